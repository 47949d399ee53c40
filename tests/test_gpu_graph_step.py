"""The timed step as the benchmark runs it: reset the committed length, draft
the block, greedy verify-accept against the target's logits, commit the
accepted rows, all captured in one CUDA graph and replayed.

Replays must give what eager calls give, bit for bit, and what the oracle
gives: drafts (where the oracle's top-2 margin exceeds 1e-2), accept outputs
(exactly), committed K/V rows (within 1e-2 of max-abs) and lengths.
"""
import numpy as np
import pytest

from oracle import dflash_oracle as O
from block_diffusion_speculative_draft_gb300 import synth
from block_diffusion_speculative_draft_gb300.configs import TINY, QWEN3_4B
from block_diffusion_speculative_draft_gb300.workload import commit_contexts, contexts
from tests.gpu_util import gpu_available, rel_err

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not gpu_available(), reason="needs a GPU")]

if gpu_available():
    import torch
    from block_diffusion_speculative_draft_gb300 import api
    DEV = torch.device("cuda:0")


def _run(cfg, check_draft_vs_oracle: bool):
    W = synth.drafter_weights(cfg)
    model = api.DeviceDrafter(cfg, synth.FloatWeights(W), DEV)
    ctx = contexts(cfg)
    b, B = cfg.b, cfg.B
    kv = api.KVCache(cfg, b, int(ctx.max()) + 2 * B, DEV)
    ws = api.workspace(cfg, b, B, DEV)
    hids = commit_contexts(api, torch, cfg, model, kv, ws, ctx, B, DEV)
    torch.cuda.synchronize()
    len0 = kv.len.clone()
    t0_host = synth.tokens(cfg.seed, "t0", b, cfg.V)
    t0 = torch.from_numpy(t0_host).to(DEV)
    draft = torch.empty((b, B - 1), dtype=torch.int32, device=DEV)
    api.dflash_draft_block(model, kv, t0, draft, ws)
    torch.cuda.synchronize()
    draft_eager = draft.cpu().numpy()
    nacc = synth.accept_lengths(cfg.seed, "acc", b, B - 1, cfg.accept_mean)
    lg_host = synth.verify_logits(cfg.seed, "verify", draft_eager, cfg.R, cfg.V, nacc)
    logits = torch.from_numpy(lg_host).to(DEV)
    blk_host = np.stack([synth.target_hidden(cfg.seed, f"blk{j}", B, cfg.k * cfg.H) for j in range(b)])
    blk = torch.from_numpy(blk_host).to(DEV)
    n_out = torch.empty(b, dtype=torch.int32, device=DEV)
    corr = torch.empty(b, dtype=torch.int32, device=DEV)
    emitted = torch.empty((b, cfg.R), dtype=torch.int32, device=DEV)
    nxt = torch.empty(b, dtype=torch.int32, device=DEV)
    vws = torch.zeros(api.dflash_verify_workspace_size(b, cfg.R, cfg.V), dtype=torch.uint8, device=DEV)

    def step():
        kv.len.copy_(len0)
        api.dflash_draft_block(model, kv, t0, draft, ws)
        api.dflash_verify_accept(logits, draft, n_out, corr, emitted, nxt, vws)
        api.dflash_kv_commit(model, kv, blk, n_out, ws)

    step()  # eager
    torch.cuda.synchronize()
    eager = [x.cpu().numpy() for x in (draft, n_out, corr, emitted, nxt, kv.len, kv.k, kv.v)]
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream(device=DEV)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    with torch.cuda.graph(g):
        step()
    for rep in range(3):
        g.replay()
        torch.cuda.synchronize()
        got = [x.cpu().numpy() for x in (draft, n_out, corr, emitted, nxt, kv.len, kv.k, kv.v)]
        for a, e in zip(got, eager):
            assert np.array_equal(a.view(np.uint8), e.view(np.uint8)), rep
    assert api.dflash_get_status() == 0

    dr, n, c, em, nx, lens, kc, vc = eager
    assert np.array_equal(dr, draft_eager)
    D = O.Drafter(cfg, W)
    for j in range(b):
        on, oc, oem, onx = O.verify_accept(lg_host[j], dr[j])
        assert (n[j], c[j], nx[j]) == (on, oc, onx)
        assert np.array_equal(em[j], oem)
        assert n[j] == nacc[j]
        keep = O.commit_rows(on, B)
        C = int(ctx[j])
        assert lens[j] == C + keep
        cr = O.context_rows(D, blk_host[j][:keep])
        for l in range(cfg.L):
            k, v = O.context_kv_layer(D, l, cr, C + np.arange(keep))
            assert rel_err(kc[l, j, :, C:C + keep].transpose(1, 0, 2), k) <= 1e-2
            assert rel_err(vc[l, j, :, C:C + keep].transpose(1, 0, 2), v) <= 1e-2
        if check_draft_vs_oracle:
            Ks, Vs = O.context_kv(D, hids[j])
            ref = O.draft_block(D, int(t0_host[j]), Ks, Vs, want_logits=False)
            ok = ref["margin"] > 1e-2
            assert ok.sum() >= (B - 1) // 2
            assert np.array_equal(dr[j][ok], ref["draft"][ok])
    D.drop()


@pytest.mark.parametrize("early", [False, True], ids=["stream-order", "early-launch"])
def test_graph_step_tiny(early):
    with api.launch_mode(api.LAUNCH_EARLY if early else api.LAUNCH_STREAM_ORDER):
        _run(TINY, True)


@pytest.mark.parametrize("early", [False, True], ids=["stream-order", "early-launch"])
def test_graph_step_qwen3_4b_shape(early):
    with api.launch_mode(api.LAUNCH_EARLY if early else api.LAUNCH_STREAM_ORDER):
        _run(QWEN3_4B, True)
