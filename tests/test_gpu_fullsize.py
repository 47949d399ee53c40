"""Whole-step GPU parity at the full workload sizes (Qwen3-4B-shaped,
Qwen3-8B-shaped, 27B-class at 64 / 2048 / 4096 context rows, batched 8 x
Qwen3-8B-shaped with ragged contexts), in the launch configuration bench.py
times (early-launch mode, one stream), through the C ABI.

The oracle recomputes sampled sequences one by one (all of them when b = 1,
two of eight for the batched workload).  Tolerances as in the tiny tests:
hidden states and logits within 2e-2 x max-abs, draft tokens bit-exact where
the oracle's top-2 margin exceeds 1e-2, accept outputs bit-exact, committed
K/V rows within 1e-2 x max-abs, rejected rows never written.
"""
import numpy as np
import pytest

from oracle import dflash_oracle as O
from block_diffusion_speculative_draft_gb300 import configs, synth
from block_diffusion_speculative_draft_gb300.workload import commit_contexts, contexts
from tests.gpu_util import gpu_available, rel_err

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not gpu_available(), reason="needs a GPU")]

if gpu_available():
    import torch
    from block_diffusion_speculative_draft_gb300 import api
    DEV = torch.device("cuda:0")

CASES = ([(configs.QWEN3_4B, [0]), (configs.QWEN3_8B, [0])]
         + [(configs.DENSE_27B.with_ctx((c,)), [0]) for c in configs.DENSE_27B_CTX_SWEEP]
         + [(configs.BATCHED_8B, [1, 6])])


@pytest.fixture(autouse=True)
def _early_launch():
    with api.launch_mode(api.LAUNCH_EARLY):
        yield


@pytest.mark.parametrize("cfg,seqs", CASES, ids=[f"{c.name}-ctx{c.ctx[0] if c.ctx else 'ragged'}" for c, _ in CASES])
def test_fullsize_step(cfg, seqs):
    W = synth.drafter_weights(cfg)
    model = api.DeviceDrafter(cfg, synth.FloatWeights(W), DEV)
    ctx = contexts(cfg)
    b = cfg.b
    rps = 64 if b > 1 else cfg.B
    kv = api.KVCache(cfg, b, int(ctx.max()) + cfg.B, DEV)
    ws = api.workspace(cfg, b, max(rps, cfg.B), DEV)
    hids = commit_contexts(api, torch, cfg, model, kv, ws, ctx, rps, DEV)
    t0 = synth.tokens(cfg.seed, "t0", b, cfg.V)
    last = torch.from_numpy(t0).to(DEV)
    paths = [api.dflash_draft_block]
    outs = []
    for fn in paths:
        draft = torch.empty((b, cfg.B - 1), dtype=torch.int32, device=DEV)
        hidden = torch.empty((b, cfg.B - 1, cfg.H), dtype=torch.float32, device=DEV)
        logits = torch.empty((b, cfg.B - 1, cfg.V), dtype=torch.float32, device=DEV)
        fn(model, kv, last, draft, ws, hidden=hidden, logits=logits)
        torch.cuda.synchronize()
        assert api.dflash_get_status() == 0
        outs.append((draft.cpu().numpy(), hidden.cpu().numpy(), logits.cpu().numpy()))
    # the argmax-only pass (no optional outputs: final RMSNorm folded away)
    draft_fast = torch.empty((b, cfg.B - 1), dtype=torch.int32, device=DEV)
    api.dflash_draft_block(model, kv, last, draft_fast, ws)
    torch.cuda.synchronize()
    assert api.dflash_get_status() == 0
    draft_fast = draft_fast.cpu().numpy()
    D = O.Drafter(cfg, W, cache=False)
    for j in seqs:
        Ks, Vs = O.context_kv(D, hids[j])
        ref = O.draft_block(D, int(t0[j]), Ks, Vs)
        ok = ref["margin"] > 1e-2
        for draft, hidden, logits in outs:
            assert rel_err(hidden[j], ref["hidden"]) <= 2e-2
            assert rel_err(logits[j], ref["logits"]) <= 2e-2
            assert np.array_equal(draft[j][ok], ref["draft"][ok])
        assert np.array_equal(draft_fast[j][ok], ref["draft"][ok])
        # committed context K/V of this sequence, two layers sampled
        C = int(ctx[j])
        for l in sorted({0, cfg.L - 1}):
            gk = kv.k[l, j, :, :C, :].float().cpu().numpy().transpose(1, 0, 2)
            gv = kv.v[l, j, :, :C, :].float().cpu().numpy().transpose(1, 0, 2)
            assert rel_err(gk, Ks[l]) <= 1e-2 and rel_err(gv, Vs[l]) <= 1e-2
    # verify-accept on the GPU drafts (planted target logits) and the commit
    # of the accepted rows with rollback of the rest
    drafts = outs[0][0]
    nacc = synth.accept_lengths(cfg.seed, "acc", b, cfg.B - 1, cfg.accept_mean)
    lg = synth.verify_logits(cfg.seed, "verify", drafts, cfg.R, cfg.V, nacc)
    n_out = torch.empty(b, dtype=torch.int32, device=DEV)
    corr = torch.empty(b, dtype=torch.int32, device=DEV)
    emitted = torch.empty((b, cfg.R), dtype=torch.int32, device=DEV)
    api.dflash_verify_accept(torch.from_numpy(lg).to(DEV), torch.from_numpy(drafts).to(DEV), n_out, corr, emitted)
    blk = np.stack([synth.target_hidden(cfg.seed, f"blk{j}", cfg.B, cfg.k * cfg.H) for j in range(b)])
    len_before = kv.len.cpu().numpy().copy()
    api.dflash_kv_commit(model, kv, torch.from_numpy(blk).to(DEV), n_out, ws)
    torch.cuda.synchronize()
    n_gpu = n_out.cpu().numpy()
    for j in range(b):
        n, c, e, _ = O.verify_accept(lg[j], drafts[j])
        assert n_gpu[j] == n == nacc[j] and int(corr[j]) == c
        assert np.array_equal(emitted[j].cpu().numpy(), e)
    assert np.array_equal(kv.len.cpu().numpy(), len_before + n_gpu + 1)
    j = seqs[0]
    C, n = int(len_before[j]), int(n_gpu[j])
    c_rows = O.context_rows(D, blk[j][:n + 1])
    k_ref, v_ref = O.context_kv_layer(D, 0, c_rows, C + np.arange(n + 1))
    gk = kv.k[0, j, :, C:C + n + 1, :].float().cpu().numpy().transpose(1, 0, 2)
    gv = kv.v[0, j, :, C:C + n + 1, :].float().cpu().numpy().transpose(1, 0, 2)
    assert rel_err(gk, k_ref) <= 1e-2 and rel_err(gv, v_ref) <= 1e-2
    assert not kv.k[0, j, :, C + n + 1:, :].any()  # rejected rows never written
