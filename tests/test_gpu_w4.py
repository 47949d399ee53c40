"""W4A16 (int4 codes, one fp16 scale per row and 128-column group) on the
GPU against the oracle, through the C ABI.

Tolerances as for int8: packed codes and scales bit-exact; the projection
alone within 1e-3 of the output's max-abs; a whole drafter step within
2e-2 x max-abs for hidden states and logits, drafts bit-exact where the
oracle's top-2 margin exceeds 1e-2, committed K/V within 1e-2 x max-abs.
"""
import dataclasses

import numpy as np
import pytest

from oracle import dflash_oracle as O
from block_diffusion_speculative_draft_gb300 import synth
from block_diffusion_speculative_draft_gb300.configs import TINY, QWEN3_4B
from block_diffusion_speculative_draft_gb300.workload import commit_contexts, contexts
from tests.gpu_util import gpu_available, rel_err, unpack_tiled_q4

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not gpu_available(), reason="needs a GPU")]

if gpu_available():
    import torch
    from block_diffusion_speculative_draft_gb300 import api
    from tests.test_gpu_drafter import _check_cache, _check_draft
    DEV = torch.device("cuda:0")


@pytest.mark.parametrize("N,K,layout,dtype", [
    (128, 128, 0, "f32"), (256, 512, 0, "f16"), (384, 256, 0, "bf16"), (256, 384, 1, "f32"), (768, 512, 1, "f16")])
def test_pack4_bit_exact(N, K, layout, dtype):
    rng = np.random.default_rng(N + K + 4)
    w = (rng.standard_normal((N, K)) * rng.lognormal(-3, 1, (N, 1))).astype(np.float32)
    w[3] = 0.0
    w[5, 128:256] = 0.0  # one zero group
    if dtype == "f16":
        w = w.astype(np.float16)
        tw = torch.from_numpy(w).to(DEV)
        w = w.astype(np.float32)
    elif dtype == "bf16":
        w = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(w))
        tw = torch.from_numpy(w).to(DEV).to(torch.bfloat16)
    else:
        tw = torch.from_numpy(w).to(DEV)
    qd, sd = api.dflash_pack_w4a16(tw, layout)
    torch.cuda.synchronize()
    q_ref, s_ref = O.pack_w4a16(w)
    assert np.array_equal(sd.cpu().numpy().view(np.uint16), s_ref.view(np.uint16))
    q, s_tiles = unpack_tiled_q4(qd.cpu().numpy(), N, K, layout)
    assert np.array_equal(s_tiles.view(np.uint16), s_ref.view(np.uint16))
    assert np.array_equal(q, q_ref)


@pytest.mark.parametrize("M,N,K,layout", [
    (16, 768, 512, 0), (16, 512, 1536, 0), (15, 3072, 512, 1), (5, 256, 256, 0), (32, 1024, 2560, 0),
    (17, 384, 640, 0), (128, 512, 1024, 0), (1, 128, 128, 0), (40, 640, 384, 1)])
def test_w4a16_linear(M, N, K, layout):
    q, s = synth.w4_grid(5, f"lin4{M}{N}{K}", N, K)
    x = synth.target_hidden(5, f"x{M}{K}", M, K)
    qd, _ = api.dflash_pack_w4a16(torch.from_numpy(synth.w4_float(q, s)).to(DEV), layout)
    desc = api.w8_desc(qd, None, N, K, layout, bits=4)
    y = api.dflash_w8a16_linear(desc, torch.from_numpy(x).to(DEV)).cpu().numpy()
    ref = O.linear(x.astype(np.float64), O.dequant_w4(q, s))
    assert rel_err(y, ref) <= 1e-3


def _w4_model(cfg, rps, extra_cap=64):
    W = synth.drafter_weights(cfg, bits=4)
    model = api.DeviceDrafter(cfg, synth.FloatWeights(W), DEV, bits=4)
    ctx = contexts(cfg)
    kv = api.KVCache(cfg, cfg.b, int(ctx.max()) + extra_cap, DEV)
    ws = api.workspace(cfg, cfg.b, rps, DEV)
    hids = commit_contexts(api, torch, cfg, model, kv, ws, ctx, rps, DEV)
    return W, model, ctx, kv, ws, hids


@pytest.mark.parametrize("cfg", [TINY, dataclasses.replace(TINY, b=3, ctx=(), ctx_range=(20, 90), seed=1400)],
                         ids=["tiny", "tiny-b3-ragged"])
def test_w4_tiny_commit_and_draft(cfg):
    W, model, ctx, kv, ws, hids = _w4_model(cfg, 16)
    _check_cache(cfg, W, kv, hids, ctx, range(cfg.b))
    _check_draft(cfg, W, model, kv, ws, hids, ctx)


def test_w4_qwen3_4b_shape():
    cfg = QWEN3_4B
    W, model, ctx, kv, ws, hids = _w4_model(cfg, cfg.B, extra_cap=cfg.B)
    t0 = synth.tokens(cfg.seed, "t0", cfg.b, cfg.V)
    last = torch.from_numpy(t0).to(DEV)
    draft = torch.empty((cfg.b, cfg.B - 1), dtype=torch.int32, device=DEV)
    hidden = torch.empty((cfg.b, cfg.B - 1, cfg.H), dtype=torch.float32, device=DEV)
    logits = torch.empty((cfg.b, cfg.B - 1, cfg.V), dtype=torch.float32, device=DEV)
    api.dflash_draft_block(model, kv, last, draft, ws, hidden=hidden, logits=logits)
    fast = torch.empty_like(draft)
    api.dflash_draft_block(model, kv, last, fast, ws)
    torch.cuda.synchronize()
    assert api.dflash_get_status() == 0
    D = O.Drafter(cfg, W, cache=False)
    Ks, Vs = O.context_kv(D, hids[0])
    n = int(ctx[0])
    for l in sorted({0, cfg.L - 1}):
        gk = kv.k[l, 0, :, :n, :].float().cpu().numpy().transpose(1, 0, 2)
        gv = kv.v[l, 0, :, :n, :].float().cpu().numpy().transpose(1, 0, 2)
        assert rel_err(gk, Ks[l]) <= 1e-2 and rel_err(gv, Vs[l]) <= 1e-2
    ref = O.draft_block(D, int(t0[0]), Ks, Vs)
    assert rel_err(hidden[0].cpu().numpy(), ref["hidden"]) <= 2e-2
    assert rel_err(logits[0].cpu().numpy(), ref["logits"]) <= 2e-2
    ok = ref["margin"] > 1e-2
    assert np.array_equal(draft[0].cpu().numpy()[ok], ref["draft"][ok])
    assert np.array_equal(fast[0].cpu().numpy()[ok], ref["draft"][ok])
    D.drop()
