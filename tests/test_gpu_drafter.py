"""Whole-step GPU parity: dflash_kv_commit + dflash_draft_block against the
oracle, through the C ABI.

Tolerances (from the drafter contract): hidden states and logits within
max-abs error <= 2e-2 x the oracle tensor's max-abs; draft tokens bit-exact
wherever the oracle's top-2 logit margin exceeds 1e-2; the committed K/V
cache within 1e-2 x max-abs (fp16 storage); lengths and untouched rows exact.
"""
import numpy as np
import pytest

from oracle import dflash_oracle as O
from block_diffusion_speculative_draft_gb300 import synth
from block_diffusion_speculative_draft_gb300.configs import TINY
from block_diffusion_speculative_draft_gb300.workload import commit_contexts, contexts
from tests.gpu_util import gpu_available, rel_err

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not gpu_available(), reason="needs a GPU")]

if gpu_available():
    import torch
    from block_diffusion_speculative_draft_gb300 import api
    DEV = torch.device("cuda:0")

TOL = 2e-2


def _setup(cfg, rows_per_seq, extra_cap=64):
    W = synth.drafter_weights(cfg)
    model = api.DeviceDrafter(cfg, synth.FloatWeights(W), DEV)
    ctx = contexts(cfg)
    kv = api.KVCache(cfg, cfg.b, int(ctx.max()) + extra_cap, DEV)
    ws = api.workspace(cfg, cfg.b, rows_per_seq, DEV)
    hids = commit_contexts(api, torch, cfg, model, kv, ws, ctx, rows_per_seq, DEV)
    return W, model, ctx, kv, ws, hids


def _check_draft(cfg, W, model, kv, ws, hids, ctx, seqs=None):
    b = cfg.b
    t0 = synth.tokens(cfg.seed, "t0", b, cfg.V)
    last = torch.from_numpy(t0).to(DEV)
    draft = torch.empty((b, cfg.B - 1), dtype=torch.int32, device=DEV)
    hidden = torch.empty((b, cfg.B - 1, cfg.H), dtype=torch.float32, device=DEV)
    logits = torch.empty((b, cfg.B - 1, cfg.V), dtype=torch.float32, device=DEV)
    fn = api.dflash_draft_block
    fn(model, kv, last, draft, ws, hidden=hidden, logits=logits)
    # without the optional outputs the final RMSNorm is folded into the last
    # GEMM (argmax only); its drafts must meet the same bar
    draft_fast = torch.empty_like(draft)
    fn(model, kv, last, draft_fast, ws)
    torch.cuda.synchronize()
    assert api.dflash_get_status() == 0
    D = O.Drafter(cfg, W)
    seqs = range(b) if seqs is None else seqs
    out = {}
    for j in seqs:
        Ks, Vs = O.context_kv(D, hids[j])
        ref = O.draft_block(D, int(t0[j]), Ks, Vs)
        eh = rel_err(hidden[j].cpu().numpy(), ref["hidden"])
        el = rel_err(logits[j].cpu().numpy(), ref["logits"])
        assert eh <= TOL, (j, eh)
        assert el <= TOL, (j, el)
        ok = ref["margin"] > 1e-2
        got = draft[j].cpu().numpy()
        assert np.array_equal(got[ok], ref["draft"][ok]), (j, got, ref["draft"], ref["margin"])
        fast = draft_fast[j].cpu().numpy()
        assert np.array_equal(fast[ok], ref["draft"][ok]), (j, fast, ref["draft"], ref["margin"])
        out[j] = (ref, Ks, Vs)
    D.drop()
    return draft.cpu().numpy(), out


def _check_cache(cfg, W, kv, hids, ctx, seqs):
    D = O.Drafter(cfg, W)
    kc = kv.k.cpu().numpy()
    vc = kv.v.cpu().numpy()
    lens = kv.len.cpu().numpy()
    for j in seqs:
        C = int(ctx[j])
        assert lens[j] == C
        Ks, Vs = O.context_kv(D, hids[j])
        for l in range(cfg.L):
            gk = kc[l, j, :, :C, :].transpose(1, 0, 2)
            gv = vc[l, j, :, :C, :].transpose(1, 0, 2)
            assert rel_err(gk, Ks[l]) <= 1e-2
            assert rel_err(gv, Vs[l]) <= 1e-2
            assert not kc[l, j, :, C:, :].any()  # nothing past the committed rows


def test_tiny_commit_and_draft():
    cfg = TINY
    W, model, ctx, kv, ws, hids = _setup(cfg, cfg.B)
    _check_cache(cfg, W, kv, hids, ctx, range(cfg.b))
    _check_draft(cfg, W, model, kv, ws, hids, ctx)


def test_tiny_long_context_multi_tile_splits():
    # a 1000-row context gives attention splits of several 64-key tiles, the
    # path where helper warps compute the second key half of every tile
    cfg = TINY.with_ctx((1000,))
    W, model, ctx, kv, ws, hids = _setup(cfg, 64)
    _check_draft(cfg, W, model, kv, ws, hids, ctx)


@pytest.mark.parametrize("lens", [(4000,), (4000, 100)])
def test_tiny_two_block_query_tile_long_context(lens):
    """The attention shape of the 27B-class drafter (40 query heads over 8 kv
    heads, d 128, block 32: 160 query rows per kv head, two 128-row MMA
    blocks) over a long context, where each split gets six 64-key tiles: the
    launch that runs the tensor-memory attention.  With a 100-row second
    sequence most of that sequence's splits hold no keys at all."""
    import dataclasses
    cfg = dataclasses.replace(TINY, nq=40, nkv=8, d=128, B=32, D=None, b=len(lens), ctx=lens,
                              seed=1200 + len(lens))
    W, model, ctx, kv, ws, hids = _setup(cfg, 256)
    _check_draft(cfg, W, model, kv, ws, hids, ctx)


def test_tiny_prefill_chunk_sizes_agree():
    # the same context committed 5 rows or 64 rows at a time gives one cache
    cfg = TINY.with_ctx((37,))
    W, model, ctx, kv, ws, hids = _setup(cfg, 5)
    ws64 = api.workspace(cfg, cfg.b, 64, DEV)
    kv2 = api.KVCache(cfg, cfg.b, kv.cap, DEV)
    commit_contexts(api, torch, cfg, model, kv2, ws64, ctx, 64, DEV)
    torch.cuda.synchronize()
    assert torch.equal(kv.len, kv2.len)
    assert torch.equal(kv.k, kv2.k) and torch.equal(kv.v, kv2.v)
    _check_cache(cfg, W, kv, hids, ctx, range(cfg.b))


def test_tiny_loop_commit_rollback():
    """draft -> verify (planted logits) -> commit of rows 0..n: the cache gains
    exactly n+1 rows at positions len..len+n; rows of the rejected suffix are
    never written; the next draft matches the oracle on the grown context."""
    cfg = TINY
    W, model, ctx, kv, ws, hids = _setup(cfg, cfg.B)
    drafts, _ = _check_draft(cfg, W, model, kv, ws, hids, ctx)
    R, Dn = cfg.B, cfg.B - 1
    nacc = np.array([5], np.int32)
    lg = synth.verify_logits(cfg.seed, "loop", drafts, R, cfg.V, nacc)
    n_out = torch.empty(1, dtype=torch.int32, device=DEV)
    corr = torch.empty(1, dtype=torch.int32, device=DEV)
    api.dflash_verify_accept(torch.from_numpy(lg).to(DEV), torch.from_numpy(drafts).to(DEV), n_out, corr)
    blk = synth.target_hidden(cfg.seed, "blk", cfg.B, cfg.k * cfg.H)
    api.dflash_kv_commit(model, kv, torch.from_numpy(blk[None]).to(DEV), n_out, ws)
    torch.cuda.synchronize()
    assert int(n_out[0]) == 5
    C = int(ctx[0])
    assert int(kv.len[0]) == C + 6
    hids2 = [np.concatenate([hids[0], blk[:6]])]
    _check_cache(cfg, W, kv, hids2, np.array([C + 6]), [0])
    _check_draft(cfg, W, model, kv, ws, hids2, np.array([C + 6]))


def test_capacity_overflow_flags_and_skips():
    cfg = TINY.with_ctx((40,))
    W = synth.drafter_weights(cfg)
    model = api.DeviceDrafter(cfg, synth.FloatWeights(W), DEV)
    kv = api.KVCache(cfg, 1, 48, DEV)
    ws = api.workspace(cfg, 1, cfg.B, DEV)
    api.dflash_get_status(clear=True)
    hid = synth.target_hidden(cfg.seed, "cap", 3 * cfg.B, cfg.k * cfg.H)
    n = torch.tensor([cfg.B - 1], dtype=torch.int32, device=DEV)
    for c in range(3):  # 16 + 16 fit in 48, the third 16 fit, a fourth would not
        api.dflash_kv_commit(model, kv, torch.from_numpy(hid[None, c * 16:(c + 1) * 16]).to(DEV), n, ws)
    assert api.dflash_get_status() == 0 and int(kv.len[0]) == 48
    before = kv.k.clone()
    api.dflash_kv_commit(model, kv, torch.from_numpy(hid[None, :16]).to(DEV), n, ws)
    st = api.dflash_get_status()
    assert st & api.DEV_KV_CAPACITY
    assert int(kv.len[0]) == 48 and torch.equal(before, kv.k)


def test_bad_token_flag():
    cfg = TINY
    W = synth.drafter_weights(cfg)
    model = api.DeviceDrafter(cfg, synth.FloatWeights(W), DEV)
    kv = api.KVCache(cfg, 1, 64, DEV)
    ws = api.workspace(cfg, 1, cfg.B, DEV)
    api.dflash_get_status(clear=True)
    draft = torch.empty((1, cfg.B - 1), dtype=torch.int32, device=DEV)
    api.dflash_draft_block(model, kv, torch.tensor([cfg.V + 5], dtype=torch.int32, device=DEV), draft, ws)
    assert api.dflash_get_status() & api.DEV_BAD_TOKEN


@pytest.mark.parametrize("b,lo,hi", [(2, 20, 70), (4, 16, 90)])
def test_tiny_batched_ragged(b, lo, hi):
    """Ragged batches: b = 2 (32 block rows) and b = 4 (64 block rows) cover
    both launch shapes of the draft step; every sequence matches the oracle."""
    import dataclasses
    cfg = dataclasses.replace(TINY, b=b, ctx=(), ctx_range=(lo, hi), seed=1100 + b)
    W, model, ctx, kv, ws, hids = _setup(cfg, cfg.B)
    _check_cache(cfg, W, kv, hids, ctx, range(b))
    _check_draft(cfg, W, model, kv, ws, hids, ctx)
