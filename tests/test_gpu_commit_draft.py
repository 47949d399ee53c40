"""Commit and draft in one pass (dflash_commit_draft_block) against the two
separate calls and against the oracle.

From identical states, the fused pass must leave the same lengths, the same
cache (within fp16 storage, 1e-2 x max-abs) and the same block outputs
(hidden states and logits within 2e-2 x max-abs, drafts equal wherever the
top-2 logit margin exceeds 1e-2) as dflash_kv_commit followed by
dflash_draft_block; and the oracle, given the grown context, must agree with
it on the same terms.
"""
import dataclasses

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

# the last case has the 27B-class attention shape (160 query rows per kv
# head) over 4000 context rows: the tensor-memory attention, with the rows
# the folded commit appends gathered after its dependency wait
CASES = [TINY, dataclasses.replace(TINY, b=3, ctx=(), ctx_range=(20, 90), seed=1200), QWEN3_4B,
         dataclasses.replace(TINY, nq=40, nkv=8, d=128, B=32, D=None, ctx=(4000,), seed=1210)]


@pytest.mark.parametrize("cfg", CASES, ids=["tiny", "tiny-b3-ragged", "qwen3-4b", "tiny-two-block-ctx4000"])
def test_commit_draft_matches_commit_then_draft(cfg):
    b, B = cfg.b, cfg.B
    rps = B
    W = synth.drafter_weights(cfg)
    model = api.DeviceDrafter(cfg, synth.FloatWeights(W), DEV)
    ctx = contexts(cfg)
    cap = int(ctx.max()) + 2 * B
    kvs, wss = [], []
    for _ in range(2):
        kv = api.KVCache(cfg, b, cap, DEV)
        ws = api.workspace(cfg, b, rps, DEV)
        hids = commit_contexts(api, torch, cfg, model, kv, ws, ctx, rps, DEV)
        kvs.append(kv)
        wss.append(ws)
    blk = np.stack([synth.target_hidden(cfg.seed, f"cd{j}", rps, cfg.k * cfg.H) for j in range(b)])
    nacc = synth.accept_lengths(cfg.seed, "cd-acc", b, B - 1, cfg.accept_mean)
    nacc[0] = B - 1  # one full accept: every row committed
    blk_d = torch.from_numpy(blk).to(DEV)
    n_d = torch.from_numpy(nacc.astype(np.int32)).to(DEV)
    t0 = torch.from_numpy(synth.tokens(cfg.seed, "cd-t0", b, cfg.V)).to(DEV)
    outs = []
    for path in ("two calls", "one pass"):
        kv, ws = kvs[len(outs)], wss[len(outs)]
        draft = torch.empty((b, B - 1), dtype=torch.int32, device=DEV)
        hidden = torch.empty((b, B - 1, cfg.H), dtype=torch.float32, device=DEV)
        logits = torch.empty((b, B - 1, cfg.V), dtype=torch.float32, device=DEV)
        if path == "two calls":
            api.dflash_kv_commit(model, kv, blk_d, n_d, ws)
            api.dflash_draft_block(model, kv, t0, draft, ws, hidden=hidden, logits=logits)
        else:
            api.dflash_commit_draft_block(model, kv, blk_d, n_d, t0, draft, ws, hidden=hidden, logits=logits)
        torch.cuda.synchronize()
        assert api.dflash_get_status() == 0
        outs.append((draft.cpu().numpy(), hidden.cpu().numpy(), logits.cpu().numpy(), kv.len.cpu().numpy()))
    (da, ha, la, lena), (db, hb, lb, lenb) = outs
    assert np.array_equal(lena, lenb)
    assert np.array_equal(lena, ctx + nacc + 1)
    for l in range(cfg.L):
        for j in range(b):
            n = int(lena[j])
            ka = kvs[0].k[l, j, :, :n].float().cpu().numpy()
            kb = kvs[1].k[l, j, :, :n].float().cpu().numpy()
            va = kvs[0].v[l, j, :, :n].float().cpu().numpy()
            vb = kvs[1].v[l, j, :, :n].float().cpu().numpy()
            assert rel_err(kb, ka) <= 1e-2 and rel_err(vb, va) <= 1e-2
    D = O.Drafter(cfg, W, cache=False)
    for j in range(b):
        assert rel_err(hb[j], ha[j]) <= 2e-2 and rel_err(lb[j], la[j]) <= 2e-2
        srt = np.sort(la[j], axis=-1)
        ok = (srt[:, -1] - srt[:, -2]) > 1e-2
        assert np.array_equal(db[j][ok], da[j][ok])
    # the oracle with the grown context (sequence 0: a full accept)
    j = 0
    grown = np.concatenate([hids[j], blk[j][: int(nacc[j]) + 1]], axis=0)
    Ks, Vs = O.context_kv(D, grown)
    ref = O.draft_block(D, int(t0[j]), Ks, Vs)
    assert rel_err(hb[j], ref["hidden"]) <= 2e-2
    assert rel_err(lb[j], ref["logits"]) <= 2e-2
    ok = ref["margin"] > 1e-2
    assert np.array_equal(db[j][ok], ref["draft"][ok])
    D.drop()
