"""Bitwise repeatability of the draft pass.

Every reduction in the pass has a fixed order (split-K in split order through
cluster shared memory, the attention merge in split order, no float atomics),
so repeated passes over the same cache must give identical bits.  A pass that
drifts between runs has a race even when each run stays within the oracle
tolerance.  Eight sequences of the batched Qwen3-8B shape give 128 block rows,
the launches of the 128-row projection kernel; the 27B-class shape at 4096
context rows gives the 32-row tensor-memory projections (two CTAs per SM)
and the tensor-memory attention.  One layer keeps both short.
"""
import dataclasses

import pytest

from block_diffusion_speculative_draft_gb300 import configs, synth
from block_diffusion_speculative_draft_gb300.workload import commit_contexts, contexts
from tests.gpu_util import gpu_available

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not gpu_available(), reason="needs a GPU")]

if gpu_available():
    import torch
    from block_diffusion_speculative_draft_gb300 import api
    DEV = torch.device("cuda:0")


CASES = [("b8-qwen3-8b", "early"), ("b8-qwen3-8b", "stream"), ("27b-class-ctx4096", "early")]


def _cfg(name):
    if name == "b8-qwen3-8b":
        return dataclasses.replace(configs.BATCHED_8B, L=1, ctx=(2048,), ctx_range=None)
    return dataclasses.replace(configs.DENSE_27B, L=1, ctx=(4096,))


@pytest.mark.parametrize("shape,mode", CASES)
def test_draft_pass_repeats_bitwise(shape, mode):
    cfg = _cfg(shape)
    with api.launch_mode(api.LAUNCH_EARLY if mode == "early" else api.LAUNCH_STREAM_ORDER):
        W = synth.drafter_weights(cfg)
        model = api.DeviceDrafter(cfg, synth.FloatWeights(W), DEV)
        ctx = contexts(cfg)
        kv = api.KVCache(cfg, cfg.b, int(ctx.max()) + cfg.B, DEV)
        ws = api.workspace(cfg, cfg.b, 64, DEV)
        commit_contexts(api, torch, cfg, model, kv, ws, ctx, 64, DEV)
        t0 = torch.from_numpy(synth.tokens(cfg.seed, "t0", cfg.b, cfg.V)).to(DEV)
        outs = []
        for _ in range(6):
            draft = torch.empty((cfg.b, cfg.B - 1), dtype=torch.int32, device=DEV)
            hidden = torch.empty((cfg.b, cfg.B - 1, cfg.H), dtype=torch.float32, device=DEV)
            api.dflash_draft_block(model, kv, t0, draft, ws, hidden=hidden)
            torch.cuda.synchronize()
            outs.append((draft.clone(), hidden.clone()))
        assert api.dflash_get_status() == 0
        for d, h in outs[1:]:
            assert torch.equal(h, outs[0][1]), float((h - outs[0][1]).abs().max())
            assert torch.equal(d, outs[0][0])
