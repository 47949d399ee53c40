"""Shared set-up for whole-step GPU parity tests and bench.py: builds the
synthetic drafter on the device, commits each sequence's context through
dflash_kv_commit, and computes the oracle's view of the same inputs.
(Test and measurement infrastructure; the oracle parts run on the CPU.)"""
from __future__ import annotations

import numpy as np

from block_diffusion_speculative_draft_gb300 import synth


def contexts(cfg) -> np.ndarray:
    if cfg.ctx_range is not None:
        return synth.ragged_contexts(cfg.seed, "ctx", cfg.b, *cfg.ctx_range)
    c = list(cfg.ctx) * cfg.b if len(cfg.ctx) == 1 else list(cfg.ctx)
    return np.asarray(c[:cfg.b], np.int32)


def context_hidden(cfg, j: int, C: int) -> np.ndarray:
    return synth.target_hidden(cfg.seed, f"ctx{j}", C, cfg.k * cfg.H)


def commit_contexts(api, torch, cfg, model, kv, ws, ctx, rows_per_seq: int, dev):
    """Prefill each sequence's committed context in chunks of rows_per_seq
    hidden rows (n = rows - 1 per chunk, -1 once a sequence is done)."""
    b = cfg.b
    W = cfg.k * cfg.H
    hids = [context_hidden(cfg, j, int(ctx[j])) for j in range(b)]
    cmax = int(max(ctx))
    for c0 in range(0, cmax, rows_per_seq):
        blk = np.zeros((b, rows_per_seq, W), np.float16)
        n = np.full(b, -1, np.int32)
        for j in range(b):
            r = min(rows_per_seq, int(ctx[j]) - c0)
            if r > 0:
                blk[j, :r] = hids[j][c0:c0 + r]
                n[j] = r - 1
        api.dflash_kv_commit(model, kv, torch.from_numpy(blk).to(dev), torch.from_numpy(n).to(dev), ws)
    return hids
