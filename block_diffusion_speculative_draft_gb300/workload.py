"""Synthetic workload set-up shared by bench.py and the GPU tests: per-sequence
context lengths, the target hidden rows of each context, and the prefill of
the draft KV cache through dflash_kv_commit."""
from __future__ import annotations

import numpy as np

from . import synth


def contexts(cfg) -> np.ndarray:
    """Committed context length per sequence: the workload's fixed lengths or
    a seeded uniform draw for ragged batches."""
    if cfg.ctx_range is not None:
        return synth.ragged_contexts(cfg.seed, "ctx", cfg.b, *cfg.ctx_range)
    c = list(cfg.ctx) * cfg.b if len(cfg.ctx) == 1 else list(cfg.ctx)
    return np.asarray(c[:cfg.b], np.int32)


def context_hidden(cfg, j: int, C: int) -> np.ndarray:
    return synth.target_hidden(cfg.seed, f"ctx{j}", C, cfg.k * cfg.H)


def commit_contexts(api, torch, cfg, model, kv, ws, ctx, rows_per_seq: int, dev):
    """Prefill each sequence's context in chunks of rows_per_seq target hidden
    rows (n = rows - 1 per chunk, -1 once a sequence is complete).  Returns the
    host hidden rows of every sequence."""
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
