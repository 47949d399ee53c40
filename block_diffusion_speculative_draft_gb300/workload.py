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


def commit_contexts(api, torch, cfg, model, kv, ws, ctx, rows_per_seq: int, dev, hids=None):
    """Prefill each sequence's context in chunks of rows_per_seq target hidden
    rows (n = rows - 1 per chunk, -1 once a sequence is complete).  Returns the
    host hidden rows of every sequence (drawn per sequence unless given)."""
    b = cfg.b
    W = cfg.k * cfg.H
    if hids is None:
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


# ---------------------------------------------------------------------------
# Draft || verify overlap (mirror-sd README, "How It Works": the draft runs
# concurrently with the target's verify).  The target itself is not part of
# this library, so a synthetic stand-in plays its verify forward: one int4
# QMM, logits[r] = W_t h[r], from the block's target hidden rows h [B][k H] to
# the R = B verify logits rows, with W_t a seeded int4 [V][k H] matrix (group
# scales, packed by dflash_pack_w4a16).  Its only role is to occupy the GPU
# the way a weight-streaming target forward does while a draft is in flight.
# ---------------------------------------------------------------------------
STANDIN_CHUNK = synth.LM_CHUNK  # rows per independently seeded part of W_t


def standin_chunks(cfg):
    """Row ranges [r0, r1) of the stand-in weight, one seeded int4 grid each."""
    return [(r0, min(cfg.V, r0 + STANDIN_CHUNK)) for r0 in range(0, cfg.V, STANDIN_CHUNK)]


def standin_grid(cfg, c: int):
    """Host int4 codes [r1 - r0][k H] and group scales of chunk c of W_t."""
    r0, r1 = standin_chunks(cfg)[c]
    return synth.w4_grid(cfg.seed, f"standin{c}", r1 - r0, cfg.k * cfg.H)


class TargetStandIn:
    """W_t resident on the device as one packed int4 matrix [V][k H]."""

    def __init__(self, api, torch, cfg, dev):
        V, K = cfg.V, cfg.k * cfg.H
        self.cfg = cfg
        self.q = torch.empty(api.dflash_w4a16_packed_bytes(V, K), dtype=torch.uint8, device=dev)
        per_row = api.dflash_w4a16_packed_bytes(128, K) // 128
        for c, (r0, r1) in enumerate(standin_chunks(cfg)):
            q, s = standin_grid(cfg, c)
            w = torch.from_numpy(synth.w4_float(q, s)).to(dev)
            part = self.q[r0 * per_row:r1 * per_row]
            api.dflash_pack_w4a16(w, 0, q=part, s=torch.empty((r1 - r0, K // 128), dtype=torch.float16,
                                                              device=dev))
            del w
        torch.cuda.synchronize()
        self.desc = api.w8_desc(self.q, None, V, K, 0, bits=4)

    def bytes(self) -> int:
        V, K = self.cfg.V, self.cfg.k * self.cfg.H
        return V * K // 2 + V * (K // 128) * 2


class Group:
    """One group of sequences of the overlapped loop with everything a step
    touches: drafter KV cache and workspace, last tokens, the block's target
    hidden rows, verify logits, accept outputs."""

    def __init__(self, api, torch, cfg, model, dev, ctx, hid_rows, t0, tag: str):
        b, B, V = cfg.b, cfg.B, cfg.V
        self.kv = api.KVCache(cfg, b, int(max(ctx)) + 2 * B, dev)
        self.ws = api.workspace(cfg, b, B, dev)
        self.hids = commit_contexts(api, torch, cfg, model, self.kv, self.ws, ctx, B, dev, hids=hid_rows)
        self.len0 = self.kv.len.clone()
        self.t0 = torch.from_numpy(np.asarray(t0, np.int32)).to(dev)
        self.blk_host = np.stack([synth.target_hidden(cfg.seed, f"{tag}blk{j}", B, cfg.k * cfg.H)
                                  for j in range(b)])
        self.blk = torch.from_numpy(self.blk_host).to(dev)
        self.draft = torch.empty((b, B - 1), dtype=torch.int32, device=dev)
        self.logits = torch.empty((b, cfg.R, V), dtype=torch.float32, device=dev)
        self.n = torch.empty(b, dtype=torch.int32, device=dev)
        self.corr = torch.empty(b, dtype=torch.int32, device=dev)
        self.emitted = torch.empty((b, cfg.R), dtype=torch.int32, device=dev)
        self.nxt = torch.empty(b, dtype=torch.int32, device=dev)
        self.vws = torch.zeros(api.dflash_verify_workspace_size(b, cfg.R, V), dtype=torch.uint8, device=dev)
        # the target stand-in's workspace (each group runs on its own stream)
        need = api.dflash_w8a16_linear_workspace_size(b * B, V, cfg.k * cfg.H)
        self.tws = torch.zeros(max(need, 256), dtype=torch.uint8, device=dev)


def group_step(api, cfg, model, standin, g, stream=None, reset: bool = False):
    """One speculative step of one group, stream-ordered: draft the block, the
    stand-in's verify forward, greedy verify-accept, commit of the accepted
    rows (reset first restores the committed lengths, for repeated timing)."""
    if reset:
        g.kv.len.copy_(g.len0)
    api.dflash_draft_block(model, g.kv, g.t0, g.draft, g.ws, stream=stream)
    api.dflash_w8a16_linear(standin.desc, g.blk.view(-1, cfg.k * cfg.H), ws=g.tws, stream=stream,
                            y=g.logits.view(-1, cfg.V))
    api.dflash_verify_accept(g.logits, g.draft, g.n, g.corr, g.emitted, g.nxt, g.vws, stream=stream)
    api.dflash_kv_commit(model, g.kv, g.blk, g.n, g.ws, stream=stream)


def run_serial(api, torch, cfg, model, standin, groups, reset: bool = False):
    """Every group's step, one after another on the current stream."""
    for g in groups:
        group_step(api, cfg, model, standin, g, reset=reset)


def run_overlapped(api, torch, cfg, model, standin, groups, side, reset: bool = False, stagger: bool = False):
    """Group 0 on the current stream, group i > 0 on side[i - 1]; forked from
    and joined back into the current stream, so it can be graph-captured.
    With stagger, group i starts once group i - 1's draft is done, so each
    draft runs beside the previous group's verify forward (the pages' draft ||
    verify pairing); otherwise the groups run freely side by side."""
    main = torch.cuda.current_stream()
    streams = [main] + list(side)
    for s in streams[1:]:
        s.wait_stream(main)
    prev_draft = None
    for g, s in zip(groups, streams):
        with torch.cuda.stream(s):
            if stagger and prev_draft is not None:
                s.wait_event(prev_draft)
            if reset:
                g.kv.len.copy_(g.len0)
            api.dflash_draft_block(model, g.kv, g.t0, g.draft, g.ws, stream=s)
            prev_draft = torch.cuda.Event()
            prev_draft.record(s)
            api.dflash_w8a16_linear(standin.desc, g.blk.view(-1, cfg.k * cfg.H), ws=g.tws, stream=s,
                                    y=g.logits.view(-1, cfg.V))
            api.dflash_verify_accept(g.logits, g.draft, g.n, g.corr, g.emitted, g.nxt, g.vws, stream=s)
            api.dflash_kv_commit(model, g.kv, g.blk, g.n, g.ws, stream=s)
    for s in streams[1:]:
        main.wait_stream(s)
