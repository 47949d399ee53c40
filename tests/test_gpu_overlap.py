"""Draft || verify overlap on two streams, with the int4 QMM stand-in for the
target's verify forward.

Overlap must not change a single result: from identical states, running the
groups side by side (free, or staggered so each draft runs beside the
previous group's verify forward), eagerly or replayed from a CUDA graph,
gives bit-identical drafts, accept outputs, logits, lengths and committed
cache rows to running them one after another.  Every mode runs several
times (a race shows up only in some runs), and every mode's committed K/V
rows are also checked against the oracle's context path, so a mismatch
says which mode is wrong.  The stand-in's logits match the oracle's int4
linear within 1e-3 of max-abs (all rows for the tiny workload, sampled row
ranges at full size), and the accept outputs equal the oracle's greedy rule
on those logits.
"""
import numpy as np
import pytest

from oracle import dflash_oracle as O
from block_diffusion_speculative_draft_gb300 import synth
from block_diffusion_speculative_draft_gb300.configs import TINY, QWEN3_4B
from block_diffusion_speculative_draft_gb300 import workload as WL
from tests.gpu_util import gpu_available, rel_err

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not gpu_available(), reason="needs a GPU")]

if gpu_available():
    import torch
    from block_diffusion_speculative_draft_gb300 import api
    DEV = torch.device("cuda:0")


def _groups(cfg, model, ngroups=2):
    ctx = WL.contexts(cfg)
    gs = []
    for i in range(ngroups):
        hids = [synth.target_hidden(cfg.seed, f"ovl-g{i}-ctx{j}", int(ctx[j]), cfg.k * cfg.H) for j in range(cfg.b)]
        t0 = synth.tokens(cfg.seed, f"ovl-g{i}-t0", cfg.b, cfg.V)
        gs.append(WL.Group(api, torch, cfg, model, DEV, ctx, hids, t0, f"ovl-g{i}-"))
    return gs


def _snapshot(cfg, gs):
    out = []
    for g in gs:
        lens = g.kv.len.cpu().numpy()
        rows = [(g.kv.k[:, j, :, :int(lens[j])].cpu().numpy(), g.kv.v[:, j, :, :int(lens[j])].cpu().numpy())
                for j in range(cfg.b)]
        out.append(dict(draft=g.draft.cpu().numpy(), logits=g.logits.cpu().numpy(), n=g.n.cpu().numpy(),
                        corr=g.corr.cpu().numpy(), emitted=g.emitted.cpu().numpy(), nxt=g.nxt.cpu().numpy(),
                        len=lens, rows=rows))
    return out


def _same(a, b):
    for gi, (ga, gb) in enumerate(zip(a, b)):
        for k in ("draft", "logits", "n", "corr", "emitted", "nxt", "len"):
            assert np.array_equal(ga[k], gb[k]), (gi, k)
        for (ka, va), (kb, vb) in zip(ga["rows"], gb["rows"]):
            assert np.array_equal(ka.view(np.uint16), kb.view(np.uint16)), (gi, "K rows")
            assert np.array_equal(va.view(np.uint16), vb.view(np.uint16)), (gi, "V rows")


REPS = 4  # runs of every mode


def _oracle_rows(cfg, W, gs, snap):
    """The oracle's K/V [L][rows][nkv][d] of each group's and sequence's
    committed rows (the accept lengths of `snap`) at their positions."""
    D = O.Drafter(cfg, W)
    out = []
    for g, sg in zip(gs, snap):
        l0 = g.len0.cpu().numpy()
        per = []
        for j in range(cfg.b):
            keep = O.commit_rows(int(sg["n"][j]), cfg.B)
            c = O.context_rows(D, g.blk_host[j][:keep])
            kv = [O.context_kv_layer(D, l, c, int(l0[j]) + np.arange(keep)) for l in range(cfg.L)]
            per.append((int(l0[j]), keep, np.stack([k for k, _ in kv]), np.stack([v for _, v in kv])))
        out.append(per)
    D.drop()
    return out


def _committed_err(snap, expect):
    """Max relative error of the committed rows [len0, len) of every group
    and sequence against the oracle's."""
    errs = []
    for sg, per in zip(snap, expect):
        for j, (l0, keep, k, v) in enumerate(per):
            assert int(sg["len"][j]) == l0 + keep
            gk, gv = sg["rows"][j]
            errs.append(rel_err(gk[:, :, l0:, :].transpose(0, 2, 1, 3), k))
            errs.append(rel_err(gv[:, :, l0:, :].transpose(0, 2, 1, 3), v))
    return max(errs)


def _run_all_ways(cfg, W, model, standin, gs):
    side = [torch.cuda.Stream(device=DEV) for _ in gs[1:]]
    WL.run_serial(api, torch, cfg, model, standin, gs, reset=True)
    torch.cuda.synchronize()
    ref = _snapshot(cfg, gs)
    expect = _oracle_rows(cfg, W, gs, ref)
    assert _committed_err(ref, expect) <= 1e-2
    modes = {
        "serial": lambda: WL.run_serial(api, torch, cfg, model, standin, gs, reset=True),
        "free": lambda: WL.run_overlapped(api, torch, cfg, model, standin, gs, side, reset=True),
        "staggered": lambda: WL.run_overlapped(api, torch, cfg, model, standin, gs, side, reset=True,
                                               stagger=True),
    }
    for name in list(modes):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            modes[name]()
        modes["graph " + name] = g.replay
    for name, fn in modes.items():
        for r in range(REPS):
            fn()
            torch.cuda.synchronize()
            snap = _snapshot(cfg, gs)
            assert _committed_err(snap, expect) <= 1e-2, (name, r)
            _same(ref, snap)
    assert api.dflash_get_status() == 0
    return ref


def _check_standin_and_accept(cfg, gs, snap, row_ranges):
    K = cfg.k * cfg.H
    chunks = WL.standin_chunks(cfg)
    for g, s in zip(gs, snap):
        for j in range(cfg.b):
            h = g.blk_host[j].astype(np.float64)
            for c, lo, hi in row_ranges:
                q, sc = WL.standin_grid(cfg, c)
                ref = O.linear(h, O.dequant_w4(q[lo:hi], sc[lo:hi]))
                r0 = chunks[c][0]
                assert rel_err(s["logits"][j][:, r0 + lo:r0 + hi], ref) <= 1e-3
            n, corr, em, nxt = O.verify_accept(s["logits"][j], s["draft"][j])
            assert s["n"][j] == n and s["corr"][j] == corr and s["nxt"][j] == nxt
            assert np.array_equal(s["emitted"][j][:n + 1], np.asarray(em)[:n + 1])


def test_overlap_tiny():
    cfg = TINY
    W = synth.drafter_weights(cfg)
    model = api.DeviceDrafter(cfg, synth.FloatWeights(W), DEV)
    standin = WL.TargetStandIn(api, torch, cfg, DEV)
    gs = _groups(cfg, model, 3)
    snap = _run_all_ways(cfg, W, model, standin, gs)
    _check_standin_and_accept(cfg, gs, snap, [(0, 0, cfg.V)])
    for g, s in zip(gs, snap):
        assert np.array_equal(s["len"], g.len0.cpu().numpy() + s["n"] + 1)


def test_overlap_qwen3_4b_shape():
    cfg = QWEN3_4B
    W = synth.drafter_weights(cfg)
    model = api.DeviceDrafter(cfg, synth.FloatWeights(W), DEV)
    standin = WL.TargetStandIn(api, torch, cfg, DEV)
    gs = _groups(cfg, model, 2)
    snap = _run_all_ways(cfg, W, model, standin, gs)
    last = len(WL.standin_chunks(cfg)) - 1
    _check_standin_and_accept(cfg, gs, snap, [(0, 0, 256), (7, 4000, 4256), (last, 4224, 4480)])
