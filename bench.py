#!/usr/bin/env python
"""Benchmark of the DFlash hot path on one GB300 (or N independent replicas).

One step = one pass of the whole hot path over one block: the draft step
(block embedding .. lm-head argmax), the greedy verify-accept against the
target's logits, and the draft-KV commit of the accepted rows.  Inputs are
seeded synthetic tensors with the drafter workload's shapes (no trained
weights, prompts or datasets exist here); they stand in for the pages'
Qwen3-class drafters and prompt suites.  The committed context length is
reset before every step so every step sees the same context.

Prints ONE JSON line (rank 0).  `--impl reference` times the CPU oracle as it
stands on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from block_diffusion_speculative_draft_gb300 import configs, synth  # noqa: E402

METRIC = "draft-step µs & weight GB/s vs ~8 TB/s HBM; verify-accept blocks/s (1×GB300)"
DEFAULT_CFG = configs.QWEN3_4B
FALLBACK_HBM_GBS = 6800.0

# dram__bytes_read.sum + dram__bytes_write.sum per launch from one ncu capture
# of the named kernel on the named workload, keyed by a hash of the kernel's
# source file; ignored (reported null) once that source has changed.
NCU_TRAFFIC = {
    "lmhead_kernel": {"workload": "qwen3-4b-shaped-5L-h2560-b16-ctx512", "bytes": 781344512,
                      "src": "c2a3fcc391c2da2a"},
}


def src_hash(name: str) -> str:
    p = os.path.join(ROOT, "block_diffusion_speculative_draft_gb300", "csrc", name)
    with open(p, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def launches_per_step(cfg, folded: bool = False) -> int:
    # draft: embed+norm, per layer qkv/attn/o/gu/down (the RMSNorms between
    # them, and the final one, are applied inside the GEMM epilogues), lm-head
    draft = 5 * cfg.L + 2
    verify = 1
    if folded:  # commit folded into the draft: its fc GEMM and the length update
        return draft + verify + 2
    commit = 2 + (cfg.L + 7) // 8  # fc, K/V of up to 8 layers per launch, length update
    return draft + verify + commit


# ----------------------------------------------------------- oracle leg ----
def oracle_step_time(cfg, W, hid_ctx, t0, blk_hid, logits_fn, n_steps=1):
    """Times the oracle's own step (draft + verify-accept + commit of the
    accepted rows) for one sequence; dequantisation happens inside, as the
    oracle stands."""
    from oracle import dflash_oracle as O
    D = O.Drafter(cfg, W)
    Ks, Vs = O.context_kv(D, hid_ctx)
    C = hid_ctx.shape[0]
    D.drop()
    times = []
    for _ in range(n_steps):
        t = time.perf_counter()
        ref = O.draft_block(D, t0, Ks, Vs, want_logits=False)
        lg = logits_fn(ref["draft"])
        n, corr, emitted, nxt = O.verify_accept(lg, ref["draft"])
        keep = O.commit_rows(n, cfg.B)
        c = O.context_rows(D, blk_hid[:keep])
        for l in range(cfg.L):
            O.context_kv_layer(D, l, c, C + np.arange(keep))
        times.append(time.perf_counter() - t)
        D.drop()
    return times


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The slowest rank's value (every rank returns it); world 1 is a no-op."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, units_per_rank: int, steps: int, total_ms: float) -> float:
    """Units all ranks processed per second over the slowest rank's time."""
    return world * units_per_rank * steps / (total_ms / 1e3)


def cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def pick_config(args):
    """The named workload (--config), else the default Qwen3-4B shape."""
    return configs.BY_NAME[args.config] if getattr(args, "config", None) else DEFAULT_CFG


def run_reference(args, rank, world):
    if rank != 0:
        return
    cfg = pick_config(args)
    W = synth.drafter_weights(cfg)
    C = cfg.ctx[0]
    hid = synth.target_hidden(cfg.seed, "ctx0", C, cfg.k * cfg.H)
    blk = synth.target_hidden(cfg.seed, "blk", cfg.B, cfg.k * cfg.H)
    t0 = int(synth.tokens(cfg.seed, "t0", 1, cfg.V)[0])
    nacc = synth.accept_lengths(cfg.seed, "acc", 1, cfg.B - 1, cfg.accept_mean)

    def logits_fn(draft):
        return synth.verify_logits(cfg.seed, "verify", draft[None], cfg.R, cfg.V, nacc)[0]

    steps = max(1, args.steps)
    cap_s = 150.0  # seconds of oracle work for the whole arm
    warm = oracle_step_time(cfg, W, hid, t0, blk, logits_fn, 1)
    nwarm = max(0, min(args.warmup, int(0.3 * cap_s / max(warm[0], 1e-3))) - 1)
    if nwarm:
        oracle_step_time(cfg, W, hid, t0, blk, logits_fn, nwarm)
    run = max(1, min(steps, int(0.7 * cap_s / max(warm[0], 1e-3))))
    ts = oracle_step_time(cfg, W, hid, t0, blk, logits_fn, run)
    per = statistics.median(ts)
    value = cfg.b / per
    out = {"metric": METRIC, "value": value, "unit": "blocks/s", "n_gpus": world, "steps": run,
           "warmup": 1 + nwarm, "ms_per_step": per * 1e3, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": cfg.name, "b": cfg.b, "B": cfg.B, "ctx": C},
           "impl": "reference",
           "cpu_baseline": {"value": value, "unit": "blocks/s", "cores": cores(), "kind": "oracle",
                            "sample": f"{run} oracle step(s) (draft + verify-accept + commit) of one "
                                      f"sequence of {cfg.name}; {steps} requested"},
           "e2e": {"value": value, "unit": "blocks/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


# -------------------------------------------------------------- GPU leg ----
def run_ours(args, rank, world, local_rank):
    import torch
    from block_diffusion_speculative_draft_gb300 import api
    from block_diffusion_speculative_draft_gb300.workload import commit_contexts, contexts

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    cfg = pick_config(args)
    b = cfg.b
    W = synth.drafter_weights(cfg)
    model = api.DeviceDrafter(cfg, W, dev)
    ctx = contexts(cfg)
    kv = api.KVCache(cfg, b, int(ctx.max()) + 2 * cfg.B, dev)
    ws = api.workspace(cfg, b, cfg.B, dev)
    commit_contexts(api, torch, cfg, model, kv, ws, ctx, cfg.B, dev)
    torch.cuda.synchronize()
    len0 = kv.len.clone()

    t0 = torch.from_numpy(synth.tokens(cfg.seed, "t0", b, cfg.V)).to(dev)
    draft = torch.empty((b, cfg.B - 1), dtype=torch.int32, device=dev)
    api.dflash_draft_block(model, kv, t0, draft, ws)
    torch.cuda.synchronize()
    nacc = synth.accept_lengths(cfg.seed, "acc", b, cfg.B - 1, cfg.accept_mean)
    lg_host = synth.verify_logits(cfg.seed, "verify", draft.cpu().numpy(), cfg.R, cfg.V, nacc)
    logits = torch.from_numpy(lg_host).to(dev)
    blk_host = np.stack([synth.target_hidden(cfg.seed, f"blk{j}", cfg.B, cfg.k * cfg.H) for j in range(b)])
    blk = torch.from_numpy(blk_host).to(dev)
    n_out = torch.empty(b, dtype=torch.int32, device=dev)
    corr = torch.empty(b, dtype=torch.int32, device=dev)
    emitted = torch.empty((b, cfg.R), dtype=torch.int32, device=dev)
    nxt = torch.empty(b, dtype=torch.int32, device=dev)
    vws = torch.zeros(api.dflash_verify_workspace_size(b, cfg.R, cfg.V), dtype=torch.uint8, device=dev)

    def step():
        kv.len.copy_(len0)
        api.dflash_draft_block(model, kv, t0, draft, ws)
        api.dflash_verify_accept(logits, draft, n_out, corr, emitted, nxt, vws)
        api.dflash_kv_commit(model, kv, blk, n_out, ws)

    def step_folded():
        # the same work per step with the commit of the previous verify's
        # accepted rows folded into this step's draft pass
        kv.len.copy_(len0)
        api.dflash_commit_draft_block(model, kv, blk, n_out, t0, draft, ws)
        api.dflash_verify_accept(logits, draft, n_out, corr, emitted, nxt, vws)

    def draft_only():
        api.dflash_draft_block(model, kv, t0, draft, ws)

    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(3):
            step_folded()
            step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    assert api.dflash_get_status() == 0, "device status flagged during warm-up"

    def capture(fn, reps=1):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(reps):
                fn()
        return g

    g_step = capture(step)
    g_folded = capture(step_folded)
    g_draft = capture(draft_only)
    g_fused = None
    if cfg.M <= 32:
        try:
            api.dflash_draft_block_fused(model, kv, t0, draft, ws)
            torch.cuda.synchronize()
            g_fused = capture(lambda: api.dflash_draft_block_fused(model, kv, t0, draft, ws))
        except api.DflashError:
            g_fused = None
    VREP = 100
    g_verify = capture(lambda: api.dflash_verify_accept(logits, draft, n_out, corr, emitted, nxt, vws), VREP)
    # temperature speculative-sampling accept on the same rows (T = 0.8,
    # uniforms drawn once on the device)
    u_acc = torch.rand((b, cfg.B - 1), device=dev).clamp_(1e-7, 1 - 1e-7)
    u_smp = torch.rand((b, cfg.V), device=dev).clamp_(1e-7, 1 - 1e-7)
    sws = torch.zeros(api.dflash_verify_sample_workspace_size(b, cfg.R, cfg.V), dtype=torch.uint8, device=dev)
    s_n, s_c = torch.empty_like(n_out), torch.empty_like(corr)
    g_sample = capture(lambda: api.dflash_verify_accept_sample(logits, draft, 0.8, u_acc, u_smp, s_n, s_c,
                                                               ws=sws), VREP)
    M1 = b * (cfg.B - 1)
    lm_idx = torch.empty(M1, dtype=torch.int32, device=dev)
    lmws = torch.zeros(4096, dtype=torch.uint8, device=dev)
    hbuf = torch.zeros((M1, cfg.H), dtype=torch.bfloat16, device=dev)
    g_lm = capture(lambda: api.dflash_lmhead_argmax(hbuf.view(torch.int16), model.lm_t, lm_idx, ws=lmws))

    def timed(g, K, W_):
        for _ in range(W_):
            g.replay()
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
        evs[0].record()
        for i in range(K):
            g.replay()
            evs[i + 1].record()
        torch.cuda.synchronize()
        per = [evs[i].elapsed_time(evs[i + 1]) for i in range(K)]
        total = max_over_ranks(evs[0].elapsed_time(evs[K]), world, dev)
        return total, per

    K, Wm = args.steps, max(3, args.warmup)
    with ClockSampler(local_rank) as clk:
        total_ms, per_ms = timed(g_step, K, Wm)
    clocks = clk.summary()
    fold_total, _ = timed(g_folded, K, Wm)
    _, draft_ms = timed(g_draft, K, Wm)
    fused_ms = timed(g_fused, K, Wm)[1] if g_fused is not None else None
    _, ver_ms = timed(g_verify, max(3, K // 5), 2)
    _, smp_ms = timed(g_sample, max(3, K // 5), 2)
    _, lm_ms = timed(g_lm, K, Wm)
    assert api.dflash_get_status() == 0, "device status flagged during the timed region"

    # end to end through the public API with host buffers: H2D of the step's
    # inputs (last token, target logits, target hidden rows), D2H of results
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    h_t0, h_lg, h_blk = pin(t0.cpu().numpy()), pin(lg_host), pin(blk_host)
    o_draft = torch.empty_like(draft, device="cpu").pin_memory()
    o_n = torch.empty_like(n_out, device="cpu").pin_memory()
    o_em = torch.empty_like(emitted, device="cpu").pin_memory()
    o_nx = torch.empty_like(nxt, device="cpu").pin_memory()
    h2d = h_t0.numel() * 4 + h_lg.numel() * 4 + h_blk.numel() * 2
    d2h = (o_draft.numel() + o_n.numel() + o_em.numel() + o_nx.numel()) * 4

    def e2e_step():
        t0.copy_(h_t0, non_blocking=True)
        logits.copy_(h_lg, non_blocking=True)
        blk.copy_(h_blk, non_blocking=True)
        g_step.replay()
        o_draft.copy_(draft, non_blocking=True)
        o_n.copy_(n_out, non_blocking=True)
        o_em.copy_(emitted, non_blocking=True)
        o_nx.copy_(nxt, non_blocking=True)

    for _ in range(Wm):
        e2e_step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(K):
        e2e_step()
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)

    # the same draft step with int4 projections (W4A16, group scales in the
    # packed tiles); the cache and inputs are the ones above
    W4 = synth.drafter_weights(cfg, bits=4)
    m4 = api.DeviceDrafter(cfg, W4, dev, bits=4)
    del W4
    draft4 = torch.empty_like(draft)
    api.dflash_draft_block(m4, kv, t0, draft4, ws)
    torch.cuda.synchronize()
    g_draft4 = capture(lambda: api.dflash_draft_block(m4, kv, t0, draft4, ws))
    _, draft4_ms = timed(g_draft4, K, Wm)
    assert api.dflash_get_status() == 0, "device status flagged during the int4 draft timing"
    del g_draft4, m4

    # draft || verify overlap: two groups (sequence sets) of this workload on
    # two streams, each step = draft, the int4 QMM stand-in for the target's
    # verify forward, verify-accept, commit; serial vs side by side
    overlap = None
    if b == 1 and not args.no_overlap:
        from block_diffusion_speculative_draft_gb300 import workload as WL
        standin = WL.TargetStandIn(api, torch, cfg, dev)
        groups = []
        for i in range(2):
            hids = [synth.target_hidden(cfg.seed, f"ovl-g{i}-ctx{j}", int(ctx[j]), cfg.k * cfg.H)
                    for j in range(b)]
            groups.append(WL.Group(api, torch, cfg, model, dev, ctx, hids,
                                   synth.tokens(cfg.seed, f"ovl-g{i}-t0", b, cfg.V), f"ovl-g{i}-"))
        side = [torch.cuda.Stream(device=dev)]
        WL.run_serial(api, torch, cfg, model, standin, groups, reset=True)
        WL.run_overlapped(api, torch, cfg, model, standin, groups, side, reset=True, stagger=True)
        torch.cuda.synchronize()
        g_ser = capture(lambda: WL.run_serial(api, torch, cfg, model, standin, groups, reset=True))
        g_free = capture(lambda: WL.run_overlapped(api, torch, cfg, model, standin, groups, side, reset=True))
        g_stag = capture(lambda: WL.run_overlapped(api, torch, cfg, model, standin, groups, side, reset=True,
                                                   stagger=True))
        g_qmm = capture(lambda: api.dflash_w8a16_linear(standin.desc, groups[0].blk.view(-1, cfg.k * cfg.H),
                                                        ws=standin.ws, y=groups[0].logits.view(-1, cfg.V)))
        ser_ms, _ = timed(g_ser, K, Wm)
        free_ms, _ = timed(g_free, K, Wm)
        stag_ms, _ = timed(g_stag, K, Wm)
        _, qmm_ms = timed(g_qmm, K, Wm)
        assert api.dflash_get_status() == 0, "device status flagged during the overlap timing"
        nb = 2 * b
        best = min(free_ms, stag_ms)
        overlap = {
            "workload": f"2 groups x {cfg.name}; target stand-in: int4 QMM [{cfg.V}][{cfg.k * cfg.H}] "
                        f"({standin.bytes() / 1e6:.0f} MB) from the block's target hidden rows to its logits",
            "serial_ms_per_step": ser_ms / K, "free_ms_per_step": free_ms / K, "staggered_ms_per_step": stag_ms / K,
            "blocks_per_s_serial": whole_job_rate(world, nb, K, ser_ms),
            "blocks_per_s_free": whole_job_rate(world, nb, K, free_ms),
            "blocks_per_s_staggered": whole_job_rate(world, nb, K, stag_ms),
            "standin_qmm_us": statistics.median(qmm_ms) * 1e3,
            "draft_time_hidden_frac": (ser_ms - best) / K / (nb * statistics.median(draft_ms)),
        }
        del g_ser, g_free, g_stag, g_qmm, groups, standin

    hbm, peak_kind = peaks()
    ms_step = total_ms / K
    value = whole_job_rate(world, b, K, total_ms)
    dms = statistics.median(draft_ms)
    step_bytes = cfg.step_bytes(list(ctx))
    lm_bytes = cfg.V * cfg.H * 2 + M1 * cfg.H * 2 + M1 * 4
    lm_avg_ms = statistics.mean(lm_ms)
    lm_gbs = lm_bytes / (lm_avg_ms * 1e-3) / 1e9
    tr = NCU_TRAFFIC.get("lmhead_kernel")
    traffic = tr["bytes"] if tr and tr["src"] == src_hash("k_lmhead.cu") and tr["workload"] == cfg.name else None
    out = {
        "metric": METRIC, "value": value, "unit": "blocks/s", "n_gpus": world, "steps": K, "warmup": Wm,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int8xf16->f32 (W8A16), bf16 lm-head, fp16 KV", "data": "synthetic",
        "config": {"workload": cfg.name, "b": b, "B": cfg.B, "ctx": [int(c) for c in ctx], "L": cfg.L,
                   "H": cfg.H, "V": cfg.V, "l2": "inputs larger than L2: weights+lm-head "
                   f"{step_bytes / 1e9:.2f} GB streamed per step", "parallelism": f"replicas x{world}"},
        "step": "draft + verify-accept + commit of the accepted rows (separate calls)",
        "step_commit_folded": {"blocks_per_s": whole_job_rate(world, b, K, fold_total),
                               "ms_per_step": fold_total / K,
                               "gpu_launches_per_step": launches_per_step(cfg, folded=True)},
        "draft_step_us": {"median": dms * 1e3, "p10": float(np.percentile(draft_ms, 10)) * 1e3,
                          "p90": float(np.percentile(draft_ms, 90)) * 1e3},
        "draft_step_weight_GBps": step_bytes / (dms * 1e-3) / 1e9,
        "draft_step_w4a16": {"median_us": statistics.median(draft4_ms) * 1e3,
                             "bytes": cfg.step_bytes_w4(list(ctx)),
                             "frac_of_measured": cfg.step_bytes_w4(list(ctx))
                             / (statistics.median(draft4_ms) * 1e-3) / 1e9 / hbm},
        "draft_verify_overlap": overlap,
        "draft_step_fused_kernel_us": None if fused_ms is None else statistics.median(fused_ms) * 1e3,
        "step_roofline": {"bytes": step_bytes, "frac_of_measured": step_bytes / (dms * 1e-3) / 1e9 / hbm,
                          "frac_of_8TBps": step_bytes / (dms * 1e-3) / 1e9 / 8000.0},
        "verify_accept_blocks_per_s": b / (statistics.median(ver_ms) / VREP / 1e3),
        "verify_sample_blocks_per_s": b / (statistics.median(smp_ms) / VREP / 1e3),
        "roofline": {"kernel": "lmhead_kernel (bf16 GEMV + fused argmax)", "bound": "hbm", "achieved": lm_gbs,
                     "peak": hbm, "unit": "GB/s", "frac": lm_gbs / hbm, "traffic": traffic,
                     "peak_kind": peak_kind, "algorithmic_bytes_per_launch": lm_bytes},
        "clocks": clocks,
        "gpu_launches": K * launches_per_step(cfg),
        "e2e": {"value": whole_job_rate(world, b, K, e2e_ms), "unit": "blocks/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        C = int(ctx[0])
        hid = synth.target_hidden(cfg.seed, "ctx0", C, cfg.k * cfg.H)

        def logits_fn(dr):
            return synth.verify_logits(cfg.seed, "verify", dr[None], cfg.R, cfg.V, nacc[:1])[0]

        ts = oracle_step_time(cfg, W, hid, int(t0[0]), blk_host[0], logits_fn, 1)
        out["cpu_baseline"] = {"value": 1.0 / ts[0], "unit": "blocks/s", "cores": cores(), "kind": "oracle",
                               "sample": f"1 oracle step (draft + verify-accept + commit) of sequence 0 of "
                                         f"{cfg.name}, {ts[0]:.1f} s"}
    if rank == 0:
        print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-overlap", action="store_true", help="skip the two-stream draft || verify measurement")
    ap.add_argument("--config", default=None, choices=sorted(configs.BY_NAME),
                    help="another workload of the parity suite (default: the Qwen3-4B-shaped one)")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local_rank)
        dist.init_process_group(backend)
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
