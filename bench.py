#!/usr/bin/env python
"""Benchmark of the DFlash hot path on one GB300 (or N independent replicas).

One step = one pass of the whole hot path over one block: the draft step
(block embedding .. lm-head argmax), the greedy verify-accept against the
target's logits, and the draft-KV commit of the accepted rows.  Inputs are
seeded synthetic tensors with the drafter workload's shapes (no trained
weights, prompts or datasets exist here); they stand in for the pages'
Qwen3-class drafters and prompt suites.  The committed context length is
reset before every step so every step sees the same context.

The default workload is the 27B-class drafter of the mirror-sd README's
"Results" table (5 layers, hidden 5120, block 32) with 4096 committed
context rows; the draft step is also timed at 64 and 2048 rows, the table's
other contexts.  The headline runs in the library's early-launch mode (one
stream on a dedicated GPU); the stream-order mode is timed beside it.

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
DEFAULT_CFG = configs.DENSE_27B.with_ctx((4096,))
CTX_SWEEP = configs.DENSE_27B_CTX_SWEEP
FALLBACK_HBM_GBS = 6800.0

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) over
# algorithmic bytes, from full ncu captures of the named kernel on the
# Qwen3-4B-shaped workload (the capture size rule keeps the 27B-class launches
# out of a full capture; both kernels read every weight byte once whatever
# the shape, so traffic scales with the algorithmic bytes).  Keyed by a hash
# of the kernel's source file: reported null once that source has changed.
NCU_TRAFFIC = {
    # DRAM read + write over algorithmic bytes of four captured launches of
    # each kernel on the 27B-class step (32 rows)
    "w8_gemm_kernel": {"ratio": 534.574 / 533.504, "src": "db60a83621a45e58",
                       "capture": "profiles/w8_gemm_kernel_27b-class.md"},
    "wmma_gemm_kernel": {"ratio": 211.481 / 216.351, "src": "db60a83621a45e58",
                         "capture": "profiles/wmma_gemm_kernel_27b-class.md"},
    "lmhead_kernel": {"ratio": 781.06 / 777.99, "src": "01ee840985b7ff35",
                      "capture": "profiles/lmhead_kernel_qwen3-4b.md"},
    # two launches, 8 x Qwen3-8B-shaped batch (120 rows)
    "lmhead_tc_kernel": {"ratio": 2497.985 / 2491.286, "src": "01ee840985b7ff35",
                         "capture": "profiles/lmhead_tc_kernel_b8-qwen3-8b.md"},
}


def traffic_for(kernel: str, source: str, algorithmic_bytes: float):
    """Per-launch DRAM traffic estimate (None once the kernel has changed)."""
    t = NCU_TRAFFIC.get(kernel)
    if not t or t["src"] != src_hash(source):
        return None
    return t["ratio"] * algorithmic_bytes


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
    """The named workload (--config), else the default 27B-class drafter at
    4096 context rows."""
    return configs.BY_NAME[args.config] if getattr(args, "config", None) else DEFAULT_CFG


def config_dict(cfg, ctx, world: int) -> dict:
    """The `config` object both arms print for a workload."""
    step_bytes = cfg.step_bytes(list(ctx))
    return {"workload": cfg.name, "b": cfg.b, "B": cfg.B, "ctx": [int(c) for c in ctx], "L": cfg.L,
            "H": cfg.H, "V": cfg.V,
            "l2": f"inputs larger than L2: {step_bytes / 1e9:.2f} GB of weights, lm-head and KV streamed per step",
            "parallelism": f"replicas x{world}"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    from block_diffusion_speculative_draft_gb300.workload import contexts
    cfg = pick_config(args)
    W = synth.drafter_weights(cfg)
    ctx = contexts(cfg)
    C = int(ctx[0])
    hid = synth.target_hidden(cfg.seed, "ctx0", C, cfg.k * cfg.H)
    blk = synth.target_hidden(cfg.seed, "blk0", cfg.B, cfg.k * cfg.H)
    t0 = int(synth.tokens(cfg.seed, "t0", cfg.b, cfg.V)[0])
    nacc = synth.accept_lengths(cfg.seed, "acc", cfg.b, cfg.B - 1, cfg.accept_mean)

    def logits_fn(draft):
        return synth.verify_logits(cfg.seed, "verify", draft[None], cfg.R, cfg.V, nacc[:1])[0]

    steps = max(1, args.steps)
    cap_s = 150.0  # seconds of oracle work for the whole arm
    warm = oracle_step_time(cfg, W, hid, t0, blk, logits_fn, 1)
    nwarm = max(0, min(args.warmup, int(0.3 * cap_s / max(warm[0], 1e-3))) - 1)
    if nwarm:
        oracle_step_time(cfg, W, hid, t0, blk, logits_fn, nwarm)
    run = max(1, min(steps, int(0.7 * cap_s / max(warm[0], 1e-3))))
    ts = oracle_step_time(cfg, W, hid, t0, blk, logits_fn, run)
    per = statistics.median(ts)
    value = 1.0 / per  # one sequence per oracle step
    out = {"metric": METRIC, "value": value, "unit": "blocks/s", "n_gpus": world, "steps": run,
           "warmup": 1 + nwarm, "ms_per_step": per * 1e3, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config_dict(cfg, ctx, world),
           "impl": "reference",
           "cpu_baseline": {"value": value, "unit": "blocks/s", "cores": cores(), "kind": "oracle",
                            "sample": f"{run} oracle step(s) (draft + verify-accept + commit) of sequence 0 of "
                                      f"{cfg.name}; {steps} requested"},
           "e2e": {"value": value, "unit": "blocks/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


# -------------------------------------------------------------- GPU leg ----
def timed_graph(torch, g, K, W_, world, dev):
    """K replays of a CUDA graph after W_ warm-up replays: (total ms over the
    slowest rank, per-replay ms).  Events on the current stream, a barrier and
    a synchronize on both sides."""
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
    return max_over_ranks(evs[0].elapsed_time(evs[K]), world, dev), per


def capture(torch, fn, reps=1):
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()  # one eager run: kernel attributes and caches are set before capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        for _ in range(reps):
            fn()
    return g


def med_us(ms_list) -> float:
    return statistics.median(ms_list) * 1e3


def run_ours(args, rank, world, local_rank):
    import torch
    from block_diffusion_speculative_draft_gb300 import api
    from block_diffusion_speculative_draft_gb300.workload import commit_contexts, contexts

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    cfg = pick_config(args)
    b, B = cfg.b, cfg.B
    K, Wm = args.steps, max(3, args.warmup)
    hbm, peak_kind = peaks()
    W = synth.drafter_weights(cfg)
    model = api.DeviceDrafter(cfg, synth.FloatWeights(W), dev)
    ctx = contexts(cfg)
    # context sweep: (label, committed length per sequence); the default
    # workload also times the pages' other contexts, any other workload its own
    if b == 1 and args.config is None:
        sweep = [(str(C), [C]) for C in sorted(set(int(c) for c in CTX_SWEEP) | {int(ctx[0])})]
    else:
        sweep = [("ctx", [int(c) for c in ctx])]
    cmax = max(max(lens) for _, lens in sweep)
    # one cache holding the largest context: context row j depends only on
    # target row j and position j, so a shorter context is the same cache
    # with a smaller committed length
    kv = api.KVCache(cfg, b, cmax + 2 * B, dev)
    ws = api.workspace(cfg, b, B, dev)
    full_ctx = np.maximum(ctx, cmax) if len(sweep) > 1 else ctx
    head_label = str(int(ctx[0])) if len(sweep) > 1 else "ctx"
    commit_contexts(api, torch, cfg, model, kv, ws, full_ctx, B, dev)
    torch.cuda.synchronize()
    len0 = torch.from_numpy(np.asarray(ctx, np.int32)).to(dev)
    kv.len.copy_(len0)

    t0 = torch.from_numpy(synth.tokens(cfg.seed, "t0", b, cfg.V)).to(dev)
    # the step's outputs (drafts, accept count, correction token, next token,
    # emitted tokens) are views of one device buffer, each 16-byte aligned, so
    # the end-to-end loop brings them back with a single copy
    al4 = lambda n: (n + 3) // 4 * 4
    o_sz = [b * (B - 1), b, b, b, b * cfg.R]
    o_off = np.cumsum([0] + [al4(n) for n in o_sz])
    outbuf = torch.zeros(int(o_off[-1]), dtype=torch.int32, device=dev)
    draft, n_out, corr, nxt, emitted = (outbuf[int(o_off[i]):int(o_off[i]) + o_sz[i]] for i in range(5))
    draft, emitted = draft.view(b, B - 1), emitted.view(b, cfg.R)
    api.dflash_draft_block(model, kv, t0, draft, ws)
    torch.cuda.synchronize()
    nacc = synth.accept_lengths(cfg.seed, "acc", b, B - 1, cfg.accept_mean)
    lg_host = synth.verify_logits(cfg.seed, "verify", draft.cpu().numpy(), cfg.R, cfg.V, nacc)
    logits = torch.from_numpy(lg_host).to(dev)
    blk_host = np.stack([synth.target_hidden(cfg.seed, f"blk{j}", B, cfg.k * cfg.H) for j in range(b)])
    blk = torch.from_numpy(blk_host).to(dev)
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

    results = {}
    for mode, mname in ((api.LAUNCH_EARLY, "early"), (api.LAUNCH_STREAM_ORDER, "stream_order")):
        with api.launch_mode(mode):
            g_step = capture(torch, step)
            if mode == api.LAUNCH_EARLY:
                with ClockSampler(local_rank) as clk:
                    total_ms, _ = timed_graph(torch, g_step, K, Wm, world, dev)
                clocks = clk.summary()
            else:
                total_ms, _ = timed_graph(torch, g_step, K, Wm, world, dev)
            res = {"step_total_ms": total_ms, "draft_us": {}}
            for label, lens in sweep:
                cl = torch.tensor(lens, dtype=torch.int32, device=dev)

                def draft_only():
                    kv.len.copy_(cl)
                    api.dflash_draft_block(model, kv, t0, draft, ws)

                _, per = timed_graph(torch, capture(torch, draft_only), K, Wm, world, dev)
                res["draft_us"][label] = per
            kv.len.copy_(len0)
            results[mname] = res
            del g_step
    assert api.dflash_get_status() == 0, "device status flagged during the timed region"
    early = results["early"]
    dms = statistics.median(early["draft_us"][head_label])

    with api.launch_mode(api.LAUNCH_EARLY):
        fold_total, _ = timed_graph(torch, capture(torch, step_folded), K, Wm, world, dev)
        VREP = 100
        _, ver_ms = timed_graph(torch, capture(torch, lambda: api.dflash_verify_accept(
            logits, draft, n_out, corr, emitted, nxt, vws), VREP), max(3, K // 20), 2, world, dev)
        # temperature speculative-sampling accept on the same rows (T = 0.8,
        # uniforms drawn once on the device)
        u_acc = torch.rand((b, B - 1), device=dev).clamp_(1e-7, 1 - 1e-7)
        u_smp = torch.rand((b, cfg.V), device=dev).clamp_(1e-7, 1 - 1e-7)
        sws = torch.zeros(api.dflash_verify_sample_workspace_size(b, cfg.R, cfg.V), dtype=torch.uint8, device=dev)
        s_n, s_c = torch.empty_like(n_out), torch.empty_like(corr)
        _, smp_ms = timed_graph(torch, capture(torch, lambda: api.dflash_verify_accept_sample(
            logits, draft, 0.8, u_acc, u_smp, s_n, s_c, ws=sws), VREP), max(3, K // 20), 2, world, dev)
        # the lm-head alone (same table, bf16 rows)
        M1 = b * (B - 1)
        lm_idx = torch.empty(M1, dtype=torch.int32, device=dev)
        lmws = torch.zeros(4096, dtype=torch.uint8, device=dev)
        hbuf = torch.zeros((M1, cfg.H), dtype=torch.bfloat16, device=dev)
        _, lm_ms = timed_graph(torch, capture(torch, lambda: api.dflash_lmhead_argmax(
            hbuf.view(torch.int16), model.lm_t, lm_idx, ws=lmws)), K, Wm, world, dev)
        # the projection kernel alone, over the step's 4 L layer matrices in
        # the step's order (plain fp32 store epilogue, same weight stream)
        xs = torch.zeros((cfg.M, max(cfg.H, cfg.F, cfg.nq * cfg.d)), dtype=torch.float16, device=dev)
        ys = torch.empty((cfg.M, max(cfg.nqkv, cfg.H, 2 * cfg.F)), dtype=torch.float32, device=dev)
        mats = []  # (name, descriptor) in step order
        for l in range(cfg.L):
            for name in ("qkv", "o", "gu", "down"):
                mats.append((name, getattr(model, name)[l]))

        # the library runs a projection on its tensor-memory kernel above 32
        # rows, and from 17 rows when the weight matrix has >= 40 MiB; each
        # kernel's launches are timed as their own group, in step order
        def on_tcgen05(m):
            return cfg.M > 32 or (cfg.M > 16 and m.N * m.K >= 40 << 20)

        def projections(ms):
            def run():
                for m in ms:
                    api.dflash_w8a16_linear(m, xs.view(-1)[:cfg.M * m.K].view(cfg.M, m.K),
                                            y=ys.view(-1)[:cfg.M * m.N].view(cfg.M, m.N))
            return run

        proj = {}
        for kname, sel in (("w8_gemm_kernel", [nm for nm in mats if on_tcgen05(nm[1])]),
                           ("wmma_gemm_kernel", [nm for nm in mats if not on_tcgen05(nm[1])])):
            if not sel:
                continue
            ms = [m for _, m in sel]
            pb = sum(m.N * m.K + 2 * m.N + 2 * cfg.M * m.K + 4 * cfg.M * m.N for m in ms)
            _, pms = timed_graph(torch, capture(torch, projections(ms)), K, Wm, world, dev)
            proj[kname] = {"bytes": pb, "ms": pms, "n": len(ms),
                           "what": "/".join(dict.fromkeys(n for n, _ in sel))}

        # end to end through the public API with host buffers, every step:
        # H2D of the step's inputs (last token, target logits, target hidden
        # rows) from pinned memory, the three C-ABI calls issued eagerly, D2H
        # of the drafts and accept outputs
        pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
        h_t0, h_lg, h_blk = pin(t0.cpu().numpy()), pin(lg_host), pin(blk_host)
        o_all = torch.empty_like(outbuf, device="cpu").pin_memory()
        o_n = o_all[int(o_off[1]):int(o_off[1]) + b]
        h2d = h_t0.numel() * 4 + h_lg.numel() * 4 + h_blk.numel() * 2
        d2h = o_all.numel() * 4

        def copies_in():
            t0.copy_(h_t0, non_blocking=True)
            logits.copy_(h_lg, non_blocking=True)
            blk.copy_(h_blk, non_blocking=True)

        def copies_out():
            o_all.copy_(outbuf, non_blocking=True)  # drafts, accept outputs, emitted tokens

        def e2e_eager():
            copies_in()
            step()
            copies_out()

        # the same, with the target logits and hidden rows (needed only by
        # verify and commit) copied on a side stream while the draft pass
        # runs; the side stream waits for the previous step's commit, which
        # last read those buffers
        side = torch.cuda.Stream(device=dev)
        ev_in, ev_done = torch.cuda.Event(), torch.cuda.Event()
        ev_done.record()

        def e2e_overlapped():
            cur = torch.cuda.current_stream()
            with torch.cuda.stream(side):
                side.wait_event(ev_done)
                logits.copy_(h_lg, non_blocking=True)
                blk.copy_(h_blk, non_blocking=True)
                ev_in.record(side)
            t0.copy_(h_t0, non_blocking=True)
            kv.len.copy_(len0)
            api.dflash_draft_block(model, kv, t0, draft, ws)
            cur.wait_event(ev_in)
            api.dflash_verify_accept(logits, draft, n_out, corr, emitted, nxt, vws)
            api.dflash_kv_commit(model, kv, blk, n_out, ws)
            ev_done.record(cur)
            copies_out()

        g_step = capture(torch, step)

        def e2e_graph():
            copies_in()
            g_step.replay()
            copies_out()

        # the same calls and copies captured once into a CUDA graph whose side
        # branch copies the target logits and hidden rows while the draft pass
        # runs: every replay moves that step's inputs in and its results out
        def overlapped_body():
            cur = torch.cuda.current_stream()
            side.wait_stream(cur)
            with torch.cuda.stream(side):
                logits.copy_(h_lg, non_blocking=True)
                blk.copy_(h_blk, non_blocking=True)
            t0.copy_(h_t0, non_blocking=True)
            kv.len.copy_(len0)
            api.dflash_draft_block(model, kv, t0, draft, ws)
            cur.wait_stream(side)
            api.dflash_verify_accept(logits, draft, n_out, corr, emitted, nxt, vws)
            api.dflash_kv_commit(model, kv, blk, n_out, ws)
            copies_out()

        g_ov, g_ov_err = None, None
        try:
            g_ov = capture(torch, overlapped_body)
        except Exception as exc:  # a runtime that cannot capture the pinned copies
            g_ov_err = f"{type(exc).__name__}: {exc}"[:200]
            torch.cuda.synchronize()

        def timed_host(fn):
            for _ in range(Wm):
                fn()
            torch.cuda.synchronize()
            if world > 1:
                torch.distributed.barrier()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(K):
                fn()
            e1.record()
            torch.cuda.synchronize()
            return max_over_ranks(e0.elapsed_time(e1), world, dev)

        e2e_ms = timed_host(e2e_overlapped)
        # the accept counts that came back are the planted ones
        assert np.array_equal(o_n.numpy(), np.asarray(nacc, dtype=np.int32)), "overlapped end-to-end step"
        e2e_serial_ms = timed_host(e2e_eager)
        e2e_graph_ms = timed_host(e2e_graph)
        e2e_gov_ms = None
        if g_ov is not None:
            o_n.zero_()
            e2e_gov_ms = timed_host(g_ov.replay)
            assert np.array_equal(o_n.numpy(), np.asarray(nacc, dtype=np.int32)), "graph-overlapped end-to-end step"
            del g_ov
        assert api.dflash_get_status() == 0, "device status flagged during the API timing"
        del g_step

    # the same draft step with int4 projections (W4A16, group scales in the
    # packed tiles); the cache and inputs are the ones above
    w4 = None
    if not args.no_w4:
        W4 = synth.drafter_weights(cfg, bits=4)
        m4 = api.DeviceDrafter(cfg, synth.FloatWeights(W4), dev, bits=4)
        del W4
        draft4 = torch.empty_like(draft)
        with api.launch_mode(api.LAUNCH_EARLY):
            _, d4 = timed_graph(torch, capture(torch, lambda: api.dflash_draft_block(m4, kv, t0, draft4, ws)),
                                K, Wm, world, dev)
        assert api.dflash_get_status() == 0, "device status flagged during the int4 draft timing"
        b4 = cfg.step_bytes_w4(list(ctx))
        w4 = {"median_us": med_us(d4), "bytes": b4, "frac_of_measured": b4 / (statistics.median(d4) * 1e-3) / 1e9 / hbm}
        del m4

    overlap = None if args.no_overlap else overlap_measurement(torch, api, args, world, dev, K, Wm)

    ms_step = early["step_total_ms"] / K
    value = whole_job_rate(world, b, K, early["step_total_ms"])
    step_bytes = cfg.step_bytes(list(ctx))
    lm_bytes = cfg.V * cfg.H * 2 + M1 * cfg.H * 2 + M1 * 4
    lm_gbs = lm_bytes / (statistics.mean(lm_ms) * 1e-3) / 1e9
    def proj_roofline(kname):
        p = proj[kname]
        t = statistics.mean(p["ms"])
        gbs = p["bytes"] / (t * 1e-3) / 1e9
        label = ("w8_gemm_kernel (tcgen05 W8A16 projection" if kname == "w8_gemm_kernel"
                 else "wmma_gemm_kernel (warp-level W8A16 projection")
        return {"kernel": f"{label}, {cfg.M} rows): the {p['n']} {p['what']} projections of one draft step, "
                          "launched back to back alone",
                "bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                "traffic": traffic_for(kname, "k_gemm_w8.cu", p["bytes"] / p["n"]), "peak_kind": peak_kind,
                "algorithmic_bytes_per_launch": p["bytes"] / p["n"], "avg_launch_us": t / p["n"] * 1e3,
                "total_us": t * 1e3}

    # the dominant projection kernel: the group with the larger total time
    order = sorted(proj, key=lambda k: -statistics.mean(proj[k]["ms"]))
    roofline = proj_roofline(order[0])
    roofline_other = proj_roofline(order[1]) if len(order) > 1 else None
    # the library's lm-head runs on tensor memory for 33 to 128 rows
    lm_kernel = "lmhead_tc_kernel" if 32 < M1 <= 128 and cfg.H % 64 == 0 else "lmhead_kernel"
    traffic_lm = traffic_for(lm_kernel, "k_lmhead.cu", lm_bytes)
    sweep_out = {}
    for label, lens in sweep:
        cb = cfg.step_bytes(lens)
        sweep_out[label] = {}
        for mname, res in results.items():
            dm = statistics.median(res["draft_us"][label])
            sweep_out[label][mname] = {
                "median_us": dm * 1e3, "p10_us": float(np.percentile(res["draft_us"][label], 10)) * 1e3,
                "p90_us": float(np.percentile(res["draft_us"][label], 90)) * 1e3, "bytes": cb,
                "frac_of_measured": cb / (dm * 1e-3) / 1e9 / hbm, "frac_of_8TBps": cb / (dm * 1e-3) / 1e9 / 8000.0}
    out = {
        "metric": METRIC, "value": value, "unit": "blocks/s", "n_gpus": world, "steps": K, "warmup": Wm,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int8xf16->f32 (W8A16), bf16 lm-head, fp16 KV", "data": "synthetic",
        "config": config_dict(cfg, ctx, world),
        "launch_mode": "early (programmatic dependent launch; one stream on a dedicated GPU)",
        "step": "draft + verify-accept + commit of the accepted rows (separate calls, one CUDA graph)",
        "step_stream_order": {"ms_per_step": results["stream_order"]["step_total_ms"] / K,
                              "blocks_per_s": whole_job_rate(world, b, K, results["stream_order"]["step_total_ms"])},
        "step_commit_folded": {"blocks_per_s": whole_job_rate(world, b, K, fold_total), "ms_per_step": fold_total / K,
                               "gpu_launches_per_step": launches_per_step(cfg, folded=True)},
        "draft_step_us": {"median": dms * 1e3, "p10": float(np.percentile(early["draft_us"][head_label], 10)) * 1e3,
                          "p90": float(np.percentile(early["draft_us"][head_label], 90)) * 1e3},
        "draft_step_ctx_sweep": sweep_out,
        "draft_step_weight_GBps": step_bytes / (dms * 1e-3) / 1e9,
        "step_roofline": {"bytes": step_bytes, "frac_of_measured": step_bytes / (dms * 1e-3) / 1e9 / hbm,
                          "frac_of_8TBps": step_bytes / (dms * 1e-3) / 1e9 / 8000.0},
        "draft_step_w4a16": w4,
        "draft_verify_overlap": overlap,
        "verify_accept_blocks_per_s": b / (statistics.median(ver_ms) / VREP / 1e3),
        "verify_sample_blocks_per_s": b / (statistics.median(smp_ms) / VREP / 1e3),
        "roofline": roofline,
        "roofline_projections_other_kernel": roofline_other,
        "roofline_lmhead": {"kernel": (f"{lm_kernel} (bf16 {'tcgen05 GEMM' if lm_kernel == 'lmhead_tc_kernel' else 'GEMV'}"
                                       f" + fused argmax, {M1} rows), alone"), "bound": "hbm",
                            "achieved": lm_gbs, "peak": hbm, "unit": "GB/s", "frac": lm_gbs / hbm,
                            "traffic": traffic_lm, "algorithmic_bytes_per_launch": lm_bytes,
                            "avg_launch_us": statistics.mean(lm_ms) * 1e3},
        "clocks": clocks,
        "gpu_launches": K * launches_per_step(cfg),
        "e2e": ({"value": whole_job_rate(world, b, K, e2e_gov_ms), "unit": "blocks/s", "h2d_bytes_per_step": h2d,
                 "d2h_bytes_per_step": d2h,
                 "path": "pinned host buffers in, dflash_draft_block + dflash_verify_accept + dflash_kv_commit, "
                         "results back to pinned host buffers, all captured once into a CUDA graph replayed "
                         "every step; the target logits and hidden rows are copied on a side branch of the "
                         "graph while the draft pass runs (verify waits for them)"}
                if e2e_gov_ms is not None else
                {"value": whole_job_rate(world, b, K, e2e_ms), "unit": "blocks/s", "h2d_bytes_per_step": h2d,
                 "d2h_bytes_per_step": d2h, "graph_capture_error": g_ov_err,
                 "path": "pinned host buffers in, dflash_draft_block + dflash_verify_accept + dflash_kv_commit "
                         "called every step, results back to pinned host buffers; the target logits and hidden "
                         "rows are copied on a second stream while the draft pass runs (verify waits for them)"}),
        "e2e_eager_overlapped": {"value": whole_job_rate(world, b, K, e2e_ms), "unit": "blocks/s",
                                 "path": "the calls issued eagerly every step, the target logits and hidden rows "
                                         "copied on a second stream while the draft pass runs"},
        "e2e_serial": {"value": whole_job_rate(world, b, K, e2e_serial_ms), "unit": "blocks/s",
                       "path": "the calls issued eagerly with every copy on the step's stream, before and after "
                               "the calls"},
        "e2e_graph": {"value": whole_job_rate(world, b, K, e2e_graph_ms), "unit": "blocks/s",
                      "path": "every copy on the step's stream around a replay of the captured step"},
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


def overlap_measurement(torch, api, args, world, dev, K, Wm):
    """Draft || verify overlap on two streams (mirror-sd README, "How It
    Works"): two groups of the Qwen3-4B-shaped workload, each step = draft,
    the int4 QMM stand-in for the target's verify forward, verify-accept,
    commit; serial vs side by side.  Several streams run at once, so the
    library runs in stream-order mode."""
    from block_diffusion_speculative_draft_gb300 import workload as WL
    cfg = configs.QWEN3_4B
    b = cfg.b
    model = api.DeviceDrafter(cfg, synth.FloatWeights(synth.drafter_weights(cfg)), dev)
    ctx = WL.contexts(cfg)
    standin = WL.TargetStandIn(api, torch, cfg, dev)
    groups = []
    for i in range(2):
        hids = [synth.target_hidden(cfg.seed, f"ovl-g{i}-ctx{j}", int(ctx[j]), cfg.k * cfg.H) for j in range(b)]
        groups.append(WL.Group(api, torch, cfg, model, dev, ctx, hids,
                               synth.tokens(cfg.seed, f"ovl-g{i}-t0", b, cfg.V), f"ovl-g{i}-"))
    side = [torch.cuda.Stream(device=dev)]
    with api.launch_mode(api.LAUNCH_STREAM_ORDER):
        g_ser = capture(torch, lambda: WL.run_serial(api, torch, cfg, model, standin, groups, reset=True))
        g_free = capture(torch, lambda: WL.run_overlapped(api, torch, cfg, model, standin, groups, side, reset=True))
        g_stag = capture(torch, lambda: WL.run_overlapped(api, torch, cfg, model, standin, groups, side,
                                                          reset=True, stagger=True))
        g_qmm = capture(torch, lambda: api.dflash_w8a16_linear(standin.desc, groups[0].blk.view(-1, cfg.k * cfg.H),
                                                                ws=groups[0].tws, y=groups[0].logits.view(-1, cfg.V)))
        g_draft = capture(torch, lambda: api.dflash_draft_block(model, groups[0].kv, groups[0].t0, groups[0].draft,
                                                                groups[0].ws))
        ser_ms, _ = timed_graph(torch, g_ser, K, Wm, world, dev)
        free_ms, _ = timed_graph(torch, g_free, K, Wm, world, dev)
        stag_ms, _ = timed_graph(torch, g_stag, K, Wm, world, dev)
        _, qmm_ms = timed_graph(torch, g_qmm, K, Wm, world, dev)
        _, dr_ms = timed_graph(torch, g_draft, K, Wm, world, dev)
    assert api.dflash_get_status() == 0, "device status flagged during the overlap timing"
    nb = 2 * b
    best = min(free_ms, stag_ms)
    return {
        "workload": f"2 groups x {cfg.name}; target stand-in: int4 QMM [{cfg.V}][{cfg.k * cfg.H}] "
                    f"({standin.bytes() / 1e6:.0f} MB) from the block's target hidden rows to its logits",
        "launch_mode": "stream order (several streams at once)",
        "serial_ms_per_step": ser_ms / K, "free_ms_per_step": free_ms / K, "staggered_ms_per_step": stag_ms / K,
        "blocks_per_s_serial": whole_job_rate(world, nb, K, ser_ms),
        "blocks_per_s_free": whole_job_rate(world, nb, K, free_ms),
        "blocks_per_s_staggered": whole_job_rate(world, nb, K, stag_ms),
        "standin_qmm_us": med_us(qmm_ms), "draft_us": med_us(dr_ms),
        "draft_time_hidden_frac": (ser_ms - best) / K / (nb * statistics.median(dr_ms)),
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-overlap", action="store_true", help="skip the two-stream draft || verify measurement")
    ap.add_argument("--no-w4", action="store_true", help="skip the int4 (W4A16) draft timing")
    ap.add_argument("--config", default=None, choices=sorted(configs.BY_NAME),
                    help="another workload of the parity suite (default: the 27B-class drafter at 4096 "
                         "context rows)")
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
