"""Seeded synthetic inputs shared by the oracle tests, the GPU tests and bench.py.

This module only draws numbers and rounds them to their storage type once; it
holds none of the drafter's arithmetic.  Both sides of every parity check read
the same bits from here.  No trained weights, prompts or datasets exist on
either machine, so these tensors stand in for the drafters and prompt suites
the pages measure (mirror-sd README "Results"; dflash-mlx summary
"Benchmarks"; mlx-dspark v0.0.3 "Head-to-head"), with the same shapes.

Recipe (per workload seed):
  * int8 weight grid: integers uniform in [-127, 127]; one random column per
    row is set to +-127 so that every row's absmax is exactly 127 * scale;
  * per-output-channel scale: fp16 of lognormal(mu=-6, sigma=0.3);
  * the float weight handed to the packer is that grid times its row scale,
    so W8A16 packing of it is lossless;
  * RMSNorm gammas 1 + N(0, 0.02) in fp32;
  * embedding and lm-head: bf16 of N(0, 0.02);
  * target hidden rows: fp16 of N(0, 1), k*H wide;
  * verify logits: fp32 N(0, 1), with the first n rows planted so that the
    draft token is the row maximum and row n planted so that it is not.
"""
from __future__ import annotations

import zlib
from typing import Dict, Iterable, List, Tuple

import numpy as np

LM_CHUNK = 8192  # rows per independently seeded chunk of a vocab-sized table


def rng_for(seed: int, *tags) -> np.random.Generator:
    """Generator keyed by (seed, tags): independent of generation order."""
    words = [int(seed) & 0xFFFFFFFF]
    for t in tags:
        if isinstance(t, (int, np.integer)):
            words.append(int(t) & 0xFFFFFFFF)
        else:
            words.append(zlib.crc32(str(t).encode()))
    return np.random.default_rng(np.random.SeedSequence(words))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest-even) and return the 16-bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(u: np.ndarray) -> np.ndarray:
    return (np.asarray(u, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def w8_grid(seed: int, name: str, N: int, K: int) -> Tuple[np.ndarray, np.ndarray]:
    """int8 grid q[N][K] (row absmax 127) and fp16 row scales s[N]."""
    rng = rng_for(seed, "w8", name)
    q = rng.integers(-127, 128, size=(N, K), dtype=np.int8)
    col = rng.integers(0, K, size=N)
    sign = np.where(rng.integers(0, 2, size=N) == 1, 127, -127).astype(np.int8)
    q[np.arange(N), col] = sign
    s = rng.lognormal(mean=-6.0, sigma=0.3, size=N).astype(np.float16)
    return q, s


def w4_grid(seed: int, name: str, N: int, K: int) -> Tuple[np.ndarray, np.ndarray]:
    """int4 grid q[N][K] in [-7, 7] (absmax 7 in every 128-column group) and
    fp16 scales s[N][K / 128]; magnitudes comparable to w8_grid's."""
    rng = rng_for(seed, "w4", name)
    G = K // 128
    q = rng.integers(-7, 8, size=(N, K), dtype=np.int8)
    col = rng.integers(0, 128, size=(N, G)) + 128 * np.arange(G)[None, :]
    sign = np.where(rng.integers(0, 2, size=(N, G)) == 1, 7, -7).astype(np.int8)
    q[np.arange(N)[:, None], col] = sign
    s = rng.lognormal(mean=-3.1, sigma=0.3, size=(N, G)).astype(np.float16)
    return q, s


def w4_float(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """The synthetic float weight on each group's int4 grid, as fp32."""
    return q.astype(np.float32) * np.repeat(s.astype(np.float32), 128, axis=1)


def w8_float(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """The synthetic float weight on each row's int8 grid, as fp32."""
    return q.astype(np.float32) * s.astype(np.float32)[:, None]


def gamma(seed: int, name: str, shape) -> np.ndarray:
    rng = rng_for(seed, "gamma", name)
    return (1.0 + 0.02 * rng.standard_normal(shape)).astype(np.float32)


def bf16_table(seed: int, name: str, V: int, H: int) -> np.ndarray:
    """bf16 bit patterns of N(0, 0.02) [V][H], seeded per LM_CHUNK rows."""
    out = np.empty((V, H), dtype=np.uint16)
    for c0 in range(0, V, LM_CHUNK):
        c1 = min(V, c0 + LM_CHUNK)
        rng = rng_for(seed, "bf16", name, c0 // LM_CHUNK)
        out[c0:c1] = f32_to_bf16_bits(0.02 * rng.standard_normal((c1 - c0, H), dtype=np.float32))
    return out


def bf16_rows(seed: int, name: str, rows: int, H: int, std: float = 1.0) -> np.ndarray:
    rng = rng_for(seed, "bf16rows", name)
    return f32_to_bf16_bits(std * rng.standard_normal((rows, H), dtype=np.float32))


def target_hidden(seed: int, name: str, rows: int, width: int) -> np.ndarray:
    """fp16 N(0, 1) target hidden rows [rows][k*H]."""
    rng = rng_for(seed, "hid", name)
    return rng.standard_normal((rows, width), dtype=np.float32).astype(np.float16)


def tokens(seed: int, name: str, n: int, V: int) -> np.ndarray:
    rng = rng_for(seed, "tok", name)
    return rng.integers(0, V, size=n).astype(np.int32)


def truncated_geometric_ratio(mean: float, D: int) -> float:
    """r with E[n] = mean for pmf(n) proportional to r**n on n in [0, D]."""
    def m(r):
        n = np.arange(D + 1, dtype=np.float64)
        w = np.power(r, n)
        return float((n * w).sum() / w.sum())
    lo, hi = 1e-6, 1e3
    for _ in range(200):
        mid = np.sqrt(lo * hi)
        if m(mid) < mean:
            lo = mid
        else:
            hi = mid
    return float(np.sqrt(lo * hi))


def accept_lengths(seed: int, name: str, b: int, D: int, mean=None) -> np.ndarray:
    """Per-sequence accept lengths: uniform on [0, D] when mean is None,
    else truncated geometric with the given mean."""
    rng = rng_for(seed, "acc", name)
    if mean is None:
        return rng.integers(0, D + 1, size=b).astype(np.int32)
    r = truncated_geometric_ratio(mean, D)
    n = np.arange(D + 1, dtype=np.float64)
    p = np.power(r, n)
    p /= p.sum()
    return rng.choice(D + 1, size=b, p=p).astype(np.int32)


def ragged_contexts(seed: int, name: str, b: int, lo: int, hi: int) -> np.ndarray:
    rng = rng_for(seed, "ctx", name)
    return rng.integers(lo, hi + 1, size=b).astype(np.int32)


def verify_logits(seed: int, name: str, draft: np.ndarray, R: int, V: int,
                  n_accept: np.ndarray) -> np.ndarray:
    """fp32 N(0,1) logits [b][R][V] planted so that rows r < n[j] have their
    maximum at draft[j][r] and row n[j] (when it is a draft row) does not."""
    draft = np.asarray(draft, dtype=np.int64)
    b, D = draft.shape
    rng = rng_for(seed, "logits", name)
    lg = rng.standard_normal((b, R, V), dtype=np.float32)
    for j in range(b):
        n = int(n_accept[j])
        for r in range(min(n, D)):
            lg[j, r, draft[j, r]] = lg[j, r].max() + np.float32(1.0)
        if n < D:
            row = lg[j, n]
            if int(np.argmax(row)) == int(draft[j, n]):
                row[draft[j, n]] = row.min() - np.float32(1.0)
    return lg


def drafter_weights(cfg, with_float: bool = False, bits: int = 8) -> Dict[str, object]:
    """All drafter tensors for a workload (host numpy arrays); bits = 4 draws
    the projections on int4 grids with per-128-column group scales.

    W8 matrices are stored as (q, s) in their logical row order:
      qkv  [(nq + 2 nkv) d][H]  rows: q heads, then k heads, then v heads
      o    [H][nq d]
      gu   [2F][H]              rows: F gate rows, then F up rows
      down [H][F]
      fc   [H][k H]
    """
    sd, L, H, d, F = cfg.seed, cfg.L, cfg.H, cfg.d, cfg.F
    W: Dict[str, object] = {}
    grid = w4_grid if bits == 4 else w8_grid
    W["fc"] = grid(sd, "fc", H, cfg.k * H)
    for l in range(L):
        W[f"qkv{l}"] = grid(sd, f"qkv{l}", cfg.nqkv, H)
        W[f"o{l}"] = grid(sd, f"o{l}", H, cfg.nq * d)
        W[f"gu{l}"] = grid(sd, f"gu{l}", 2 * F, H)
        W[f"down{l}"] = grid(sd, f"down{l}", H, F)
    W["gamma_hid"] = gamma(sd, "hid", (H,))
    W["gamma_in"] = gamma(sd, "in", (L, H))
    W["gamma_post"] = gamma(sd, "post", (L, H))
    W["gamma_q"] = gamma(sd, "q", (L, d))
    W["gamma_k"] = gamma(sd, "k", (L, d))
    W["gamma_final"] = gamma(sd, "final", (H,))
    W["embed"] = bf16_table(sd, "embed", cfg.V, H)
    W["lm_head"] = bf16_table(sd, "lm_head", cfg.V, H)
    return W


class FloatWeights:
    """A read-only view of drafter_weights' dict in which every projection
    matrix reads as its float weight (fp32, grid times scale) and every other
    entry as stored.  Each matrix is built on access, so a consumer that
    takes them one at a time holds one float matrix at a time."""

    def __init__(self, W: Dict[str, object]):
        self.W = W

    def __getitem__(self, name: str):
        v = self.W[name]
        if isinstance(v, tuple):
            q, s = v
            return w4_float(q, s) if s.ndim == 2 else w8_float(q, s)
        return v

    def __contains__(self, name: str) -> bool:
        return name in self.W

    def keys(self):
        return self.W.keys()


W8_NAMES = ("qkv", "o", "gu", "down")


def w8_names(cfg) -> List[str]:
    return ["fc"] + [f"{n}{l}" for l in range(cfg.L) for n in W8_NAMES]
