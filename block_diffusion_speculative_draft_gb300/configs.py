"""Drafter workloads: shapes of the DFlash drafters the pages run.

Each workload is a few-layer W8A16 drafter that fills a block of B positions
in one non-causal pass (mlx-dspark v0.0.3 release notes, "Highlights"; mirror-sd
README, "How It Works": 5 drafter layers, block 32). Hidden sizes follow the
Qwen3-4B / Qwen3-8B / 27B-class targets that the pages pair with their drafters
(mirror-sd README, "Supported Models" and "Results" table).

Conventions that the pages leave open are fixed here: RMSNorm eps 1e-6 and
RoPE base 1e6 (Qwen3 conventions), mask token id V-1.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional


@dataclasses.dataclass(frozen=True)
class DrafterConfig:
    name: str
    L: int            # drafter layers
    H: int            # hidden size
    nq: int           # query heads
    nkv: int          # key/value heads
    d: int            # head_dim
    F: int            # SwiGLU FFN width
    V: int            # vocabulary (shared embedding / lm-head rows)
    B: int            # block size (position 0 = last accepted token, rest = mask)
    k: int            # hooked target layers; target hidden rows are k*H wide
    b: int = 1        # batch of independent sequences
    ctx: tuple = ()   # committed context length per sequence (fixed workloads)
    ctx_range: Optional[tuple] = None  # (lo, hi) uniform ragged contexts
    accept_mean: Optional[float] = None  # truncated-geometric mean accept length
    D: Optional[int] = None  # drafts verified per block (default B-1)
    rope_theta: float = 1.0e6
    eps: float = 1.0e-6
    seed: int = 1000

    @property
    def mask_id(self) -> int:
        return self.V - 1

    @property
    def R(self) -> int:
        """Target rows verified per block: one per block position."""
        return self.B

    @property
    def n_draft(self) -> int:
        return self.B - 1 if self.D is None else self.D

    @property
    def nqkv(self) -> int:
        return (self.nq + 2 * self.nkv) * self.d

    @property
    def M(self) -> int:
        return self.B * self.b

    def with_ctx(self, ctx) -> "DrafterConfig":
        return dataclasses.replace(self, ctx=tuple(ctx))

    # algorithmic bytes of one draft step (weights + scales + lm-head + KV read)
    def layer_weight_bytes(self) -> int:
        H, d = self.H, self.d
        per = H * self.nqkv + self.nq * d * H + 2 * self.F * H + self.F * H
        return self.L * per

    def scale_bytes(self) -> int:
        per = self.nqkv + self.H + 2 * self.F + self.H
        return 2 * self.L * per

    def lmhead_bytes(self) -> int:
        return 2 * self.V * self.H

    def kv_read_bytes(self, ctx: List[int]) -> int:
        return self.L * sum(int(c) for c in ctx) * self.nkv * self.d * 2 * 2

    def step_bytes(self, ctx: List[int]) -> int:
        return (self.layer_weight_bytes() + self.scale_bytes()
                + self.lmhead_bytes() + self.kv_read_bytes(ctx))

    def step_bytes_w4(self, ctx: List[int]) -> int:
        # int4 codes (half a byte per weight) + one fp16 scale per 128 weights
        lw = self.layer_weight_bytes()
        return lw // 2 + lw // 64 + self.lmhead_bytes() + self.kv_read_bytes(ctx)

    def commit_weight_bytes(self) -> int:
        fc = self.H * self.k * self.H + 2 * self.H
        kv = self.L * (2 * self.nkv * self.d * self.H + 2 * 2 * self.nkv * self.d)
        return fc + kv


TINY = DrafterConfig(
    name="tiny-1L-h512-v4096-b16", L=1, H=512, nq=8, nkv=2, d=64, F=1536,
    V=4096, B=16, k=3, b=1, ctx=(64,), D=16, seed=1000)

QWEN3_4B = DrafterConfig(
    name="qwen3-4b-shaped-5L-h2560-b16-ctx512", L=5, H=2560, nq=32, nkv=8,
    d=128, F=9728, V=151936, B=16, k=3, b=1, ctx=(512,), accept_mean=6.0,
    seed=1001)

QWEN3_8B = DrafterConfig(
    name="qwen3-8b-shaped-5L-h4096-b16-ctx2048", L=5, H=4096, nq=32, nkv=8,
    d=128, F=12288, V=151936, B=16, k=5, b=1, ctx=(2048,), accept_mean=6.0,
    seed=1002)

DENSE_27B = DrafterConfig(
    name="27b-class-5L-h5120-b32", L=5, H=5120, nq=40, nkv=8, d=128,
    F=17408, V=151936, B=32, k=5, b=1, ctx=(2048,), accept_mean=17.0,
    seed=1003)

BATCHED_8B = DrafterConfig(
    name="qwen3-8b-shaped-b8-ragged-256-8192", L=5, H=4096, nq=32, nkv=8,
    d=128, F=12288, V=151936, B=16, k=5, b=8, ctx_range=(256, 8192),
    accept_mean=6.0, seed=1004)

ALL = [TINY, QWEN3_4B, QWEN3_8B, DENSE_27B, BATCHED_8B]
BY_NAME = {c.name: c for c in ALL}
DENSE_27B_CTX_SWEEP = (64, 2048, 4096)
