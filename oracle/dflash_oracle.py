"""Oracle: a plain, slow CPU restatement of one DFlash draft step, the greedy
verify-accept that follows it, and the draft-KV commit.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or links
this module; only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline
leg (and its --impl reference arm) may use it.  It shares no code with the CUDA
library: every step below is written out from the pages' description, in
float64 numpy, one sequence at a time, with no blocking or fusion.

Sources (web pages on DFlash; cited by page title and section):
  [mirror-sd]  mirror-sd README: "The Story" (Phase 2: per-head Q/K norm over
               128 dims; Phase 3: neox split-half RoPE as
               mx.fast.rope(traditional=False), int8 weights with per-channel
               fp16 scales), "How It Works" (5 drafter layers, int8 constants
               dequantised affinely; step = target verify, draft, accept
               matching prefix + correction token).
  [dspark]     mlx-dspark v0.0.3 release notes, "Highlights": the drafter
               denoises a whole block in one parallel pass and reuses the
               target's embedding and lm-head; greedy output is identical to
               plain decoding up to fp ties; "Notes": KV rollback.
  [dflash-mlx] dflash-mlx summary, "What It Does" / "How it works": drafter
               conditioned on intermediate target activations, longest
               matching prefix accepted, one target forward verifies a block.

Where the pages are silent the plainest reading is taken and the docstring of
the function that takes it says so.  Parity status of each function is stated
in its docstring.  The whole-drafter composition has no worked example in the
pages; it is pinned by invariants instead (a layer with zero output
projections is the identity, context order does not matter, greedy
speculative decoding reproduces plain greedy decoding).  The conventions it
takes where the pages are silent (norm placement on the context path, RoPE
base, eps) are readings no pin can fix: for those choices parity is
"parity unpinned".
"""
from __future__ import annotations

from typing import Dict, List, Sequence, Tuple

import numpy as np

F64 = np.float64


# ----------------------------------------------------------------------------
# storage decoding (inputs arrive rounded to their storage types)
# ----------------------------------------------------------------------------
def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64 (exact).  Pinned on patterns
    decoded by hand (normal, subnormal, signed zero, largest finite, inf)."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(F64)


# ----------------------------------------------------------------------------
# W8A16 quantisation  [mirror-sd "The Story", Phase 3; "How It Works"]
# ----------------------------------------------------------------------------
def dequant_w8(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """w[n][k] = q[n][k] * s[n]: affine int8 dequantisation with a per-output
    -channel fp16 scale and zero offset.  Pinned: exact (q*s fits in fp32)."""
    return q.astype(F64) * np.asarray(s, dtype=np.float16).astype(F64)[:, None]


def pack_w8a16(w: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Per-output-channel symmetric int8 quantisation of w[N][K] (fp32).

    s[n] = fp16(absmax_n / 127), the division in fp32 and rounded to nearest
    even; q = clamp(rint(w / s), -127, 127) with the division in fp32 using the
    rounded s; rows whose s is 0 get q = 0.  Pinned: round trip on the int8
    grid is exact; |w - q s| <= s/2 elementwise; max|q| = 127 on every row.
    """
    w32 = np.asarray(w, dtype=np.float32)
    amax = np.abs(w32).max(axis=1)
    s = (amax / np.float32(127.0)).astype(np.float32).astype(np.float16)
    s32 = s.astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.rint(w32 / s32[:, None])
    r = np.where(s32[:, None] == 0, np.float32(0), r)
    q = np.clip(r, -127, 127).astype(np.int8)
    return q, s


GROUP4 = 128  # columns per int4 scale group


def dequant_w4(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """w[n][k] = q[n][k] * s[n][k / 128]: int4 values (in [-7, 7]) with one
    fp16 scale per output row and 128-column group.  A 4-bit drafter is the
    pages' default (mlx-dspark v0.0.3 release notes, "Notes": drafter
    quantisation does not affect acceptance, 4-bit stays the default); the
    symmetric format and the group size are a reading (the pages give neither).  Pinned:
    exact (q * s fits in fp32)."""
    sg = np.repeat(np.asarray(s, dtype=np.float16).astype(F64), GROUP4, axis=1)
    return q.astype(F64) * sg


def pack_w4a16(w: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Symmetric int4 quantisation of w[N][K] (fp32), K a multiple of 128.

    s[n][g] = fp16(absmax over row n, columns [128 g, 128 g + 128) / 7), the
    division in fp32 rounded to nearest even; q = clamp(rint(w / s), -7, 7)
    with the division in fp32 using the rounded s; groups whose s is 0 get
    q = 0.  Pinned: round trip on the int4 grid is exact; |w - q s| <= s/2;
    max|q| = 7 in every group."""
    w32 = np.asarray(w, dtype=np.float32)
    N, K = w32.shape
    g = w32.reshape(N, K // GROUP4, GROUP4)
    amax = np.abs(g).max(axis=2)
    s = (amax / np.float32(7.0)).astype(np.float32).astype(np.float16)
    s32 = s.astype(np.float32)[:, :, None]
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.rint(g / s32)
    r = np.where(s32 == 0, np.float32(0), r)
    q = np.clip(r, -7, 7).astype(np.int8).reshape(N, K)
    return q, s


# ----------------------------------------------------------------------------
# norms and rotary embedding
# ----------------------------------------------------------------------------
def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """y = x / sqrt(mean(x^2) + eps) * g over the last axis.  Pinned: RMS 1
    before gamma at eps=0; RMS sqrt(ms/(ms+eps)) otherwise."""
    x = np.asarray(x, dtype=F64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(g, dtype=F64)


def head_rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """Per-head Q/K RMSNorm: x[..., heads, d] normalised over each head's d
    values separately, never over all channels at once [mirror-sd "The
    Story", Phase 2 and 3].  Pinned: every head vector has RMS 1 before gamma;
    a global norm fails that check."""
    return rmsnorm(x, g, eps)


def rope_neox(x: np.ndarray, pos, theta: float) -> np.ndarray:
    """neox split-half rotary embedding [mirror-sd "The Story", Phase 3: the
    mx.fast.rope(traditional=False) convention].  Element i pairs with
    i + d/2 and rotates by pos * theta^(-2i/d):
        y_i       = x_i cos - x_{i+d/2} sin
        y_{i+d/2} = x_{i+d/2} cos + x_i sin
    x[..., d]; pos broadcasts against x[..., 0].  Pinned: identity at pos 0,
    norm-preserving, relative-position identity, pair (0, d/2) turns by pos."""
    x = np.asarray(x, dtype=F64)
    d = x.shape[-1]
    half = d // 2
    inv = np.power(F64(theta), -2.0 * np.arange(half, dtype=F64) / d)
    ang = np.asarray(pos, dtype=F64)[..., None] * inv
    c, s = np.cos(ang), np.sin(ang)
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def silu(z: np.ndarray) -> np.ndarray:
    z = np.asarray(z, dtype=F64)
    return z / (1.0 + np.exp(-z))


# ----------------------------------------------------------------------------
# block attention: non-causal GQA over [context K/V || block K/V]
# ----------------------------------------------------------------------------
def attention_gqa(q: np.ndarray, k: np.ndarray, v: np.ndarray) -> np.ndarray:
    """q[T][nq][d], k/v[S][nkv][d] -> o[T][nq][d].  Every query sees every key
    (the block is drafted in one non-causal pass [dspark "Highlights"]); query
    head h reads kv head h // (nq / nkv); scores scaled by 1/sqrt(d); softmax
    with the maximum subtracted.  Pinned: equal keys give mean(V); one key
    gives v; GQA head mapping; agrees with torch SDPA in float64."""
    q, k, v = (np.asarray(a, dtype=F64) for a in (q, k, v))
    T, nq, d = q.shape
    nkv = k.shape[1]
    grp = nq // nkv
    o = np.empty((T, nq, d), dtype=F64)
    for h in range(nq):
        kh, vh = k[:, h // grp, :], v[:, h // grp, :]
        sc = q[:, h, :] @ kh.T / np.sqrt(F64(d))
        sc = sc - sc.max(axis=1, keepdims=True)
        p = np.exp(sc)
        p /= p.sum(axis=1, keepdims=True)
        o[:, h, :] = p @ vh
    return o


# ----------------------------------------------------------------------------
# drafter weights view
# ----------------------------------------------------------------------------
class Drafter:
    """Dequantised float64 view of a drafter's tensors (lazy per matrix).

    W maps names to (q, s) pairs for W8 matrices (s per row) or W4
    matrices (s per row and 128-column group) in logical row order
    (qkv rows: q heads | k heads | v heads; gu rows: gate F | up F) and to
    arrays for gammas and the bf16 embedding / lm-head bit patterns."""

    def __init__(self, cfg, W: Dict[str, object], cache: bool = True):
        self.cfg, self.W, self.cache = cfg, W, cache
        self._cache: Dict[str, np.ndarray] = {}

    def w(self, name: str) -> np.ndarray:
        if name in self._cache:
            return self._cache[name]
        q, s = self.W[name]
        w = dequant_w4(q, s) if np.ndim(s) == 2 else dequant_w8(q, s)
        if self.cache:
            self._cache[name] = w
        return w

    def drop(self):
        self._cache.clear()


def linear(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """y = x W^T for W[N][K] (row n is output channel n)."""
    return np.asarray(x, dtype=F64) @ w.T


# ----------------------------------------------------------------------------
# context path: projected target hidden rows -> per-layer context K/V
# ----------------------------------------------------------------------------
def context_rows(D: Drafter, hid: np.ndarray) -> np.ndarray:
    """c = RMSNorm(fc(h); gamma_hid) for target hidden rows h[rows][k H]
    (fp16 storage).  The drafter is conditioned on intermediate target
    activations, not logits [dflash-mlx "What It Does"]; the projection and
    norm placement are the plainest reading (parity unpinned by the pages)."""
    cfg = D.cfg
    h = np.asarray(hid, dtype=np.float16).astype(F64)
    return rmsnorm(linear(h, D.w("fc")), D.W["gamma_hid"], cfg.eps)


def context_kv_layer(D: Drafter, l: int, c: np.ndarray, pos: np.ndarray):
    """Layer l's context K/V for context rows c at absolute positions pos:
    K = RoPE(QKnorm(Wk c)), V = Wv c, with the layer's own Wk/Wv."""
    cfg = D.cfg
    nq, nkv, d = cfg.nq, cfg.nkv, cfg.d
    wqkv = D.w(f"qkv{l}")
    wk = wqkv[nq * d:(nq + nkv) * d]
    wv = wqkv[(nq + nkv) * d:(nq + 2 * nkv) * d]
    k = linear(c, wk).reshape(-1, nkv, d)
    v = linear(c, wv).reshape(-1, nkv, d)
    k = head_rmsnorm(k, D.W["gamma_k"][l], cfg.eps)
    k = rope_neox(k, np.asarray(pos)[:, None], cfg.rope_theta)
    return k, v


def context_kv(D: Drafter, hid: np.ndarray, pos0: int = 0):
    """All layers' context K/V for committed hidden rows at positions
    pos0, pos0+1, ...  Returns lists K[l][rows][nkv][d], V[l]."""
    c = context_rows(D, hid)
    pos = pos0 + np.arange(c.shape[0])
    Ks, Vs = [], []
    for l in range(D.cfg.L):
        k, v = context_kv_layer(D, l, c, pos)
        Ks.append(k)
        Vs.append(v)
    return Ks, Vs


# ----------------------------------------------------------------------------
# one draft step for one sequence
# ----------------------------------------------------------------------------
def argmax_lowest(x: np.ndarray) -> np.ndarray:
    """Index of the maximum along the last axis; ties go to the lowest index."""
    return np.argmax(x, axis=-1)


def top2_margin(x: np.ndarray) -> np.ndarray:
    """Gap between the largest and the second-largest entry of each row
    (counting repeats, so a tied maximum gives 0).  The GPU's draft tokens
    are compared with the oracle's only where this gap exceeds 1e-2.  Pinned
    on hand-worked rows (ties, all-negative rows)."""
    part = np.partition(x, -2, axis=-1)
    return part[..., -1] - part[..., -2]


def draft_block(D: Drafter, t0: int, ctxK: List[np.ndarray], ctxV: List[np.ndarray],
                want_logits: bool = True, lm_chunk: int = 16384) -> Dict[str, np.ndarray]:
    """One block-diffusion draft pass for one sequence [dspark "Highlights";
    mirror-sd "How It Works"].

    Block slot 0 holds the last accepted token t0, slots 1..B-1 the mask token
    embedding; slot i sits at position C + i where C = committed context
    length.  Per layer (pre-norm):
        u = RMSNorm(x; gamma_in)
        q, k, v = Wq u, Wk u, Wv u       (int8 weights x fp16 scales)
        q, k = RoPE(QKnorm(q)), RoPE(QKnorm(k))   per head
        x += Wo attn(q, [ctxK || k], [ctxV || v])  (non-causal, GQA)
        u = RMSNorm(x; gamma_post)
        x += Wdown (silu(Wgate u) * Wup u)
    then h = RMSNorm(x[1:]; gamma_final), logits = h W_lm^T and
    draft[i] = argmax(logits[i]) (lowest index on ties): slot i+1 predicts its
    own token.  Returns draft [B-1], hidden h [B-1][H], logits [B-1][V] (when
    asked), margin [B-1] (top-2 logit gap)."""
    cfg = D.cfg
    H, nq, nkv, d, F, B = cfg.H, cfg.nq, cfg.nkv, cfg.d, cfg.F, cfg.B
    C = ctxK[0].shape[0] if ctxK else 0
    E = D.W["embed"]
    x = np.empty((B, H), dtype=F64)
    x[0] = bf16_to_f64(E[t0])
    x[1:] = bf16_to_f64(E[cfg.mask_id])[None, :]
    pos = C + np.arange(B)
    for l in range(cfg.L):
        u = rmsnorm(x, D.W["gamma_in"][l], cfg.eps)
        qkv = linear(u, D.w(f"qkv{l}"))
        q = qkv[:, :nq * d].reshape(B, nq, d)
        k = qkv[:, nq * d:(nq + nkv) * d].reshape(B, nkv, d)
        v = qkv[:, (nq + nkv) * d:].reshape(B, nkv, d)
        q = rope_neox(head_rmsnorm(q, D.W["gamma_q"][l], cfg.eps), pos[:, None], cfg.rope_theta)
        k = rope_neox(head_rmsnorm(k, D.W["gamma_k"][l], cfg.eps), pos[:, None], cfg.rope_theta)
        Kall = np.concatenate([ctxK[l], k], axis=0) if C else k
        Vall = np.concatenate([ctxV[l], v], axis=0) if C else v
        o = attention_gqa(q, Kall, Vall).reshape(B, nq * d)
        x = x + linear(o, D.w(f"o{l}"))
        u = rmsnorm(x, D.W["gamma_post"][l], cfg.eps)
        gu = linear(u, D.w(f"gu{l}"))
        g = silu(gu[:, :F]) * gu[:, F:]
        x = x + linear(g, D.w(f"down{l}"))
    h = rmsnorm(x[1:], D.W["gamma_final"], cfg.eps)
    logits = lmhead_logits(h, D.W["lm_head"], chunk=lm_chunk)
    out = {"draft": argmax_lowest(logits).astype(np.int32), "hidden": h,
           "margin": top2_margin(logits)}
    if want_logits:
        out["logits"] = logits
    return out


def lmhead_logits(h: np.ndarray, w_bits: np.ndarray, chunk: int = 16384) -> np.ndarray:
    """logits = h W_lm^T with the target's shared bf16 lm-head [dspark
    "Highlights": the drafter reuses the target's embedding and lm-head],
    computed over vocabulary chunks.  Pinned on hand-built tables whose
    vocabulary spans several chunk boundaries."""
    h = np.asarray(h, dtype=F64)
    V = w_bits.shape[0]
    out = np.empty((h.shape[0], V), dtype=F64)
    for c0 in range(0, V, chunk):
        c1 = min(V, c0 + chunk)
        out[:, c0:c1] = h @ bf16_to_f64(w_bits[c0:c1]).T
    return out


def lmhead_argmax(h_bits: np.ndarray, w_bits: np.ndarray):
    """argmax over the vocabulary of bf16 h[M][H] . bf16 W[V][H]^T, lowest
    index on ties; also the maximum logit and the top-2 margin.  Pinned on a
    hand-worked 9-row table with a tied maximum."""
    lg = lmhead_logits(bf16_to_f64(h_bits), w_bits)
    return argmax_lowest(lg).astype(np.int32), lg.max(axis=-1), top2_margin(lg), lg


# ----------------------------------------------------------------------------
# greedy verify-accept  [mirror-sd "How It Works" step 3; dflash-mlx "How it
# works": truncate at the first error, the target supplies the next token]
# ----------------------------------------------------------------------------
def verify_accept(logits: np.ndarray, draft: np.ndarray):
    """One sequence.  logits[R][V] (fp32 target rows; row r predicts the token
    after block input r), draft[D] with D <= R.

      a_r  = argmax logits[r] (lowest index on ties)
      n    = number of leading i < D with draft[i] == a_i
      corr = a_n if n < R else -1          (the correction / bonus token)
      emitted = draft[0:n] ++ [corr]  (padded with -1 to R entries)
      next_tok = last emitted token (position 0 of the next block)

    Pinned: brute force over tiny vocabularies; planted full / zero accepts;
    greedy equivalence of the whole loop with a toy target."""
    a = argmax_lowest(np.asarray(logits))
    R = a.shape[0]
    Dn = len(draft)
    n = 0
    while n < Dn and int(draft[n]) == int(a[n]):
        n += 1
    corr = int(a[n]) if n < R else -1
    emitted = np.full(R, -1, dtype=np.int32)
    emitted[:n] = np.asarray(draft[:n], dtype=np.int32)
    if corr >= 0:
        emitted[n] = corr
        next_tok = corr
    else:
        next_tok = int(draft[n - 1]) if n > 0 else -1
    return n, corr, emitted, next_tok


# ----------------------------------------------------------------------------
# temperature speculative-sampling accept  [mlx-dspark v0.0.3 release notes,
# "Highlights": with --temperature > 0 the loop stays lossless, every emitted
# token an exact sample from the target at temperature T, "via the same
# acceptance rule as DSpark"]
# ----------------------------------------------------------------------------
def softmax_t(z: np.ndarray, T: float) -> np.ndarray:
    """Target distribution at temperature T over the last axis, float64."""
    zt = np.asarray(z, dtype=F64) / F64(T)
    zt = zt - zt.max(axis=-1, keepdims=True)
    e = np.exp(zt)
    return e / e.sum(axis=-1, keepdims=True)


def gumbel_scores(z_row: np.ndarray, T: float, u: np.ndarray) -> np.ndarray:
    """Gumbel-max scores z/T - log(-log u), in float32 (the precision the
    sample decision is taken in): argmax of the scores is an exact draw from
    softmax(z/T) when u is uniform on (0, 1).  Pinned: frequencies against
    softmax_t."""
    zf = np.asarray(z_row, dtype=np.float32) / np.float32(T)
    uf = np.asarray(u, dtype=np.float32)
    return zf - np.log(-np.log(uf))


def verify_accept_sample(logits: np.ndarray, draft: np.ndarray, T: float, u_acc: np.ndarray,
                         u_sample: np.ndarray, exclude_rejected: bool = True):
    """One sequence of speculative sampling at temperature T > 0.

    The pages name the property (an exact sample from the target at T) and
    "the same acceptance rule as DSpark" without writing it out; the plainest
    reading is the standard speculative-sampling rule.  This drafter proposes
    greedily, so its proposal distribution q_i is one-hot at draft[i] and the
    rule reads:

      p_i  = softmax(logits[i] / T)
      draft i (in order) is accepted iff u_acc[i] < min(1, p_i(x_i) / q_i(x_i)) = p_i(x_i)
      n    = number of leading accepted drafts
      corr = a draw from the residual max(0, p_n - q_n) (p_n without x_n,
             renormalised) if n < D; a draw from p_D if n = D < R; -1 if
             n = D = R
      emitted / next_tok as in verify_accept.

    The one categorical draw uses the Gumbel-max trick over u_sample[V] (one
    uniform per vocabulary entry; the residual excludes x_n).  Random numbers
    are inputs.  Accept probabilities are float64; the draw is decided in
    float32 (gumbel_scores).  exclude_rejected=False is a deliberately wrong
    variant kept for the negative-control test.

    Pinned: T -> 0 equals verify_accept; emitted-token frequencies against
    p_0 and p_1 by chi-square (a wrong residual fails).
    Returns n, corr, emitted, next_tok, and diagnostics (accept probabilities,
    the u - p margins, the top-2 score gap of the draw)."""
    z = np.asarray(logits)
    R, V = z.shape
    x = np.asarray(draft, dtype=np.int64)
    Dn = len(x)
    p_acc = np.array([softmax_t(z[i], T)[x[i]] for i in range(Dn)], dtype=F64)
    n = 0
    while n < Dn and float(u_acc[n]) < p_acc[n]:
        n += 1
    row = n if n < Dn else (Dn if Dn < R else -1)
    gap = np.inf
    if row < 0:
        corr = -1
    else:
        sc = gumbel_scores(z[row], T, u_sample).astype(F64)
        if n < Dn and exclude_rejected:
            sc[x[n]] = -np.inf
        corr = int(argmax_lowest(sc))
        srt = np.sort(sc)
        gap = float(srt[-1] - srt[-2])
    emitted = np.full(R, -1, dtype=np.int32)
    emitted[:n] = x[:n]
    if corr >= 0:
        emitted[n] = corr
        next_tok = corr
    else:
        next_tok = int(x[n - 1]) if n > 0 else -1
    diag = {"p_accept": p_acc, "u_minus_p": np.asarray(u_acc[:Dn], dtype=F64) - p_acc, "row": row,
            "score_gap": gap}
    return n, corr, emitted, next_tok, diag


def commit_rows(n: int, rows: int) -> int:
    """Rows of the verified block whose target hidden state enters the
    drafter's context: block inputs 0..n (the last token plus the n accepted
    drafts); the rejected suffix is rolled back by never being written
    [dspark "Notes": KV rollback].  Clamped to the rows provided."""
    return max(0, min(int(n) + 1, int(rows)))
