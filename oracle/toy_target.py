"""Tiny random causal target and the speculative loop around the oracle drafter.

TEST INFRASTRUCTURE ONLY (see oracle/dflash_oracle.py).  Used to pin the
whole draft -> verify -> accept -> commit loop against plain greedy decoding:
the pages state that greedy speculative output equals the target's own greedy
output up to fp ties [mlx-dspark v0.0.3 release notes, opening paragraph;
dflash-mlx summary, "Key Points": lossless; agentlens dflash-mlx "Highlights"].

The target computes every position with the same per-row code whether it is
fed one token (plain greedy) or a whole block (verify), so the two decodings
see bit-identical logits and equality is exact here, not up to ties.
"""
from __future__ import annotations

from typing import Dict, List, Optional

import numpy as np

from . import dflash_oracle as O

F64 = np.float64


class ToyTarget:
    """2-layer causal pre-norm transformer over a shared bf16 embedding and
    lm-head, exposing k = 3 hidden layers (embedding output and both layer
    outputs, concatenated) to the drafter [dflash-mlx "What It Does": the
    drafter reads intermediate target activations]."""

    def __init__(self, V: int, H: int, nh: int, embed_bits, lm_bits, seed: int = 7):
        rng = np.random.default_rng(seed)
        self.V, self.H, self.nh, self.d = V, H, nh, H // nh
        self.E = O.bf16_to_f64(embed_bits)
        self.Wlm = O.bf16_to_f64(lm_bits)
        sc = 1.0 / np.sqrt(H)
        self.layers = []
        for _ in range(2):
            self.layers.append({
                "wq": rng.standard_normal((H, H)) * sc, "wk": rng.standard_normal((H, H)) * sc,
                "wv": rng.standard_normal((H, H)) * sc, "wo": rng.standard_normal((H, H)) * sc,
                "w1": rng.standard_normal((2 * H, H)) * sc, "w2": rng.standard_normal((H, 2 * H)) * sc,
            })
        self.reset()

    def reset(self):
        self.K: List[List[np.ndarray]] = [[] for _ in self.layers]
        self.Vc: List[List[np.ndarray]] = [[] for _ in self.layers]

    def length(self) -> int:
        return len(self.K[0])

    def truncate(self, n: int):
        """Roll the target cache back to its first n positions."""
        for l in range(len(self.layers)):
            del self.K[l][n:]
            del self.Vc[l][n:]

    def step(self, tok: int):
        """Append one token; return (logits[V], hidden[3H]) for it."""
        x = self.E[int(tok)].copy()
        hid = [x.copy()]
        ones = np.ones(self.H)
        for l, P in enumerate(self.layers):
            u = O.rmsnorm(x, ones, 1e-6)
            q, k, v = P["wq"] @ u, P["wk"] @ u, P["wv"] @ u
            self.K[l].append(k)
            self.Vc[l].append(v)
            Ks, Vs = np.stack(self.K[l]), np.stack(self.Vc[l])
            o = np.empty(self.H)
            for h in range(self.nh):
                sl = slice(h * self.d, (h + 1) * self.d)
                s = Ks[:, sl] @ q[sl] / np.sqrt(self.d)
                p = np.exp(s - s.max())
                o[sl] = (p / p.sum()) @ Vs[:, sl]
            x = x + P["wo"] @ o
            u = O.rmsnorm(x, ones, 1e-6)
            x = x + P["w2"] @ np.maximum(P["w1"] @ u, 0.0)
            hid.append(x.copy())
        logits = self.Wlm @ O.rmsnorm(x, ones, 1e-6)
        return logits, np.concatenate(hid)


def greedy(target: ToyTarget, prompt: List[int], n_new: int) -> List[int]:
    """Plain greedy decoding: the reference token stream."""
    target.reset()
    for t in prompt:
        logits, _ = target.step(t)
    out = []
    tok = int(np.argmax(logits))
    while len(out) < n_new:
        out.append(tok)
        logits, _ = target.step(tok)
        tok = int(np.argmax(logits))
    return out


def speculative(target: ToyTarget, drafter_fn, prompt: List[int], n_new: int, B: int,
                ctx_check: Optional[list] = None) -> Dict[str, object]:
    """Block speculative decoding with greedy verify-accept.

    drafter_fn(t0, ctx_hidden_rows, history) -> B-1 draft tokens.  Each step:
    the target runs the block [t0, d_0..d_{B-2}] (one row per position),
    oracle.verify_accept picks n and the correction token, the target cache
    keeps rows 0..n and the drafter context gains the hidden rows 0..n
    (oracle.commit_rows)."""
    target.reset()
    ctx_hidden: List[np.ndarray] = []
    for t in prompt:
        logits, hid = target.step(t)
        ctx_hidden.append(hid)
    out = [int(np.argmax(logits))]
    accepts = []
    history = list(prompt)
    while len(out) < n_new:
        t0 = out[-1]
        draft = np.asarray(drafter_fn(t0, np.stack(ctx_hidden), history + [t0]), dtype=np.int64)
        base = target.length()
        rows_logits, rows_hid = [], []
        for tok in [t0] + list(draft):
            lg, hd = target.step(tok)
            rows_logits.append(lg)
            rows_hid.append(hd)
        n, corr, emitted, next_tok = O.verify_accept(np.stack(rows_logits), draft)
        keep = O.commit_rows(n, B)
        target.truncate(base + keep)
        ctx_hidden.extend(rows_hid[:keep])
        history.extend([t0] + [int(t) for t in draft[:n]])
        accepts.append(n)
        out.extend(int(t) for t in draft[:n])
        if corr >= 0:
            out.append(corr)
        if ctx_check is not None:
            ctx_check.append((list(history), np.stack(ctx_hidden)))
    return {"tokens": out[:n_new], "accepts": accepts}
