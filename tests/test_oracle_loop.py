"""Whole-loop pin: greedy speculative decoding with the oracle's verify-accept
and commit rule reproduces plain greedy decoding of a toy target exactly
(mlx-dspark v0.0.3 release notes: greedy output identical to plain decoding up
to fp ties; the toy target computes each row identically in both modes, so
equality here is exact), and the drafter context after every step holds
exactly the target hidden rows of the accepted tokens (rollback of the
rejected suffix)."""
import dataclasses

import numpy as np
import pytest

from oracle import dflash_oracle as O
from oracle.toy_target import ToyTarget, greedy, speculative
from block_diffusion_speculative_draft_gb300 import synth
from block_diffusion_speculative_draft_gb300.configs import DrafterConfig

MICRO = DrafterConfig(name="micro", L=1, H=64, nq=4, nkv=2, d=16, F=128, V=512,
                      B=8, k=3, b=1, ctx=(0,), seed=77)


@pytest.fixture(scope="module")
def setup():
    W = synth.drafter_weights(MICRO)
    D = O.Drafter(MICRO, W)
    tgt = ToyTarget(MICRO.V, MICRO.H, 4, W["embed"], W["lm_head"], seed=5)
    prompt = [int(t) for t in synth.tokens(3, "prompt", 12, MICRO.V)]
    n_new = 48
    ref = greedy(tgt, prompt, n_new + MICRO.B + 1)
    return W, D, tgt, prompt, n_new, ref


def _oracle_drafter(D):
    def fn(t0, ctx_hidden, history):
        Ks, Vs = O.context_kv(D, ctx_hidden.astype(np.float16))
        return O.draft_block(D, t0, Ks, Vs, want_logits=False)["draft"]
    return fn


def _perfect(ref, prompt, B, corrupt=None):
    def fn(t0, ctx_hidden, history):
        m = len(history) - len(prompt)  # ref tokens emitted so far, t0 included
        d = list(ref[m:m + B - 1])
        if corrupt is not None:
            i = corrupt(m)
            if i is not None and i < len(d):
                d[i] = (d[i] + 1) % 512
        return d
    return fn


@pytest.mark.parametrize("kind", ["oracle", "perfect", "corrupt", "random"])
def test_greedy_equivalence(setup, kind):
    W, D, tgt, prompt, n_new, ref = setup
    B = MICRO.B
    rng = np.random.default_rng(0)
    if kind == "oracle":
        fn = _oracle_drafter(D)
    elif kind == "perfect":
        fn = _perfect(ref, prompt, B)
    elif kind == "corrupt":
        fn = _perfect(ref, prompt, B, corrupt=lambda m: (m * 7) % (B + 2))
    else:
        fn = lambda t0, c, h: rng.integers(0, MICRO.V, B - 1)
    checks = []
    res = speculative(tgt, fn, prompt, n_new, B, ctx_check=checks)
    assert res["tokens"] == ref[:n_new]
    if kind == "perfect":
        assert all(a == B - 1 for a in res["accepts"])
    if kind == "corrupt":
        assert any(a < B - 1 for a in res["accepts"]) and any(a == B - 1 for a in res["accepts"])
    # committed drafter context == target hidden rows of exactly the accepted
    # history (rejected suffix rolled back)
    for hist, ctx in checks[:4] + checks[-2:]:
        tgt.reset()
        rows = [tgt.step(t)[1] for t in hist]
        assert np.array_equal(np.stack(rows), ctx)


def test_context_rows_are_independent_of_chunking(setup):
    W, D, *_ = setup
    hid = synth.target_hidden(5, "chunk", 40, MICRO.k * MICRO.H)
    K, V = O.context_kv(D, hid, 0)
    K1, V1 = O.context_kv(D, hid[:17], 0)
    K2, V2 = O.context_kv(D, hid[17:], 17)
    for l in range(MICRO.L):
        assert np.allclose(np.concatenate([K1[l], K2[l]]), K[l], rtol=1e-13, atol=1e-13)
        assert np.allclose(np.concatenate([V1[l], V2[l]]), V[l], rtol=1e-13, atol=1e-13)


def test_draft_block_structure(setup):
    W, D, *_ = setup
    hid = synth.target_hidden(5, "ctx", 20, MICRO.k * MICRO.H)
    Ks, Vs = O.context_kv(D, hid)
    out = O.draft_block(D, 3, Ks, Vs)
    B = MICRO.B
    assert out["draft"].shape == (B - 1,) and out["logits"].shape == (B - 1, MICRO.V)
    assert np.array_equal(out["draft"], np.argmax(out["logits"], axis=1))
    # final RMSNorm: h / gamma_final has unit RMS up to eps
    hn = out["hidden"] / W["gamma_final"][None].astype(np.float64)
    assert np.allclose(np.sqrt(np.mean(hn * hn, axis=1)), 1.0, rtol=1e-5)
    # non-causal block: slot 0's token changes every draft row's logits
    out2 = O.draft_block(D, 4, Ks, Vs)
    assert np.all(np.abs(out2["logits"] - out["logits"]).max(axis=1) > 0)
    # the context conditions every slot
    out3 = O.draft_block(D, 3, [k[:10] for k in Ks], [v[:10] for v in Vs])
    assert np.all(np.abs(out3["logits"] - out["logits"]).max(axis=1) > 0)


def _zero(W, name):
    q, s = W[name]
    W[name] = (np.zeros_like(q), s)


def _one_layer_from(W2, l):
    """A 1-layer weight dict holding layer l of a 2-layer one."""
    W1 = {k: v for k, v in W2.items() if not k[-1].isdigit()}
    for m in ("qkv", "o", "gu", "down"):
        W1[f"{m}0"] = W2[f"{m}{l}"]
    for gname in ("gamma_in", "gamma_post", "gamma_q", "gamma_k"):
        W1[gname] = W2[gname][l:l + 1]
    return W1


@pytest.mark.parametrize("zeroed", [0, 1])
def test_zero_branch_layer_is_the_identity(zeroed):
    # a layer whose o and down projections are zero adds nothing to the
    # residual stream, so a 2-layer drafter with one such layer equals the
    # 1-layer drafter made of the other layer -- exactly (pins the residual
    # wiring, the layer order and which gammas / K/V each layer uses)
    cfg2 = dataclasses.replace(MICRO, L=2, seed=91)
    W2 = synth.drafter_weights(cfg2)
    _zero(W2, f"o{zeroed}")
    _zero(W2, f"down{zeroed}")
    keep = 1 - zeroed
    W1 = _one_layer_from(W2, keep)
    D2, D1 = O.Drafter(cfg2, W2), O.Drafter(MICRO, W1)
    hid = synth.target_hidden(5, "idl", 24, MICRO.k * MICRO.H)
    K2, V2 = O.context_kv(D2, hid)
    K1, V1 = O.context_kv(D1, hid)
    a = O.draft_block(D2, 11, K2, V2)
    b = O.draft_block(D1, 11, K1, V1)
    assert np.array_equal(a["logits"], b["logits"]) and np.array_equal(a["draft"], b["draft"])
    # negative control: without the zeroing the 2-layer drafter differs
    W2b = synth.drafter_weights(cfg2)
    D2b = O.Drafter(cfg2, W2b)
    Kb, Vb = O.context_kv(D2b, hid)
    assert np.abs(O.draft_block(D2b, 11, Kb, Vb)["logits"] - b["logits"]).max() > 1e-3


def test_context_order_does_not_matter(setup):
    # context keys carry their positions inside K (RoPE applied at commit), and
    # the block attends to all of them without a mask: permuting the context
    # rows (K and V together) leaves the draft unchanged
    W, D, *_ = setup
    hid = synth.target_hidden(5, "perm", 30, MICRO.k * MICRO.H)
    Ks, Vs = O.context_kv(D, hid)
    perm = np.random.default_rng(4).permutation(30)
    a = O.draft_block(D, 7, Ks, Vs)
    b = O.draft_block(D, 7, [k[perm] for k in Ks], [v[perm] for v in Vs])
    assert np.allclose(a["logits"], b["logits"], rtol=1e-12, atol=1e-12)
    # negative control: permuting K alone (breaking the K/V pairing) changes it
    c = O.draft_block(D, 7, [k[perm] for k in Ks], Vs)
    assert np.abs(c["logits"] - a["logits"]).max() > 1e-6
