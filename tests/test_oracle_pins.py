"""Pins of the oracle against what the pages and the mathematics fix.

Every check here is independent of the oracle's own formulas: exact
representability, closed forms, invariants, library routines on special
cases, brute force on tiny inputs and hand-worked examples from the pages.
Negative controls plant a plausible mistake in the oracle (on the CPU) and
show that a pin catches it.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import dflash_oracle as O
from block_diffusion_speculative_draft_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- W8A16 -----
def test_dequant_is_exact_in_fp32():
    # int8 (8 bits) x fp16 (11-bit significand) fits fp32's 24 bits exactly,
    # so the float64 dequantisation must equal the fp32 product bit for bit.
    q, s = synth.w8_grid(11, "pin", 64, 256)
    w64 = O.dequant_w8(q, s)
    w32 = q.astype(np.float32) * s.astype(np.float32)[:, None]
    assert np.array_equal(w64, w32.astype(np.float64))
    # orientation: the scale belongs to the output channel (row)
    q1 = np.zeros((3, 5), np.int8)
    q1[1, 4] = 2
    s1 = np.array([1.0, 0.5, 4.0], np.float16)
    w = O.dequant_w8(q1, s1)
    assert w[1, 4] == 1.0 and np.count_nonzero(w) == 1


def test_pack_round_trip_on_int8_grid():
    # every synthetic row has absmax exactly 127 * s, so packing is lossless
    q, s = synth.w8_grid(12, "pin", 96, 384)
    q2, s2 = O.pack_w8a16(synth.w8_float(q, s))
    assert np.array_equal(q2, q)
    assert np.array_equal(s2.view(np.uint16), s.view(np.uint16))


def test_pack_error_bound_and_range():
    rng = np.random.default_rng(3)
    w = (rng.standard_normal((128, 200)) * rng.lognormal(-3, 1, (128, 1))).astype(np.float32)
    w[5] = 0.0  # an all-zero row
    q, s = O.pack_w8a16(w)
    s32 = s.astype(np.float32)
    assert np.all(np.abs(q.astype(np.int32)) <= 127)
    assert s[5] == 0 and not q[5].any()
    nz = s32 > 0
    # rounding to nearest: |w - q s| <= s/2 (+ fp32 rounding of w/s)
    err = np.abs(w.astype(np.float64) - O.dequant_w8(q, s))
    assert np.all(err[nz] <= s32[nz, None] * (0.5 + 1e-6) + 1e-30)
    # the row maximum maps to +-127 (or +-126 after fp16 rounding of s up)
    assert np.all(np.abs(q[nz]).max(axis=1) >= 126)


def test_pack_negative_control(monkeypatch):
    # truncation instead of round-to-nearest violates the s/2 bound
    rng = np.random.default_rng(4)
    w = rng.standard_normal((32, 64)).astype(np.float32)
    monkeypatch.setattr(O.np, "rint", np.trunc)
    q, s = O.pack_w8a16(w)
    err = np.abs(w.astype(np.float64) - O.dequant_w8(q, s))
    assert np.any(err > s.astype(np.float64)[:, None] * 0.5 * (1 + 1e-6))


# ---------------------------------------------------------------- W4A16 -----
def test_dequant_w4_is_exact_and_grouped():
    # int4 x fp16 is exact in fp32; the scale of column k is group k // 128
    q, s = synth.w4_grid(13, "pin4", 16, 512)
    w64 = O.dequant_w4(q, s)
    w32 = q.astype(np.float32) * np.repeat(s.astype(np.float32), 128, axis=1)
    assert np.array_equal(w64, w32.astype(np.float64))
    q1 = np.zeros((2, 256), np.int8)
    q1[1, 127] = 3
    q1[1, 128] = 5
    s1 = np.array([[1.0, 1.0], [0.5, 2.0]], np.float16)
    w = O.dequant_w4(q1, s1)
    assert w[1, 127] == 1.5 and w[1, 128] == 10.0 and np.count_nonzero(w) == 2


def test_pack_w4_round_trip_on_int4_grid():
    # every synthetic group has absmax exactly 7 * s, so packing is lossless
    q, s = synth.w4_grid(14, "pin4", 48, 384)
    assert np.abs(q).max() == 7
    q2, s2 = O.pack_w4a16(synth.w4_float(q, s))
    assert np.array_equal(q2, q)
    assert np.array_equal(s2.view(np.uint16), s.view(np.uint16))


def test_pack_w4_error_bound_and_range():
    rng = np.random.default_rng(5)
    w = (rng.standard_normal((64, 384)) * rng.lognormal(-2, 1, (64, 1))).astype(np.float32)
    w[3, 128:256] = 0.0  # an all-zero group
    q, s = O.pack_w4a16(w)
    assert s.shape == (64, 3)
    assert np.all(np.abs(q.astype(np.int32)) <= 7)
    assert s[3, 1] == 0 and not q[3, 128:256].any()
    sg = np.repeat(s.astype(np.float32), 128, axis=1)
    nz = sg > 0
    err = np.abs(w.astype(np.float64) - O.dequant_w4(q, s))
    assert np.all(err[nz] <= sg[nz] * (0.5 + 1e-6) + 1e-30)
    # each group's maximum maps to +-7 (or +-6 after fp16 rounding of s up)
    g = np.abs(q.reshape(64, 3, 128)).max(axis=2)
    assert np.all(g[s > 0] >= 6)


def test_pack_w4_negative_control(monkeypatch):
    # one scale per row instead of per group loses the small groups' precision
    rng = np.random.default_rng(6)
    w = rng.standard_normal((8, 256)).astype(np.float32)
    w[:, 128:] *= 1e-3
    q, s = O.pack_w4a16(w)
    ok = np.abs(w.astype(np.float64) - O.dequant_w4(q, s))
    s_row = np.repeat(s.max(axis=1, keepdims=True), 2, axis=1)
    bad = np.abs(w.astype(np.float64) - O.dequant_w4(np.clip(np.rint(
        w / np.repeat(s_row.astype(np.float32), 128, axis=1)), -7, 7).astype(np.int8), s_row))
    assert np.max(bad[:, 128:]) > 5 * np.max(ok[:, 128:])


def test_linear_orientation():
    # a single nonzero weight q[n0][k0] routes input channel k0 to output n0
    x = np.arange(1, 13, dtype=np.float64).reshape(2, 6)
    q = np.zeros((4, 6), np.int8)
    q[2, 5] = 3
    s = np.ones(4, np.float16)
    y = O.linear(x, O.dequant_w8(q, s))
    assert y.shape == (2, 4)
    assert np.array_equal(y[:, 2], 3 * x[:, 5])
    assert np.count_nonzero(y[:, [0, 1, 3]]) == 0


# ---------------------------------------------------------------- norms -----
def test_rmsnorm_unit_rms_and_eps():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((7, 96)) * 3.0
    y = O.rmsnorm(x, np.ones(96), 0.0)
    assert np.allclose(np.sqrt(np.mean(y * y, axis=1)), 1.0, rtol=1e-12)
    eps = 0.5
    ms = np.mean(x * x, axis=1)
    y = O.rmsnorm(x, np.ones(96), eps)
    assert np.allclose(np.sqrt(np.mean(y * y, axis=1)), np.sqrt(ms / (ms + eps)), rtol=1e-12)
    g = rng.standard_normal(96)
    assert np.allclose(O.rmsnorm(x, g, 0.0), O.rmsnorm(x, np.ones(96), 0.0) * g)


def test_head_norm_is_per_head():
    # per-head norm over d values: each head vector has RMS 1 before gamma
    rng = np.random.default_rng(6)
    nh, d = 8, 128
    x = rng.standard_normal((5, nh, d)) * rng.lognormal(0, 2, (1, nh, 1))
    y = O.head_rmsnorm(x, np.ones(d), 0.0)
    assert np.allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, rtol=1e-12)
    # negative control: a global norm over all channels fails the per-head
    # check (the ANE bug the mirror-sd README describes in Phase 2)
    g = O.rmsnorm(x.reshape(5, nh * d), np.ones(nh * d), 0.0).reshape(5, nh, d)
    rms = np.sqrt(np.mean(g * g, axis=-1))
    assert not np.allclose(rms, 1.0, rtol=1e-2)


# ----------------------------------------------------------------- rope -----
@pytest.mark.parametrize("d", [64, 128])
def test_rope_identity_at_zero_and_norm(d):
    rng = np.random.default_rng(7)
    x = rng.standard_normal((9, 4, d))
    assert np.array_equal(O.rope_neox(x, np.zeros((9, 1)), 1e6), x)
    pos = rng.integers(0, 10000, (9, 1))
    y = O.rope_neox(x, pos, 1e6)
    assert np.allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-12)


def test_rope_relative_position():
    rng = np.random.default_rng(8)
    d = 128
    q, k = rng.standard_normal(d), rng.standard_normal(d)
    for p, pp in [(37, 5), (4096, 4000), (8191, 1)]:
        lhs = O.rope_neox(q, p, 1e6) @ O.rope_neox(k, pp, 1e6)
        rhs = O.rope_neox(q, p - pp, 1e6) @ k
        assert abs(lhs - rhs) < 1e-9 * (1 + abs(rhs))


def test_rope_split_half_convention_and_frequencies():
    # neox split-half: element i pairs with i + d/2 (mirror-sd "The Story",
    # Phase 3), not with i + 1 as in the interleaved form.
    d = 128
    e0 = np.zeros(d)
    e0[0] = 1.0
    y = O.rope_neox(e0, 1.0, 10000.0)
    # pair 0 has frequency theta^0 = 1: turns by exactly pos radians
    assert abs(y[0] - 0.5403023058681397174) < 1e-15
    assert abs(y[d // 2] - 0.84147098480789650665) < 1e-15
    assert np.count_nonzero(np.abs(y) > 1e-15) == 2 and abs(y[1]) == 0
    y5 = O.rope_neox(e0, 5.0, 10000.0)
    assert abs(y5[0] - 0.28366218546322626447) < 1e-14
    assert abs(y5[d // 2] + 0.95892427466313846889) < 1e-14
    # pair i turns by pos * theta^(-2i/d); literals are that closed form
    # evaluated to 20 digits (RoFormer frequencies; base 1e4 and 1e6)
    table = {(10000.0, 128, 1): 0.86596432336006535235,
             (10000.0, 128, 2): 0.7498942093324558273,
             (10000.0, 128, 63): 0.00011547819846894581797,
             (1e6, 128, 1): 0.805842187761481817,
             (1e6, 128, 63): 1.2409377607517195661e-6,
             (1e6, 64, 1): 0.64938163157621131513,
             (1e6, 64, 31): 1.5399265260594919896e-6}
    for (theta, dd, i), f in table.items():
        e = np.zeros(dd)
        e[i] = 1.0
        y = O.rope_neox(e, 1.0, theta)
        ang = math.atan2(y[i + dd // 2], y[i])
        assert abs(ang - f) < 1e-15 * max(1.0, f) + 1e-18, (theta, dd, i)


# ------------------------------------------------------------ attention -----
def test_attention_closed_forms():
    rng = np.random.default_rng(9)
    T, nq, nkv, d, S = 6, 8, 2, 64, 11
    q = rng.standard_normal((T, nq, d))
    k = np.repeat(rng.standard_normal((1, nkv, d)), S, axis=0)  # all keys equal
    v = rng.standard_normal((S, nkv, d))
    o = O.attention_gqa(q, k, v)
    for h in range(nq):
        assert np.allclose(o[:, h], v[:, h // 4].mean(axis=0)[None], rtol=1e-12)
    o1 = O.attention_gqa(q, k[:1], v[:1])  # one key: output is that value
    for h in range(nq):
        assert np.allclose(o1[:, h], v[0, h // 4][None], rtol=1e-12)


def test_attention_gqa_head_mapping():
    # kv heads carry distinct constant values: q head h must read h // (nq/nkv)
    T, nq, nkv, d, S = 3, 8, 4, 16, 5
    rng = np.random.default_rng(10)
    q = rng.standard_normal((T, nq, d))
    k = rng.standard_normal((S, nkv, d))
    v = np.zeros((S, nkv, d))
    for g in range(nkv):
        v[:, g, :] = 10.0 * g + 1.0
    o = O.attention_gqa(q, k, v)
    for h in range(nq):
        assert np.allclose(o[:, h, :], 10.0 * (h // 2) + 1.0)


def test_attention_matches_torch_sdpa_float64():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(11)
    T, nq, nkv, d, S = 16, 8, 2, 64, 80
    q = rng.standard_normal((T, nq, d))
    k = rng.standard_normal((S, nkv, d))
    v = rng.standard_normal((S, nkv, d))
    o = O.attention_gqa(q, k, v)
    tq = torch.from_numpy(q).permute(1, 0, 2)[None]
    tk = torch.from_numpy(np.repeat(k, nq // nkv, axis=1)).permute(1, 0, 2)[None]
    tv = torch.from_numpy(np.repeat(v, nq // nkv, axis=1)).permute(1, 0, 2)[None]
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv)[0].permute(1, 0, 2).numpy()
    assert np.allclose(o, ref, rtol=1e-12, atol=1e-12)


def test_silu_closed_forms():
    z = np.array([-50.0, -3.0, 0.0, 2.5, 60.0])
    s = O.silu(z)
    assert s[2] == 0.0
    assert abs(s[0]) < 1e-19 and abs(s[4] - 60.0) < 1e-20
    # silu(z) - silu(-z) = z for all z
    assert np.allclose(O.silu(z) - O.silu(-z), z, rtol=1e-14, atol=1e-14)


# --------------------------------------------------------------- accept -----
def test_accept_golden_cases():
    with open(os.path.join(GOLDEN, "accept_cases.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        a = np.asarray(c["a"])
        V = int(a.max()) + 3
        logits = np.zeros((len(a), V), np.float32)
        logits[np.arange(len(a)), a] = 1.0
        n, corr, emitted, nt = O.verify_accept(logits, np.asarray(c["draft"]))
        assert (n, corr, list(emitted), nt) == (c["n"], c["corr"], c["emitted"], c["next_tok"]), c


def _brute_accept(a, draft, R):
    # longest prefix by enumeration: the largest k with all of draft[:k] == a[:k]
    best = 0
    for k in range(len(draft) + 1):
        if all(draft[i] == a[i] for i in range(k)):
            best = k
    corr = a[best] if best < R else -1
    return best, corr


@pytest.mark.parametrize("R", [1, 2, 3, 4, 5])
def test_accept_brute_force_tiny_vocab(R):
    import itertools
    V = 3
    for a in itertools.product(range(V), repeat=R):
        logits = np.full((R, V), -1.0, np.float32)
        logits[np.arange(R), a] = 2.0
        for Dn in {R - 1, R} - {0}:
            for dr in itertools.product(range(V), repeat=Dn):
                n, corr, emitted, nt = O.verify_accept(logits, np.asarray(dr))
                bn, bc = _brute_accept(a, dr, R)
                assert (n, corr) == (bn, bc)
                exp = list(dr[:bn]) + ([bc] if bc >= 0 else [])
                assert list(emitted[:len(exp)]) == exp
                assert all(e == -1 for e in emitted[len(exp):])


def test_argmax_ties_go_to_lowest_index():
    lg = np.array([[0.0, 3.0, 1.0, 3.0], [5.0, 5.0, 5.0, 5.0]], np.float32)
    assert list(O.argmax_lowest(lg)) == [1, 0]
    n, corr, _, _ = O.verify_accept(lg, np.array([3]))
    assert (n, corr) == (0, 1)


def test_accept_planted_synthetic_logits():
    # the generator's planting: draft == target argmax on rows < n, not at n
    b, R, V = 6, 16, 4096
    draft = synth.tokens(1, "pin", b * (R - 1), V).reshape(b, R - 1)
    n_acc = np.array([0, 1, 5, 14, 15, 7])
    lg = synth.verify_logits(1, "pin", draft, R, V, n_acc)
    for j in range(b):
        n, corr, emitted, nt = O.verify_accept(lg[j], draft[j])
        assert n == n_acc[j]
        assert corr == int(np.argmax(lg[j, n]))
        assert nt == corr


# -------------------------------------------------------- generator pins -----
def test_truncated_geometric_means():
    for mean, D in [(6.0, 15), (17.0, 31)]:
        r = synth.truncated_geometric_ratio(mean, D)
        n = np.arange(D + 1)
        p = r ** n / (r ** n).sum()
        assert abs((n * p).sum() - mean) < 1e-9
    assert synth.truncated_geometric_ratio(17.0, 31) > 1.0  # above midpoint


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 3.0e-3], np.float32)
    u = synth.f32_to_bf16_bits(x)
    back = synth.bf16_bits_to_f32(u)
    assert back[0] == 1.0 and back[1] == 1.0  # tie to even (down)
    assert back[2] == 1.0 + 4 * 2 ** -8        # tie to even (up)
    assert back[3] == -2.5
    assert abs(back[4] - 3.0e-3) <= 3.0e-3 * 2 ** -8
