"""Pins for the oracle's temperature speculative-sampling accept.

The pages fix the property — with temperature T > 0 every emitted token is an
exact sample from the target at T (mlx-dspark v0.0.3 release notes,
"Highlights") — so the pins test that property by counting: emitted tokens of
many seeded draws must follow softmax(logits / T) (chi-square), a sampler with
a wrong residual must fail the same count, and T -> 0 must reduce to the
greedy rule.
"""
import numpy as np

from oracle import dflash_oracle as O

# 99.9 % quantiles of chi-square with k - 1 degrees of freedom
CHI2_999 = {4: 18.47, 5: 20.52, 7: 24.32}


def _uniforms(rng, shape):
    # odd multiples of 2^-24: exact in fp32, never 0 or 1
    k = rng.integers(0, 1 << 23, size=shape)
    return ((2 * k + 1) * 2.0 ** -24).astype(np.float32)


def _chi2(counts, p):
    n = counts.sum()
    e = n * p
    return float(((counts - e) ** 2 / e).sum())


def _draws(z, draft, T, N, seed, exclude=True):
    rng = np.random.default_rng(seed)
    R, V = z.shape
    first = np.zeros(V, dtype=np.int64)
    second = np.zeros(V, dtype=np.int64)
    for _ in range(N):
        u_acc = _uniforms(rng, len(draft))
        u_s = _uniforms(rng, V)
        n, corr, em, _, _ = O.verify_accept_sample(z, draft, T, u_acc, u_s, exclude_rejected=exclude)
        first[em[0]] += 1
        if n >= 1:  # draft[0] accepted: the next token is a draw from p_1
            second[em[1]] += 1
    return first, second


def _case():
    rng = np.random.default_rng(7)
    z = rng.normal(0, 1.5, size=(3, 5)).astype(np.float32)
    draft = np.array([int(np.argsort(z[0])[-2]), int(np.argmax(z[1]))])  # x_0 is not the mode
    return z, draft


def test_emitted_tokens_follow_the_target_at_temperature():
    z, draft = _case()
    T = 0.8
    first, second = _draws(z, draft, T, 20000, seed=11)
    assert _chi2(first, O.softmax_t(z[0], T)) < CHI2_999[4]
    assert second.sum() > 2000
    assert _chi2(second, O.softmax_t(z[1], T)) < CHI2_999[4]


def test_residual_that_keeps_the_rejected_token_is_caught():
    # negative control: resampling from p_n itself (x_n not removed) over-weights
    # x_n, and the same count rejects it
    z, draft = _case()
    T = 0.8
    first, _ = _draws(z, draft, T, 20000, seed=11, exclude=False)
    assert _chi2(first, O.softmax_t(z[0], T)) > 10 * CHI2_999[4]


def test_bonus_row_after_full_accept_follows_p_D():
    rng = np.random.default_rng(3)
    z = rng.normal(0, 1.0, size=(2, 6)).astype(np.float32)
    draft = np.array([int(np.argmax(z[0]))])
    z[0, draft[0]] += 6.0  # accept almost always
    T = 1.3
    counts = np.zeros(6, dtype=np.int64)
    g = np.random.default_rng(5)
    for _ in range(12000):
        n, corr, em, _, d = O.verify_accept_sample(z, draft, T, _uniforms(g, 1), _uniforms(g, 6))
        if n == 1:
            assert d["row"] == 1
            counts[corr] += 1
    assert counts.sum() > 11000
    assert _chi2(counts, O.softmax_t(z[1], T)) < CHI2_999[5]


def test_gumbel_max_frequencies():
    z = np.array([0.3, -1.0, 2.0, 0.0, 1.1, -0.4, 0.9, 0.2], dtype=np.float32)
    T = 0.9
    g = np.random.default_rng(17)
    counts = np.zeros(8, dtype=np.int64)
    for _ in range(20000):
        counts[int(np.argmax(O.gumbel_scores(z, T, _uniforms(g, 8))))] += 1
    assert _chi2(counts, O.softmax_t(z, T)) < CHI2_999[7]


def test_zero_temperature_limit_is_the_greedy_rule():
    rng = np.random.default_rng(23)
    for trial in range(40):
        R, V = 6, 40
        z = rng.normal(0, 1, size=(R, V)).astype(np.float32)
        a = np.argmax(z, axis=1)
        k = int(rng.integers(0, R))
        draft = a[: R - 1].copy()
        if k < R - 1:
            draft[k] = (a[k] + 1 + int(rng.integers(0, V - 1))) % V
        srt = np.sort(z, axis=1)
        if np.min(srt[:, -1] - srt[:, -2]) < 0.05:
            continue
        g = np.random.default_rng(trial)
        got = O.verify_accept_sample(z, draft, 1e-3, _uniforms(g, R - 1), _uniforms(g, V))
        ref = O.verify_accept(z, draft)
        assert got[0] == ref[0] and got[1] == ref[1]
        assert np.array_equal(got[2], ref[2]) and got[3] == ref[3]


def test_full_accept_without_a_bonus_row():
    z = np.zeros((2, 4), dtype=np.float32)
    z[0, 1] = z[1, 3] = 30.0
    n, corr, em, nxt, d = O.verify_accept_sample(z, np.array([1, 3]), 1.0, np.full(2, 0.5, np.float32),
                                                 np.full(4, 0.5, np.float32))
    assert (n, corr, nxt, d["row"]) == (2, -1, 3, -1)
    assert em.tolist() == [1, 3]
