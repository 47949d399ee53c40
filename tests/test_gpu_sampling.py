"""GPU temperature speculative-sampling accept through the C ABI.

Parity with the oracle: accept lengths, correction tokens and emitted rows
are compared exactly wherever the decisions have a margin (|u - p| > 1e-4
for every accept test taken, top-2 Gumbel score gap > 1e-3 for the draw —
the kernel decides in fp32, the oracle's accept probabilities are float64);
inside a margin the GPU's choice must still be a valid one.  Exactness of
the GPU sampler itself is checked by counting over thousands of sequences,
and T -> 0 must reproduce the greedy kernel.
"""
import numpy as np
import pytest

from oracle import dflash_oracle as O
from tests.gpu_util import gpu_available

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not gpu_available(), reason="needs a GPU")]

if gpu_available():
    import torch
    from block_diffusion_speculative_draft_gb300 import api
    DEV = torch.device("cuda:0")

CHI2_999 = {4: 18.47, 5: 20.52}


def _uniforms(rng, shape):
    k = rng.integers(0, 1 << 23, size=shape)
    return ((2 * k + 1) * 2.0 ** -24).astype(np.float32)


def _run(lg, draft, T, ua, us):
    b, R, V = lg.shape
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    n = torch.empty(b, dtype=torch.int32, device=DEV)
    c = torch.empty(b, dtype=torch.int32, device=DEV)
    em = torch.empty((b, R), dtype=torch.int32, device=DEV)
    nx = torch.empty(b, dtype=torch.int32, device=DEV)
    api.dflash_verify_accept_sample(t(lg), t(draft), T, t(ua), t(us), n, c, em, nx)
    torch.cuda.synchronize()
    assert api.dflash_get_status() == 0
    return n.cpu().numpy(), c.cpu().numpy(), em.cpu().numpy(), nx.cpu().numpy()


def _case(seed, b, R, V, scale=3.0):
    rng = np.random.default_rng(seed)
    lg = rng.normal(0, scale, size=(b, R, V)).astype(np.float32)
    a = lg.argmax(axis=2)
    draft = a[:, : R - 1].astype(np.int32).copy()
    # lift the draft tokens so acceptance is likely but not certain
    for j in range(b):
        for i in range(R - 1):
            lg[j, i, draft[j, i]] += float(rng.uniform(0, 4))
        k = int(rng.integers(0, R))
        if k < R - 1:
            draft[j, k] = (draft[j, k] + 1 + int(rng.integers(0, V - 1))) % V
    return rng, lg, draft


@pytest.mark.parametrize("b,V,T", [(6, 4096, 0.6), (6, 4096, 1.0), (4, 4096, 2.5), (2, 151936, 0.8)])
def test_sample_accept_matches_the_oracle(b, V, T):
    R = 16
    rng, lg, draft = _case(100 + V + b, b, R, V)
    ua = _uniforms(rng, (b, R - 1))
    us = _uniforms(rng, (b, V))
    n, c, em, nx = _run(lg, draft, T, ua, us)
    compared = 0
    for j in range(b):
        rn, rc, rem, rnx, d = O.verify_accept_sample(lg[j], draft[j], T, ua[j], us[j])
        taken = np.abs(d["u_minus_p"][: min(rn + 1, R - 1)])
        if np.all(taken > 1e-4):
            assert n[j] == rn
            if rc < 0:
                assert c[j] == -1
            elif d["score_gap"] > 1e-3:
                assert c[j] == rc and np.array_equal(em[j], rem) and nx[j] == rnx
                compared += 1
            else:  # a near tie in fp32: any top-scoring token is a valid draw
                sc = O.gumbel_scores(lg[j, d["row"]], T, us[j]).astype(np.float64)
                if rn < R - 1:
                    assert c[j] != draft[j, rn]
                    sc[draft[j, rn]] = -np.inf
                assert sc[c[j]] >= sc.max() - 1e-3
    assert compared >= b // 2


def test_gpu_sampler_is_exact_by_counting():
    # thousands of sequences with the same target rows: emitted tokens must
    # follow softmax(z / T) (first token always; second when the first draft
    # was accepted)
    rng = np.random.default_rng(41)
    b, R, V, T = 8192, 3, 5, 0.9
    z = rng.normal(0, 1.2, size=(R, V)).astype(np.float32)
    x0 = int(np.argsort(z[0])[-2])
    x1 = int(np.argmax(z[1]))
    lg = np.broadcast_to(z, (b, R, V)).copy()
    draft = np.tile(np.array([x0, x1], dtype=np.int32), (b, 1))
    ua = _uniforms(rng, (b, 2))
    us = _uniforms(rng, (b, V))
    n, c, em, _ = _run(lg, draft, T, ua, us)

    def chi2(counts, p):
        e = counts.sum() * p
        return float(((counts - e) ** 2 / e).sum())

    first = np.bincount(em[:, 0], minlength=V)
    assert chi2(first, O.softmax_t(z[0], T)) < CHI2_999[4]
    acc = n >= 1
    second = np.bincount(em[acc, 1], minlength=V)
    assert second.sum() > 1000
    assert chi2(second, O.softmax_t(z[1], T)) < CHI2_999[4]


def test_low_temperature_is_the_greedy_kernel():
    b, R, V = 4, 16, 151936
    rng, lg, draft = _case(7, b, R, V, scale=1.0)
    # make every row's maximum unique by a clear gap
    top = lg.argmax(axis=2)
    for j in range(b):
        for r in range(R):
            lg[j, r, top[j, r]] += 1.0
    ua = _uniforms(rng, (b, R - 1))
    us = _uniforms(rng, (b, V))
    n, c, em, nx = _run(lg, draft, 1e-3, ua, us)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    gn = torch.empty(b, dtype=torch.int32, device=DEV)
    gc = torch.empty(b, dtype=torch.int32, device=DEV)
    gem = torch.empty((b, R), dtype=torch.int32, device=DEV)
    gnx = torch.empty(b, dtype=torch.int32, device=DEV)
    api.dflash_verify_accept(t(lg), t(draft), gn, gc, gem, gnx)
    torch.cuda.synchronize()
    assert np.array_equal(n, gn.cpu().numpy()) and np.array_equal(c, gc.cpu().numpy())
    assert np.array_equal(em, gem.cpu().numpy()) and np.array_equal(nx, gnx.cpu().numpy())


def test_draft_token_outside_the_vocabulary_is_rejected():
    b, R, V = 2, 4, 1000
    rng, lg, draft = _case(9, b, R, V)
    for j in range(b):
        for i in range(R - 1):
            lg[j, i, draft[j, i]] += 50.0  # certain accept
    draft[0, 1] = V + 7
    draft[1, 0] = -3
    n, c, em, _ = _run(lg, draft, 1.0, _uniforms(rng, (b, R - 1)), _uniforms(rng, (b, V)))
    assert n.tolist() == [1, 0]
    assert 0 <= c[0] < V and 0 <= c[1] < V
