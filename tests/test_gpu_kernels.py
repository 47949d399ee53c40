"""GPU parity of each kernel against the oracle, through the C ABI.

Tolerances: bit-exact for integer work (packed codes, argmax indices,
accept lengths and tokens); the W8A16 GEMM alone within 1e-3 of the output's
max-abs (fp16 activations x exact int8 with fp32 accumulation against a
float64 oracle on the same fp16 inputs); draft argmax compared only where the
oracle's top-2 margin exceeds 1e-2.
"""
import numpy as np
import pytest

from oracle import dflash_oracle as O
from block_diffusion_speculative_draft_gb300 import synth
from tests.gpu_util import gpu_available, rel_err, unpack_tiled_q

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not gpu_available(), reason="needs a GPU")]

if gpu_available():
    import torch
    from block_diffusion_speculative_draft_gb300 import api
    DEV = torch.device("cuda:0")


# ------------------------------------------------------------------ pack ----
@pytest.mark.parametrize("N,K,layout,dtype", [
    (128, 128, 0, "f32"), (256, 512, 0, "f16"), (384, 256, 0, "bf16"), (256, 384, 1, "f32"), (768, 512, 0, "f32")])
def test_pack_bit_exact(N, K, layout, dtype):
    rng = np.random.default_rng(N + K)
    w = (rng.standard_normal((N, K)) * rng.lognormal(-3, 1, (N, 1))).astype(np.float32)
    w[3] = 0.0
    if dtype == "f16":
        w = w.astype(np.float16)
        tw = torch.from_numpy(w).to(DEV)
        w = w.astype(np.float32)
    elif dtype == "bf16":
        bits = synth.f32_to_bf16_bits(w)
        w = synth.bf16_bits_to_f32(bits)
        tw = torch.from_numpy(w).to(DEV).to(torch.bfloat16)
    else:
        tw = torch.from_numpy(w).to(DEV)
    qd, sd = api.dflash_pack_w8a16(tw, layout)
    torch.cuda.synchronize()
    q_ref, s_ref = O.pack_w8a16(w)
    assert np.array_equal(sd.cpu().numpy().view(np.uint16), s_ref.view(np.uint16))
    q = unpack_tiled_q(qd.cpu().numpy(), N, K, layout)
    assert np.array_equal(q, q_ref)


# ------------------------------------------------------------------ K1 ------
@pytest.mark.parametrize("M,N,K,layout", [
    (16, 768, 512, 0), (16, 512, 1536, 0), (15, 3072, 512, 1), (5, 256, 256, 0), (32, 1024, 2560, 0),
    (17, 384, 640, 0), (128, 512, 1024, 0), (1, 128, 128, 0), (40, 640, 384, 1), (64, 768, 512, 0),
    (100, 640, 2560, 1), (300, 512, 768, 0), (33, 128, 4096, 0),
    # one split over a long K: every ring slot and A buffer cycles several times
    (64, 19584, 1024, 0), (32, 19584, 1024, 0), (128, 19584, 1024, 1),
    # 32 rows of a projection large enough for the tensor-memory kernel
    (32, 20480, 2560, 0), (31, 20480, 2560, 1)])
def test_w8a16_linear(M, N, K, layout):
    q, s = synth.w8_grid(5, f"lin{M}{N}{K}", N, K)
    x = synth.target_hidden(5, f"x{M}{K}", M, K)
    qd, sd = api.dflash_pack_w8a16(torch.from_numpy(synth.w8_float(q, s)).to(DEV), layout)
    desc = api.w8_desc(qd, sd, N, K, layout)
    y = api.dflash_w8a16_linear(desc, torch.from_numpy(x).to(DEV)).cpu().numpy()
    ref = O.linear(x.astype(np.float64), O.dequant_w8(q, s))
    assert rel_err(y, ref) <= 1e-3


# ------------------------------------------------------------------ K4 ------
@pytest.mark.parametrize("M,V,H", [(15, 4096, 512), (16, 5000, 256), (31, 9000, 640), (1, 300, 64),
                                   (120, 2048, 512), (33, 1027, 128)])
def test_lmhead_argmax(M, V, H):
    hb = synth.bf16_rows(7, f"h{M}", M, H)
    wb = synth.bf16_table(7, f"w{V}{H}", V, H)
    idx = torch.empty(M, dtype=torch.int32, device=DEV)
    mx = torch.empty(M, dtype=torch.float32, device=DEV)
    lg = torch.empty((M, V), dtype=torch.float32, device=DEV)
    th = torch.from_numpy(hb.view(np.int16)).to(DEV)
    tw = torch.from_numpy(wb.view(np.int16)).to(DEV)
    for _ in range(2):  # second call checks the workspace re-zeroing
        api.dflash_lmhead_argmax(th, tw, idx, mx, lg)
    torch.cuda.synchronize()
    ridx, rmax, margin, rlg = O.lmhead_argmax(hb, wb)
    ok = margin > 1e-2
    assert ok.sum() >= M // 2
    assert np.array_equal(idx.cpu().numpy()[ok], ridx[ok])
    assert rel_err(lg.cpu().numpy(), rlg) <= 1e-4
    assert np.allclose(mx.cpu().numpy(), rmax, rtol=1e-4, atol=1e-4)


def test_lmhead_ties_lowest_index():
    H, V, M = 64, 1000, 3
    hb = synth.f32_to_bf16_bits(np.ones((M, H), np.float32))
    w = np.zeros((V, H), np.float32)
    w[[7, 300, 999], :] = 0.5   # equal maxima: lowest index wins
    w[500, :] = -1.0
    wb = synth.f32_to_bf16_bits(w)
    idx = api.dflash_lmhead_argmax(torch.from_numpy(hb.view(np.int16)).to(DEV),
                                   torch.from_numpy(wb.view(np.int16)).to(DEV))
    assert idx.cpu().numpy().tolist() == [7, 7, 7]


# ------------------------------------------------------------------ K5 ------
@pytest.mark.parametrize("b,R,D,V", [(1, 16, 16, 4096), (1, 16, 15, 151936), (1, 32, 31, 151936),
                                     (8, 16, 15, 151936), (3, 5, 4, 4093), (2, 1, 1, 17), (4, 8, 8, 1000)])
def test_verify_accept_bit_exact(b, R, D, V):
    draft = synth.tokens(9, f"d{b}{R}", b * D, V).reshape(b, D)
    nacc = synth.accept_lengths(9, f"n{b}{R}", b, D)
    lg = synth.verify_logits(9, f"l{b}{R}{V}", draft, R, V, nacc)
    n_out = torch.empty(b, dtype=torch.int32, device=DEV)
    corr = torch.empty(b, dtype=torch.int32, device=DEV)
    emitted = torch.empty((b, R), dtype=torch.int32, device=DEV)
    nxt = torch.empty(b, dtype=torch.int32, device=DEV)
    tl, td = torch.from_numpy(lg).to(DEV), torch.from_numpy(draft).to(DEV)
    for _ in range(2):
        api.dflash_verify_accept(tl, td, n_out, corr, emitted, nxt)
    torch.cuda.synchronize()
    for j in range(b):
        n, c, e, nt = O.verify_accept(lg[j], draft[j])
        assert int(n_out[j]) == n == min(int(nacc[j]), D)
        assert int(corr[j]) == c and int(nxt[j]) == nt
        assert np.array_equal(emitted[j].cpu().numpy(), e)


def test_verify_accept_ties_and_golden():
    import json, os
    with open(os.path.join(os.path.dirname(__file__), "golden", "accept_cases.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        a = np.asarray(c["a"])
        R, V = len(a), 16
        lg = np.zeros((1, R, V), np.float32)
        lg[0, np.arange(R), a] = 1.0
        lg[0, :, V - 1] = 1.0  # a tie at a higher index must lose
        dr = np.asarray(c["draft"], np.int32)[None]
        n_out = torch.empty(1, dtype=torch.int32, device=DEV)
        corr = torch.empty(1, dtype=torch.int32, device=DEV)
        emitted = torch.empty((1, R), dtype=torch.int32, device=DEV)
        nxt = torch.empty(1, dtype=torch.int32, device=DEV)
        api.dflash_verify_accept(torch.from_numpy(lg).to(DEV), torch.from_numpy(dr).to(DEV), n_out, corr,
                                 emitted, nxt)
        assert (int(n_out[0]), int(corr[0]), emitted[0].cpu().tolist(), int(nxt[0])) == \
            (c["n"], c["corr"], c["emitted"], c["next_tok"]), c
