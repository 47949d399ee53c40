"""Host-side logic that the GPU runs depend on, checked on the CPU: the
algorithmic byte counts the roofline divides by, the stand-in target's row
chunks, and the test helper that decodes packed int4 tiles (so that the GPU
packer's bit-exact test compares against a correct reading of the layout)."""
import numpy as np

from oracle import dflash_oracle as O
from block_diffusion_speculative_draft_gb300.configs import QWEN3_4B, TINY, ALL
from block_diffusion_speculative_draft_gb300 import workload as WL
from tests.gpu_util import unpack_tiled_q, unpack_tiled_q4


def test_step_bytes_by_hand():
    c = QWEN3_4B
    # per layer: q|k|v (32 + 2 * 8 heads of 128) x 2560, o 2560 x 4096,
    # gate|up 2 * 9728 x 2560, down 2560 x 9728, one byte per int8 weight
    per_layer = 2560 * 6144 + 2560 * 4096 + 2 * 9728 * 2560 + 2560 * 9728
    weights = 5 * per_layer
    scales = 2 * 5 * (6144 + 2560 + 2 * 9728 + 2560)
    lm = 2 * 151936 * 2560
    kv = 5 * 512 * 8 * 128 * 2 * 2
    assert c.step_bytes([512]) == weights + scales + lm + kv == 1293332480
    assert c.step_bytes_w4([512]) == weights // 2 + weights // 64 + lm + kv == 1048596480


def test_standin_chunks_cover_the_vocabulary():
    for cfg in ALL:
        ch = WL.standin_chunks(cfg)
        assert ch[0][0] == 0 and ch[-1][1] == cfg.V
        assert all(a[1] == b[0] for a, b in zip(ch, ch[1:]))
        assert all((r1 - r0) % 128 == 0 and r1 - r0 <= WL.STANDIN_CHUNK for r0, r1 in ch)
    assert WL.standin_chunks(TINY) == [(0, 4096)]


def _pack4_by_element(q, s, layout):
    """The packed int4 layout written element by element: tile (nt, kt) of
    8448 bytes; lane chunk (warp w, k-step ks, lane l) at 8 (256 w + 32 ks + l)
    holds two words, word f for m-group 2w + f; nibble k of a word is element
    (row g + 8 (k & 1), column 2t + (k >> 2) + 8 ((k >> 1) & 1)) of the lane's
    fragment (g = l / 4, t = l % 4), stored as q + 8; the tile's 128 packed
    rows' scales follow at byte 8192."""
    N, K = q.shape
    KT = K // 128
    buf = np.zeros((N // 128) * KT * 8448, np.uint8)

    def lrow(pr):
        if layout != 1:
            return pr
        tl, rr = pr >> 7, pr & 127
        return tl * 64 + rr if rr < 64 else N // 2 + tl * 64 + rr - 64

    for nt in range(N // 128):
        for kt in range(KT):
            base = (nt * KT + kt) * 8448
            for r in range(128):
                buf[base + 8192 + 2 * r:base + 8194 + 2 * r] = np.array([s[lrow(nt * 128 + r), kt]], "<f2").view(np.uint8)
            for w in range(4):
                for ks in range(8):
                    for ln in range(32):
                        g, t = ln // 4, ln % 4
                        words = []
                        for f in range(2):
                            wd = 0
                            for k in range(8):
                                row = lrow(nt * 128 + (2 * w + f) * 16 + g + 8 * (k & 1))
                                col = kt * 128 + ks * 16 + 2 * t + (k >> 2) + 8 * ((k >> 1) & 1)
                                wd |= (int(q[row, col]) + 8) << (4 * k)
                            words.append(wd)
                        off = base + 8 * (256 * w + 32 * ks + ln)
                        buf[off:off + 8] = np.array(words, "<u4").view(np.uint8)
    return buf


def test_int4_tile_decoder_reads_the_layout():
    rng = np.random.default_rng(3)
    w = rng.standard_normal((256, 256)).astype(np.float32)
    q, s = O.pack_w4a16(w)
    for layout in (0, 1):
        q2, s2 = unpack_tiled_q4(_pack4_by_element(q, s, layout), 256, 256, layout)
        assert np.array_equal(q2, q)
        assert np.array_equal(s2.view(np.uint16), s.view(np.uint16))


def _pack8_by_element(q, layout):
    """Byte image of the packed int8 tiles built element by element from the
    layout rule (tile (nt, kt) at (nt K/128 + kt) 16 KB; within the tile,
    column c of packed row r, c = 16 g + j, goes to chunk g ^ (r % 8) of the
    row at byte 4 (j % 8 // 2) + (j % 2) + 2 (j // 8); q + 128)."""
    N, K = q.shape
    KT = K // 128
    buf = np.zeros(N * K, np.uint8)
    for p in range(N):
        nt, r = p // 128, p % 128
        if layout == 1:
            lr = nt * 64 + r if r < 64 else N // 2 + nt * 64 + (r - 64)
        else:
            lr = p
        for c in range(K):
            kt, cc = c // 128, c % 128
            g, j = cc // 16, cc % 16
            byte = 4 * ((j % 8) // 2) + (j % 2) + 2 * (j // 8)
            off = (nt * KT + kt) * 16384 + r * 128 + ((g ^ (r % 8)) * 16) + byte
            buf[off] = (int(q[lr, c]) + 128) & 0xFF
    return buf


def test_int8_tile_decoder_reads_the_layout():
    rng = np.random.default_rng(4)
    q = rng.integers(-127, 128, size=(256, 256)).astype(np.int8)
    for layout in (0, 1):
        assert np.array_equal(unpack_tiled_q(_pack8_by_element(q, layout), 256, 256, layout), q)


def test_float_weights_view_reads_grid_times_scale():
    """The host view handed to DeviceDrafter: matrices read as grid x scale
    (row scales for int8, 128-column group scales for int4), every other entry
    as stored."""
    from block_diffusion_speculative_draft_gb300 import synth
    W8 = synth.drafter_weights(TINY)
    F8 = synth.FloatWeights(W8)
    q, s = W8["o0"]
    w = F8["o0"]
    assert w.dtype == np.float32 and w.shape == q.shape
    r, c = 3, 5
    assert w[r, c] == np.float32(q[r, c]) * np.float32(s[r])
    assert F8["gamma_in"] is W8["gamma_in"] and F8["embed"] is W8["embed"]
    W4 = synth.drafter_weights(TINY, bits=4)
    q4, s4 = W4["down0"]
    w4 = synth.FloatWeights(W4)["down0"]
    assert w4[r, 130] == np.float32(q4[r, 130]) * np.float32(s4[r, 1])
    assert w4[r, 127] == np.float32(q4[r, 127]) * np.float32(s4[r, 0])


def _tiled_attention(s, v, tile=64, thresh=8.0):
    """The tensor-memory attention's per-split loop in float64: scores s
    [rows][keys] in log2 units, a reference maximum raised only when a tile's
    maximum exceeds it by more than `thresh`, O and the sum rescaled only
    then.  Returns the split's normalised output, its log2 log-sum-exp and
    the largest p it formed."""
    rows, keys = s.shape
    mref = np.full(rows, -np.inf)
    lsum = np.zeros(rows)
    o = np.zeros((rows, v.shape[1]))
    pmax = 0.0
    for t0 in range(0, keys, tile):
        st = s[:, t0:t0 + tile]
        mnew = np.maximum(mref, st.max(axis=1))
        resc = np.isfinite(mref) & (mnew - mref > thresh)
        corr = np.where(resc, np.exp2(np.where(resc, mref - mnew, 0.0)), 1.0)
        mref = np.where(~np.isfinite(mref) | resc, mnew, mref)
        o *= corr[:, None]
        lsum *= corr
        p = np.exp2(st - mref[:, None])
        pmax = max(pmax, float(p.max()))
        o += p @ v[t0:t0 + tile]
        lsum += p.sum(axis=1)
    return o / lsum[:, None], mref + np.log2(lsum), pmax


def test_conditional_rescale_softmax_is_softmax():
    """A reference maximum that lags the running maximum by up to 8 (log2
    units) leaves every p <= 2^8 and gives the same normalised attention as
    softmax by definition; the split merge by log-sum-exp weights does too."""
    rng = np.random.default_rng(7)
    rows, keys, d = 40, 6 * 64 + 17, 32
    v = rng.standard_normal((keys, d))
    # scores that climb slowly (the reference stays stale) and then jump
    # (the reference is raised and O rescaled)
    ramp = np.linspace(0.0, 6.0, keys)[None, :]
    jump = np.where(np.arange(keys) >= 4 * 64, 20.0, 0.0)[None, :]
    s = rng.standard_normal((rows, keys)) * 2.0 + ramp + jump
    ref = np.exp2(s - s.max(axis=1, keepdims=True))
    ref = (ref / ref.sum(axis=1, keepdims=True)) @ v
    out, _, pmax = _tiled_attention(s, v)
    assert np.abs(out - ref).max() <= 1e-12 * np.abs(ref).max()
    assert pmax <= 2.0 ** 8
    # without the jump the reference never moves after the first tile
    _, _, pmax2 = _tiled_attention(s - jump, v)
    assert 1.0 < pmax2 <= 2.0 ** 8
    # split the keys in 3 and merge: weights 2^(lse - max lse)
    bounds = [0, 192, 320, keys]
    parts = [_tiled_attention(s[:, a:b], v[a:b]) for a, b in zip(bounds[:-1], bounds[1:])]
    lse = np.stack([p[1] for p in parts])
    w = np.exp2(lse - lse.max(axis=0))
    merged = sum(w[i][:, None] * parts[i][0] for i in range(len(parts))) / w.sum(axis=0)[:, None]
    assert np.abs(merged - ref).max() <= 1e-12 * np.abs(ref).max()
