"""Helpers for the GPU parity tests (test infrastructure)."""
import numpy as np

try:
    import torch
except Exception:  # pragma: no cover
    torch = None


def gpu_available() -> bool:
    return torch is not None and torch.cuda.is_available()


def unpack_tiled_q(qbytes: np.ndarray, N: int, K: int, layout: int = 0) -> np.ndarray:
    """Restates the packed int8 layout of include/dflash.h's packer to recover
    the logical q[N][K]: 128x128 tiles in (row-tile, k-tile) order, each
    [packed row 128][128 bytes]; the 16 columns of group g of row r sit in the
    16-byte chunk at r*128 + (g ^ (r % 8))*16, whose bytes 4t..4t+3 hold
    columns 2t, 2t+1, 2t+8, 2t+9 of the group; bytes are q + 128.  Packed row
    p of a gate|up matrix is logical row (p // 128)*64 + p % 128 for
    p % 128 < 64, else N/2 + (p // 128)*64 + p % 128 - 64."""
    KT = K // 128
    t = qbytes.reshape(N // 128, KT, 128, 8, 16).astype(np.int16) - 128
    r = np.arange(128)
    e = np.arange(16)
    col_of_byte = 2 * (e >> 2) + (e & 1) + ((e >> 1) & 1) * 8
    q = np.empty((N, K), np.int8)
    for nt in range(N // 128):
        pr = nt * 128 + r
        if layout == 1:
            tl, rr = pr >> 7, pr & 127
            lr = np.where(rr < 64, tl * 64 + rr, N // 2 + tl * 64 + (rr - 64))
        else:
            lr = pr
        for kt in range(KT):
            for g in range(8):
                slot = g ^ (r & 7)
                chunk = t[nt, kt, r, slot, :]  # [128][16] bytes of group g
                q[lr[:, None], kt * 128 + g * 16 + col_of_byte[None, :]] = chunk
    return q


def rel_err(got, ref) -> float:
    ref = np.asarray(ref, np.float64)
    return float(np.abs(np.asarray(got, np.float64) - ref).max() / max(np.abs(ref).max(), 1e-30))


def unpack_tiled_q4(qbytes: np.ndarray, N: int, K: int, layout: int = 0):
    """Restates the packed int4 layout of include/dflash.h's packer: 128x128
    tiles of 8448 bytes in (row-tile, k-tile) order; bytes [0, 8192) are
    [warp 4][k16 step 8][lane 32][two 32-bit fragment words], nibble k of a
    word = element (row g + 8 (k & 1), column 2t + (k >> 2) + 8 ((k >> 1) & 1))
    of the lane's m16k16 fragment, stored as q + 8; bytes [8192, 8448) are the
    fp16 scales of the tile's 128 packed rows for its column group.  Returns
    the logical q[N][K] (int8) and the in-tile scales s[N][K/128] (fp16)."""
    KT = K // 128
    t = qbytes.reshape(N // 128, KT, 8448)
    words = np.ascontiguousarray(t[:, :, :8192]).view("<u4").reshape(N // 128, KT, 4, 8, 32, 2)
    sc = np.ascontiguousarray(t[:, :, 8192:]).view("<f2").reshape(N // 128, KT, 128)
    q = np.empty((N, K), np.int8)
    s = np.empty((N, KT), np.float16)
    lane = np.arange(32)
    g, tt = lane // 4, lane % 4
    k = np.arange(8)
    rows = g[:, None] + ((k & 1) * 8)[None, :]                               # [32][8]
    cols = 2 * tt[:, None] + ((k >> 2) + ((k >> 1) & 1) * 8)[None, :]        # [32][8]

    def logical(pr):
        if layout != 1:
            return pr
        tl, rr = pr >> 7, pr & 127
        return np.where(rr < 64, tl * 64 + rr, N // 2 + tl * 64 + (rr - 64))

    for nt in range(N // 128):
        s[logical(nt * 128 + np.arange(128))] = sc[nt].T
        for w in range(4):
            for f in range(2):
                lr = logical(nt * 128 + (2 * w + f) * 16 + rows)
                for ks in range(8):
                    wd = words[nt, :, w, ks, :, f]                            # [KT][32]
                    nib = ((wd[:, :, None] >> (4 * k[None, None, :])) & 15).astype(np.int16) - 8
                    for kt in range(KT):
                        q[lr, kt * 128 + ks * 16 + cols] = nib[kt]
    return q, s
