"""Thin Python binding over libdflash.so (include/dflash.h).

Argument marshalling only: every step of the draft, verify-accept and commit
runs in the library's CUDA kernels.  PyTorch supplies device memory
(`tensor.data_ptr()`) and streams (`torch.cuda.current_stream().cuda_stream`).
The functions carry the C entry points' names.  There is no fallback: if the
library is missing or no GPU is present, the first call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, List, Optional

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libdflash.so")

DFLASH_OK = 0
STATUS_NAMES = {0: "ok", -1: "EINVAL", -2: "EUNSUPPORTED", -3: "ECUDA", -4: "ECAPACITY", -5: "EWORKSPACE"}
DTYPE_F32, DTYPE_F16, DTYPE_BF16 = 0, 1, 2
LAYOUT_PLAIN, LAYOUT_GATEUP = 0, 1
DEV_KV_CAPACITY, DEV_BAD_TOKEN, DEV_BAD_LENGTH, DEV_WAIT_TIMEOUT = 0x1, 0x2, 0x4, 0x100

EXPORTS = [
    "dflash_version", "dflash_status_string", "dflash_workspace_size", "dflash_pack_w8a16",
    "dflash_w4a16_packed_bytes", "dflash_pack_w4a16",
    "dflash_w8a16_linear_workspace_size", "dflash_w8a16_linear", "dflash_draft_block",
    "dflash_lmhead_workspace_size", "dflash_lmhead_argmax", "dflash_verify_workspace_size",
    "dflash_verify_accept", "dflash_verify_accept_noalloc", "dflash_verify_sample_workspace_size",
    "dflash_verify_accept_sample", "dflash_kv_commit", "dflash_commit_draft_block", "dflash_set_launch_mode",
    "dflash_get_launch_mode", "dflash_get_status",
]
LAUNCH_STREAM_ORDER, LAUNCH_EARLY = 0, 1


class DflashError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(code, code)} ({code})")
        self.code = code


# ------------------------------------------------------------ C structs ----
class Config(ctypes.Structure):
    _fields_ = [("L", ctypes.c_int32), ("H", ctypes.c_int32), ("nq", ctypes.c_int32), ("nkv", ctypes.c_int32),
                ("d", ctypes.c_int32), ("F", ctypes.c_int32), ("V", ctypes.c_int32), ("B", ctypes.c_int32),
                ("k", ctypes.c_int32), ("mask_id", ctypes.c_int32), ("rope_theta", ctypes.c_float),
                ("eps", ctypes.c_float)]


class W8(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("s", ctypes.c_void_p), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("layout", ctypes.c_int32), ("bits", ctypes.c_int32)]


class Weights(ctypes.Structure):
    _fields_ = [("cfg", Config), ("fc", W8), ("qkv", ctypes.POINTER(W8)), ("o", ctypes.POINTER(W8)),
                ("gu", ctypes.POINTER(W8)), ("down", ctypes.POINTER(W8)),
                ("gamma_hid", ctypes.c_void_p), ("gamma_in", ctypes.c_void_p), ("gamma_post", ctypes.c_void_p),
                ("gamma_q", ctypes.c_void_p), ("gamma_k", ctypes.c_void_p), ("gamma_final", ctypes.c_void_p),
                ("embed", ctypes.c_void_p), ("lm_head", ctypes.c_void_p)]


class KV(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("len", ctypes.c_void_p), ("b", ctypes.c_int32),
                ("cap", ctypes.c_int32)]


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libdflash.so and declare its signatures; raises if it is absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libdflash.so not built ({path}); run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    PSZ = ctypes.POINTER(ctypes.c_size_t)
    sig = {
        "dflash_version": ([], ctypes.c_char_p),
        "dflash_status_string": ([I32], ctypes.c_char_p),
        "dflash_workspace_size": ([ctypes.POINTER(Config), I32, I32, PSZ], I32),
        "dflash_pack_w8a16": ([P, I32, I64, I64, I32, P, P, P], I32),
        "dflash_w4a16_packed_bytes": ([I64, I64, PSZ], I32),
        "dflash_pack_w4a16": ([P, I32, I64, I64, I32, P, P, P], I32),
        "dflash_w8a16_linear_workspace_size": ([I64, I64, I64, PSZ], I32),
        "dflash_w8a16_linear": ([ctypes.POINTER(W8), P, I64, P, P, SZ, P], I32),
        "dflash_draft_block": ([ctypes.POINTER(Weights), ctypes.POINTER(KV), P, P, P, P, P, SZ, P], I32),
        "dflash_lmhead_workspace_size": ([I64, PSZ], I32),
        "dflash_lmhead_argmax": ([P, P, I64, I64, I64, P, P, P, P, SZ, P], I32),
        "dflash_verify_workspace_size": ([I32, I32, I64, PSZ], I32),
        "dflash_verify_accept": ([P, P, I32, I32, I32, I64, P, P, P, P, P, SZ, P], I32),
        "dflash_verify_accept_noalloc": ([P, P, I32, I32, I32, I64, P, P, P, P, P], I32),
        "dflash_verify_sample_workspace_size": ([I32, I32, I64, PSZ], I32),
        "dflash_verify_accept_sample": ([P, P, I32, I32, I32, I64, ctypes.c_float, P, P, P, P, P, P, P, SZ, P],
                                        I32),
        "dflash_kv_commit": ([ctypes.POINTER(Weights), ctypes.POINTER(KV), P, I32, P, P, SZ, P], I32),
        "dflash_commit_draft_block": ([ctypes.POINTER(Weights), ctypes.POINTER(KV), P, I32, P, P, P, P, P, P, SZ, P],
                                      I32),
        "dflash_set_launch_mode": ([I32], I32),
        "dflash_get_launch_mode": ([], I32),
        "dflash_get_status": ([ctypes.POINTER(ctypes.c_int32), I32], I32),
    }
    if set(sig) != set(EXPORTS):  # every export is called with declared argument types
        raise RuntimeError(f"binding signatures out of step with exports: {set(sig) ^ set(EXPORTS)}")
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def _check(fn: str, rc: int):
    if rc != DFLASH_OK:
        raise DflashError(fn, rc)


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream=None) -> int:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _torch():
    import torch
    if not torch.cuda.is_available():
        raise RuntimeError("dflash needs a CUDA GPU; no CPU path exists")
    return torch


# ---------------------------------------------------------- entry points ----
def dflash_version() -> str:
    return load_library().dflash_version().decode()


def dflash_workspace_size(cfg, b: int, rows_per_seq: int) -> int:
    n = ctypes.c_size_t(0)
    _check("dflash_workspace_size", load_library().dflash_workspace_size(
        ctypes.byref(to_c_config(cfg)), b, rows_per_seq, ctypes.byref(n)))
    return n.value


def dflash_pack_w8a16(w, layout: int = LAYOUT_PLAIN, stream=None):
    """Pack a device weight w[N][K] (fp32/fp16/bf16 tensor); returns (q, s)
    device tensors: q uint8 [N*K] tiled, s fp16 [N] logical order."""
    torch = _torch()
    dt = {torch.float32: DTYPE_F32, torch.float16: DTYPE_F16, torch.bfloat16: DTYPE_BF16}[w.dtype]
    N, K = w.shape
    w = w.contiguous()
    q = torch.empty(N * K, dtype=torch.uint8, device=w.device)
    s = torch.empty(N, dtype=torch.float16, device=w.device)
    _check("dflash_pack_w8a16", load_library().dflash_pack_w8a16(
        w.data_ptr(), dt, N, K, layout, q.data_ptr(), s.data_ptr(), _stream(stream)))
    return q, s


def dflash_w4a16_packed_bytes(N: int, K: int) -> int:
    n = ctypes.c_size_t(0)
    _check("dflash_w4a16_packed_bytes", load_library().dflash_w4a16_packed_bytes(N, K, ctypes.byref(n)))
    return n.value


def dflash_pack_w4a16(w, layout: int = LAYOUT_PLAIN, stream=None, q=None, s=None):
    """Pack a device weight w[N][K] to int4 with per-128-column group scales;
    returns (q, s): q uint8 tiles (scales included), s fp16 [N][K/128].  `q`
    and `s` may be given (contiguous device buffers of those sizes), e.g. a
    128-row-aligned slice of a larger matrix's tiles."""
    torch = _torch()
    lib = load_library()
    dt = {torch.float32: DTYPE_F32, torch.float16: DTYPE_F16, torch.bfloat16: DTYPE_BF16}[w.dtype]
    N, K = w.shape
    w = w.contiguous()
    nbytes = dflash_w4a16_packed_bytes(N, K)
    if q is None:
        q = torch.empty(nbytes, dtype=torch.uint8, device=w.device)
    if s is None:
        s = torch.empty((N, K // 128), dtype=torch.float16, device=w.device)
    if q.numel() < nbytes or s.numel() < N * (K // 128) or not (q.is_contiguous() and s.is_contiguous()):
        raise ValueError("dflash_pack_w4a16: output buffers too small or not contiguous")
    _check("dflash_pack_w4a16", lib.dflash_pack_w4a16(
        w.data_ptr(), dt, N, K, layout, q.data_ptr(), s.data_ptr(), _stream(stream)))
    return q, s


def w8_desc(q, s, N: int, K: int, layout: int = LAYOUT_PLAIN, bits: int = 8) -> W8:
    return W8(q.data_ptr(), s.data_ptr() if s is not None else None, N, K, layout, bits)


def dflash_w8a16_linear_workspace_size(M: int, N: int, K: int) -> int:
    n = ctypes.c_size_t(0)
    _check("dflash_w8a16_linear_workspace_size",
           load_library().dflash_w8a16_linear_workspace_size(M, N, K, ctypes.byref(n)))
    return n.value


def dflash_w8a16_linear(desc: W8, x, ws=None, stream=None, y=None):
    """y[M][N] fp32 = W8(desc) applied to fp16 x[M][K] (y may be given).  ws:
    a zero-filled uint8 workspace of dflash_w8a16_linear_workspace_size bytes
    (allocated here when not given)."""
    torch = _torch()
    lib = load_library()
    M = x.shape[0]
    need = dflash_w8a16_linear_workspace_size(M, desc.N, desc.K)
    if ws is None:
        ws = torch.zeros(max(need, 256), dtype=torch.uint8, device=x.device)
    elif ws.numel() < need:
        raise ValueError(f"dflash_w8a16_linear: workspace of {ws.numel()} bytes, {need} needed")
    if y is None:
        y = torch.empty((M, desc.N), dtype=torch.float32, device=x.device)
    elif y.numel() < M * desc.N or not y.is_contiguous() or y.dtype != torch.float32:
        raise ValueError("dflash_w8a16_linear: y must be contiguous fp32 with M*N elements")
    _check("dflash_w8a16_linear", lib.dflash_w8a16_linear(
        ctypes.byref(desc), x.data_ptr(), M, y.data_ptr(), ws.data_ptr(), ws.numel(), _stream(stream)))
    return y


def dflash_lmhead_argmax(h, w, idx=None, maxlogit=None, logits=None, ws=None, stream=None):
    """h bf16-bits int16/uint16 or bf16 tensor [M][H]; w [V][H] likewise."""
    torch = _torch()
    lib = load_library()
    M, H = h.shape
    V = w.shape[0]
    n = ctypes.c_size_t(0)
    _check("dflash_lmhead_workspace_size", lib.dflash_lmhead_workspace_size(M, ctypes.byref(n)))
    if ws is None:
        ws = torch.zeros(n.value, dtype=torch.uint8, device=h.device)
    if idx is None:
        idx = torch.empty(M, dtype=torch.int32, device=h.device)
    _check("dflash_lmhead_argmax", lib.dflash_lmhead_argmax(
        h.data_ptr(), w.data_ptr(), M, V, H, idx.data_ptr(), _ptr(maxlogit), _ptr(logits), ws.data_ptr(),
        ws.numel(), _stream(stream)))
    return idx


def dflash_verify_workspace_size(b: int, R: int, V: int) -> int:
    n = ctypes.c_size_t(0)
    _check("dflash_verify_workspace_size", load_library().dflash_verify_workspace_size(b, R, V, ctypes.byref(n)))
    return n.value


def dflash_verify_accept(logits, draft, n_out, corr_out, emitted=None, next_tok=None, ws=None, stream=None):
    """logits fp32 [b][R][V], draft int32 [b][D] (device tensors)."""
    torch = _torch()
    b, R, V = logits.shape
    D = draft.shape[1]
    if ws is None:
        ws = torch.zeros(dflash_verify_workspace_size(b, R, V), dtype=torch.uint8, device=logits.device)
    _check("dflash_verify_accept", load_library().dflash_verify_accept(
        logits.data_ptr(), draft.data_ptr(), b, R, D, V, n_out.data_ptr(), corr_out.data_ptr(), _ptr(emitted),
        _ptr(next_tok), ws.data_ptr(), ws.numel(), _stream(stream)))


def dflash_verify_sample_workspace_size(b: int, R: int, V: int) -> int:
    n = ctypes.c_size_t(0)
    _check("dflash_verify_sample_workspace_size",
           load_library().dflash_verify_sample_workspace_size(b, R, V, ctypes.byref(n)))
    return n.value


def dflash_verify_accept_sample(logits, draft, temperature: float, u_accept, u_sample, n_out, corr_out,
                                emitted=None, next_tok=None, ws=None, stream=None):
    """Temperature speculative-sampling accept.  logits fp32 [b][R][V], draft
    int32 [b][D], u_accept fp32 [b][D], u_sample fp32 [b][V] (uniforms in
    (0, 1)), all device tensors."""
    torch = _torch()
    b, R, V = logits.shape
    D = draft.shape[1]
    if ws is None:
        ws = torch.zeros(dflash_verify_sample_workspace_size(b, R, V), dtype=torch.uint8, device=logits.device)
    _check("dflash_verify_accept_sample", load_library().dflash_verify_accept_sample(
        logits.data_ptr(), draft.data_ptr(), b, R, D, V, float(temperature), u_accept.data_ptr(),
        u_sample.data_ptr(), n_out.data_ptr(), corr_out.data_ptr(), _ptr(emitted), _ptr(next_tok),
        ws.data_ptr(), ws.numel(), _stream(stream)))


def dflash_verify_accept_noalloc(logits, draft, n_out, corr_out, emitted=None, next_tok=None, stream=None):
    """Same result as dflash_verify_accept without a workspace: for callers
    that cannot allocate device memory, the library's own fixed device scratch
    is used (one shared array per GPU; serialise overlapping calls)."""
    b, R, V = logits.shape
    D = draft.shape[1]
    _check("dflash_verify_accept_noalloc", load_library().dflash_verify_accept_noalloc(
        logits.data_ptr(), draft.data_ptr(), b, R, D, V, n_out.data_ptr(), corr_out.data_ptr(), _ptr(emitted),
        _ptr(next_tok), _stream(stream)))


def dflash_draft_block(model: "DeviceDrafter", kv: "KVCache", last_tok, draft_out, ws, hidden=None, logits=None,
                       stream=None):
    _check("dflash_draft_block", load_library().dflash_draft_block(
        ctypes.byref(model.c), ctypes.byref(kv.c), last_tok.data_ptr(), draft_out.data_ptr(), _ptr(hidden),
        _ptr(logits), ws.data_ptr(), ws.numel(), _stream(stream)))


def dflash_kv_commit(model: "DeviceDrafter", kv: "KVCache", hid, n, ws, stream=None):
    """hid fp16 [b][rows_per_seq][k*H]; n int32 [b] (device)."""
    rps = hid.shape[1]
    _check("dflash_kv_commit", load_library().dflash_kv_commit(
        ctypes.byref(model.c), ctypes.byref(kv.c), hid.data_ptr(), rps, n.data_ptr(), ws.data_ptr(), ws.numel(),
        _stream(stream)))


def dflash_commit_draft_block(model: "DeviceDrafter", kv: "KVCache", hid, n, last_tok, draft_out, ws, hidden=None,
                              logits=None, stream=None):
    """dflash_kv_commit(hid, n) and dflash_draft_block(last_tok) in one pass.
    hid fp16 [b][rows_per_seq][k*H], n int32 [b], last_tok int32 [b]."""
    rps = hid.shape[1]
    _check("dflash_commit_draft_block", load_library().dflash_commit_draft_block(
        ctypes.byref(model.c), ctypes.byref(kv.c), hid.data_ptr(), rps, n.data_ptr(), last_tok.data_ptr(),
        draft_out.data_ptr(), _ptr(hidden), _ptr(logits), ws.data_ptr(), ws.numel(), _stream(stream)))


def dflash_set_launch_mode(mode: int):
    """LAUNCH_STREAM_ORDER (default) or LAUNCH_EARLY (dedicated GPU, one
    stream only; see include/dflash.h)."""
    _check("dflash_set_launch_mode", load_library().dflash_set_launch_mode(mode))


def dflash_get_launch_mode() -> int:
    return load_library().dflash_get_launch_mode()


class launch_mode:
    """Context manager: the given launch mode inside, the previous one after."""

    def __init__(self, mode: int):
        self.mode = mode

    def __enter__(self):
        self.prev = dflash_get_launch_mode()
        dflash_set_launch_mode(self.mode)
        return self

    def __exit__(self, *exc):
        dflash_set_launch_mode(self.prev)


def dflash_get_status(clear: bool = True) -> int:
    v = ctypes.c_int32(0)
    _check("dflash_get_status", load_library().dflash_get_status(ctypes.byref(v), 1 if clear else 0))
    return v.value


# ------------------------------------------------------- device objects ----
def to_c_config(cfg) -> Config:
    return Config(cfg.L, cfg.H, cfg.nq, cfg.nkv, cfg.d, cfg.F, cfg.V, cfg.B, cfg.k, cfg.mask_id,
                  cfg.rope_theta, cfg.eps)


class DeviceDrafter:
    """A drafter's tensors resident on the GPU, packed by dflash_pack_w8a16
    (bits 8) or dflash_pack_w4a16 (bits 4).

    `weights` maps names to host arrays: the projection matrices "fc",
    "qkv{l}", "o{l}", "gu{l}", "down{l}" as float weights [N][K] (anything
    numpy can turn into fp32; the gate|up matrix holds F gate rows then F up
    rows), the fp32 RMSNorm gammas "gamma_hid" [H], "gamma_in" / "gamma_post"
    [L][H], "gamma_q" / "gamma_k" [L][d], "gamma_final" [H], and the bf16 bit
    patterns (uint16) of "embed" and "lm_head" [V][H].  Matrices are read one
    at a time, uploaded as fp32 and packed on the device, so a mapping that
    builds each matrix on access keeps at most one float matrix alive."""

    def __init__(self, cfg, weights, device="cuda", bits: int = 8):
        torch = _torch()
        self.cfg = cfg
        self.keep: List[object] = []
        dev = torch.device(device)
        if bits not in (4, 8):
            raise ValueError("bits must be 4 or 8")
        self.bits = bits
        W = weights

        def pack(name, layout=LAYOUT_PLAIN):
            w = torch.from_numpy(np.ascontiguousarray(W[name], dtype=np.float32)).to(dev)
            if w.dim() != 2:
                raise ValueError(f"{name}: expected a 2-D float weight")
            N, K = w.shape
            if bits == 4:
                qd, sd = dflash_pack_w4a16(w, layout)
            else:
                qd, sd = dflash_pack_w8a16(w, layout)
            del w
            self.keep += [qd, sd]
            return W8(qd.data_ptr(), sd.data_ptr(), N, K, layout, bits)

        def up(a, dtype=None):
            t = torch.from_numpy(np.ascontiguousarray(a)).to(dev)
            self.keep.append(t)
            return t.data_ptr()

        L = cfg.L
        self.fc = pack("fc")
        self.qkv = (W8 * L)(*[pack(f"qkv{l}") for l in range(L)])
        self.o = (W8 * L)(*[pack(f"o{l}") for l in range(L)])
        self.gu = (W8 * L)(*[pack(f"gu{l}", LAYOUT_GATEUP) for l in range(L)])
        self.down = (W8 * L)(*[pack(f"down{l}") for l in range(L)])
        torch.cuda.synchronize()
        self.embed_t = torch.from_numpy(np.ascontiguousarray(W["embed"]).view(np.int16)).to(dev)
        self.lm_t = torch.from_numpy(np.ascontiguousarray(W["lm_head"]).view(np.int16)).to(dev)
        self.keep += [self.embed_t, self.lm_t]
        self.c = Weights(to_c_config(cfg), self.fc,
                         ctypes.cast(self.qkv, ctypes.POINTER(W8)), ctypes.cast(self.o, ctypes.POINTER(W8)),
                         ctypes.cast(self.gu, ctypes.POINTER(W8)), ctypes.cast(self.down, ctypes.POINTER(W8)),
                         up(W["gamma_hid"]), up(W["gamma_in"]), up(W["gamma_post"]), up(W["gamma_q"]),
                         up(W["gamma_k"]), up(W["gamma_final"]), self.embed_t.data_ptr(), self.lm_t.data_ptr())


class KVCache:
    """Draft KV cache [L][b][nkv][cap][d] fp16 (K after norm + RoPE) and
    per-sequence lengths (device int32)."""

    def __init__(self, cfg, b: int, cap: int, device="cuda"):
        torch = _torch()
        shape = (cfg.L, b, cfg.nkv, cap, cfg.d)
        self.k = torch.zeros(shape, dtype=torch.float16, device=device)
        self.v = torch.zeros(shape, dtype=torch.float16, device=device)
        self.len = torch.zeros(b, dtype=torch.int32, device=device)
        self.b, self.cap = b, cap
        self.c = KV(self.k.data_ptr(), self.v.data_ptr(), self.len.data_ptr(), b, cap)


def workspace(cfg, b: int, rows_per_seq: int, device="cuda"):
    """Zero-filled workspace for dflash_draft_block / dflash_kv_commit."""
    torch = _torch()
    return torch.zeros(dflash_workspace_size(cfg, b, rows_per_seq), dtype=torch.uint8, device=device)
