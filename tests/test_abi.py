"""CPU-side checks of the C ABI: the library builds, loads without a GPU,
exports every entry point include/dflash.h declares, and rejects bad
arguments on the host before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dflash.h")


@pytest.fixture(scope="module")
def lib():
    from block_diffusion_speculative_draft_gb300 import build, api
    build.build()
    return api.load_library()


def declared_functions():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"DFLASH_API\s+[\w\s\*]+?\b(dflash_\w+)\s*\(", src)))


def test_header_declares_the_five_calls():
    names = declared_functions()
    for n in ["dflash_pack_w8a16", "dflash_draft_block", "dflash_lmhead_argmax", "dflash_verify_accept",
              "dflash_kv_commit"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    from block_diffusion_speculative_draft_gb300 import api
    for n in declared_functions():
        assert hasattr(lib, n), n
    assert set(declared_functions()) == set(api.EXPORTS)


def test_host_only_calls(lib):
    from block_diffusion_speculative_draft_gb300 import api
    from block_diffusion_speculative_draft_gb300.configs import ALL
    assert api.dflash_version().startswith("dflash")
    assert lib.dflash_status_string(-4) == b"KV capacity exceeded"
    for cfg in ALL:
        n = api.dflash_workspace_size(cfg, cfg.b, cfg.B)
        assert n > 0
    assert api.dflash_verify_workspace_size(1, 16, 151936) > 0


def test_bad_arguments_rejected_on_host(lib):
    from block_diffusion_speculative_draft_gb300 import api
    from block_diffusion_speculative_draft_gb300.configs import TINY
    P = None
    n = ctypes.c_size_t(0)
    # null pointers / bad sizes never reach the GPU
    assert lib.dflash_pack_w8a16(P, 0, 128, 128, 0, P, P, P) == -1
    assert lib.dflash_verify_accept(P, P, 1, 16, 15, 100, P, P, P, P, P, 0, P) == -1
    assert lib.dflash_verify_workspace_size(1, 16, 151936, None) == -1
    assert lib.dflash_lmhead_workspace_size(0, ctypes.byref(n)) == -1
    assert lib.dflash_draft_block(None, None, P, P, P, P, P, 0, P) == -1
    assert lib.dflash_kv_commit(None, None, P, 16, P, P, 0, P) == -1
    # unsupported shapes
    cfg = api.to_c_config(TINY)
    cfg.d = 96
    assert lib.dflash_workspace_size(ctypes.byref(cfg), 1, 16, ctypes.byref(n)) == -2
    cfg = api.to_c_config(TINY)
    cfg.H = 500
    assert lib.dflash_workspace_size(ctypes.byref(cfg), 1, 16, ctypes.byref(n)) == -2
    cfg = api.to_c_config(TINY)
    cfg.mask_id = TINY.V
    assert lib.dflash_workspace_size(ctypes.byref(cfg), 1, 16, ctypes.byref(n)) == -1
    # D > R and a non-128 packed shape
    x = ctypes.c_void_p(16)
    assert lib.dflash_verify_accept(x, x, 1, 4, 5, 100, x, x, P, P, x, 1 << 20, P) == -1
    assert lib.dflash_pack_w8a16(x, 0, 100, 128, 0, x, x, P) == -2
    # sampling accept: temperature must be finite and > 0, uniforms present,
    # workspace large enough
    ws_need = api.dflash_verify_sample_workspace_size(1, 4, 100)
    assert ws_need > 0
    for T in (0.0, -1.0, float("inf"), float("nan")):
        assert lib.dflash_verify_accept_sample(x, x, 1, 4, 3, 100, T, x, x, x, x, P, P, x, ws_need, P) == -1
    assert lib.dflash_verify_accept_sample(x, x, 1, 4, 3, 100, 1.0, P, x, x, x, P, P, x, ws_need, P) == -1
    assert lib.dflash_verify_accept_sample(x, x, 1, 4, 5, 100, 1.0, x, x, x, x, P, P, x, ws_need, P) == -1
    assert lib.dflash_verify_accept_sample(x, x, 1, 4, 3, 100, 1.0, x, x, x, x, P, P, x, ws_need - 1, P) == -5


def test_weights_struct_checked_before_launch(lib):
    """A dflash_weights whose descriptors disagree with the config is
    rejected with EINVAL on the host."""
    from block_diffusion_speculative_draft_gb300 import api
    from block_diffusion_speculative_draft_gb300.configs import TINY as c
    fake = ctypes.c_void_p(256)
    w8 = api.W8(256, 256, c.H, c.k * c.H, 0)
    L = c.L
    arr = (api.W8 * L)(*[api.W8(256, 256, 1, 1, 0) for _ in range(L)])  # wrong shapes
    W = api.Weights(api.to_c_config(c), w8, ctypes.cast(arr, ctypes.POINTER(api.W8)),
                    ctypes.cast(arr, ctypes.POINTER(api.W8)), ctypes.cast(arr, ctypes.POINTER(api.W8)),
                    ctypes.cast(arr, ctypes.POINTER(api.W8)), 256, 256, 256, 256, 256, 256, 256, 256)
    kv = api.KV(256, 256, 256, 1, 64)
    assert lib.dflash_draft_block(ctypes.byref(W), ctypes.byref(kv), fake, fake, None, None, fake, 1 << 30,
                                  None) == -1


def test_int4_entry_points_checked_on_host(lib):
    from block_diffusion_speculative_draft_gb300 import api
    n = ctypes.c_size_t(0)
    assert lib.dflash_w4a16_packed_bytes(128, 256, ctypes.byref(n)) == 0 and n.value == 2 * 8448
    assert api.dflash_w4a16_packed_bytes(256, 384) == 2 * 3 * 8448
    assert lib.dflash_w4a16_packed_bytes(100, 128, ctypes.byref(n)) == -2
    assert lib.dflash_w4a16_packed_bytes(128, 128, None) == -1
    P, x = None, ctypes.c_void_p(256)
    assert lib.dflash_pack_w4a16(P, 0, 128, 128, 0, x, x, P) == -1
    assert lib.dflash_pack_w4a16(x, 0, 128, 128, 0, x, P, P) == -1
    assert lib.dflash_pack_w4a16(x, 3, 128, 128, 0, x, x, P) == -1          # unknown dtype
    assert lib.dflash_pack_w4a16(x, 0, 128, 100, 0, x, x, P) == -2          # K not a multiple of 128
    assert lib.dflash_pack_w4a16(x, 0, 128, 128, 0, ctypes.c_void_p(264), x, P) == -1  # q_out misaligned


def _tiny_weights(api, c, bits=8, fc_bits=None, s_ptr=256):
    def d(N, K, layout=0, b=bits):
        return api.W8(256, s_ptr, N, K, layout, b)
    L = c.L
    arr = lambda N, K, layout=0: (api.W8 * L)(*[d(N, K, layout) for _ in range(L)])
    qkv, o = arr(c.nqkv, c.H), arr(c.H, c.nq * c.d)
    gu, down = arr(2 * c.F, c.H, 1), arr(c.H, c.F)
    P = lambda a: ctypes.cast(a, ctypes.POINTER(api.W8))
    W = api.Weights(api.to_c_config(c), d(c.H, c.k * c.H, 0, bits if fc_bits is None else fc_bits),
                    P(qkv), P(o), P(gu), P(down), 256, 256, 256, 256, 256, 256, 256, 256)
    return W, (qkv, o, gu, down)


def test_weight_bits_checked_before_launch(lib):
    """bits must be 0, 8 or 4 and the same for every matrix; int4 matrices
    need no scale pointer; the single-kernel step refuses int4.  Every case
    returns on the host (a workspace that is too small is the last check
    before any launch)."""
    from block_diffusion_speculative_draft_gb300 import api
    from block_diffusion_speculative_draft_gb300.configs import TINY as c
    fake = ctypes.c_void_p(256)
    kv = api.KV(256, 256, 256, 1, 64)

    def draft(W, fn=lib.dflash_draft_block):
        return fn(ctypes.byref(W), ctypes.byref(kv), fake, fake, None, None, None, 0, None)

    for bits in (0, 8, 4):
        W, keep = _tiny_weights(api, c, bits)
        assert draft(W) == -5, bits                      # valid: only the workspace is missing
    W, keep = _tiny_weights(api, c, 4, s_ptr=None)
    assert draft(W) == -5                                # int4 needs no scale array
    W, keep = _tiny_weights(api, c, 8, s_ptr=None)
    assert draft(W) == -1                                # int8 does
    W, keep = _tiny_weights(api, c, 5)
    assert draft(W) == -1
    W, keep = _tiny_weights(api, c, 4, fc_bits=8)
    assert draft(W) == -1                                # mixed widths


def test_launch_mode_switch(lib):
    from block_diffusion_speculative_draft_gb300 import api
    assert lib.dflash_get_launch_mode() == api.LAUNCH_STREAM_ORDER  # the default
    with api.launch_mode(api.LAUNCH_EARLY):
        assert lib.dflash_get_launch_mode() == api.LAUNCH_EARLY
    assert lib.dflash_get_launch_mode() == api.LAUNCH_STREAM_ORDER
    assert lib.dflash_set_launch_mode(2) == -1 and lib.dflash_set_launch_mode(-1) == -1
    assert lib.dflash_get_launch_mode() == api.LAUNCH_STREAM_ORDER
