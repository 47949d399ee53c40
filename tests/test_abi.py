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
