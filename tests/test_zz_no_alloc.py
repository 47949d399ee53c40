"""The allocation-free verify-accept against the workspace one.

Some callers cannot allocate device memory (an allocator owned by someone
else, a capture that forbids allocation, a bare C host); for them the
library offers dflash_verify_accept_noalloc, whose scratch is a fixed array
inside the library.  This test calls it through the C ABI twice in a row on
the same inputs and checks that both calls give exactly the result of
dflash_verify_accept (integer outputs: bit-exact), so leftovers from one call
cannot leak into the next.  It lives in its own file, collected last, and
passes alone in a fresh process or after every other test.
"""
import numpy as np
import pytest

from block_diffusion_speculative_draft_gb300 import synth
from tests.gpu_util import gpu_available

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not gpu_available(), reason="needs a GPU")]


@pytest.mark.parametrize("b,R,D,V", [(1, 16, 15, 151936), (8, 16, 15, 151936), (3, 5, 4, 4093), (2, 32, 31, 50000)])
def test_noalloc_matches_workspace_version(b, R, D, V):
    import torch
    from block_diffusion_speculative_draft_gb300 import api
    dev = torch.device("cuda:0")
    draft = synth.tokens(21, f"na{b}{R}", b * D, V).reshape(b, D)
    nacc = synth.accept_lengths(21, f"nn{b}{R}", b, D)
    lg = synth.verify_logits(21, f"nl{b}{R}{V}", draft, R, V, nacc)
    tl, td = torch.from_numpy(lg).to(dev), torch.from_numpy(draft).to(dev)

    def outs():
        return [torch.full((b,), -7, dtype=torch.int32, device=dev), torch.full((b,), -7, dtype=torch.int32, device=dev),
                torch.full((b, R), -7, dtype=torch.int32, device=dev), torch.full((b,), -7, dtype=torch.int32, device=dev)]

    ref = outs()
    api.dflash_verify_accept(tl, td, *ref)
    for _ in range(2):  # two calls in a row share the fixed scratch
        got = outs()
        api.dflash_verify_accept_noalloc(tl, td, *got)
        torch.cuda.synchronize()
        for r, g in zip(ref, got):
            assert torch.equal(r, g)
    assert np.array_equal(ref[0].cpu().numpy(), np.minimum(nacc, D))


def test_noalloc_rejects_oversized_batch():
    import torch
    from block_diffusion_speculative_draft_gb300 import api
    dev = torch.device("cuda:0")
    b, R, V = 2000, 2, 64  # 2000 per-sequence counters do not fit the fixed scratch
    lg = torch.zeros((b, R, V), dtype=torch.float32, device=dev)
    dr = torch.zeros((b, 1), dtype=torch.int32, device=dev)
    n = torch.empty(b, dtype=torch.int32, device=dev)
    c = torch.empty(b, dtype=torch.int32, device=dev)
    with pytest.raises(api.DflashError) as e:
        api.dflash_verify_accept_noalloc(lg, dr, n, c)
    assert e.value.code == -5
