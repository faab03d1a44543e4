"""gdn_prefill_noalloc: the chunked prefill with the library's fixed scratch.

It exists for callers that cannot allocate device memory (code that must not
call cudaMalloc while it runs, plugins whose host framework owns all device
allocations, runtimes without a device allocator), so it cannot ask them for a
workspace.  Its results must match the normal entry point, gdn_prefill with a
caller workspace, on the same inputs; two calls in a row check that the shared
scratch carries nothing from one call into the next.  This file is collected
last on purpose (a failure here leaves every other test already run).
"""
import ctypes

import pytest
import torch

from gated_deltanet_linear_03_gb300 import synth
from helpers import to_device


@pytest.fixture(scope="module")
def gdn():
    from gated_deltanet_linear_03_gb300 import _build, gdn as g
    _build.build()
    g.load_library()
    return g


def _pair(gdn, inp):
    d = to_device(inp)
    cu = inp.cu_seqlens.tolist()
    ref_out, ref_fin = gdn.prefill(d.q, d.k, d.v, d.log_alpha, d.beta, d.cu_seqlens, init_state=d.init_state,
                                   algo="chunked", out_dtype=torch.float32, cu_seqlens_host=cu)
    out, fin = gdn.prefill_noalloc(d.q, d.k, d.v, d.log_alpha, d.beta, d.cu_seqlens, init_state=d.init_state,
                                   out_dtype=torch.float32, cu_seqlens_host=cu)
    torch.cuda.synchronize()
    assert gdn.device_error() == 0
    return out, fin, ref_out, ref_fin


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_twice(gdn):
    """The same kernels on the same inputs as gdn_prefill, so the results must be identical bit for bit.  The
    small ragged case runs again after the 4096-token case, so that its second call finds the larger call's
    contents still in the shared scratch."""
    small = synth.prefill_inputs([300, 65, 1], hk=4, hv=8, seed=71, init_std=0.02)
    large = synth.prefill_inputs([4096], seed=72)             # the largest size the scratch holds
    for inp in (small, large, small):                         # calls in a row on the shared scratch
        out, fin, ref_out, ref_fin = _pair(gdn, inp)
        assert torch.equal(out, ref_out)
        assert torch.equal(fin, ref_fin)


def test_noalloc_rejects_problems_beyond_the_scratch(gdn):
    """Needs more than 97 MiB of scratch: refused on the host before any GPU work."""
    lib = gdn.load_library()
    T = 4096 + 64
    cu = (ctypes.c_int32 * 2)(0, T)
    st = ctypes.c_int(-1)
    need = lib.gdn_prefill_workspace_size(1, T, 16, 32, 128, 128, cu, 0, ctypes.byref(st))
    assert st.value == 0 and need > gdn.NOALLOC_SCRATCH_BYTES
    fake = ctypes.c_void_p(0x10000)
    r = lib.gdn_prefill_noalloc(1, T, 16, 32, 128, 128, fake, fake, fake, fake, fake, None, fake, cu, fake, 0,
                                None, 0, 1.0, None, 1e-6, None, None, None)
    assert r == 7   # GDN_ERR_WORKSPACE
