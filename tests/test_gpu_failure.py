"""The bounded-wait failure path on the GPU: a device-side wait that runs out ends its kernel with
GDN_ERR_TIMEOUT in the device error word, which gdn_device_error reports and clears, and the CUDA
context stays usable (nothing faults, traps or hangs)."""
import pytest
import torch

import oracle
from gated_deltanet_linear_03_gb300 import synth
from helpers import check_prefill, oracle_args, to_device

pytestmark = pytest.mark.gpu

GDN_ERR_TIMEOUT = 5


@pytest.fixture(scope="module")
def gdn():
    from gated_deltanet_linear_03_gb300 import gdn as g
    g.load_library()
    return g


def test_wait_that_runs_out_reports_timeout_and_context_survives(gdn):
    assert gdn.device_error() == 0
    stream = torch.cuda.Stream()
    gdn.selftest_bounded_wait(20_000, stream=stream)          # gives up after 20 ms
    assert gdn.device_error(stream) == GDN_ERR_TIMEOUT
    assert gdn.device_error(stream) == 0                        # reading clears the word

    # the context still runs the recurrence correctly
    inp = synth.prefill_inputs([100, 37], hk=2, hv=4, seed=21, init_std=0.02)
    ref_out, ref_fin = oracle.prefill(*oracle_args(inp))
    d = to_device(inp)
    out, fin = gdn.prefill(d.q, d.k, d.v, d.log_alpha, d.beta, d.cu_seqlens, init_state=d.init_state,
                           out_dtype=torch.float32, algo="chunked", cu_seqlens_host=inp.cu_seqlens.tolist())
    torch.cuda.synchronize()
    check_prefill(out, fin, ref_out, ref_fin, what="after a timed-out wait")
    assert gdn.device_error() == 0


def test_wait_limit_bounds_the_kernel_time(gdn):
    """The limit holds: a 50 ms wait ends after about 50 ms, not the kernels' 1 s."""
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    gdn.selftest_bounded_wait(50_000)
    end.record()
    torch.cuda.synchronize()
    ms = start.elapsed_time(end)
    assert 45.0 <= ms <= 500.0, ms
    assert gdn.device_error() == GDN_ERR_TIMEOUT
