"""GPU parity of the in-kernel query/key preparation (qk_norm, q_scale) against the fp64 oracle, on every
path: chunked (tcgen05), both mappings of the direct scan, the no-alloc entry point and the decode step.
The inputs are raw projections (N(0, 1) entries times a per-vector length in [0.25, 4]), which the kernels
must L2-normalise before the recurrence; q is then scaled by 1/sqrt(dk)."""
import math

import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_linear_03_gb300 import synth
from helpers import check_prefill, max_abs_err, np32, oracle_args, to_device, OUT_ATOL

pytestmark = pytest.mark.gpu

SCALE = 1.0 / math.sqrt(128)


@pytest.fixture(scope="module")
def gdn():
    from gated_deltanet_linear_03_gb300 import gdn as g
    g.load_library()
    return g


CASES = {
    # (lengths, algo): chunked; register scan (long, and few tokens in one sequence); streaming scan
    "chunked_ragged": ([200, 1, 64, 130], "chunked"),
    "scan_T200": ([200, 37], "scan"),
    "scan_single_T8": ([8], "scan"),
    "scan_short_batch": ([5, 32, 1, 17, 9, 0, 3, 12], "scan"),
    "auto_short": ([4, 9], "auto"),
}


@pytest.mark.parametrize("case", list(CASES))
def test_qk_norm_matches_oracle(gdn, case):
    lengths, algo = CASES[case]
    inp = synth.prefill_inputs(lengths, seed=51, init_std=0.02, raw_qk=True)
    ref_out, ref_fin = oracle.prefill(*oracle_args(inp), qk_norm=True, q_scale=SCALE)
    d = to_device(inp)
    out, fin = gdn.prefill(d.q, d.k, d.v, d.log_alpha, d.beta, d.cu_seqlens, init_state=d.init_state, algo=algo,
                           cu_seqlens_host=inp.cu_seqlens.tolist(), qk_norm=True, q_scale=SCALE)
    torch.cuda.synchronize()
    check_prefill(out, fin, ref_out, ref_fin, what=case)


@pytest.mark.parametrize("algo", ["chunked", "scan"])
def test_q_scale_alone(gdn, algo):
    """qk_norm off, q_scale != 1: unit keys as given, queries scaled in the kernel."""
    inp = synth.prefill_inputs([150, 40], seed=52, init_std=0.02, scale_q=False)
    ref_out, ref_fin = oracle.prefill(*oracle_args(inp), q_scale=SCALE)
    d = to_device(inp)
    out, fin = gdn.prefill(d.q, d.k, d.v, d.log_alpha, d.beta, d.cu_seqlens, init_state=d.init_state, algo=algo,
                           cu_seqlens_host=inp.cu_seqlens.tolist(), q_scale=SCALE)
    torch.cuda.synchronize()
    check_prefill(out, fin, ref_out, ref_fin, what=f"q_scale {algo}")


def test_qk_norm_noalloc(gdn):
    inp = synth.prefill_inputs([300], seed=53, init_std=0.02, raw_qk=True)
    ref_out, ref_fin = oracle.prefill(*oracle_args(inp), qk_norm=True, q_scale=SCALE)
    d = to_device(inp)
    out, fin = gdn.prefill_noalloc(d.q, d.k, d.v, d.log_alpha, d.beta, d.cu_seqlens, init_state=d.init_state,
                                   cu_seqlens_host=inp.cu_seqlens.tolist(), qk_norm=True, q_scale=SCALE)
    torch.cuda.synchronize()
    check_prefill(out, fin, ref_out, ref_fin, what="noalloc qk_norm")


@pytest.mark.parametrize("d", [128, 64, 32])
def test_qk_norm_decode(gdn, d):
    di = synth.decode_inputs(6, 3, hk=2, hv=4, dk=d, dv=d, seed=54, raw_qk=True)
    st = di.state.cuda()
    ref = di.state.double().numpy()
    for t in range(3):
        args = (di.q[t], di.k[t], di.v[t], di.log_alpha[t], di.beta[t])
        out = gdn.decode_step(st, *[x.cuda() for x in args], out_dtype=torch.float32, qk_norm=True, q_scale=SCALE)
        ref_out, ref = oracle.decode_step(ref, *[np32(x) for x in args], qk_norm=True, q_scale=SCALE)
        torch.cuda.synchronize()
        assert max_abs_err(out, ref_out) <= OUT_ATOL
    g = np32(st).astype(np.float64)
    rel = np.sqrt(((g - ref) ** 2).sum(axis=(-1, -2))) / np.sqrt((ref ** 2).sum(axis=(-1, -2)))
    assert rel.max() <= 1e-3
