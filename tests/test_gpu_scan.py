"""GPU parity of the direct-scan prefill (GDN_ALGO_SCAN) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_linear_03_gb300 import synth
from helpers import as_bf16_inputs, check_prefill, oracle_args, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gdn():
    from gated_deltanet_linear_03_gb300 import gdn as g
    g.load_library()
    return g


def run(gdn, inp, algo, out_dtype=torch.bfloat16, with_init=True):
    d = to_device(inp)
    return gdn.prefill(d.q, d.k, d.v, d.log_alpha, d.beta, d.cu_seqlens,
                       init_state=d.init_state if with_init else None, out_dtype=out_dtype, algo=algo,
                       cu_seqlens_host=inp.cu_seqlens.tolist())


CASES = {
    "tiny_T64_d32": lambda: as_bf16_inputs(synth.tiny_case()),
    "model_T200": lambda: synth.prefill_inputs([200], seed=21),
    "ragged_init": lambda: synth.prefill_inputs([1, 63, 64, 65, 130, 0, 7], seed=22, init_std=0.02),
    "slow_decay_T256": lambda: synth.prefill_inputs([256], seed=23, gates="slow", init_std=0.02),
    "d64_group4": lambda: synth.prefill_inputs([100, 37], hk=1, hv=4, dk=64, dv=64, seed=24, init_std=0.1),
    # At most 32 tokens per sequence and more (sequence, head, 16-row) slices than one wave of the register
    # scan on a 152-SM GB300 (3 per SM): the row-streaming short-sequence mapping.
    "short_ragged": lambda: synth.prefill_inputs([3, 16, 1, 9, 0, 32], seed=27, init_std=0.02),
    "short_slow_T32": lambda: synth.prefill_inputs([32, 31], seed=28, gates="slow", init_std=0.02),
    "short_d64": lambda: synth.prefill_inputs([5, 2, 17, 9], hk=8, hv=32, dk=64, dv=64, seed=29, init_std=0.1),
    "short_d32": lambda: as_bf16_inputs(synth.prefill_inputs([8, 3, 1, 5, 2, 7, 4, 6], hk=8, hv=32, dk=32, dv=32,
                                                             seed=30, gates="tiny", scale_q=False,
                                                             qkv_dtype=torch.float32)),
    # few tokens in a single sequence: the register scan
    "short_single_T8": lambda: synth.prefill_inputs([8], seed=31, init_std=0.02),
}


@pytest.mark.parametrize("case", list(CASES))
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_scan_matches_oracle(gdn, case, out_dtype):
    inp = CASES[case]()
    ref_out, ref_fin = oracle.prefill(*oracle_args(inp))
    out, fin = run(gdn, inp, "scan", out_dtype)
    torch.cuda.synchronize()
    check_prefill(out, fin, ref_out, ref_fin, what=case)


def test_scan_in_place_state(gdn):
    inp = synth.prefill_inputs([50, 70], seed=25, init_std=0.05)
    ref_out, ref_fin = oracle.prefill(*oracle_args(inp))
    d = to_device(inp)
    st = d.init_state.clone()
    out, fin = gdn.prefill(d.q, d.k, d.v, d.log_alpha, d.beta, d.cu_seqlens, init_state=st, final_state=st,
                           algo="scan")
    torch.cuda.synchronize()
    assert fin.data_ptr() == st.data_ptr()
    check_prefill(out, st, ref_out, ref_fin, what="in-place")


@pytest.mark.parametrize("lengths", [[3, 16, 1, 9], [8], [200], [40, 1, 100]])
def test_auto_matches_oracle(gdn, lengths):
    """algo="auto" (gdn_prefill_algo's choice) against the oracle, on short and longer sequences."""
    inp = synth.prefill_inputs(lengths, seed=26, init_std=0.02)
    cu = inp.cu_seqlens.tolist()
    resolved = gdn.resolve_algo(len(lengths), cu[-1], 16, 32, 128, 128, cu)
    assert resolved == ("scan" if max(lengths) <= 16 else "chunked")
    ref_out, ref_fin = oracle.prefill(*oracle_args(inp))
    out, fin = run(gdn, inp, "auto")
    torch.cuda.synchronize()
    check_prefill(out, fin, ref_out, ref_fin, what=f"auto {lengths} -> {resolved}")
