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
