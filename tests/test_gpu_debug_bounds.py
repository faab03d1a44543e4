"""The bounds-checking build (GDN_DEBUG_BOUNDS): every global address a kernel computes and every tensor-copy
coordinate is checked against the extent of its buffer before use; an access out of range is skipped and
recorded in the device error word (GDN_ERR_INTERNAL), never trapped.  It stands in for compute-sanitizer,
which is not available on these GPUs.

Each path runs in that build on the addressing-heavy cases (ragged packing with empty, 1-token and
partial-chunk sequences, head groupings, fused options, the 128K-token layer) and must record nothing and
give exactly the normal build's results; a case whose device-side sequence table contradicts the host's
shows the device check firing.
"""
import ctypes

import pytest
import torch

from gated_deltanet_linear_03_gb300 import synth
from helpers import to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def libs():
    from gated_deltanet_linear_03_gb300 import _build, gdn
    gdn.load_library()
    dbg = gdn.bind(_build.build(debug=True))
    assert gdn.device_error() == 0 and gdn.device_error(lib=dbg) == 0
    return gdn, dbg


def both(gdn, dbg, fn):
    """fn(lib) under the normal and the checking build; the results must be identical and nothing recorded."""
    ref = fn(None)
    got = fn(dbg)
    torch.cuda.synchronize()
    assert gdn.device_error(lib=dbg) == 0, "the bounds-checking build recorded an out-of-range access"
    for a, b in zip(ref, got):
        if a is not None:
            assert torch.equal(a, b)


CASES = {
    "ragged": lambda: synth.prefill_inputs([1, 63, 64, 65, 130, 0, 7], seed=101, init_std=0.02),
    "group3_gates": lambda: synth.prefill_inputs([77, 1], hk=1, hv=3, seed=102, raw_gates="per_head"),
    "short_many": lambda: synth.prefill_inputs([32, 5, 17, 1, 32, 9, 30, 2], seed=103, init_std=0.02),
    "raw_qk_norm": lambda: synth.prefill_inputs([200, 3, 64], seed=104, init_std=0.02, raw_qk=True),
}


@pytest.mark.parametrize("algo", ["chunked", "scan"])
@pytest.mark.parametrize("case", list(CASES))
def test_prefill_paths_record_nothing(libs, case, algo):
    gdn, dbg = libs
    inp = CASES[case]()
    d = to_device(inp)
    kw = dict(init_state=d.init_state, out_dtype=torch.float32, algo=algo, cu_seqlens_host=inp.cu_seqlens.tolist())
    if inp.gate_scale is not None:
        kw.update(gate_scale=inp.gate_scale.cuda(), gate_bias=inp.gate_bias.cuda())
    if case == "raw_qk_norm":
        kw.update(qk_norm=True, q_scale=0.088, norm_weight=torch.linspace(0.5, 2.0, 128, device="cuda"))
    both(gdn, dbg, lambda lib: gdn.prefill(d.q, d.k, d.v, d.log_alpha, d.beta, d.cu_seqlens, lib=lib, **kw))


def test_long_layer_records_nothing(libs):
    gdn, dbg = libs
    inp = synth.prefill_inputs([131072], seed=105, device="cuda")
    both(gdn, dbg, lambda lib: gdn.prefill(inp.q, inp.k, inp.v, inp.log_alpha, inp.beta, inp.cu_seqlens.cuda(),
                                           algo="chunked", cu_seqlens_host=[0, 131072], lib=lib))


def test_decode_records_nothing(libs):
    gdn, dbg = libs
    di = synth.decode_inputs(3, 1, seed=106, raw_gates="per_head")
    args = [x[0].cuda() for x in (di.q, di.k, di.v, di.log_alpha, di.beta)]
    w = torch.linspace(0.5, 2.0, 128, device="cuda")
    g = dict(gate_scale=di.gate_scale.cuda(), gate_bias=di.gate_bias.cuda())
    for kw in ({}, dict(norm_weight=w), dict(qk_norm=True, q_scale=0.1, **g)):
        def step(lib):
            st = di.state.cuda()
            out = gdn.decode_step(st, *args, out_dtype=torch.float32, lib=lib, **kw)
            return out, st
        both(gdn, dbg, step)


def test_device_check_fires_on_a_contradicting_sequence_table(libs):
    """cu_seqlens on the device says [0, 1, 128] while the host copy says [0, 64, 128]: the launch is planned
    for 2 chunks but the device table needs 3.  The state pass finds the second sequence's chunks beyond the
    planned range, records GDN_ERR_INTERNAL and skips it; nothing out of range is touched."""
    gdn, dbg = libs
    inp = synth.prefill_inputs([64, 64], hk=2, hv=4, seed=107)
    d = to_device(inp)
    bad = torch.tensor([0, 1, 128], dtype=torch.int32, device="cuda")
    for lib in (None, dbg):
        gdn.prefill(d.q, d.k, d.v, d.log_alpha, d.beta, bad, algo="chunked", cu_seqlens_host=[0, 64, 128], lib=lib)
        assert gdn.device_error(lib=lib) == 6   # GDN_ERR_INTERNAL, then cleared
        assert gdn.device_error(lib=lib) == 0
