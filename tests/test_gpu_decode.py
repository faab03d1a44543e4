"""GPU parity of gdn_decode_step against the fp64 oracle (through the C ABI)."""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_linear_03_gb300 import synth
from helpers import OUT_ATOL, STATE_RTOL, max_abs_err, np32, state_rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gdn():
    from gated_deltanet_linear_03_gb300 import gdn as g
    g.load_library()
    return g


@pytest.mark.parametrize("d,hk,hv,n", [(128, 16, 32, 30), (64, 2, 4, 3), (32, 2, 2, 5)])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_decode_chain_matches_oracle(gdn, d, hk, hv, n, out_dtype):
    steps = 4
    di = synth.decode_inputs(n, steps, hk=hk, hv=hv, dk=d, dv=d, seed=7 + d)
    st_gpu = di.state.cuda()
    st_ref = di.state.double().numpy()
    for s in range(steps):
        args = [x[s] for x in (di.q, di.k, di.v, di.log_alpha, di.beta)]
        out = gdn.decode_step(st_gpu, *[a.cuda() for a in args], out_dtype=out_dtype)
        o_ref, st_ref = oracle.decode_step(st_ref, *[np32(a) for a in args])
        torch.cuda.synchronize()
        assert max_abs_err(out, o_ref) <= OUT_ATOL
        assert state_rel_err(st_gpu, st_ref) <= STATE_RTOL


def test_decode_identity_gate_is_bit_exact(gdn):
    """alpha = 1, beta = 0 leaves the state unchanged bit for bit."""
    n, d = 3, 128
    di = synth.decode_inputs(n, 1, seed=11)
    st = di.state.cuda()
    before = st.clone()
    la = torch.zeros(n, 32, device="cuda")
    b = torch.zeros(n, 32, device="cuda")
    out = gdn.decode_step(st, di.q[0].cuda(), di.k[0].cuda(), di.v[0].cuda(), la, b, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(st, before)
    # o = S q exactly up to fp32 rounding of the dot product
    qe = di.q[0].float().repeat_interleave(2, dim=1).cuda()
    ref = torch.einsum("nhij,nhj->nhi", before.double(), qe.double())
    assert (out.double() - ref).abs().max().item() < 1e-5


def test_decode_zero_batch_is_noop(gdn):
    st = torch.zeros(0, 32, 128, 128, device="cuda")
    e = torch.zeros(0, 16, 128, device="cuda", dtype=torch.bfloat16)
    v = torch.zeros(0, 32, 128, device="cuda", dtype=torch.bfloat16)
    g = torch.zeros(0, 32, device="cuda")
    out = gdn.decode_step(st, e, e, v, g, g)
    assert out.shape == (0, 32, 128)


def test_decode_30_layers_256_steps(gdn):
    """The full decode workload: 30 layer states (32 v heads x 128 x 128 fp32), 256 chained steps with fresh
    bf16 inputs, bf16 outputs.  Three sampled layers follow the oracle through every step; the error must not
    grow past the tolerance over the chain."""
    steps = 256
    di = synth.decode_30(steps=steps)
    layers = [0, 13, 29]
    st_gpu = di.state.cuda()
    q, k, v, la, b = (x.cuda() for x in (di.q, di.k, di.v, di.log_alpha, di.beta))
    outs = []
    for s in range(steps):
        outs.append(gdn.decode_step(st_gpu, q[s], k[s], v[s], la[s], b[s]))
    torch.cuda.synchronize()
    st_ref = di.state[layers].double().numpy()
    worst = 0.0
    for s in range(steps):
        args = [np32(x[s][layers]) for x in (di.q, di.k, di.v, di.log_alpha, di.beta)]
        o_ref, st_ref = oracle.decode_step(st_ref, *args)
        worst = max(worst, max_abs_err(outs[s][layers], o_ref))
    assert worst <= OUT_ATOL, worst
    assert state_rel_err(st_gpu[layers], st_ref) <= STATE_RTOL
