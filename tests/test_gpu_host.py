"""gdn_prefill_host: the prefill on inputs and outputs in host memory (copies in, kernels, copies out, all
enqueued by the library).  Its results must match the fp64 oracle and be bit-identical to gdn_prefill run on
device copies of the same inputs; two plans alternated on two streams must not disturb each other."""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_linear_03_gb300 import synth
from helpers import check_prefill, oracle_args, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gdn():
    from gated_deltanet_linear_03_gb300 import gdn as g
    g.load_library()
    return g


def host_args(inp, pinned=True):
    def h(t):
        t = t.contiguous()
        return t.pin_memory() if pinned else t.clone()
    return [h(x) for x in (inp.q, inp.k, inp.v, inp.log_alpha, inp.beta)], \
        (None if inp.init_state is None else h(inp.init_state.float()))


def device_reference(gdn, inp, algo, out_dtype):
    d = to_device(inp)
    out, fin = gdn.prefill(d.q, d.k, d.v, d.log_alpha, d.beta, d.cu_seqlens, init_state=d.init_state,
                           out_dtype=out_dtype, algo=algo, cu_seqlens_host=inp.cu_seqlens.tolist())
    torch.cuda.synchronize()
    return out.cpu(), fin.cpu()


@pytest.mark.parametrize("algo", ["chunked", "scan", "auto"])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("pinned", [True, False])
def test_host_call_matches_oracle_and_device_call(gdn, algo, out_dtype, pinned):
    inp = synth.prefill_inputs([150, 1, 0, 77], seed=81, init_std=0.02)
    (q, k, v, la, b), s0 = host_args(inp, pinned)
    out, fin = gdn.prefill_host(q, k, v, la, b, inp.cu_seqlens.tolist(), init_state=s0, out_dtype=out_dtype,
                                algo=algo)
    assert not out.is_cuda and not fin.is_cuda
    ref_out, ref_fin = oracle.prefill(*oracle_args(inp))
    check_prefill(out, fin, ref_out, ref_fin, what=f"host {algo}")
    dev_out, dev_fin = device_reference(gdn, inp, "chunked" if algo == "auto" else algo, out_dtype)
    assert torch.equal(out, dev_out) and torch.equal(fin, dev_fin)
    assert gdn.device_error() == 0


def test_host_call_without_init_or_final_state(gdn):
    inp = synth.prefill_inputs([130], seed=82)
    (q, k, v, la, b), _ = host_args(inp)
    out, fin = gdn.prefill_host(q, k, v, la, b, [0, 130], final_state=False)
    assert fin is None
    dev_out, _ = device_reference(gdn, inp, "chunked", torch.bfloat16)
    assert torch.equal(out, dev_out)


def test_host_call_empty_batch_returns_initial_state(gdn):
    inp = synth.prefill_inputs([0, 0], seed=83, init_std=0.02)
    (q, k, v, la, b), s0 = host_args(inp)
    out, fin = gdn.prefill_host(q, k, v, la, b, [0, 0, 0], init_state=s0, algo="scan")
    assert out.numel() == 0
    assert torch.equal(fin, s0)


def test_two_plans_alternated_on_two_streams(gdn):
    """Two problems, each with its own staging, run alternately on two streams several times: the copies
    of one overlap the other's kernels, and each keeps producing its own results."""
    inputs = [synth.prefill_inputs([300, 45], seed=84, init_std=0.02), synth.prefill_inputs([200], seed=85)]
    plans, refs = [], []
    for inp in inputs:
        (q, k, v, la, b), s0 = host_args(inp)
        plans.append(gdn.HostPrefillPlan(q, k, v, la, b, inp.cu_seqlens.tolist(), init_state=s0))
        refs.append(device_reference(gdn, inp, "chunked", torch.bfloat16))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for _ in range(3):
        for p, s in zip(plans, streams):
            p.run(s)
    torch.cuda.synchronize()
    for p, (ref_out, ref_fin) in zip(plans, refs):
        assert torch.equal(p.out, ref_out) and torch.equal(p.final_state, ref_fin)
    assert plans[0].h2d_bytes == sum(t.numel() * t.element_size() for t in plans[0].tensors[:6]) + 12
    assert plans[0].d2h_bytes == 345 * 32 * 128 * 2 + 2 * 32 * 128 * 128 * 4


def test_host_call_with_query_key_preparation_and_output_norm(gdn):
    """The host call forwards the in-kernel options: raw q/k normalised in the kernels, output norm fused."""
    inp = synth.prefill_inputs([150, 90], seed=86, init_std=0.02, raw_qk=True)
    (q, k, v, la, b), s0 = host_args(inp)
    w = torch.linspace(0.5, 2.0, 128)
    scale = 1.0 / np.sqrt(128)
    out, fin = gdn.prefill_host(q, k, v, la, b, inp.cu_seqlens.tolist(), init_state=s0, out_dtype=torch.float32,
                                qk_norm=True, q_scale=scale, norm_weight=w.cuda(), norm_eps=1e-6)
    ref_out, ref_fin = oracle.prefill(*oracle_args(inp), qk_norm=True, q_scale=scale, norm_weight=w.numpy(),
                                      norm_eps=1e-6)
    check_prefill(out, fin, ref_out, ref_fin, what="host with options")
