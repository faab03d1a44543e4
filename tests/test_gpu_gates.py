"""GPU parity of the gates computed inside the kernels, through the C ABI.

With gate_scale / gate_bias the log_alpha and beta arrays carry each token's raw
projections a and y, and every kernel forms log_alpha = -c_h softplus(a + b_h)
and beta = sigmoid(y) where it loads them (the configured workloads' gate recipe
with per-value-head parameters; the state and its gate stay fp32, "Optimizing
on-device inference for Apple Silicon", section "Keep recurrent state on chip").
Each path is compared with the fp64 oracle given the same raw inputs and
parameters, at the tolerances of the other parity tests.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_linear_03_gb300 import synth
from helpers import OUT_ATOL, STATE_RTOL, check_prefill, max_abs_err, np32, oracle_args, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gdn():
    from gated_deltanet_linear_03_gb300 import gdn as g
    g.load_library()
    return g


def gate_kw(inp, dev="cuda"):
    return dict(gate_scale=inp.gate_scale.to(dev), gate_bias=inp.gate_bias.to(dev))


def oracle_ref(inp, **kw):
    return oracle.prefill(*oracle_args(inp), gate_scale=inp.gate_scale.numpy(), gate_bias=inp.gate_bias.numpy(),
                          **kw)


CASES = {
    # (lengths, kwargs of synth.prefill_inputs)
    "chunked_ragged": ([1, 63, 64, 65, 200, 0, 7], dict(hk=4, hv=8, seed=81, init_std=0.02, raw_gates="per_head")),
    "chunked_4k_config": ([4096], dict(seed=82, raw_gates="config")),
    "group3": ([150], dict(hk=1, hv=3, seed=83, init_std=0.05, raw_gates="per_head")),
}


@pytest.mark.parametrize("algo", ["chunked", "scan"])
@pytest.mark.parametrize("case", list(CASES))
def test_prefill_gates_match_oracle(gdn, case, algo):
    lengths, kw = CASES[case]
    inp = synth.prefill_inputs(lengths, **kw)
    ref_out, ref_fin = oracle_ref(inp)
    d = to_device(inp)
    out, fin = gdn.prefill(d.q, d.k, d.v, d.log_alpha, d.beta, d.cu_seqlens, init_state=d.init_state,
                           out_dtype=torch.float32, algo=algo, cu_seqlens_host=inp.cu_seqlens.tolist(), **gate_kw(inp))
    torch.cuda.synchronize()
    assert gdn.device_error() == 0
    check_prefill(out, fin, ref_out, ref_fin, what=f"{case}/{algo}")


@pytest.mark.parametrize("d", [32, 64])
def test_scan_gates_small_heads(gdn, d):
    inp = synth.prefill_inputs([90, 33], hk=2, hv=4, dk=d, dv=d, seed=84, init_std=0.05, raw_gates="per_head")
    ref_out, ref_fin = oracle_ref(inp)
    x = to_device(inp)
    out, fin = gdn.prefill(x.q, x.k, x.v, x.log_alpha, x.beta, x.cu_seqlens, init_state=x.init_state,
                           out_dtype=torch.float32, algo="scan", cu_seqlens_host=inp.cu_seqlens.tolist(),
                           **gate_kw(inp))
    torch.cuda.synchronize()
    check_prefill(out, fin, ref_out, ref_fin, what=f"scan d={d}")


def test_short_sequences_row_streaming_scan_gates(gdn):
    """At most 32 tokens per sequence and more than one wave of 16-row CTAs: the row-streaming scan."""
    inp = synth.prefill_inputs([32, 5, 17, 1, 32, 9, 30, 2], seed=85, init_std=0.02, raw_gates="per_head")
    ref_out, ref_fin = oracle_ref(inp)
    x = to_device(inp)
    out, fin = gdn.prefill(x.q, x.k, x.v, x.log_alpha, x.beta, x.cu_seqlens, init_state=x.init_state,
                           out_dtype=torch.float32, algo="scan", cu_seqlens_host=inp.cu_seqlens.tolist(),
                           **gate_kw(inp))
    torch.cuda.synchronize()
    check_prefill(out, fin, ref_out, ref_fin, what="short scan")


def test_chunked_gates_with_qk_preparation(gdn):
    """Raw q/k projections and raw gates together: every input of the layer prepared inside the kernels."""
    inp = synth.prefill_inputs([300, 77], seed=86, init_std=0.02, raw_qk=True, raw_gates="per_head")
    scale = 1.0 / np.sqrt(128)
    ref_out, ref_fin = oracle_ref(inp, qk_norm=True, q_scale=scale)
    x = to_device(inp)
    for algo in ("chunked", "scan"):
        out, fin = gdn.prefill(x.q, x.k, x.v, x.log_alpha, x.beta, x.cu_seqlens, init_state=x.init_state,
                               out_dtype=torch.float32, algo=algo, cu_seqlens_host=inp.cu_seqlens.tolist(),
                               qk_norm=True, q_scale=scale, **gate_kw(inp))
        torch.cuda.synchronize()
        check_prefill(out, fin, ref_out, ref_fin, what=f"qk+gates {algo}")


def test_gates_agree_with_precomputed_gates(gdn):
    """The same layer with the gates finished by the caller (the oracle's map, rounded to fp32) and with the
    gates formed in the kernels: both meet the oracle, and they differ from each other by fp32 gate rounding
    only."""
    inp = synth.prefill_inputs([500], hk=4, hv=8, seed=87, init_std=0.02, raw_gates="per_head")
    c = inp.gate_scale.double().numpy()
    b = inp.gate_bias.double().numpy()
    a = inp.log_alpha.double().numpy()
    y = inp.beta.double().numpy()
    x = a + b
    la = torch.from_numpy((-c * (np.maximum(x, 0) + np.log1p(np.exp(-np.abs(x))))).astype(np.float32))
    bt = torch.from_numpy((1 / (1 + np.exp(-y))).astype(np.float32))
    d = to_device(inp)
    cu = inp.cu_seqlens.tolist()
    o1, f1 = gdn.prefill(d.q, d.k, d.v, d.log_alpha, d.beta, d.cu_seqlens, init_state=d.init_state,
                         out_dtype=torch.float32, cu_seqlens_host=cu, **gate_kw(inp))
    o2, f2 = gdn.prefill(d.q, d.k, d.v, la.cuda(), bt.cuda(), d.cu_seqlens, init_state=d.init_state,
                         out_dtype=torch.float32, cu_seqlens_host=cu)
    torch.cuda.synchronize()
    assert (o1 - o2).abs().max().item() <= 1e-4
    assert ((f1 - f2).flatten(2).norm(dim=-1) / f2.flatten(2).norm(dim=-1)).max().item() <= 1e-5


def test_decode_chain_with_gates(gdn):
    di = synth.decode_inputs(3, 16, seed=88, raw_gates="per_head")
    st = di.state.cuda()
    ref = di.state.double().numpy()
    g = dict(gate_scale=di.gate_scale.numpy(), gate_bias=di.gate_bias.numpy())
    for t in range(16):
        args = [x[t] for x in (di.q, di.k, di.v, di.log_alpha, di.beta)]
        out = gdn.decode_step(st, *[a.cuda() for a in args], out_dtype=torch.float32,
                              gate_scale=di.gate_scale.cuda(), gate_bias=di.gate_bias.cuda())
        o_ref, ref = oracle.decode_step(ref, *[np32(a) for a in args], **g)
        torch.cuda.synchronize()
        assert max_abs_err(out, o_ref) <= OUT_ATOL
    rel = np.sqrt(((np32(st) - ref) ** 2).sum(axis=(-1, -2))) / np.sqrt((ref ** 2).sum(axis=(-1, -2)))
    assert rel.max() <= STATE_RTOL


def test_noalloc_and_host_calls_with_gates(gdn):
    inp = synth.prefill_inputs([200, 65], hk=4, hv=8, seed=89, init_std=0.02, raw_gates="per_head")
    d = to_device(inp)
    cu = inp.cu_seqlens.tolist()
    ref_out, ref_fin = gdn.prefill(d.q, d.k, d.v, d.log_alpha, d.beta, d.cu_seqlens, init_state=d.init_state,
                                   out_dtype=torch.float32, cu_seqlens_host=cu, **gate_kw(inp))
    out, fin = gdn.prefill_noalloc(d.q, d.k, d.v, d.log_alpha, d.beta, d.cu_seqlens, init_state=d.init_state,
                                   out_dtype=torch.float32, cu_seqlens_host=cu, **gate_kw(inp))
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out) and torch.equal(fin, ref_fin)
    hq = [t.contiguous().pin_memory() for t in (inp.q, inp.k, inp.v, inp.log_alpha, inp.beta)]
    out_h, fin_h = gdn.prefill_host(*hq, cu, init_state=inp.init_state.pin_memory(), out_dtype=torch.float32,
                                    algo="chunked", **gate_kw(inp))
    assert torch.equal(out_h, ref_out.cpu()) and torch.equal(fin_h, ref_fin.cpu())
