"""GPU parity of the fused output normalisation (o / sqrt(mean(o^2) + eps) * w per head) against the fp64
oracle.  Normalised outputs are O(1), so they are compared in fp32 against the 2e-3 bound, and in bf16
against the bf16 rounding of the reference (relative 2^-8)."""
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


def weight(d, seed):
    gen = torch.Generator().manual_seed(seed)
    return 0.5 + 1.5 * torch.rand(d, generator=gen)


def bf16_ok(out, ref):
    ref = np.asarray(ref, np.float64)
    return np.all(np.abs(np32(out).astype(np.float64) - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-3)


# d = 128: one 512-thread CTA per head; d = 64: one 128-thread CTA per head; d = 32: one warp per head,
# including a batch whose rows leave the last CTA partly empty (n * hv * 32 not a multiple of 128)
@pytest.mark.parametrize("d,hk,hv,n", [(128, 16, 32, 30), (128, 2, 4, 1), (64, 2, 4, 3), (32, 2, 2, 5), (32, 1, 1, 3)])
@pytest.mark.parametrize("qk_norm", [False, True])
def test_decode_with_output_norm(gdn, d, hk, hv, n, qk_norm):
    steps = 3
    di = synth.decode_inputs(n, steps, hk=hk, hv=hv, dk=d, dv=d, seed=60 + d, raw_qk=qk_norm)
    w = weight(d, 61)
    scale = 1.0 / np.sqrt(d) if qk_norm else 1.0
    st_gpu = di.state.cuda()
    st_ref = di.state.double().numpy()
    for s in range(steps):
        args = [x[s] for x in (di.q, di.k, di.v, di.log_alpha, di.beta)]
        dev = [a.cuda() for a in args]
        out = gdn.decode_step(st_gpu, *dev, out_dtype=torch.float32, qk_norm=qk_norm, q_scale=scale,
                              norm_weight=w.cuda(), norm_eps=1e-6)
        o_ref, st_ref = oracle.decode_step(st_ref, *[np32(a) for a in args], qk_norm=qk_norm, q_scale=scale,
                                           norm_weight=w.numpy(), norm_eps=1e-6)
        torch.cuda.synchronize()
        assert max_abs_err(out, o_ref) <= OUT_ATOL
        assert state_rel_err(st_gpu, st_ref) <= STATE_RTOL


def test_decode_output_norm_bf16(gdn):
    di = synth.decode_inputs(30, 1, seed=62)
    w = weight(128, 63)
    st = di.state.cuda()
    args = [x[0] for x in (di.q, di.k, di.v, di.log_alpha, di.beta)]
    out = gdn.decode_step(st, *[a.cuda() for a in args], norm_weight=w.cuda())
    o_ref, _ = oracle.decode_step(di.state.double().numpy(), *[np32(a) for a in args], norm_weight=w.numpy())
    torch.cuda.synchronize()
    assert bf16_ok(out, o_ref)


PREFILL_CASES = {
    # lengths, algo, d: the chunked pass (cluster of 4 slices, per-chunk exchange, partial last chunks and a
    # 1-token sequence), the register scan (cluster of d/16 slices, per 64-token block), the streaming scan
    # (a batch of short sequences: cluster of 4 for d = 128, one CTA per head below)
    "chunked_ragged": ([200, 1, 64, 130], "chunked", 128),
    "chunked_T64": ([64], "chunked", 128),
    "scan_long": ([150, 70], "scan", 128),
    "scan_single_short": ([8], "scan", 128),
    "scan_short_batch": ([5, 32, 1, 17, 9, 0, 3, 12], "scan", 128),
    "scan_long_d64": ([100, 37], "scan", 64),
    "scan_short_batch_d64": ([5, 2, 17, 9], "scan", 64),
    "scan_long_d32": ([90, 3], "scan", 32),
    "scan_short_batch_d32": ([8, 3, 1, 5, 2, 7, 4, 6], "scan", 32),
}


@pytest.mark.parametrize("case", list(PREFILL_CASES))
@pytest.mark.parametrize("qk_norm", [False, True])
def test_prefill_with_output_norm(gdn, case, qk_norm):
    lengths, algo, d = PREFILL_CASES[case]
    hk, hv = (16, 32) if d == 128 else (8, 32)
    inp = synth.prefill_inputs(lengths, hk=hk, hv=hv, dk=d, dv=d, seed=64, init_std=0.02, raw_qk=qk_norm)
    w = weight(d, 65)
    scale = 1.0 / np.sqrt(d) if qk_norm else 1.0
    kw = dict(qk_norm=qk_norm, q_scale=scale, norm_weight=w.numpy(), norm_eps=1e-6)
    from helpers import oracle_args, to_device, check_prefill
    ref_out, ref_fin = oracle.prefill(*oracle_args(inp), **kw)
    dv_ = to_device(inp)
    kw["norm_weight"] = w.cuda()
    out, fin = gdn.prefill(dv_.q, dv_.k, dv_.v, dv_.log_alpha, dv_.beta, dv_.cu_seqlens, init_state=dv_.init_state,
                           out_dtype=torch.float32, algo=algo, cu_seqlens_host=inp.cu_seqlens.tolist(), **kw)
    torch.cuda.synchronize()
    check_prefill(out, fin, ref_out, ref_fin, what=f"{case} qk_norm={qk_norm}")


def test_prefill_output_norm_noalloc_and_phases(gdn):
    from helpers import oracle_args, to_device, check_prefill
    inp = synth.prefill_inputs([300, 5], seed=66, init_std=0.02)
    w = weight(128, 67)
    ref_out, ref_fin = oracle.prefill(*oracle_args(inp), norm_weight=w.numpy())
    d = to_device(inp)
    cu = inp.cu_seqlens.tolist()
    out, fin = gdn.prefill_noalloc(d.q, d.k, d.v, d.log_alpha, d.beta, d.cu_seqlens, init_state=d.init_state,
                                   out_dtype=torch.float32, cu_seqlens_host=cu, norm_weight=w.cuda())
    torch.cuda.synchronize()
    check_prefill(out, fin, ref_out, ref_fin, what="noalloc norm")
    plan = gdn.PrefillPlan(d.q, d.k, d.v, d.log_alpha, d.beta, d.cu_seqlens, init_state=d.init_state,
                           out_dtype=torch.float32, cu_seqlens_host=cu, norm_weight=w.cuda())
    plan.run_phase("prep")
    plan.run_phase("pass")
    torch.cuda.synchronize()
    check_prefill(plan.out, plan.final_state, ref_out, ref_fin, what="phases norm")


# The chunked pass carries the norm in every form the host can pick: many short sequences (several per CTA,
# with raw gates: the multi-sequence, gated instantiation), eight long ones (one sequence per CTA: 1024
# four-CTA clusters over several waves), both with raw q/k and bf16 outputs as a model would run them.
NORM_PASS_FORMS = {
    "many_short_raw_gates": ([37, 0, 129, 64, 1, 300, 65, 2, 90, 17, 250, 3], dict(raw_gates="per_head")),
    "eight_long": ([600, 520, 700, 513, 640, 600, 530, 610], {}),
}


@pytest.mark.parametrize("form", list(NORM_PASS_FORMS))
def test_chunked_norm_every_pass_form(gdn, form):
    lengths, extra = NORM_PASS_FORMS[form]
    inp = synth.prefill_inputs(lengths, seed=68, init_std=0.02, raw_qk=True, **extra)
    w = weight(128, 69)
    kw = dict(qk_norm=True, q_scale=1.0 / np.sqrt(128), norm_weight=w.numpy(), norm_eps=1e-6)
    gk = {}
    if inp.gate_scale is not None:
        kw.update(gate_scale=inp.gate_scale.numpy(), gate_bias=inp.gate_bias.numpy())
        gk = dict(gate_scale=inp.gate_scale.cuda(), gate_bias=inp.gate_bias.cuda())
    from helpers import oracle_args, to_device
    ref_out, ref_fin = oracle.prefill(*oracle_args(inp), **kw)
    dv_ = to_device(inp)
    kw.update(norm_weight=w.cuda(), **gk)
    out, fin = gdn.prefill(dv_.q, dv_.k, dv_.v, dv_.log_alpha, dv_.beta, dv_.cu_seqlens, init_state=dv_.init_state,
                           out_dtype=torch.bfloat16, algo="chunked", cu_seqlens_host=inp.cu_seqlens.tolist(), **kw)
    torch.cuda.synchronize()
    assert gdn.device_error() == 0
    assert bf16_ok(out, ref_out), f"{form}: bf16 normalised outputs"
    assert state_rel_err(fin, ref_fin) <= STATE_RTOL, f"{form}: final state"
