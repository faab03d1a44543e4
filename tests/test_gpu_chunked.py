"""GPU parity of the chunked (tcgen05) prefill against the fp64 oracle, through the C ABI.

Cases span several chunks and ragged tails (lengths that are not multiples of
64, empty sequences, one-token sequences), sequence buckets (one state-pass CTA
carrying several sequences one after another), both head groupings the kernels
specialise on, slow-decay gates that make the carried state matter, and the
full model-shaped workloads (4K exhaustively; 128K and the ragged 8-sequence
batch on sampled heads, where the oracle checks every token of those heads).
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_linear_03_gb300 import synth
from gated_deltanet_linear_03_gb300.synth import PrefillInputs
from helpers import (OUT_ATOL, STATE_RTOL, as_bf16_inputs, check_prefill, max_abs_err, oracle_args,
                     state_rel_err, to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gdn():
    from gated_deltanet_linear_03_gb300 import gdn as g
    g.load_library()
    return g


def run(gdn, inp, algo="chunked", out_dtype=torch.bfloat16):
    d = to_device(inp)
    out, fin = gdn.prefill(d.q, d.k, d.v, d.log_alpha, d.beta, d.cu_seqlens, init_state=d.init_state,
                           out_dtype=out_dtype, algo=algo, cu_seqlens_host=inp.cu_seqlens.tolist())
    torch.cuda.synchronize()
    assert gdn.device_error() == 0
    return out, fin


CASES = {
    "T200": lambda: synth.prefill_inputs([200], seed=31),
    "ragged_init": lambda: synth.prefill_inputs([1, 63, 64, 65, 130, 0, 7], seed=32, init_std=0.02),
    "slow_T1024_S1": lambda: synth.prefill_inputs([1024], seed=33, gates="slow"),
    "slow_ragged_S2": lambda: synth.prefill_inputs([100, 257, 31, 700], seed=34, gates="slow", init_std=0.02),
    "group1": lambda: synth.prefill_inputs([150, 90], hk=4, hv=4, seed=35, init_std=0.05),
    "group4": lambda: synth.prefill_inputs([129, 64], hk=2, hv=8, seed=36, init_std=0.05),
    "group3_odd": lambda: synth.prefill_inputs([77], hk=1, hv=3, seed=37, init_std=0.05),
    # 8 value heads: the state pass runs 4 buckets of consecutive sequences, each CTA carrying the state
    # through several sequences (empty ones first, in the middle and last), with slow decay and initial states
    "buckets_many_seqs": lambda: synth.prefill_inputs([0, 1, 63, 64, 65, 0, 130, 7, 200, 0, 2, 64, 0], hk=2, hv=8,
                                                      seed=38, gates="slow", init_std=0.05),
}


@pytest.mark.parametrize("case", list(CASES))
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_chunked_matches_oracle(gdn, case, out_dtype):
    inp = CASES[case]()
    ref_out, ref_fin = oracle.prefill(*oracle_args(inp))
    out, fin = run(gdn, inp, "chunked", out_dtype)
    check_prefill(out, fin, ref_out, ref_fin, what=case)


def pad_heads(inp: PrefillInputs, d: int = 128) -> PrefillInputs:
    """Zero-pad q/k/v and the state to head size d: the recurrence on the padded
    problem equals the original on the first dims and is zero elsewhere."""
    def pad(x, dims):
        shape = list(x.shape)
        for ax in dims:
            shape[ax] = d
        y = torch.zeros(shape, dtype=x.dtype)
        sl = tuple(slice(0, s) for s in x.shape)
        y[sl] = x
        return y
    s0 = None if inp.init_state is None else pad(inp.init_state, [-1, -2])
    return PrefillInputs(pad(inp.q, [-1]), pad(inp.k, [-1]), pad(inp.v, [-1]), inp.log_alpha, inp.beta, s0,
                         inp.cu_seqlens)


def test_tiny_case_via_zero_padding(gdn):
    """The 64-token, 2-head, d=32 case (fp32 draws rounded to bf16), run by the d=128 chunked kernels."""
    inp = as_bf16_inputs(synth.tiny_case())
    ref_out, ref_fin = oracle.prefill(*oracle_args(inp))
    out, fin = run(gdn, pad_heads(inp), "chunked", torch.float32)
    assert torch.count_nonzero(out[..., 32:]).item() == 0
    assert torch.count_nonzero(fin[..., 32:, :]).item() == 0 and torch.count_nonzero(fin[..., 32:]).item() == 0
    check_prefill(out[..., :32].contiguous(), fin[..., :32, :32].contiguous(), ref_out, ref_fin, what="tiny")


def test_split_prompt_composes(gdn):
    """prefill(T) == prefill(T1) then prefill(T - T1) from its final state (also across chunk borders)."""
    inp = synth.prefill_inputs([300], seed=38, init_std=0.02)
    out, fin = run(gdn, inp, "chunked", torch.float32)
    for t1 in (64, 100):
        a = PrefillInputs(inp.q[:t1], inp.k[:t1], inp.v[:t1], inp.log_alpha[:t1], inp.beta[:t1], inp.init_state,
                          torch.tensor([0, t1], dtype=torch.int32))
        o1, f1 = run(gdn, a, "chunked", torch.float32)
        b = PrefillInputs(inp.q[t1:], inp.k[t1:], inp.v[t1:], inp.log_alpha[t1:], inp.beta[t1:], f1.cpu(),
                          torch.tensor([0, 300 - t1], dtype=torch.int32))
        o2, f2 = run(gdn, b, "chunked", torch.float32)
        assert (torch.cat([o1, o2]) - out).abs().max().item() < 1e-4
        assert ((f2 - fin).norm() / fin.norm()).item() < 1e-5


def test_in_place_state_and_empty_batch(gdn):
    inp = synth.prefill_inputs([90, 0, 40], seed=39, init_std=0.05)
    ref_out, ref_fin = oracle.prefill(*oracle_args(inp))
    d = to_device(inp)
    st = d.init_state.clone()
    out, fin = gdn.prefill(d.q, d.k, d.v, d.log_alpha, d.beta, d.cu_seqlens, init_state=st, final_state=st,
                           algo="chunked", out_dtype=torch.float32)
    torch.cuda.synchronize()
    check_prefill(out, st, ref_out, ref_fin, what="in-place")
    # all sequences empty: final state is the initial state
    e = synth.prefill_inputs([0, 0], seed=40, init_std=0.05)
    de = to_device(e)
    out, fin = gdn.prefill(de.q, de.k, de.v, de.log_alpha, de.beta, de.cu_seqlens, init_state=de.init_state,
                           algo="chunked")
    torch.cuda.synchronize()
    assert out.shape[0] == 0 and torch.equal(fin, de.init_state)


def test_alpha_zero_and_identity_gates(gdn):
    """log_alpha = -inf resets (GPU clamps it at -20); log_alpha = 0, beta = 0 keeps the state."""
    inp = synth.prefill_inputs([130], hk=2, hv=4, seed=41, init_std=0.05)
    inp.log_alpha[::7] = -float("inf")
    ref_out, ref_fin = oracle.prefill(*oracle_args(inp))
    out, fin = run(gdn, inp, "chunked", torch.float32)
    check_prefill(out, fin, ref_out, ref_fin, what="alpha=0")
    inp.log_alpha.zero_()
    inp.beta.zero_()
    out, fin = run(gdn, inp, "chunked", torch.float32)
    assert ((fin.cpu() - inp.init_state).norm() / inp.init_state.norm()).item() < 1e-5


def test_prefill_4k_full(gdn):
    """Single-layer prefill at the model shape: T=4096, 16 q/k heads, 32 v heads, d=128."""
    inp = synth.prefill_4k()
    ref_out, ref_fin = oracle.prefill(*oracle_args(inp))
    out, fin = run(gdn, inp, "chunked")
    e = check_prefill(out, fin, ref_out, ref_fin, what="4k chunked")
    out2, fin2 = run(gdn, inp, "scan")
    check_prefill(out2, fin2, ref_out, ref_fin, what="4k scan")
    print("4k chunked errors", e)


def sampled_heads(inp: PrefillInputs, heads):
    """Inputs restricted to some value heads (with the q/k heads they read)."""
    T, hk, dk = inp.q.shape
    hv = inp.v.shape[1]
    g = hv // hk
    qh = [h // g for h in heads]
    s0 = None if inp.init_state is None else inp.init_state[:, heads]
    return (inp.q[:, qh].float().numpy(), inp.k[:, qh].float().numpy(), inp.v[:, heads].float().numpy(),
            inp.log_alpha[:, heads].numpy(), inp.beta[:, heads].numpy(), inp.cu_seqlens.numpy(),
            None if s0 is None else s0.double().numpy())


@pytest.fixture(scope="module")
def full_size():
    """The two full-size workloads with the oracle's outputs and final states on three value heads."""
    heads = [0, 17, 31]
    cases = {}
    for which in ("long_128k", "ragged_8"):
        inp = getattr(synth, which)()
        q, k, v, la, b, cu, s0 = sampled_heads(inp, heads)
        # each sampled v head with its own q/k head: hk = hv = len(heads)
        cases[which] = (inp, oracle.prefill(q, k, v, la, b, cu, s0))
    return heads, cases


@pytest.mark.parametrize("algo", ["chunked", "scan"])
@pytest.mark.parametrize("which", ["long_128k", "ragged_8"])
def test_full_size_sampled_heads(gdn, full_size, which, algo):
    heads, cases = full_size
    inp, (ref_out, ref_fin) = cases[which]
    out, fin = run(gdn, inp, algo)
    check_prefill(out[:, heads].contiguous(), fin[:, heads].contiguous(), ref_out, ref_fin,
                  what=f"{which} {algo}")


@pytest.mark.parametrize("lengths", [
    [600] * 70,                           # 70 sequences of 10 chunks: one state-pass CTA per sequence (beyond the
                                          # 64-entry bucket table: the first chunks come from cu_seqlens)
    [40, 0, 1, 64, 65, 0, 129] * 10,      # 70 short ones: one CTA carries them all, empty ones included
])
def test_many_sequences_bucket_layouts(gdn, lengths):
    heads = [0, 13, 31]
    inp = synth.prefill_inputs(lengths, seed=1301 + len(set(lengths)), init_std=0.02)
    ref_out, ref_fin = oracle.prefill(*sampled_heads(inp, heads))
    out, fin = run(gdn, inp, "chunked", torch.float32)
    check_prefill(out[:, heads].contiguous(), fin[:, heads].contiguous(), ref_out, ref_fin,
                  what=f"{len(lengths)} sequences")


def test_long_128k_then_decode(gdn, full_size):
    """The long-context case end to end: the 128K-token prefill emits its final state, and 64 batch-1
    decode steps continue from it in place.  Sampled heads follow the oracle's own continuation from the
    oracle's final state; both paths' final states agree with each other as well."""
    heads, cases = full_size
    inp, (_, ref_fin) = cases["long_128k"]
    out_c, fin_c = run(gdn, inp, "chunked")
    _, fin_s = run(gdn, inp, "scan")
    assert state_rel_err(fin_c[:, heads], ref_fin) <= STATE_RTOL
    diff = (fin_c - fin_s).flatten(2).norm(dim=-1) / fin_s.flatten(2).norm(dim=-1)
    assert diff.max().item() <= 2 * STATE_RTOL
    steps = 64
    di = synth.decode_inputs(1, steps, seed=1006)
    qh = [h // (inp.v.shape[1] // inp.q.shape[1]) for h in heads]
    state = fin_c.clone()
    ref = np.asarray(ref_fin, np.float64)
    for t in range(steps):
        args = (di.q[t], di.k[t], di.v[t], di.log_alpha[t], di.beta[t])
        o = gdn.decode_step(state, *[x.cuda() for x in args], out_dtype=torch.float32)
        o_ref, ref = oracle.decode_step(ref, di.q[t][:, qh].float().numpy(), di.k[t][:, qh].float().numpy(),
                                        di.v[t][:, heads].float().numpy(), di.log_alpha[t][:, heads].numpy(),
                                        di.beta[t][:, heads].numpy())
        torch.cuda.synchronize()
        assert max_abs_err(o[:, heads].contiguous(), o_ref) <= OUT_ATOL, t
    assert state_rel_err(state[:, heads].contiguous(), ref) <= STATE_RTOL
