"""Pins of the fp64 CPU oracle against facts fixed by the definition itself.

The recurrence (per value head, state S of shape dv x dk):
    S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,   o_t = S_t q_t,
is the gated delta update that "Optimizing on-device inference for Apple
Silicon" describes in words (section "Qwen creates three workload shapes").
None of these checks re-types the oracle's expanded update; each uses a
closed form, an invariant, a hand-worked example or a differently arranged
brute-force formula, chosen so that a dropped term, a wrong sign, an index
slip or a transposed operand fails at least one of them.  Shapes use dk != dv
so that a transposed state cannot pass.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def rand_case(rng, T, hk=1, hv=1, dk=3, dv=5, unit_k=True, init=True, gates="mixed"):
    q = rng.standard_normal((T, hk, dk)).astype(np.float32)
    k = rng.standard_normal((T, hk, dk)).astype(np.float32)
    if unit_k:
        k = (k / np.linalg.norm(k, axis=-1, keepdims=True)).astype(np.float32)
    v = rng.standard_normal((T, hv, dv)).astype(np.float32)
    if gates == "mixed":
        la = (-np.log1p(np.exp(rng.standard_normal((T, hv))))).astype(np.float32)
        b = (1 / (1 + np.exp(-rng.standard_normal((T, hv))))).astype(np.float32)
    else:
        la, b = gates
    s0 = rng.standard_normal((1, hv, dv, dk)) if init else None
    return q, k, v, la, b, s0


def one_seq(T):
    return np.array([0, T], np.int32)


# ---------------------------------------------------------------- worked example (hand-derived)

def test_worked_example_by_hand():
    g = json.load(open(os.path.join(HERE, "golden", "worked_example_d2.json")))
    q = np.array(g["q"], np.float32)[:, None, :]
    k = np.array(g["k"], np.float32)[:, None, :]
    v = np.array(g["v"], np.float32)[:, None, :]
    la = np.log(np.array(g["alpha"], np.float64)).astype(np.float32)[:, None]
    b = np.array(g["beta"], np.float32)[:, None]
    out, fin = oracle.prefill(q, k, v, la, b, one_seq(3))
    np.testing.assert_allclose(out[:, 0, :], np.array(g["out"]), atol=1e-6)
    np.testing.assert_allclose(fin[0, 0], np.array(g["final_state"]), atol=1e-6)


# ---------------------------------------------------------------- P1: alpha = 1, beta = 0

def test_identity_gate_keeps_state():
    rng = np.random.default_rng(1)
    T = 9
    q, k, v, _, _, s0 = rand_case(rng, T)
    la = np.zeros((T, 1), np.float32)
    b = np.zeros((T, 1), np.float32)
    out, fin = oracle.prefill(q, k, v, la, b, one_seq(T), s0)
    assert np.array_equal(fin, s0)
    np.testing.assert_allclose(out[:, 0, :], (s0[0, 0] @ q[:, 0, :].T.astype(np.float64)).T, atol=1e-13)


# ---------------------------------------------------------------- P2: alpha = 0 resets the state

def test_zero_alpha_resets_to_rank_one():
    rng = np.random.default_rng(2)
    T = 6
    q, k, v, _, b, s0 = rand_case(rng, T)
    la = np.full((T, 1), -np.inf, np.float32)
    out, fin = oracle.prefill(q, k, v, la, b, one_seq(T), s0)
    kk = k[:, 0, :].astype(np.float64)
    qq = q[:, 0, :].astype(np.float64)
    vv = v[:, 0, :].astype(np.float64)
    bb = b[:, 0].astype(np.float64)
    np.testing.assert_allclose(fin[0, 0], bb[-1] * np.outer(vv[-1], kk[-1]), atol=1e-13)
    expect_o = bb[:, None] * vv * np.sum(kk * qq, axis=1)[:, None]
    np.testing.assert_allclose(out[:, 0, :], expect_o, atol=1e-13)


# ---------------------------------------------------------------- P3: beta = 1, unit key => S_t k_t = v_t

@pytest.mark.parametrize("T", [1, 2, 5, 11])
def test_full_beta_writes_value_exactly(T):
    rng = np.random.default_rng(3 + T)
    q, k, v, la, _, s0 = rand_case(rng, T)
    b = np.ones((T, 1), np.float32)
    kk = k[:, 0, :].astype(np.float64)
    # unit norm in fp64 terms for the check (k is fp32-rounded; renormalise exactly representable)
    _, fin = oracle.prefill(q, k, v, la, b, one_seq(T), s0)
    nk = float(kk[-1] @ kk[-1])
    # S_T k_T = alpha S (k - k (k.k)) + v (k.k) = v when |k| = 1; allow for the fp32 rounding of |k|
    resid = fin[0, 0] @ kk[-1] - v[-1, 0].astype(np.float64)
    assert np.max(np.abs(resid)) < 1e-6 * (1 + np.max(np.abs(fin)))
    assert abs(nk - 1) < 1e-6


# ---------------------------------------------------------------- P4: literal matrix form

def literal(q, k, v, la, b, s0, group=1):
    T, hk, dk = q.shape
    hv, dv = v.shape[1], v.shape[2]
    out = np.zeros((T, hv, dv))
    fin = np.zeros((1, hv, dv, dk))
    for h in range(hv):
        S = np.zeros((dv, dk)) if s0 is None else s0[0, h].copy()
        for t in range(T):
            kt = k[t, h // group].astype(np.float64)[:, None]
            vt = v[t, h].astype(np.float64)[:, None]
            a = math.exp(float(la[t, h]))
            G = np.eye(dk) - float(b[t, h]) * (kt @ kt.T)
            S = a * (S @ G) + float(b[t, h]) * (vt @ kt.T)
            out[t, h] = S @ q[t, h // group].astype(np.float64)
        fin[0, h] = S
    return out, fin


def test_literal_matrix_form_matches():
    rng = np.random.default_rng(4)
    T = 13
    q, k, v, la, b, s0 = rand_case(rng, T, hk=2, hv=4, dk=3, dv=5, unit_k=False)
    out, fin = oracle.prefill(q, k, v, la, b, one_seq(T), s0)
    ref_o, ref_s = literal(q, k, v, la, b, s0, group=2)
    np.testing.assert_allclose(out, ref_o, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(fin, ref_s, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- P5: splitting the prompt keeps the output

@pytest.mark.parametrize("T1", [0, 1, 7, 16, 20])
def test_split_prefill_composes(T1):
    rng = np.random.default_rng(5)
    T = 20
    q, k, v, la, b, s0 = rand_case(rng, T, hk=1, hv=2, dk=4, dv=3)
    out, fin = oracle.prefill(q, k, v, la, b, one_seq(T), s0)
    o1, f1 = oracle.prefill(q[:T1], k[:T1], v[:T1], la[:T1], b[:T1], one_seq(T1), s0)
    o2, f2 = oracle.prefill(q[T1:], k[T1:], v[T1:], la[T1:], b[T1:], one_seq(T - T1), f1)
    np.testing.assert_allclose(np.concatenate([o1, o2]), out, atol=1e-13)
    np.testing.assert_allclose(f2, fin, atol=1e-13)


# ---------------------------------------------------------------- P6: chunked form equals the scan

@pytest.mark.parametrize("C", [1, 2, 4, 8, 16, 32, 64])
@pytest.mark.parametrize("T", [1, 5, 64, 70, 131])
def test_chunked_equals_sequential(C, T):
    rng = np.random.default_rng(1000 * C + T)
    q, k, v, la, b, s0 = rand_case(rng, T, hk=1, hv=2, dk=8, dv=6)
    out, fin = oracle.prefill(q, k, v, la, b, one_seq(T), s0)
    oc, fc = oracle.prefill_chunked(q, k, v, la, b, one_seq(T), s0, chunk=C)
    np.testing.assert_allclose(oc, out, rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(fc, fin, rtol=1e-10, atol=1e-11)


def test_chunked_ragged_equals_sequential():
    rng = np.random.default_rng(61)
    lens = [3, 64, 0, 77, 1]
    T = sum(lens)
    q, k, v, la, b, _ = rand_case(rng, T, hk=2, hv=4, dk=8, dv=8, init=False)
    s0 = rng.standard_normal((len(lens), 4, 8, 8))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    out, fin = oracle.prefill(q, k, v, la, b, cu, s0)
    oc, fc = oracle.prefill_chunked(q, k, v, la, b, cu, s0, chunk=16)
    np.testing.assert_allclose(oc, out, rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(fc, fin, rtol=1e-10, atol=1e-11)


# ---------------------------------------------------------------- P7: linearity in (S0, V)

def test_linear_in_state_and_values():
    rng = np.random.default_rng(7)
    T = 17
    q, k, v, la, b, s0 = rand_case(rng, T, dk=4, dv=3)
    # values on a 1/256 grid, so that a1*v + a2*v2 below is exact in fp32
    v = (np.round(v * 256) / 256).astype(np.float32)
    v2 = (np.round(rng.standard_normal(v.shape) * 256) / 256).astype(np.float32)
    s02 = rng.standard_normal(s0.shape)
    a1, a2 = 0.5, -2.0
    o1, f1 = oracle.prefill(q, k, v, la, b, one_seq(T), s0)
    o2, f2 = oracle.prefill(q, k, v2, la, b, one_seq(T), s02)
    vm = (a1 * v.astype(np.float64) + a2 * v2.astype(np.float64))
    assert np.array_equal(vm.astype(np.float32).astype(np.float64), vm)
    om, fm = oracle.prefill(q, k, vm.astype(np.float32), la, b, one_seq(T), a1 * s0 + a2 * s02)
    np.testing.assert_allclose(om, a1 * o1 + a2 * o2, atol=1e-12)
    np.testing.assert_allclose(fm, a1 * f1 + a2 * f2, atol=1e-12)


# ---------------------------------------------------------------- P8: orthonormal keys, closed form

def test_orthonormal_keys_closed_form():
    rng = np.random.default_rng(8)
    dk, dv, T = 6, 4, 6
    perm = rng.permutation(dk)
    k = np.zeros((T, 1, dk), np.float32)
    k[np.arange(T), 0, perm[:T]] = 1.0
    q = rng.standard_normal((T, 1, dk)).astype(np.float32)
    v = rng.standard_normal((T, 1, dv)).astype(np.float32)
    la = (-np.log1p(np.exp(rng.standard_normal((T, 1))))).astype(np.float32)
    b = (1 / (1 + np.exp(-rng.standard_normal((T, 1))))).astype(np.float32)
    s0 = rng.standard_normal((1, 1, dv, dk))
    out, fin = oracle.prefill(q, k, v, la, b, one_seq(T), s0)
    alpha = np.exp(la[:, 0].astype(np.float64))
    beta = b[:, 0].astype(np.float64)
    # column j is touched only at the token t* whose key is e_j:
    #   before t*: c <- alpha c ; at t*: c <- alpha (1 - beta) c + beta v ; after: c <- alpha c
    expect = np.zeros((dv, dk))
    for j in range(dk):
        hits = np.nonzero(perm[:T] == j)[0]
        decay = np.prod(alpha)
        if hits.size == 0:
            expect[:, j] = decay * s0[0, 0, :, j]
        else:
            ts = int(hits[0])
            after = np.prod(alpha[ts + 1:])
            expect[:, j] = decay * (1 - beta[ts]) * s0[0, 0, :, j] + beta[ts] * after * v[ts, 0]
    np.testing.assert_allclose(fin[0, 0], expect, atol=1e-13)


# ---------------------------------------------------------------- P9: parallel (sum over sources) form

def test_parallel_form_brute_force():
    rng = np.random.default_rng(9)
    dk, dv, T = 3, 4, 7
    q, k, v, la, b, s0 = rand_case(rng, T, dk=dk, dv=dv, unit_k=False)
    out, fin = oracle.prefill(q, k, v, la, b, one_seq(T), s0)
    k64, v64 = k.astype(np.float64), v.astype(np.float64)
    G = [math.exp(float(la[r, 0])) * (np.eye(dk) - float(b[r, 0]) * np.outer(k64[r, 0], k64[r, 0]))
         for r in range(T)]

    def prod(lo, hi):  # G_lo G_{lo+1} ... G_hi (right-multiplied transitions)
        P = np.eye(dk)
        for r in range(lo, hi + 1):
            P = P @ G[r]
        return P

    for t in range(T):
        St = s0[0, 0] @ prod(0, t)
        for s in range(t + 1):
            St = St + float(b[s, 0]) * np.outer(v64[s, 0], k64[s, 0]) @ prod(s + 1, t)
        np.testing.assert_allclose(out[t, 0], St @ q[t, 0].astype(np.float64), atol=1e-12)
        if t == T - 1:
            np.testing.assert_allclose(fin[0, 0], St, atol=1e-12)


# ---------------------------------------------------------------- query/key preparation (qk_norm, q_scale)

def test_qk_norm_single_token_by_hand():
    """dk = 2, S0 = 0, one token: S = beta v k_n^T and o = S q_n with k_n = k / sqrt(|k|^2 + 1e-6)."""
    q = np.array([[[1.0, 2.0]]], np.float32)
    k = np.array([[[3.0, 4.0]]], np.float32)
    v = np.array([[[2.0, -1.0, 0.5]]], np.float32)
    la = np.array([[0.0]], np.float32)
    b = np.array([[0.5]], np.float32)
    scale = 0.25
    out, fin = oracle.prefill(q, k, v, la, b, one_seq(1), qk_norm=True, q_scale=scale)
    kn = np.array([3.0, 4.0]) / math.sqrt(25.0 + 1e-6)
    qn = np.array([1.0, 2.0]) / math.sqrt(5.0 + 1e-6) * scale
    S = 0.5 * np.outer([2.0, -1.0, 0.5], kn)
    np.testing.assert_allclose(fin[0, 0], S, rtol=1e-14)
    np.testing.assert_allclose(out[0, 0], S @ qn, rtol=1e-14)


@pytest.mark.parametrize("path", ["prefill", "chunked", "decode"])
def test_qk_norm_ignores_the_length_of_q_and_k(path):
    """With qk_norm, rescaling any token's q or k by a positive factor changes nothing (up to the 1e-6
    floor under the norm, kept negligible here by norms far above it)."""
    rng = np.random.default_rng(40)
    T = 9
    q, k, v, la, b, s0 = rand_case(rng, T, hk=2, hv=4, dk=6, dv=5, unit_k=False)
    cq = rng.uniform(0.5, 4.0, (T, 2, 1)).astype(np.float32)
    ck = rng.uniform(0.5, 4.0, (T, 2, 1)).astype(np.float32)
    def run(qq, kk):
        if path == "prefill":
            return oracle.prefill(qq, kk, v, la, b, one_seq(T), s0, qk_norm=True, q_scale=0.3)
        if path == "chunked":
            return oracle.prefill_chunked(qq, kk, v, la, b, one_seq(T), s0, chunk=4, qk_norm=True, q_scale=0.3)
        st0 = np.repeat(s0, T, axis=0)   # T independent states, one token each
        return oracle.decode_step(st0, qq, kk, v, la, b, qk_norm=True, q_scale=0.3)
    o1, f1 = run(q, k)
    o2, f2 = run(q * cq, k * ck)   # the rescaled inputs are rounded to fp32: agreement to ~1e-7 relative
    np.testing.assert_allclose(o2, o1, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(f2, f1, rtol=1e-5, atol=1e-6)


def test_qk_norm_on_unit_vectors_is_the_plain_recurrence():
    rng = np.random.default_rng(41)
    T = 7
    q, k, v, la, b, s0 = rand_case(rng, T, hk=1, hv=2, dk=5, dv=3)
    q = (q / np.linalg.norm(q, axis=-1, keepdims=True)).astype(np.float32)
    o1, f1 = oracle.prefill(q, k, v, la, b, one_seq(T), s0)
    o2, f2 = oracle.prefill(q, k, v, la, b, one_seq(T), s0, qk_norm=True)
    # 1/sqrt(|x|^2 + 1e-6) differs from 1 by ~5e-7 (plus the fp32 rounding of the unit vectors)
    np.testing.assert_allclose(o2, o1, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(f2, f1, rtol=1e-5, atol=1e-6)


def test_q_scale_scales_outputs_only():
    """o = S q is linear in q; the state never reads q."""
    rng = np.random.default_rng(42)
    T = 6
    q, k, v, la, b, s0 = rand_case(rng, T, hk=1, hv=2, dk=4, dv=3)
    o1, f1 = oracle.prefill(q, k, v, la, b, one_seq(T), s0)
    o2, f2 = oracle.prefill(q, k, v, la, b, one_seq(T), s0, q_scale=0.125)
    np.testing.assert_array_equal(f2, f1)
    np.testing.assert_allclose(o2, 0.125 * o1, rtol=1e-13, atol=1e-15)


def test_chunked_with_qk_norm_equals_sequential():
    rng = np.random.default_rng(43)
    T = 23
    q, k, v, la, b, s0 = rand_case(rng, T, hk=1, hv=2, dk=5, dv=4, unit_k=False)
    o1, f1 = oracle.prefill(q, k, v, la, b, one_seq(T), s0, qk_norm=True, q_scale=0.5)
    o2, f2 = oracle.prefill_chunked(q, k, v, la, b, one_seq(T), s0, chunk=8, qk_norm=True, q_scale=0.5)
    np.testing.assert_allclose(o2, o1, rtol=1e-9, atol=1e-10)
    np.testing.assert_allclose(f2, f1, rtol=1e-9, atol=1e-10)


# ---------------------------------------------------------------- output normalisation

def test_output_norm_by_hand():
    """o = (3, 4): mean of squares 12.5; with eps 0.5 the divisor is sqrt(13) = 3.6055..."""
    o = np.array([[3.0, 4.0]])
    got = oracle.rms_norm(o, np.array([2.0, -1.0]), 0.5)
    np.testing.assert_allclose(got, [[6.0 / math.sqrt(13.0), -4.0 / math.sqrt(13.0)]], rtol=1e-15)


def test_output_norm_properties():
    """With unit weight the normalised output has mean square ms/(ms + eps); scaling v (so o) by c > 0
    leaves it unchanged up to eps; the state never depends on the norm."""
    rng = np.random.default_rng(44)
    T = 6
    q, k, v, la, b, s0 = rand_case(rng, T, hk=1, hv=2, dk=4, dv=5)
    s0 = None
    raw, f0 = oracle.prefill(q, k, v, la, b, one_seq(T), s0)
    o1, f1 = oracle.prefill(q, k, v, la, b, one_seq(T), s0, norm_weight=np.ones(5), norm_eps=1e-9)
    ms = (raw ** 2).mean(axis=-1)
    np.testing.assert_allclose((o1 ** 2).mean(axis=-1), ms / (ms + 1e-9), rtol=1e-12)
    np.testing.assert_array_equal(f1, f0)
    o2, _ = oracle.prefill(q, k, (v * 3.0).astype(np.float32), la, b, one_seq(T), s0, norm_weight=np.ones(5),
                           norm_eps=1e-9)
    np.testing.assert_allclose(o2, o1, rtol=1e-6, atol=1e-7)
    w = rng.uniform(0.5, 2.0, 5)
    o3, _ = oracle.prefill(q, k, v, la, b, one_seq(T), s0, norm_weight=w, norm_eps=1e-9)
    np.testing.assert_allclose(o3, o1 * w, rtol=1e-13)


def test_output_norm_decode_matches_prefill():
    rng = np.random.default_rng(45)
    q, k, v, la, b, s0 = rand_case(rng, 1, hk=1, hv=2, dk=4, dv=4)
    w = rng.uniform(0.5, 2.0, 4)
    o_p, f_p = oracle.prefill(q, k, v, la, b, one_seq(1), s0, norm_weight=w)
    o_d, f_d = oracle.decode_step(s0, q, k, v, la, b, norm_weight=w)
    np.testing.assert_allclose(o_d, o_p, rtol=1e-14)
    np.testing.assert_array_equal(f_d, f_p)


# ---------------------------------------------------------------- decode, packing, grouping

def test_decode_chain_equals_prefill():
    rng = np.random.default_rng(10)
    T = 5
    q, k, v, la, b, s0 = rand_case(rng, T, hk=2, hv=4, dk=4, dv=3)
    out, fin = oracle.prefill(q, k, v, la, b, one_seq(T), s0)
    st = s0.copy()
    for t in range(T):
        o, st = oracle.decode_step(st, q[t:t + 1], k[t:t + 1], v[t:t + 1], la[t:t + 1], b[t:t + 1])
        np.testing.assert_array_equal(o[0], out[t])
    np.testing.assert_array_equal(st, fin)


def test_decode_batch_is_independent():
    rng = np.random.default_rng(11)
    n = 3
    q, k, v, la, b, _ = rand_case(rng, n, hk=1, hv=2, dk=4, dv=4)
    st = rng.standard_normal((n, 2, 4, 4))
    o, s1 = oracle.decode_step(st, q, k, v, la, b)
    for i in range(n):
        oi, si = oracle.decode_step(st[i:i + 1], q[i:i + 1], k[i:i + 1], v[i:i + 1], la[i:i + 1], b[i:i + 1])
        np.testing.assert_array_equal(o[i], oi[0])
        np.testing.assert_array_equal(s1[i], si[0])


def test_ragged_equals_separate_calls():
    rng = np.random.default_rng(12)
    lens = [4, 0, 9, 1]
    T = sum(lens)
    q, k, v, la, b, _ = rand_case(rng, T, hk=1, hv=2, dk=3, dv=2, init=False)
    s0 = rng.standard_normal((len(lens), 2, 2, 3))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    out, fin = oracle.prefill(q, k, v, la, b, cu, s0)
    for n in range(len(lens)):
        a, e = cu[n], cu[n + 1]
        o, f = oracle.prefill(q[a:e], k[a:e], v[a:e], la[a:e], b[a:e], one_seq(e - a), s0[n:n + 1])
        np.testing.assert_array_equal(out[a:e], o)
        np.testing.assert_array_equal(fin[n], f[0])


def test_group_mapping_is_repeat_interleave():
    rng = np.random.default_rng(13)
    T = 6
    q, k, v, la, b, s0 = rand_case(rng, T, hk=2, hv=6, dk=3, dv=2)
    out, fin = oracle.prefill(q, k, v, la, b, one_seq(T), s0)
    qe, ke = np.repeat(q, 3, axis=1), np.repeat(k, 3, axis=1)
    o2, f2 = oracle.prefill(qe, ke, v, la, b, one_seq(T), s0)
    np.testing.assert_array_equal(out, o2)
    np.testing.assert_array_equal(fin, f2)


def test_zero_length_sequence_passes_state_through():
    rng = np.random.default_rng(14)
    q, k, v, la, b, _ = rand_case(rng, 0, hk=1, hv=1)
    s0 = rng.standard_normal((2, 1, 5, 3))
    out, fin = oracle.prefill(q, k, v, la, b, np.array([0, 0, 0], np.int32), s0)
    assert out.shape == (0, 1, 5)
    np.testing.assert_array_equal(fin, s0)


# ---------------------------------------------------------------- planted mistakes are caught

def test_pins_catch_a_planted_mistake():
    """A forgotten alpha inside the delta (S <- aS + b(v - S k)k^T) must fail the closed form."""
    rng = np.random.default_rng(15)
    T = 5
    q, k, v, la, b, s0 = rand_case(rng, T, dk=4, dv=3)
    S = s0[0, 0].copy()
    for t in range(T):
        a = math.exp(float(la[t, 0]))
        kt = k[t, 0].astype(np.float64)
        S = a * S + float(b[t, 0]) * np.outer(v[t, 0] - S @ kt, kt)  # the planted slip
    _, fin = oracle.prefill(q, k, v, la, b, one_seq(T), s0)
    _, ref = literal(q, k, v, la, b, s0)
    np.testing.assert_allclose(fin, ref, atol=1e-12)
    assert np.max(np.abs(S - ref[0, 0])) > 1e-3


# ---------------------------------------------------------------- gates computed from raw inputs
# log_alpha = -c_h softplus(a + b_h), beta = sigmoid(y) (the configured workloads' gate recipe with per-head
# parameters).  A one-token step from S0 = e_0 e_1^T with k = e_0 and q = e_1 gives, by hand,
#     S1 = alpha S0 (I - beta e_0 e_0^T) + beta v e_0^T = [[0, alpha], [beta v_1 ... ]]
# (S0 e_0 = 0), so S1[0, 1] = alpha and, with v = e_1, S1[1, 0] = beta: the gates can be read off the state.

def _gate_probe(a, y, c, b):
    """alpha and beta the oracle applies for raw inputs a, y (arrays [n]) and head parameters c, b."""
    n = len(a)
    s0 = np.zeros((n, 1, 2, 2))
    s0[:, 0, 0, 1] = 1.0
    e0 = np.tile(np.array([1, 0], np.float32), (n, 1, 1))
    e1 = np.tile(np.array([0, 1], np.float32), (n, 1, 1))
    la = np.asarray(a, np.float32).reshape(n, 1)
    bt = np.asarray(y, np.float32).reshape(n, 1)
    out, s1 = oracle.decode_step(s0, e1, e0, e1, la, bt, gate_scale=np.array([c], np.float32),
                                 gate_bias=np.array([b], np.float32))
    np.testing.assert_array_equal(s1[:, 0, 0, 0], 0.0)
    np.testing.assert_allclose(out[:, 0, 0], s1[:, 0, 0, 1], rtol=1e-15)   # o = S1 e_1: (alpha, 0)
    return s1[:, 0, 0, 1], s1[:, 0, 1, 0]


def test_gates_by_hand():
    # softplus(ln(e - 1)) = 1 and sigmoid(ln 3) = 3/4; softplus(0) = ln 2 and sigmoid(0) = 1/2
    a = np.float32(math.log(math.e - 1.0))
    alpha, beta = _gate_probe([a, 0.0], [math.log(3.0), 0.0], 0.5, 0.0)
    np.testing.assert_allclose(alpha[0], math.exp(-0.5 * math.log1p(math.exp(float(a)))), rtol=1e-14)
    np.testing.assert_allclose(alpha[0], math.exp(-0.5), rtol=1e-6)       # a is ln(e - 1) rounded to fp32
    np.testing.assert_allclose(beta[0], 0.75, rtol=1e-7)                  # ln 3 rounded to fp32
    np.testing.assert_allclose(alpha[1], 2.0 ** -0.5, rtol=1e-15)         # exp(-0.5 ln 2)
    np.testing.assert_allclose(beta[1], 0.5, rtol=1e-15)
    # the bias shifts the argument: a + b = 0 with b = 3
    alpha, _ = _gate_probe([-3.0], [0.0], 2.0, 3.0)
    np.testing.assert_allclose(alpha[0], 0.25, rtol=1e-15)                # exp(-2 ln 2)


def test_gates_tails():
    # softplus(x) -> x for large x, -> e^x for very negative x (kept, not rounded to 0)
    alpha, beta = _gate_probe([30.0, -40.0], [40.0, -40.0], 0.5, 0.0)
    np.testing.assert_allclose(alpha[0], math.exp(-0.5 * (30.0 + math.exp(-30.0))), rtol=1e-14)
    np.testing.assert_allclose(beta[0], 1.0, rtol=1e-15)
    np.testing.assert_allclose(beta[1], math.exp(-40.0), rtol=1e-6)
    # a large scale makes the small-x tail visible in alpha: -log alpha = c softplus(-30) = c e^-30 (1 - ...)
    alpha, _ = _gate_probe([-30.0], [0.0], 1.0e6, 0.0)
    np.testing.assert_allclose(-math.log(alpha[0]), 1.0e6 * math.log1p(math.exp(-30.0)), rtol=1e-8)
    np.testing.assert_allclose(-math.log(alpha[0]), 1.0e6 * math.exp(-30.0), rtol=1e-8)


def test_gates_are_in_range_and_monotone():
    rng = np.random.default_rng(5)
    a = np.sort(rng.standard_normal(64).astype(np.float32) * 4)
    y = np.sort(rng.standard_normal(64).astype(np.float32) * 4)
    alpha, beta = _gate_probe(a, y, 0.7, 1.3)
    assert np.all(alpha > 0) and np.all(alpha <= 1) and np.all(beta > 0) and np.all(beta < 1)
    assert np.all(np.diff(alpha) <= 0) and np.all(np.diff(beta) >= 0)    # alpha falls with a, beta rises with y
    alpha0, _ = _gate_probe(a, y, 0.0, 1.3)
    np.testing.assert_array_equal(alpha0, 1.0)                            # c = 0: nothing decays


def test_gates_reproduce_the_configured_recipe():
    """With c = 0.5, b = 2 (model) or c = 1, b = 0 (tiny) the map is the configs' own gate recipe, drawn by the
    input generator with a library softplus/sigmoid on the same normal variates."""
    from gated_deltanet_linear_03_gb300 import synth
    for kind, kw in (("model", dict(hk=2, hv=4, dk=8, dv=8)), ("tiny", dict(hk=2, hv=2, dk=8, dv=8))):
        fin_gates = synth.prefill_inputs([50, 30], seed=11, gates=kind, init_std=0.1, **kw)
        raw = synth.prefill_inputs([50, 30], seed=11, gates=kind, init_std=0.1, raw_gates="config", **kw)
        args = lambda x: (x.q.float().numpy(), x.k.float().numpy(), x.v.float().numpy())
        cu = raw.cu_seqlens.numpy()
        s0 = raw.init_state.double().numpy()
        o1, f1 = oracle.prefill(*args(fin_gates), fin_gates.log_alpha.numpy(), fin_gates.beta.numpy(), cu, s0)
        o2, f2 = oracle.prefill(*args(raw), raw.log_alpha.numpy(), raw.beta.numpy(), cu, s0,
                                gate_scale=raw.gate_scale.numpy(), gate_bias=raw.gate_bias.numpy())
        # the generator's gates are fp32 values of the same map: agreement to fp32 rounding of the gates
        np.testing.assert_allclose(o2, o1, rtol=2e-5, atol=2e-6)
        np.testing.assert_allclose(f2, f1, rtol=2e-5, atol=2e-6)


def test_gates_decode_chain_equals_prefill():
    from gated_deltanet_linear_03_gb300 import synth
    inp = synth.prefill_inputs([40], hk=2, hv=4, dk=8, dv=8, seed=12, init_std=0.1, raw_gates="per_head")
    g = dict(gate_scale=inp.gate_scale.numpy(), gate_bias=inp.gate_bias.numpy())
    q, k, v = inp.q.float().numpy(), inp.k.float().numpy(), inp.v.float().numpy()
    out, fin = oracle.prefill(q, k, v, inp.log_alpha.numpy(), inp.beta.numpy(), inp.cu_seqlens.numpy(),
                              inp.init_state.double().numpy(), **g)
    st = inp.init_state.double().numpy()
    for t in range(40):
        o, st = oracle.decode_step(st, q[t:t + 1], k[t:t + 1], v[t:t + 1], inp.log_alpha.numpy()[t:t + 1],
                                   inp.beta.numpy()[t:t + 1], **g)
        np.testing.assert_allclose(o[0], out[t], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(st, fin, rtol=1e-12, atol=1e-14)
