"""CPU rounding model of the GPU's blocked (chunked) arithmetic, checked against the fp64 oracle.

The chunked kernels do not evaluate the textbook W/U form: they fold the triangular inverse into two
state-independent matrices per chunk ("Optimizing on-device inference for Apple Silicon", section "Qwen
creates three workload shapes": blocks that expose matrix operations), with g the running log-decay,
Gamma_i = e^{g_L - g_i} and T = (I + strict_lower(beta_i e^{g_i - g_j} k_i.k_j))^-1:

    P = K^T diag(Gamma) T,   R = lower_incl(e^{g_i - g_j} q_i.k_j) T
    X = diag(beta) V - diag(beta e^g) K S0^T
    O = diag(e^g) Q S0^T + R X,   S_L^T = e^{g_L} S0^T + P X

This module restates that form in numpy (float64), with optional rounding of P, R, X and the state
operand S exactly where the kernels round them: a bf16 hi part taken by truncation (the low 16 bits of
the fp32 value dropped) plus a round-to-nearest bf16 lo part, or a single bf16.  It pins:
  * the reformulated algebra itself (no rounding) against the sequential oracle;
  * the kernels' rounding (hi + lo everywhere) far inside the stated tolerance;
  * that storing P as one bf16 would break the 1e-3 state tolerance, which is why the kernels keep
    the split on everything that feeds the carried state.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_linear_03_gb300 import synth
from helpers import STATE_RTOL, oracle_args


def _bf16_rn(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64)).to(torch.bfloat16).double().numpy()


def _bf16_trunc(x):
    bits = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) & np.uint32(0xFFFF0000)
    return bits.view(np.float32).astype(np.float64)


def _split(x):
    """hi (truncated bf16) + lo (round-to-nearest bf16 of the fp32 remainder), as the kernels form it."""
    x32 = np.asarray(x, dtype=np.float32).astype(np.float64)
    hi = _bf16_trunc(x32)
    return hi + _bf16_rn(x32 - hi)


ROUND = {"none": lambda x: x, "split": _split, "bf16": _bf16_rn}


def blocked_prefill(inp, heads, *, p="none", rest="none", C=64):
    """Outputs and final states of the listed value heads by the kernels' blocked form.  `p` rounds P;
    `rest` rounds R, X and the state operand S."""
    q, k, v, la, b, cu, s0 = oracle_args(inp)
    T, hk, d = q.shape
    hv = v.shape[1]
    grp = hv // hk
    rp, rr = ROUND[p], ROUND[rest]
    out = np.zeros((T, hv, d))
    fin = np.zeros((len(cu) - 1, hv, d, d))
    for n in range(len(cu) - 1):
        for h in heads:
            S = np.zeros((d, d)) if s0 is None else s0[n, h].copy()   # rows: value index, columns: key index
            for t0 in range(cu[n], cu[n + 1], C):
                L = min(C, cu[n + 1] - t0)
                K = k[t0:t0 + L, h // grp].astype(np.float64)
                Q = q[t0:t0 + L, h // grp].astype(np.float64)
                V = v[t0:t0 + L, h].astype(np.float64)
                bt = b[t0:t0 + L, h].astype(np.float64)
                g = np.cumsum(np.clip(la[t0:t0 + L, h].astype(np.float64), -20.0, 0.0))
                decay = np.exp(np.minimum(g[:, None] - g[None, :], 0.0))
                Tm = np.linalg.inv(np.eye(L) + np.tril(bt[:, None] * decay * (K @ K.T), -1))
                P = rp(K.T @ (np.exp(g[-1] - g)[:, None] * Tm))
                R = rr(np.tril(decay * (Q @ K.T)) @ Tm)
                Sop = rr(S)
                X = rr(bt[:, None] * V - (bt * np.exp(g))[:, None] * (K @ Sop.T))
                out[t0:t0 + L, h] = np.exp(g)[:, None] * (Q @ Sop.T) + R @ X
                S = np.exp(g[-1]) * S + (P @ X).T
            fin[n, h] = S
    return out, fin


def _errors(inp, heads, **kw):
    ref_out, ref_fin = oracle.prefill(*oracle_args(inp))
    out, fin = blocked_prefill(inp, heads, **kw)
    hs = list(heads)
    e_out = float(np.abs(out[:, hs] - ref_out[:, hs]).max())
    diff = np.sqrt(((fin[:, hs] - ref_fin[:, hs]) ** 2).sum(axis=(-1, -2)))
    norm = np.sqrt((ref_fin[:, hs] ** 2).sum(axis=(-1, -2)))
    return e_out, float((diff / np.maximum(norm, 1e-30)).max())


CASES = {
    # the model's gates, 1024 tokens; slow decay (the carried state matters); ragged with initial states,
    # empty and one-token sequences and partial chunks
    "model_gates": (lambda: synth.prefill_inputs([1024], seed=41), (0, 17)),
    "slow_decay": (lambda: synth.prefill_inputs([1024], seed=33, gates="slow"), (0, 9)),
    "ragged_init": (lambda: synth.prefill_inputs([64, 1, 0, 129, 63, 7, 66], seed=31, init_std=0.02), (3, 30)),
}


@pytest.mark.parametrize("case", list(CASES))
def test_blocked_algebra_equals_the_sequential_scan(case):
    make, heads = CASES[case]
    e_out, e_state = _errors(make(), heads)
    assert e_out < 1e-9 and e_state < 1e-9, (e_out, e_state)


@pytest.mark.parametrize("case", list(CASES))
def test_kernel_rounding_stays_far_inside_the_tolerance(case):
    make, heads = CASES[case]
    e_out, e_state = _errors(make(), heads, p="split", rest="split")
    assert e_state < STATE_RTOL / 50 and e_out < 1e-4, (e_out, e_state)


@pytest.mark.parametrize("case", ["model_gates", "slow_decay"])
def test_single_bf16_p_breaks_the_state_tolerance(case):
    """The tolerance holds per head; over eight heads the worst one breaks it (1.7e-3 on both cases)."""
    make, _ = CASES[case]
    _, e_state = _errors(make(), range(0, 32, 4), p="bf16", rest="split")
    assert e_state > STATE_RTOL, e_state
