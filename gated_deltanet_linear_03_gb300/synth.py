"""Seeded synthetic inputs for the Gated DeltaNet recurrence.

This module only draws random numbers and shapes them into the input
conventions of the library (it holds none of the recurrence's arithmetic), so
the CUDA path, the oracle-based tests and the benchmark can all use it.

Distributions follow the workloads the library is measured on:
  * q, k ~ N(0, 1), L2-normalised per head over the key dimension; q is also
    multiplied by 1/sqrt(dk) for the model-shaped cases; stored as bf16.
  * v ~ N(0, 1), bf16.
  * log_alpha = -0.5 * softplus(N(0,1) + 2) per token per value head
    ("model" gates, alpha around 0.33), or -softplus(N(0,1)) for the tiny
    case, or -softplus(N(0,1) - 6) for the slow-decay stress gates
    (alpha around 0.998).  fp32.
  * beta = sigmoid(N(0,1)) (scaled by 0.1 for the stress gates).  fp32.
  * raw gates (``raw_gates``), for the in-kernel gate computation: the same
    two normal draws are returned unmapped (a, y), with per-value-head
    parameters gate_scale c and gate_bias b: either the constants of the
    recipe above ("config": c = 0.5, b = 2 for the model gates; c = 1, b = 0
    for the tiny ones) or per-head draws ("per_head": c ~ U[0.25, 1.5],
    b ~ U[-0.5, 2.5]).
  * initial states ~ N(0, std^2) fp32 when requested.
  * ragged lengths are log-uniform in [lo, hi].

Everything is generated on the CPU with ``torch.Generator`` seeds, so that the
oracle and the GPU consume identical bytes.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Optional, Sequence

import torch
import torch.nn.functional as F


@dataclass
class PrefillInputs:
    q: torch.Tensor          # [T, hk, dk] bf16
    k: torch.Tensor          # [T, hk, dk] bf16
    v: torch.Tensor          # [T, hv, dv] bf16
    log_alpha: torch.Tensor  # [T, hv] fp32
    beta: torch.Tensor       # [T, hv] fp32
    init_state: Optional[torch.Tensor]  # [N, hv, dv, dk] fp32 or None
    cu_seqlens: torch.Tensor  # [N + 1] int32
    gate_scale: Optional[torch.Tensor] = None   # [hv] fp32: log_alpha/beta hold raw inputs when set
    gate_bias: Optional[torch.Tensor] = None    # [hv] fp32

    @property
    def shape(self):
        T, hk, dk = self.q.shape
        return dict(T=T, hk=hk, hv=self.v.shape[1], dk=dk, dv=self.v.shape[2],
                    n_seqs=self.cu_seqlens.numel() - 1)


@dataclass
class DecodeInputs:
    state: torch.Tensor      # [n, hv, dv, dk] fp32
    q: torch.Tensor          # [steps, n, hk, dk] bf16
    k: torch.Tensor          # [steps, n, hk, dk] bf16
    v: torch.Tensor          # [steps, n, hv, dv] bf16
    log_alpha: torch.Tensor  # [steps, n, hv] fp32
    beta: torch.Tensor       # [steps, n, hv] fp32
    gate_scale: Optional[torch.Tensor] = None   # [hv] fp32: log_alpha/beta hold raw inputs when set
    gate_bias: Optional[torch.Tensor] = None    # [hv] fp32


def _unit(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-12)


# (c, b) of the recipe log_alpha = -c softplus(z + b) for the gate kinds that have that form
GATE_RECIPE = {"model": (0.5, 2.0), "tiny": (1.0, 0.0)}


def _gates(shape, gen, kind: str, raw: Optional[str] = None):
    """(log_alpha, beta), or with ``raw`` the unmapped draws (a, y) and the [hv] gate parameters."""
    z1 = torch.randn(shape, generator=gen, device=gen.device)
    z2 = torch.randn(shape, generator=gen, device=gen.device)
    if raw is not None:
        hv = shape[-1]
        if raw == "config":
            if kind not in GATE_RECIPE:
                raise ValueError(f"the {kind} gates have no (c, b) recipe")
            c, b = GATE_RECIPE[kind]
            scale, bias = torch.full((hv,), c), torch.full((hv,), b)
        elif raw == "per_head":
            scale = 0.25 + 1.25 * torch.rand(hv, generator=gen, device=gen.device)
            bias = -0.5 + 3.0 * torch.rand(hv, generator=gen, device=gen.device)
        else:
            raise ValueError(raw)
        return z1, z2, scale.float().cpu(), bias.float().cpu()
    if kind == "model":
        return -0.5 * F.softplus(z1 + 2.0), torch.sigmoid(z2)
    if kind == "tiny":
        return -F.softplus(z1), torch.sigmoid(z2)
    if kind == "slow":
        return -F.softplus(z1 - 6.0), 0.1 * torch.sigmoid(z2)
    raise ValueError(kind)


def qkv(T: int, hk: int, hv: int, dk: int, dv: int, gen, *, scale_q: bool = True, raw_qk: bool = False):
    """q, k unit vectors (q scaled by 1/sqrt(dk) when ``scale_q``), v ~ N(0, 1).  With ``raw_qk`` q and k are
    raw projections instead: N(0, 1) entries times a per-vector length drawn from [0.25, 4], for the
    in-kernel query/key preparation to normalise."""
    dev = gen.device
    q = torch.randn(T, hk, dk, generator=gen, device=dev)
    k = torch.randn(T, hk, dk, generator=gen, device=dev)
    v = torch.randn(T, hv, dv, generator=gen, device=dev)
    if raw_qk:
        q = q * (0.25 + 3.75 * torch.rand(T, hk, 1, generator=gen, device=dev))
        k = k * (0.25 + 3.75 * torch.rand(T, hk, 1, generator=gen, device=dev))
        return q, k, v
    q, k = _unit(q), _unit(k)
    if scale_q:
        q = q / math.sqrt(dk)
    return q, k, v


def prefill_inputs(lengths: Sequence[int], *, hk=16, hv=32, dk=128, dv=128, seed=1001,
                   gates="model", init_std: float = 0.0, scale_q: bool = True,
                   qkv_dtype=torch.bfloat16, raw_qk: bool = False, raw_gates: Optional[str] = None,
                   device=None) -> PrefillInputs:
    """Packed prefill inputs for sequences of the given lengths.  With a CUDA ``device`` the draws come from
    that device's generator (same recipe and seed, different numbers): for timing large workloads only,
    never for comparison with the oracle."""
    gen = torch.Generator(device=device or "cpu").manual_seed(seed)
    T = int(sum(lengths))
    q, k, v = qkv(T, hk, hv, dk, dv, gen, scale_q=scale_q, raw_qk=raw_qk)
    g = _gates((T, hv), gen, gates, raw_gates)
    la, b = g[0], g[1]
    cu = torch.zeros(len(lengths) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(list(lengths), dtype=torch.int64), 0).to(torch.int32)
    s0 = None
    if init_std > 0:
        s0 = torch.randn(len(lengths), hv, dv, dk, generator=gen, device=gen.device) * init_std
    return PrefillInputs(q.to(qkv_dtype), k.to(qkv_dtype), v.to(qkv_dtype),
                         la.float().contiguous(), b.float().contiguous(), s0, cu,
                         *(g[2:] if raw_gates else (None, None)))


def log_uniform_lengths(n: int, lo: int, hi: int, seed: int) -> list:
    gen = torch.Generator().manual_seed(seed)
    u = torch.rand(n, generator=gen, dtype=torch.float64)
    return [int(math.floor(math.exp(math.log(lo) + float(x) * (math.log(hi) - math.log(lo)))))
            for x in u]


def decode_inputs(n: int, steps: int, *, hk=16, hv=32, dk=128, dv=128, seed=1002,
                  state_std: float = 0.02, gates="model", raw_qk: bool = False, raw_gates: Optional[str] = None,
                  device=None) -> DecodeInputs:
    """``n`` independent states (one per layer) and ``steps`` tokens of fresh inputs (``device`` as in
    ``prefill_inputs``)."""
    gen = torch.Generator(device=device or "cpu").manual_seed(seed)
    state = torch.randn(n, hv, dv, dk, generator=gen, device=gen.device) * state_std
    q, k, v = qkv(steps * n, hk, hv, dk, dv, gen, raw_qk=raw_qk)
    g = _gates((steps * n, hv), gen, gates, raw_gates)
    la, b = g[0], g[1]
    bf = torch.bfloat16
    return DecodeInputs(state.contiguous(),
                        q.reshape(steps, n, hk, dk).to(bf), k.reshape(steps, n, hk, dk).to(bf),
                        v.reshape(steps, n, hv, dv).to(bf),
                        la.reshape(steps, n, hv).contiguous(), b.reshape(steps, n, hv).contiguous(),
                        *(g[2:] if raw_gates else (None, None)))


# Named workloads -----------------------------------------------------------------------------

def tiny_case(seed: int = 1000) -> PrefillInputs:
    """1 sequence, T=64, 2 heads, dk=dv=32, fp32 draws (rounded to bf16 for the GPU)."""
    return prefill_inputs([64], hk=2, hv=2, dk=32, dv=32, seed=seed, gates="tiny",
                          scale_q=False, qkv_dtype=torch.float32)


def prefill_4k(seed: int = 1001) -> PrefillInputs:
    """Single-layer prefill, one 4096-token sequence, 16 q/k heads, 32 v heads, d=128."""
    return prefill_inputs([4096], seed=seed)


def long_128k(seed: int = 1003) -> PrefillInputs:
    return prefill_inputs([131072], seed=seed)


def ragged_8(seed: int = 1004) -> PrefillInputs:
    """8 packed sequences, lengths log-uniform in [256, 32768], initial states ~ N(0, 0.02^2)."""
    return prefill_inputs(log_uniform_lengths(8, 256, 32768, seed), seed=seed, init_std=0.02)


def decode_30(steps: int = 256, seed: int = 1002) -> DecodeInputs:
    """30 layers of batch-1 decode state (32 v heads x 128 x 128 fp32 each)."""
    return decode_inputs(30, steps, seed=seed)
