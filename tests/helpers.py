"""Shared test helpers: conversions to the oracle's inputs and the parity checks.

Tolerances (stated for bf16 q/k/v with fp32 state and accumulation):
  outputs       max |o_gpu - o_oracle| <= 2e-3 (on the returned dtype)
  final states  per (sequence, head) ||S_gpu - S_oracle||_F / ||S_oracle||_F <= 1e-3
                (absolute 1e-6 when the oracle's norm is 0)
"""
import numpy as np
import torch

OUT_ATOL = 2e-3
STATE_RTOL = 1e-3


def np32(t: torch.Tensor) -> np.ndarray:
    """Exact float32 copy of a CPU/GPU tensor (bf16 values are exact in fp32)."""
    return t.detach().float().cpu().numpy()


def oracle_args(inp):
    return (np32(inp.q), np32(inp.k), np32(inp.v), np32(inp.log_alpha), np32(inp.beta),
            inp.cu_seqlens.cpu().numpy().astype(np.int32),
            None if inp.init_state is None else inp.init_state.double().cpu().numpy())


def to_device(inp, dev="cuda"):
    from gated_deltanet_linear_03_gb300.synth import PrefillInputs
    bf = torch.bfloat16
    return PrefillInputs(inp.q.to(bf).to(dev), inp.k.to(bf).to(dev), inp.v.to(bf).to(dev),
                         inp.log_alpha.to(dev), inp.beta.to(dev),
                         None if inp.init_state is None else inp.init_state.to(dev),
                         inp.cu_seqlens.to(dev))


def as_bf16_inputs(inp):
    """The bf16-rounded copy of an fp32-drawn case, as the GPU consumes it."""
    from gated_deltanet_linear_03_gb300.synth import PrefillInputs
    bf = torch.bfloat16
    return PrefillInputs(inp.q.to(bf), inp.k.to(bf), inp.v.to(bf), inp.log_alpha, inp.beta,
                         inp.init_state, inp.cu_seqlens)


def max_abs_err(got: torch.Tensor, ref: np.ndarray) -> float:
    if ref.size == 0:
        return 0.0
    return float(np.max(np.abs(np32(got).astype(np.float64) - ref)))


def state_rel_err(got: torch.Tensor, ref: np.ndarray) -> float:
    """Worst per-(sequence, head) relative Frobenius error."""
    g = np32(got).astype(np.float64)
    diff = np.sqrt(((g - ref) ** 2).sum(axis=(-1, -2)))
    norm = np.sqrt((ref ** 2).sum(axis=(-1, -2)))
    rel = np.where(norm > 0, diff / np.where(norm > 0, norm, 1.0), diff / 1e-3)
    return float(rel.max()) if rel.size else 0.0


def check_prefill(out, fin, ref_out, ref_fin, *, out_atol=OUT_ATOL, state_rtol=STATE_RTOL, what=""):
    e_o = max_abs_err(out, ref_out)
    e_s = state_rel_err(fin, ref_fin) if fin is not None else 0.0
    assert e_o <= out_atol, f"{what}: output max|err| {e_o:.3e} > {out_atol}"
    assert e_s <= state_rtol, f"{what}: state rel err {e_s:.3e} > {state_rtol}"
    return e_o, e_s
