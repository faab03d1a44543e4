"""CPU oracle for the Gated DeltaNet recurrence (fp64).

TEST INFRASTRUCTURE ONLY: the test-suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use it; the product library never imports it
and shares no code with it.  The arithmetic lives in ``gdn_oracle.c`` (plain
C, fp64, sequential per (sequence, head), OpenMP across independent heads);
this module only compiles that file with the host C compiler and marshals
numpy arrays across ctypes.

Functions (all inputs numpy, see ``gdn_oracle.c`` for the definition):
  prefill          sequential scan over packed sequences (optionally with the
                   gates computed from raw inputs: gate_scale / gate_bias)
  prefill_chunked  blocked (chunked) evaluation of the same recurrence
  decode_step      one token applied to a batch of independent states

Every function here is pinned by ``tests/test_oracle_pins.py`` against
closed forms, invariants and brute-force formulas (none is "parity
unpinned").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libgdn_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/libgdn_oracle.so`` (idempotent)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = f"{_LIB_PATH}.{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            Dbl = ctypes.c_double
            lib.gdn_oracle_prefill.argtypes = [I, P, I, I, I, I, P, P, P, P, P, P, P, P, I, Dbl, P, P, I]
            lib.gdn_oracle_prefill_chunked.argtypes = [I, P, I, I, I, I, P, P, P, P, P, P, P, P, I, I, Dbl, I]
            lib.gdn_oracle_decode_step.argtypes = [I, I, I, I, I, P, P, P, P, P, P, P, I, Dbl, P, P, I]
            for f in (lib.gdn_oracle_prefill, lib.gdn_oracle_prefill_chunked, lib.gdn_oracle_decode_step):
                f.restype = I
            lib.gdn_oracle_max_threads.restype = I
            _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().gdn_oracle_max_threads())


def _f32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _shapes(q, k, v):
    if q.ndim != 3 or k.shape != q.shape or v.ndim != 3 or v.shape[0] != q.shape[0]:
        raise ValueError("q,k must be [T, hk, dk] and v [T, hv, dv]")
    T, hk, dk = q.shape
    _, hv, dv = v.shape
    return T, hk, dk, hv, dv


def rms_norm(out, weight, eps):
    """Output normalisation (fp64): every head's output vector o (the last axis) becomes
    o / sqrt(mean(o^2) + eps) * weight.  The pages' decode path fuses "the recurrent update with its
    normalisation" ("Optimizing on-device inference for Apple Silicon", section "Reduce intermediate and
    state traffic"); they give neither the norm nor its weights, and this root-mean-square norm over the
    value dimension with a per-channel weight is our reading."""
    o = np.asarray(out, dtype=np.float64)
    w = np.asarray(weight, dtype=np.float64)
    return o / np.sqrt((o * o).mean(axis=-1, keepdims=True) + float(eps)) * w


def _gate_params(gate_scale, gate_bias, hv):
    if (gate_scale is None) != (gate_bias is None):
        raise ValueError("gate_scale and gate_bias go together")
    if gate_scale is None:
        return None, None
    c, b = _f32(gate_scale), _f32(gate_bias)
    if c.shape != (hv,) or b.shape != (hv,):
        raise ValueError("gate_scale and gate_bias must be [hv]")
    return c, b


def prefill(q, k, v, log_alpha, beta, cu_seqlens, init_state=None, *, n_threads=None,
            want_out=True, qk_norm=False, q_scale=1.0, norm_weight=None, norm_eps=1e-6,
            gate_scale=None, gate_bias=None):
    """Sequential fp64 scan.  Returns (out [T,hv,dv] fp64 or None, final_state [N,hv,dv,dk] fp64).

    ``qk_norm``: L2-normalise every q and k head vector first (x / sqrt(|x|^2 + 1e-6)); q is then
    multiplied by ``q_scale``.  ``norm_weight`` ([dv]): apply :func:`rms_norm` to the outputs.
    ``gate_scale`` / ``gate_bias`` ([hv] each): ``log_alpha`` and ``beta`` hold the raw per-token inputs
    a and y, and the gates are log_alpha = -c_h softplus(a + b_h), beta = sigmoid(y) (see
    ``gdn_oracle.c``)."""
    q, k, v = _f32(q), _f32(k), _f32(v)
    la, b = _f32(log_alpha), _f32(beta)
    T, hk, dk, hv, dv = _shapes(q, k, v)
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    N = cu.shape[0] - 1
    if cu[0] != 0 or cu[-1] != T:
        raise ValueError("cu_seqlens must start at 0 and end at T")
    s0 = None if init_state is None else _f64(init_state)
    gc, gb = _gate_params(gate_scale, gate_bias, hv)
    out = np.zeros((T, hv, dv), np.float64) if want_out else None
    fin = np.zeros((N, hv, dv, dk), np.float64)
    rc = _load().gdn_oracle_prefill(N, _ptr(cu), hk, hv, dk, dv, _ptr(q), _ptr(k), _ptr(v),
                                    _ptr(la), _ptr(b), _ptr(s0), _ptr(out), _ptr(fin),
                                    int(bool(qk_norm)), float(q_scale), _ptr(gc), _ptr(gb),
                                    int(n_threads or max_threads()))
    if rc:
        raise RuntimeError(f"gdn_oracle_prefill failed: {rc}")
    if norm_weight is not None and out is not None:
        out = rms_norm(out, norm_weight, norm_eps)
    return out, fin


def prefill_chunked(q, k, v, log_alpha, beta, cu_seqlens, init_state=None, *, chunk,
                    n_threads=None, qk_norm=False, q_scale=1.0):
    """Blocked fp64 evaluation with chunk size ``chunk``; same return as :func:`prefill`."""
    q, k, v = _f32(q), _f32(k), _f32(v)
    la, b = _f32(log_alpha), _f32(beta)
    T, hk, dk, hv, dv = _shapes(q, k, v)
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    N = cu.shape[0] - 1
    s0 = None if init_state is None else _f64(init_state)
    out = np.zeros((T, hv, dv), np.float64)
    fin = np.zeros((N, hv, dv, dk), np.float64)
    rc = _load().gdn_oracle_prefill_chunked(N, _ptr(cu), hk, hv, dk, dv, _ptr(q), _ptr(k), _ptr(v),
                                            _ptr(la), _ptr(b), _ptr(s0), _ptr(out), _ptr(fin),
                                            int(chunk), int(bool(qk_norm)), float(q_scale),
                                            int(n_threads or max_threads()))
    if rc:
        raise RuntimeError(f"gdn_oracle_prefill_chunked failed: {rc}")
    return out, fin


def decode_step(state, q, k, v, log_alpha, beta, *, n_threads=None, qk_norm=False, q_scale=1.0,
                norm_weight=None, norm_eps=1e-6, gate_scale=None, gate_bias=None):
    """One token per state.  state [n,hv,dv,dk]; q,k [n,hk,dk]; v [n,hv,dv]; gates [n,hv].

    Returns (out [n,hv,dv] fp64, new_state fp64); the input array is not modified.
    """
    q, k, v = _f32(q), _f32(k), _f32(v)
    la, b = _f32(log_alpha), _f32(beta)
    n, hk, dk, hv, dv = _shapes(q, k, v)
    st = np.array(state, dtype=np.float64, order="C", copy=True)
    if st.shape != (n, hv, dv, dk):
        raise ValueError("state must be [n, hv, dv, dk]")
    gc, gb = _gate_params(gate_scale, gate_bias, hv)
    out = np.zeros((n, hv, dv), np.float64)
    rc = _load().gdn_oracle_decode_step(n, hk, hv, dk, dv, _ptr(st), _ptr(q), _ptr(k), _ptr(v),
                                        _ptr(la), _ptr(b), _ptr(out), int(bool(qk_norm)), float(q_scale),
                                        _ptr(gc), _ptr(gb), int(n_threads or max_threads()))
    if rc:
        raise RuntimeError(f"gdn_oracle_decode_step failed: {rc}")
    if norm_weight is not None:
        out = rms_norm(out, norm_weight, norm_eps)
    return out, st


if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv))
