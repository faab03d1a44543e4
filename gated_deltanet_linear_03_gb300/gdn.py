"""Thin ctypes binding of libgdn (include/gdn.h).

Argument marshalling only: every step of the recurrence runs in the CUDA
kernels of ``libgdn.so``.  Torch provides device memory and streams.  There is
no CPU fallback: if the library is missing or no GPU is present, calls raise.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence, Tuple

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgdn.so")

GDN_OK = 0
STATUS_NAMES = {0: "GDN_OK", 1: "GDN_ERR_INVALID_ARG", 2: "GDN_ERR_UNSUPPORTED", 3: "GDN_ERR_ALIGNMENT",
                4: "GDN_ERR_CUDA", 5: "GDN_ERR_TIMEOUT", 6: "GDN_ERR_INTERNAL", 7: "GDN_ERR_WORKSPACE"}
ALGO = {"chunked": 0, "scan": 1, "auto": 2}
DTYPE = {torch.bfloat16: 0, torch.float32: 1}

# every symbol include/gdn.h declares
EXPORTS = ("gdn_prefill", "gdn_prefill_chunked_phase", "gdn_prefill_workspace_size", "gdn_decode_step",
           "gdn_device_error", "gdn_status_string", "gdn_version", "gdn_prefill_noalloc", "gdn_prefill_algo",
           "gdn_prefill_host", "gdn_prefill_host_staging_size", "gdn_selftest_bounded_wait",
           "gdn_prefill_pass_plan")
NOALLOC_SCRATCH_BYTES = 97 * 1024 * 1024
PHASE = {"prep": 1, "pass": 2}


class GdnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} ({lib_status_string(status)})")


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libgdn.so (built by ``__graft_entry__.build()``); raises if it is missing.  The handle is kept:
    the wrappers below use it unless given another one (``lib=``)."""
    global _lib
    if _lib is not None:
        return _lib
    _lib = bind(path)
    return _lib


def bind(path: str) -> ctypes.CDLL:
    """A configured handle of a library with the gdn.h ABI at ``path`` (e.g. the bounds-checking build
    ``libgdn_debug.so``), not kept as the default."""
    if not os.path.exists(path):
        raise RuntimeError(f"{os.path.basename(path)} not found at {path}; build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    F = ctypes.c_float
    lib.gdn_prefill.argtypes = [I, I, I, I, I, I, P, P, P, P, P, P, P, P, P, I, P, I, F, P, F, P, P, I, P, Z, P]
    lib.gdn_prefill.restype = I
    lib.gdn_prefill_chunked_phase.argtypes = [I, I, I, I, I, I, I, P, P, P, P, P, P, P, P, P, I, P, I, F, P, F, P, P,
                                              P, Z, P]
    lib.gdn_prefill_chunked_phase.restype = I
    lib.gdn_prefill_noalloc.argtypes = [I, I, I, I, I, I, P, P, P, P, P, P, P, P, P, I, P, I, F, P, F, P, P, P]
    lib.gdn_prefill_noalloc.restype = I
    lib.gdn_prefill_workspace_size.argtypes = [I, I, I, I, I, I, P, I, ctypes.POINTER(I)]
    lib.gdn_prefill_workspace_size.restype = Z
    lib.gdn_prefill_host.argtypes = [I, I, I, I, I, I, P, P, P, P, P, P, P, P, I, P, I, F, P, F, P, P, I, P, Z, P]
    lib.gdn_prefill_host.restype = I
    lib.gdn_prefill_host_staging_size.argtypes = [I, I, I, I, I, I, P, I, I, I, I, ctypes.POINTER(I)]
    lib.gdn_prefill_host_staging_size.restype = Z
    lib.gdn_prefill_algo.argtypes = [I, I, I, I, I, I, P]
    lib.gdn_prefill_algo.restype = I
    lib.gdn_prefill_pass_plan.argtypes = [I, I, I, P, I, P, I]
    lib.gdn_prefill_pass_plan.restype = I
    lib.gdn_decode_step.argtypes = [I, I, I, I, I, P, P, P, P, P, P, P, I, I, ctypes.c_float, P, ctypes.c_float, P,
                                    P, P]
    lib.gdn_decode_step.restype = I
    lib.gdn_device_error.argtypes = [P]
    lib.gdn_device_error.restype = I
    lib.gdn_selftest_bounded_wait.argtypes = [I, P]
    lib.gdn_selftest_bounded_wait.restype = I
    lib.gdn_status_string.argtypes = [I]
    lib.gdn_status_string.restype = ctypes.c_char_p
    lib.gdn_version.restype = I
    return lib


def lib_status_string(status: int) -> str:
    try:
        return load_library().gdn_status_string(int(status)).decode()
    except Exception:  # pragma: no cover
        return "?"


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream, device=None) -> ctypes.c_void_p:
    """The stream to enqueue on: ``stream``, else the current stream of ``device`` (the tensors' device)."""
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _gate_tensors(gate_scale, gate_bias, hv: int):
    """The optional gate parameters: both or neither, fp32 [hv]."""
    if (gate_scale is None) != (gate_bias is None):
        raise ValueError("gate_scale and gate_bias go together")
    if gate_scale is not None:
        _need(gate_scale, "gate_scale", torch.float32, 1)
        _need(gate_bias, "gate_bias", torch.float32, 1)
        if gate_scale.numel() != hv or gate_bias.numel() != hv:
            raise ValueError(f"gate_scale and gate_bias must have hv = {hv} entries")


def _same_device(device: torch.device, **tensors):
    """Every tensor lives on ``device``: the library launches on the current device, which the wrappers make
    the tensors' device, and refuses pointers of any other device."""
    for name, t in tensors.items():
        if t is not None and t.device != device:
            raise ValueError(f"{name} is on {t.device}, the other tensors on {device}")


def _need(t: torch.Tensor, name: str, dtype, ndim: int):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {ndim}-d tensor")


def _host_cu(cu_seqlens: torch.Tensor, cu_host) -> Tuple[ctypes.Array, list]:
    vals = [int(x) for x in (cu_host if cu_host is not None else cu_seqlens.cpu().tolist())]
    arr = (ctypes.c_int32 * len(vals))(*vals)
    return arr, vals


def resolve_algo(n_seqs: int, total_tokens: int, hk: int, hv: int, dk: int, dv: int,
                 cu_seqlens_host: Sequence[int]) -> str:
    """The algorithm ``algo="auto"`` runs for this problem (``gdn_prefill_algo``)."""
    lib = load_library()
    arr = (ctypes.c_int32 * len(cu_seqlens_host))(*[int(x) for x in cu_seqlens_host])
    a = lib.gdn_prefill_algo(n_seqs, total_tokens, hk, hv, dk, dv, arr)
    if a < 0:
        raise GdnError(1, "gdn_prefill_algo")
    return {v: k for k, v in ALGO.items()}[a]


def pass_plan(cu_seqlens_host: Sequence[int], hv: int, multiprocessors: int = 152) -> list:
    """The state pass's buckets (``gdn_prefill_pass_plan``): the first sequence of each bucket, then n_seqs."""
    lib = load_library()
    n = len(cu_seqlens_host) - 1
    arr = (ctypes.c_int32 * len(cu_seqlens_host))(*[int(x) for x in cu_seqlens_host])
    out = (ctypes.c_int * (n + 1))()
    nb = lib.gdn_prefill_pass_plan(n, int(cu_seqlens_host[-1]), hv, arr, multiprocessors, out, n + 1)
    if nb < 1:
        raise GdnError(1, "gdn_prefill_pass_plan")
    return list(out[:nb + 1])


def workspace_size(n_seqs: int, total_tokens: int, hk: int, hv: int, dk: int, dv: int,
                   cu_seqlens_host: Sequence[int], algo: str = "chunked", lib=None) -> int:
    lib = lib or load_library()
    arr = (ctypes.c_int32 * len(cu_seqlens_host))(*[int(x) for x in cu_seqlens_host])
    st = ctypes.c_int(0)
    n = lib.gdn_prefill_workspace_size(n_seqs, total_tokens, hk, hv, dk, dv, arr, ALGO[algo], ctypes.byref(st))
    if st.value != GDN_OK:
        raise GdnError(st.value, "gdn_prefill_workspace_size")
    return int(n)


def prefill(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, log_alpha: torch.Tensor,
            beta: torch.Tensor, cu_seqlens: torch.Tensor, *, init_state: Optional[torch.Tensor] = None,
            out: Optional[torch.Tensor] = None, out_dtype=torch.bfloat16,
            final_state=True, algo: str = "chunked", workspace: Optional[torch.Tensor] = None,
            cu_seqlens_host: Optional[Sequence[int]] = None, stream=None, qk_norm: bool = False,
            q_scale: float = 1.0, norm_weight: Optional[torch.Tensor] = None, norm_eps: float = 1e-6,
            gate_scale: Optional[torch.Tensor] = None, gate_bias: Optional[torch.Tensor] = None, lib=None):
    """Run ``gdn_prefill``.  Returns ``(out, final_state)``.  ``lib``: a handle from :func:`bind` instead of the
    default library.

    ``gate_scale`` / ``gate_bias`` (fp32 [hv] each): ``log_alpha`` and ``beta`` hold raw per-token inputs a, y and
    the kernels compute log_alpha = -gate_scale softplus(a + gate_bias), beta = sigmoid(y).

    ``qk_norm`` / ``q_scale``: the in-kernel query/key preparation (every q and k head vector
    L2-normalised, then q multiplied by ``q_scale``); the defaults use q and k as given.
    ``norm_weight`` (fp32 [dv]): fuse the output normalisation o / sqrt(mean(o^2) + norm_eps) * weight.

    ``final_state`` may be ``True`` (allocate), ``False``/``None`` (do not emit)
    or a tensor to write into (it may be ``init_state`` for an in-place update).
    """
    lib = lib or load_library()
    _need(q, "q", torch.bfloat16, 3)
    _need(k, "k", torch.bfloat16, 3)
    _need(v, "v", torch.bfloat16, 3)
    _need(log_alpha, "log_alpha", torch.float32, 2)
    _need(beta, "beta", torch.float32, 2)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    T, hk, dk = q.shape
    hv, dv = v.shape[1], v.shape[2]
    n_seqs = cu_seqlens.numel() - 1
    if init_state is not None:
        _need(init_state, "init_state", torch.float32, 4)
    if out is None:
        out = torch.empty(T, hv, dv, device=q.device, dtype=out_dtype)
    else:
        _need(out, "out", out.dtype, 3)
    if final_state is True:
        final_state = torch.empty(n_seqs, hv, dv, dk, device=q.device, dtype=torch.float32)
    elif final_state is False:
        final_state = None
    elif final_state is not None:
        _need(final_state, "final_state", torch.float32, 4)
    cu_arr, cu_vals = _host_cu(cu_seqlens, cu_seqlens_host)
    need = workspace_size(n_seqs, T, hk, hv, dk, dv, cu_vals, algo, lib=lib) if n_seqs > 0 else 0
    if need and workspace is None:
        workspace = torch.empty(need, device=q.device, dtype=torch.uint8)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _gate_tensors(gate_scale, gate_bias, hv)
    _same_device(q.device, k=k, v=v, log_alpha=log_alpha, beta=beta, cu_seqlens=cu_seqlens, init_state=init_state,
                 out=out, final_state=final_state, norm_weight=norm_weight, workspace=workspace,
                 gate_scale=gate_scale, gate_bias=gate_bias)
    with torch.cuda.device(q.device):
        st = lib.gdn_prefill(n_seqs, T, hk, hv, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta),
                             _ptr(init_state), _ptr(cu_seqlens), cu_arr, _ptr(out), DTYPE[out.dtype],
                             _ptr(final_state), int(bool(qk_norm)), float(q_scale), _ptr(norm_weight),
                             float(norm_eps), _ptr(gate_scale), _ptr(gate_bias), ALGO[algo], _ptr(workspace),
                             ws_bytes, _stream_ptr(stream, q.device))
    if st != GDN_OK:
        raise GdnError(st, "gdn_prefill")
    return out, final_state


def prefill_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, log_alpha: torch.Tensor,
                    beta: torch.Tensor, cu_seqlens: torch.Tensor, *, init_state: Optional[torch.Tensor] = None,
                    out: Optional[torch.Tensor] = None, out_dtype=torch.bfloat16, final_state=True,
                    cu_seqlens_host: Optional[Sequence[int]] = None, stream=None, qk_norm: bool = False,
                    q_scale: float = 1.0, norm_weight: Optional[torch.Tensor] = None, norm_eps: float = 1e-6,
                    gate_scale: Optional[torch.Tensor] = None, gate_bias: Optional[torch.Tensor] = None):
    """Run ``gdn_prefill_noalloc``: the chunked prefill using the library's fixed
    scratch instead of a workspace (for callers that cannot allocate device
    memory; see include/gdn.h for its size limit and sharing rules).
    Returns ``(out, final_state)``; ``out``/``final_state`` are allocated here
    only when not passed in."""
    lib = load_library()
    _need(q, "q", torch.bfloat16, 3)
    _need(k, "k", torch.bfloat16, 3)
    _need(v, "v", torch.bfloat16, 3)
    _need(log_alpha, "log_alpha", torch.float32, 2)
    _need(beta, "beta", torch.float32, 2)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    T, hk, dk = q.shape
    hv, dv = v.shape[1], v.shape[2]
    n_seqs = cu_seqlens.numel() - 1
    if init_state is not None:
        _need(init_state, "init_state", torch.float32, 4)
    if out is None:
        out = torch.empty(T, hv, dv, device=q.device, dtype=out_dtype)
    if final_state is True:
        final_state = torch.empty(n_seqs, hv, dv, dk, device=q.device, dtype=torch.float32)
    elif final_state is False:
        final_state = None
    cu_arr, _ = _host_cu(cu_seqlens, cu_seqlens_host)
    _gate_tensors(gate_scale, gate_bias, hv)
    _same_device(q.device, k=k, v=v, log_alpha=log_alpha, beta=beta, cu_seqlens=cu_seqlens, init_state=init_state,
                 out=out, final_state=final_state, norm_weight=norm_weight, gate_scale=gate_scale, gate_bias=gate_bias)
    with torch.cuda.device(q.device):   # the scratch used is the one of the current device
        st = lib.gdn_prefill_noalloc(n_seqs, T, hk, hv, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha),
                                     _ptr(beta), _ptr(init_state), _ptr(cu_seqlens), cu_arr, _ptr(out),
                                     DTYPE[out.dtype], _ptr(final_state), int(bool(qk_norm)), float(q_scale),
                                     _ptr(norm_weight), float(norm_eps), _ptr(gate_scale), _ptr(gate_bias),
                                     _stream_ptr(stream, q.device))
    if st != GDN_OK:
        raise GdnError(st, "gdn_prefill_noalloc")
    return out, final_state


def _need_host(t: torch.Tensor, name: str, dtype, ndim: int):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.is_cuda:
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {ndim}-d tensor")


def host_staging_size(n_seqs: int, total_tokens: int, hk: int, hv: int, dk: int, dv: int,
                      cu_seqlens_host: Sequence[int], out_dtype=torch.bfloat16, init_state: bool = False,
                      final_state: bool = True, algo: str = "chunked") -> int:
    """Bytes of device staging ``gdn_prefill_host`` needs for this problem."""
    lib = load_library()
    arr = (ctypes.c_int32 * len(cu_seqlens_host))(*[int(x) for x in cu_seqlens_host])
    st = ctypes.c_int(0)
    n = lib.gdn_prefill_host_staging_size(n_seqs, total_tokens, hk, hv, dk, dv, arr, DTYPE[out_dtype],
                                          int(bool(init_state)), int(bool(final_state)), ALGO[algo],
                                          ctypes.byref(st))
    if st.value != GDN_OK:
        raise GdnError(st.value, "gdn_prefill_host_staging_size")
    return int(n)


class HostPrefillPlan:
    """Pre-marshalled arguments of one ``gdn_prefill_host`` problem: inputs and outputs in host memory, the
    copies and the kernels enqueued by the library on one stream.  ``out`` and ``final_state`` are
    allocated here in page-locked host memory unless passed in; ``staging`` is allocated on ``device``
    unless passed in.  ``run`` only enqueues: synchronise the stream before reading the outputs or changing
    the inputs.  Two plans with their own staging, run alternately on two streams, overlap one call's
    copies with the other's kernels."""

    def __init__(self, q, k, v, log_alpha, beta, cu_seqlens_host, *, init_state=None, out=None,
                 out_dtype=torch.bfloat16, final_state=True, algo="chunked", staging=None, device=None,
                 qk_norm=False, q_scale=1.0, norm_weight=None, norm_eps=1e-6, gate_scale=None, gate_bias=None):
        self.lib = load_library()
        _need_host(q, "q", torch.bfloat16, 3)
        _need_host(k, "k", torch.bfloat16, 3)
        _need_host(v, "v", torch.bfloat16, 3)
        _need_host(log_alpha, "log_alpha", torch.float32, 2)
        _need_host(beta, "beta", torch.float32, 2)
        if init_state is not None:
            _need_host(init_state, "init_state", torch.float32, 4)
        if norm_weight is not None:
            _need(norm_weight, "norm_weight", torch.float32, 1)
        T, hk, dk = q.shape
        hv, dv = v.shape[1], v.shape[2]
        cu_vals = [int(x) for x in (cu_seqlens_host.tolist() if isinstance(cu_seqlens_host, torch.Tensor)
                                    else cu_seqlens_host)]
        n_seqs = len(cu_vals) - 1
        self.cu_arr = (ctypes.c_int32 * len(cu_vals))(*cu_vals)
        if out is None:
            out = torch.empty(T, hv, dv, dtype=out_dtype, pin_memory=True)
        _need_host(out, "out", out.dtype, 3)
        if final_state is True:
            final_state = torch.empty(n_seqs, hv, dv, dk, dtype=torch.float32, pin_memory=True)
        elif final_state is False:
            final_state = None
        if final_state is not None:
            _need_host(final_state, "final_state", torch.float32, 4)
        need = host_staging_size(n_seqs, T, hk, hv, dk, dv, cu_vals, out.dtype, init_state is not None,
                                 final_state is not None, algo)
        if staging is None:
            staging = torch.empty(need, dtype=torch.uint8, device=device or torch.device("cuda"))
        _gate_tensors(gate_scale, gate_bias, hv)
        _same_device(staging.device, norm_weight=norm_weight, gate_scale=gate_scale, gate_bias=gate_bias)
        self.device = staging.device
        self.out, self.final_state, self.staging = out, final_state, staging
        self.tensors = (q, k, v, log_alpha, beta, init_state, norm_weight, gate_scale, gate_bias)
        self.head = (n_seqs, T, hk, hv, dk, dv)
        self.ptrs = (_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(init_state), self.cu_arr,
                     _ptr(out), DTYPE[out.dtype], _ptr(final_state))
        self.qk = (int(bool(qk_norm)), float(q_scale), _ptr(norm_weight), float(norm_eps), _ptr(gate_scale),
                   _ptr(gate_bias))
        self.tail = (ALGO[algo], _ptr(staging), staging.numel() * staging.element_size())
        self.h2d_bytes = sum(t.numel() * t.element_size() for t in (q, k, v, log_alpha, beta, init_state)
                             if t is not None) + 4 * len(cu_vals)
        self.d2h_bytes = sum(t.numel() * t.element_size() for t in (out, final_state) if t is not None)

    def run(self, stream=None):
        with torch.cuda.device(self.device):
            st = self.lib.gdn_prefill_host(*self.head, *self.ptrs, *self.qk, *self.tail,
                                           _stream_ptr(stream, self.device))
        if st != GDN_OK:
            raise GdnError(st, "gdn_prefill_host")
        return self.out, self.final_state


def prefill_host(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, log_alpha: torch.Tensor, beta: torch.Tensor,
                 cu_seqlens_host, *, stream=None, **kw):
    """Run ``gdn_prefill_host`` once on host tensors and wait for it: returns ``(out, final_state)`` in host
    memory.  Keyword arguments as for ``HostPrefillPlan``."""
    plan = HostPrefillPlan(q, k, v, log_alpha, beta, cu_seqlens_host, **kw)
    plan.run(stream)
    (stream or torch.cuda.current_stream(plan.device)).synchronize()
    return plan.out, plan.final_state


class PrefillPlan:
    """Pre-marshalled arguments of one gdn_prefill problem, for repeated calls
    with little host overhead (benchmarks, CUDA-graph capture).  All tensors
    must stay alive and unmoved while the plan is used."""

    def __init__(self, q, k, v, log_alpha, beta, cu_seqlens, *, init_state=None, out=None,
                 out_dtype=torch.bfloat16, final_state=True, algo="chunked", workspace=None,
                 cu_seqlens_host=None, qk_norm=False, q_scale=1.0, norm_weight=None, norm_eps=1e-6,
                 gate_scale=None, gate_bias=None):
        self.lib = load_library()
        _need(q, "q", torch.bfloat16, 3)
        _need(k, "k", torch.bfloat16, 3)
        _need(v, "v", torch.bfloat16, 3)
        _need(log_alpha, "log_alpha", torch.float32, 2)
        _need(beta, "beta", torch.float32, 2)
        _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
        T, hk, dk = q.shape
        hv, dv = v.shape[1], v.shape[2]
        n_seqs = cu_seqlens.numel() - 1
        if out is None:
            out = torch.empty(T, hv, dv, device=q.device, dtype=out_dtype)
        if final_state is True:
            final_state = torch.empty(n_seqs, hv, dv, dk, device=q.device, dtype=torch.float32)
        elif final_state is False:
            final_state = None
        self.cu_arr, cu_vals = _host_cu(cu_seqlens, cu_seqlens_host)
        need = workspace_size(n_seqs, T, hk, hv, dk, dv, cu_vals, algo)
        if need and workspace is None:
            workspace = torch.empty(need, device=q.device, dtype=torch.uint8)
        self.out, self.final_state, self.workspace = out, final_state, workspace
        self.tensors = (q, k, v, log_alpha, beta, cu_seqlens, init_state, gate_scale, gate_bias)
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        self.algo = ALGO[algo]
        self.head = (n_seqs, T, hk, hv, dk, dv)
        self.ptrs = (_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(init_state), _ptr(cu_seqlens),
                     self.cu_arr, _ptr(out), DTYPE[out.dtype], _ptr(final_state))
        self.ws = (_ptr(workspace), ws_bytes)
        self.qk = (int(bool(qk_norm)), float(q_scale), _ptr(norm_weight), float(norm_eps), _ptr(gate_scale),
                   _ptr(gate_bias))
        self.norm_weight = norm_weight
        _gate_tensors(gate_scale, gate_bias, hv)
        _same_device(q.device, k=k, v=v, log_alpha=log_alpha, beta=beta, cu_seqlens=cu_seqlens,
                     init_state=init_state, out=out, final_state=final_state, norm_weight=norm_weight,
                     workspace=workspace, gate_scale=gate_scale, gate_bias=gate_bias)
        self.device = q.device

    def run(self, stream=None):
        with torch.cuda.device(self.device):
            st = self.lib.gdn_prefill(*self.head, *self.ptrs, *self.qk, self.algo, *self.ws,
                                      _stream_ptr(stream, self.device))
        if st != GDN_OK:
            raise GdnError(st, "gdn_prefill")
        return self.out, self.final_state

    def run_phase(self, phase: str, stream=None):
        with torch.cuda.device(self.device):
            st = self.lib.gdn_prefill_chunked_phase(PHASE[phase], *self.head, *self.ptrs, *self.qk, *self.ws,
                                                    _stream_ptr(stream, self.device))
        if st != GDN_OK:
            raise GdnError(st, "gdn_prefill_chunked_phase")


def decode_step(state: torch.Tensor, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                log_alpha: torch.Tensor, beta: torch.Tensor, *, out: Optional[torch.Tensor] = None,
                out_dtype=torch.bfloat16, stream=None, qk_norm: bool = False, q_scale: float = 1.0,
                norm_weight: Optional[torch.Tensor] = None, norm_eps: float = 1e-6,
                gate_scale: Optional[torch.Tensor] = None, gate_bias: Optional[torch.Tensor] = None,
                lib=None) -> torch.Tensor:
    """Run ``gdn_decode_step`` (state updated in place).  Returns ``out``.

    ``norm_weight`` (fp32 [dv]): fuse the output normalisation o / sqrt(mean(o^2) + norm_eps) * weight.
    ``lib``: a handle from :func:`bind` instead of the default library."""
    lib = lib or load_library()
    _need(state, "state", torch.float32, 4)
    _need(q, "q", torch.bfloat16, 3)
    _need(k, "k", torch.bfloat16, 3)
    _need(v, "v", torch.bfloat16, 3)
    _need(log_alpha, "log_alpha", torch.float32, 2)
    _need(beta, "beta", torch.float32, 2)
    n, hk, dk = q.shape
    hv, dv = v.shape[1], v.shape[2]
    if out is None:
        out = torch.empty(n, hv, dv, device=q.device, dtype=out_dtype)
    _gate_tensors(gate_scale, gate_bias, hv)
    _same_device(state.device, q=q, k=k, v=v, log_alpha=log_alpha, beta=beta, out=out, norm_weight=norm_weight,
                 gate_scale=gate_scale, gate_bias=gate_bias)
    with torch.cuda.device(state.device):
        st = lib.gdn_decode_step(n, hk, hv, dk, dv, _ptr(state), _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha),
                                 _ptr(beta), _ptr(out), DTYPE[out.dtype], int(bool(qk_norm)), float(q_scale),
                                 _ptr(norm_weight), float(norm_eps), _ptr(gate_scale), _ptr(gate_bias),
                                 _stream_ptr(stream, state.device))
    if st != GDN_OK:
        raise GdnError(st, "gdn_decode_step")
    return out


def device_error(stream=None, device=None, lib=None) -> int:
    """Synchronise and return the device-side error status (0 = none) of ``device`` (default: the current
    device; the error word is per device, shared by all of its streams) kept by ``lib`` (default library)."""
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(device):
        return int((lib or load_library()).gdn_device_error(_stream_ptr(stream, device)))


def selftest_bounded_wait(limit_us: int, stream=None) -> None:
    """Run ``gdn_selftest_bounded_wait``: one CTA waits for a barrier phase that nothing completes and gives
    up after ``limit_us`` microseconds, recording GDN_ERR_TIMEOUT for ``device_error`` to report."""
    st = load_library().gdn_selftest_bounded_wait(int(limit_us), _stream_ptr(stream))
    if st != GDN_OK:
        raise GdnError(st, "gdn_selftest_bounded_wait")
