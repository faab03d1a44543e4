"""GB300 (sm_103a) Gated DeltaNet recurrence: chunked and direct-scan prefill,
batch decode step, behind the C ABI in include/gdn.h.

    from gated_deltanet_linear_03_gb300 import gdn
    out, final_state = gdn.prefill(q, k, v, log_alpha, beta, cu_seqlens)
    out = gdn.decode_step(state, q, k, v, log_alpha, beta)

The binding (``gdn``) is imported lazily so that ``synth`` (input generators)
can be used without loading the CUDA library.
"""
import importlib

__all__ = ["gdn", "synth"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
