"""Host-only checks of the C ABI: the library loads, exports every symbol that
include/gdn.h declares, and rejects invalid arguments before touching the GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from gated_deltanet_linear_03_gb300 import _build, gdn
    _build.build()
    return gdn.load_library()


def header_symbols():
    text = open(os.path.join(ROOT, "include", "gdn.h")).read()
    return set(re.findall(r"GDN_API\s+[\w\s\*]+?\b(gdn_\w+)\s*\(", text))


def test_header_declares_the_binding_exports():
    from gated_deltanet_linear_03_gb300 import gdn
    assert header_symbols() == set(gdn.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    for name in header_symbols():
        assert hasattr(lib, name), name


def test_version_and_status_strings(lib):
    assert lib.gdn_version() >= 100
    for code in range(8):
        s = lib.gdn_status_string(code).decode()
        assert s.startswith("GDN_")
    assert lib.gdn_status_string(99).decode() == "unknown gdn_status"


def _cu(vals):
    return (ctypes.c_int32 * len(vals))(*vals)


FAKE = 0x10000  # an aligned address that is never dereferenced: validation fails first


def prefill(lib, **kw):
    a = dict(n_seqs=1, T=64, hk=1, hv=2, dk=128, dv=128, q=FAKE, k=FAKE * 2, v=FAKE * 3, la=FAKE * 4,
             b=FAKE * 5, s0=None, cu=FAKE * 6, cu_host=_cu([0, 64]), out=FAKE * 7, odt=0, fin=None,
             algo=1, ws=None, wsb=0, qkn=0, qs=1.0, nw=None, ne=1e-6, gc=None, gb=None)
    a.update(kw)
    P = ctypes.c_void_p
    return lib.gdn_prefill(a["n_seqs"], a["T"], a["hk"], a["hv"], a["dk"], a["dv"], P(a["q"]), P(a["k"]),
                           P(a["v"]), P(a["la"]), P(a["b"]), P(a["s0"]), P(a["cu"]), a["cu_host"], P(a["out"]),
                           a["odt"], P(a["fin"]), a["qkn"], a["qs"], P(a["nw"]), a["ne"], P(a["gc"]), P(a["gb"]),
                           a["algo"], P(a["ws"]), a["wsb"], None)


def test_prefill_rejects_bad_heads(lib):
    assert prefill(lib, hk=3, hv=4) == 1          # hv % hk
    assert prefill(lib, dk=48, dv=48) == 2        # unsupported head size
    assert prefill(lib, dk=128, dv=64) == 2       # dk != dv
    assert prefill(lib, dk=64, dv=64, algo=0) == 2   # chunked path implements d = 128 only
    assert prefill(lib, hk=0) == 1


def test_prefill_rejects_bad_cu_seqlens(lib):
    assert prefill(lib, cu_host=_cu([0, 65])) == 1               # does not end at T
    assert prefill(lib, n_seqs=2, cu_host=_cu([0, 40, 30])) == 1  # decreasing
    assert prefill(lib, cu_host=_cu([1, 64])) == 1                # does not start at 0
    assert prefill(lib, cu_host=None) == 1
    assert prefill(lib, cu=None) == 1
    assert prefill(lib, n_seqs=0, cu_host=_cu([0])) == 1


def test_prefill_rejects_bad_dtype_algo_pointers(lib):
    assert prefill(lib, odt=7) == 2
    assert prefill(lib, qkn=2) == 1                 # qk_norm is 0 or 1
    assert prefill(lib, qkn=1, qs=float("inf")) == 1
    assert prefill(lib, qs=float("nan")) == 1
    assert prefill(lib, nw=FAKE * 50, ne=float("nan")) == 1
    assert prefill(lib, nw=FAKE * 50 + 8) == 3
    assert prefill(lib, algo=5) == 2
    assert prefill(lib, q=None) == 1
    assert prefill(lib, q=FAKE + 4) == 3          # misaligned
    assert prefill(lib, out=FAKE * 2) == 1        # out overlaps k
    assert prefill(lib, fin=FAKE * 3, s0=FAKE * 40) == 1   # final_state overlaps v
    assert prefill(lib, gc=FAKE * 60) == 1                 # gate_scale without gate_bias
    assert prefill(lib, gb=FAKE * 60) == 1
    assert prefill(lib, gc=FAKE * 60 + 4, gb=FAKE * 61) == 3   # misaligned gate parameters
    assert prefill(lib, gc=FAKE * 7, gb=FAKE * 61) == 1    # out overlaps gate_scale


def test_chunked_requires_workspace(lib):
    st = ctypes.c_int(-1)
    need = lib.gdn_prefill_workspace_size(1, 64, 1, 2, 128, 128, _cu([0, 64]), 0, ctypes.byref(st))
    assert st.value == 0
    if need > 0:
        assert prefill(lib, algo=0, ws=None, wsb=0) == 7
        assert prefill(lib, algo=0, ws=FAKE * 1000, wsb=need - 1) == 7
        assert prefill(lib, algo=0, ws=FAKE * 1000 + 16, wsb=need) == 3   # not 256-byte aligned


def test_workspace_size_validation(lib):
    st = ctypes.c_int(-1)
    assert lib.gdn_prefill_workspace_size(1, 64, 1, 2, 128, 128, _cu([0, 64]), 1, ctypes.byref(st)) == 0
    assert st.value == 0
    assert lib.gdn_prefill_workspace_size(1, 64, 3, 2, 128, 128, _cu([0, 64]), 0, ctypes.byref(st)) == 0
    assert st.value == 1
    assert lib.gdn_prefill_workspace_size(1, 64, 1, 2, 128, 128, _cu([0, 64]), 9, ctypes.byref(st)) == 0
    assert st.value == 2
    assert lib.gdn_prefill_workspace_size(1, 64, 1, 2, 64, 64, _cu([0, 64]), 0, ctypes.byref(st)) == 0
    assert st.value == 2


def test_decode_rejects_bad_args(lib):
    P = ctypes.c_void_p

    def dec(n=1, hk=1, hv=2, d=128, state=FAKE, q=FAKE * 2, k=FAKE * 3, v=FAKE * 4, la=FAKE * 5, b=FAKE * 6,
            out=FAKE * 7, odt=0, qkn=0, qs=1.0, nw=None, ne=1e-6, gc=None, gb=None):
        return lib.gdn_decode_step(n, hk, hv, d, d, P(state), P(q), P(k), P(v), P(la), P(b), P(out), odt, qkn, qs,
                                   P(nw), ne, P(gc), P(gb), None)

    assert dec(hk=3, hv=4) == 1
    assert dec(d=96) == 2
    assert dec(n=-1) == 1
    assert dec(n=0) == 0                     # nothing to do, nothing launched
    assert dec(state=None) == 1
    assert dec(q=FAKE + 8) == 3
    assert dec(odt=3) == 2
    assert dec(out=FAKE) == 1                # out overlaps state
    assert dec(qkn=-1) == 1
    assert dec(qs=float("inf")) == 1
    assert dec(nw=FAKE * 9, ne=-1.0) == 1    # negative eps
    assert dec(nw=FAKE * 9 + 4) == 3         # misaligned weight
    assert dec(gc=FAKE * 20) == 1            # gate_scale without gate_bias
    assert dec(gc=FAKE * 20, gb=FAKE * 21 + 8) == 3
    assert dec(gc=FAKE, gb=FAKE * 21) == 1   # gate_scale overlaps state


def test_auto_algo_rule(lib):
    """gdn_prefill_algo: the scan for short sequences (<= 16 tokens, or <= 32 with at most 64 (sequence,
    head) pairs) and whenever d != 128, the chunked path otherwise; -1 for invalid arguments."""
    algo = lambda n, hv, d, cu: lib.gdn_prefill_algo(n, cu[-1], 1, hv, d, d, _cu(cu))
    assert algo(1, 32, 128, [0, 16]) == 1
    assert algo(1, 32, 128, [0, 32]) == 1
    assert algo(1, 32, 128, [0, 33]) == 0
    assert algo(8, 32, 128, [0, 2, 4, 6, 8, 10, 12, 14, 16]) == 1
    assert algo(8, 32, 128, list(range(0, 9 * 24, 24))) == 0    # 256 (sequence, head) pairs of 24 tokens
    assert algo(2, 32, 128, [0, 1, 30]) == 1                     # 64 pairs, longest 29
    assert algo(1, 32, 128, [0, 4096]) == 0
    assert algo(1, 4, 64, [0, 4096]) == 1                        # chunked implements d = 128 only
    assert algo(1, 32, 128, [0, 5]) == 1
    assert lib.gdn_prefill_algo(1, 64, 3, 2, 128, 128, _cu([0, 64])) == -1   # hv % hk
    assert lib.gdn_prefill_algo(1, 64, 1, 2, 128, 128, _cu([0, 63])) == -1   # cu does not end at T


def test_auto_workspace_matches_resolved_algo(lib):
    st = ctypes.c_int(-1)
    for cu in ([0, 16], [0, 200], [0, 64, 200]):
        n = len(cu) - 1
        resolved = lib.gdn_prefill_algo(n, cu[-1], 1, 32, 128, 128, _cu(cu))
        want = lib.gdn_prefill_workspace_size(n, cu[-1], 1, 32, 128, 128, _cu(cu), resolved, ctypes.byref(st))
        got = lib.gdn_prefill_workspace_size(n, cu[-1], 1, 32, 128, 128, _cu(cu), 2, ctypes.byref(st))
        assert st.value == 0 and got == want
        assert (got == 0) == (resolved == 1)


def test_auto_requires_workspace_only_when_chunked(lib):
    # 200 tokens resolves to the chunked path, which needs a workspace
    assert prefill(lib, T=200, cu_host=_cu([0, 200]), algo=2, ws=None, wsb=0) == 7


# gdn_prefill_host: the staging layout and the checks made before anything is enqueued
def _r256(x):
    return (x + 255) // 256 * 256


def host_size(lib, T=64, n=1, hk=1, hv=2, d=128, odt=0, init=0, fin=1, algo=0, cu=None):
    st = ctypes.c_int(-1)
    cu = cu or _cu([0, T])
    size = lib.gdn_prefill_host_staging_size(n, T, hk, hv, d, d, cu, odt, init, fin, algo, ctypes.byref(st))
    return size, st.value


def test_host_staging_size_is_the_sum_of_its_pieces(lib):
    T, n, hk, hv, d = 200, 2, 2, 4, 128
    cu = _cu([0, 150, 200])
    st = ctypes.c_int(-1)
    ws = lib.gdn_prefill_workspace_size(n, T, hk, hv, d, d, cu, 0, ctypes.byref(st))
    assert st.value == 0 and ws > 0
    state = n * hv * d * d * 4
    for odt, ob in ((0, 2), (1, 4)):
        for init in (0, 1):
            for fin in (0, 1):
                expect = (2 * _r256(T * hk * d * 2) + _r256(T * hv * d * 2) + 2 * _r256(T * hv * 4)
                          + init * _r256(state) + _r256((n + 1) * 4) + _r256(T * hv * d * ob)
                          + fin * _r256(state) + _r256(ws))
                size, s = host_size(lib, T, n, hk, hv, d, odt, init, fin, 0, cu)
                assert s == 0 and size == expect, (odt, init, fin)
    size, s = host_size(lib, T, n, hk, hv, d, 0, 0, 1, 1, cu)   # the scan needs no workspace
    assert s == 0 and size == (2 * _r256(T * hk * d * 2) + _r256(T * hv * d * 2) + 2 * _r256(T * hv * 4)
                               + _r256((n + 1) * 4) + _r256(T * hv * d * 2) + _r256(state))


def test_host_staging_size_rejects_invalid_problems(lib):
    assert host_size(lib, hk=3, hv=4) == (0, 1)
    assert host_size(lib, d=64, algo=0) == (0, 2)          # chunked path implements d = 128 only
    assert host_size(lib, odt=5) == (0, 2)
    assert host_size(lib, cu=_cu([0, 63])) == (0, 1)
    assert host_size(lib, algo=9) == (0, 2)


def prefill_host(lib, **kw):
    a = dict(n_seqs=1, T=64, hk=1, hv=2, dk=128, dv=128, q=FAKE, k=FAKE, v=FAKE, la=FAKE, b=FAKE, s0=None,
             cu_host=_cu([0, 64]), out=FAKE, odt=0, fin=FAKE, qkn=0, qs=1.0, nw=None, ne=1e-6, gc=None,
             gb=None, algo=0, stg=FAKE * 16, stgb=1 << 40)
    a.update(kw)
    P = ctypes.c_void_p
    return lib.gdn_prefill_host(a["n_seqs"], a["T"], a["hk"], a["hv"], a["dk"], a["dv"], P(a["q"]), P(a["k"]),
                                P(a["v"]), P(a["la"]), P(a["b"]), P(a["s0"]), a["cu_host"], P(a["out"]), a["odt"],
                                P(a["fin"]), a["qkn"], a["qs"], P(a["nw"]), a["ne"], P(a["gc"]), P(a["gb"]),
                                a["algo"], P(a["stg"]), a["stgb"], None)


def test_prefill_host_validates_before_enqueueing(lib):
    need, s = host_size(lib)
    assert s == 0
    assert prefill_host(lib, stgb=need - 1) == 7            # staging too small
    assert prefill_host(lib, stg=None) == 7
    assert prefill_host(lib, stg=FAKE * 16 + 128) == 3      # staging not 256-byte aligned
    assert prefill_host(lib, q=None) == 1
    assert prefill_host(lib, out=None) == 1
    assert prefill_host(lib, qkn=2) == 1
    assert prefill_host(lib, qs=float("nan")) == 1
    assert prefill_host(lib, nw=FAKE + 4) == 3              # norm_weight is a 16-byte aligned device array
    assert prefill_host(lib, nw=FAKE, ne=-1.0) == 1
    assert prefill_host(lib, odt=3) == 2
    assert prefill_host(lib, hk=3, hv=4) == 1
    assert prefill_host(lib, cu_host=_cu([0, 65])) == 1
    assert prefill_host(lib, gb=FAKE) == 1                   # gate_bias without gate_scale
    assert prefill_host(lib, T=0, cu_host=_cu([0, 0]), fin=None) == 0   # nothing to do: returns at once


def test_selftest_bounded_wait_rejects_limits_out_of_range(lib):
    # validated on the host before anything is launched
    for bad in (0, -5, 1000001):
        assert lib.gdn_selftest_bounded_wait(bad, None) == 1  # GDN_ERR_INVALID_ARG


def test_pointers_off_the_current_device_are_refused(lib):
    """A well-formed call whose pointers are not device memory of the current device is refused before any
    launch: GDN_ERR_INVALID_ARG where a GPU is present, GDN_ERR_CUDA (the runtime cannot be asked) without
    one.  FAKE is an address that no allocation owns."""
    allowed = {1, 4}
    assert prefill(lib) in allowed
    assert prefill_host(lib, stgb=1 << 40) in allowed

    def dec():
        P = ctypes.c_void_p
        return lib.gdn_decode_step(1, 1, 2, 128, 128, P(FAKE), P(FAKE * 2), P(FAKE * 3), P(FAKE * 4), P(FAKE * 5),
                                   P(FAKE * 6), P(FAKE * 7), 0, 0, 1.0, None, 1e-6, None, None, None)
    assert dec() in allowed


@pytest.mark.gpu
def test_host_memory_is_refused_on_a_gpu(lib):
    """Host tensors in place of device tensors: GDN_ERR_INVALID_ARG, nothing launched, no device error."""
    import torch
    from gated_deltanet_linear_03_gb300 import gdn, synth
    inp = synth.prefill_inputs([64], hk=1, hv=2, seed=3)
    dev = torch.device("cuda:0")
    d = [t.to(dev) for t in (inp.q, inp.k, inp.v, inp.log_alpha, inp.beta, inp.cu_seqlens)]
    out_dev = torch.empty(64, 2, 128, dtype=torch.bfloat16, device=dev)
    P = ctypes.c_void_p
    host_q = inp.q.contiguous()
    cu = _cu(inp.cu_seqlens.tolist())
    with torch.cuda.device(dev):
        for q_ptr, out_ptr in ((host_q.data_ptr(), out_dev.data_ptr()), (d[0].data_ptr(), host_q.data_ptr())):
            st = lib.gdn_prefill(1, 64, 1, 2, 128, 128, P(q_ptr), P(d[1].data_ptr()), P(d[2].data_ptr()),
                                 P(d[3].data_ptr()), P(d[4].data_ptr()), None, P(d[5].data_ptr()), cu, P(out_ptr), 0,
                                 None, 0, 1.0, None, 1e-6, None, None, 1, None, 0, None)
            assert st == 1
        state = torch.zeros(1, 2, 128, 128, dtype=torch.float32)            # host state
        st = lib.gdn_decode_step(1, 1, 2, 128, 128, P(state.data_ptr()), P(d[0].data_ptr()), P(d[1].data_ptr()),
                                 P(d[2].data_ptr()), P(d[3].data_ptr()), P(d[4].data_ptr()), P(out_dev.data_ptr()),
                                 0, 0, 1.0, None, 1e-6, None, None, None)
        assert st == 1
    assert gdn.device_error() == 0
