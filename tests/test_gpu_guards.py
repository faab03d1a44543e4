"""Guard canaries: no kernel writes outside the buffers it is given.

compute-sanitizer is not available on these GPUs, so stray writes are looked for
directly.  Every buffer a call writes (out, final_state, the workspace, the
decode state, the host call's staging) is carved out of a larger allocation
whose bands on both sides hold a known byte pattern; after the call the bands
must be intact.  The cases are the ones where addressing is most delicate:
ragged packing with empty, 1-token and partial-chunk sequences, every head
grouping, the short-sequence scan, fp32 and bf16 outputs, and the 128K-token
layer, whose workspace offsets run past 2^31 bytes.
"""
import pytest
import torch

from gated_deltanet_linear_03_gb300 import synth
from helpers import to_device

pytestmark = pytest.mark.gpu

GUARD = 1 << 16        # guard band on each side, bytes
PATTERN = 0xA5


@pytest.fixture(scope="module")
def gdn():
    from gated_deltanet_linear_03_gb300 import gdn as g
    g.load_library()
    return g


class Guarded:
    """A device buffer of `shape`/`dtype` between two guard bands of PATTERN bytes (256-byte aligned)."""

    def __init__(self, shape, dtype, device="cuda"):
        numel = 1
        for s in shape:
            numel *= s
        self.nbytes = numel * torch.empty((), dtype=dtype).element_size()
        self.raw = torch.full((GUARD + ((self.nbytes + 255) // 256) * 256 + GUARD,), PATTERN, dtype=torch.uint8,
                              device=device)
        self.tensor = self.raw[GUARD:GUARD + self.nbytes].view(dtype).view(*shape)

    def intact(self) -> bool:
        lo = self.raw[:GUARD]
        hi = self.raw[GUARD + self.nbytes:]
        return bool((lo == PATTERN).all().item()) and bool((hi == PATTERN).all().item())


def run_guarded(gdn, inp, algo, out_dtype, **kw):
    d = to_device(inp)
    T, hk, dk = inp.q.shape
    hv, dv = inp.v.shape[1], inp.v.shape[2]
    n = inp.cu_seqlens.numel() - 1
    cu = inp.cu_seqlens.tolist()
    out = Guarded((T, hv, dv), out_dtype)
    fin = Guarded((n, hv, dv, dk), torch.float32)
    need = gdn.workspace_size(n, T, hk, hv, dk, dv, cu, algo)
    ws = Guarded((max(need, 1),), torch.uint8)
    gdn.prefill(d.q, d.k, d.v, d.log_alpha, d.beta, d.cu_seqlens, init_state=d.init_state, out=out.tensor,
                final_state=fin.tensor, algo=algo, workspace=ws.tensor if need else None, cu_seqlens_host=cu, **kw)
    torch.cuda.synchronize()
    assert gdn.device_error() == 0
    return out, fin, ws


CASES = {
    "ragged": lambda: synth.prefill_inputs([1, 63, 64, 65, 130, 0, 7], seed=91, init_std=0.02),
    "group4": lambda: synth.prefill_inputs([129, 64], hk=2, hv=8, seed=92, init_std=0.05),
    "group3_gates": lambda: synth.prefill_inputs([77, 1], hk=1, hv=3, seed=93, raw_gates="per_head"),
    "short_many": lambda: synth.prefill_inputs([32, 5, 17, 1, 32, 9, 30, 2], seed=94, init_std=0.02),
    "buckets": lambda: synth.prefill_inputs([0, 65, 1, 0, 130, 64, 3, 0], seed=99, init_std=0.02),   # one state-pass CTA carries all eight
}


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("algo", ["chunked", "scan"])
@pytest.mark.parametrize("case", list(CASES))
def test_prefill_writes_stay_inside(gdn, case, algo, out_dtype):
    inp = CASES[case]()
    kw = {}
    if inp.gate_scale is not None:
        kw = dict(gate_scale=inp.gate_scale.cuda(), gate_bias=inp.gate_bias.cuda())
    out, fin, ws = run_guarded(gdn, inp, algo, out_dtype, **kw)
    assert out.intact() and fin.intact() and ws.intact(), case


def test_fused_options_write_stay_inside(gdn):
    """q/k preparation and the output normalisation (cluster kernels) together."""
    inp = synth.prefill_inputs([200, 3, 64], seed=95, init_std=0.02, raw_qk=True)
    w = torch.linspace(0.5, 2.0, 128, device="cuda")
    for algo in ("chunked", "scan"):
        out, fin, ws = run_guarded(gdn, inp, algo, torch.bfloat16, qk_norm=True, q_scale=0.088, norm_weight=w)
        assert out.intact() and fin.intact() and ws.intact(), algo


def test_long_layer_writes_stay_inside(gdn):
    """131072 tokens: 2048 chunks x 32 heads; the workspace is 3.2 GB, its offsets pass 2^31 bytes."""
    inp = synth.prefill_inputs([131072], seed=96, device="cuda")
    out, fin, ws = run_guarded(gdn, inp, "chunked", torch.bfloat16)
    assert out.intact() and fin.intact() and ws.intact()


def test_decode_writes_stay_inside(gdn):
    di = synth.decode_inputs(5, 1, seed=97)
    state = Guarded(tuple(di.state.shape), torch.float32)
    state.tensor.copy_(di.state.cuda())
    out = Guarded((5, 32, 128), torch.bfloat16)
    args = [x[0].cuda() for x in (di.q, di.k, di.v, di.log_alpha, di.beta)]
    w = torch.linspace(0.5, 2.0, 128, device="cuda")
    for kw in ({}, dict(norm_weight=w), dict(qk_norm=True, q_scale=0.1)):
        gdn.decode_step(state.tensor, *args, out=out.tensor, **kw)
        torch.cuda.synchronize()
        assert state.intact() and out.intact(), kw
    assert gdn.device_error() == 0


def test_host_call_staging_stays_inside(gdn):
    inp = synth.prefill_inputs([300, 65, 1], hk=4, hv=8, seed=98, init_std=0.02)
    cu = inp.cu_seqlens.tolist()
    need = gdn.host_staging_size(3, 366, 4, 8, 128, 128, cu, init_state=True)
    stg = Guarded((need,), torch.uint8)
    hq = [t.contiguous().pin_memory() for t in (inp.q, inp.k, inp.v, inp.log_alpha, inp.beta)]
    gdn.prefill_host(*hq, cu, init_state=inp.init_state.pin_memory(), staging=stg.tensor)
    assert stg.intact()
    assert gdn.device_error() == 0
