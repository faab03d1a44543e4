"""Host logic of the chunked path's state pass: how sequences are grouped into buckets (gdn_prefill_pass_plan).

A bucket is a run of consecutive sequences that one state-pass CTA per (value head, 32-row slice) carries one
after another.  The host picks one wave of multi-sequence buckets or one bucket per sequence from the chunk
counts alone; these tests check the plan's invariants and the crossover points that the GB300 sweep of N
sequences of T tokens measured (one bucket up to 256 tokens per sequence for eight sequences, one per sequence
from 512).  No GPU is needed.
"""
import ctypes
import itertools

import numpy as np
import pytest

from gated_deltanet_linear_03_gb300 import gdn

SLICES = 4   # 32-row slices of a d = 128 head: CTAs per (bucket, value head)
GB300_SMS = 152


@pytest.fixture(scope="module", autouse=True)
def lib():
    from gated_deltanet_linear_03_gb300 import _build
    _build.build()
    return gdn.load_library()


def cu(lengths):
    return [0] + list(itertools.accumulate(int(x) for x in lengths))


def chunks(lengths):
    return [(int(x) + 63) // 64 for x in lengths]


def plan(lengths, hv=32, sms=GB300_SMS):
    return gdn.pass_plan(cu(lengths), hv, sms)


def random_lengths(rng, n):
    kind = rng.integers(3)
    if kind == 0:
        return rng.integers(0, 200, n)
    if kind == 1:
        return np.exp(rng.uniform(0, np.log(20000), n)).astype(int)
    return rng.choice([0, 1, 63, 64, 65, 128, 700, 4096], n)


@pytest.mark.parametrize("seed", range(40))
def test_buckets_partition_the_sequences_in_order(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 90))
    lengths = random_lengths(rng, n)
    hv = int(rng.choice([1, 3, 8, 32, 64]))
    sms = int(rng.choice([8, 132, 152, 1000]))
    p = plan(lengths, hv, sms)
    nb = len(p) - 1
    assert p[0] == 0 and p[-1] == n
    assert all(a < b for a, b in zip(p, p[1:])), p
    assert 1 <= nb <= n
    if 1 < nb < n:   # several sequences per bucket only as one wave of CTAs (at most 64 buckets)
        assert nb * hv * SLICES <= sms and nb <= 64, (nb, hv, sms)


def test_crossover_points_of_the_sweep():
    assert plan([4096]) == [0, 1]
    for t in (1, 64, 128, 256):
        assert plan([t] * 8) == [0, 8], t           # eight short sequences share the CTAs of one bucket
    for t in (512, 1024, 4096):
        assert plan([t] * 8) == list(range(9)), t   # long ones get one bucket each


def test_plan_depends_on_chunk_counts_only():
    rng = np.random.default_rng(7)
    for _ in range(20):
        c = rng.integers(0, 40, int(rng.integers(1, 30)))
        full = [64 * x for x in c]
        ragged = [0 if x == 0 else 64 * (x - 1) + int(rng.integers(1, 65)) for x in c]
        assert chunks(full) == chunks(ragged)
        assert plan(full, 8) == plan(ragged, 8)


def test_one_sequence_is_one_bucket_whatever_its_length():
    for t in (0, 1, 64, 65, 131072):
        assert plan([t]) == [0, 1]


def test_empty_sequences_only():
    assert plan([0, 0, 0]) == [0, 3]


def test_equal_sequences_split_evenly():
    # hv = 8: 32 CTAs per bucket, so up to four buckets fit one wave of 152 SMs
    p = plan([640] * 16, hv=8)
    sizes = [b - a for a, b in zip(p, p[1:])]
    assert max(sizes) - min(sizes) <= 1, p


def test_multi_bucket_layout_balances_chunks():
    # the longest bucket carries no more than an even share of the chunks plus one sequence
    rng = np.random.default_rng(11)
    for _ in range(30):
        lengths = rng.integers(1, 3000, int(rng.integers(5, 40)))
        p = plan(lengths, hv=8)
        nb = len(p) - 1
        if nb in (1, len(lengths)):
            continue
        c = chunks(lengths)
        per = [sum(c[a:b]) for a, b in zip(p, p[1:])]
        assert max(per) <= -(-sum(c) // nb) + max(c), (per, c)


def test_invalid_arguments_are_refused(lib):
    arr = (ctypes.c_int32 * 3)(0, 10, 20)
    out = (ctypes.c_int * 3)()
    assert lib.gdn_prefill_pass_plan(2, 20, 0, arr, 152, out, 3) == -1     # hv < 1
    assert lib.gdn_prefill_pass_plan(2, 20, 8, arr, 0, out, 3) == -1       # no multiprocessors
    assert lib.gdn_prefill_pass_plan(2, 21, 8, arr, 152, out, 3) == -1     # cu_seqlens does not end at T
    assert lib.gdn_prefill_pass_plan(2, 20, 8, arr, 152, None, 3) == -1    # no output array
    bad = (ctypes.c_int32 * 3)(0, 15, 10)
    assert lib.gdn_prefill_pass_plan(2, 10, 8, bad, 152, out, 3) == -1     # decreasing
    long8 = (ctypes.c_int32 * 9)(*cu([1024] * 8))
    out9 = (ctypes.c_int * 9)()
    assert lib.gdn_prefill_pass_plan(8, 8192, 32, long8, 152, out9, 8) == -1   # 9 entries needed
    assert lib.gdn_prefill_pass_plan(8, 8192, 32, long8, 152, out9, 9) == 8
