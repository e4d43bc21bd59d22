"""The scheduler kernel's metadata equals the restated plan, integer for
integer, on random cases: zero-length units, more partitions than tiles,
one partition, and more units than the kernel keeps in shared memory."""

import numpy as np
import pytest
import torch

import mla_paged_kv_gb300 as mla
from oracle import mla_sched

pytestmark = pytest.mark.gpu


def _gpu_plan(lengths, num_parts, default_length=-1, request_local=False):
    n = len(lengths) if lengths is not None else 1
    sched = torch.full((num_parts * 8,), -7, dtype=torch.int32, device="cuda")
    off = torch.full((n + 1,), -7, dtype=torch.int32, device="cuda")
    d = None if lengths is None else torch.tensor(lengths, dtype=torch.int32, device="cuda")
    fn = mla.mla_get_metadata_request_local if request_local else mla.mla_get_metadata
    fn(d, n, num_parts, sched, off, default_length)
    torch.cuda.synchronize()
    return sched.cpu().reshape(-1, 8).tolist(), off.cpu().tolist()


@pytest.mark.parametrize("seed,n,parts,lo,hi,zero_frac", [
    (1, 64, 76, 2048, 4096, 0.0),
    (2, 1, 76, 65536, 65536, 0.0),
    (3, 16, 38, 4096, 8192, 0.0),
    (4, 50, 7, 0, 300, 0.3),
    (5, 300, 152, 1, 5000, 0.1),
    (6, 5000, 76, 0, 700, 0.2),
    (7, 9, 1, 10, 2000, 0.0),
    (8, 3, 200, 1, 130, 0.0),
])
def test_sched_kernel_matches_plan(seed, n, parts, lo, hi, zero_frac):
    rng = np.random.default_rng(seed)
    lens = rng.integers(lo, hi + 1, size=n)
    lens[rng.random(n) < zero_frac] = 0
    lens = lens.tolist()
    ref_sched, ref_off = mla_sched.plan(lens, parts, 4)
    sched, off = _gpu_plan(lens, parts)
    assert sched == [list(e) for e in ref_sched]
    assert off == ref_off


def test_sched_kernel_cap_search_by_hand():
    """Requests of 2, 1, 1, 1 tiles over 4 partitions (F = 4): the plan's cap is
    c0 = 6, one request per partition (tests/test_sched.py works it out); the
    plain cap c0 + F = 10 would leave the last partition empty."""
    sched, off = _gpu_plan([128, 64, 64, 64], 4)
    assert sched == [[0, 0, 1, 0, 0, 0, 0, 0], [1, 0, 2, 0, 0, 0, 0, 0], [2, 0, 3, 0, 0, 0, 0, 0],
                     [3, 0, 4, 0, 0, 0, 0, 0]]
    assert off == [0, 1, 2, 3, 4]


@pytest.mark.parametrize("parts", [76, 128, 129])
def test_sched_kernel_search_limit(parts):
    """At most 128 partitions take the cap search; 129 take the single walk with
    c0 + F.  Both sides apply the same limit."""
    rng = np.random.default_rng(parts)
    lens = rng.integers(1, 3000, size=40).tolist()
    ref_sched, ref_off = mla_sched.plan(lens, parts, 4)
    sched, off = _gpu_plan(lens, parts)
    assert sched == [list(e) for e in ref_sched]
    assert off == ref_off


def test_sched_kernel_default_length():
    ref_sched, ref_off = mla_sched.plan([2048], 76, 4)
    sched, off = _gpu_plan(None, 76, default_length=2048)
    assert sched == [list(e) for e in ref_sched]
    assert off == ref_off


@pytest.mark.parametrize("seed,n,parts,lo,hi,zero_frac", [
    (11, 16, 76, 64, 2048, 0.0),        # sparse-like: 16 query tokens, top-k lengths
    (12, 64, 76, 2048, 4096, 0.0),
    (13, 76, 76, 1, 5000, 0.0),         # one part per unit
    (14, 40, 76, 0, 3000, 0.3),
    (15, 100, 76, 1, 500, 0.0),         # more units than parts: native plan
    (16, 3, 200, 1, 130, 0.0),          # units run out of tiles before parts run out
    (17, 1000, 1024, 0, 4000, 0.5),
    (18, 2000, 76, 0, 100, 0.99),       # above the request-local unit limit: native plan
])
def test_request_local_kernel_matches_plan(seed, n, parts, lo, hi, zero_frac):
    rng = np.random.default_rng(seed)
    lens = rng.integers(lo, hi + 1, size=n)
    lens[rng.random(n) < zero_frac] = 0
    lens = lens.tolist()
    if n > 1024:
        ref_sched, ref_off = mla_sched.plan(lens, parts, 4)
    else:
        ref_sched, ref_off = mla_sched.plan_request_local(lens, parts, 4)
    sched, off = _gpu_plan(lens, parts, request_local=True)
    assert sched == [list(e) for e in ref_sched]
    assert off == ref_off
