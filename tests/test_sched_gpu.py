"""The scheduler kernel's metadata equals the restated plan, integer for
integer, on random cases: zero-length units, more partitions than tiles,
one partition, and more units than the kernel keeps in shared memory."""

import numpy as np
import pytest
import torch

import mla_paged_kv_gb300 as mla
from oracle import mla_sched

pytestmark = pytest.mark.gpu


def _gpu_plan(lengths, num_parts, default_length=-1):
    n = len(lengths) if lengths is not None else 1
    sched = torch.full((num_parts * 8,), -7, dtype=torch.int32, device="cuda")
    off = torch.full((n + 1,), -7, dtype=torch.int32, device="cuda")
    d = None if lengths is None else torch.tensor(lengths, dtype=torch.int32, device="cuda")
    mla.mla_get_metadata(d, n, num_parts, sched, off, default_length)
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


def test_sched_kernel_default_length():
    ref_sched, ref_off = mla_sched.plan([2048], 76, 4)
    sched, off = _gpu_plan(None, 76, default_length=2048)
    assert sched == [list(e) for e in ref_sched]
    assert off == ref_off
