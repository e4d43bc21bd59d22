"""The device timeout paths on a real GPU, in a form that faults and hangs
nothing.

The test instance of the pack kernel withholds the arrival that completes
each block's bulk-copy barrier, so that block's bounded wait (200 us) runs
out.  The block must report MLA_ERR_TIMEOUT, give its tile a zero mask, make
the withheld arrival, wait for its own copies and exit without storing.

The test instance of the dense decode kernel never loads the first own K
tile of each CTA, and its waits have a 200 us budget: the Q K^T thread's
wait runs out, the CTA unwinds every role, the peer CTA's waits for the
messages that never come run out as well, and the grid ends.  For a cache
of FP8 records the same hook runs the test instance of the sparse kernel,
which never computes the first tile's scores: the softmax warps' wait for
them runs out, the pairs of warps leave their named barriers together, the
producers leave theirs together, and the MMA thread drains and frees TMEM.

Either way the context and the stream must stay usable, which a normal
call right after checks against the oracle."""

import numpy as np
import pytest
import torch

import mla_paged_kv_gb300 as mla
from mla_paged_kv_gb300 import workloads as wl
from oracle import mla_oracle as orc
from tests.parity import compare, dense_oracle, to_dev

pytestmark = pytest.mark.gpu

MLA_ERR_TIMEOUT = 4


def test_pack_wait_runs_out_reports_timeout_and_the_next_call_is_exact():
    case = wl.sparse_case(2, 1, 16, topk=192, pages_per_req=8, topk_lengths=[[192], [70]], seed=99)
    kv8, ind, tl = case.kv8.cuda(), case.indices.cuda(), case.topk_length.cuda()
    n_bytes = mla.mla_packed_kv_workspace_bytes(2, 192)
    rec_bytes = 2 * 3 * 64 * 656
    packed = torch.full((n_bytes,), 0xAB, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_test_pack_timeout(kv8, ind, tl, packed, status)
    torch.cuda.synchronize()
    assert int(status.item()) == MLA_ERR_TIMEOUT
    got = packed.cpu().numpy()
    assert not got[rec_bytes:].any()                  # every tile's mask is zero
    assert (got[:rec_bytes] == 0xAB).all()            # no record was stored

    # same process, same stream: the normal pack is unaffected
    packed.fill_(0xAB)
    status.zero_()
    mla.mla_pack_selected_kv(kv8, ind, tl, packed, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref, bad = orc.pack_selected(case.kv8.numpy(), case.indices.numpy(), case.topk_length.numpy())
    assert bad == 0 and np.array_equal(packed.cpu().numpy(), ref)


@pytest.mark.parametrize("lens", [[700, 300], [64, 2000, 1]])
def test_dense_decode_wait_runs_out_reports_timeout_and_the_next_call_is_exact(lens):
    import time
    case = wl.dense_case(len(lens), 1, 64, 0, seqlens=lens, seed=97 + len(lens))
    c = to_dev(case)
    B = case.batch
    pl = mla.plan(c.cache_seqlens, B, 64, num_parts=mla.mla_num_parts_dense(1, 64, 1))
    out = torch.zeros(B, 1, 64, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(B, 1, 64, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    mla.mla_test_decode_timeout(c.q, c.kv, c.block_table, c.cache_seqlens, pl.sched, pl.split_offset,
                                pl.num_parts, pl.workspace, out, lse, status, False, case.scale)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(status.item()) == MLA_ERR_TIMEOUT
    assert elapsed < 1.5                              # the 200 us budgets, not the 2 s ones

    # same process, same stream: the normal decode is unaffected
    status.zero_()
    out.fill_(float("nan"))
    mla.mla_decode_fwd(c.q, c.kv, c.block_table, c.cache_seqlens, pl.sched, pl.split_offset, pl.num_parts,
                       pl.workspace, out, lse, status, False, case.scale)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ro, rl = dense_oracle(case)
    compare(out, lse, ro, rl)


@pytest.mark.parametrize("lens", [[700, 300], [64, 2000, 1]])
def test_fp8_record_decode_wait_runs_out_reports_timeout_and_the_next_call_is_exact(lens):
    import time
    case = wl.dense_fp8_case(len(lens), 1, 64, 0, seqlens=lens, seed=91 + len(lens))
    q, kv8, bt, sl = case.q.cuda(), case.kv8.cuda(), case.block_table.cuda(), case.cache_seqlens.cuda()
    B = case.batch
    pl = mla.plan(sl, B, 64, num_parts=mla.mla_num_parts_dense(1, 64, 1))
    out = torch.zeros(B, 1, 64, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(B, 1, 64, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    mla.mla_test_decode_timeout(q, kv8, bt, sl, pl.sched, pl.split_offset, pl.num_parts, pl.workspace, out, lse,
                                status, False, case.scale)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(status.item()) == MLA_ERR_TIMEOUT
    assert elapsed < 1.5                              # the 200 us budgets, not the 2 s ones

    status.zero_()
    out.fill_(float("nan"))
    mla.mla_decode_fwd(q, kv8, bt, sl, pl.sched, pl.split_offset, pl.num_parts, pl.workspace, out, lse, status,
                       False, case.scale)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ro, rl = orc.dense_fp8_decode(case.q.double().numpy(), case.kv8.numpy(), case.block_table.numpy(),
                                  case.cache_seqlens.numpy(), False, case.scale)
    compare(out, lse, ro, rl)
