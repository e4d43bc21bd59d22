"""Dense decode over a paged cache of FP8 records, on the GPU through the C ABI,
against the oracle (dense_fp8_decode)."""

import numpy as np
import pytest
import torch

import mla_paged_kv_gb300 as mla
from mla_paged_kv_gb300 import workloads as wl
from oracle import mla_oracle as orc
from tests.parity import compare

pytestmark = pytest.mark.gpu


def run(case, num_parts=None, block_table=None):
    q, kv8 = case.q.cuda(), case.kv8.cuda()
    bt = (case.block_table if block_table is None else block_table).cuda()
    sl = case.cache_seqlens.cuda()
    B, s_q, h_q = case.batch, case.s_q, case.h_q
    ul = torch.empty(B * s_q, dtype=torch.int32, device="cuda")
    mla.mla_dense_fp8_unit_lengths(sl, s_q, case.causal, ul)
    pl = mla.plan(ul, B * s_q, h_q, sparse=True, num_parts=num_parts, device=torch.device("cuda"))
    out = torch.full((B, s_q, h_q, 512), float("nan"), device="cuda", dtype=torch.bfloat16)
    lse = torch.full((B, s_q, h_q), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_dense_fp8_decode_fwd(q, kv8, bt, ul, pl.sched, pl.split_offset, pl.num_parts, pl.workspace, out, lse,
                                 status, case.scale)
    torch.cuda.synchronize()
    return out, lse, int(status.item()), ul.cpu()


def oracle(case):
    return orc.dense_fp8_decode(case.q.double().numpy(), case.kv8.numpy(), case.block_table.numpy(),
                                case.cache_seqlens.numpy(), case.causal, case.scale)


@pytest.mark.parametrize("h_q,s_q,causal,lens", [(16, 1, False, [1, 63]), (64, 1, False, [64, 65, 500]),
                                                 (128, 1, False, [2000, 130]), (128, 2, True, [2, 700]),
                                                 (64, 3, True, [3, 64, 1200]), (32, 2, False, [0, 300])])
def test_dense_fp8_small(h_q, s_q, causal, lens):
    case = wl.dense_fp8_case(len(lens), s_q, h_q, 0, seqlens=lens, causal=causal, seed=h_q + s_q + sum(lens))
    out, lse, st, _ = run(case)
    assert st == 0
    ro, rl = oracle(case)
    compare(out, lse, ro, rl)


@pytest.mark.parametrize("num_parts", [1, 7])
def test_dense_fp8_split_counts(num_parts):
    case = wl.dense_fp8_case(3, 2, 128, 0, seqlens=[900, 130, 2000], causal=True, seed=num_parts + 90)
    out, lse, st, _ = run(case, num_parts=num_parts)
    assert st == 0
    ro, rl = oracle(case)
    compare(out, lse, ro, rl)


def test_dense_fp8_unit_lengths_exact():
    case = wl.dense_fp8_case(4, 3, 16, 0, seqlens=[0, 1, 2, 500], causal=True, seed=91)
    _, _, _, ul = run(case)
    want = [max(L - 3 + i + 1, 0) for L in [0, 1, 2, 500] for i in range(3)]
    assert ul.tolist() == want


def test_dense_fp8_bad_page_is_reported_and_masked():
    case = wl.dense_fp8_case(2, 1, 64, 0, seqlens=[300, 200], seed=92)
    bt = case.block_table.clone()
    bt[0, 2] = case.kv8.shape[0] + 5                 # keys 128..191 of request 0 point outside the pool
    out, lse, st, _ = run(case, block_table=bt)
    assert st == 5                                   # MLA_ERR_BAD_INDEX
    # the oracle over every other slot (sparse selection with those 64 slots masked)
    ind = np.full((2, 1, 320), -1, dtype=np.int64)
    for b, L in enumerate([300, 200]):
        j = np.arange(L)
        ind[b, 0, :L] = case.block_table.numpy()[b, j // 64] * 64 + j % 64
    ind[0, 0, 128:192] = -1
    ro, rl, _ = orc.sparse_decode(case.q.double().numpy(), case.kv8.numpy(), ind, None, case.scale)
    compare(out, lse, ro, rl)
