"""Dense decode over a paged cache of FP8 records (mla_decode_fwd with
MLA_DTYPE_FP8_RECORD), on the GPU through the C ABI, against the oracle
(dense_fp8_decode).  The records are FlashMLA PR #200's ("FP8 KV cache
format"); the path runs the sparse kernel with the block table as its slot
source, a whole request as its unit and the dense plan, so the scores stay
exact in codes and scales and the plain bars hold for peaky queries too."""

import dataclasses

import numpy as np
import pytest
import torch

import mla_paged_kv_gb300 as mla
from mla_paged_kv_gb300 import workloads as wl
from oracle import mla_oracle as orc
from tests.parity import compare

pytestmark = pytest.mark.gpu


def run(case, num_parts=None, block_table=None, out_dtype=torch.bfloat16):
    q, kv8 = case.q.cuda(), case.kv8.cuda()
    bt = (case.block_table if block_table is None else block_table).cuda()
    sl = case.cache_seqlens.cuda()
    B, s_q, h_q = case.batch, case.s_q, case.h_q
    if num_parts is None:
        num_parts = mla.mla_num_parts_dense(s_q, h_q, 1)
    pl = mla.plan(sl, B, s_q * h_q, num_parts=num_parts)
    out = torch.full((B, s_q, h_q, 512), float("nan"), device="cuda", dtype=out_dtype)
    lse = torch.full((B, s_q, h_q), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_decode_fwd(q, kv8, bt, sl, pl.sched, pl.split_offset, pl.num_parts, pl.workspace, out, lse, status,
                       case.causal, case.scale)
    torch.cuda.synchronize()
    return out, lse, int(status.item())


def oracle(case, block_table=None):
    bt = case.block_table if block_table is None else block_table
    return orc.dense_fp8_decode(case.q.double().numpy(), case.kv8.numpy(), bt.numpy(),
                                case.cache_seqlens.numpy(), case.causal, case.scale)


# h_q = 64 with s_q = 3: 192 rows, two row blocks, the first holding tokens
# 0 and 1; h_q = 128 with s_q = 2: one token per row block
@pytest.mark.parametrize("h_q,s_q,causal,lens", [(16, 1, False, [1, 63]), (64, 1, False, [64, 65, 500]),
                                                 (128, 1, False, [2000, 130]), (128, 2, True, [2, 700]),
                                                 (64, 3, True, [3, 64, 1200]), (32, 2, False, [0, 300]),
                                                 (128, 4, True, [1, 127, 129]), (16, 8, True, [8, 65])])
def test_dense_fp8_small(h_q, s_q, causal, lens):
    case = wl.dense_fp8_case(len(lens), s_q, h_q, 0, seqlens=lens, causal=causal, seed=h_q + s_q + sum(lens))
    out, lse, st = run(case)
    assert st == 0
    ro, rl = oracle(case)
    compare(out, lse, ro, rl)


@pytest.mark.parametrize("num_parts", [1, 7, 40])
def test_dense_fp8_split_counts(num_parts):
    case = wl.dense_fp8_case(3, 2, 128, 0, seqlens=[900, 130, 2000], causal=True, seed=num_parts + 90)
    out, lse, st = run(case, num_parts=num_parts)
    assert st == 0
    ro, rl = oracle(case)
    compare(out, lse, ro, rl)


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.float16])
def test_dense_fp8_peaky_queries_meet_the_plain_bars(out_dtype):
    """q x 8 exercises the running-max rescale; with exact scores the plain
    bars hold (no separate bound), in every output type, and a second call
    gives the same bits."""
    case = wl.dense_fp8_case(2, 1, 128, 0, seqlens=[1500, 333], q_scale=8.0, seed=193)
    o1, l1, st = run(case, out_dtype=out_dtype)
    assert st == 0 and o1.dtype == out_dtype
    ro, rl = oracle(case)
    compare(o1, l1, ro, rl)
    o2, l2, _ = run(case, out_dtype=out_dtype)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("num_parts", [1, 5])
def test_dense_fp8_direct_and_combined_outputs(num_parts):
    """One split per request (num_parts 1: written by the decode kernel
    itself) and several (through the combine), for each output type."""
    case = wl.dense_fp8_case(2, 2, 64, 0, seqlens=[700, 64], causal=True, seed=199)
    ro, rl = oracle(case)
    for dt in (torch.bfloat16, torch.float16, torch.float32):
        out, lse, st = run(case, num_parts=num_parts, out_dtype=dt)
        assert st == 0
        compare(out, lse, ro, rl)


def test_dense_fp8_bad_page_is_reported_and_masked():
    case = wl.dense_fp8_case(2, 1, 64, 0, seqlens=[300, 200], seed=195)
    bt = case.block_table.clone()
    bt[0, 2] = case.kv8.shape[0] + 5                 # keys 128..191 of request 0 point outside the pool
    out, lse, st = run(case, block_table=bt)
    assert st == 5                                   # MLA_ERR_BAD_INDEX
    ro, rl = oracle(case, block_table=bt)            # the oracle masks those keys
    compare(out, lse, ro, rl)
    # the same result as a selection of every other slot through the sparse oracle
    ind = np.full((2, 1, 320), -1, dtype=np.int64)
    for b, L in enumerate([300, 200]):
        j = np.arange(L)
        ind[b, 0, :L] = case.block_table.numpy()[b, j // 64] * 64 + j % 64
    ind[0, 0, 128:192] = -1
    rs, rls, _ = orc.sparse_decode(case.q.double().numpy(), case.kv8.numpy(), ind, None, case.scale)
    compare(out, lse, rs, rls)


@pytest.mark.parametrize("q_scale", [1.0, 8.0])
def test_dense_fp8_decode_helper(q_scale):
    case = wl.dense_fp8_case(2, 2, 64, 0, seqlens=[400, 90], causal=True, q_scale=q_scale, seed=196)
    out, lse = mla.decode(case.q.cuda(), case.kv8.cuda(), case.block_table.cuda(), case.cache_seqlens.cuda(),
                          causal=True, softmax_scale=case.scale)
    torch.cuda.synchronize()
    ro, rl = oracle(case)
    compare(out, lse, ro, rl)


def test_dense_fp8_every_code_value():
    """Every non-NaN E4M3 byte (subnormals, +-0, +-448) in the keys of one
    request: each enters the score as its exact value."""
    case = wl.dense_fp8_case(1, 1, 64, 0, seqlens=[640], seed=197)
    kv8 = case.kv8.clone()
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    bt = case.block_table.numpy()
    for p in range(10):                               # the request's 10 pages
        page = kv8[bt[0, p]].numpy()
        page[:, :512] = np.resize(np.roll(codes, 37 * p), (64, 512))
        kv8[bt[0, p]] = torch.from_numpy(page)
    case = dataclasses.replace(case, kv8=kv8)
    out, lse, st = run(case)
    assert st == 0
    ro, rl = oracle(case)
    compare(out, lse, ro, rl)


def test_dense_fp8_equals_the_token_selection():
    """s_q = 1: the dense FP8 call and a native sparse call whose selection
    lists the request's keys in order run the same arithmetic on the same
    records under the same plan: equal bit for bit."""
    case = wl.dense_fp8_case(3, 1, 128, 0, seqlens=[1000, 64, 300], seed=198)
    out, lse, st = run(case)
    assert st == 0
    B, topk = 3, 1024
    ind = torch.full((B, 1, topk), -1, dtype=torch.int32)
    for b, L in enumerate([1000, 64, 300]):
        j = torch.arange(L)
        ind[b, 0, :L] = case.block_table[b, j // 64] * 64 + j % 64
    sl = case.cache_seqlens.cuda()
    pl = mla.plan(sl, B, 128, num_parts=mla.mla_num_parts_dense(1, 128, 1))
    out_s = torch.empty_like(out)
    lse_s = torch.empty_like(lse)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_sparse_fp8_decode_fwd(case.q.cuda(), case.kv8.cuda(), ind.cuda(), sl.reshape(B, 1), pl.sched,
                                  pl.split_offset, pl.num_parts, pl.workspace, out_s, lse_s, status, case.scale)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    out_d, lse_d, _ = run(case, num_parts=pl.num_parts)
    assert torch.equal(out_d, out_s) and torch.equal(lse_d, lse_s)
