"""Dense MLA decode on the GPU through the C ABI, element by element against the oracle."""

import numpy as np
import pytest
import torch

import mla_paged_kv_gb300 as mla
from mla_paged_kv_gb300 import workloads as wl
from oracle import mla_sched
from tests.parity import compare, dense_oracle, to_dev

pytestmark = pytest.mark.gpu


def run_dense(case, num_parts=None, split_path=False, out_dtype=None):
    c = to_dev(case)
    B, s_q, h_q = case.batch, case.s_q, case.h_q
    if num_parts is None:
        num_parts = mla.mla_num_parts_dense(s_q, h_q, case.h_kv)
    pl = mla.plan(c.cache_seqlens, B, s_q * h_q, num_parts=num_parts)
    if out_dtype is None:
        out_dtype = torch.float32 if case.out_fp32 else case.q.dtype
    out = torch.full((B, s_q, h_q, 512), float("nan"), device="cuda", dtype=out_dtype)
    lse = torch.full((B, s_q, h_q), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    if split_path:
        mla.mla_decode_splits(c.q, c.kv, c.block_table, c.cache_seqlens, pl.sched, pl.split_offset, pl.num_parts,
                              pl.workspace, out, lse, status, case.causal, case.scale)
        mla.mla_combine(pl.workspace, pl.split_offset, B, s_q * h_q, pl.num_parts, out, lse, status)
    else:
        mla.mla_decode_fwd(c.q, c.kv, c.block_table, c.cache_seqlens, pl.sched, pl.split_offset, pl.num_parts,
                           pl.workspace, out, lse, status, case.causal, case.scale)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, mla.mla_status_string(int(status.item()))
    return out, lse, pl


@pytest.mark.parametrize("lens", [[1], [63], [64], [65], [127, 200], [1000, 3, 64]])
@pytest.mark.parametrize("h_q", [16, 128])
def test_dense_small_lengths(lens, h_q):
    case = wl.dense_case(len(lens), 1, h_q, 0, seqlens=lens, seed=sum(lens) + h_q)
    out, lse, _ = run_dense(case)
    ro, rl = dense_oracle(case)
    compare(out, lse, ro, rl)


@pytest.mark.parametrize("num_parts", [1, 2, 5, 40])
def test_dense_split_counts(num_parts):
    case = wl.dense_case(3, 1, 64, 0, seqlens=[900, 130, 2000], seed=num_parts)
    out, lse, pl = run_dense(case, num_parts=num_parts)
    ro, rl = dense_oracle(case)
    compare(out, lse, ro, rl)
    # scheduler metadata equals the plan, integer for integer
    sched, off = mla_sched.plan(case.cache_seqlens.tolist(), num_parts, 4)
    assert pl.sched.cpu().reshape(-1, 8).tolist() == [list(e) for e in sched]
    assert pl.split_offset.cpu().tolist() == off


def test_dense_splits_then_combine_entry_points():
    case = wl.dense_case(2, 1, 32, 0, seqlens=[700, 1500], seed=3)
    out, lse, _ = run_dense(case, num_parts=7, split_path=True)
    ro, rl = dense_oracle(case)
    compare(out, lse, ro, rl)


@pytest.mark.parametrize("h_q,lens", [(16, [65536] + [64] * 9),        # 160 rows: quarter-row combine
                                        (128, [32768] + [64] * 63)])    # 8192 rows: whole-row combine
def test_dense_combine_unit_with_many_splits(h_q, lens):
    """One long request among short ones: its more than 32 splits go through the
    combine's loop past the first 32 LSEs (and past the first batch of rows)."""
    case = wl.dense_case(len(lens), 1, h_q, 0, seqlens=lens, seed=31 + h_q)
    out, lse, pl = run_dense(case, num_parts=76)
    so = pl.split_offset.cpu().tolist()
    assert so[1] - so[0] > 32 and all(so[i + 1] - so[i] >= 1 for i in range(len(lens)))
    ro, rl = dense_oracle(case)
    compare(out, lse, ro, rl)


@pytest.mark.parametrize("lens", [[1, 2], [64, 65], [300, 129]])
def test_dense_causal_two_tokens(lens):
    case = wl.dense_case(len(lens), 2, 128, 0, seqlens=lens, causal=True, seed=11 + sum(lens))
    out, lse, _ = run_dense(case)
    ro, rl = dense_oracle(case)
    compare(out, lse, ro, rl)


def test_dense_peaky_queries():
    case = wl.dense_case(2, 1, 128, 0, seqlens=[1500, 333], q_scale=8.0, seed=21)
    out, lse, _ = run_dense(case)
    ro, rl = dense_oracle(case)
    compare(out, lse, ro, rl)


def test_dense_tiny_fp32_out():
    case = wl.make("dense_b1_hq16_sk256_fp32out")
    out, lse, _ = run_dense(case)
    assert out.dtype == torch.float32
    ro, rl = dense_oracle(case)
    compare(out, lse, ro, rl)


def test_dense_empty_request():
    case = wl.dense_case(3, 1, 16, 0, seqlens=[0, 70, 0], seed=5)
    out, lse, _ = run_dense(case)
    ro, rl = dense_oracle(case)
    compare(out, lse, ro, rl)


def test_dense_rows_spanning_two_blocks():
    case = wl.dense_case(2, 2, 96, 0, seqlens=[260, 90], causal=True, seed=31)   # 192 rows per request
    out, lse, _ = run_dense(case)
    ro, rl = dense_oracle(case)
    compare(out, lse, ro, rl)


def test_dense_is_deterministic():
    case = wl.dense_case(2, 1, 128, 0, seqlens=[1200, 800], seed=41)
    o1, l1, _ = run_dense(case, num_parts=9)
    o2, l2, _ = run_dense(case, num_parts=9)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_dense_block_table_permutation():
    case = wl.dense_case(2, 1, 64, 0, seqlens=[500, 260], seed=51)
    o1, l1, _ = run_dense(case, num_parts=4)
    P = case.kv.shape[0]
    perm = torch.randperm(P, generator=torch.Generator().manual_seed(1))
    kv2 = torch.empty_like(case.kv)
    kv2[perm] = case.kv
    bt = case.block_table
    bt2 = torch.where(bt >= 0, perm[bt.clamp(min=0).long()].to(torch.int32), bt)
    case2 = wl.DenseCase(q=case.q, kv=kv2, block_table=bt2, cache_seqlens=case.cache_seqlens, causal=False,
                         scale=case.scale, out_fp32=False)
    o2, l2, _ = run_dense(case2, num_parts=4)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_dense_request_local_plan():
    case = wl.dense_case(5, 2, 64, 0, seqlens=[900, 130, 2000, 64, 3000], causal=True, seed=61)
    c = to_dev(case)
    pl = mla.plan(c.cache_seqlens, 5, 2 * 64, request_local=True)
    out, lse = mla.decode(c.q, c.kv, c.block_table, c.cache_seqlens, causal=True, softmax_scale=case.scale, pl=pl)
    torch.cuda.synchronize()
    ro, rl = dense_oracle(case)
    compare(out, lse, ro, rl)


# ---------------------------------------------------------------- several latent KV heads; fp16

@pytest.mark.parametrize("h_kv,h_q,s_q,causal", [(2, 128, 1, False), (4, 128, 2, True), (2, 64, 3, True),
                                                 (4, 16, 1, False), (3, 96, 2, False), (2, 256, 1, False)])
def test_dense_kv_heads(h_kv, h_q, s_q, causal):
    case = wl.dense_case(3, s_q, h_q, 0, seqlens=[65, 700, 2000], causal=causal, h_kv=h_kv, seed=h_kv * h_q + s_q)
    out, lse, _ = run_dense(case)
    ro, rl = dense_oracle(case)
    compare(out, lse, ro, rl)


@pytest.mark.parametrize("num_parts", [1, 40])
def test_dense_kv_heads_split_counts(num_parts):
    case = wl.dense_case(3, 2, 64, 0, seqlens=[900, 130, 2000], causal=True, h_kv=2, seed=num_parts + 500)
    out, lse, _ = run_dense(case, num_parts=num_parts, split_path=True)
    ro, rl = dense_oracle(case)
    compare(out, lse, ro, rl)


@pytest.mark.parametrize("h_q,s_q,causal,out_dtype", [(128, 1, False, torch.float16), (64, 2, True, torch.float16),
                                                      (128, 1, False, torch.float32), (16, 1, False, torch.bfloat16)])
def test_dense_fp16(h_q, s_q, causal, out_dtype):
    case = wl.dense_case(2, s_q, h_q, 0, seqlens=[300, 1500], causal=causal, dtype=torch.float16, seed=h_q + s_q)
    out, lse, _ = run_dense(case, out_dtype=out_dtype)
    assert out.dtype == out_dtype
    ro, rl = dense_oracle(case)
    compare(out, lse, ro, rl)


def test_dense_fp16_kv_heads_peaky():
    case = wl.dense_case(2, 2, 64, 0, seqlens=[1000, 2100], causal=True, h_kv=2, dtype=torch.float16, q_scale=8.0,
                         seed=601)
    out, lse, _ = run_dense(case, num_parts=7)
    ro, rl = dense_oracle(case)
    compare(out, lse, ro, rl)


def test_dense_kv_heads_static_workspace():
    case = wl.dense_case(2, 1, 128, 0, seqlens=[500, 1300], h_kv=4, dtype=torch.float16, seed=602)
    c = to_dev(case)
    pl = mla.plan(c.cache_seqlens, 2, 128)
    out = torch.empty(2, 1, 128, 512, dtype=torch.float16, device="cuda")
    lse = torch.empty(2, 1, 128, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_decode_fwd_static_ws(c.q, c.kv, c.block_table, c.cache_seqlens, pl.sched, pl.split_offset, pl.num_parts,
                                 out, lse, status, case.causal, case.scale)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ro, rl = dense_oracle(case)
    compare(out, lse, ro, rl)


def test_num_parts_dense_counts_row_blocks():
    base = mla.mla_num_parts(128, False)
    assert mla.mla_num_parts_dense(1, 128, 1) == base
    assert mla.mla_num_parts_dense(2, 128, 1) == mla.mla_num_parts(256, False)
    assert mla.mla_num_parts_dense(1, 128, 2) == max(base // 2, 1)      # two head groups of 64 heads
    assert mla.mla_num_parts_dense(3, 96, 3) == max(base // 3, 1)       # 3 groups, each one block of 3 tokens x 32 heads
    assert mla.mla_num_parts_dense(5, 64, 2) == max(base // 4, 1)       # 2 groups of 32 heads x 2 blocks (4 + 1 tokens)


# ---------------------------------------------------------------- block-table entries outside the pool

@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("num_parts", [2, 76])      # 76 parts per 2 requests: the instance staging Q in the V ring
@pytest.mark.parametrize("bad_entry", [-7, 10 ** 6])
def test_dense_out_of_pool_page_is_masked_and_reported(dtype, num_parts, bad_entry):
    """A block-table entry outside [0, num_pages) masks the 64 keys of its
    page (the oracle's reading) and sets MLA_ERR_BAD_INDEX; both requests
    still match the oracle, the untouched one bit for bit against a clean run."""
    case = wl.dense_case(2, 2, 128, 0, seqlens=[700, 333], causal=True, dtype=dtype, seed=81)
    bt = case.block_table.clone()
    bt[0, 3] = bad_entry                               # keys 192..255 of request 0
    bad = wl.DenseCase(q=case.q, kv=case.kv, block_table=bt, cache_seqlens=case.cache_seqlens, causal=True,
                       scale=case.scale, out_fp32=False)
    c = to_dev(bad)
    pl = mla.plan(c.cache_seqlens, 2, 256, num_parts=num_parts)
    out = torch.full((2, 2, 128, 512), float("nan"), device="cuda", dtype=dtype)
    lse = torch.full((2, 2, 128), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_decode_fwd(c.q, c.kv, c.block_table, c.cache_seqlens, pl.sched, pl.split_offset, pl.num_parts,
                       pl.workspace, out, lse, status, True, case.scale)
    torch.cuda.synchronize()
    assert int(status.item()) == 5                     # MLA_ERR_BAD_INDEX
    ro, rl = dense_oracle(bad)
    compare(out, lse, ro, rl)
    clean_o, clean_l, _ = run_dense(case, num_parts=num_parts)
    assert torch.equal(out[1], clean_o[1]) and torch.equal(lse[1], clean_l[1])
