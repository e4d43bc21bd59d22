"""Dense decode over a paged cache of FP8 records, on the GPU through the C ABI,
against the oracle (dense_fp8_decode)."""

import dataclasses

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


# ------------------------------------------- the same cache through the dense kernel (dtype FP8_RECORD)
# Each NoPE value enters the MMAs as code * scale rounded to fp16 (relative
# error <= 2^-11 + 2^-20: one rounding of the product up to 2^-20 from the
# split of the scale), and q and the RoPE dims as fp16 (exact for values in
# fp16's normal range); the oracle keeps every value exact.  For unit-scale
# inputs the result meets the bf16 bar.  In general each score moves by at
# most scale * (2^-11 + 2^-20) * sum_d |q_d k_d| (+ fp16 subnormal slack), and
# the LSE, being 1-Lipschitz in the largest score change, by at most the
# largest such bound over the row's keys: lse_bound() below, which the
# peaky-query test uses.


def lse_bound(case):
    """Per-row bound on |lse - lse*| for fp16-rounded K (see above), plus fp32 slack."""
    recs = case.kv8.numpy().reshape(-1, 656)
    codes = torch.from_numpy(recs[:, :512].copy()).view(torch.float8_e4m3fn).double().numpy()
    sc = recs[:, 512:528].copy().view(np.float32).astype(np.float64)
    rope = torch.from_numpy(recs[:, 528:].copy()).view(torch.bfloat16).double().numpy()
    k = np.abs(np.concatenate([codes * np.repeat(sc, 128, axis=1), rope], axis=1)).reshape(-1, 64, 576)
    q = np.abs(case.q.double().numpy())
    bt, L = case.block_table.numpy(), case.cache_seqlens.numpy()
    out = np.zeros(q.shape[:3])
    for b in range(q.shape[0]):
        if L[b] == 0:
            continue
        j = np.arange(L[b])
        dots = np.einsum("shd,jd->shj", q[b], k[bt[b, j // 64], j % 64])
        out[b] = case.scale * ((2.0 ** -11 + 2.0 ** -20) * dots.max(-1) + 576 * 2.0 ** -25 * q[b].max(-1)) + 1e-5
    return out

def run_records(case, num_parts=None, block_table=None, out_dtype=torch.bfloat16):
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


@pytest.mark.parametrize("h_q,s_q,causal,lens", [(16, 1, False, [1, 63]), (64, 1, False, [64, 65, 500]),
                                                 (128, 1, False, [2000, 130]), (128, 2, True, [2, 700]),
                                                 (64, 3, True, [3, 64, 1200]), (32, 2, False, [0, 300])])
def test_dense_fp8_records_small(h_q, s_q, causal, lens):
    case = wl.dense_fp8_case(len(lens), s_q, h_q, 0, seqlens=lens, causal=causal, seed=h_q + s_q + sum(lens))
    out, lse, st = run_records(case)
    assert st == 0
    ro, rl = oracle(case)
    compare(out, lse, ro, rl)


@pytest.mark.parametrize("num_parts", [1, 7, 40])
def test_dense_fp8_records_split_counts(num_parts):
    case = wl.dense_fp8_case(3, 2, 128, 0, seqlens=[900, 130, 2000], causal=True, seed=num_parts + 190)
    out, lse, st = run_records(case, num_parts=num_parts)
    assert st == 0
    ro, rl = oracle(case)
    compare(out, lse, ro, rl)


def test_dense_fp8_records_fp32_out_peaky_and_deterministic():
    """q x 8: the output still meets the bf16 bar; the LSE meets the bound
    derived from the fp16 rounding of K (the bf16 LSE bar assumes exact K)."""
    case = wl.dense_fp8_case(2, 1, 128, 0, seqlens=[1500, 333], q_scale=8.0, seed=193)
    o1, l1, st = run_records(case, out_dtype=torch.float32)
    assert st == 0 and o1.dtype == torch.float32
    ro, rl = oracle(case)
    import tests.parity as par
    o = o1.double().cpu().numpy()
    assert np.abs(o - ro).max() <= par.MAX_ABS
    assert np.linalg.norm(o - ro) / np.linalg.norm(ro) <= par.REL_FRO
    assert (np.abs(l1.double().cpu().numpy() - rl) <= lse_bound(case)).all()
    o2, l2, _ = run_records(case, out_dtype=torch.float32)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_dense_fp8_records_agree_with_the_exact_score_path():
    case = wl.dense_fp8_case(3, 1, 128, 0, seqlens=[777, 64, 1500], seed=194)
    out_r, lse_r, st = run_records(case)
    assert st == 0
    out_e, lse_e, st, _ = run(case)
    assert st == 0
    compare(out_r, lse_r, out_e.double().cpu().numpy(), lse_e.double().cpu().numpy())


def test_dense_fp8_records_bad_page_is_reported_and_masked():
    case = wl.dense_fp8_case(2, 1, 64, 0, seqlens=[300, 200], seed=195)
    bt = case.block_table.clone()
    bt[0, 2] = case.kv8.shape[0] + 5                 # keys 128..191 of request 0 point outside the pool
    out, lse, st = run_records(case, block_table=bt)
    assert st == 5                                   # MLA_ERR_BAD_INDEX
    ro, rl = orc.dense_fp8_decode(case.q.double().numpy(), case.kv8.numpy(), bt.numpy(),
                                  case.cache_seqlens.numpy(), case.causal, case.scale)   # those keys masked
    compare(out, lse, ro, rl)


@pytest.mark.parametrize("q_scale", [1.0, 8.0])
def test_dense_fp8_decode_helper_default_is_exact(q_scale):
    """mla.decode on an FP8-record cache takes the exact-score path by
    default: the plain bars hold even for peaky queries (q x 8)."""
    case = wl.dense_fp8_case(2, 2, 64, 0, seqlens=[400, 90], causal=True, q_scale=q_scale, seed=196)
    out, lse = mla.decode(case.q.cuda(), case.kv8.cuda(), case.block_table.cuda(), case.cache_seqlens.cuda(),
                          causal=True, softmax_scale=case.scale)
    torch.cuda.synchronize()
    ro, rl = oracle(case)
    compare(out, lse, ro, rl)


def test_dense_fp8_decode_helper_fast_option():
    case = wl.dense_fp8_case(2, 2, 64, 0, seqlens=[400, 90], causal=True, seed=198)
    out, lse = mla.decode(case.q.cuda(), case.kv8.cuda(), case.block_table.cuda(), case.cache_seqlens.cuda(),
                          causal=True, softmax_scale=case.scale, fast_fp8=True)
    torch.cuda.synchronize()
    ro, rl = oracle(case)
    compare(out, lse, ro, rl)


def test_dense_fp8_records_every_code_value():
    """Every non-NaN E4M3 byte (subnormals, +-0, +-448) in the keys of one
    request: the in-kernel decode takes each to code * scale exactly before
    the single fp16 rounding."""
    case = wl.dense_fp8_case(1, 1, 64, 0, seqlens=[640], seed=197)
    kv8 = case.kv8.clone()
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    bt = case.block_table.numpy()
    for p in range(10):                               # the request's 10 pages
        page = kv8[bt[0, p]].numpy()
        page[:, :512] = np.resize(np.roll(codes, 37 * p), (64, 512))
        kv8[bt[0, p]] = torch.from_numpy(page)
    case = dataclasses.replace(case, kv8=kv8)
    out, lse, st = run_records(case)
    assert st == 0
    ro, rl = oracle(case)
    compare(out, lse, ro, rl)
