"""Sparse FP8 MLA decode and the record unpack on the GPU, against the oracle."""

import numpy as np
import pytest
import torch

import mla_paged_kv_gb300 as mla
from mla_paged_kv_gb300 import workloads as wl
from oracle import mla_oracle as orc
from tests.parity import compare, to_dev

pytestmark = pytest.mark.gpu


def run_sparse(case, indices=None, topk_length="case", num_parts=None):
    c = to_dev(case)
    ind = c.indices if indices is None else indices.to("cuda")
    tl = c.topk_length if isinstance(topk_length, str) else (None if topk_length is None else topk_length.cuda())
    B, s_q, h_q = case.batch, case.s_q, case.h_q
    lens = None if tl is None else tl.reshape(-1).contiguous()
    pl = mla.plan(lens, B * s_q, h_q, sparse=True, default_length=ind.shape[2], num_parts=num_parts,
                  device=torch.device("cuda"))
    out = torch.full((B, s_q, h_q, 512), float("nan"), device="cuda", dtype=torch.bfloat16)
    lse = torch.full((B, s_q, h_q), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_sparse_fp8_decode_fwd(c.q, c.kv8, ind, tl, pl.sched, pl.split_offset, pl.num_parts, pl.workspace,
                                  out, lse, status, case.scale)
    torch.cuda.synchronize()
    return out, lse, int(status.item())


def oracle(case, indices=None, topk_length="case"):
    ind = case.indices if indices is None else indices
    tl = case.topk_length if isinstance(topk_length, str) else topk_length
    o, l, bad = orc.sparse_decode(case.q.double().numpy(), case.kv8.numpy(), ind.numpy(),
                                  None if tl is None else tl.numpy(), case.scale)
    return o, l, bad


@pytest.mark.parametrize("h_q", [16, 64, 128])
@pytest.mark.parametrize("topk", [64, 200])
def test_sparse_small(h_q, topk):
    case = wl.sparse_case(2, 1, h_q, topk=topk, pages_per_req=8, topk_lo=topk // 3, topk_hi=topk, seed=h_q + topk)
    out, lse, st = run_sparse(case)
    assert st == 0
    ro, rl, _ = oracle(case)
    compare(out, lse, ro, rl)


@pytest.mark.parametrize("tl", [0, 1, 63, 64, 65, 128])
def test_sparse_topk_length_edges(tl):
    case = wl.sparse_case(2, 1, 64, topk=128, pages_per_req=4, topk_lengths=[[tl], [max(tl - 1, 0)]], seed=tl)
    out, lse, st = run_sparse(case)
    assert st == 0
    ro, rl, _ = oracle(case)
    compare(out, lse, ro, rl)


def test_sparse_minus_one_inside_prefix_and_duplicates():
    case = wl.sparse_case(2, 2, 128, topk=192, pages_per_req=8, topk_lo=150, topk_hi=192, seed=77)
    ind = case.indices.clone()
    ind[0, 0, 5] = -1
    ind[0, 1, 0:40:3] = -1
    ind[1, 0, 10] = ind[1, 0, 11]          # duplicate counts twice
    ind[1, 1, 100] = ind[1, 1, 0]
    out, lse, st = run_sparse(case, indices=ind)
    assert st == 0
    ro, rl, _ = oracle(case, indices=ind)
    compare(out, lse, ro, rl)


def test_sparse_null_topk_length():
    case = wl.sparse_case(2, 1, 128, topk=128, pages_per_req=4, topk_lengths=[[128], [128]], seed=9)
    ind = case.indices.clone()
    ind[1, 0, 64:] = -1
    out, lse, st = run_sparse(case, indices=ind, topk_length=None)
    assert st == 0
    ro, rl, _ = oracle(case, indices=ind, topk_length=None)
    compare(out, lse, ro, rl)


def test_sparse_bad_index_is_reported_and_masked():
    case = wl.sparse_case(1, 1, 32, topk=64, pages_per_req=4, topk_lengths=[[64]], seed=12)
    ind = case.indices.clone()
    ind[0, 0, 7] = case.kv8.shape[0] * 64 + 5
    out, lse, st = run_sparse(case, indices=ind)
    assert st == 5                          # MLA_ERR_BAD_INDEX
    ro, rl, bad = oracle(case, indices=ind)
    assert bad == 1
    compare(out, lse, ro, rl)


@pytest.mark.parametrize("num_parts", [1, 3, 50])
def test_sparse_split_counts(num_parts):
    case = wl.sparse_case(3, 1, 128, topk=512, pages_per_req=16, topk_lo=200, topk_hi=512, seed=num_parts)
    out, lse, st = run_sparse(case, num_parts=num_parts)
    assert st == 0
    ro, rl, _ = oracle(case)
    compare(out, lse, ro, rl)


def test_sparse_peaky_queries():
    case = wl.sparse_case(2, 1, 128, topk=256, pages_per_req=8, topk_lo=100, topk_hi=256, q_scale=8.0, seed=3)
    out, lse, st = run_sparse(case)
    assert st == 0
    ro, rl, _ = oracle(case)
    compare(out, lse, ro, rl)


def test_unpack_is_bit_exact():
    case = wl.sparse_case(2, 2, 8, topk=256, pages_per_req=8, topk_lo=100, topk_hi=256, seed=5)
    idx = case.indices.reshape(-1).clone()
    idx[3] = case.kv8.shape[0] * 64           # out of the pool -> zero row + status
    k = torch.full((idx.numel(), 576), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_sparse_fp8_unpack(case.kv8.cuda(), idx.cuda(), k, status)
    torch.cuda.synchronize()
    ref, bad = orc.unpack_records(case.kv8.numpy(), idx.numpy())
    assert bad == 1 and int(status.item()) == 5
    got = k.cpu().numpy()
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_unpack_every_e4m3_code():
    # two pages of records whose 512 code bytes run through all 256 codes
    # (except the two NaN codes), with scales that are powers of two and
    # arbitrary fp32 values, so the product is checked bit for bit
    n = 128
    kv8 = torch.zeros(2, 64, 656, dtype=torch.uint8)
    flat = kv8.view(n, 656)
    codes = torch.arange(512, dtype=torch.int64) % 256
    codes[codes == 0x7F] = 0x7E
    codes[codes == 0xFF] = 0xFE
    for r in range(n):
        flat[r, :512] = torch.roll(codes, shifts=r).to(torch.uint8)
        sc = torch.tensor([1.0, 0.5 ** (r % 9), 3.0517578125e-05 * (r + 1), 1.7 + r], dtype=torch.float32)
        flat[r, 512:528] = sc.view(torch.uint8)
        flat[r, 528:656] = torch.randn(64, generator=torch.Generator().manual_seed(r)).to(torch.bfloat16).view(torch.uint8)
    idx = torch.arange(n, dtype=torch.int32)
    k = torch.full((n, 576), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_sparse_fp8_unpack(kv8.cuda(), idx.cuda(), k, status)
    torch.cuda.synchronize()
    ref, bad = orc.unpack_records(kv8.numpy(), idx.numpy())
    assert bad == 0 and int(status.item()) == 0
    assert np.array_equal(k.cpu().numpy().view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("b,s_q,h_q", [(4, 4, 64), (2, 8, 128), (1, 16, 64)])
def test_sparse_request_local_plan(b, s_q, h_q):
    """h_q=64 and s_q>1 query shapes of the sparse path under the request-local plan,
    and the same inputs under the native plan."""
    case = wl.sparse_case(b, s_q, h_q, topk=512, pages_per_req=16, topk_lo=64, topk_hi=512, seed=b * 100 + s_q)
    ro, rl, _ = oracle(case)
    c = to_dev(case)
    for local in (True, False):
        pl = mla.plan(c.topk_length.reshape(-1).contiguous(), b * s_q, h_q, sparse=True, default_length=512,
                      device=torch.device("cuda"), request_local=local)
        out, lse = mla.sparse_decode(c.q, c.kv8, c.indices, c.topk_length, softmax_scale=case.scale, pl=pl)
        torch.cuda.synchronize()
        compare(out, lse, ro, rl)
