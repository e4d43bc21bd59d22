"""Packed selected-KV path on the GPU (FlashMLA PR #200, sections "SM90
packing kernel" and "Packed attention specialization"): the pack against the
oracle's byte-for-byte gather, the packed attention (the sparse kernel
reading the packed records in place of the gathered ones) against the
oracle, and the packed result against the native sparse call under the same
plan: the page's packed attention reuses the native dequantisation pipeline,
so the two agree bit for bit."""

import numpy as np
import pytest
import torch

import mla_paged_kv_gb300 as mla
from mla_paged_kv_gb300 import workloads as wl
from oracle import mla_oracle as orc
from tests.parity import compare

pytestmark = pytest.mark.gpu


def gpu_pack(case, ind):
    B, s_q, topk = ind.shape
    packed = torch.full((mla.mla_packed_kv_workspace_bytes(B * s_q, topk),), 0xAB, dtype=torch.uint8,
                        device="cuda")                     # every byte must be written
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_pack_selected_kv(case.kv8.cuda(), ind.cuda(), case.topk_length.cuda(), packed, status)
    torch.cuda.synchronize()
    return packed.cpu().numpy(), int(status.item())


def run_packed(case, packed_np, topk, num_parts=None):
    B, s_q, h_q = case.q.shape[:3]
    tl = case.topk_length.cuda()
    pl = mla.plan(tl.reshape(-1).contiguous(), B * s_q, h_q, sparse=True, default_length=topk,
                  num_parts=num_parts, device=torch.device("cuda"))
    out = torch.full((B, s_q, h_q, 512), float("nan"), device="cuda", dtype=torch.bfloat16)
    lse = torch.full((B, s_q, h_q), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_sparse_fp8_packed_decode_fwd(case.q.cuda(), torch.from_numpy(packed_np).cuda(), topk, tl, pl.sched,
                                         pl.split_offset, pl.num_parts, pl.workspace, out, lse, status, case.scale)
    torch.cuda.synchronize()
    return out, lse, int(status.item()), pl


def case_with_holes(B, s_q, h_q, topk, pages, lengths, seed):
    case = wl.sparse_case(B, s_q, h_q, topk=topk, pages_per_req=pages, topk_lengths=lengths, seed=seed)
    ind = case.indices.clone()
    ind[0, 0, 2:topk:11] = -1                  # masked inside the prefix
    if B > 1:
        ind[1, 0, 1] = ind[1, 0, 0]            # a duplicate counts twice
    return case, ind


@pytest.mark.parametrize("topk,lengths", [(64, [[64], [17]]), (130, [[130], [65]]), (200, [[0], [199]]),
                                          (256, [[256], [128]])])
def test_pack_is_byte_exact(topk, lengths):
    case, ind = case_with_holes(2, 1, 16, topk, 8, lengths, seed=topk)
    got, st = gpu_pack(case, ind)
    ref, bad = orc.pack_selected(case.kv8.numpy(), ind.numpy(), case.topk_length.numpy())
    assert bad == 0 and st == 0
    assert got.shape == ref.shape and np.array_equal(got, ref)


def test_pack_reports_bad_index_and_masks_it():
    case, ind = case_with_holes(1, 2, 16, 128, 4, [[128, 100]], seed=31)
    ind[0, 1, 50] = case.kv8.shape[0] * 64
    ind[0, 1, 120] = -5                        # past unit 1's prefix: ignored
    got, st = gpu_pack(case, ind)
    ref, bad = orc.pack_selected(case.kv8.numpy(), ind.numpy(), case.topk_length.numpy())
    assert bad == 1 and st == 5                # MLA_ERR_BAD_INDEX
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("h_q,topk,s_q", [(16, 64, 1), (64, 200, 2), (128, 130, 1), (128, 512, 2)])
def test_packed_decode_matches_oracle(h_q, topk, s_q):
    lengths = [[topk] * s_q, [max(topk // 3, 1)] * s_q]
    case, ind = case_with_holes(2, s_q, h_q, topk, 16, lengths, seed=h_q + topk)
    packed, _ = orc.pack_selected(case.kv8.numpy(), ind.numpy(), case.topk_length.numpy())
    out, lse, st, _ = run_packed(case, packed, topk)
    assert st == 0
    ro, rl = orc.packed_decode(case.q.double().numpy(), packed, topk, case.topk_length.numpy(), case.scale)
    compare(out, lse, ro, rl)


def run_native(case, ind, pl):
    B, s_q, h_q = case.q.shape[:3]
    out = torch.full((B, s_q, h_q, 512), float("nan"), device="cuda", dtype=torch.bfloat16)
    lse = torch.full((B, s_q, h_q), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_sparse_fp8_decode_fwd(case.q.cuda(), case.kv8.cuda(), ind.cuda(), case.topk_length.cuda(), pl.sched,
                                  pl.split_offset, pl.num_parts, pl.workspace, out, lse, status, case.scale)
    torch.cuda.synchronize()
    return out, lse, int(status.item())


@pytest.mark.parametrize("num_parts", [1, 7, None])
def test_packed_equals_native_under_the_same_plan(num_parts):
    """Same records, same masks, same plan, same arithmetic: the packed and
    the native results are equal bit for bit."""
    case, ind = case_with_holes(3, 1, 128, 384, 16, [[384], [200], [1]], seed=41)
    got, st = gpu_pack(case, ind)
    assert st == 0
    out_p, lse_p, st, pl = run_packed(case, got, 384, num_parts=num_parts)
    assert st == 0
    out_n, lse_n, st = run_native(case, ind, pl)
    assert st == 0
    assert torch.equal(out_p, out_n) and torch.equal(lse_p, lse_n)


def test_packed_full_size_workload():
    """16 query tokens x 128 heads, top-k 2048 over a 128K-token pool: the pack
    byte for byte, the packed attention against the oracle and bit for bit
    against the native call (both plan from the same lengths)."""
    case = wl.make("sparse_fp8_b16_hq128_topk2048")
    packed = mla.pack_selected_kv(case.kv8.cuda(), case.indices.cuda(), case.topk_length.cuda())
    out, lse = mla.packed_sparse_decode(case.q.cuda(), packed, 2048, case.topk_length.cuda(),
                                        softmax_scale=case.scale)
    torch.cuda.synchronize()
    ref, bad = orc.pack_selected(case.kv8.numpy(), case.indices.numpy(), case.topk_length.numpy())
    assert bad == 0 and np.array_equal(packed.cpu().numpy(), ref)
    ro, rl = orc.packed_decode(case.q.double().numpy(), ref, 2048, case.topk_length.numpy(), case.scale)
    compare(out, lse, ro, rl)
    out_n, lse_n = mla.sparse_decode(case.q.cuda(), case.kv8.cuda(), case.indices.cuda(), case.topk_length.cuda(),
                                     softmax_scale=case.scale)
    torch.cuda.synchronize()
    assert torch.equal(out, out_n) and torch.equal(lse, lse_n)


@pytest.mark.parametrize("where", ["middle", "last"])
def test_packed_topk_length_above_topk(where):
    """topk_length may exceed topk: the plan counts tiles from the lengths as
    given, only the first topk slots exist.  The walked tiles past them carry
    no key (no read past the unit's records or masks), and every split the
    plan counts is written, so the result equals the oracle's (which takes
    min(topk_length, topk))."""
    topk = 192
    lengths = [[topk], [topk], [topk]]
    case, ind = case_with_holes(3, 1, 128, topk, 16, lengths, seed=77)
    tl = case.topk_length.clone()
    tl[1 if where == "middle" else 2, 0] = topk + 300  # five phantom tiles past the unit's three
    case.topk_length = tl
    packed, _ = orc.pack_selected(case.kv8.numpy(), ind.numpy(), tl.numpy())
    for num_parts in (5, 23):                           # partitions beginning inside the phantom tiles
        out, lse, st, pl = run_packed(case, packed, topk, num_parts=num_parts)
        assert st == 0
        ro, rl = orc.packed_decode(case.q.double().numpy(), packed, topk, tl.numpy(), case.scale)
        compare(out, lse, ro, rl)


def test_packed_and_native_with_peaky_queries():
    """q x 8 exercises the running-max rescale: both paths keep the scores
    exact in codes and scales, so the plain bars hold, and they agree bit for
    bit."""
    topk = 256
    case, ind = case_with_holes(2, 1, 128, topk, 16, [[topk], [150]], seed=88)
    case.q = case.q * 8
    packed, _ = orc.pack_selected(case.kv8.numpy(), ind.numpy(), case.topk_length.numpy())
    out, lse, st, pl = run_packed(case, packed, topk)
    assert st == 0
    ro, rl = orc.packed_decode(case.q.double().numpy(), packed, topk, case.topk_length.numpy(), case.scale)
    compare(out, lse, ro, rl)
    out_n, lse_n, st = run_native(case, ind, pl)
    assert st == 0
    rn, rln, _ = orc.sparse_decode(case.q.double().numpy(), case.kv8.numpy(), ind.numpy(),
                                   case.topk_length.numpy(), case.scale)
    compare(out_n, lse_n, rn, rln)
    assert torch.equal(out, out_n) and torch.equal(lse, lse_n)
