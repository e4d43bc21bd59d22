"""Many units per partition: batches of a thousand or more short requests, so
that every CTA pair walks through dozens of units (a Q load, an epilogue and
a row-sum exchange each, with the barrier phases running on across units),
and the combine sees tens of thousands of rows.  Ragged lengths with zeros
and page-boundary lengths; every request is checked against the oracle."""

import numpy as np
import pytest
import torch

import mla_paged_kv_gb300 as mla
from mla_paged_kv_gb300 import workloads as wl
from oracle import mla_oracle as orc
from tests.parity import compare, dense_oracle, sparse_oracle, to_dev

pytestmark = pytest.mark.gpu


def ragged_lengths(n, hi, seed, specials=(0, 1, 63, 64, 65, 127, 128, 129)):
    rng = np.random.default_rng(seed)
    lens = rng.integers(0, hi + 1, n)
    lens[:len(specials)] = specials
    rng.shuffle(lens)
    return lens.tolist()


@pytest.mark.parametrize("batch,s_q,h_q,causal,hi,h_kv,dtype", [
    (1500, 1, 16, False, 200, 1, torch.bfloat16),
    (700, 2, 32, True, 300, 1, torch.bfloat16),
    (700, 1, 64, False, 200, 2, torch.float16),   # two latent KV heads, fp16 cache and output
])
def test_dense_many_short_requests(batch, s_q, h_q, causal, hi, h_kv, dtype):
    lens = ragged_lengths(batch, hi, seed=batch + h_q)  # causal with L < s_q: rows that see no key
    case = wl.dense_case(batch, s_q, h_q, 0, seqlens=lens, causal=causal, seed=batch + s_q, h_kv=h_kv,
                         dtype=dtype)
    c = to_dev(case)
    pl = mla.plan(c.cache_seqlens, batch, s_q * h_q, num_parts=mla.mla_num_parts_dense(s_q, h_q, h_kv))
    # more units than partitions by far: each partition runs through many units
    assert batch >= 8 * pl.num_parts
    out = torch.full((batch, s_q, h_q, 512), float("nan"), dtype=dtype, device="cuda")
    lse = torch.full((batch, s_q, h_q), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_decode_fwd(c.q, c.kv, c.block_table, c.cache_seqlens, pl.sched, pl.split_offset, pl.num_parts,
                       pl.workspace, out, lse, status, causal, case.scale)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ro, rl = dense_oracle(case)
    compare(out, lse, ro, rl)


def test_sparse_many_query_tokens():
    batch, s_q, h_q, topk = 500, 2, 64, 128
    tl = np.array(ragged_lengths(batch * s_q, topk, seed=7, specials=(0, 1, 63, 64, 65, 127, 128)))
    case = wl.sparse_case(batch, s_q, h_q, topk=topk, pages_per_req=4, topk_lengths=tl.reshape(batch, s_q),
                          seed=8)
    c = to_dev(case)
    pl = mla.plan(c.topk_length.reshape(-1).contiguous(), batch * s_q, h_q, sparse=True, default_length=topk)
    assert batch * s_q >= 8 * pl.num_parts
    out = torch.full((batch, s_q, h_q, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((batch, s_q, h_q), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_sparse_fp8_decode_fwd(c.q, c.kv8, c.indices, c.topk_length, pl.sched, pl.split_offset, pl.num_parts,
                                  pl.workspace, out, lse, status, case.scale)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ro, rl = sparse_oracle(case)
    compare(out, lse, ro, rl)


def test_dense_fp8_many_short_requests():
    batch, h_q = 1200, 16
    lens = ragged_lengths(batch, 200, seed=21)
    case = wl.dense_fp8_case(batch, 1, h_q, 0, seqlens=lens, seed=22)
    q, kv8, bt, sl = case.q.cuda(), case.kv8.cuda(), case.block_table.cuda(), case.cache_seqlens.cuda()
    out, lse = mla.decode(q, kv8, bt, sl, softmax_scale=case.scale)
    torch.cuda.synchronize()
    ro, rl = orc.dense_fp8_decode(case.q.double().numpy(), case.kv8.numpy(), case.block_table.numpy(),
                                  case.cache_seqlens.numpy(), False, case.scale)
    compare(out, lse, ro, rl)
