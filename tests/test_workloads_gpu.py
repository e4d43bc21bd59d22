"""The named workloads at their full sizes, in the launch configuration
bench.py times (partition count from mla_num_parts, default plan), against the
oracle on every request (the vectorised fp64 oracle takes well under a second
per workload)."""

import pytest
import torch

import mla_paged_kv_gb300 as mla
from mla_paged_kv_gb300 import workloads as wl
from tests.parity import compare, dense_oracle, sparse_oracle, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["dense_b1_hq16_sk256_fp32out", "dense_b64_hq128_sk2048to4096",
                                  "dense_b1_hq64_sk65536", "dense_b16_sq2causal_hq128_sk4096to8192",
                                  "dense_b64_hq128_sk2048to4096_fp16", "dense_b32_hkv2_hq128_sk2048to4096"])
def test_dense_workload_full_size(name):
    case = wl.make(name)
    c = to_dev(case)
    out, lse = mla.decode(c.q, c.kv, c.block_table, c.cache_seqlens, causal=case.causal, softmax_scale=case.scale,
                          out_fp32=case.out_fp32)
    torch.cuda.synchronize()
    ro, rl = dense_oracle(case)
    compare(out, lse, ro, rl)


@pytest.mark.parametrize("name", ["sparse_fp8_b16_hq128_topk2048", "sparse_fp8_b4_sq4_hq64_topk2048",
                                  "sparse_fp8_b2_sq8_hq128_topk2048"])
def test_sparse_workload_full_size(name):
    case = wl.make(name)
    c = to_dev(case)
    out, lse = mla.sparse_decode(c.q, c.kv8, c.indices, c.topk_length, softmax_scale=case.scale)
    torch.cuda.synchronize()
    ro, rl = sparse_oracle(case)
    compare(out, lse, ro, rl)


def test_dense_fp8_workload_full_size():
    """64 requests x 128 heads over a 2048-4096-token FP8 record cache
    (mla_decode_fwd, dtype FP8_RECORD), in the launch configuration the bench
    times; the oracle checks 6 of the requests."""
    from oracle import mla_oracle as orc
    case = wl.make("dense_fp8_b64_hq128_sk2048to4096")
    out, lse = mla.decode(case.q.cuda(), case.kv8.cuda(), case.block_table.cuda(), case.cache_seqlens.cuda(),
                          softmax_scale=case.scale)
    torch.cuda.synchronize()
    bs = [0, 1, 17, 31, 50, 63]
    ro, rl = orc.dense_fp8_decode(case.q.double().numpy(), case.kv8.numpy(), case.block_table.numpy(),
                                  case.cache_seqlens.numpy(), False, case.scale, batches=bs)
    compare(out[bs], lse[bs], ro[bs], rl[bs])
