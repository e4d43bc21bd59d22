"""mla_decode_fwd_static_ws: the decode entry point for callers that cannot
allocate device memory (a plain C host program with no device allocator, or a
serving runtime that reserved nearly all of HBM up front and forbids
allocation on the decode path).  It keeps the split partials in the
library's fixed device array instead of a caller workspace.

Its results must match mla_decode_fwd (caller workspace) on the same inputs,
call after call, although every call reuses the same array.  The file name
puts it last in collection, so it also runs after every other GPU test in
the same process; it passes alone in a fresh process as well.
"""

import ctypes

import pytest
import torch

import mla_paged_kv_gb300 as mla
from mla_paged_kv_gb300 import workloads as wl
from tests.parity import compare, to_dev

MLA_ERR_INVALID_ARG = 1
MLA_ERR_UNSUPPORTED = 2
STATIC_WORKSPACE_BYTES = 64 << 20


def _null_call(lib, batch, s_q, h_q, num_parts):
    n = None
    # ..., batch, s_q, h_q, h_kv = 1, dtype = bf16, causal = 0, scale, sched, split_offset, num_parts, out,
    # out_type = bf16, lse, status, stream
    return lib.mla_decode_fwd_static_ws(n, n, n, 1, 1, n, batch, s_q, h_q, 1, 0, 0, 1.0 / 24.0, n, n, num_parts, n, 0,
                                        n, n, ctypes.c_void_p(0))


def test_static_ws_refuses_oversize_before_any_device_call():
    lib = mla.load_library()
    # 4096 requests x 128 rows with 76 parts need ~1.1 GB of partials: refused on the host
    assert mla.mla_workspace_bytes(4096, 128, 76) > STATIC_WORKSPACE_BYTES
    assert _null_call(lib, 4096, 1, 128, 76) == MLA_ERR_UNSUPPORTED
    assert _null_call(lib, 0, 1, 128, 76) == MLA_ERR_INVALID_ARG
    assert _null_call(lib, 4, 1, 128, 0) == MLA_ERR_INVALID_ARG


def _run(case, num_parts, static):
    c = to_dev(case)
    B, s_q, h_q = case.batch, case.s_q, case.h_q
    pl = mla.plan(c.cache_seqlens, B, s_q * h_q, num_parts=num_parts)
    out = torch.full((B, s_q, h_q, 512), float("nan"), device="cuda", dtype=torch.bfloat16)
    lse = torch.full((B, s_q, h_q), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    if static:
        mla.mla_decode_fwd_static_ws(c.q, c.kv, c.block_table, c.cache_seqlens, pl.sched, pl.split_offset,
                                     pl.num_parts, out, lse, status, case.causal, case.scale)
    else:
        mla.mla_decode_fwd(c.q, c.kv, c.block_table, c.cache_seqlens, pl.sched, pl.split_offset, pl.num_parts,
                           pl.workspace, out, lse, status, case.causal, case.scale)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, mla.mla_status_string(int(status.item()))
    return out, lse


@pytest.mark.gpu
def test_static_ws_matches_caller_workspace_on_consecutive_calls():
    # two different problems, so the second call lays its partials over what
    # the first one left in the shared array; then the first one again
    a = wl.dense_case(4, 1, 128, 0, seqlens=[3000, 1, 700, 4096], seed=71)
    b = wl.dense_case(3, 2, 64, 0, seqlens=[900, 130, 2000], causal=True, seed=72)
    ref = {"a": _run(a, None, static=False), "b": _run(b, 40, static=False)}
    for name, case, parts in (("a", a, None), ("b", b, 40), ("a", a, None)):
        out, lse = _run(case, parts, static=True)
        ro, rl = ref[name]
        compare(out, lse, ro.double().cpu().numpy(), rl.double().cpu().numpy())
