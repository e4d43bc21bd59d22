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
    kv = c.kv8 if hasattr(c, "kv8") else c.kv          # FP8 records, or the 16-bit cache (h_kv >= 1)
    h_kv = 1 if kv.dim() == 3 else kv.shape[2]
    if num_parts is None:
        num_parts = mla.mla_num_parts_dense(s_q, h_q, h_kv)
    pl = mla.plan(c.cache_seqlens, B, s_q * h_q, num_parts=num_parts)
    out = torch.full((B, s_q, h_q, 512), float("nan"), device="cuda", dtype=case.q.dtype)
    lse = torch.full((B, s_q, h_q), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    if static:
        mla.mla_decode_fwd_static_ws(c.q, kv, c.block_table, c.cache_seqlens, pl.sched, pl.split_offset,
                                     pl.num_parts, out, lse, status, case.causal, case.scale)
    else:
        mla.mla_decode_fwd(c.q, kv, c.block_table, c.cache_seqlens, pl.sched, pl.split_offset, pl.num_parts,
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


# The other cache types go through the same array: fp16, two latent KV heads,
# and FP8 records (the sparse kernel under the dense plan, same partials).
KINDS = {
    "fp16": lambda: wl.dense_case(3, 1, 128, 0, seqlens=[2500, 90, 1300], dtype=torch.float16, seed=73),
    "hkv2": lambda: wl.dense_case(3, 2, 128, 0, seqlens=[700, 2200, 64], causal=True, h_kv=2, seed=74),
    "fp8_records": lambda: wl.dense_fp8_case(3, 1, 128, 0, seqlens=[1800, 5, 900], seed=75),
}


@pytest.mark.gpu
@pytest.mark.parametrize("kind", sorted(KINDS))
def test_static_ws_other_cache_types_on_consecutive_calls(kind):
    case = KINDS[kind]()
    ro, rl = _run(case, None, static=False)
    for _ in range(2):
        out, lse = _run(case, None, static=True)
        compare(out, lse, ro.double().cpu().numpy(), rl.double().cpu().numpy())


@pytest.mark.gpu
def test_static_ws_fp8_records_just_under_the_limit():
    """The largest FP8-record batch whose workspace (partials, then LSEs)
    still fits the array: the last LSE ends inside it."""
    parts = mla.mla_num_parts_dense(1, 128, 1)
    B = 1
    while mla.mla_workspace_bytes(B + 1, 128, parts) <= STATIC_WORKSPACE_BYTES:
        B += 1
    assert STATIC_WORKSPACE_BYTES - mla.mla_workspace_bytes(B, 128, parts) < 128 * 2052 + 512
    case = wl.dense_fp8_case(B, 1, 128, 64, 320, seed=76)
    ro, rl = _run(case, parts, static=False)
    for _ in range(2):
        out, lse = _run(case, parts, static=True)
        compare(out, lse, ro.double().cpu().numpy(), rl.double().cpu().numpy())
