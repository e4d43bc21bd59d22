"""MLA decode over a paged KV cache, GB300 (sm_103a) native.

Thin ctypes binding over libmla_paged_kv.so (see include/mla_paged_kv.h).
Functions named ``mla_*`` mirror the C entry points one to one: they only
marshal torch tensors into pointers, sizes and the current CUDA stream; every
step of the computation runs in the library's CUDA kernels.  The helpers
below them (``plan``, ``decode``, ``sparse_decode``) allocate outputs with
torch and check the device status word.

There is no fallback: if the library is missing or the GPU is not sm_103a,
the calls raise.
"""

from __future__ import annotations

import ctypes
import math
import os

import torch

from .build import LIB_PATH

__all__ = [
    "MlaError", "load_library", "mla_status_string", "mla_num_parts", "mla_workspace_bytes",
    "mla_get_metadata", "mla_decode_fwd", "mla_decode_splits", "mla_combine",
    "mla_sparse_fp8_decode_fwd", "mla_sparse_fp8_unpack", "mla_decode_fwd_static_ws",
    "mla_packed_kv_workspace_bytes", "mla_pack_selected_kv", "mla_sparse_fp8_packed_decode_fwd",
    "mla_get_metadata_request_local", "mla_num_parts_dense", "mla_test_pack_timeout", "mla_test_decode_timeout", "plan",
    "decode",
    "sparse_decode", "pack_selected_kv", "packed_sparse_decode",
    "EXPORTED_SYMBOLS",
]

EXPORTED_SYMBOLS = (
    "mla_status_string", "mla_num_parts", "mla_workspace_bytes", "mla_get_metadata", "mla_decode_fwd",
    "mla_decode_splits", "mla_combine", "mla_sparse_fp8_decode_fwd", "mla_sparse_fp8_unpack",
    "mla_decode_fwd_static_ws", "mla_packed_kv_workspace_bytes", "mla_pack_selected_kv",
    "mla_sparse_fp8_packed_decode_fwd", "mla_get_metadata_request_local", "mla_num_parts_dense",
    "mla_test_pack_timeout", "mla_test_decode_timeout",
)

_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_SZ = ctypes.c_size_t

_SIGS = {
    "mla_status_string": (ctypes.c_char_p, [_I]),
    "mla_num_parts": (_I, [_I, _I]),
    "mla_num_parts_dense": (_I, [_I, _I, _I]),
    "mla_workspace_bytes": (_SZ, [_I, _I, _I]),
    "mla_get_metadata": (_I, [_P, _I, _I, _I, _P, _P, _P]),
    "mla_get_metadata_request_local": (_I, [_P, _I, _I, _I, _P, _P, _P]),
    "mla_decode_fwd": (_I, [_P, _P, _P, _I, _I, _P, _I, _I, _I, _I, _I, _I, _F, _P, _P, _I, _P, _SZ, _P, _I, _P,
                            _P, _P]),
    "mla_decode_splits": (_I, [_P, _P, _P, _I, _I, _P, _I, _I, _I, _I, _I, _I, _F, _P, _P, _I, _P, _SZ, _P, _I,
                               _P, _P, _P]),
    "mla_combine": (_I, [_P, _SZ, _P, _I, _I, _I, _P, _I, _P, _P, _P]),
    "mla_sparse_fp8_decode_fwd": (_I, [_P, _P, _I, _P, _I, _P, _I, _I, _I, _F, _P, _P, _I, _P, _SZ, _P, _P, _P,
                                       _P]),
    "mla_sparse_fp8_unpack": (_I, [_P, _I, _P, _I, _P, _P, _P]),
    "mla_decode_fwd_static_ws": (_I, [_P, _P, _P, _I, _I, _P, _I, _I, _I, _I, _I, _I, _F, _P, _P, _I, _P, _I,
                                      _P, _P, _P]),
    "mla_packed_kv_workspace_bytes": (_SZ, [_I, _I]),
    "mla_pack_selected_kv": (_I, [_P, _I, _P, _I, _P, _I, _P, _SZ, _P, _P]),
    "mla_test_pack_timeout": (_I, [_P, _I, _P, _I, _P, _I, _P, _SZ, _P, _P]),
    "mla_test_decode_timeout": (_I, [_P, _P, _P, _I, _I, _P, _I, _I, _I, _I, _I, _I, _F, _P, _P, _I, _P, _SZ, _P,
                                     _I, _P, _P, _P]),
    "mla_sparse_fp8_packed_decode_fwd": (_I, [_P, _P, _SZ, _I, _P, _I, _I, _I, _F, _P, _P, _I, _P, _SZ, _P, _P, _P,
                                              _P]),
}

_lib = None


class MlaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {mla_status_string(code)} ({code})")


def load_library(path: str = LIB_PATH):
    """Load libmla_paged_kv.so (built by ``build.build()``) and declare its signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with mla_paged_kv_gb300.build.build()")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(rc: int, where: str):
    if rc != 0:
        raise MlaError(rc, where)


def _need(t, dtype, name, dims=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if dims is not None and t.dim() != dims:
        raise ValueError(f"{name} must have {dims} dims, got {tuple(t.shape)}")


# ---------------------------------------------------------------- C entry points


def mla_status_string(code: int) -> str:
    return load_library().mla_status_string(int(code)).decode()


def mla_num_parts(rows_per_unit: int, is_sparse_fp8: bool = False) -> int:
    n = load_library().mla_num_parts(int(rows_per_unit), int(bool(is_sparse_fp8)))
    if n < 0:
        raise MlaError(-n, "mla_num_parts")
    return n


def mla_num_parts_dense(s_q: int, h_q: int, h_kv: int = 1) -> int:
    n = load_library().mla_num_parts_dense(int(s_q), int(h_q), int(h_kv))
    if n < 1:
        raise MlaError(-n, "mla_num_parts_dense")
    return n


def mla_workspace_bytes(n_units: int, rows_per_unit: int, num_parts: int) -> int:
    return int(load_library().mla_workspace_bytes(int(n_units), int(rows_per_unit), int(num_parts)))


def _metadata(fn, lengths, n_units, num_parts, sched, split_offset, default_length, stream):
    if lengths is not None:
        _need(lengths, torch.int32, "lengths")
    _need(sched, torch.int32, "sched")
    _need(split_offset, torch.int32, "split_offset")
    if sched.numel() < num_parts * 8 or split_offset.numel() < n_units + 1:
        raise ValueError("sched / split_offset too small")
    _check(getattr(load_library(), fn)(_ptr(lengths), int(default_length), int(n_units), int(num_parts),
                                       _ptr(sched), _ptr(split_offset), _stream(stream)), fn)


def mla_get_metadata(lengths, n_units, num_parts, sched, split_offset, default_length=-1, stream=None):
    _metadata("mla_get_metadata", lengths, n_units, num_parts, sched, split_offset, default_length, stream)


def mla_get_metadata_request_local(lengths, n_units, num_parts, sched, split_offset, default_length=-1,
                                   stream=None):
    _metadata("mla_get_metadata_request_local", lengths, n_units, num_parts, sched, split_offset, default_length,
              stream)


DTYPE_BF16, DTYPE_FP32, DTYPE_FP16, DTYPE_FP8_RECORD = 0, 1, 2, 3   # mla_dtype_t
_DTYPE_CODE = {torch.bfloat16: DTYPE_BF16, torch.float32: DTYPE_FP32, torch.float16: DTYPE_FP16}


def _dense_inputs(q, kv, block_table, cache_seqlens, out, lse, status):
    """Checks shared by the dense entry points; returns (h_kv, dtype code, out type code).
    kv is the 16-bit latent cache of q's dtype, or (uint8 [pages, 64, 656])
    a cache of FP8 records with a bf16 q."""
    if q.dtype not in (torch.bfloat16, torch.float16):
        raise TypeError("q must be bf16 or fp16")
    _need(q, q.dtype, "q", 4)
    if kv.dtype == torch.uint8:
        if q.dtype != torch.bfloat16 or kv.dim() != 3 or kv.shape[1] != 64 or kv.shape[2] != 656:
            raise TypeError("an FP8 record cache is uint8 [pages, 64, 656] and goes with a bf16 q")
        _need(kv, torch.uint8, "kv")
    elif kv.dtype != q.dtype or kv.dim() not in (3, 4):
        raise TypeError("kv must have q's dtype and be [pages, 64, 576] or [pages, 64, h_kv, 576]")
    else:
        _need(kv, q.dtype, "kv")
    _need(block_table, torch.int32, "block_table", 2)
    _need(cache_seqlens, torch.int32, "cache_seqlens", 1)
    _need(lse, torch.float32, "lse")
    _need(status, torch.int32, "status")
    if out.dtype not in _DTYPE_CODE:
        raise TypeError("out must be bf16, fp16 or fp32")
    B, s_q, h_q, d = q.shape
    fp8 = kv.dtype == torch.uint8
    h_kv = 1 if kv.dim() == 3 else kv.shape[2]
    if d != 576 or kv.shape[1] != 64 or (kv.shape[-1] != 576 and not fp8) or h_q % h_kv:
        raise ValueError("q must be [B, s_q, h_q, 576], kv [pages, 64, (h_kv,) 576] with h_kv dividing h_q")
    if tuple(out.shape) != (B, s_q, h_q, 512) or tuple(lse.shape) != (B, s_q, h_q):
        raise ValueError("out must be [B, s_q, h_q, 512] and lse [B, s_q, h_q]")
    if block_table.shape[0] != B or cache_seqlens.shape[0] != B:
        raise ValueError("block_table / cache_seqlens batch mismatch")
    return h_kv, (DTYPE_FP8_RECORD if fp8 else _DTYPE_CODE[q.dtype]), _DTYPE_CODE[out.dtype]


def _dense_args(q, kv, block_table, cache_seqlens, sched, split_offset, num_parts, workspace, out, lse, status,
                causal, softmax_scale, stream):
    h_kv, dt, ot = _dense_inputs(q, kv, block_table, cache_seqlens, out, lse, status)
    _need(workspace, torch.uint8, "workspace")
    B, s_q, h_q, _ = q.shape
    return (_ptr(q), _ptr(kv), _ptr(block_table), block_table.shape[1], kv.shape[0], _ptr(cache_seqlens), B, s_q,
            h_q, h_kv, dt, int(bool(causal)), float(softmax_scale), _ptr(sched), _ptr(split_offset),
            int(num_parts), _ptr(workspace), workspace.numel(), _ptr(out), ot, _ptr(lse), _ptr(status),
            _stream(stream))


def mla_decode_fwd(q, kv, block_table, cache_seqlens, sched, split_offset, num_parts, workspace, out, lse, status,
                   causal=False, softmax_scale=1.0 / 24.0, stream=None):
    """Dense decode.  q/kv bf16 or fp16 (same type), kv [pages, 64, 576] or
    [pages, 64, h_kv, 576]; or a bf16 q over FP8 records, kv uint8
    [pages, 64, 656].  out bf16, fp16 or fp32."""
    args = _dense_args(q, kv, block_table, cache_seqlens, sched, split_offset, num_parts, workspace, out, lse,
                       status, causal, softmax_scale, stream)
    _check(load_library().mla_decode_fwd(*args), "mla_decode_fwd")


def mla_decode_splits(q, kv, block_table, cache_seqlens, sched, split_offset, num_parts, workspace, out, lse,
                      status, causal=False, softmax_scale=1.0 / 24.0, stream=None):
    args = _dense_args(q, kv, block_table, cache_seqlens, sched, split_offset, num_parts, workspace, out, lse,
                       status, causal, softmax_scale, stream)
    _check(load_library().mla_decode_splits(*args), "mla_decode_splits")


def mla_test_decode_timeout(q, kv, block_table, cache_seqlens, sched, split_offset, num_parts, workspace, out, lse,
                            status, causal=False, softmax_scale=1.0 / 24.0, stream=None):
    """Test hook: the dense kernel instance whose first own K tile never
    loads, so that a bounded wait runs out (*status = MLA_ERR_TIMEOUT)."""
    args = _dense_args(q, kv, block_table, cache_seqlens, sched, split_offset, num_parts, workspace, out, lse,
                       status, causal, softmax_scale, stream)
    _check(load_library().mla_test_decode_timeout(*args), "mla_test_decode_timeout")


def mla_decode_fwd_static_ws(q, kv, block_table, cache_seqlens, sched, split_offset, num_parts, out, lse, status,
                             causal=False, softmax_scale=1.0 / 24.0, stream=None):
    """mla_decode_fwd for callers with no device scratch to give: the library
    keeps the split partials in its own fixed device array (64 MiB per GPU).
    Nothing is allocated; a problem whose partials do not fit raises
    MLA_ERR_UNSUPPORTED."""
    h_kv, dt, ot = _dense_inputs(q, kv, block_table, cache_seqlens, out, lse, status)
    B, s_q, h_q, _ = q.shape
    rc = load_library().mla_decode_fwd_static_ws(
        _ptr(q), _ptr(kv), _ptr(block_table), block_table.shape[1], kv.shape[0], _ptr(cache_seqlens), B, s_q, h_q,
        h_kv, dt, int(bool(causal)), float(softmax_scale), _ptr(sched), _ptr(split_offset), int(num_parts),
        _ptr(out), ot, _ptr(lse), _ptr(status), _stream(stream))
    _check(rc, "mla_decode_fwd_static_ws")


def mla_combine(workspace, split_offset, n_units, rows_per_unit, num_parts, out, lse, status=None, stream=None):
    _need(workspace, torch.uint8, "workspace")
    _check(load_library().mla_combine(_ptr(workspace), workspace.numel(), _ptr(split_offset), int(n_units),
                                      int(rows_per_unit), int(num_parts), _ptr(out),
                                      _DTYPE_CODE[out.dtype], _ptr(lse), _ptr(status), _stream(stream)), "mla_combine")


def mla_sparse_fp8_decode_fwd(q, kv8, indices, topk_length, sched, split_offset, num_parts, workspace, out, lse,
                              status, softmax_scale=1.0 / 24.0, stream=None):
    _need(q, torch.bfloat16, "q", 4)
    _need(kv8, torch.uint8, "kv8", 3)
    _need(indices, torch.int32, "indices", 3)
    if topk_length is not None:
        _need(topk_length, torch.int32, "topk_length", 2)
    _need(out, torch.bfloat16, "out", 4)
    B, s_q, h_q, d = q.shape
    if d != 576 or kv8.shape[1:] != (64, 656):
        raise ValueError("q must be [B, s_q, h_q, 576] and kv8 [pages, 64, 656]")
    if tuple(indices.shape[:2]) != (B, s_q):
        raise ValueError("indices must be [B, s_q, topk]")
    _check(load_library().mla_sparse_fp8_decode_fwd(
        _ptr(q), _ptr(kv8), kv8.shape[0], _ptr(indices), indices.shape[2], _ptr(topk_length), B, s_q, h_q,
        float(softmax_scale), _ptr(sched), _ptr(split_offset), int(num_parts), _ptr(workspace), workspace.numel(),
        _ptr(out), _ptr(lse), _ptr(status), _stream(stream)), "mla_sparse_fp8_decode_fwd")


def mla_sparse_fp8_unpack(kv8, indices, k_out, status, stream=None):
    _need(kv8, torch.uint8, "kv8", 3)
    _need(indices, torch.int32, "indices")
    _need(k_out, torch.float32, "k_out")
    n = indices.numel()
    if k_out.numel() < n * 576:
        raise ValueError("k_out too small")
    _check(load_library().mla_sparse_fp8_unpack(_ptr(kv8), kv8.shape[0], _ptr(indices), n, _ptr(k_out),
                                                _ptr(status), _stream(stream)), "mla_sparse_fp8_unpack")


def mla_packed_kv_workspace_bytes(n_units: int, topk: int) -> int:
    return int(load_library().mla_packed_kv_workspace_bytes(int(n_units), int(topk)))


def _pack(name, kv8, indices, topk_length, packed, status, stream):
    _need(kv8, torch.uint8, "kv8", 3)
    _need(indices, torch.int32, "indices", 3)
    if topk_length is not None:
        _need(topk_length, torch.int32, "topk_length", 2)
    _need(packed, torch.uint8, "packed")
    B, s_q, topk = indices.shape
    _check(getattr(load_library(), name)(_ptr(kv8), kv8.shape[0], _ptr(indices), topk, _ptr(topk_length), B * s_q,
                                         _ptr(packed), packed.numel(), _ptr(status), _stream(stream)), name)


def mla_pack_selected_kv(kv8, indices, topk_length, packed, status, stream=None):
    _pack("mla_pack_selected_kv", kv8, indices, topk_length, packed, status, stream)


def mla_test_pack_timeout(kv8, indices, topk_length, packed, status, stream=None):
    """Test hook: the pack with every block's bounded wait made to run out (MLA_ERR_TIMEOUT)."""
    _pack("mla_test_pack_timeout", kv8, indices, topk_length, packed, status, stream)


def mla_sparse_fp8_packed_decode_fwd(q, packed, topk, topk_length, sched, split_offset, num_parts, workspace, out,
                                     lse, status, softmax_scale=1.0 / 24.0, stream=None):
    _need(q, torch.bfloat16, "q", 4)
    _need(packed, torch.uint8, "packed")
    if topk_length is not None:
        _need(topk_length, torch.int32, "topk_length", 2)
    _need(out, torch.bfloat16, "out", 4)
    B, s_q, h_q, d = q.shape
    if d != 576:
        raise ValueError("q must be [B, s_q, h_q, 576]")
    _check(load_library().mla_sparse_fp8_packed_decode_fwd(
        _ptr(q), _ptr(packed), packed.numel(), int(topk), _ptr(topk_length), B, s_q, h_q, float(softmax_scale),
        _ptr(sched), _ptr(split_offset), int(num_parts), _ptr(workspace), workspace.numel(), _ptr(out), _ptr(lse),
        _ptr(status), _stream(stream)), "mla_sparse_fp8_packed_decode_fwd")


# ---------------------------------------------------------------- helpers


class Plan:
    """Scheduler output for one batch: reused by every layer of that batch."""

    def __init__(self, sched, split_offset, num_parts, n_units, rows, workspace):
        self.sched = sched
        self.split_offset = split_offset
        self.num_parts = num_parts
        self.n_units = n_units
        self.rows = rows
        self.workspace = workspace


def plan(lengths, n_units, rows_per_unit, sparse=False, default_length=-1, num_parts=None, stream=None,
         device=None, request_local=False) -> Plan:
    """Run the scheduler kernel (native or request-local plan) and allocate the split workspace."""
    dev = device if device is not None else (lengths.device if lengths is not None else torch.device("cuda"))
    parts = mla_num_parts(rows_per_unit, sparse) if num_parts is None else int(num_parts)
    sched = torch.empty(parts * 8, dtype=torch.int32, device=dev)
    split_offset = torch.empty(n_units + 1, dtype=torch.int32, device=dev)
    fn = mla_get_metadata_request_local if request_local else mla_get_metadata
    fn(lengths, n_units, parts, sched, split_offset, default_length, stream)
    ws = torch.empty(mla_workspace_bytes(n_units, rows_per_unit, parts), dtype=torch.uint8, device=dev)
    return Plan(sched, split_offset, parts, n_units, rows_per_unit, ws)


def check_status(status: torch.Tensor, where: str):
    code = int(status.item())
    if code != 0:
        raise MlaError(code, where)


def decode(q, kv, block_table, cache_seqlens, causal=False, softmax_scale=None, out_fp32=False, pl=None,
           check=True):
    """Dense decode with freshly allocated outputs; returns (out, lse).  The
    cache is bf16 or fp16 latent rows, or FP8 records (uint8 [pages, 64, 656],
    bf16 q)."""
    B, s_q, h_q, _ = q.shape
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(576)
    if pl is None:
        h_kv = 1 if kv.dim() == 3 else kv.shape[2]
        pl = plan(cache_seqlens, B, s_q * h_q, num_parts=mla_num_parts_dense(s_q, h_q, h_kv))
    out = torch.empty(B, s_q, h_q, 512, dtype=torch.float32 if out_fp32 else q.dtype, device=q.device)
    lse = torch.empty(B, s_q, h_q, dtype=torch.float32, device=q.device)
    status = torch.zeros(1, dtype=torch.int32, device=q.device)
    mla_decode_fwd(q, kv, block_table, cache_seqlens, pl.sched, pl.split_offset, pl.num_parts, pl.workspace, out,
                   lse, status, causal, softmax_scale)
    if check:
        check_status(status, "mla_decode_fwd")
    return out, lse


def sparse_decode(q, kv8, indices, topk_length=None, softmax_scale=None, pl=None, check=True):
    """Sparse FP8 decode with freshly allocated outputs; returns (out, lse)."""
    B, s_q, h_q, _ = q.shape
    topk = indices.shape[2]
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(576)
    if pl is None:
        lens = None if topk_length is None else topk_length.reshape(-1)
        pl = plan(lens, B * s_q, h_q, sparse=True, default_length=topk, device=q.device)
    out = torch.empty(B, s_q, h_q, 512, dtype=torch.bfloat16, device=q.device)
    lse = torch.empty(B, s_q, h_q, dtype=torch.float32, device=q.device)
    status = torch.zeros(1, dtype=torch.int32, device=q.device)
    mla_sparse_fp8_decode_fwd(q, kv8, indices, topk_length, pl.sched, pl.split_offset, pl.num_parts, pl.workspace,
                              out, lse, status, softmax_scale)
    if check:
        check_status(status, "mla_sparse_fp8_decode_fwd")
    return out, lse


def pack_selected_kv(kv8, indices, topk_length=None, check=True):
    """Pack the selected records into a freshly allocated packed workspace."""
    B, s_q, topk = indices.shape
    packed = torch.empty(mla_packed_kv_workspace_bytes(B * s_q, topk), dtype=torch.uint8, device=kv8.device)
    status = torch.zeros(1, dtype=torch.int32, device=kv8.device)
    mla_pack_selected_kv(kv8, indices, topk_length, packed, status)
    if check:
        check_status(status, "mla_pack_selected_kv")
    return packed


def packed_sparse_decode(q, packed, topk, topk_length=None, softmax_scale=None, pl=None, check=True):
    """Sparse FP8 decode over a packed workspace; returns (out, lse)."""
    B, s_q, h_q, _ = q.shape
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(576)
    if pl is None:
        lens = None if topk_length is None else topk_length.reshape(-1)
        pl = plan(lens, B * s_q, h_q, sparse=True, default_length=topk, device=q.device)
    out = torch.empty(B, s_q, h_q, 512, dtype=torch.bfloat16, device=q.device)
    lse = torch.empty(B, s_q, h_q, dtype=torch.float32, device=q.device)
    status = torch.zeros(1, dtype=torch.int32, device=q.device)
    mla_sparse_fp8_packed_decode_fwd(q, packed, topk, topk_length, pl.sched, pl.split_offset, pl.num_parts,
                                     pl.workspace, out, lse, status, softmax_scale)
    if check:
        check_status(status, "mla_sparse_fp8_packed_decode_fwd")
    return out, lse
