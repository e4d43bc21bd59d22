"""The C-ABI library loads and exports every entry point the header declares (CPU only).

Also checks the host-side argument validation that returns before any
launch and needs no GPU: null pointers and bad sizes come back as
MLA_ERR_INVALID_ARG.
"""

import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mla_paged_kv.h")


@pytest.fixture(scope="module")
def lib_path():
    from mla_paged_kv_gb300 import build
    if not os.path.exists(build.LIB_PATH):
        build.build()
    return build.LIB_PATH


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^(?:const char\*|int|size_t)\s+(mla_\w+)\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    assert names == sorted(["mla_status_string", "mla_num_parts", "mla_workspace_bytes", "mla_get_metadata",
                            "mla_decode_fwd", "mla_decode_splits", "mla_combine", "mla_sparse_fp8_decode_fwd",
                            "mla_sparse_fp8_unpack", "mla_decode_fwd_static_ws", "mla_packed_kv_workspace_bytes",
                            "mla_pack_selected_kv", "mla_sparse_fp8_packed_decode_fwd",
                            "mla_get_metadata_request_local", "mla_num_parts_dense", "mla_test_pack_timeout",
                            "mla_test_decode_timeout"])


def test_library_exports_every_declared_symbol(lib_path):
    out = subprocess.run(["nm", "-D", "--defined-only", lib_path], capture_output=True, text=True, check=True)
    exported = set(re.findall(r"\sT\s(mla_\w+)$", out.stdout, flags=re.M))
    assert set(declared_functions()) <= exported
    lib = ctypes.CDLL(lib_path)
    for name in declared_functions():
        assert getattr(lib, name) is not None


def test_python_binding_names_match(lib_path):
    import mla_paged_kv_gb300 as mla
    assert set(mla.EXPORTED_SYMBOLS) == set(declared_functions())
    for name in declared_functions():
        assert callable(getattr(mla, name))


def test_host_validation_without_gpu(lib_path):
    lib = ctypes.CDLL(lib_path)
    lib.mla_status_string.restype = ctypes.c_char_p
    assert lib.mla_status_string(0) == b"MLA_OK"
    assert b"unknown" in lib.mla_status_string(99)
    lib.mla_workspace_bytes.restype = ctypes.c_size_t
    lib.mla_workspace_bytes.argtypes = [ctypes.c_int] * 3
    # (n_units + num_parts) slots x rows x (512 + 1) fp32: fp32 O, then fp32 LSE,
    # each region 256-byte aligned (36,771,840 bytes at 64 x 128 rows, 76 parts)
    assert lib.mla_workspace_bytes(64, 128, 76) == (64 + 76) * 128 * 512 * 4 + (64 + 76) * 128 * 4
    assert lib.mla_workspace_bytes(1, 3, 1) == 2 * 3 * 2048 + 256
    assert lib.mla_workspace_bytes(0, 0, 1) == 0
    null = ctypes.c_void_p(0)
    lib.mla_get_metadata.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                     ctypes.c_void_p, ctypes.c_void_p]
    assert lib.mla_get_metadata(null, -1, 4, 2, null, null, null) == 1          # MLA_ERR_INVALID_ARG
    assert lib.mla_get_metadata(null, 10, 0, 2, ctypes.c_void_p(16), ctypes.c_void_p(16), null) == 1
    # q, kv, block_table, max_pages, num_pages, seqlens, batch, s_q, h_q, h_kv, dtype, causal, scale, sched,
    # split_offset, num_parts, workspace, workspace_bytes, out, out_type, lse, status, stream
    args = [null] * 3 + [1, 1, null, 1, 1, 1, 1, 0, 0, 0.04, null, null, 1, null, 0, null, 0, null, null, null]
    lib.mla_decode_fwd.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 2 + [ctypes.c_void_p] + \
        [ctypes.c_int] * 6 + [ctypes.c_float] + [ctypes.c_void_p] * 2 + [ctypes.c_int, ctypes.c_void_p,
                                                                           ctypes.c_size_t, ctypes.c_void_p,
                                                                           ctypes.c_int] + [ctypes.c_void_p] * 3
    assert lib.mla_decode_fwd(*args) == 1
    lib.mla_sparse_fp8_unpack.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
                                          ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    assert lib.mla_sparse_fp8_unpack(null, 1, null, 4, null, null, null) == 1
    # packed workspace: [units, tiles, 64, 656] records, then [units, tiles] uint64 masks
    lib.mla_packed_kv_workspace_bytes.restype = ctypes.c_size_t
    lib.mla_packed_kv_workspace_bytes.argtypes = [ctypes.c_int, ctypes.c_int]
    assert lib.mla_packed_kv_workspace_bytes(16, 2048) == 16 * 32 * (64 * 656 + 8)
    assert lib.mla_packed_kv_workspace_bytes(3, 65) == 3 * 2 * (64 * 656 + 8)
    assert lib.mla_packed_kv_workspace_bytes(3, 0) == 0
    lib.mla_pack_selected_kv.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
                                         ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t,
                                         ctypes.c_void_p, ctypes.c_void_p]
    assert lib.mla_pack_selected_kv(null, 1, null, 64, null, 1, null, 0, null, null) == 1
    # a workspace smaller than the layout is refused before any launch
    p16 = ctypes.c_void_p(256)
    assert lib.mla_pack_selected_kv(p16, 1, p16, 64, null, 1, p16, 64 * 656, p16, null) == 1

    # pools whose slot count does not fit int32 are refused before any launch (pack, test hook, unpack)
    big = (1 << 31) // 64
    assert lib.mla_pack_selected_kv(p16, big, p16, 64, null, 1, p16, 1 << 20, p16, null) == 2   # UNSUPPORTED
    lib.mla_test_pack_timeout.argtypes = lib.mla_pack_selected_kv.argtypes
    assert lib.mla_test_pack_timeout(p16, big, p16, 64, null, 1, p16, 1 << 20, p16, null) == 2
    assert lib.mla_test_pack_timeout(null, 1, null, 64, null, 1, null, 0, null, null) == 1
    assert lib.mla_sparse_fp8_unpack(p16, big, p16, 4, p16, p16, null) == 2
