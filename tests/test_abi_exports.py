"""CPU checks of the C ABI: the library builds for sm_103a, loads without a
GPU, and exports every function include/dsa_indexer.h declares."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsa_indexer.h")


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"DSA_API\s+[\w\s\*]+?\b(dsa_\w+)\s*\(", text)


@pytest.fixture(scope="module")
def lib_path():
    from sparse_attention_paged_dsa_gb300 import build
    return build.build()


def test_header_declares_the_entry_points():
    names = set(declared_functions())
    assert {"dsa_indexer_scores", "dsa_indexer_topk", "dsa_indexer_fused", "dsa_indexer_workspace_size",
            "dsa_indexer_get_error", "dsa_status_string"} <= names


def test_library_exports_every_declared_symbol(lib_path):
    out = subprocess.run(["nm", "-D", "--defined-only", lib_path], capture_output=True, text=True, check=True)
    exported = set(re.findall(r"\sT\s(\w+)$", out.stdout, re.M))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, f"not exported: {missing}"
    lib = ctypes.CDLL(lib_path)
    for n in declared_functions():
        assert hasattr(lib, n)


def documented_workspace_bytes(rows, max_context, slots=True):
    """The workspace size the header documents: a 256-byte header and, for the fused
    calls without a scores row, live-score slots (M x 4 B per row)."""
    M = max_context // 4
    up = lambda n: (n + 255) // 256 * 256
    parts = [256]
    if slots:
        parts.append(rows * M * 4)
    return sum(up(p) for p in parts)


def test_host_only_queries_without_gpu(lib_path):
    lib = ctypes.CDLL(lib_path)
    lib.dsa_indexer_workspace_size.argtypes = [ctypes.c_int32, ctypes.c_int64, ctypes.c_int32]
    lib.dsa_indexer_workspace_size.restype = ctypes.c_size_t
    lib.dsa_indexer_workspace_size_mtp.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32]
    lib.dsa_indexer_workspace_size_mtp.restype = ctypes.c_size_t
    lib.dsa_status_string.argtypes = [ctypes.c_int]
    lib.dsa_status_string.restype = ctypes.c_char_p
    for batch, ctx in ((64, 131072), (2, 1024), (1, 8192), (64, 1 << 20), (7, 33 * 256)):
        assert lib.dsa_indexer_workspace_size(batch, ctx, 2048) == documented_workspace_bytes(batch, ctx)
    assert lib.dsa_indexer_workspace_size(64, 131072, 2048) == 256 + 64 * 32768 * 4
    assert lib.dsa_indexer_workspace_size_mtp(16, 3, 8192, 64) == documented_workspace_bytes(48, 8192)
    assert lib.dsa_indexer_workspace_size(0, 131072, 2048) == 0
    assert lib.dsa_indexer_workspace_size(4, 1000, 8) == 0
    assert lib.dsa_status_string(0) == b"ok"
