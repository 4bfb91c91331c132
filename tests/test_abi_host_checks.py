"""CPU checks of the C ABI's host-side argument checks: every rejected call returns the status
include/dsa_indexer.h documents (DSA_ERR_INVALID_ARG, DSA_ERR_UNSUPPORTED or DSA_ERR_WORKSPACE)
before it makes any CUDA call, so these run without a GPU.  The pointers are never dereferenced on
these paths; they are plain addresses chosen for their alignment."""
import ctypes

import pytest

OK, INVALID, UNSUPPORTED, WORKSPACE = 0, 1, 2, 3
A16 = 0x100000        # 16-byte (and 256-byte) aligned address
A4 = 0x100004         # 4-byte aligned only
A8 = 0x100008         # 8-byte aligned only
P = ctypes.c_void_p


@pytest.fixture(scope="module")
def lib():
    from sparse_attention_paged_dsa_gb300 import build
    lib = ctypes.CDLL(build.build())
    lib.dsa_indexer_fused.argtypes = [P, P, P, ctypes.c_int64, P, P, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32,
                                      P, P, P, ctypes.c_size_t, P]
    lib.dsa_indexer_scores.argtypes = [P, P, P, ctypes.c_int64, P, P, ctypes.c_int32, ctypes.c_int64, P, P,
                                       ctypes.c_size_t, P]
    lib.dsa_indexer_topk.argtypes = [P, P, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, P, P, ctypes.c_size_t, P]
    lib.dsa_indexer_workspace_size.argtypes = [ctypes.c_int32, ctypes.c_int64, ctypes.c_int32]
    lib.dsa_indexer_workspace_size.restype = ctypes.c_size_t
    for f in (lib.dsa_indexer_fused, lib.dsa_indexer_scores, lib.dsa_indexer_topk):
        f.restype = ctypes.c_int
    return lib


def fused_args(**over):
    a = dict(q=A16, w=A16, pool=A16, pages=64, table=A16, seq=A16, batch=2, ctx=8192, k=16, topk=A16,
             scores=None, ws=A16, wsb=1 << 30, stream=None)
    a.update(over)
    return [a["q"], a["w"], a["pool"], a["pages"], a["table"], a["seq"], a["batch"], a["ctx"], a["k"], a["topk"],
            a["scores"], a["ws"], a["wsb"], a["stream"]]


@pytest.mark.parametrize("over, status", [
    (dict(batch=0), INVALID),                  # no request
    (dict(batch=-3), INVALID),
    (dict(batch=1025), UNSUPPORTED),           # past DSA_MAX_BATCH
    (dict(ctx=0), INVALID),
    (dict(ctx=8192 + 4), INVALID),             # not a whole number of 256-token pages
    (dict(ctx=(1 << 24) + 256), UNSUPPORTED),  # past the 16M-token row limit
    (dict(q=None), INVALID),
    (dict(w=None), INVALID),
    (dict(pool=None), INVALID),
    (dict(table=None), INVALID),
    (dict(seq=None), INVALID),
    (dict(topk=None), INVALID),
    (dict(q=A8), INVALID),                     # q must be 16-byte aligned
    (dict(pool=A8), INVALID),
    (dict(w=A4), INVALID),
    (dict(table=A4 + 1), INVALID),             # int32 arrays must be 4-byte aligned
    (dict(seq=A4 + 2), INVALID),
    (dict(topk=A4 + 1), INVALID),
    (dict(scores=A8), INVALID),                # an optional row must be 16-byte aligned
    (dict(pages=0), INVALID),
    (dict(pages=1 << 31), INVALID),
    (dict(k=0), INVALID),
    (dict(k=8192 // 4 + 1), INVALID),          # k above the row width
    (dict(ws=None), WORKSPACE),
    (dict(ws=A16 + 16), WORKSPACE),            # the workspace must be 256-byte aligned
    (dict(wsb=255), WORKSPACE),                # smaller than the header
])
def test_fused_rejects_bad_arguments(lib, over, status):
    assert lib.dsa_indexer_fused(*fused_args(**over)) == status


def test_fused_workspace_must_hold_the_live_slots_without_a_row(lib):
    need = lib.dsa_indexer_workspace_size(2, 8192, 16)
    assert need > 256
    # without a scores row the workspace holds the live-score slots; with one, the header suffices
    # (the call then goes on to CUDA, which this check stops short of: only the shortfall is tested)
    assert lib.dsa_indexer_fused(*fused_args(wsb=need - 1)) == WORKSPACE


@pytest.mark.parametrize("over, status", [
    (dict(batch=0), INVALID),
    (dict(batch=2000), UNSUPPORTED),
    (dict(ctx=100), INVALID),
    (dict(q=None), INVALID),
    (dict(q=A8), INVALID),
    (dict(scores=None), INVALID),
    (dict(scores=A8), INVALID),
    (dict(pages=0), INVALID),
    (dict(ws=None), WORKSPACE),
    (dict(wsb=128), WORKSPACE),
])
def test_scores_rejects_bad_arguments(lib, over, status):
    a = dict(q=A16, w=A16, pool=A16, pages=64, table=A16, seq=A16, batch=2, ctx=8192, scores=A16, ws=A16,
             wsb=1 << 20, stream=None)
    a.update(over)
    args = [a["q"], a["w"], a["pool"], a["pages"], a["table"], a["seq"], a["batch"], a["ctx"], a["scores"],
            a["ws"], a["wsb"], a["stream"]]
    assert lib.dsa_indexer_scores(*args) == status


@pytest.mark.parametrize("over, status", [
    (dict(batch=0), INVALID),
    (dict(batch=1025), UNSUPPORTED),
    (dict(ctx=1000), INVALID),
    (dict(scores=None), INVALID),
    (dict(scores=A8), INVALID),
    (dict(seq=None), INVALID),
    (dict(topk=A4 + 2), INVALID),
    (dict(k=0), INVALID),
    (dict(k=2049), INVALID),                   # 8192 / 4 = 2048 positions per row
    (dict(ws=A16 + 64), WORKSPACE),
    (dict(wsb=0), WORKSPACE),
])
def test_topk_rejects_bad_arguments(lib, over, status):
    a = dict(scores=A16, seq=A16, batch=2, ctx=8192, k=16, topk=A16, ws=A16, wsb=1 << 20, stream=None)
    a.update(over)
    args = [a["scores"], a["seq"], a["batch"], a["ctx"], a["k"], a["topk"], a["ws"], a["wsb"], a["stream"]]
    assert lib.dsa_indexer_topk(*args) == status


@pytest.mark.parametrize("over, status", [
    (dict(batch=0), INVALID),
    (dict(batch=1025), UNSUPPORTED),
    (dict(codes=None), INVALID),
    (dict(codes=A8), INVALID),                 # codes must be 16-byte aligned
    (dict(scales=None), INVALID),
    (dict(scales=A8), INVALID),                # scales must be 16-byte aligned
    (dict(q=A8), INVALID),
    (dict(pages=0), INVALID),
    (dict(k=0), INVALID),
    (dict(ws=None), WORKSPACE),
])
def test_fused_fp8_rejects_bad_arguments(lib, over, status):
    f = lib.dsa_indexer_fused_fp8
    f.argtypes = [P, P, P, P, ctypes.c_int64, P, P, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, P, P, P,
                  ctypes.c_size_t, P]
    f.restype = ctypes.c_int
    a = dict(q=A16, w=A16, codes=A16, scales=A16, pages=64, table=A16, seq=A16, batch=2, ctx=8192, k=16,
             topk=A16, scores=None, ws=A16, wsb=1 << 30, stream=None)
    a.update(over)
    assert f(a["q"], a["w"], a["codes"], a["scales"], a["pages"], a["table"], a["seq"], a["batch"], a["ctx"],
             a["k"], a["topk"], a["scores"], a["ws"], a["wsb"], a["stream"]) == status


@pytest.mark.parametrize("over, status", [
    (dict(next_n=0), INVALID),
    (dict(next_n=5), INVALID),                 # 1 <= next_n <= DSA_MAX_NEXT_N = 4
    (dict(batch=0), INVALID),
    (dict(q=None), INVALID),
    (dict(k=0), INVALID),
    (dict(ws=A16 + 128), WORKSPACE),
])
def test_fused_mtp_rejects_bad_arguments(lib, over, status):
    f = lib.dsa_indexer_fused_mtp
    f.argtypes = [P, P, P, ctypes.c_int64, P, P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, P,
                  P, P, ctypes.c_size_t, P]
    f.restype = ctypes.c_int
    a = dict(q=A16, w=A16, pool=A16, pages=64, table=A16, seq=A16, batch=2, next_n=2, ctx=8192, k=16, topk=A16,
             scores=None, ws=A16, wsb=1 << 30, stream=None)
    a.update(over)
    assert f(a["q"], a["w"], a["pool"], a["pages"], a["table"], a["seq"], a["batch"], a["next_n"], a["ctx"],
             a["k"], a["topk"], a["scores"], a["ws"], a["wsb"], a["stream"]) == status


@pytest.mark.parametrize("over, status", [
    (dict(batch=0), INVALID),
    (dict(batch=257), INVALID),                # past DSA_PROJ_MAX_TOKENS
    (dict(d=32), INVALID),                     # d_model a multiple of 64
    (dict(d=7168 + 32), INVALID),
    (dict(x=None), INVALID),
    (dict(x=A8), INVALID),
    (dict(wq=A8), INVALID),
    (dict(ww=None), INVALID),
    (dict(qo=A4 + 1), INVALID),
    (dict(wo=None), INVALID),
    (dict(ws=None), WORKSPACE),
    (dict(wsb=255), WORKSPACE),
])
def test_qw_proj_rejects_bad_arguments(lib, over, status):
    f = lib.dsa_indexer_qw_proj
    f.argtypes = [P, P, P, ctypes.c_int32, ctypes.c_int64, P, P, P, ctypes.c_size_t, P]
    f.restype = ctypes.c_int
    lib.dsa_indexer_qw_proj_workspace_size.argtypes = [ctypes.c_int32, ctypes.c_int64]
    lib.dsa_indexer_qw_proj_workspace_size.restype = ctypes.c_size_t
    a = dict(x=A16, wq=A16, ww=A16, batch=64, d=7168, qo=A16, wo=A16, ws=A16, wsb=1 << 20, stream=None)
    a.update(over)
    assert f(a["x"], a["wq"], a["ww"], a["batch"], a["d"], a["qo"], a["wo"], a["ws"], a["wsb"], a["stream"]) == status
    assert lib.dsa_indexer_qw_proj_workspace_size(64, 7168) == 256
    assert lib.dsa_indexer_qw_proj_workspace_size(0, 7168) == 0
    assert lib.dsa_indexer_qw_proj_workspace_size(64, 100) == 0


@pytest.mark.parametrize("over, status", [
    (dict(batch=0), INVALID),
    (dict(ctx=1000), INVALID),
    (dict(q=None), INVALID),
    (dict(q=A8), INVALID),
    (dict(kv=A8), INVALID),
    (dict(out=A8), INVALID),
    (dict(lse=A4), INVALID),
    (dict(topk=None), INVALID),
    (dict(pages=0), INVALID),
    (dict(k=0), INVALID),
    (dict(k=2049), INVALID),                   # past DSA_MLA_MAX_TOPK
    (dict(scale=float("nan")), INVALID),
    (dict(scale=float("inf")), INVALID),
    (dict(ws=None), WORKSPACE),
    (dict(wsb=0), WORKSPACE),
    (dict(pages=1 << 25), UNSUPPORTED),        # cache rows past 32-bit coordinates
])
def test_sparse_mla_rejects_bad_arguments(lib, over, status):
    f = lib.dsa_sparse_mla_decode
    f.argtypes = [P, P, ctypes.c_int64, P, P, ctypes.c_int32, ctypes.c_int64, P, ctypes.c_int32, ctypes.c_float,
                  P, P, P, ctypes.c_size_t, P]
    f.restype = ctypes.c_int
    a = dict(q=A16, kv=A16, pages=64, table=A16, seq=A16, batch=2, ctx=8192, topk=A16, k=64, scale=0.04,
             out=A16, lse=A16, ws=A16, wsb=1 << 30, stream=None)
    a.update(over)
    assert f(a["q"], a["kv"], a["pages"], a["table"], a["seq"], a["batch"], a["ctx"], a["topk"], a["k"], a["scale"],
             a["out"], a["lse"], a["ws"], a["wsb"], a["stream"]) == status
