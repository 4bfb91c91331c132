"""GPU test of dsa_indexer_fused_noalloc, the fused entry point that takes no
workspace (for callers that cannot allocate device memory: its scratch is a
fixed device array inside the library).

It is called through the C ABI and compared with dsa_indexer_fused given a
caller-allocated workspace, on two calls in a row (the second call reuses the
scratch the first one left behind).  Collected last so that a stop-at-first-
failure run has already run every other test.
"""
import ctypes

import numpy as np
import pytest

from sparse_attention_paged_dsa_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _noalloc(lib):
    f = lib.dsa_indexer_fused_noalloc
    p, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    f.argtypes = [p, p, p, i64, p, p, i32, i64, i32, p, p]
    f.restype = ctypes.c_int
    return f


def _get_error(lib):
    f = lib.dsa_indexer_noalloc_get_error
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
    f.restype = ctypes.c_int
    return f


def _read_error(lib, stream, clear=1):
    code = ctypes.c_uint32(0)
    assert _get_error(lib)(ctypes.byref(code), clear, stream) == 0
    return int(code.value)


def _call(f, case, dev, topk, stream, k=None):
    q, w, pool, table, seq = dev
    P = ctypes.c_void_p
    return f(P(q.data_ptr()), P(w.data_ptr()), P(pool.data_ptr()), case.num_pages, P(table.data_ptr()),
             P(seq.data_ptr()), case.batch, case.max_context, case.k if k is None else k, P(topk.data_ptr()),
             stream)


def test_noalloc_matches_fused_on_two_calls_in_a_row(gpu_lib):
    import torch
    b = gpu_lib
    f = _noalloc(b.load())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    cases = [I.workload("b64_ctx128k_loguniform"),
             I.make_case(name="second", batch=9, max_context=65536,
                         seq_lens=[65536, 1, 0, 40000, 257, 5, 65000, 1000, 32768], num_pages=1200, k=1024,
                         seed=31)]
    for case in cases:
        dev = b.to_device(case)
        want = b.dsa_indexer_fused(*dev, case.max_context, case.k)
        got = torch.full((case.batch, case.k), -7, dtype=torch.int32, device="cuda")
        assert _call(f, case, dev, got, stream) == b.DSA_OK
        torch.cuda.synchronize()
        np.testing.assert_array_equal(got.cpu().numpy(), want.cpu().numpy())


def test_noalloc_rejects_shapes_beyond_its_scratch(gpu_lib):
    import torch
    b = gpu_lib
    f = _noalloc(b.load())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    case = I.make_case(name="big", batch=64, max_context=1 << 20, seq_lens=[512] * 64, num_pages=256, k=2048,
                       seed=4)  # 64 x 262144 fp32 slots = 64 MiB > 16 MiB
    dev = b.to_device(case)
    out = torch.full((case.batch, case.k), -7, dtype=torch.int32, device="cuda")
    assert _call(f, case, dev, out, stream) == b.DSA_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert int(out.min()) == -7 and int(out.max()) == -7


def test_noalloc_checks_arguments_first_and_reports_device_errors(gpu_lib):
    """Rejected calls launch nothing; a live page id outside the pool is flagged in the scratch's
    error word, which dsa_indexer_noalloc_get_error reads back (sticky until cleared)."""
    import torch
    b = gpu_lib
    lib = b.load()
    f = _noalloc(lib)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    case = I.make_case(name="errs", batch=3, max_context=8192, seq_lens=[8192, 600, 3000], num_pages=64, k=256,
                       seed=17)
    dev = list(b.to_device(case))
    out = torch.full((case.batch, case.k), -7, dtype=torch.int32, device="cuda")
    _read_error(lib, stream)  # start from a clear word
    assert _call(f, case, dev, out, stream, k=0) == b.DSA_ERR_INVALID_ARG
    assert _call(f, case, dev, out, stream, k=case.max_context // 4 + 1) == b.DSA_ERR_INVALID_ARG
    # batch past the limit (buffers of the full size, so that nothing could be read out of bounds)
    B2 = 2000
    P = ctypes.c_void_p
    q2 = torch.zeros((B2, 32, 64), dtype=torch.bfloat16, device="cuda")
    w2 = torch.zeros((B2, 32), dtype=torch.float32, device="cuda")
    t2 = torch.zeros((B2, 32), dtype=torch.int32, device="cuda")
    s2 = torch.ones((B2,), dtype=torch.int32, device="cuda")
    o2 = torch.empty((B2, 4), dtype=torch.int32, device="cuda")
    assert f(P(q2.data_ptr()), P(w2.data_ptr()), P(dev[2].data_ptr()), case.num_pages, P(t2.data_ptr()),
             P(s2.data_ptr()), B2, 8192, 4, P(o2.data_ptr()), stream) == b.DSA_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert int(out.min()) == -7 and int(out.max()) == -7
    assert _read_error(lib, stream) == 0
    # a bad page id in row 1's live range
    table = dev[3].clone()
    table[1, 1] = case.num_pages + 5
    dev[3] = table
    assert _call(f, case, dev, out, stream) == b.DSA_OK
    assert _read_error(lib, stream, clear=0) == b.DEVERR_BAD_PAGE
    assert _read_error(lib, stream, clear=1) == b.DEVERR_BAD_PAGE  # still there: sticky until cleared
    assert _read_error(lib, stream) == 0
