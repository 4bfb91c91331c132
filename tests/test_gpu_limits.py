"""GPU parity at the boundary's size limits.

* DSA_MAX_BATCH = 1024 requests in one call (the per-request tables fill one
  warp's 32 rows per lane) with ragged lengths 0..4096 tokens.
* max_context = 2^24 tokens, the largest row (4,194,304 C4 positions = 32768
  two-page units: the largest unit index the kernels encode), one request
  that fills it; scores are compared with the oracle on windows at the start,
  the middle and the end of the row (the oracle on the same query and the
  window's pages), the top-k (2048 of 4M, the global-memory selection path)
  with an exact sort of the kernel's own scores.
* Just past each limit the call is rejected on the host.
"""
import numpy as np
import pytest

from sparse_attention_paged_dsa_gb300 import inputs as I

from _parity import check_scores, check_topk, own_topk

pytestmark = pytest.mark.gpu


def test_max_batch_ragged(gpu_lib, oracle):
    import torch
    rng = np.random.default_rng(2024)
    seqs = rng.integers(0, 4097, size=1024)
    seqs[:8] = [0, 1, 4, 5, 255, 256, 257, 4096]
    case = I.make_case(name="maxbatch", batch=1024, max_context=4096, seq_lens=seqs, num_pages=9000, k=64,
                       seed=31)
    q, w, pool, table, seq = gpu_lib.to_device(case)
    ws = gpu_lib.new_workspace(case.batch, case.max_context, case.k)
    s = gpu_lib.dsa_indexer_scores(q, w, pool, table, seq, case.max_context, workspace=ws)
    t = gpu_lib.dsa_indexer_fused(q, w, pool, table, seq, case.max_context, case.k, workspace=ws)
    torch.cuda.synchronize()
    assert gpu_lib.get_error(ws) == 0
    s, t = s.cpu().numpy(), t.cpu().numpy()
    ref = oracle.case_scores(case)
    check_scores(case, s, ref)
    check_topk(case, t, ref, gpu_scores=s)


def test_max_context_one_full_row(gpu_lib, oracle):
    import torch
    ctx = 1 << 24
    W = ctx // 256
    case = I.make_case(name="maxctx", batch=1, max_context=ctx, seq_lens=[ctx], num_pages=W, k=2048, seed=33)
    q, w, pool, table, seq = gpu_lib.to_device(case)
    ws = gpu_lib.new_workspace(1, ctx, case.k)
    s = gpu_lib.dsa_indexer_scores(q, w, pool, table, seq, ctx, workspace=ws)
    t = gpu_lib.dsa_indexer_fused(q, w, pool, table, seq, ctx, case.k, workspace=ws)
    torch.cuda.synchronize()
    assert gpu_lib.get_error(ws) == 0
    s, t = s.cpu().numpy()[0], t.cpu().numpy()[0]
    n = ctx // 4
    assert np.all(np.isfinite(s))
    for p0 in (0, W // 2 - 1, W - 2):  # two pages at the start, across the middle, at the end
        sub = I.IndexerCase("win", case.q, case.w, case.key_pool, case.page_table[:, p0:p0 + 2].copy(),
                            np.array([512], np.int32), 512, case.k)
        ref = oracle.case_scores(sub)[0]
        got = s[p0 * 64:(p0 + 2) * 64]
        rel = np.abs(got - ref).max() / np.abs(ref).max()
        assert rel <= 3e-3, (p0, rel)
    np.testing.assert_array_equal(t, own_topk(s, n, case.k))


def test_past_the_limits_rejected(gpu_lib):
    import ctypes
    import torch
    b = gpu_lib
    lib = b.load()
    P = ctypes.c_void_p
    buf = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    ptr = P(buf.data_ptr())
    s = P(torch.cuda.current_stream().cuda_stream)
    # batch 1025 and max_context 2^24 + 256: nothing launched, status says why
    assert lib.dsa_indexer_scores(ptr, ptr, ptr, 1, ptr, ptr, 1025, 1024, ptr, ptr, 1 << 16, s) == b.DSA_ERR_UNSUPPORTED
    assert lib.dsa_indexer_scores(ptr, ptr, ptr, 1, ptr, ptr, 1, (1 << 24) + 256, ptr, ptr, 1 << 16, s) == \
        b.DSA_ERR_UNSUPPORTED
    assert lib.dsa_indexer_workspace_size(1025, 1024, 1) == 0
    torch.cuda.synchronize()
    assert int(buf.count_nonzero()) == 0


@pytest.mark.parametrize("path", ["bf16", "fp8", "two_token", "four_token"])
def test_short_mixed_rows_query_slots(gpu_lib, oracle, path):
    """1024 requests of one to three two-page units in a mixed order, so that consecutive rows
    start on units of either producer warp and the two query slots turn over every few units;
    repeated five times, each run must leave the error word clear and match the oracle."""
    import torch
    rng = np.random.default_rng(4049)
    seqs = rng.choice(np.array([1, 512, 513, 1024, 1025, 1536]), size=1024)
    case = I.make_case(name="shortrows", batch=1024, max_context=2048, seq_lens=seqs, num_pages=4096, k=64,
                       seed=41)
    q, w, pool, table, seq = gpu_lib.to_device(case)
    ws = gpu_lib.new_workspace(case.batch, case.max_context, case.k)
    if path == "fp8":
        f = I.with_fp8_keys(case)
        codes, scales = gpu_lib.to_device_fp8(f)
        ref = oracle.case_scores_fp8(f)
        run = lambda: gpu_lib.dsa_indexer_scores_fp8(q, w, codes, scales, table, seq, case.max_context, workspace=ws)
    elif path in ("two_token", "four_token"):
        m = I.with_next_n(case, 2 if path == "two_token" else 4)
        qm = torch.from_numpy(m.q.view("int16")).cuda().view(torch.bfloat16)
        wm = torch.from_numpy(m.w).cuda()
        ref = oracle.case_scores_mtp(m).reshape(-1, case.max_context // 4)
        run = lambda: gpu_lib.dsa_indexer_scores_mtp(qm, wm, pool, table, seq, case.max_context,
                                                     workspace=ws).reshape(-1, case.max_context // 4)
    else:
        ref = oracle.case_scores(case)
        run = lambda: gpu_lib.dsa_indexer_scores(q, w, pool, table, seq, case.max_context, workspace=ws)
    live = np.isfinite(ref)
    for _ in range(5):
        s = run()
        torch.cuda.synchronize()
        assert gpu_lib.get_error(ws) == 0
        s = s.cpu().numpy()
        assert np.array_equal(np.isfinite(s), live)
        for r in range(ref.shape[0]):
            if live[r].any():
                rel = np.abs(s[r][live[r]] - ref[r][live[r]]).max() / np.abs(ref[r][live[r]]).max()
                assert rel <= 3e-3, f"row {r}: {rel}"
