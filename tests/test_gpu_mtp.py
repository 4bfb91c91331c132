"""GPU parity of the multi-token indexer (next_n query tokens per request) against the oracle.

Reading (see the header): the request's seq_len counts all next_n tokens; token j scores
the keys of its causal prefix of seq_len - (next_n - 1 - j) tokens and writes row
b x next_n + j.  The kernel reads each key page once for all tokens (N = 32 next_n in one
MMA).  Same tolerances as the single-token path; integer inputs are bit-exact.
"""
import ctypes

import numpy as np
import pytest

from sparse_attention_paged_dsa_gb300 import inputs as I

from _parity import check_scores, check_topk

pytestmark = pytest.mark.gpu


def _flat(case):
    """The batch x next_n token rows as an ordinary case (for the row-wise checks)."""
    B, Q = case.q.shape[0], case.q.shape[1]
    seq = np.asarray(case.seq_lens, dtype=np.int64)
    seq_j = np.stack([np.maximum(seq - (Q - 1 - j), 0) for j in range(Q)], axis=1).reshape(-1)
    return I.IndexerCase(case.name + "_flat", case.q.reshape(B * Q, 32, 64), case.w.reshape(B * Q, 32),
                         case.key_pool, np.repeat(case.page_table, Q, axis=0), seq_j.astype(np.int32),
                         case.max_context, case.k)


def _to_dev(b, case):
    import torch
    q = torch.from_numpy(case.q.view("int16")).cuda().view(torch.bfloat16)
    w = torch.from_numpy(case.w).cuda()
    pool = torch.from_numpy(case.key_pool.view("int16")).cuda().view(torch.bfloat16)
    return q, w, pool, torch.from_numpy(case.page_table).cuda(), torch.from_numpy(case.seq_lens).cuda()


def _run_mtp(b, case):
    """mtp scores, mtp top-k on them, fused with rows, fused without rows (must agree)."""
    import torch
    q, w, pool, table, seq = _to_dev(b, case)
    B, Q = case.q.shape[0], case.q.shape[1]
    ws = torch.zeros(b.workspace_size_mtp(B, Q, case.max_context, case.k), dtype=torch.uint8, device="cuda")
    s = b.dsa_indexer_scores_mtp(q, w, pool, table, seq, case.max_context, workspace=ws)
    t = b.dsa_indexer_topk_mtp(s, seq, case.max_context, case.k, workspace=ws)
    s2 = torch.full_like(s, 7.0)
    t2 = b.dsa_indexer_fused_mtp(q, w, pool, table, seq, case.max_context, case.k, scores=s2, workspace=ws)
    t3 = b.dsa_indexer_fused_mtp(q, w, pool, table, seq, case.max_context, case.k, workspace=ws)
    torch.cuda.synchronize()
    assert b.get_error(ws) == 0
    out = [x.cpu().numpy() for x in (s, t, s2, t2, t3)]
    np.testing.assert_array_equal(out[0].view(np.uint32), out[2].view(np.uint32))
    np.testing.assert_array_equal(out[1], out[3])
    np.testing.assert_array_equal(out[1], out[4])
    return out[0], out[1]


@pytest.mark.parametrize("next_n", [2, 3, 4])
@pytest.mark.parametrize("name", ["b16_ctx8k_mixed", "b64_ctx128k_loguniform", "b64_ctx1m_seq512"])
def test_mtp_named_workloads(gpu_lib, oracle, name, next_n):
    case = I.with_next_n(I.workload(name), next_n)
    s, t = _run_mtp(gpu_lib, case)
    ref = oracle.case_scores_mtp(case)
    B = case.batch
    f = _flat(case)
    check_scores(f, s.reshape(B * next_n, -1), ref.reshape(B * next_n, -1))
    check_topk(f, t.reshape(B * next_n, -1), ref.reshape(B * next_n, -1), gpu_scores=s.reshape(B * next_n, -1))


def test_mtp_dense_128k_sampled_rows(gpu_lib, oracle):
    case = I.with_next_n(I.workload("b64_ctx128k_dense"), 2)
    s, t = _run_mtp(gpu_lib, case)
    rows = [0, 31, 63]
    sub = I.IndexerCase("dense_mtp_rows", case.q[rows], case.w[rows], case.key_pool, case.page_table[rows],
                        case.seq_lens[rows], case.max_context, case.k)
    ref = oracle.case_scores_mtp(sub)
    f = _flat(sub)
    check_scores(f, s[rows].reshape(6, -1), ref.reshape(6, -1))
    check_topk(f, t[rows].reshape(6, -1), ref.reshape(6, -1), gpu_scores=s[rows].reshape(6, -1))


def test_mtp_integer_inputs_bit_exact(gpu_lib, oracle):
    base = I.make_case(name="mtpint", batch=6, max_context=16384, seq_lens=[16384, 1, 2, 5, 4097, 9999],
                       num_pages=400, k=300, seed=91, key_dist="int")
    case = I.with_next_n(base, 3, dist="int")
    s, t = _run_mtp(gpu_lib, case)
    ref = oracle.case_scores_mtp(case)
    live = np.isfinite(ref)
    np.testing.assert_array_equal(s[live].astype(np.float64), ref[live])
    assert np.all(s[~live].view(np.uint32) == 0xFF800000)
    np.testing.assert_array_equal(t, oracle.topk_mtp(ref, case.seq_lens, case.max_context, case.k))


def test_mtp_ragged_short_lengths(gpu_lib, oracle):
    seqs = [0, 1, 2, 3, 4, 5, 6, 7, 255, 256, 257, 4096]
    base = I.make_case(name="mtprag", batch=len(seqs), max_context=4096, seq_lens=seqs, num_pages=200, k=7,
                       seed=93)
    case = I.with_next_n(base, 4)
    s, t = _run_mtp(gpu_lib, case)
    ref = oracle.case_scores_mtp(case)
    f = _flat(case)
    check_scores(f, s.reshape(len(seqs) * 4, -1), ref.reshape(len(seqs) * 4, -1))
    check_topk(f, t.reshape(len(seqs) * 4, -1), ref.reshape(len(seqs) * 4, -1),
               gpu_scores=s.reshape(len(seqs) * 4, -1))


def test_mtp_one_token_equals_single_token_path(gpu_lib):
    base = I.workload("b64_ctx128k_loguniform")
    case = I.with_next_n(base, 1)
    s, t = _run_mtp(gpu_lib, case)
    import torch
    q, w, pool, table, seq = gpu_lib.to_device(base)
    ws = gpu_lib.new_workspace(base.batch, base.max_context, base.k)
    s1 = gpu_lib.dsa_indexer_scores(q, w, pool, table, seq, base.max_context, workspace=ws)
    t1 = gpu_lib.dsa_indexer_topk(s1, seq, base.max_context, base.k, workspace=ws)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(s[:, 0].view(np.uint32), s1.cpu().numpy().view(np.uint32))
    np.testing.assert_array_equal(t[:, 0], t1.cpu().numpy())


def test_mtp_last_token_equals_single_token_scores(gpu_lib):
    """Token next_n - 1 carries the base case's query and full length: same scores as the
    single-token kernel up to fp32 summation order (the same order here: bit-identical)."""
    import torch
    base = I.workload("b16_ctx8k_mixed")
    case = I.with_next_n(base, 4)
    s, _ = _run_mtp(gpu_lib, case)
    q, w, pool, table, seq = gpu_lib.to_device(base)
    s1 = gpu_lib.dsa_indexer_scores(q, w, pool, table, seq, base.max_context)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(s[:, 3].view(np.uint32), s1.cpu().numpy().view(np.uint32))


def test_mtp_host_argument_checks(gpu_lib):
    import torch
    b = gpu_lib
    lib = b.load()
    case = I.with_next_n(I.make_case(name="mtpargs", batch=2, max_context=1024, seq_lens=[1024, 10],
                                     num_pages=8, k=16, seed=1), 2)
    q, w, pool, table, seq = _to_dev(b, case)
    scores = torch.empty((2, 2, 256), dtype=torch.float32, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    P = ctypes.c_void_p
    stream = P(torch.cuda.current_stream().cuda_stream)

    def call(next_n):
        return lib.dsa_indexer_scores_mtp(P(q.data_ptr()), P(w.data_ptr()), P(pool.data_ptr()), 8,
                                          P(table.data_ptr()), P(seq.data_ptr()), 2, next_n, 1024,
                                          P(scores.data_ptr()), P(ws.data_ptr()), 256, stream)
    assert call(2) == b.DSA_OK
    for bad in (0, 5, -1):
        assert call(bad) == b.DSA_ERR_INVALID_ARG
    assert lib.dsa_indexer_workspace_size_mtp(2, 5, 1024, 16) == 0
    torch.cuda.synchronize()
    assert b.get_error(ws) == 0
