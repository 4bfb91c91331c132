"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Covers the five named workloads (full size; the dense 128K one is checked on
sampled rows by the oracle and on every row by properties), plus exact-integer
inputs (bit-exact), ragged tails, odd table widths, long rows past the top-k
shared-memory cache, shared pages, page-permutation and dead-entry
invariance, and agreement of the three entry points.
"""
import numpy as np
import pytest

from sparse_attention_paged_dsa_gb300 import inputs as I

from _parity import check_scores, check_topk, own_topk

pytestmark = pytest.mark.gpu


def _run_all(b, case):
    """scores API, top-k API on it, fused with row, fused without row."""
    import torch
    q, w, pool, table, seq = b.to_device(case)
    ws = b.new_workspace(case.batch, case.max_context, case.k)
    s = b.dsa_indexer_scores(q, w, pool, table, seq, case.max_context, workspace=ws)
    t = b.dsa_indexer_topk(s, seq, case.max_context, case.k, workspace=ws)
    s2 = torch.full_like(s, 7.0)
    t2 = b.dsa_indexer_fused(q, w, pool, table, seq, case.max_context, case.k, scores=s2, workspace=ws)
    t3 = b.dsa_indexer_fused(q, w, pool, table, seq, case.max_context, case.k, workspace=ws)
    torch.cuda.synchronize()
    assert b.get_error(ws) == 0
    out = [x.cpu().numpy() for x in (s, t, s2, t2, t3)]
    np.testing.assert_array_equal(out[0].view(np.uint32), out[2].view(np.uint32))
    np.testing.assert_array_equal(out[1], out[3])
    np.testing.assert_array_equal(out[1], out[4])
    return out[0], out[1]


@pytest.mark.parametrize("name", ["b1_ctx8k_seq512", "b16_ctx8k_mixed", "b64_ctx128k_loguniform",
                                  "b64_ctx1m_seq512"])
def test_named_workload_full(gpu_lib, oracle, name):
    case = I.workload(name)
    s, t = _run_all(gpu_lib, case)
    ref = oracle.case_scores(case)
    stats = check_scores(case, s, ref)
    check_topk(case, t, ref, gpu_scores=s)
    print(name, "max rel err", max(r for r, _ in stats))


def test_dense_128k_sampled_rows(gpu_lib, oracle):
    case = I.workload("b64_ctx128k_dense")
    s, t = _run_all(gpu_lib, case)
    rows = [0, 17, 40, 63]
    sub = I.IndexerCase("dense_rows", case.q[rows], case.w[rows], case.key_pool, case.page_table[rows],
                        case.seq_lens[rows], case.max_context, case.k)
    ref = oracle.case_scores(sub)
    check_scores(sub, s[rows], ref)
    check_topk(sub, t[rows], ref, gpu_scores=s[rows])
    # every row: all live, finite, and the top-k is exact on its own scores
    assert np.all(np.isfinite(s))
    for b in range(case.batch):
        np.testing.assert_array_equal(t[b], own_topk(s[b], 32768, case.k))


def test_dense_128k_literal_shared_pool(gpu_lib, oracle):
    """8192-page pool shared by all rows (each page referenced by 4 rows)."""
    case = I.workload("b64_ctx128k_dense", literal_pool=True)
    s, t = _run_all(gpu_lib, case)
    rows = [3, 33]
    sub = I.IndexerCase("lit_rows", case.q[rows], case.w[rows], case.key_pool, case.page_table[rows],
                        case.seq_lens[rows], case.max_context, case.k)
    ref = oracle.case_scores(sub)
    check_scores(sub, s[rows], ref)
    check_topk(sub, t[rows], ref, gpu_scores=s[rows])


def test_exact_integer_inputs_bit_exact(gpu_lib, oracle):
    """Integer q, k in [-4, 4] and w = +-2^-j: every partial sum is exact in fp32."""
    case = I.make_case(name="int", batch=8, max_context=16384,
                       seq_lens=[16384, 1, 5, 300, 4097, 8000, 12345, 9999], num_pages=512, k=700,
                       seed=77, key_dist="int")
    s, t = _run_all(gpu_lib, case)
    ref = oracle.case_scores(case)
    live = np.isfinite(ref)
    np.testing.assert_array_equal(s[live].astype(np.float64), ref[live])
    assert np.all(np.isneginf(s[~live]))
    np.testing.assert_array_equal(t, oracle.topk(ref, case.seq_lens, case.max_context, case.k))


@pytest.mark.parametrize("k", [1, 64, 300, 2048])
def test_ragged_lengths_and_k(gpu_lib, oracle, k):
    seqs = [0, 1, 3, 4, 5, 255, 256, 257, 1023, 8192, 512, 7777]
    case = I.make_case(name="ragged", batch=len(seqs), max_context=8192, seq_lens=seqs, num_pages=300,
                       k=k, seed=5 + k)
    s, t = _run_all(gpu_lib, case)
    ref = oracle.case_scores(case)
    check_scores(case, s, ref)
    check_topk(case, t, ref, gpu_scores=s)


def test_k_equals_row_width(gpu_lib, oracle):
    case = I.make_case(name="kmax", batch=3, max_context=4096, seq_lens=[4096, 100, 0], num_pages=40,
                       k=1024, seed=9)
    s, t = _run_all(gpu_lib, case)
    ref = oracle.case_scores(case)
    check_scores(case, s, ref)
    check_topk(case, t, ref, gpu_scores=s)


def test_odd_table_width(gpu_lib, oracle):
    """max_context = 33 pages: the last work unit of a full row is half outside the row."""
    case = I.make_case(name="odd", batch=4, max_context=33 * 256, seq_lens=[33 * 256, 33 * 256 - 3, 32 * 256 + 1, 77],
                       num_pages=200, k=500, seed=11)
    s, t = _run_all(gpu_lib, case)
    ref = oracle.case_scores(case)
    check_scores(case, s, ref)
    check_topk(case, t, ref, gpu_scores=s)


def test_long_rows_beyond_topk_cache(gpu_lib, oracle):
    """65536 live positions per row: the top-k re-reads scores from global memory."""
    case = I.make_case(name="long", batch=2, max_context=262144, seq_lens=[262144, 200001], num_pages=2048,
                       k=2048, seed=13)
    s, t = _run_all(gpu_lib, case)
    ref = oracle.case_scores(case)
    check_scores(case, s, ref)
    check_topk(case, t, ref, gpu_scores=s)


def test_dead_entries_and_page_permutation_bit_identical(gpu_lib):
    base = I.make_case(name="inv", batch=6, max_context=32768, seq_lens=[32768, 1, 9000, 20000, 257, 4],
                       num_pages=700, k=256, seed=21)
    rnd = I.make_case(name="inv", batch=6, max_context=32768, seq_lens=[32768, 1, 9000, 20000, 257, 4],
                      num_pages=700, k=256, seed=21, dead_fill="random")
    s0, t0 = _run_all(gpu_lib, base)
    s1, t1 = _run_all(gpu_lib, rnd)
    np.testing.assert_array_equal(s0.view(np.uint32), s1.view(np.uint32))
    np.testing.assert_array_equal(t0, t1)
    perm = np.random.default_rng(3).permutation(base.num_pages)
    pool2 = np.empty_like(base.key_pool)
    pool2[perm] = base.key_pool
    table2 = np.where(base.page_table >= 0, perm[np.maximum(base.page_table, 0)], -1).astype(np.int32)
    moved = I.IndexerCase("perm", base.q, base.w, pool2, table2, base.seq_lens, base.max_context, base.k)
    s2, t2 = _run_all(gpu_lib, moved)
    np.testing.assert_array_equal(s0.view(np.uint32), s2.view(np.uint32))
    np.testing.assert_array_equal(t0, t2)


def test_shared_pages_across_rows(gpu_lib, oracle):
    case = I.make_case(name="shared", batch=5, max_context=16384, seq_lens=[16384] * 5, num_pages=70, k=333,
                       seed=23, page_reuse=True)
    s, t = _run_all(gpu_lib, case)
    ref = oracle.case_scores(case)
    check_scores(case, s, ref)
    check_topk(case, t, ref, gpu_scores=s)


def test_repeat_runs_bitwise_deterministic(gpu_lib):
    case = I.workload("b64_ctx128k_loguniform")
    s0, t0 = _run_all(gpu_lib, case)
    s1, t1 = _run_all(gpu_lib, case)
    np.testing.assert_array_equal(s0.view(np.uint32), s1.view(np.uint32))
    np.testing.assert_array_equal(t0, t1)


def _topk_on_rows(b, rows, n_live, k):
    """The top-k entry point on crafted fp32 rows (row width = rows.shape[1])."""
    import torch
    B, M = rows.shape
    s = torch.from_numpy(np.ascontiguousarray(rows, dtype=np.float32)).cuda()
    seq = torch.from_numpy((np.asarray(n_live, dtype=np.int64) * 4).astype(np.int32)).cuda()
    t = b.dsa_indexer_topk(s, seq, 4 * M, k)
    torch.cuda.synchronize()
    return t.cpu().numpy()


def test_topk_rows_at_the_sample_edges(gpu_lib, oracle):
    """The sampled top-k takes its threshold from a sixteenth of the row's scores, the four at
    positions 64 g .. 64 g + 3 of every group g.  Rows just past k (the sample cannot bound the
    k-th key: every key a candidate), rows of a few thousand keys, and a full row whose sampled
    keys are 8x the others (the sampled keys are the row's
    extremes, so too few keys pass and the exact path runs): the fused and unfused results
    must agree with each other and with the oracle's."""
    k = 2048
    n_rows = [32768, k + 1, k + 13, 2600, 2900, 3100, 4500]
    case = I.make_case(name="edges", batch=len(n_rows), max_context=131072, seq_lens=[4 * n for n in n_rows],
                       num_pages=800, k=k, seed=31)
    vals = I.bf16_bits_to_f32(case.key_pool)
    t = np.arange(0, 32768)
    t = t[t % 64 < 4]                                              # the sampled positions
    vals[case.page_table[0, t // 64], t % 64] *= np.float32(8.0)  # exact in bf16
    case.key_pool = I.f32_to_bf16_bits(vals)
    s, tk = _run_all(gpu_lib, case)
    ref = oracle.case_scores(case)
    check_scores(case, s, ref)
    check_topk(case, tk, ref, gpu_scores=s)


def test_topk_rows_that_defeat_the_sample(gpu_lib, oracle):
    """Rows where the sampled positions score high (too few keys pass the sampled threshold),
    where every 4th position does, rows with all scores equal (too many pass), heavy ties, and ragged live lengths: every
    path of the top-k kernel must give the exact top-k (ties to the lower position)."""
    rng = np.random.default_rng(99)
    M, k = 32768, 2048
    rows, n_live = [], []
    r = rng.standard_normal(M).astype(np.float32)
    r[0::4] += 100.0
    rows.append(r); n_live.append(M)                       # a quarter of the row (and of the sample) high
    r = rng.standard_normal(M).astype(np.float32)
    r[np.arange(M) % 64 < 4] += 100.0
    rows.append(r); n_live.append(M)                       # samples all high: fallback (too few)
    rows.append(np.full(M, 1.5, np.float32)); n_live.append(M)   # one value: fallback (too many)
    rows.append(np.floor(rng.standard_normal(M) * 3).astype(np.float32)); n_live.append(M)  # ties
    r = rng.standard_normal(M).astype(np.float32)
    rows.append(r); n_live.append(30001)                   # ragged, n % 4 == 1
    r = rng.standard_normal(M).astype(np.float32)
    r[:8] = 50.0
    rows.append(r); n_live.append(2051)                    # barely more than k
    r = -np.abs(rng.standard_normal(M)).astype(np.float32)
    r[::7] = -0.0
    rows.append(r); n_live.append(M)                       # negative scores and (only negative) zeros
    rows = np.stack(rows)
    got = _topk_on_rows(gpu_lib, rows, n_live, k)
    for i, n in enumerate(n_live):
        ref = oracle.topk_row(rows[i].astype(np.float64), n, k)
        np.testing.assert_array_equal(got[i], ref, err_msg=f"row {i}")


def test_topk_infinite_scores(gpu_lib, oracle):
    """Rows holding +inf and -inf scores (a caller's row through dsa_indexer_topk): more +inf
    keys than k (the threshold sits at +inf and ties resolve to the lower positions), a few +inf
    among many -inf, and a row whose k-th largest score is -inf."""
    rng = np.random.default_rng(4321)
    M, k = 32768, 2048
    rows, n_live = [], []
    r = rng.standard_normal(M).astype(np.float32)
    r[rng.choice(M, 3000, replace=False)] = np.inf
    rows.append(r); n_live.append(M)
    r = rng.standard_normal(M).astype(np.float32)
    r[rng.choice(M, 20000, replace=False)] = -np.inf
    r[rng.choice(M, 100, replace=False)] = np.inf
    rows.append(r); n_live.append(M)
    r = np.full(M, -np.inf, np.float32)
    r[rng.choice(M, 1000, replace=False)] = rng.standard_normal(1000).astype(np.float32)
    rows.append(r); n_live.append(M)
    r = rng.standard_normal(M).astype(np.float32)
    r[rng.choice(29999, 2500, replace=False)] = np.inf
    rows.append(r); n_live.append(29999)                    # ragged tail
    rows = np.stack(rows)
    got = _topk_on_rows(gpu_lib, rows, n_live, k)
    for i, n in enumerate(n_live):
        ref = oracle.topk_row(rows[i].astype(np.float64), n, k)
        np.testing.assert_array_equal(got[i], ref, err_msg=f"row {i}")


@pytest.mark.parametrize("k", [1, 7, 100, 1000, 4096])
def test_topk_sample_rule_across_k(gpu_lib, oracle, k):
    """The sampled path's threshold rank depends on k and n: rows from a few hundred keys to a full
    32768-key row, continuous and heavily tied scores, for k from 1 to 4096."""
    rng = np.random.default_rng(500 + k)
    M = 32768
    n_live = [300, 1000, 2600, 5000, 20000, 32768, 32768]
    rows = rng.standard_normal((len(n_live), M)).astype(np.float32)
    rows[-1] = np.floor(rows[-1] * 2.0)                     # a handful of distinct values
    got = _topk_on_rows(gpu_lib, rows, n_live, k)
    for i, n in enumerate(n_live):
        ref = oracle.topk_row(rows[i].astype(np.float64), n, k)
        np.testing.assert_array_equal(got[i], ref, err_msg=f"row {i} (n = {n})")


def _topk_by_bits(row, n, k):
    """The contract's order written out on the bits: -0 taken as +0, then a float's sign-magnitude
    bits mapped to an unsigned key that rises with the value and extends it to NaNs (positive NaNs
    above +inf, negative ones below -inf); the k largest keys, equal keys to the lower position,
    listed in ascending position and padded with -1."""
    u = row[:n].view(np.uint32).astype(np.uint64)
    u = np.where(u == 0x80000000, 0, u)
    key = np.where(u & 0x80000000, (~u) & 0xFFFFFFFF, u | 0x80000000)
    order = np.lexsort((np.arange(n), -key.astype(np.int64)))[: min(k, n)]
    out = np.full(k, -1, np.int32)
    out[: order.size] = np.sort(order)
    return out


def test_topk_nan_scores(gpu_lib, oracle):
    """NaN scores in a caller's row rank by their bits (positive NaNs above +inf, negative ones
    below -inf, payloads in bit order), on the sampled path, its fallback and the short-row path."""
    rng = np.random.default_rng(77)
    M, k = 32768, 2048
    pos_nan = (0x7FC00000 + rng.integers(0, 1 << 20, 400)).astype(np.uint32).view(np.float32)
    neg_nan = (0xFFC00000 + rng.integers(0, 1 << 20, 400)).astype(np.uint32).view(np.float32)
    rows, n_live = [], []
    r = rng.standard_normal(M).astype(np.float32)
    r[rng.choice(M, 400, replace=False)] = pos_nan          # a few hundred NaNs above everything
    r[rng.choice(M, 50, replace=False)] = np.inf
    rows.append(r); n_live.append(M)
    r = rng.standard_normal(M).astype(np.float32)
    r[rng.choice(M, 400, replace=False)] = neg_nan          # NaNs below everything: never taken
    rows.append(r); n_live.append(M)
    r = np.full(M, np.float32(1.0))
    r[rng.choice(M, 3000, replace=False)] = pos_nan[rng.integers(0, 400, 3000)]  # more NaNs than k
    rows.append(r); n_live.append(M)
    r = rng.standard_normal(M).astype(np.float32)
    r[np.arange(M) % 64 < 4] = pos_nan[rng.integers(0, 400, M // 16)]  # every sampled key a NaN
    rows.append(r); n_live.append(30001)
    rows = np.stack(rows)
    got = _topk_on_rows(gpu_lib, rows, n_live, k)
    for i, n in enumerate(n_live):
        np.testing.assert_array_equal(got[i], _topk_by_bits(rows[i], n, k), err_msg=f"row {i}")
    # the rule agrees with the oracle on rows without NaN
    plain = rng.standard_normal(M).astype(np.float32)
    np.testing.assert_array_equal(_topk_by_bits(plain, M, k), oracle.topk_row(plain.astype(np.float64), M, k))
    short = rng.standard_normal((1, 256)).astype(np.float32)
    short[0, rng.choice(200, 30, replace=False)] = pos_nan[:30]
    short[0, rng.choice(200, 30, replace=False)] = neg_nan[:30]
    got = _topk_on_rows(gpu_lib, short, [200], 50)
    np.testing.assert_array_equal(got[0], _topk_by_bits(short[0], 200, 50))


def _signed_zero_rows(rng, M):
    """Rows whose k-th largest score is 0 and that hold both +0 and -0 (equal in fp32 order,
    so they tie and go to the lower position whatever their sign)."""
    rows, n_live = [], []
    zeros = np.sort(rng.choice(M, 3000, replace=False))    # more zeros than k: k cuts the zero band
    for first in (-0.0, 0.0):                               # both sign orders along the positions
        r = -np.abs(rng.standard_normal(M)).astype(np.float32) - 0.5
        if first == 0.0:
            signs = np.where(np.arange(zeros.size) % 2 == 0, np.float32(0.0), np.float32(-0.0))
        else:
            signs = np.where(np.arange(zeros.size) % 2 == 0, np.float32(-0.0), np.float32(0.0))
        r[zeros] = signs
        rows.append(r); n_live.append(M)
    r = np.where(rng.random(M) < 0.5, np.float32(-0.0), np.float32(0.0)).astype(np.float32)
    rows.append(r); n_live.append(M)                        # every score a signed zero
    r = -np.abs(rng.standard_normal(M)).astype(np.float32) - 0.5
    r[zeros[:1500]] = np.float32(-0.0)
    r[zeros[1500:]] = np.float32(0.0)                       # every -0 before every +0
    r[:40] = 3.0
    rows.append(r); n_live.append(M)
    return np.stack(rows), n_live


def test_topk_signed_zeros_tie(gpu_lib, oracle):
    """+0 and -0 are equal scores: the top-k takes the lower positions among them, as the oracle
    (which ranks in fp64, where -0 == +0) does, through the single-token and multi-token entry points."""
    import torch
    rng = np.random.default_rng(1234)
    M, k = 32768, 2048
    rows, n_live = _signed_zero_rows(rng, M)
    assert np.signbit(rows[0][rows[0] == 0]).any() and (~np.signbit(rows[0][rows[0] == 0])).any()
    got = _topk_on_rows(gpu_lib, rows, n_live, k)
    for i, n in enumerate(n_live):
        ref = oracle.topk_row(rows[i].astype(np.float64), n, k)
        np.testing.assert_array_equal(got[i], ref, err_msg=f"row {i}")
    # a short row (k < n <= 256: ranked by direct comparison) of mixed zeros
    short = np.full((1, 256), -1.0, np.float32)
    short[0, :200] = np.where(rng.random(200) < 0.5, np.float32(-0.0), np.float32(0.0))
    short[0, 7] = 1.0
    got = _topk_on_rows(gpu_lib, short, [230], 50)
    np.testing.assert_array_equal(got[0], oracle.topk_row(short[0].astype(np.float64), 230, 50))
    # the same rows through the multi-token entry point: two tokens per request, token j of
    # request b is row 2b + j (both tokens see the whole row: seq_len = 4M gives n = M for both)
    B2 = (rows.shape[0] + 1) // 2
    pad = np.concatenate([rows, rows[:1]]) if rows.shape[0] % 2 else rows
    s = torch.from_numpy(np.ascontiguousarray(pad.reshape(B2, 2, M), dtype=np.float32)).cuda()
    seq = torch.full((B2,), 4 * M, dtype=torch.int32, device="cuda")
    t = gpu_lib.dsa_indexer_topk_mtp(s, seq, 4 * M, k)
    torch.cuda.synchronize()
    t = t.cpu().numpy().reshape(-1, k)
    for i in range(rows.shape[0]):
        ref = oracle.topk_row(pad[i].astype(np.float64), M, k)
        np.testing.assert_array_equal(t[i], ref, err_msg=f"multi-token row {i}")


def test_many_short_requests(gpu_lib, oracle):
    """1024 requests of one to three units each: every CTA of the persistent grid starts several
    requests, so the query-tile ring and the epilogue's head weights turn over at nearly every
    unit; each request's query sits at its own power-of-two magnitude (2^-40 .. 2^40), so a unit
    scored with another request's query or weights would miss the tolerance by orders of magnitude."""
    rng = np.random.default_rng(22)
    B = 1024
    seq = rng.integers(1, 1537, size=B)
    seq[::89] = 0
    base = I.make_case(name="short_many_bf16", batch=B, max_context=2048, seq_lens=seq, num_pages=B * 8 + 16,
                       k=16, seed=24)
    q = I.bf16_bits_to_f32(base.q).astype(np.float64) * (2.0 ** rng.integers(-40, 41, size=B))[:, None, None]
    case = I.IndexerCase("short_many_bf16", I.f32_to_bf16_bits(q.astype(np.float32)), base.w, base.key_pool,
                         base.page_table, base.seq_lens, base.max_context, base.k)
    s, t = _run_all(gpu_lib, case)
    ref = oracle.case_scores(case)
    check_scores(case, s, ref)
    check_topk(case, t, ref, gpu_scores=s)
