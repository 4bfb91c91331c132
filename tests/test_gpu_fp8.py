"""GPU parity of the fp8 key-cache path against the fp64 oracle.

The cache stores each C4 key as 64 OCP e4m3 codes plus one positive fp32
scale (k = scale x e4m3(code)); the oracle decodes the codes by the e4m3
definition in fp64.  The kernel widens the codes to bf16 (exact) and applies
the scale after the head sum, so the only error is fp32 accumulation: the
same 3e-3 row-normwise bar as the bf16 path, and bit-exactness on integer
inputs.  Covers the named workloads, integer keys at scale 1 and 2, ragged
lengths and an odd table width, NaN codes outside the live range, bad page
ids, and the host argument checks of the two fp8 entry points.
"""
import ctypes

import numpy as np
import pytest

from sparse_attention_paged_dsa_gb300 import inputs as I

from _parity import check_scores, check_topk, own_topk

pytestmark = pytest.mark.gpu


def _run_fp8(b, case):
    """fp8 scores API, top-k API on it, fp8 fused with row, fp8 fused without row."""
    import torch
    q, w, _, table, seq = b.to_device(case)
    codes, scales = b.to_device_fp8(case)
    ws = b.new_workspace(case.batch, case.max_context, case.k)
    s = b.dsa_indexer_scores_fp8(q, w, codes, scales, table, seq, case.max_context, workspace=ws)
    t = b.dsa_indexer_topk(s, seq, case.max_context, case.k, workspace=ws)
    s2 = torch.full_like(s, 7.0)
    t2 = b.dsa_indexer_fused_fp8(q, w, codes, scales, table, seq, case.max_context, case.k, scores=s2,
                                 workspace=ws)
    t3 = b.dsa_indexer_fused_fp8(q, w, codes, scales, table, seq, case.max_context, case.k, workspace=ws)
    torch.cuda.synchronize()
    err = b.get_error(ws)
    out = [x.cpu().numpy() for x in (s, t, s2, t2, t3)]
    np.testing.assert_array_equal(out[0].view(np.uint32), out[2].view(np.uint32))
    np.testing.assert_array_equal(out[1], out[3])
    np.testing.assert_array_equal(out[1], out[4])
    return out[0], out[1], err


@pytest.mark.parametrize("name", ["b1_ctx8k_seq512", "b16_ctx8k_mixed", "b64_ctx128k_loguniform",
                                  "b64_ctx1m_seq512"])
def test_fp8_named_workload(gpu_lib, oracle, name):
    case = I.with_fp8_keys(I.workload(name))
    s, t, err = _run_fp8(gpu_lib, case)
    assert err == 0
    ref = oracle.case_scores_fp8(case)
    stats = check_scores(case, s, ref)
    check_topk(case, t, ref, gpu_scores=s)
    print(name, "fp8 max rel err", max(r for r, _ in stats))


def test_fp8_dense_128k_sampled_rows(gpu_lib, oracle):
    case = I.with_fp8_keys(I.workload("b64_ctx128k_dense"))
    s, t, err = _run_fp8(gpu_lib, case)
    assert err == 0
    rows = [0, 29, 63]
    sub = I.IndexerCase("dense_fp8_rows", case.q[rows], case.w[rows], case.key_pool, case.page_table[rows],
                        case.seq_lens[rows], case.max_context, case.k, key_codes=case.key_codes,
                        key_scales=case.key_scales)
    ref = oracle.case_scores_fp8(sub)
    check_scores(sub, s[rows], ref)
    check_topk(sub, t[rows], ref, gpu_scores=s[rows])
    assert np.all(np.isfinite(s))
    for b in range(case.batch):
        np.testing.assert_array_equal(t[b], own_topk(s[b], 32768, case.k))


@pytest.mark.parametrize("scale", [1.0, 2.0, 0.25])
def test_fp8_integer_keys_bit_exact(gpu_lib, oracle, scale):
    """Integer keys in [-4, 4] stored as e4m3(k / scale) with a power-of-two scale are exact,
    so every partial sum is exact in fp32 and the scores equal the oracle's bit for bit."""
    base = I.make_case(name="int8", batch=6, max_context=16384, seq_lens=[16384, 1, 5, 4097, 12345, 300],
                       num_pages=400, k=600, seed=78, key_dist="int")
    k = I.bf16_bits_to_f32(base.key_pool).astype(np.float64)
    codes = I.f32_to_e4m3_codes(k / scale)
    case = I.IndexerCase("int8", base.q, base.w, base.key_pool, base.page_table, base.seq_lens, base.max_context,
                         base.k, key_codes=codes, key_scales=np.full(codes.shape[:2], scale, np.float32))
    s, t, err = _run_fp8(gpu_lib, case)
    assert err == 0
    ref = oracle.case_scores_fp8(case)
    np.testing.assert_array_equal(ref, oracle.case_scores(base))  # the fp8 cache holds these keys exactly
    live = np.isfinite(ref)
    np.testing.assert_array_equal(s[live].astype(np.float64), ref[live])
    assert np.all(s[~live].view(np.uint32) == 0xFF800000)
    np.testing.assert_array_equal(t, oracle.topk(ref, case.seq_lens, case.max_context, case.k))


@pytest.mark.parametrize("k", [1, 300, 2048])
def test_fp8_ragged_lengths_and_k(gpu_lib, oracle, k):
    seqs = [0, 1, 3, 4, 5, 255, 256, 257, 1023, 8192, 512, 7777]
    case = I.with_fp8_keys(I.make_case(name="ragged8", batch=len(seqs), max_context=8192, seq_lens=seqs,
                                       num_pages=300, k=k, seed=50 + k))
    s, t, err = _run_fp8(gpu_lib, case)
    assert err == 0
    ref = oracle.case_scores_fp8(case)
    check_scores(case, s, ref)
    check_topk(case, t, ref, gpu_scores=s)


def test_fp8_odd_table_width_and_shared_pages(gpu_lib, oracle):
    case = I.with_fp8_keys(I.make_case(name="odd8", batch=4, max_context=33 * 256,
                                       seq_lens=[33 * 256, 33 * 256 - 3, 32 * 256 + 1, 77], num_pages=40, k=500,
                                       seed=12, page_reuse=True))
    s, t, err = _run_fp8(gpu_lib, case)
    assert err == 0
    ref = oracle.case_scores_fp8(case)
    check_scores(case, s, ref)
    check_topk(case, t, ref, gpu_scores=s)


def test_fp8_nan_codes_outside_live_range_do_not_leak(gpu_lib):
    """Entries past each row's live length and pages no row reads hold e4m3 NaN codes (0x7F)
    and NaN scales: the scores stay bit-identical to the clean cache."""
    case = I.with_fp8_keys(I.make_case(name="nan8", batch=5, max_context=16384,
                                       seq_lens=[16384, 1, 4099, 9001, 250], num_pages=400, k=128, seed=31))
    s0, t0, _ = _run_fp8(gpu_lib, case)
    codes = case.key_codes.copy()
    scales = case.key_scales.copy()
    used = np.zeros((case.num_pages, 64), bool)
    for b, n in enumerate(case.live_positions()):
        for t in range(int(n)):
            used[case.page_table[b, t // 64], t % 64] = True
    codes[~used] = 0x7F
    scales[~used] = np.float32(np.nan)
    dirty = I.IndexerCase("nan8d", case.q, case.w, case.key_pool, case.page_table, case.seq_lens,
                          case.max_context, case.k, key_codes=codes, key_scales=scales)
    s1, t1, err = _run_fp8(gpu_lib, dirty)
    assert err == 0
    np.testing.assert_array_equal(s0.view(np.uint32), s1.view(np.uint32))
    np.testing.assert_array_equal(t0, t1)


def test_fp8_bad_page_scores_neg_inf_and_sets_bit(gpu_lib, oracle):
    case = I.with_fp8_keys(I.make_case(name="bad8", batch=3, max_context=4096, seq_lens=[4096, 700, 300],
                                       num_pages=40, k=64, seed=41))
    table = case.page_table.copy()
    table[0, 3] = case.num_pages + 5
    table[1, 0] = -7
    bad = I.IndexerCase("bad8", case.q, case.w, case.key_pool, table, case.seq_lens, case.max_context, case.k,
                        key_codes=case.key_codes, key_scales=case.key_scales)
    s, t, err = _run_fp8(gpu_lib, bad)
    assert err & gpu_lib.DEVERR_BAD_PAGE
    ref = oracle.case_scores_fp8(case)
    assert np.all(np.isneginf(s[0, 192:256])) and np.all(np.isneginf(s[1, 0:64]))
    keep = np.ones_like(s, bool)
    keep[0, 192:256] = False
    keep[1, 0:64] = False
    live = np.isfinite(ref) & keep
    err_rel = np.abs(s[live] - ref[live]).max() / np.abs(ref[live]).max()
    assert err_rel <= 3e-3


def test_fp8_host_argument_checks(gpu_lib):
    import torch
    b = gpu_lib
    lib = b.load()
    case = I.with_fp8_keys(I.make_case(name="args8", batch=2, max_context=1024, seq_lens=[1024, 10], num_pages=8,
                                       k=16, seed=1))
    q, w, _, table, seq = b.to_device(case)
    codes, scales = b.to_device_fp8(case)
    scores = torch.empty((2, 256), dtype=torch.float32, device="cuda")
    topk = torch.empty((2, 16), dtype=torch.int32, device="cuda")
    ws = b.new_workspace(2, 1024, 16)
    P = ctypes.c_void_p
    stream = P(torch.cuda.current_stream().cuda_stream)

    def call(fused=False, **kw):
        a = dict(codes=P(codes.data_ptr()), scales=P(scales.data_ptr()), out=P(scores.data_ptr()),
                 ws=P(ws.data_ptr()), wsb=ws.numel(), ctx=1024, k=16, np_=8)
        a.update(kw)
        if fused:
            return lib.dsa_indexer_fused_fp8(P(q.data_ptr()), P(w.data_ptr()), a["codes"], a["scales"], a["np_"],
                                             P(table.data_ptr()), P(seq.data_ptr()), 2, a["ctx"], a["k"],
                                             P(topk.data_ptr()), None, a["ws"], a["wsb"], stream)
        return lib.dsa_indexer_scores_fp8(P(q.data_ptr()), P(w.data_ptr()), a["codes"], a["scales"], a["np_"],
                                          P(table.data_ptr()), P(seq.data_ptr()), 2, a["ctx"], a["out"], a["ws"],
                                          a["wsb"], stream)

    assert call() == b.DSA_OK
    assert call(fused=True) == b.DSA_OK
    torch.cuda.synchronize()
    sentinel = scores.clone()
    assert call(codes=None) == b.DSA_ERR_INVALID_ARG
    assert call(scales=None) == b.DSA_ERR_INVALID_ARG
    assert call(codes=P(codes.data_ptr() + 8)) == b.DSA_ERR_INVALID_ARG
    assert call(scales=P(scales.data_ptr() + 4)) == b.DSA_ERR_INVALID_ARG
    assert call(np_=0) == b.DSA_ERR_INVALID_ARG
    assert call(ctx=1000) == b.DSA_ERR_INVALID_ARG
    assert call(ws=None) == b.DSA_ERR_WORKSPACE
    assert call(fused=True, k=0) == b.DSA_ERR_INVALID_ARG
    assert call(fused=True, wsb=256) == b.DSA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.equal(scores.view(torch.int32), sentinel.view(torch.int32))
    assert b.get_error(ws) == 0


def test_fp8_query_dynamic_range(gpu_lib, oracle):
    """The kernel feeds the fp8 MMA a query split into two e4m3 terms under a per-head
    power-of-two scale.  Queries whose heads differ in magnitude by 2^+-12, whose elements span
    2^20 within a head, whose rows sit at 2^+-60, that hold bf16 subnormals, or whose heads are all
    zero must still meet the score tolerance against the oracle."""
    rng = np.random.default_rng(7)
    base = I.with_fp8_keys(I.make_case(name="qrange", batch=6, max_context=4096,
                                       seq_lens=[4096, 4000, 3000, 2048, 1500, 777], num_pages=120, k=64,
                                       seed=17))
    q = I.bf16_bits_to_f32(base.q).astype(np.float64)
    q[0] *= 2.0 ** rng.integers(-12, 13, size=(32, 1))                 # heads 2^-12 .. 2^12 apart
    q[1] *= np.where(rng.random((32, 64)) < 0.5, 2.0 ** -20, 1.0)      # elements 2^20 apart in a head
    q[2] *= 2.0 ** 60
    q[3] *= 2.0 ** -60
    q[4, ::2] = 0.0                                                     # every other head all zero
    q5 = (rng.integers(1, 0x80, size=(32, 64)) * rng.choice([-1, 1], size=(32, 64))).astype(np.int64)
    q5_bits = np.where(q5 < 0, 0x8000 | (-q5), q5).astype(np.uint16)  # bf16 subnormals
    q5_bits[:, :8] = I.f32_to_bf16_bits(rng.standard_normal((32, 8)).astype(np.float32) * 2.0 ** -125)
    qb = I.f32_to_bf16_bits(q.astype(np.float32))
    qb[5] = q5_bits
    case = I.IndexerCase("qrange", qb, base.w, base.key_pool, base.page_table, base.seq_lens, base.max_context,
                         base.k, key_codes=base.key_codes, key_scales=base.key_scales)
    s, t, err = _run_fp8(gpu_lib, case)
    assert err == 0
    ref = oracle.case_scores_fp8(case)
    rows = [0, 1, 2, 3, 4]  # row 5's scores are below the fp32 normal range: checked for sign/finiteness
    sub = I.IndexerCase("qrange_rows", qb[rows], base.w[rows], base.key_pool, base.page_table[rows],
                        base.seq_lens[rows], base.max_context, base.k)
    check_scores(sub, s[rows], ref[rows])
    n5 = int(case.live_positions()[5])
    assert np.all(np.isfinite(s[5, :n5])) and np.all(np.isneginf(s[5, n5:]))
    np.testing.assert_allclose(s[5, :n5], ref[5, :n5], rtol=0, atol=float(np.abs(ref[5, :n5]).max()) * 3e-3 + 1e-44)


def test_fp8_many_short_requests(gpu_lib, oracle):
    """Every CTA of the persistent grid starts several requests (1024 requests of one to three
    units each), so the query-split ring turns over at nearly every unit; each request's query
    sits at its own power-of-two magnitude (2^-40 .. 2^40) with some heads all zero, so a split
    that used another request's scale or tile would miss the tolerance by orders of magnitude."""
    rng = np.random.default_rng(21)
    B = 1024
    seq = rng.integers(1, 1537, size=B)                      # up to 384 C4 positions: 1 to 3 units
    seq[::97] = 0                                            # a few empty requests
    base = I.with_fp8_keys(I.make_case(name="short_many", batch=B, max_context=2048, seq_lens=seq,
                                       num_pages=B * 8 + 16, k=16, seed=23))
    q = I.bf16_bits_to_f32(base.q).astype(np.float64)
    q *= (2.0 ** rng.integers(-40, 41, size=B))[:, None, None]
    q[rng.random(B) < 0.2, ::3] = 0.0                        # some requests with every third head zero
    case = I.IndexerCase("short_many", I.f32_to_bf16_bits(q.astype(np.float32)), base.w, base.key_pool,
                         base.page_table, base.seq_lens, base.max_context, base.k,
                         key_codes=base.key_codes, key_scales=base.key_scales)
    s, t, err = _run_fp8(gpu_lib, case)
    assert err == 0
    ref = oracle.case_scores_fp8(case)
    check_scores(case, s, ref)
    check_topk(case, t, ref, gpu_scores=s)
