"""GPU parity of the sparse multi-head latent attention decode (row f1) against the fp64 oracle.

Tolerance from the arithmetic.  Scores are exact bf16 products summed in fp32; the softmax
weights reach the tensor cores as bf16 (and the row sum adds the same rounded values), so each
normalised weight is within 2^-8 of its exact value, relatively:
    |o - o_ref| <= 2^-8 * sum_t w_t |v_t| = 2^-8 * o_abs   (o_abs from the oracle)
plus fp32 accumulation far below that; the test allows twice the bound, 2^-7 * o_abs + 1e-6.
lse: the row sum of rounded weights is within 2^-9 relatively, so |lse - lse_ref| <= 2^-8 +
1e-5 |lse|.  Cases: one block; many requests with ragged top-k rows split across CTAs and
merged; holes, duplicates, positions past the live length and empty rows; the running-max
rescale (late blocks dominate); the indexer's own top-k rows on a mixed-length workload; the
full 64-request, 128K-context workload sampled; more requests than SMs and the maximum batch
(one split each, several waves); a zero scale (the plain mean); determinism; host argument checks."""
import numpy as np
import pytest

from sparse_attention_paged_dsa_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _dev(mc):
    import torch
    t16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view("int16")).cuda().view(torch.bfloat16)
    return (t16(mc.q), t16(mc.kv), torch.from_numpy(mc.page_table).cuda(), torch.from_numpy(mc.seq_lens).cuda(),
            torch.from_numpy(mc.topk).cuda())


def _run(b, mc):
    import torch
    q, kv, table, seq, topk = _dev(mc)
    ws = torch.zeros(b.sparse_mla_workspace_size(mc.batch, mc.topk.shape[1]), dtype=torch.uint8, device="cuda")
    o, lse = b.dsa_sparse_mla_decode(q, kv, table, seq, mc.max_context, topk, mc.sm_scale, workspace=ws)
    torch.cuda.synchronize()
    assert b.get_error(ws) == 0
    return o.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def _check(o, lse, mc, oracle, rows=None):
    rows = range(mc.batch) if rows is None else rows
    for b in rows:
        sub = lambda a: a[b:b + 1]
        o_ref, lse_ref, o_abs = oracle.sparse_mla_decode(sub(mc.q), mc.kv, sub(mc.page_table), sub(mc.topk),
                                                         mc.sm_scale, I.MLA_DV, seq_lens=sub(mc.seq_lens))
        if np.isneginf(lse_ref[0]).all():
            assert np.all(o[b] == 0.0) and np.all(np.isneginf(lse[b])), f"request {b}: empty selection"
            continue
        bad = np.abs(o[b] - o_ref[0]) > 2.0 ** -7 * o_abs[0] + 1e-6
        assert not bad.any(), f"request {b}: o off at {np.argwhere(bad)[:4]}, " \
                              f"{o[b][bad][:4]} vs {o_ref[0][bad][:4]}"
        dl = np.abs(lse[b] - lse_ref[0])
        assert np.all(dl <= 2.0 ** -8 + 1e-5 * np.abs(lse_ref[0])), f"request {b}: lse off by {dl.max()}"


def test_mla_one_block(gpu_lib, oracle):
    """One request, 64 of its 128 live entries: a single block, no split."""
    mc = I.mla_case(I.workload("b1_ctx8k_seq512"), k=64)
    o, lse = _run(gpu_lib, mc)
    _check(o, lse, mc, oracle)


def test_mla_mixed_lengths_split(gpu_lib, oracle):
    """16 requests of 256..8192 tokens, k = 2048 clamped to the live length: up to 32 blocks per
    row shared among several CTAs per request and merged by log-sum-exp."""
    mc = I.mla_case(I.workload("b16_ctx8k_mixed"))
    o, lse = _run(gpu_lib, mc)
    _check(o, lse, mc, oracle)


def test_mla_ragged_rows(gpu_lib, oracle):
    """k = 100 (a ragged last block): holes of -1 inside the row, positions at or past the live
    length, a duplicated position, and a request with no used entry."""
    case = I.make_case(name="ragged", batch=4, max_context=8192, seq_lens=[4000, 8192, 300, 1],
                       num_pages=160, k=100, seed=77)
    mc = I.mla_case(case)
    topk = mc.topk.copy()
    topk[0, 5:20] = -1                      # holes
    topk[0, 30] = 1000                      # live length is 1000: skipped
    topk[0, 31] = 999                       # the last live position
    topk[1, 60] = topk[1, 3]                # counted twice
    topk[2, :] = -1
    topk[2, 0] = 74                         # one used entry: o is that entry's value part
    topk[3, :] = -1                         # nothing used: o = 0, lse = -inf
    mc.topk = topk
    o, lse = _run(gpu_lib, mc)
    _check(o, lse, mc, oracle)
    assert np.all(o[3] == 0.0) and np.all(np.isneginf(lse[3]))


def test_mla_running_max_rescale(gpu_lib, oracle):
    """80 requests (one CTA each, 16 blocks): the cache pages of the first half of every row are
    scaled by 1/4 and the rest by 4 (exact in bf16), so a late block's maximum exceeds the running
    maximum by far more than 2^8 and the accumulated output is rescaled in tensor memory."""
    case = I.make_case(name="rescale", batch=80, max_context=4096, seq_lens=[4096] * 80, num_pages=1280,
                       k=1024, seed=78)
    mc = I.mla_case(case, sm_scale=1.0 / 24.0)
    kv = I.bf16_bits_to_f32(mc.kv)
    for b in range(case.batch):
        pages = case.page_table[b, :16]
        kv[pages[:8]] *= np.float32(0.25)
        kv[pages[8:]] *= np.float32(4.0)
    mc.kv = I.f32_to_bf16_bits(kv)
    o, lse = _run(gpu_lib, mc)
    _check(o, lse, mc, oracle)


def test_mla_indexer_topk_rows(gpu_lib, oracle):
    """The rows the indexer selects (the oracle's top-k on the mixed-length workload) as input."""
    case = I.workload("b16_ctx8k_mixed")
    topk = oracle.case_topk(case)
    mc = I.mla_case(case, topk=topk)
    o, lse = _run(gpu_lib, mc)
    _check(o, lse, mc, oracle)


@pytest.mark.slow
def test_mla_full_workload_sampled(gpu_lib, oracle):
    """64 requests at 128K context, k = 2048 of 32768 live entries each (the dense workload's
    table on its 8192-page pool): eight requests checked against the oracle, all outputs finite."""
    mc = I.mla_case(I.workload("b64_ctx128k_dense", literal_pool=True))
    o, lse = _run(gpu_lib, mc)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    _check(o, lse, mc, oracle, rows=[0, 9, 17, 26, 33, 42, 51, 63])


def test_mla_deterministic(gpu_lib):
    mc = I.mla_case(I.workload("b16_ctx8k_mixed"))
    o1, l1 = _run(gpu_lib, mc)
    o2, l2 = _run(gpu_lib, mc)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_mla_host_checks(gpu_lib):
    import torch
    b = gpu_lib
    mc = I.mla_case(I.workload("b1_ctx8k_seq512"), k=64)
    q, kv, table, seq, topk = _dev(mc)
    with pytest.raises(b.DsaError):
        b.dsa_sparse_mla_decode(q, kv, table, seq, mc.max_context, topk, float("nan"))
    big = torch.zeros((1, 2049), dtype=torch.int32, device="cuda")
    ws_ok = torch.zeros(b.sparse_mla_workspace_size(1, 2048), dtype=torch.uint8, device="cuda")
    with pytest.raises(b.DsaError):  # k past 2048: refused by the library itself
        b.dsa_sparse_mla_decode(q, kv, table, seq, mc.max_context, big, 0.1, workspace=ws_ok)
    ws = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(b.DsaError):
        b.dsa_sparse_mla_decode(q, kv, table, seq, mc.max_context, topk, 0.1, workspace=ws)
    assert b.sparse_mla_workspace_size(1, 0) == 0 and b.sparse_mla_workspace_size(1, 2049) == 0


def test_mla_more_requests_than_sms(gpu_lib, oracle):
    """200 requests (more than the SMs: one split each, no merge, several waves of CTAs),
    k = 1000 (a ragged last block), lengths 1..4096 tokens; every request checked."""
    rng = np.random.default_rng(91)
    seqs = rng.integers(1, 4097, size=200)
    case = I.make_case(name="many", batch=200, max_context=4096, seq_lens=seqs, num_pages=3400, k=1000, seed=92)
    mc = I.mla_case(case)
    o, lse = _run(gpu_lib, mc)
    _check(o, lse, mc, oracle)


def test_mla_max_batch(gpu_lib, oracle):
    """1024 requests (the boundary's maximum), k = 64, lengths 1..2048 tokens: about seven waves of
    CTAs, one split each; every request checked."""
    rng = np.random.default_rng(93)
    seqs = rng.integers(1, 2049, size=1024)
    case = I.make_case(name="maxb", batch=1024, max_context=2048, seq_lens=seqs, num_pages=8192, k=64, seed=94)
    mc = I.mla_case(case)
    o, lse = _run(gpu_lib, mc)
    _check(o, lse, mc, oracle)


def test_mla_zero_scale_is_the_mean(gpu_lib, oracle):
    """sm_scale = 0: every used entry has weight 1/n, so o is the plain mean of the used value rows
    and lse = log n (checked against the oracle, which computes the same softmax)."""
    mc = I.mla_case(I.workload("b16_ctx8k_mixed"), sm_scale=0.0)
    o, lse = _run(gpu_lib, mc)
    _check(o, lse, mc, oracle)
    n = (mc.topk >= 0).sum(axis=1)
    np.testing.assert_allclose(lse[:, 0], np.log(n), rtol=1e-5)


def test_mla_workspace_reused(gpu_lib, oracle):
    """Three calls on one workspace, on two different inputs: each result equals a call on a fresh
    workspace (nothing a call leaves in the workspace changes the next one)."""
    import torch
    b = gpu_lib
    mc1 = I.mla_case(I.workload("b16_ctx8k_mixed"))
    mc2 = I.mla_case(I.workload("b16_ctx8k_mixed"), sm_scale=0.02)
    ws = torch.zeros(b.sparse_mla_workspace_size(mc1.batch, mc1.topk.shape[1]), dtype=torch.uint8, device="cuda")
    outs = []
    for mc in (mc1, mc2, mc1):
        q, kv, table, seq, topk = _dev(mc)
        o, lse = b.dsa_sparse_mla_decode(q, kv, table, seq, mc.max_context, topk, mc.sm_scale, workspace=ws)
        torch.cuda.synchronize()
        assert b.get_error(ws, clear=False) == 0
        outs.append((o.cpu().numpy(), lse.cpu().numpy()))
    for (o, lse), mc in zip(outs, (mc1, mc2, mc1)):
        of, lf = _run(b, mc)
        assert np.array_equal(o, of) and np.array_equal(lse, lf)


def test_mla_bad_page_ids(gpu_lib, oracle):
    """A live page id outside [0, num_pages) sets the bad-page bit and is never read: requests
    whose pages are all valid still match the oracle, on the same call (the row gathers take
    another row of the request in place of the bad entry, so nothing outside the cache is read)."""
    import torch
    from sparse_attention_paged_dsa_gb300 import binding as b
    mc = I.mla_case(I.workload("b16_ctx8k_mixed"))
    table = mc.page_table.copy()
    n_pages = mc.kv.shape[0]
    bad_rows = [3, 7]
    for r in bad_rows:   # the first page of these requests (their top-k rows use it): out of range, then negative
        n = (int(mc.seq_lens[r]) + 3) // 4
        assert ((mc.topk[r] >= 0) & (mc.topk[r] < min(64, n))).any()
    for r in bad_rows:
        table[r, 0] = n_pages + 5 if r == 3 else -7
    q, kv, _, seq, topk = _dev(mc)
    t = torch.from_numpy(table).cuda()
    ws = torch.zeros(b.sparse_mla_workspace_size(mc.batch, mc.topk.shape[1]), dtype=torch.uint8, device="cuda")
    o, lse = b.dsa_sparse_mla_decode(q, kv, t, seq, mc.max_context, topk, mc.sm_scale, workspace=ws)
    torch.cuda.synchronize()
    assert b.get_error(ws) & 0x2, "bad-page bit not set"
    good = [r for r in range(mc.batch) if r not in bad_rows]
    _check(o.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), mc, oracle, rows=good)
