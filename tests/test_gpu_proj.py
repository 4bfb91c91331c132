"""GPU parity of the q/w projection (row f4) against the fp64 oracle.

q is stored as bf16, so each element must lie within bf16 rounding (2^-8 relative) of the fp64
oracle, plus a small fp32-accumulation slack, and equal the oracle rounded to bf16 on integer
inputs; w is fp32.
Covers token counts across the N paddings (1, 5, 32, 64, 100, 256), model widths from one 64-wide
atom to 7168 (uneven split-K ranges), determinism, the chain projection -> scores, and the host
argument checks."""
import ctypes

import numpy as np
import pytest

from sparse_attention_paged_dsa_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _rand(seed, B, d, scale=1.0):
    rng = np.random.default_rng(seed)
    x = I.f32_to_bf16_bits((rng.standard_normal((B, d)) * scale).astype(np.float32))
    wq = I.f32_to_bf16_bits((rng.standard_normal((2048, d)) / np.sqrt(d)).astype(np.float32))
    ww = I.f32_to_bf16_bits((rng.standard_normal((32, d)) / np.sqrt(d)).astype(np.float32))
    return x, wq, ww


def _run(b, x, wq, ww):
    import torch
    t = lambda a: torch.from_numpy(a.view("int16")).cuda().view(torch.bfloat16)
    q, w = b.dsa_indexer_qw_proj(t(x), t(wq), t(ww))
    torch.cuda.synchronize()
    return q.view(torch.int16).cpu().numpy().view(np.uint16), w.cpu().numpy()


def _check(q_bits, w, q_ref, w_ref):
    """q: bf16 rounding to nearest is within 2^-8 of the value (half a unit in the last of 8
    significant bits, at the bottom of a binade); the fp32 accumulation adds at most ~2^-20 of the
    row's largest |q| here.  w: fp32, relative 1e-5 of the row's largest |w|."""
    q = I.bf16_bits_to_f32(q_bits).astype(np.float64)
    for b in range(q.shape[0]):
        slack = 2.0 ** -20 * np.abs(q_ref[b]).max()
        bad = np.abs(q[b] - q_ref[b]) > 2.0 ** -8 * np.abs(q_ref[b]) + slack
        assert not bad.any(), f"q row {b}: {np.argwhere(bad)[:4]}"
        sw = np.abs(w_ref[b]).max()
        assert np.abs(w[b] - w_ref[b]).max() <= 1e-5 * sw + 1e-30, f"w row {b}"


@pytest.mark.parametrize("B,d", [(1, 64), (5, 448), (32, 1024), (64, 7168), (100, 1536), (256, 2048)])
def test_proj_random(gpu_lib, oracle, B, d):
    x, wq, ww = _rand(B * 1000 + d, B, d)
    q, w = _run(gpu_lib, x, wq, ww)
    q_ref, w_ref = oracle.qw_proj(x, wq, ww)
    _check(q, w, q_ref, w_ref)


def test_proj_integer_inputs_exact(gpu_lib, oracle):
    """Integer x and weights in [-4, 4], d = 512: every sum is an exact fp32 integer; q equals the
    oracle's value rounded to bf16 (nearest even), w equals it exactly."""
    rng = np.random.default_rng(5)
    B, d = 40, 512
    f = lambda shape: I.f32_to_bf16_bits(rng.integers(-4, 5, size=shape).astype(np.float32))
    x, wq, ww = f((B, d)), f((2048, d)), f((32, d))
    q, w = _run(gpu_lib, x, wq, ww)
    q_ref, w_ref = oracle.qw_proj(x, wq, ww)
    np.testing.assert_array_equal(q, I.f32_to_bf16_bits(q_ref.astype(np.float32)))
    np.testing.assert_array_equal(w.astype(np.float64), w_ref)


def test_proj_deterministic(gpu_lib):
    x, wq, ww = _rand(9, 64, 7168)
    q0, w0 = _run(gpu_lib, x, wq, ww)
    q1, w1 = _run(gpu_lib, x, wq, ww)
    np.testing.assert_array_equal(q0, q1)
    np.testing.assert_array_equal(w0.view(np.uint32), w1.view(np.uint32))


def test_proj_feeds_the_indexer(gpu_lib, oracle):
    """Projection outputs go straight into the scores entry point; the scores match the oracle
    evaluated on the oracle's own projection (rounded to the stored formats)."""
    import torch
    B, d = 8, 2048
    x, wq, ww = _rand(11, B, d)
    case = I.make_case(name="chain", batch=B, max_context=8192, seq_lens=[8192, 4000, 3, 700, 8192, 1, 256, 5000],
                       num_pages=300, k=100, seed=12)
    q_bits, w = _run(gpu_lib, x, wq, ww)
    q_ref, w_ref = oracle.qw_proj(x, wq, ww)
    chained = I.IndexerCase("chain", q_bits.reshape(B, 32, 64), w.astype(np.float32), case.key_pool,
                            case.page_table, case.seq_lens, case.max_context, case.k)
    qd, wd, pool, table, seq = gpu_lib.to_device(chained)
    s = gpu_lib.dsa_indexer_scores(qd, wd, pool, table, seq, case.max_context)
    torch.cuda.synchronize()
    ref = oracle.case_scores(chained)
    from _parity import check_scores
    check_scores(chained, s.cpu().numpy(), ref)


def test_proj_host_argument_checks(gpu_lib):
    import torch
    b = gpu_lib
    lib = b.load()
    assert lib.dsa_indexer_qw_proj_workspace_size(0, 64) == 0
    assert lib.dsa_indexer_qw_proj_workspace_size(257, 64) == 0
    assert lib.dsa_indexer_qw_proj_workspace_size(4, 100) == 0
    assert lib.dsa_indexer_qw_proj_workspace_size(4, 0) == 0
    x = torch.zeros((4, 128), dtype=torch.bfloat16, device="cuda")
    wq = torch.zeros((2048, 128), dtype=torch.bfloat16, device="cuda")
    ww = torch.zeros((32, 128), dtype=torch.bfloat16, device="cuda")
    q = torch.empty((4, 32, 64), dtype=torch.bfloat16, device="cuda")
    w = torch.empty((4, 32), dtype=torch.float32, device="cuda")
    n = lib.dsa_indexer_qw_proj_workspace_size(4, 128)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    P = ctypes.c_void_p
    s = P(torch.cuda.current_stream().cuda_stream)
    call = lambda **k: lib.dsa_indexer_qw_proj(k.get("x", P(x.data_ptr())), P(wq.data_ptr()), P(ww.data_ptr()),
                                               k.get("B", 4), k.get("d", 128), P(q.data_ptr()), P(w.data_ptr()),
                                               P(ws.data_ptr()), k.get("wsb", n), s)
    assert call() == b.DSA_OK
    assert call(x=None) == b.DSA_ERR_INVALID_ARG
    assert call(x=P(x.data_ptr() + 2)) == b.DSA_ERR_INVALID_ARG
    assert call(d=96) == b.DSA_ERR_INVALID_ARG
    assert call(B=0) == b.DSA_ERR_INVALID_ARG
    assert call(wsb=n - 4) == b.DSA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert b.get_error(ws) == 0
    assert torch.count_nonzero(q.view(torch.int16)) == 0 and torch.count_nonzero(w) == 0
