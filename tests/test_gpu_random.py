"""GPU parity on seeded random shapes: batch, max_context, lengths (including 0, 1..3 tokens, a
full row and a partial last page) and k drawn at random, through the scores, top-k and both
fused entry points (which must agree bit for bit), the multi-token and fp8 entry points, and the
sparse-MLA decode over random top-k rows; every result against the fp64 oracle."""
import numpy as np
import pytest

from sparse_attention_paged_dsa_gb300 import inputs as I

from _parity import check_scores, check_topk
from test_gpu_mtp import _flat, _run_mtp
from test_gpu_parity import _run_all

pytestmark = pytest.mark.gpu


def _random_case(seed):
    rng = np.random.default_rng(7000 + seed)
    batch = int(rng.integers(1, 25))
    max_context = 256 * int(rng.integers(1, 257))           # 256 .. 65536 tokens
    M = max_context // 4
    kinds = rng.integers(0, 6, size=batch)
    seq = np.where(kinds == 0, 0,
          np.where(kinds == 1, rng.integers(1, 4, size=batch),
          np.where(kinds == 2, max_context,
          np.where(kinds == 3, max_context - rng.integers(0, 256, size=batch),
                   rng.integers(0, max_context + 1, size=batch)))))
    seq = np.clip(seq, 0, max_context)
    k = int(rng.integers(1, min(M, 4096) + 1))
    pages = int(((seq + 255) // 256).sum()) + 8
    return I.make_case(name=f"rand{seed}", batch=batch, max_context=max_context, seq_lens=seq, num_pages=pages,
                       k=k, seed=8000 + seed, outlier_frac=0.01 if seed % 3 == 0 else 0.0)


@pytest.mark.parametrize("seed", range(16))
def test_random_shapes(gpu_lib, oracle, seed):
    case = _random_case(seed)
    s, t = _run_all(gpu_lib, case)
    ref = oracle.case_scores(case)
    check_scores(case, s, ref)
    check_topk(case, t, ref, gpu_scores=s)


@pytest.mark.parametrize("seed", range(6))
def test_random_shapes_multi_token(gpu_lib, oracle, seed):
    base = _random_case(100 + seed)
    Q = 2 + seed % 3
    case = I.with_next_n(base, Q)
    s, t = _run_mtp(gpu_lib, case)
    ref = oracle.case_scores_mtp(case)
    B = case.batch
    f = _flat(case)
    check_scores(f, s.reshape(B * Q, -1), ref.reshape(B * Q, -1))
    check_topk(f, t.reshape(B * Q, -1), ref.reshape(B * Q, -1), gpu_scores=s.reshape(B * Q, -1))


@pytest.mark.parametrize("seed", range(6))
def test_random_shapes_fp8(gpu_lib, oracle, seed):
    from test_gpu_fp8 import _run_fp8
    case = I.with_fp8_keys(_random_case(200 + seed))
    s, t, err = _run_fp8(gpu_lib, case)
    assert err == 0
    ref = oracle.case_scores_fp8(case)
    check_scores(case, s, ref)
    check_topk(case, t, ref, gpu_scores=s)


@pytest.mark.parametrize("seed", range(6))
def test_random_shapes_sparse_mla(gpu_lib, oracle, seed):
    """The decode over random top-k rows (holes, positions past the live length, duplicates) of a
    random indexer case: k from 1 to 2048, batches that take one or several splits per request."""
    from test_gpu_mla import _check, _run
    case = _random_case(300 + seed)
    rng = np.random.default_rng(9000 + seed)
    k = int(rng.integers(1, 2049))
    M = case.max_context // 4
    topk = rng.integers(-1, M, size=(case.batch, k)).astype(np.int32)  # -1 holes, any position
    mc = I.mla_case(case, topk)
    o, lse = _run(gpu_lib, mc)
    _check(o, lse, mc, oracle)
