"""CPU checks of the sparse-MLA input generators (no GPU): the synthetic top-k rows have the
shape of the indexer's output, and the cases are reproducible from their seed."""
import numpy as np

from sparse_attention_paged_dsa_gb300 import inputs as I


def test_random_topk_has_the_indexer_output_shape():
    """min(k, live) distinct positions below the live length, ascending, then -1 padding."""
    case = I.make_case(name="t", batch=5, max_context=8192, seq_lens=[1, 300, 4096, 8192, 0], num_pages=200, k=700,
                       seed=3)
    topk = I.random_topk(case, 700, seed=3)
    live = case.live_positions()
    assert topk.shape == (5, 700) and topk.dtype == np.int32
    for b in range(5):
        n = int(min(700, live[b]))
        row = topk[b]
        assert np.all(row[n:] == -1)
        used = row[:n]
        assert np.all(used >= 0) and np.all(used < live[b])
        assert np.all(np.diff(used) > 0)  # ascending, hence distinct


def test_random_topk_takes_all_of_a_short_row():
    case = I.make_case(name="t", batch=1, max_context=8192, seq_lens=[100], num_pages=8, k=64, seed=4)
    topk = I.random_topk(case, 64, seed=4)
    assert np.array_equal(topk[0, :25], np.arange(25)) and np.all(topk[0, 25:] == -1)


def test_mla_case_shapes_and_reproducibility():
    case = I.workload("b1_ctx8k_seq512")
    a = I.mla_case(case, k=64)
    b = I.mla_case(case, k=64)
    assert a.q.shape == (1, I.MLA_HEADS, I.MLA_DIM) and a.q.dtype == np.uint16
    assert a.kv.shape == (case.num_pages, I.PAGE_ENTRIES, I.MLA_DIM) and a.kv.dtype == np.uint16
    assert a.topk.shape == (1, 64)
    assert np.array_equal(a.q, b.q) and np.array_equal(a.kv, b.kv) and np.array_equal(a.topk, b.topk)
    assert a.page_table is case.page_table and np.array_equal(a.seq_lens, case.seq_lens)
    # given rows are kept as they are
    given = np.full((1, 10), -1, np.int32)
    given[0, :3] = [5, 1, 9]
    c = I.mla_case(case, topk=given)
    assert np.array_equal(c.topk, given)


def test_mla_case_values_are_standard_normal_bf16():
    """q and the cache are N(0, 1) rounded to bf16: mean near 0, variance near 1 over the pool."""
    a = I.mla_case(I.workload("b1_ctx8k_seq512"), k=64)
    x = I.bf16_bits_to_f32(a.kv).astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.var() - 1.0) < 0.01
    assert np.array_equal(I.f32_to_bf16_bits(I.bf16_bits_to_f32(a.kv)), a.kv)  # exact bf16 values
