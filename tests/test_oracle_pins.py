"""Pins of the fp64 CPU oracle to facts outside itself (CPU only).

Each test fixes the oracle against something it does not compute the same
way: a hand-worked example, closed forms, textbook/library routines on
special cases, invariants of the definition, and the numbers the pages print.
Together they are chosen so that a plausible slip in the oracle (a dropped
term, a wrong sign, a wrong page index, relu in the wrong place, floor in
place of ceil, ties resolved upwards) fails at least one of them; the
mutation test at the end checks exactly that on planted slips.
"""
import json
import math
import os
import re
import shutil
import subprocess

import numpy as np
import pytest

from sparse_attention_paged_dsa_gb300 import inputs as I

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16(x):
    return I.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def widen(bits):
    return I.bf16_bits_to_f32(bits).astype(np.float64)


# --------------------------------------------------------------- step 0: bf16
def test_bf16_widening_exact(oracle):
    # IEEE bit patterns: 0x3F80 = 1.0, 0xC000 = -2.0, 0x3F81 = 1 + 2^-7,
    # 0x0001 = smallest subnormal 2^-133, 0x7F7F = largest finite (2 - 2^-7) 2^127.
    assert oracle.bf16_to_double(0x3F80) == 1.0
    assert oracle.bf16_to_double(0xC000) == -2.0
    assert oracle.bf16_to_double(0x3F81) == 1.0 + 2.0 ** -7
    assert oracle.bf16_to_double(0x0001) == 2.0 ** -133
    assert oracle.bf16_to_double(0x7F7F) == (2.0 - 2.0 ** -7) * 2.0 ** 127
    assert oracle.bf16_to_double(0x8000) == 0.0 and math.copysign(1, oracle.bf16_to_double(0x8000)) < 0


# ---------------------------------------------------------- step 1: live count
@pytest.mark.parametrize("seq,n", [(0, 0), (1, 1), (3, 1), (4, 1), (5, 2), (8, 2), (255, 64),
                                   (256, 64), (257, 65), (131072, 32768), (-3, 0)])
def test_live_count_is_ceil_quarter(oracle, seq, n):
    # One C4 key per 4 tokens; a trailing 1-3 tokens still make a key.
    assert oracle.live_count(seq) == n


# ------------------------------------------------- pages' printed shape values
def test_row_width_matches_printed_shapes():
    """The printed 262208 = page_table width 4097 x 64, and ~1M -> 8192 is ~128x."""
    with open(os.path.join(GOLDEN, "printed_shapes.json")) as f:
        g = json.load(f)
    W = g["page_table_width"]
    max_context = W * I.PAGE_TOKENS
    case = I.IndexerCase("shape", np.zeros((1, 32, 64), np.uint16), np.zeros((1, 32), np.float32),
                         np.zeros((1, 64, 64), np.uint16), np.zeros((1, W), np.int32),
                         np.zeros(1, np.int32), max_context, 1)
    assert case.row_width == g["max_c4_seq_len"]
    assert case.table_width == W
    small = 8192 // I.PAGE_TOKENS * I.PAGE_ENTRIES
    assert round(case.row_width / small) == g["work_ratio_1m_to_8k"]


# --------------------------------------------------- hand-worked example (H=2)
def _hand_case():
    # H = 2 heads, D = 3 dims, E = 2 entries per page (8-token pages),
    # max_context = 16 tokens -> row width M = 4, table width W = 2.
    pool = bf16([[[1, 0, 2], [5, 5, 5]],      # page 0
                 [[9, 9, 9], [9, 9, 9]],      # page 1
                 [[1, -1, 0], [0, 2, -1]]])   # page 2
    table = np.array([[2, 0], [1, 2]], np.int32)
    seq = np.array([9, 8], np.int32)          # n = ceil(9/4) = 3, ceil(8/4) = 2
    q = bf16([[[2, 1, 0], [-1, 0, 1]],
              [[1, 1, 1], [0, 0, -1]]])
    w = np.array([[0.5, -2.0], [1.0, 1.0]], np.float32)
    return q, w, pool, table, seq


def test_hand_worked_example(oracle):
    q, w, pool, table, seq = _hand_case()
    s = oracle.scores(q, w, pool, table, seq, 16)
    # Row 0.  K[0] = page2[0] = (1,-1,0), K[1] = page2[1] = (0,2,-1), K[2] = page0[0] = (1,0,2).
    #   t=0: dots (2-1+0, -1+0+0) = (1,-1) -> relu (1,0) -> 0.5*1 - 2*0 = 0.5
    #   t=1: dots (0+2+0, 0+0-1)  = (2,-1) -> relu (2,0) -> 0.5*2       = 1.0
    #   t=2: dots (2+0+0, -1+0+2) = (2, 1) -> relu (2,1) -> 1.0 - 2.0   = -1.0
    #   t=3: past n = 3 -> -inf
    # Row 1.  K[0] = K[1] = page1 entries (9,9,9): dots (27,-9) -> relu (27,0) -> 27; t>=2 -> -inf
    expect = np.array([[0.5, 1.0, -1.0, -np.inf], [27.0, 27.0, -np.inf, -np.inf]])
    np.testing.assert_array_equal(s, expect)
    # top-k: row 0 best two are t=1 (1.0), t=0 (0.5); row 1 ties resolve to the lower position.
    np.testing.assert_array_equal(oracle.topk(s, seq, 16, 2), [[0, 1], [0, 1]])
    np.testing.assert_array_equal(oracle.topk(s, seq, 16, 1), [[1], [0]])
    np.testing.assert_array_equal(oracle.topk(s, seq, 16, 4), [[0, 1, 2, -1], [0, 1, -1, -1]])


# ------------------------------------------------------------ closed forms
def _rand_case(seed, B=3, seqs=(300, 5, 257), max_context=1024, num_pages=16, key_dist="normal"):
    return I.make_case(name="pin", batch=B, max_context=max_context, seq_lens=list(seqs),
                       num_pages=num_pages, k=37, seed=seed, key_dist=key_dist)


def test_one_hot_keys_give_weighted_relu_of_query_column(oracle):
    """k[t] = e_d  =>  s[t] = sum_h w_h relu(q[h, d]) (no dot product involved)."""
    c = _rand_case(1)
    D = I.HEAD_DIM
    pool = np.zeros_like(c.key_pool)
    d_of = {}
    for p in range(c.num_pages):
        for e in range(I.PAGE_ENTRIES):
            d = (7 * p + 3 * e) % D
            pool[p, e, d] = 0x3F80  # 1.0
            d_of[(p, e)] = d
    s = oracle.scores(c.q, c.w, pool, c.page_table, c.seq_lens, c.max_context)
    qd = widen(c.q)
    for b in range(c.batch):
        n = (int(c.seq_lens[b]) + 3) // 4
        for t in range(n):
            p = int(c.page_table[b, t // I.PAGE_ENTRIES])
            d = d_of[(p, t % I.PAGE_ENTRIES)]
            expect = float(np.dot(c.w[b].astype(np.float64), np.maximum(qd[b, :, d], 0.0)))
            assert s[b, t] == pytest.approx(expect, rel=1e-12, abs=1e-12)


def test_one_hot_weights_select_one_head(oracle):
    """w = e_h  =>  s[t] = relu(q_h . k[t]) (library matmul on the gathered keys)."""
    c = _rand_case(2)
    for h in (0, 13, 31):
        w = np.zeros_like(c.w)
        w[:, h] = 1.0
        s = oracle.scores(c.q, w, c.key_pool, c.page_table, c.seq_lens, c.max_context)
        for b in range(c.batch):
            n = (int(c.seq_lens[b]) + 3) // 4
            pages = c.page_table[b, :(n + 63) // 64]
            K = widen(c.key_pool[pages]).reshape(-1, I.HEAD_DIM)[:n]
            expect = np.maximum(K @ widen(c.q[b, h]), 0.0)
            np.testing.assert_allclose(s[b, :n], expect, rtol=1e-12, atol=1e-12)


def test_nonnegative_inputs_reduce_to_gemv(oracle):
    """q, k >= 0 make relu the identity: s = (w^T Q) K^T, a GEMV in another order."""
    c = _rand_case(3)
    q = bf16(np.abs(widen(c.q)))
    pool = bf16(np.abs(widen(c.key_pool)))
    s = oracle.scores(q, c.w, pool, c.page_table, c.seq_lens, c.max_context)
    for b in range(c.batch):
        n = (int(c.seq_lens[b]) + 3) // 4
        pages = c.page_table[b, :(n + 63) // 64]
        K = widen(pool[pages]).reshape(-1, I.HEAD_DIM)[:n]
        v = c.w[b].astype(np.float64) @ widen(q[b])
        np.testing.assert_allclose(s[b, :n], K @ v, rtol=1e-10, atol=1e-10)


def test_opposite_head_pairs_give_absolute_value(oracle):
    """q_{2i+1} = -q_{2i}, equal weights: relu(x) + relu(-x) = |x| per pair.

    Fixes that relu acts on each head's dot product before the weighted sum.
    """
    c = _rand_case(4)
    q = c.q.copy()
    q[:, 1::2, :] = q[:, 0::2, :] ^ np.uint16(0x8000)  # flip the sign bit
    w = c.w.copy()
    w[:, 1::2] = w[:, 0::2]
    s = oracle.scores(q, w, c.key_pool, c.page_table, c.seq_lens, c.max_context)
    for b in range(c.batch):
        n = (int(c.seq_lens[b]) + 3) // 4
        pages = c.page_table[b, :(n + 63) // 64]
        K = widen(c.key_pool[pages]).reshape(-1, I.HEAD_DIM)[:n]
        dots = K @ widen(q[b, 0::2]).T          # [n, 16]
        expect = np.abs(dots) @ w[b, 0::2].astype(np.float64)
        np.testing.assert_allclose(s[b, :n], expect, rtol=1e-10, atol=1e-10)


def test_positive_homogeneity_in_weights(oracle):
    c = _rand_case(5)
    s1 = oracle.case_scores(c)
    s4 = oracle.scores(c.q, (c.w * np.float32(4.0)), c.key_pool, c.page_table, c.seq_lens, c.max_context)
    live = np.isfinite(s1)
    np.testing.assert_array_equal(s4[live], 4.0 * s1[live])


# --------------------------------------------------------------- invariants
def test_minus_inf_exactly_past_live_length(oracle):
    c = I.make_case(name="tail", batch=6, max_context=2048, seq_lens=[0, 1, 4, 5, 256, 2048],
                    num_pages=64, k=8, seed=6)
    s = oracle.case_scores(c)
    for b, n in enumerate(c.live_positions()):
        assert np.all(np.isfinite(s[b, :n]))
        assert np.all(s[b, n:] == -np.inf)


def test_paged_equals_contiguous(oracle):
    """Scatter contiguous keys into pages by a random table; the oracle must read them back."""
    rng = np.random.default_rng(7)
    n, M = 300, 512
    keys = bf16(rng.standard_normal((n, I.HEAD_DIM)).astype(np.float32))
    P = (n + 63) // 64
    num_pages = 11
    slots = rng.permutation(num_pages)[:P]
    pool = bf16(rng.standard_normal((num_pages, 64, I.HEAD_DIM)).astype(np.float32))
    padded = np.zeros((P * 64, I.HEAD_DIM), np.uint16)
    padded[:n] = keys
    for j in range(P):
        pool[slots[j]] = padded[j * 64:(j + 1) * 64]
    table = np.full(M // 64, -1, np.int32)
    table[:P] = slots
    g = oracle.gather(pool, table, n)
    np.testing.assert_array_equal(g, widen(keys))
    q = bf16(rng.standard_normal((1, 32, 64)).astype(np.float32))
    w = rng.standard_normal((1, 32)).astype(np.float32)
    paged = oracle.scores(q, w, pool, table[None], np.array([4 * n - 2], np.int32), 4 * M)
    dense = oracle.scores_dense(q[0], w[0], widen(keys), M)
    np.testing.assert_array_equal(paged[0], dense)


def test_physical_page_permutation_invariance(oracle):
    c = _rand_case(8, num_pages=24)
    rng = np.random.default_rng(9)
    perm = rng.permutation(c.num_pages)          # new slot of old page p is perm[p]
    pool2 = np.empty_like(c.key_pool)
    pool2[perm] = c.key_pool
    table2 = np.where(c.page_table >= 0, perm[np.maximum(c.page_table, 0)], -1).astype(np.int32)
    np.testing.assert_array_equal(oracle.case_scores(c),
                                  oracle.scores(c.q, c.w, pool2, table2, c.seq_lens, c.max_context))


def test_dead_table_entries_and_unreferenced_pages_are_ignored(oracle):
    base = _rand_case(10, num_pages=24)
    rnd = I.make_case(name="pin", batch=3, max_context=1024, seq_lens=[300, 5, 257], num_pages=24,
                      k=37, seed=10, dead_fill="random")
    np.testing.assert_array_equal(base.page_table[base.page_table >= 0],
                                  rnd.page_table[base.page_table >= 0])
    s0 = oracle.case_scores(base)
    np.testing.assert_array_equal(s0, oracle.case_scores(rnd))
    used = set(base.page_table[base.page_table >= 0].tolist())
    pool = base.key_pool.copy()
    for p in range(base.num_pages):
        if p not in used:
            pool[p] = 0x4120  # 10.0
    np.testing.assert_array_equal(
        s0, oracle.scores(base.q, base.w, pool, base.page_table, base.seq_lens, base.max_context))


# -------------------------------------------------------------------- top-k
def _lexsort_topk(row, n, k):
    order = np.lexsort((np.arange(n), -row[:n]))   # primary: score desc, then position asc
    keep = np.sort(order[:min(k, n)])
    out = np.full(k, -1, np.int64)
    out[:keep.size] = keep
    return out


@pytest.mark.parametrize("seed", range(6))
def test_topk_equals_full_library_sort(oracle, seed):
    rng = np.random.default_rng(100 + seed)
    n = int(rng.integers(0, 700))
    M = 800
    # coarse values so that ties are frequent
    row = np.full(M, -np.inf)
    row[:n] = rng.integers(-20, 20, size=n) / 4.0
    k = int(rng.integers(1, 900))
    got = oracle.topk_row(row, n, k)
    np.testing.assert_array_equal(got, _lexsort_topk(row, n, k))


def test_topk_selection_property_brute_force(oracle):
    """Every chosen position beats every unchosen live one, ties to the lower index."""
    rng = np.random.default_rng(11)
    for _ in range(20):
        n = int(rng.integers(1, 60))
        row = rng.integers(-3, 3, size=n).astype(np.float64)
        k = int(rng.integers(1, 70))
        got = oracle.topk_row(row, n, k)
        chosen = [int(i) for i in got if i >= 0]
        assert chosen == sorted(chosen) and len(chosen) == min(k, n)
        assert all(i == -1 for i in got[len(chosen):])
        rest = [j for j in range(n) if j not in set(chosen)]
        for i in chosen:
            for j in rest:
                assert row[i] > row[j] or (row[i] == row[j] and i < j)


def test_topk_all_equal_scores_takes_lowest_positions(oracle):
    c = I.make_case(name="eq", batch=2, max_context=2048, seq_lens=[1000, 120], num_pages=16,
                    k=100, seed=12)
    pool = np.zeros_like(c.key_pool)
    pool[:, :, 0] = 0x3F80
    s = oracle.scores(c.q, c.w, pool, c.page_table, c.seq_lens, c.max_context)
    t = oracle.topk(s, c.seq_lens, c.max_context, 100)
    np.testing.assert_array_equal(t[0], np.arange(100))
    np.testing.assert_array_equal(t[1], np.r_[np.arange(30), -np.ones(70, int)])


def test_topk_empty_row_is_all_minus_one(oracle):
    row = np.full(64, -np.inf)
    np.testing.assert_array_equal(oracle.topk_row(row, 0, 5), [-1] * 5)


# ------------------------------------------------- cross-machine regression
def test_stored_oracle_values_reproduce():
    """Values written by tests/golden/make_oracle_golden.py (calls only the oracle)."""
    from oracle import oracle as o
    with open(os.path.join(GOLDEN, "oracle_small_case.json")) as f:
        g = json.load(f)
    c = I.make_case(**g["case"])
    s = o.case_scores(c)
    got = [float.hex(float(x)) for x in s[np.isfinite(s)]]
    assert got == g["live_scores_hex"]
    np.testing.assert_array_equal(o.case_topk(c, s), np.array(g["topk"]))


# ------------------------------------------------------ planted-slip check
MUTATIONS = [
    ("page index uses t % E", "int64_t j = t / E;  /* page slot", "int64_t j = t % E;  /* page slot"),
    ("entry index uses t / E", "int64_t e = t % E;  /* entry", "int64_t e = t / E;  /* entry"),
    ("relu dropped", "double r = dot > 0.0 ? dot : 0.0;", "double r = dot;"),
    ("weight dropped", "s += (double)w_row[h] * r;", "s += r;"),
    ("floor in place of ceil", "return (seq_len + 3) / 4;", "return seq_len / 4;"),
    ("ties to the higher position", "return (x->t > y->t) - (x->t < y->t);",
     "return (x->t < y->t) - (x->t > y->t);"),
    ("last head skipped", "for (int32_t h = 0; h < H; ++h) {", "for (int32_t h = 0; h < H - 1; ++h) {"),
    ("query/key dims transposed", "q_row[h * D + d]", "q_row[d * H + h]"),
]


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("label,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_slips_fail_a_pin(tmp_path, label, old, new):
    """Compile the oracle with one planted slip; the pins above must catch it."""
    import ctypes
    from oracle import oracle as o
    src = open(o.SRC).read()
    assert src.count(old) == 1, label
    mutated = tmp_path / "mut.c"
    mutated.write_text(src.replace(old, new))
    lib = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                    str(mutated), "-o", str(lib), "-lm"], check=True)
    saved_lib, saved_path = o._lib, o.LIB
    try:
        o._lib = None
        o.LIB = str(lib)
        o.build = lambda force=False: str(lib)   # use the mutant as is
        caught = False
        for pin in (test_hand_worked_example, test_opposite_head_pairs_give_absolute_value,
                    test_paged_equals_contiguous, test_topk_all_equal_scores_takes_lowest_positions,
                    test_one_hot_keys_give_weighted_relu_of_query_column):
            try:
                pin(o)
            except (AssertionError, ValueError):
                caught = True
                break
        for seq, n in [(5, 2), (257, 65)]:
            if o.live_count(seq) != n:
                caught = True
        assert caught, f"planted slip '{label}' passed every pin"
    finally:
        o._lib, o.LIB = saved_lib, saved_path
        import importlib
        importlib.reload(o)
