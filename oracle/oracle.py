"""ctypes front-end of the fp64 CPU oracle (``dsa_oracle.c``).

TEST INFRASTRUCTURE.  Only the test suite, the package smoke check and the
benchmark's CPU-baseline leg may import this module.  It never touches the
CUDA library and the CUDA library never touches it.

``build()`` compiles ``dsa_oracle.c`` with gcc (strict IEEE: no fast-math, no
contraction of multiply-add) into ``liboracle_dsa.so`` beside it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "dsa_oracle.c")
LIB = os.path.join(HERE, "liboracle_dsa.so")

_lib = None


def build(force: bool = False) -> str:
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        tmp = LIB + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
               "-fno-fast-math", SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB)
    return LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(LIB)
        i32, i64, p = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
        lib.dsa_oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.dsa_oracle_bf16_to_double.restype = ctypes.c_double
        lib.dsa_oracle_live_count.argtypes = [i64]
        lib.dsa_oracle_live_count.restype = i64
        lib.dsa_oracle_gather.argtypes = [p, i64, i32, i32, p, i64, i64, p]
        lib.dsa_oracle_gather.restype = ctypes.c_int
        lib.dsa_oracle_scores_dense.argtypes = [p, p, i32, i32, p, i64, i64, p]
        lib.dsa_oracle_scores_dense.restype = None
        lib.dsa_oracle_scores.argtypes = [p, p, i32, i32, p, i64, i32, p, p, i32, i64, p]
        lib.dsa_oracle_scores.restype = ctypes.c_int
        lib.dsa_oracle_topk_row.argtypes = [p, i64, i32, p]
        lib.dsa_oracle_topk_row.restype = ctypes.c_int
        lib.dsa_oracle_topk.argtypes = [p, p, i32, i64, i32, p]
        lib.dsa_oracle_topk.restype = ctypes.c_int
        lib.dsa_oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        lib.dsa_oracle_e4m3_to_double.restype = ctypes.c_double
        lib.dsa_oracle_gather_fp8.argtypes = [p, p, i64, i32, i32, p, i64, i64, p]
        lib.dsa_oracle_gather_fp8.restype = ctypes.c_int
        lib.dsa_oracle_scores_fp8.argtypes = [p, p, i32, i32, p, p, i64, i32, p, p, i32, i64, p]
        lib.dsa_oracle_scores_fp8.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags.c_contiguous
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what} failed with code {rc}")


def bf16_to_double(bits: int) -> float:
    return float(_load().dsa_oracle_bf16_to_double(int(bits)))


def live_count(seq_len: int) -> int:
    return int(_load().dsa_oracle_live_count(int(seq_len)))


def gather(pool, table_row, n: int, entries: int = 64) -> np.ndarray:
    """Contiguous fp64 keys [n, D] of one request read through its table row."""
    pool = np.ascontiguousarray(pool, dtype=np.uint16)
    table_row = np.ascontiguousarray(table_row, dtype=np.int32)
    D = pool.shape[-1]
    out = np.empty((max(n, 0), D), dtype=np.float64)
    rc = _load().dsa_oracle_gather(_ptr(pool), pool.shape[0], entries, D, _ptr(table_row),
                                   table_row.shape[0], n, _ptr(out))
    _check(rc, "gather")
    return out


def scores_dense(q_row, w_row, keys, row_width: int) -> np.ndarray:
    """fp64 scores of one request over contiguous keys; -inf from len(keys) on."""
    q_row = np.ascontiguousarray(q_row, dtype=np.uint16)
    w_row = np.ascontiguousarray(w_row, dtype=np.float32)
    keys = np.ascontiguousarray(keys, dtype=np.float64)
    H, D = q_row.shape
    out = np.empty(row_width, dtype=np.float64)
    _load().dsa_oracle_scores_dense(_ptr(q_row), _ptr(w_row), H, D, _ptr(keys), keys.shape[0],
                                    row_width, _ptr(out))
    return out


def scores(q, w, key_pool, page_table, seq_lens, max_context: int) -> np.ndarray:
    """fp64 scores [B, max_context/4] through the page table."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    w = np.ascontiguousarray(w, dtype=np.float32)
    pool = np.ascontiguousarray(key_pool, dtype=np.uint16)
    table = np.ascontiguousarray(page_table, dtype=np.int32)
    seq = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B, H, D = q.shape
    E = pool.shape[1]
    out = np.empty((B, max_context // 4), dtype=np.float64)
    rc = _load().dsa_oracle_scores(_ptr(q), _ptr(w), H, D, _ptr(pool), pool.shape[0], E,
                                   _ptr(table), _ptr(seq), B, max_context, _ptr(out))
    _check(rc, "scores")
    return out


def topk_row(row, n: int, k: int) -> np.ndarray:
    row = np.ascontiguousarray(row, dtype=np.float64)
    out = np.empty(k, dtype=np.int32)
    _check(_load().dsa_oracle_topk_row(_ptr(row), n, k, _ptr(out)), "topk_row")
    return out


def topk(rows, seq_lens, max_context: int, k: int) -> np.ndarray:
    """Top-k [B, k] of score rows [B, max_context/4] (any float dtype, widened)."""
    rows = np.ascontiguousarray(rows, dtype=np.float64)
    seq = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B = rows.shape[0]
    out = np.empty((B, k), dtype=np.int32)
    _check(_load().dsa_oracle_topk(_ptr(rows), _ptr(seq), B, max_context, k, _ptr(out)), "topk")
    return out


def e4m3_to_double(code: int) -> float:
    return float(_load().dsa_oracle_e4m3_to_double(int(code)))


def gather_fp8(codes, scales, table_row, n: int, entries: int = 64) -> np.ndarray:
    """Contiguous fp64 keys [n, D] (scale x decoded codes) of one request."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.float32)
    table_row = np.ascontiguousarray(table_row, dtype=np.int32)
    D = codes.shape[-1]
    out = np.empty((max(n, 0), D), dtype=np.float64)
    rc = _load().dsa_oracle_gather_fp8(_ptr(codes), _ptr(scales), codes.shape[0], entries, D,
                                       _ptr(table_row), table_row.shape[0], n, _ptr(out))
    _check(rc, "gather_fp8")
    return out


def scores_fp8(q, w, key_codes, key_scales, page_table, seq_lens, max_context: int) -> np.ndarray:
    """fp64 scores [B, max_context/4] on the fp8 cache (k = scale x e4m3(code))."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    w = np.ascontiguousarray(w, dtype=np.float32)
    codes = np.ascontiguousarray(key_codes, dtype=np.uint8)
    scales = np.ascontiguousarray(key_scales, dtype=np.float32)
    table = np.ascontiguousarray(page_table, dtype=np.int32)
    seq = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B, H, D = q.shape
    E = codes.shape[1]
    out = np.empty((B, max_context // 4), dtype=np.float64)
    rc = _load().dsa_oracle_scores_fp8(_ptr(q), _ptr(w), H, D, _ptr(codes), _ptr(scales), codes.shape[0], E,
                                       _ptr(table), _ptr(seq), B, max_context, _ptr(out))
    _check(rc, "scores_fp8")
    return out


def case_scores_fp8(case) -> np.ndarray:
    return scores_fp8(case.q, case.w, case.key_codes, case.key_scales, case.page_table, case.seq_lens,
                      case.max_context)


def scores_mtp(q, w, key_pool, page_table, seq_lens, max_context: int) -> np.ndarray:
    """fp64 scores [B, Q, max_context/4] for Q query tokens per request (q [B, Q, H, D], w [B, Q, H]).

    Token j is an ordinary indexer query whose sequence is the request's first
    seq_len - (Q - 1 - j) tokens (its causal prefix; the request's seq_len counts
    all Q tokens): the single-token definition applied once per token."""
    q = np.asarray(q)
    w = np.asarray(w)
    B, Q = q.shape[0], q.shape[1]
    seq = np.asarray(seq_lens, dtype=np.int64)
    out = np.empty((B, Q, max_context // 4), dtype=np.float64)
    for j in range(Q):
        seq_j = np.maximum(seq - (Q - 1 - j), 0).astype(np.int32)
        out[:, j] = scores(q[:, j], w[:, j], key_pool, page_table, seq_j, max_context)
    return out


def topk_mtp(rows, seq_lens, max_context: int, k: int) -> np.ndarray:
    """Top-k [B, Q, k] of score rows [B, Q, max_context/4], token j with its own causal length."""
    rows = np.asarray(rows)
    B, Q = rows.shape[0], rows.shape[1]
    seq = np.asarray(seq_lens, dtype=np.int64)
    out = np.empty((B, Q, k), dtype=np.int32)
    for j in range(Q):
        seq_j = np.maximum(seq - (Q - 1 - j), 0).astype(np.int32)
        out[:, j] = topk(rows[:, j], seq_j, max_context, k)
    return out


def case_scores_mtp(case) -> np.ndarray:
    return scores_mtp(case.q, case.w, case.key_pool, case.page_table, case.seq_lens, case.max_context)


def qw_proj(x_bits, wq_bits, ww_bits):
    """fp64 q [B, 32, 64] and w [B, 32] from the bf16 hidden state: q = x Wq^T, w = x Ww^T.

    The bf16 bit patterns are widened exactly; the products and sums are fp64 (a
    library matmul on fp64 arrays is the step)."""
    x = _bf16_bits_to_f64(x_bits)
    wq = _bf16_bits_to_f64(wq_bits)
    ww = _bf16_bits_to_f64(ww_bits)
    q = x @ wq.T
    w = x @ ww.T
    return q.reshape(x.shape[0], ww.shape[0], -1), w


def sparse_mla_decode(q_bits, kv_bits, page_table, topk_idx, sm_scale: float, dv: int, seq_lens=None):
    """fp64 sparse attention over the entries the indexer selected (multi-head latent decode).

    Follows "The Indexer O(max_context) Breakthrough", section "Phase 1: The MMA Sparse-MLA
    Decode Kernel" (attention restricted to the top-k cache entries the indexer picked, every
    head reading the same gathered entries) with the head/entry shapes read as stated in the
    design notes.  q [B, H, D] and the paged cache kv [P, E, D] are bf16 bit patterns (D = key
    width; the value is the first dv dims of each entry); topk_idx [B, K] holds C4 positions.
    Position t of request b is kv[page_table[b, t // E], t % E]; an entry is used when
    0 <= t < ceil(seq_lens[b] / 4) (any t >= 0 when seq_lens is None), others (-1 padding)
    are skipped.  For each request and head:
        s_t = sm_scale * q_h . kv_t      over the request's used entries
        o_h = sum_t softmax(s)_t kv_t[:dv],   lse_h = log sum_t exp(s_t)
    A request with no used entry gives o = 0 and lse = -inf.  Also returns
    o_abs = sum_t softmax(s)_t |kv_t[:dv]|, the scale of the rounding in a weighted sum.
    Steps as written: gather, scaled dot products, max-shifted exponentials, normalised sums."""
    q = _bf16_bits_to_f64(q_bits)
    kv_bits = np.asarray(kv_bits)
    table = np.asarray(page_table)
    idx_all = np.asarray(topk_idx)
    B, H, _ = q.shape
    E = kv_bits.shape[1]
    o = np.zeros((B, H, dv))
    o_abs = np.zeros((B, H, dv))
    lse = np.full((B, H), -np.inf)
    for b in range(B):
        idx = idx_all[b].astype(np.int64)
        keep = idx >= 0
        if seq_lens is not None:
            keep &= idx < -(-int(seq_lens[b]) // 4)
        idx = idx[keep]
        if idx.size == 0:
            continue
        rows = _bf16_bits_to_f64(kv_bits[table[b, idx // E], idx % E])  # [n, D]
        s = sm_scale * (q[b] @ rows.T)                                   # [H, n]
        m = s.max(axis=1, keepdims=True)
        p = np.exp(s - m)
        l = p.sum(axis=1, keepdims=True)
        o[b] = (p @ rows[:, :dv]) / l
        o_abs[b] = (p @ np.abs(rows[:, :dv])) / l
        lse[b] = (m + np.log(l))[:, 0]
    return o, lse, o_abs


def _bf16_bits_to_f64(bits) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def case_scores(case) -> np.ndarray:
    return scores(case.q, case.w, case.key_pool, case.page_table, case.seq_lens, case.max_context)


def case_topk(case, rows=None) -> np.ndarray:
    if rows is None:
        rows = case_scores(case)
    return topk(rows, case.seq_lens, case.max_context, case.k)
