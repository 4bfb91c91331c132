"""Seeded synthetic inputs for the decode-step DSA indexer.

This module only draws and lays out data: the query ``q`` (bf16 bits), the
head weights ``w`` (fp32), the paged C4 index-key pool (bf16 bits), the page
table and the per-request token lengths.  It holds none of the indexer's
arithmetic (no scores, no gather, no selection), so that both the CPU oracle
and the CUDA path can take their inputs from here without sharing any of the
method.

Shapes follow the problem statement of "The Moment of Breakthrough:
Validating the Indexer Fix That Unlocked 17x Throughput on Blackwell"
(section "The Context: A Long Hunt for the Hidden Wall"): one 64-dim key per
4 tokens ("C4"), 256-token pages holding 64 C4 entries, a page table of width
``max_context / 256`` per request, and an output row of ``page_table width x
64`` C4 positions.  Head count 32 and head dim 64 are the leading dims of the
``[32, 262208, 64]`` tensors quoted in "The Indexer O(max_context)
Breakthrough" (section "The Indexer O(max_context) Breakthrough").

Random numbers come from numpy's PCG64 generator, which gives the same
stream on x86 and Arm.  bf16 values are fp32 samples rounded to nearest-even.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

HEADS = 32          # indexer heads
HEAD_DIM = 64       # index-key / query dim
PAGE_TOKENS = 256   # tokens per page
C4 = 4              # tokens per compressed index key
PAGE_ENTRIES = PAGE_TOKENS // C4  # 64 C4 entries per page


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest, ties to even); uint16 bits.

    Inputs are finite samples, so no NaN handling is needed.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bits to fp32 (for building inputs, not scores)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _e4m3_table() -> np.ndarray:
    """Values of the positive finite OCP e4m3 codes 0x00..0x7E (index = code)."""
    vals = np.empty(0x7F, dtype=np.float64)
    for c in range(0x7F):
        e, m = c >> 3, c & 7
        vals[c] = (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


_E4M3 = _e4m3_table()


def f32_to_e4m3_codes(x: np.ndarray) -> np.ndarray:
    """Round to the nearest OCP e4m3 value (ties to the even code), saturating at +-448; uint8 codes."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), 448.0)
    hi = np.clip(np.searchsorted(_E4M3, a, side="left"), 0, 0x7E)
    lo = np.clip(hi - 1, 0, 0x7E)
    d_lo = a - _E4M3[lo]
    d_hi = _E4M3[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    return np.where(np.signbit(x) & (code != 0), code | np.uint8(0x80), code).astype(np.uint8)


def e4m3_codes_to_f32(c: np.ndarray) -> np.ndarray:
    """Exact values of e4m3 codes (no NaN codes expected)."""
    c = np.asarray(c, dtype=np.uint8)
    v = _E4M3[c & 0x7F]
    return np.where(c & 0x80, -v, v).astype(np.float32)


@dataclasses.dataclass
class IndexerCase:
    """One batch of indexer inputs, all host numpy arrays, C-contiguous.

    q          uint16 [B, 32, 64]      bf16 bits of the indexer query
    w          float32 [B, 32]         per-head weights
    key_pool   uint16 [P, 64, 64]      bf16 bits, page-major, entry, dim
    page_table int32 [B, W]            physical page ids (-1 or any id past the live pages)
    seq_lens   int32 [B]               tokens per request
    max_context int                    tokens; W = max_context / 256
    k          int                     top-k
    """

    name: str
    q: np.ndarray
    w: np.ndarray
    key_pool: np.ndarray
    page_table: np.ndarray
    seq_lens: np.ndarray
    max_context: int
    k: int
    seed: int = 0
    key_codes: np.ndarray = None   # uint8 [P, 64, 64] e4m3 codes (fp8 cache), or None
    key_scales: np.ndarray = None  # float32 [P, 64] positive per-key scales (fp8 cache), or None

    @property
    def batch(self) -> int:
        return int(self.q.shape[0])

    @property
    def num_pages(self) -> int:
        return int(self.key_pool.shape[0])

    @property
    def row_width(self) -> int:
        """C4 positions per output row."""
        return self.max_context // C4

    @property
    def table_width(self) -> int:
        return self.max_context // PAGE_TOKENS

    def live_positions(self) -> np.ndarray:
        """C4 entries per request that hold data: tokens/4 rounded up."""
        s = np.clip(self.seq_lens.astype(np.int64), 0, self.max_context)
        return (s + C4 - 1) // C4

    def live_key_bytes(self) -> int:
        return int(self.live_positions().sum()) * HEAD_DIM * 2


def _normal_bf16(rng: np.random.Generator, shape, scale: float = 1.0) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if scale != 1.0:
        x = x * np.float32(scale)
    return f32_to_bf16_bits(x)


def _int_bf16(rng: np.random.Generator, shape, lo: int, hi: int) -> np.ndarray:
    x = rng.integers(lo, hi + 1, size=shape).astype(np.float32)
    return f32_to_bf16_bits(x)


def make_case(
    *,
    name: str,
    batch: int,
    max_context: int,
    seq_lens,
    num_pages: int,
    k: int,
    seed: int,
    dead_fill: str = "neg1",
    key_dist: str = "normal",
    outlier_frac: float = 0.0,
    outlier_scale: float = 8.0,
    page_reuse: bool = False,
) -> IndexerCase:
    """Build a case with disjoint live page slices drawn from a shuffled pool.

    seq_lens     int sequence or array of token counts (length ``batch``)
    dead_fill    "neg1": table entries past the live pages are -1;
                 "random": they hold random valid page ids
    key_dist     "normal" (q, keys ~ N(0,1), w ~ N(0, 1/32)) or "int"
                 (q, keys integers in [-4, 4], w = +-2^-j, j in 1..4: every
                 product and partial sum is exact in fp32)
    outlier_frac each key element is independently scaled by
                 ``outlier_scale`` with this probability
    page_reuse   if the pool is smaller than the live pages, rows wrap around
                 the shuffled pool (pages shared across rows) instead of
                 failing
    """
    assert max_context % PAGE_TOKENS == 0 and max_context > 0
    rng = np.random.default_rng(seed)
    W = max_context // PAGE_TOKENS
    seq = np.asarray(seq_lens, dtype=np.int64).reshape(batch)
    live = (np.clip(seq, 0, max_context) + C4 - 1) // C4
    pages_live = (live + PAGE_ENTRIES - 1) // PAGE_ENTRIES
    total_live_pages = int(pages_live.sum())
    if total_live_pages > num_pages and not page_reuse:
        raise ValueError(f"{name}: {total_live_pages} live pages do not fit a {num_pages}-page pool")

    perm = rng.permutation(num_pages).astype(np.int32)
    table = np.full((batch, W), -1, dtype=np.int32)
    cursor = 0
    for b in range(batch):
        p = int(pages_live[b])
        idx = (np.arange(cursor, cursor + p) % num_pages)
        table[b, :p] = perm[idx]
        cursor += p
    if dead_fill == "random":
        # own stream, so that q, w and the pool are the same as with "neg1"
        dead_rng = np.random.default_rng([seed, 1])
        for b in range(batch):
            p = int(pages_live[b])
            if p < W:
                table[b, p:] = dead_rng.integers(0, num_pages, size=W - p, dtype=np.int32)
    elif dead_fill != "neg1":
        raise ValueError(dead_fill)

    if key_dist == "normal":
        q = _normal_bf16(rng, (batch, HEADS, HEAD_DIM))
        w = (rng.standard_normal(size=(batch, HEADS), dtype=np.float32)
             * np.float32(math.sqrt(1.0 / 32.0))).astype(np.float32)
        pool = _normal_bf16(rng, (num_pages, PAGE_ENTRIES, HEAD_DIM))
    elif key_dist == "int":
        q = _int_bf16(rng, (batch, HEADS, HEAD_DIM), -4, 4)
        j = rng.integers(1, 5, size=(batch, HEADS))
        sgn = np.where(rng.integers(0, 2, size=(batch, HEADS)) == 0, -1.0, 1.0)
        w = (sgn * np.ldexp(1.0, -j)).astype(np.float32)
        pool = _int_bf16(rng, (num_pages, PAGE_ENTRIES, HEAD_DIM), -4, 4)
    else:
        raise ValueError(key_dist)

    if outlier_frac > 0.0:
        mask = rng.random(size=pool.shape) < outlier_frac
        vals = bf16_bits_to_f32(pool)
        vals = np.where(mask, vals * np.float32(outlier_scale), vals)
        pool = f32_to_bf16_bits(vals)

    return IndexerCase(
        name=name,
        q=np.ascontiguousarray(q),
        w=np.ascontiguousarray(w),
        key_pool=np.ascontiguousarray(pool),
        page_table=table,
        seq_lens=seq.astype(np.int32),
        max_context=max_context,
        k=k,
        seed=seed,
    )


def with_fp8_keys(case: IndexerCase, scale: str = "absmax") -> IndexerCase:
    """The same case with an fp8 key cache made from its bf16 keys.

    scale "absmax": each key's scale is max|k| / 448 (1.0 for an all-zero key), codes are
    e4m3(k / scale); scale "one": scale 1.0 and codes e4m3(k) (exact for small integers).
    """
    k = bf16_bits_to_f32(case.key_pool).astype(np.float64)
    if scale == "absmax":
        amax = np.max(np.abs(k), axis=-1)
        sc = np.where(amax > 0, amax / 448.0, 1.0).astype(np.float32)
    elif scale == "one":
        sc = np.ones(k.shape[:-1], dtype=np.float32)
    else:
        raise ValueError(scale)
    codes = f32_to_e4m3_codes(k / sc.astype(np.float64)[..., None])
    return dataclasses.replace(case, name=case.name + "_fp8", key_codes=np.ascontiguousarray(codes),
                               key_scales=np.ascontiguousarray(sc))


def with_next_n(case: IndexerCase, next_n: int, dist: str = "normal") -> IndexerCase:
    """The same keys, table and lengths with next_n query tokens per request.

    q becomes [B, next_n, 32, 64] and w [B, next_n, 32]; the last token keeps the case's own q
    and w, the others are fresh draws from the stream [seed, 2]: q ~ N(0,1) -> bf16 and
    w ~ N(0, 1/32) ("normal"), or integer q in [-4, 4] and w = +-2^-j, j in 1..4 ("int", for
    cases made with key_dist="int").  The request's seq_len counts all next_n tokens."""
    if next_n == 1:
        return dataclasses.replace(case, q=case.q[:, None].copy(), w=case.w[:, None].copy())
    rng = np.random.default_rng([case.seed, 2])
    B = case.batch
    q = np.empty((B, next_n) + case.q.shape[1:], dtype=case.q.dtype)
    w = np.empty((B, next_n) + case.w.shape[1:], dtype=case.w.dtype)
    q[:, -1] = case.q
    w[:, -1] = case.w
    for j in range(next_n - 1):
        if dist == "int":
            q[:, j] = _int_bf16(rng, case.q.shape, -4, 4)
            sgn = rng.choice(np.array([-1.0, 1.0]), size=case.w.shape)
            w[:, j] = (sgn * np.ldexp(1.0, -rng.integers(1, 5, size=case.w.shape))).astype(np.float32)
        else:
            q[:, j] = _normal_bf16(rng, case.q.shape)
            w[:, j] = (rng.standard_normal(case.w.shape) * math.sqrt(1.0 / 32.0)).astype(np.float32)
    return dataclasses.replace(case, name=f"{case.name}_q{next_n}", q=np.ascontiguousarray(q),
                               w=np.ascontiguousarray(w))


# Sparse multi-head latent attention over the selected entries: 64 heads, 576-wide
# cache entries (512 value + 64 rotary dims), paged like the index keys.
MLA_HEADS = 64
MLA_DIM = 576
MLA_DV = 512


@dataclasses.dataclass
class MlaCase:
    """Inputs of one sparse-MLA decode call.

    q          uint16 [B, 64, 576]   bf16 bits of the attention query
    kv         uint16 [P, 64, 576]   bf16 bits of the paged cache (page, entry, dim)
    page_table int32 [B, W]          the indexer case's table
    seq_lens   int32 [B]             tokens per request
    topk       int32 [B, k]          C4 positions, -1 = unused
    sm_scale   float                 softmax scale
    """

    name: str
    q: np.ndarray
    kv: np.ndarray
    page_table: np.ndarray
    seq_lens: np.ndarray
    max_context: int
    topk: np.ndarray
    sm_scale: float

    @property
    def batch(self) -> int:
        return int(self.q.shape[0])


def random_topk(case: IndexerCase, k: int, seed: int) -> np.ndarray:
    """Rows shaped like the indexer's top-k output: min(k, live) distinct live positions per
    request drawn uniformly (stream [seed, 4]), ascending, then -1 padding."""
    rng = np.random.default_rng([seed, 4])
    live = case.live_positions()
    out = np.full((case.batch, k), -1, dtype=np.int32)
    for b in range(case.batch):
        n = int(min(k, live[b]))
        if n:
            out[b, :n] = np.sort(rng.choice(int(live[b]), size=n, replace=False)).astype(np.int32)
    return out


def mla_case(case: IndexerCase, topk=None, *, k: int = None, sm_scale: float = MLA_DIM ** -0.5) -> MlaCase:
    """Sparse-MLA inputs on an indexer case's page table and lengths: q and the cache
    ~ N(0, 1) rounded to bf16 (stream [seed, 3]), one cache page per index-key page.
    topk: given rows (e.g. the indexer's output) or random_topk(case, k or case.k)."""
    rng = np.random.default_rng([case.seed, 3])
    q = _normal_bf16(rng, (case.batch, MLA_HEADS, MLA_DIM))
    kv = np.empty((case.num_pages, PAGE_ENTRIES, MLA_DIM), dtype=np.uint16)
    step = 1024
    for p0 in range(0, case.num_pages, step):  # in chunks: large pools stay within host memory
        p1 = min(case.num_pages, p0 + step)
        kv[p0:p1] = _normal_bf16(rng, (p1 - p0, PAGE_ENTRIES, MLA_DIM))
    if topk is None:
        topk = random_topk(case, k if k is not None else case.k, case.seed)
    return MlaCase(name=case.name + "_mla", q=q, kv=kv, page_table=case.page_table, seq_lens=case.seq_lens,
                   max_context=case.max_context, topk=np.ascontiguousarray(np.asarray(topk, dtype=np.int32)),
                   sm_scale=float(sm_scale))


# The five workloads of the decode indexer, named by what they are.
WORKLOADS = ("b1_ctx8k_seq512", "b16_ctx8k_mixed", "b64_ctx128k_loguniform",
             "b64_ctx1m_seq512", "b64_ctx128k_dense")


def workload(name: str, *, literal_pool: bool = False, dead_fill: str = "neg1") -> IndexerCase:
    """The named synthetic workloads (seed 1000 + 1-based position in WORKLOADS).

    b1_ctx8k_seq512         B=1,  max_context 8192, seq 512, 64-page pool, k=64
    b16_ctx8k_mixed         B=16, max_context 8192, seq ~ U{256..8192}, 1024-page pool, k=2048
    b64_ctx128k_loguniform  B=64, max_context 131072, seq log-uniform in [512, 131072],
                            20000-page pool, k=2048
    b64_ctx1m_seq512        B=64, max_context 1048576, seq 512, 256-page pool, k=2048
    b64_ctx128k_dense       B=64, max_context 131072, seq 131072, keys with 1% x8 outliers,
                            k=2048; 32768 distinct pages (``literal_pool``: an 8192-page pool
                            that every row shares, each page referenced 4 times)
    """
    i = WORKLOADS.index(name) + 1
    seed = 1000 + i
    rng = np.random.default_rng(seed + 7919)  # seq_len draws, separate from the case stream
    if name == "b1_ctx8k_seq512":
        return make_case(name=name, batch=1, max_context=8192, seq_lens=[512], num_pages=64,
                         k=64, seed=seed, dead_fill=dead_fill)
    if name == "b16_ctx8k_mixed":
        seq = rng.integers(256, 8192 + 1, size=16)
        return make_case(name=name, batch=16, max_context=8192, seq_lens=seq, num_pages=1024,
                         k=2048, seed=seed, dead_fill=dead_fill)
    if name == "b64_ctx128k_loguniform":
        seq = np.rint(np.exp(rng.uniform(math.log(512.0), math.log(131072.0), size=64)))
        seq = np.clip(seq, 512, 131072).astype(np.int64)
        return make_case(name=name, batch=64, max_context=131072, seq_lens=seq, num_pages=20000,
                         k=2048, seed=seed, dead_fill=dead_fill)
    if name == "b64_ctx1m_seq512":
        return make_case(name=name, batch=64, max_context=1 << 20, seq_lens=[512] * 64,
                         num_pages=256, k=2048, seed=seed, dead_fill=dead_fill)
    if name == "b64_ctx128k_dense":
        return make_case(name=name, batch=64, max_context=131072, seq_lens=[131072] * 64,
                         num_pages=8192 if literal_pool else 32768, k=2048, seed=seed,
                         dead_fill=dead_fill, outlier_frac=0.01, page_reuse=literal_pool)
    raise KeyError(name)
