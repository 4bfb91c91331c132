"""Pins of the oracle's fp8 key-cache path (CPU only).

The fp8 cache stores each C4 key as 64 OCP e4m3 codes and one positive fp32
scale, k = scale x e4m3(code).  The decode is pinned to the e4m3 definition's
fixed points and to a library decoder (torch.float8_e4m3fn) over all 256
codes; the fp8 scores are pinned to the bf16-path oracle on keys that e4m3
holds exactly, to scale linearity, and to paging invariants.  Planted slips in
the decode or the scale must fail one of them.
"""
import math
import shutil
import subprocess

import numpy as np
import pytest

from sparse_attention_paged_dsa_gb300 import inputs as I


@pytest.mark.parametrize("code,value", [(0x38, 1.0), (0x40, 2.0), (0x7E, 448.0), (0x01, 2.0 ** -9),
                                        (0x07, 7 * 2.0 ** -9), (0x08, 2.0 ** -6), (0x0F, 1.875 * 2.0 ** -6),
                                        (0xB8, -1.0), (0x00, 0.0), (0x3C, 1.5), (0x47, 3.75)])
def test_e4m3_fixed_points(oracle, code, value):
    assert oracle.e4m3_to_double(code) == value


def test_e4m3_nan_codes_and_negative_zero(oracle):
    assert math.isnan(oracle.e4m3_to_double(0x7F)) and math.isnan(oracle.e4m3_to_double(0xFF))
    z = oracle.e4m3_to_double(0x80)
    assert z == 0.0 and math.copysign(1.0, z) < 0


def test_e4m3_decode_matches_library_decoder(oracle):
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    codes = torch.arange(256, dtype=torch.uint8)
    lib = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = np.array([oracle.e4m3_to_double(c) for c in range(256)])
    nan = np.isnan(lib)
    assert np.array_equal(nan, np.isnan(mine))
    np.testing.assert_array_equal(mine[~nan], lib[~nan])


def _int_case(seed=3):
    return I.make_case(name="fp8pin", batch=3, max_context=2048, seq_lens=[2048, 5, 777], num_pages=48, k=40,
                       seed=seed, key_dist="int")


def test_fp8_scores_equal_bf16_scores_on_exact_keys(oracle):
    """Integer keys in [-4, 4] are exact in e4m3 (scale 1) and as e4m3(k/2) x 2."""
    c = _int_case()
    ref = oracle.case_scores(c)
    f = I.with_fp8_keys(c, scale="one")
    np.testing.assert_array_equal(oracle.case_scores_fp8(f), ref)
    codes = I.f32_to_e4m3_codes(I.bf16_bits_to_f32(c.key_pool) / 2.0)
    halved = oracle.scores_fp8(c.q, c.w, codes, np.full(codes.shape[:2], 2.0, np.float32), c.page_table,
                               c.seq_lens, c.max_context)
    np.testing.assert_array_equal(halved, ref)


def test_fp8_scale_is_linear_and_per_key(oracle):
    c = I.with_fp8_keys(I.make_case(name="lin", batch=2, max_context=1024, seq_lens=[1024, 300], num_pages=12,
                                    k=8, seed=4))
    s1 = oracle.case_scores_fp8(c)
    s2 = oracle.scores_fp8(c.q, c.w, c.key_codes, c.key_scales * np.float32(4.0), c.page_table, c.seq_lens,
                           c.max_context)
    live = np.isfinite(s1)
    np.testing.assert_array_equal(s2[live], 4.0 * s1[live])
    # Changing one key's scale changes that position only.
    sc = c.key_scales.copy()
    page = int(c.page_table[0, 1])
    sc[page, 5] *= np.float32(2.0)
    s3 = oracle.scores_fp8(c.q, c.w, c.key_codes, sc, c.page_table, c.seq_lens, c.max_context)
    diff = np.argwhere(s3 != s1)
    assert [tuple(d) for d in diff] in ([(0, 64 + 5)], [])
    assert s3[0, 64 + 5] == 2.0 * s1[0, 64 + 5]


def test_fp8_gather_reads_scale_times_code(oracle):
    c = I.with_fp8_keys(_int_case(5), scale="absmax")
    n = 200
    g = oracle.gather_fp8(c.key_codes, c.key_scales, c.page_table[0], n)
    pages = c.page_table[0, :(n + 63) // 64]
    expect = (I.e4m3_codes_to_f32(c.key_codes[pages]).astype(np.float64)
              * c.key_scales[pages].astype(np.float64)[..., None]).reshape(-1, I.HEAD_DIM)[:n]
    np.testing.assert_array_equal(g, expect)


def test_fp8_physical_page_permutation_invariance(oracle):
    c = I.with_fp8_keys(I.make_case(name="perm8", batch=3, max_context=1024, seq_lens=[1024, 9, 500],
                                    num_pages=20, k=8, seed=6))
    perm = np.random.default_rng(1).permutation(c.num_pages)
    codes2 = np.empty_like(c.key_codes)
    codes2[perm] = c.key_codes
    sc2 = np.empty_like(c.key_scales)
    sc2[perm] = c.key_scales
    table2 = np.where(c.page_table >= 0, perm[np.maximum(c.page_table, 0)], -1).astype(np.int32)
    np.testing.assert_array_equal(oracle.case_scores_fp8(c),
                                  oracle.scores_fp8(c.q, c.w, codes2, sc2, table2, c.seq_lens, c.max_context))


FP8_MUTATIONS = [
    ("exponent bias 8", "ldexp(1.0 + (double)man / 8.0, exp - 7)", "ldexp(1.0 + (double)man / 8.0, exp - 8)"),
    ("subnormal scale 2^-10", "v = ldexp((double)man, -9);", "v = ldexp((double)man, -10);"),
    ("mantissa over 16", "ldexp(1.0 + (double)man / 8.0", "ldexp(1.0 + (double)man / 16.0"),
    ("scale dropped", "keys_out[t * D + d] = scale * dsa_oracle_e4m3_to_double(src[d]);",
     "keys_out[t * D + d] = dsa_oracle_e4m3_to_double(src[d]);"),
    ("sign dropped", "return sign ? -v : v;", "return v;"),
]


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("label,old,new", FP8_MUTATIONS, ids=[m[0] for m in FP8_MUTATIONS])
def test_planted_fp8_slips_fail_a_pin(tmp_path, label, old, new):
    from oracle import oracle as o
    src = open(o.SRC).read()
    assert src.count(old) == 1, label
    mutated = tmp_path / "mut.c"
    mutated.write_text(src.replace(old, new))
    lib = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", str(mutated), "-o",
                    str(lib), "-lm"], check=True)
    saved_lib, saved_path = o._lib, o.LIB
    try:
        o._lib = None
        o.LIB = str(lib)
        o.build = lambda force=False: str(lib)
        caught = False
        pins = [lambda: [test_e4m3_fixed_points(o, c, v) for c, v in
                         [(0x38, 1.0), (0x40, 2.0), (0x01, 2.0 ** -9), (0x0F, 1.875 * 2.0 ** -6), (0xB8, -1.0)]],
                lambda: test_fp8_scores_equal_bf16_scores_on_exact_keys(o),
                lambda: test_fp8_gather_reads_scale_times_code(o)]
        for pin in pins:
            try:
                pin()
            except (AssertionError, ValueError):
                caught = True
                break
        assert caught, f"planted slip '{label}' passed every pin"
    finally:
        o._lib, o.LIB = saved_lib, saved_path
        import importlib
        importlib.reload(o)
