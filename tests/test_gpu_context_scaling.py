"""GPU test of the O(actual) property at a fixed capture shape.

Sixty-four 512-token requests cost the fused indexer (no full-width row) at
most 1.2x more with a 1M-token max_context (page table 4096 pages wide, rows of
262144 positions) than with an 8K one (32 pages, 2048 positions): the grid
and the work depend on the live pages, not on max_context.  The pages show the
same property end to end ("The O(Actual) Indexer: Validating 128K Context at
500 tok/s on Blackwell", sections "The Benchmark Results" and "The Reasoning
Process"); the 1.2x bound is the target set for this kernel.
"""
import pytest

pytestmark = pytest.mark.gpu


def test_fused_cost_at_1m_context_within_1p2x_of_8k(gpu_lib):
    import bench
    from sparse_attention_paged_dsa_gb300 import inputs
    r = bench.context_scaling(gpu_lib, inputs, "cuda")
    print(r)
    assert r["ratio_1m_over_8k"] <= 1.2, r
