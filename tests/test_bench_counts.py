"""The benchmark's algorithmic counts (host logic, no GPU): the FLOP and byte figures that the
roofline fractions divide by, checked against the layer's shapes and the values the workload
tables quote."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_prefill_flops_match_the_quoted_totals():
    # Config 3 (T=4096): 828.39 GFLOP in the projections and 206.21 + 137.47 in the causal
    # attention (QK^T over 192 dims, PV over 128), 1,172.07 GFLOP in all.
    gemm, attn = bench.prefill_flops(4096)
    assert gemm == pytest.approx(828.39e9, rel=1e-5)
    assert attn == pytest.approx((206.21 + 137.47) * 1e9, rel=1e-4)
    assert (gemm + attn) == pytest.approx(1172.07e9, rel=1e-5)


def test_chunk_flops_reduce_to_prefill_and_grow_with_the_cache():
    for T in (1, 16, 1000):
        assert bench.chunk_flops(0, T) == bench.prefill_flops(T)
    g0, a0 = bench.chunk_flops(0, 512)
    g1, a1 = bench.chunk_flops(100, 512)
    assert g1 - g0 == 2 * 100 * 512 * 16384            # kv_b_proj over the 100 cached rows
    assert a1 - a0 == 2 * 64 * 512 * 100 * (192 + 128)  # every query also sees 100 more keys


def test_decode_attention_bytes_are_the_latent_rows_and_queries():
    lengths = [1000, 5, 131072]
    assert bench.algorithmic_bytes("decode_attention", 3, lengths) == \
        sum(n + 1 for n in lengths) * 1152 + 3 * 64 * 576 * 2
    # the weight-streaming projections read each FP8 weight byte (and its scales) once
    assert bench.wbytes("o") == 7168 * 8192 + (7168 // 128) * (8192 // 128) * 4
    assert bench.algorithmic_bytes("gemm_o", 1, [1000]) == bench.wbytes("o") + 8192 * 2 + 7168 * 2
