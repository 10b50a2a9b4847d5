"""The bench's algorithmic work formulas, which the roofline fractions divide by.

Pinned to numbers fixed outside the bench: the record size the library itself
reports (edge0_expert_record_bytes, host code, no GPU needed), the record sizes the
pages' layer shapes give (3 F l / 2 code bytes, one E4M3 scale per 16 weights, three
fp32 globals), and the consistency of the per-stage FLOPs with the per-token total.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


@pytest.mark.parametrize("latent,expected", [(1792, 1_935_360 + 12), (1280, 1_382_400 + 12)])
def test_record_bytes_match_the_layer_shapes(latent, expected):
    assert bench.record_bytes(latent) == expected


@pytest.mark.parametrize("latent", [1792, 1280])
def test_record_bytes_match_the_library(latent):
    import latent_sparse_moe_router_b300 as ext
    assert bench.record_bytes(latent) == ext.lib().edge0_expert_record_bytes(latent, bench.F)


def test_decode_bytes_of_one_145b_token():
    # D and U bf16 [1792][2560], the bf16 router [512][1792], 10 routed records and the
    # shared one, x and y bf16 [1][2560]
    dense = 2 * (1792 * 2560 * 2) + 512 * 1792 * 2
    records = 11 * (1_935_360 + 12)
    assert bench.decode_algorithmic_bytes(1792, 1, 10) == dense + records + 2 * 2560 * 2 == 41_484_420


@pytest.mark.parametrize("latent", [1792, 1280])
def test_stage_flops_add_up_to_the_per_token_total(latent):
    T = 4096
    st = bench.stage_flops(latent, T)
    assert sum(st.values()) == T * bench.flops_per_token_layer(latent)


def test_gate_up_flops_per_launch_at_16k():
    # (T K + T) rows through the gate and up matrices [2F][l], 2 flops per multiply-add
    T, latent = 16384, 1792
    assert bench.stage_flops(latent, T)["gate_up_grouped"] == 2 * (T * 10 + T) * latent * 2 * 640 == 826_781_204_480


def test_grouped_stage_flops_add_up_to_the_per_token_total():
    T, L, G = 4096, 1792, 8
    st = bench.stage_flops(L, T, G)
    assert sum(st.values()) == T * bench.flops_per_token_layer(L, G)
    # D and U of every group: G times the ungrouped projections, the experts unchanged
    one = bench.stage_flops(L, T)
    assert st["u_gemm"] == G * one["u_gemm"] and st["gate_up_grouped"] == one["gate_up_grouped"]
    assert st["xz_gemm"] - 2 * T * L * bench.E == G * (one["xz_gemm"] - 2 * T * L * bench.E)
