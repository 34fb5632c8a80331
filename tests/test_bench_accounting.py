"""The benchmark's byte and operation accounting on the CPU: the algorithmic
bytes behind every GB/s figure and roofline fraction, checked against counts
written out by hand for the workload shapes, and the restated base-3 row rule
against the oracle's."""
from __future__ import annotations

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
import oracle  # noqa: E402
import workloads  # noqa: E402


def layer(M, K, N, x="bf16"):
    return workloads.Layer(M=M, K=K, N=N, w_sigma=0.02, x_dtype=x)


def test_decode_layer_bytes_by_hand():
    L = layer(1, 2560, 6912)
    # X 2560 bf16 + packed W 6912 x 640 + y 6912 fp32 + s + gamma
    assert bench.layer_bytes(L) == 5120 + 4_423_680 + 27_648 + 4 + 4
    # the fused kernel also writes x_q: the figure quoted with the ncu summary
    assert bench.forward_kernel_bytes(L, fused=True) == 4_459_016
    # the forward on x_q reads x_q instead of X
    assert bench.forward_kernel_bytes(L, fused=False) == 4_423_680 + 2560 + 4 + 27_648 + 4


def test_base3_bytes_by_hand():
    L = layer(1, 8192, 28672)
    assert bench.weight_bytes(L, "tq5") == 28672 * 1648  # ceil(8192/5) = 1639 -> 1648
    assert bench.weight_bytes(L, "2bit") == 28672 * 2048
    assert bench.forward_kernel_bytes(L, fused=False, fmt="tq5") == 47_251_456 + 8192 + 4 + 114_688 + 4


@pytest.mark.parametrize("K", [1, 4, 5, 79, 80, 81, 2560, 3200, 6912, 8192, 8640, 28672, 40960])
def test_restated_base3_rule_matches_oracle(K):
    assert bench.tq5_row_bytes(K) == oracle.tq5_row_bytes(K)


def test_prefill_ops_and_metric():
    L = layer(2048, 2560, 6912)
    assert bench.layer_ops(L) == 2 * 2048 * 2560 * 6912  # 72.48 G
    wl = workloads.WORKLOADS["prefill"]
    assert bench.metric_for(wl)[1] == "TOPS"
    assert bench.metric_for(workloads.WORKLOADS["decode"])[1] == "GB/s"


def test_restated_routing_labels():
    # the streaming GEMV serves at most 4 tokens with K <= 32768; the rest go to the GEMM
    assert bench.gemv_fused_layer(layer(1, 28672, 8192))
    assert bench.gemv_fused_layer(layer(4, 2560, 6912))
    assert not bench.gemv_fused_layer(layer(5, 2560, 6912))
    assert not bench.gemv_fused_layer(layer(1, 32768 + 64, 100))
    assert bench.gemm_variant(layer(2048, 2560, 6912), 148) == "gemm_tc_x16_persistent_kernel"
    assert bench.gemm_variant(layer(16, 3200, 8640), 148) == "gemm_f8_kernel"
    assert bench.gemm_variant(layer(64, 3200, 8640), 148) == "gemm_f8_kernel"
    assert bench.gemm_variant(layer(1, 32768 + 64, 100), 148) == "gemm_f8_kernel"
    assert bench.gemm_variant(layer(176, 8192, 28672), 148) == "gemm_f16_sk_kernel"  # 224 tiles: stream-K
    assert bench.gemm_variant(layer(176, 28672, 8192), 148) == "gemm_f16_sk_kernel"


PEAKS = {"hbm_gbs": 6484.9, "bf16_tflops": 1755.4}  # ridge about 270.7 op/B


@pytest.mark.parametrize("M,bound", [(1, "hbm"), (16, "hbm"), (176, "tensor")])
def test_llama70b_layer_bounds_from_intensity(M, bound):
    # 2MNK over about N*K/4 bytes of packed weights: 8 op/B per token, so 1 and
    # 16 tokens (8, 128 op/B) sit below the ridge, 176 tokens (~1400) above it
    for K, N in ((8192, 28672), (28672, 8192)):
        L = layer(M, K, N)
        nbytes = bench.forward_kernel_bytes(L, fused=bench.gemv_fused_layer(L))
        assert bench.layer_bound(bench.layer_ops(L), nbytes, PEAKS) == bound


def test_layer_roofline_hbm_fraction_by_hand():
    L = layer(16, 8192, 28672)
    # 58,720,256 B of packed weights + 16*8192 B of x_q + 64 B of s + 16*28672*4 B of y + 4 B of gamma
    nbytes = 58_720_256 + 131_072 + 64 + 1_835_008 + 4
    e = bench.layer_roofline(L, 20.0, True, "2bit", PEAKS, "measured")
    assert e["algorithmic_bytes"] == nbytes and e["bound"] == "hbm" and e["unit"] == "GB/s"
    assert abs(e["achieved"] - nbytes / 20e-6 / 1e9) < 0.1
    assert abs(e["frac"] - nbytes / 20e-6 / 1e9 / 6484.9) < 1e-4


def test_layer_roofline_tensor_fraction_by_hand():
    L = layer(176, 8192, 28672)
    e = bench.layer_roofline(L, 100.0, True, "2bit", PEAKS, "measured")
    ops = 2 * 176 * 8192 * 28672
    assert e["bound"] == "tensor" and e["unit"] == "TFLOP/s" and e["algorithmic_ops"] == ops
    assert abs(e["achieved"] - ops / 100e-6 / 1e12) < 0.1


def test_default_workload_is_the_largest_single_gpu_config():
    assert bench.DEFAULT_WORKLOAD == "llama70b"
    wl = workloads.WORKLOADS[bench.DEFAULT_WORKLOAD]
    assert {L.M for L in wl.layers} == {1, 16, 176}
    assert bench.metric_for(wl)[1] == "TOPS"
