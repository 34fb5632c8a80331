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
    assert bench.gemm_variant(layer(16, 3200, 8640), 148).startswith("gemm_tc_x16_kernel")
