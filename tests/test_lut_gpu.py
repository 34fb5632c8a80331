"""The lookup-table GEMV (the table approach of the CPU kernels behind BitNet
b1.58: promptinjection.net, "4. GPU Support: The Fragile Boost") against the
CPU oracle: int32 accumulators and y bit-exact, on the decode and 70B-class
one-token layers, ragged shapes, several tokens, K over several table
slices, extreme magnitudes and the squared-ReLU epilogue."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bl():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from ternary_weight_06_b300 import build

    build.build()
    import ternary_weight_06_b300 as mod

    return mod


def lut_case(bl, p, g, xq, s, K, where, flags=0):
    y, acc = bl.bitlinear_forward_lut(torch.from_numpy(p).cuda(), torch.tensor([g], dtype=torch.float32).cuda(),
                                      torch.from_numpy(xq).cuda(), torch.from_numpy(s).cuda(), acc=True, flags=flags)
    torch.cuda.synchronize()
    y_ref, acc_ref = oracle.forward(p, g, xq, s, K, omp=True)
    if flags:
        y_ref = oracle.relu2(y_ref)
    bad = np.count_nonzero(acc.cpu().numpy() != acc_ref)
    assert bad == 0, f"{where}: {bad} accumulators differ"
    assert np.array_equal(y.cpu().numpy().view(np.uint32), y_ref.view(np.uint32)), where
    bl.bitlinear_check_device_error()


@pytest.mark.parametrize("wl_name,idx", [("decode", 0), ("decode", 1), ("llama70b", 0), ("llama70b", 1),
                                         ("skinny", 0), ("skinny", 1)])
def test_lut_full_size_layers(bl, wl_name, idx):
    wl = workloads.WORKLOADS[wl_name]
    L = wl.layers[idx]
    p, g = oracle.pack_weights(workloads.layer_weights(wl, idx).numpy())
    xq, s = oracle.quant_act(workloads.x_as_f32_numpy(workloads.layer_activations(wl, idx)))
    lut_case(bl, p, g, xq, s, L.K, f"{wl_name}[{idx}]")


@pytest.mark.parametrize("M,N,K", [(1, 1, 64), (1, 13, 128), (2, 255, 576), (3, 1000, 2560), (4, 777, 8192 + 64),
                                   (1, 130, 3 * 8192 + 128), (5, 64, 640), (1, 40, 131072)])
def test_lut_edge_shapes(bl, M, N, K):
    rng = np.random.default_rng(M * 100 + N + K)
    q = rng.integers(-1, 2, size=(N, K)).astype(np.int8)
    xq = rng.integers(-128, 128, size=(M, K)).astype(np.int8)
    s = rng.uniform(0.5, 300, size=M).astype(np.float32)
    lut_case(bl, oracle.pack(q), np.float32(0.0123), xq, s, K, f"lut M={M} N={N} K={K}")


@pytest.mark.parametrize("K", [8192, 131072])
def test_lut_extreme_magnitudes(bl, K):
    # rows of +1, -1 and alternating signs against +127 / -128 activations: |acc| up to 128 K
    N, M = 300, 2
    q = np.ones((N, K), np.int8)
    q[1::3] = -1
    q[2::3, 1::2] = -1
    xq = np.full((M, K), 127, np.int8)
    xq[1] = -128
    lut_case(bl, oracle.pack(q), np.float32(1.0), xq, np.ones((M,), np.float32), K, f"lut extreme K={K}")


def test_lut_relu2_and_equals_conditional_add_gemv(bl):
    rng = np.random.default_rng(5)
    N, K = 2000, 6912
    p = oracle.pack(rng.integers(-1, 2, size=(N, K)).astype(np.int8))
    xq = rng.integers(-127, 128, size=(1, K)).astype(np.int8)
    s = np.array([37.5], np.float32)
    lut_case(bl, p, np.float32(0.02), xq, s, K, "lut relu2", flags=bl.BITLINEAR_RELU2)
    args = (torch.from_numpy(p).cuda(), torch.tensor([0.02]).cuda(), torch.from_numpy(xq).cuda(),
            torch.from_numpy(s).cuda())
    assert torch.equal(bl.bitlinear_forward_lut(*args), bl.bitlinear_forward(*args))
