"""The base-3 weight format (five ternary weights per byte, reading R11) on the
GPU, against the oracle: the packing kernel byte for byte, and the forward's
int32 products and y bit for bit."""
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


def layer_shapes():
    """Each distinct (workload, K, N) of the decode-sized workloads once."""
    out, seen = [], set()
    for name in ("tiny", "decode", "skinny", "llama70b"):
        wl = workloads.WORKLOADS[name]
        for i, L in enumerate(wl.layers):
            if (L.K, L.N) not in seen:
                seen.add((L.K, L.N))
                out.append((name, i))
    return out


@pytest.mark.parametrize("wl_name,idx", layer_shapes())
def test_pack_tq5_full_size_bit_exact(bl, wl_name, idx):
    W = workloads.layer_weights(workloads.WORKLOADS[wl_name], idx)
    Wt, g = bl.bitlinear_pack_weights_tq5(W.cuda())
    Wp, g2 = bl.bitlinear_pack_weights(W.cuda())
    torch.cuda.synchronize()
    # gamma and the ternary codes are those of the 2-bit packing: re-encode the
    # GPU's own 2-bit output with the oracle, and compare with the oracle's pack
    q, bad = oracle.unpack(Wp.cpu().numpy(), W.shape[1])
    assert bad == 0
    ref = oracle.pack_tq5(q)
    assert g.item() == g2.item()
    diff = np.count_nonzero(Wt.cpu().numpy() != ref)
    assert diff == 0, f"{diff} base-3 bytes differ"
    if W.numel() <= 20_000_000:  # the oracle's own ternarisation on the smaller matrices
        p5, g5 = oracle.pack_weights_tq5(W.numpy())
        assert np.float32(g.item()) == g5 and np.array_equal(Wt.cpu().numpy(), p5)
    bl.bitlinear_check_device_error()


def forward_case(bl, M, N, K, seed, flags=0, x_extremes=False):
    rng = np.random.default_rng(seed)
    q = rng.integers(-1, 2, size=(N, K)).astype(np.int8)
    if x_extremes:
        q[0] = 1
        q[-1] = -1
    X = rng.standard_normal((M, K)).astype(np.float32)
    if M > 2:
        X[2] = 0.0  # an all-zero token
    if x_extremes:
        X[0] = np.abs(X[0])  # all codes positive: acc reaches 127 * K on row 0
    xq, s = oracle.quant_act(X)
    g = np.float32(0.0273)
    p5 = oracle.pack_tq5(q)
    y_ref, acc_ref = oracle.forward_tq5(p5, g, xq, s, K)
    if flags & bl.BITLINEAR_RELU2:
        y_ref = oracle.relu2(y_ref)
    y, acc = bl.bitlinear_forward_tq5(torch.from_numpy(p5).cuda(), torch.tensor([g]).cuda(),
                                      torch.from_numpy(xq).cuda(), torch.from_numpy(s).cuda(), acc=True, flags=flags)
    torch.cuda.synchronize()
    bad = np.count_nonzero(acc.cpu().numpy() != acc_ref)
    assert bad == 0, f"M={M} N={N} K={K}: {bad} int32 products differ"
    assert np.array_equal(y.cpu().numpy().view(np.uint32), y_ref.view(np.uint32)), f"M={M} N={N} K={K}: y differs"
    bl.bitlinear_check_device_error()
    return q, xq, s, g, y


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 9])
@pytest.mark.parametrize("N,K", [(7, 16), (300, 1024), (999, 6912), (64, 8192), (40, 28672), (16, 40960),
                                 (1, 2560), (150, 80)])
def test_forward_tq5_edge_shapes(bl, M, N, K):
    forward_case(bl, M, N, K, seed=M * 131 + N + K)


@pytest.mark.parametrize("M,N,K", [(1, 6912, 2560), (1, 2560, 6912), (1, 28672, 8192), (1, 8192, 28672),
                                   (4, 8640, 3200)])
def test_forward_tq5_full_size(bl, M, N, K):
    forward_case(bl, M, N, K, seed=N + K, x_extremes=True)


@pytest.mark.parametrize("M", [1, 4, 6])
def test_forward_tq5_relu2(bl, M):
    forward_case(bl, M, 513, 2560, seed=M, flags=bl.BITLINEAR_RELU2)


@pytest.mark.parametrize("M,N,K", [(1, 6912, 2560), (3, 999, 6912)])
def test_forward_tq5_equals_two_bit_forward(bl, M, N, K):
    """the two weight formats give the same y bit for bit on the GPU"""
    q, xq, s, g, y5 = forward_case(bl, M, N, K, seed=7 + M)
    y2 = bl.bitlinear_forward(torch.from_numpy(oracle.pack(q)).cuda(), torch.tensor([g]).cuda(),
                              torch.from_numpy(xq).cuda(), torch.from_numpy(s).cuda())
    torch.cuda.synchronize()
    assert torch.equal(y5.view(torch.int32), y2.view(torch.int32))
