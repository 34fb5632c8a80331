"""Live re-ternarisation of changing latent weights (the absmean quantiser
applied while the model trains from scratch: yousumm.com transcript, the
"ABS mean quantizer" paragraph; anthology note-168, "What it does").

Each simulated training step changes the latent fp32 weights; the packed
ternary weights and gamma are then rebuilt from the new values, in place, on
the step's stream.  After every step they must equal the oracle's packing of
the same latent values bit for bit.  (The pages give no backward pass, so no
gradient is modelled: the updates are seeded random changes.)
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bl():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from ternary_weight_06_b300 import build

    build.build()
    import ternary_weight_06_b300 as mod

    return mod


def updates(N, K, steps, seed):
    """Latent weights after each of `steps` seeded updates: small steps, one
    that moves many weights across the zero band, and one that rescales the
    matrix (gamma moves with it)."""
    rng = np.random.default_rng(seed)
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    out = [W.copy()]
    for t in range(steps):
        if t == 1:
            W = (W + (rng.standard_normal((N, K)) * 0.01).astype(np.float32)).astype(np.float32)
        elif t == 2:
            W = (W * np.float32(1.5)).astype(np.float32)
        else:
            W = (W + (rng.standard_normal((N, K)) * 1e-3).astype(np.float32)).astype(np.float32)
        out.append(W.copy())
    return out


@pytest.mark.parametrize("N,K", [(1000, 2560), (257, 8192), (3, 68)])
def test_repack_in_place_after_each_update(bl, N, K):
    ws = torch.empty((bl.bitlinear_pack_workspace_bytes(N, K),), dtype=torch.uint8, device="cuda")
    Wd = torch.empty((N, K), dtype=torch.float32, device="cuda")
    Wp = torch.empty((N, K // 4), dtype=torch.uint8, device="cuda")
    g = torch.empty((1,), dtype=torch.float32, device="cuda")
    prev = None
    for t, W in enumerate(updates(N, K, 4, seed=N + K)):
        Wd.copy_(torch.from_numpy(W))
        bl.bitlinear_pack_weights(Wd, W_packed=Wp, gamma=g, workspace=ws)
        torch.cuda.synchronize()
        p_ref, g_ref = oracle.pack_weights(W)
        assert np.float32(g.item()).view(np.uint32) == np.float32(g_ref).view(np.uint32), t
        got = Wp.cpu().numpy()
        assert np.array_equal(got, p_ref), t
        if prev is not None and N * K > 1000 and t != 3:  # step 3 only rescales: codes may all stay
            assert np.count_nonzero(got != prev) > 0, "an update changed no packed byte"
        prev = got
    bl.bitlinear_check_device_error()


def test_repack_step_replayed_from_a_cuda_graph(bl):
    """The re-pack captured once as a CUDA graph (as a training step would be)
    and replayed after each in-place update of the latent weights."""
    N, K = 512, 4096
    seq = updates(N, K, 3, seed=7)
    Wd = torch.from_numpy(seq[0]).cuda()
    Wp = torch.empty((N, K // 4), dtype=torch.uint8, device="cuda")
    g = torch.empty((1,), dtype=torch.float32, device="cuda")
    ws = torch.empty((bl.bitlinear_pack_workspace_bytes(N, K),), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        bl.bitlinear_pack_weights(Wd, W_packed=Wp, gamma=g, workspace=ws, stream=s)  # warm
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        bl.bitlinear_pack_weights(Wd, W_packed=Wp, gamma=g, workspace=ws, stream=s)
    for W in seq[1:]:
        Wd.copy_(torch.from_numpy(W))
        graph.replay()
        torch.cuda.synchronize()
        p_ref, g_ref = oracle.pack_weights(W)
        assert np.float32(g.item()).view(np.uint32) == np.float32(g_ref).view(np.uint32)
        assert np.array_equal(Wp.cpu().numpy(), p_ref)
    bl.bitlinear_check_device_error()
