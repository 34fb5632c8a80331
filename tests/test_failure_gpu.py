"""Failure detection on the GPU without a fault or a hang.

Every wait of the kernels on an on-chip barrier is bounded: after about two
seconds the kernel records a bit in the library's device error word, abandons
its work, lets the copies it started land, frees its tensor memory and exits.
The test hook BITLINEAR_TEST_STALL makes a kernel start none of the work its
waits depend on (no weight or row copies, or no weight expansion), so the
waits run out; this is done for the fused GEMV, the fp8, stream-K,
persistent and workspace-free tensor-core GEMMs, the staged quantisation and
the base-3 GEMV.  bitlinear_check_device_error must then report
BL_ERR_TIMEOUT, clear the word, no y may have been written, and the next call
must be exact again.
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


def test_bounded_wait_timeout_is_reported_and_cleared(bl):
    rng = np.random.default_rng(3)
    N, K = 300, 1024
    q = rng.integers(-1, 2, size=(N, K)).astype(np.int8)
    Wp = torch.from_numpy(oracle.pack(q)).cuda()
    gamma = torch.tensor([0.02], dtype=torch.float32).cuda()
    X = torch.randn((1, K), generator=torch.Generator().manual_seed(4)).to(torch.bfloat16)
    Xd = X.cuda()
    bl.bitlinear_check_device_error()  # start from a clear error word
    y = torch.full((1, N), 7.0, device="cuda")
    bl.bitlinear_quant_forward(Wp, gamma, Xd, y=y, flags=bl.BITLINEAR_TEST_STALL)
    with pytest.raises(bl.BitLinearError) as info:
        bl.bitlinear_check_device_error()
    assert info.value.status == bl.BL_ERR_TIMEOUT
    assert torch.all(y == 7.0), "a kernel that gave up must not write y"
    bl.bitlinear_check_device_error()  # the word was cleared by the previous check
    # the context is still usable and the next call is exact
    y2, xq, s = bl.bitlinear_quant_forward(Wp, gamma, Xd)
    torch.cuda.synchronize()
    xq_ref, s_ref = oracle.quant_act(X.to(torch.float32).numpy())
    y_ref, _ = oracle.forward(oracle.pack(q), np.float32(0.02), xq_ref, s_ref, K)
    assert np.array_equal(y2.cpu().numpy().view(np.uint32), y_ref.view(np.uint32))
    bl.bitlinear_check_device_error()


def test_stall_flag_rejected_where_there_is_no_hook(bl):
    Wp = torch.zeros((64, 16), dtype=torch.uint8, device="cuda")
    gamma = torch.ones((1,), device="cuda")
    X = torch.zeros((8, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(bl.BitLinearError) as info:
        bl.bitlinear_rmsnorm_quant_forward_ws(Wp, gamma, X, flags=bl.BITLINEAR_TEST_STALL)
    assert info.value.status == bl.BL_ERR_INVALID_ARG


def _stall_then_exact(bl, call, y, y_ref):
    """call(stall) runs the path; with the hook every kernel's bounded wait runs
    out: BL_ERR_TIMEOUT is reported once, y is untouched, and the same call
    without the hook is exact afterwards."""
    bl.bitlinear_check_device_error()  # start from a clear error word
    y.fill_(7.0)
    call(True)
    with pytest.raises(bl.BitLinearError) as info:
        bl.bitlinear_check_device_error()
    assert info.value.status == bl.BL_ERR_TIMEOUT
    assert torch.all(y == 7.0), "a kernel that gave up must not write y"
    bl.bitlinear_check_device_error()  # cleared
    call(False)
    torch.cuda.synchronize()
    assert np.array_equal(y.cpu().numpy().view(np.uint32), y_ref.view(np.uint32))
    bl.bitlinear_check_device_error()


@pytest.mark.parametrize("M,N,K,route", [
    (16, 256, 512, "fp8 GEMM"),
    (100, 512, 1024, "stream-K GEMM"),
    (2048, 4864, 64, "persistent GEMM"),
])
def test_bounded_waits_tensor_core_gemms(bl, M, N, K, route):
    """bitlinear_quant_forward_ws with the stall hook on each tensor-core route"""
    rng = np.random.default_rng(M + N)
    q = rng.integers(-1, 2, size=(N, K)).astype(np.int8)
    p = oracle.pack(q)
    X = torch.randn((M, K), generator=torch.Generator().manual_seed(M)).to(torch.bfloat16)
    xq_ref, s_ref = oracle.quant_act(X.to(torch.float32).numpy())
    y_ref, _ = oracle.forward(p, np.float32(0.02), xq_ref, s_ref, K, omp=True)
    Wp, gamma, Xd = torch.from_numpy(p).cuda(), torch.tensor([0.02]).cuda(), X.cuda()
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    ws = torch.empty((bl.bitlinear_forward_workspace_bytes(M, N, K),), dtype=torch.uint8, device="cuda")

    def call(stall):
        bl.bitlinear_quant_forward_ws(Wp, gamma, Xd, y=y, workspace=ws, flags=bl.BITLINEAR_TEST_STALL if stall else 0)

    _stall_then_exact(bl, call, y, y_ref)


@pytest.mark.parametrize("M", [8, 512])
def test_bounded_waits_quantisation_and_gemm(bl, M):
    """bitlinear_quant_forward with the stall hook: the GEMM without a workspace,
    and from 256 tokens the staged quantisation too"""
    N, K = 384, 1024
    rng = np.random.default_rng(M)
    q = rng.integers(-1, 2, size=(N, K)).astype(np.int8)
    p = oracle.pack(q)
    X = torch.randn((M, K), generator=torch.Generator().manual_seed(M + 1)).to(torch.bfloat16)
    xq_ref, s_ref = oracle.quant_act(X.to(torch.float32).numpy())
    y_ref, _ = oracle.forward(p, np.float32(0.03), xq_ref, s_ref, K, omp=True)
    Wp, gamma, Xd = torch.from_numpy(p).cuda(), torch.tensor([0.03]).cuda(), X.cuda()
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")

    def call(stall):
        bl.bitlinear_quant_forward(Wp, gamma, Xd, y=y, flags=bl.BITLINEAR_TEST_STALL if stall else 0)

    _stall_then_exact(bl, call, y, y_ref)


def test_bounded_waits_base3_gemv(bl):
    """bitlinear_forward_tq5 with the stall hook"""
    N, K = 600, 2560
    rng = np.random.default_rng(5)
    q = rng.integers(-1, 2, size=(N, K)).astype(np.int8)
    W = torch.from_numpy(q.astype(np.float32) * 0.7).cuda()
    Wt, gamma = bl.bitlinear_pack_weights_tq5(W)
    X = torch.randn((1, K), generator=torch.Generator().manual_seed(6)).to(torch.bfloat16).cuda()
    xq, s = bl.bitlinear_quant_act(X)
    torch.cuda.synchronize()
    y_ref, _ = oracle.forward(oracle.pack(q), gamma.cpu().numpy()[0], xq.cpu().numpy(), s.cpu().numpy(), K)
    y = torch.empty((1, N), dtype=torch.float32, device="cuda")

    def call(stall):
        bl.bitlinear_forward_tq5(Wt, gamma, xq, s, y=y, flags=bl.BITLINEAR_TEST_STALL if stall else 0)

    _stall_then_exact(bl, call, y, y_ref)
