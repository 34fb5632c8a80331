"""Failure detection on the GPU without a fault or a hang.

Every wait of the kernels on an on-chip barrier is bounded: after about two
seconds the kernel records a bit in the library's device error word, abandons
its work without touching the stage, and exits.  The test hook
BITLINEAR_TEST_STALL makes the fused GEMV's producer issue no weight copies,
so its consumers' waits run out; bitlinear_check_device_error must then report
BL_ERR_TIMEOUT, clear the word, and the next call must be correct again.
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


def test_stall_flag_rejected_on_the_multi_kernel_path(bl):
    Wp = torch.zeros((64, 16), dtype=torch.uint8, device="cuda")
    gamma = torch.ones((1,), device="cuda")
    X = torch.zeros((8, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(bl.BitLinearError) as info:
        bl.bitlinear_quant_forward(Wp, gamma, X, flags=bl.BITLINEAR_TEST_STALL)
    assert info.value.status == bl.BL_ERR_INVALID_ARG
