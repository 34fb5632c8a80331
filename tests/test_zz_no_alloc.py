"""The allocation-free packing entry point, through the C ABI.

bitlinear_pack_weights_noalloc serves callers that cannot give the library
device memory (an application whose device memory belongs to its own pool
allocator, plug-in hosts that only pass pointers): it keeps its workspace in
a fixed array in the library's device image.  Its output must equal
bitlinear_pack_weights' output exactly (the tolerance of every packing test
here: bit-exact bytes and gamma), on two calls in a row, because the shared
array keeps the previous call's contents and must be cleared by each call;
the small matrix is also checked against the CPU oracle.  This file is
collected last on purpose: if it fails, a run that stops at the first failure
has already run every other test.
"""
from __future__ import annotations

import ctypes

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


def pack_noalloc(bl, W: torch.Tensor, eps: float = 1e-5):
    N, K = W.shape
    Wp = torch.empty((N, K // 4), dtype=torch.uint8, device=W.device)
    g = torch.empty((1,), dtype=torch.float32, device=W.device)
    stream = torch.cuda.current_stream().cuda_stream
    st = bl.get_lib().bitlinear_pack_weights_noalloc(ctypes.c_void_p(W.data_ptr()), N, K, ctypes.c_float(eps),
                                                    ctypes.c_void_p(Wp.data_ptr()), ctypes.c_void_p(g.data_ptr()),
                                                    ctypes.c_void_p(stream))
    assert st == 0, bl.bitlinear_status_string(st)
    return Wp, g


def test_noalloc_pack_matches_pack_twice_in_a_row(bl):
    gen = torch.Generator().manual_seed(2024)
    # two different matrices back to back: the second call must not see the
    # first call's sums left in the shared array
    mats = [torch.randn((1000, 2560), generator=gen) * 0.02, torch.randn((777, 68), generator=gen) * 3.0]
    for W_cpu in mats:
        W = W_cpu.cuda()
        ref_p, ref_g = bl.bitlinear_pack_weights(W)
        got_p, got_g = pack_noalloc(bl, W)
        torch.cuda.synchronize()
        assert torch.equal(got_p, ref_p)
        assert np.float32(got_g.item()).view(np.uint32) == np.float32(ref_g.item()).view(np.uint32)
    p_or, g_or = oracle.pack_weights(mats[1].numpy())
    assert np.array_equal(got_p.cpu().numpy(), p_or)
    assert np.float32(got_g.item()).view(np.uint32) == np.float32(g_or).view(np.uint32)
    bl.bitlinear_check_device_error()


def test_noalloc_pack_rejects_bad_arguments(bl):
    lib = bl.get_lib()
    good = ctypes.c_void_p(0x10000)
    assert lib.bitlinear_pack_weights_noalloc(None, 4, 64, 1e-5, good, good, None) == bl.BL_ERR_INVALID_ARG
    assert lib.bitlinear_pack_weights_noalloc(good, 4, 66, 1e-5, good, good, None) == bl.BL_ERR_UNSUPPORTED_SHAPE
    assert lib.bitlinear_pack_weights_noalloc(good, 2**20, 2**13, 1e-5, good, good, None) == \
        bl.BL_ERR_UNSUPPORTED_SHAPE
    # W and W_packed need 16-byte alignment, gamma 4-byte: checked before anything is launched
    odd = ctypes.c_void_p(0x10008)
    assert lib.bitlinear_pack_weights_noalloc(odd, 4, 64, 1e-5, good, good, None) == bl.BL_ERR_MISALIGNED
    assert lib.bitlinear_pack_weights_noalloc(good, 4, 64, 1e-5, odd, good, None) == bl.BL_ERR_MISALIGNED
    assert lib.bitlinear_pack_weights_noalloc(good, 4, 64, 1e-5, good, ctypes.c_void_p(0x10002), None) == \
        bl.BL_ERR_MISALIGNED
    assert lib.bitlinear_pack_weights_noalloc(good, 4, 64, 0.0, good, good, None) == bl.BL_ERR_INVALID_ARG
