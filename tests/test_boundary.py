"""The C-ABI boundary on the CPU: the library builds, loads, exports every
entry point include/bitlinear.h declares, and rejects bad arguments on the
host before anything is launched.  No call here launches anything: every
case fails validation first (the pointers are fake and never dereferenced);
only the workspace-size query asks the runtime for the current device's SM
count, and assumes 256 SMs where there is no device."""
from __future__ import annotations

import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bitlinear.h")


@pytest.fixture(scope="module")
def bl():
    from ternary_weight_06_b300 import build

    build.build()
    import ternary_weight_06_b300 as mod

    return mod


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bitlinear_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("bitlinear_pack_weights", "bitlinear_quant_act", "bitlinear_forward",
                     "bitlinear_quant_forward", "bitlinear_check_device_error", "bitlinear_status_string",
                     "bitlinear_pack_workspace_bytes", "bitlinear_forward_workspace_bytes", "bitlinear_forward_ws",
                     "bitlinear_quant_forward_ws", "bitlinear_rmsnorm_quant_act", "bitlinear_tq5_row_bytes",
                     "bitlinear_pack_weights_tq5", "bitlinear_forward_tq5"):
        assert required in names


def test_library_exports_every_declared_symbol(bl):
    lib = ctypes.CDLL(bl.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in bitlinear.h but not exported"
    assert set(bl.EXPORTED_SYMBOLS) == set(declared_functions())


def test_binding_constants_match_the_header(bl):
    text = open(HEADER).read()
    defines = dict(re.findall(r"#define\s+(BITLINEAR_\w+)\s+(\S+)", text))
    for name in ("BITLINEAR_WEIGHTS_RESIDENT", "BITLINEAR_RELU2", "BITLINEAR_TEST_STALL"):
        assert int(defines[name].rstrip("uU"), 0) == getattr(bl, name), name
    enum = dict(re.findall(r"\b(BL_\w+)\s*=\s*(\d+)", text))
    for name, value in enum.items():
        assert getattr(bl, name) == int(value), name


def test_status_strings(bl):
    for code in range(7):
        s = bl.bitlinear_status_string(code)
        assert s.startswith("BL_")
    assert "unknown" in bl.bitlinear_status_string(99)


def test_workspace_size_is_small_constant(bl):
    assert 272 <= bl.bitlinear_pack_workspace_bytes(8192, 28672) <= 4096
    assert bl.bitlinear_pack_workspace_bytes(1, 4) == bl.bitlinear_pack_workspace_bytes(8192, 28672)


GOOD = 0x10000  # a fake, 64 KiB-aligned address: never dereferenced by these cases


def pack(bl, W=GOOD, N=8, K=64, eps=1e-5, Wp=GOOD, g=GOOD, ws=GOOD, ws_bytes=4096):
    return bl.get_lib().bitlinear_pack_weights(W, N, K, eps, Wp, g, ws, ws_bytes, None)


def test_pack_validation(bl):
    assert pack(bl, W=None) == bl.BL_ERR_INVALID_ARG
    assert pack(bl, Wp=None) == bl.BL_ERR_INVALID_ARG
    assert pack(bl, g=None) == bl.BL_ERR_INVALID_ARG
    assert pack(bl, ws=None) == bl.BL_ERR_INVALID_ARG
    assert pack(bl, N=0) == bl.BL_ERR_INVALID_ARG
    assert pack(bl, K=-4) == bl.BL_ERR_INVALID_ARG
    assert pack(bl, eps=0.0) == bl.BL_ERR_INVALID_ARG
    assert pack(bl, eps=float("nan")) == bl.BL_ERR_INVALID_ARG
    assert pack(bl, eps=float("inf")) == bl.BL_ERR_INVALID_ARG
    assert pack(bl, K=6) == bl.BL_ERR_UNSUPPORTED_SHAPE
    assert pack(bl, N=2**20, K=2**13) == bl.BL_ERR_UNSUPPORTED_SHAPE  # N*K = 2^33 > 2^32
    assert pack(bl, W=GOOD + 4) == bl.BL_ERR_MISALIGNED
    assert pack(bl, Wp=GOOD + 8) == bl.BL_ERR_MISALIGNED
    assert pack(bl, g=GOOD + 2) == bl.BL_ERR_MISALIGNED
    assert pack(bl, ws=GOOD + 8) == bl.BL_ERR_MISALIGNED
    assert pack(bl, ws_bytes=16) == bl.BL_ERR_WORKSPACE


def quant(bl, X=GOOD, dt=1, M=4, K=64, xq=GOOD, s=GOOD):
    return bl.get_lib().bitlinear_quant_act(X, dt, M, K, xq, s, None)


def test_quant_validation(bl):
    assert quant(bl, X=None) == bl.BL_ERR_INVALID_ARG
    assert quant(bl, xq=None) == bl.BL_ERR_INVALID_ARG
    assert quant(bl, s=None) == bl.BL_ERR_INVALID_ARG
    assert quant(bl, M=0) == bl.BL_ERR_INVALID_ARG
    assert quant(bl, K=0) == bl.BL_ERR_INVALID_ARG
    assert quant(bl, dt=7) == bl.BL_ERR_INVALID_ARG
    assert quant(bl, M=2**31) == bl.BL_ERR_UNSUPPORTED_SHAPE
    assert quant(bl, K=2**24 + 1) == bl.BL_ERR_UNSUPPORTED_SHAPE
    assert quant(bl, X=GOOD + 2) == bl.BL_ERR_MISALIGNED
    assert quant(bl, xq=GOOD + 1) == bl.BL_ERR_MISALIGNED
    assert quant(bl, s=GOOD + 2) == bl.BL_ERR_MISALIGNED


def fwd(bl, Wp=GOOD, g=GOOD, xq=GOOD, s=GOOD, M=1, N=16, K=64, y=GOOD, acc=None):
    return bl.get_lib().bitlinear_forward(Wp, g, xq, s, M, N, K, y, acc, None)


def test_forward_validation(bl):
    assert fwd(bl, Wp=None) == bl.BL_ERR_INVALID_ARG
    assert fwd(bl, g=None) == bl.BL_ERR_INVALID_ARG
    assert fwd(bl, xq=None) == bl.BL_ERR_INVALID_ARG
    assert fwd(bl, s=None) == bl.BL_ERR_INVALID_ARG
    assert fwd(bl, y=None) == bl.BL_ERR_INVALID_ARG
    assert fwd(bl, M=0) == bl.BL_ERR_INVALID_ARG
    assert fwd(bl, N=-1) == bl.BL_ERR_INVALID_ARG
    assert fwd(bl, K=0) == bl.BL_ERR_INVALID_ARG
    assert fwd(bl, K=96) == bl.BL_ERR_UNSUPPORTED_SHAPE  # K % 64 != 0
    assert fwd(bl, K=32) == bl.BL_ERR_UNSUPPORTED_SHAPE
    assert fwd(bl, K=131072 + 64) == bl.BL_ERR_UNSUPPORTED_SHAPE
    assert fwd(bl, M=2**31) == bl.BL_ERR_UNSUPPORTED_SHAPE
    assert fwd(bl, N=2**31) == bl.BL_ERR_UNSUPPORTED_SHAPE
    assert fwd(bl, Wp=GOOD + 4) == bl.BL_ERR_MISALIGNED
    assert fwd(bl, xq=GOOD + 8) == bl.BL_ERR_MISALIGNED
    assert fwd(bl, y=GOOD + 4) == bl.BL_ERR_MISALIGNED
    assert fwd(bl, g=GOOD + 1) == bl.BL_ERR_MISALIGNED
    assert fwd(bl, s=GOOD + 2) == bl.BL_ERR_MISALIGNED
    assert fwd(bl, acc=GOOD + 4) == bl.BL_ERR_MISALIGNED


def qfwd(bl, Wp=GOOD, g=GOOD, X=GOOD, dt=1, M=1, N=16, K=64, y=GOOD, xq=GOOD, s=GOOD, acc=None, flags=0):
    return bl.get_lib().bitlinear_quant_forward(Wp, g, X, dt, M, N, K, y, xq, s, acc, flags, None)


def test_quant_forward_validation(bl):
    for kw in ("Wp", "g", "X", "y", "xq", "s"):
        assert qfwd(bl, **{kw: None}) == bl.BL_ERR_INVALID_ARG, kw
    assert qfwd(bl, M=0) == bl.BL_ERR_INVALID_ARG
    assert qfwd(bl, dt=3) == bl.BL_ERR_INVALID_ARG
    assert qfwd(bl, flags=4) == bl.BL_ERR_INVALID_ARG
    assert qfwd(bl, K=96) == bl.BL_ERR_UNSUPPORTED_SHAPE
    assert qfwd(bl, K=131072 + 64) == bl.BL_ERR_UNSUPPORTED_SHAPE
    assert qfwd(bl, X=GOOD + 2) == bl.BL_ERR_MISALIGNED
    assert qfwd(bl, xq=GOOD + 4) == bl.BL_ERR_MISALIGNED
    assert qfwd(bl, s=GOOD + 1) == bl.BL_ERR_MISALIGNED
    assert qfwd(bl, acc=GOOD + 8) == bl.BL_ERR_MISALIGNED


def f8_workspace(M, K, sms):
    """The fp8 GEMM's workspace written out: the e4m3 operand (two rows per
    token of a token tile of M rounded up to 16, K rounded up to 512 bytes
    each), two partial-sum slots per CTA of 128 features x the token tile in
    int32, one arrival counter per CTA, and int32 sums of activations per
    (padded) token over 4096-k chunks, each part rounded up to 256 bytes."""
    up = lambda v: (v + 255) // 256 * 256  # noqa: E731
    ntm = (M + 95) // 96  # token tiles of at most 96
    bn = ((M + ntm - 1) // ntm + 15) // 16 * 16
    kpad = (K + 511) // 512 * 512
    return up(ntm * 2 * bn * kpad) + 2 * sms * bn * 128 * 4 + up(4 * sms) + up(4 * ntm * bn * ((K + 4095) // 4096))


def sk_workspace(M, K, sms):
    """The stream-K fp16 GEMM's workspace written out: the fp16 operand (M x K
    halves), two partial-sum slots per CTA of 128 features x the token tile
    (M split into tiles of at most 192, rounded up to 16) in fp32, and one
    arrival counter per CTA, the first and last part rounded up to 256 bytes."""
    up = lambda v: (v + 255) // 256 * 256  # noqa: E731
    ntm = (M + 191) // 192
    bn = ((M + ntm - 1) // ntm + 15) // 16 * 16
    return up(2 * M * K) + 2 * sms * bn * 128 * 4 + up(4 * sms)


def test_forward_workspace_bytes(bl):
    f = bl.bitlinear_forward_workspace_bytes
    sms = torch.cuda.get_device_properties(0).multi_processor_count if torch.cuda.is_available() else 256
    assert f(1, 6912, 2560) == 0 and f(4, 100, 32768) == 0  # the GEMV path needs none
    assert f(5, 100, 64) == f8_workspace(5, 64, sms)  # up to 64 tokens: the fp8 GEMM
    assert f(64, 100, 2560) == f8_workspace(64, 2560, sms)
    assert f(65, 100, 2560) == sk_workspace(65, 2560, sms)  # more: the stream-K fp16 GEMM
    assert f(176, 8192, 28672) == sk_workspace(176, 28672, sms)
    assert f(2048, 6912, 2560) == sk_workspace(2048, 2560, sms)
    assert f(1, 100, 32768 + 64) == f8_workspace(1, 32768 + 64, sms)  # K beyond the GEMV goes to a GEMM
    assert f(0, 1, 64) == 0


def fwd_ws(bl, M=8, N=16, K=64, ws=GOOD, ws_bytes=1 << 26, **kw):
    args = dict(Wp=GOOD, g=GOOD, xq=GOOD, s=GOOD, y=GOOD, acc=None)
    args.update(kw)
    return bl.get_lib().bitlinear_forward_ws(args["Wp"], args["g"], args["xq"], args["s"], M, N, K, args["y"],
                                             args["acc"], ws, ws_bytes, None)


def qfwd_ws(bl, M=8, N=16, K=64, ws=GOOD, ws_bytes=1 << 26, dt=1, flags=0, **kw):
    args = dict(Wp=GOOD, g=GOOD, X=GOOD, y=GOOD, xq=GOOD, s=GOOD, acc=None)
    args.update(kw)
    return bl.get_lib().bitlinear_quant_forward_ws(args["Wp"], args["g"], args["X"], dt, M, N, K, args["y"],
                                                   args["xq"], args["s"], args["acc"], flags, ws, ws_bytes, None)


def test_forward_ws_validation(bl):
    for kw in ("Wp", "g", "xq", "s", "y"):
        assert fwd_ws(bl, **{kw: None}) == bl.BL_ERR_INVALID_ARG, kw
    assert fwd_ws(bl, M=0) == bl.BL_ERR_INVALID_ARG
    assert fwd_ws(bl, K=96) == bl.BL_ERR_UNSUPPORTED_SHAPE
    assert fwd_ws(bl, Wp=GOOD + 4) == bl.BL_ERR_MISALIGNED
    assert fwd_ws(bl, ws=None) == bl.BL_ERR_WORKSPACE
    assert fwd_ws(bl, ws_bytes=2 * 8 * 64 - 1) == bl.BL_ERR_WORKSPACE
    assert fwd_ws(bl, ws=GOOD + 8) == bl.BL_ERR_MISALIGNED
    for kw in ("Wp", "g", "X", "y", "xq", "s"):
        assert qfwd_ws(bl, **{kw: None}) == bl.BL_ERR_INVALID_ARG, kw
    assert qfwd_ws(bl, dt=3) == bl.BL_ERR_INVALID_ARG
    assert qfwd_ws(bl, flags=4) == bl.BL_ERR_INVALID_ARG
    assert qfwd_ws(bl, X=GOOD + 2) == bl.BL_ERR_MISALIGNED
    assert qfwd_ws(bl, ws=None) == bl.BL_ERR_WORKSPACE
    assert qfwd_ws(bl, ws_bytes=100) == bl.BL_ERR_WORKSPACE
    assert qfwd_ws(bl, ws=GOOD + 4) == bl.BL_ERR_MISALIGNED


def test_rmsnorm_quant_validation(bl):
    f = bl.get_lib().bitlinear_rmsnorm_quant_act
    assert f(None, 1, 2, 64, None, 1e-5, GOOD, GOOD, None) == bl.BL_ERR_INVALID_ARG
    assert f(GOOD, 1, 2, 64, None, 1e-5, None, GOOD, None) == bl.BL_ERR_INVALID_ARG
    assert f(GOOD, 2, 2, 64, None, 1e-5, GOOD, GOOD, None) == bl.BL_ERR_INVALID_ARG  # dtype
    assert f(GOOD, 1, 0, 64, None, 1e-5, GOOD, GOOD, None) == bl.BL_ERR_INVALID_ARG
    assert f(GOOD, 1, 2, 64, None, -1.0, GOOD, GOOD, None) == bl.BL_ERR_INVALID_ARG
    assert f(GOOD, 1, 2, 64, None, float("nan"), GOOD, GOOD, None) == bl.BL_ERR_INVALID_ARG
    assert f(GOOD, 1, 2, 2**24 + 1, None, 1e-5, GOOD, GOOD, None) == bl.BL_ERR_UNSUPPORTED_SHAPE
    assert f(GOOD + 1, 1, 2, 64, None, 1e-5, GOOD, GOOD, None) == bl.BL_ERR_MISALIGNED
    assert f(GOOD + 2, 0, 2, 64, None, 1e-5, GOOD, GOOD, None) == bl.BL_ERR_MISALIGNED  # fp32 needs 4
    assert f(GOOD, 1, 2, 64, GOOD + 2, 1e-5, GOOD, GOOD, None) == bl.BL_ERR_MISALIGNED
    assert qfwd(bl, flags=bl.BITLINEAR_RELU2 | 4) == bl.BL_ERR_INVALID_ARG


def test_tq5_row_bytes(bl):
    f = bl.bitlinear_tq5_row_bytes
    assert [f(K) for K in (0, 1, 5, 80, 81, 2560, 6912, 8192, 28672)] == [0, 16, 16, 16, 32, 512, 1392, 1648, 5744]


def pack_tq5(bl, W=GOOD, N=8, K=64, eps=1e-5, Wt=GOOD, g=GOOD, ws=GOOD, ws_bytes=4096):
    return bl.get_lib().bitlinear_pack_weights_tq5(W, N, K, eps, Wt, g, ws, ws_bytes, None)


def test_pack_tq5_validation(bl):
    for kw in ("W", "Wt", "g", "ws"):
        assert pack_tq5(bl, **{kw: None}) == bl.BL_ERR_INVALID_ARG, kw
    assert pack_tq5(bl, N=0) == bl.BL_ERR_INVALID_ARG
    assert pack_tq5(bl, eps=0.0) == bl.BL_ERR_INVALID_ARG
    assert pack_tq5(bl, eps=float("inf")) == bl.BL_ERR_INVALID_ARG
    assert pack_tq5(bl, K=66) == bl.BL_ERR_UNSUPPORTED_SHAPE
    assert pack_tq5(bl, N=2**20, K=2**13) == bl.BL_ERR_UNSUPPORTED_SHAPE  # N*K > 2^32
    assert pack_tq5(bl, W=GOOD + 4) == bl.BL_ERR_MISALIGNED
    assert pack_tq5(bl, Wt=GOOD + 8) == bl.BL_ERR_MISALIGNED
    assert pack_tq5(bl, ws_bytes=16) == bl.BL_ERR_WORKSPACE


def fwd_tq5(bl, Wt=GOOD, g=GOOD, xq=GOOD, s=GOOD, M=1, N=16, K=64, y=GOOD, acc=None, flags=0):
    return bl.get_lib().bitlinear_forward_tq5(Wt, g, xq, s, M, N, K, y, acc, flags, None)


def test_forward_tq5_validation(bl):
    for kw in ("Wt", "g", "xq", "s", "y"):
        assert fwd_tq5(bl, **{kw: None}) == bl.BL_ERR_INVALID_ARG, kw
    assert fwd_tq5(bl, M=0) == bl.BL_ERR_INVALID_ARG
    assert fwd_tq5(bl, N=0) == bl.BL_ERR_INVALID_ARG
    assert fwd_tq5(bl, flags=bl.BITLINEAR_WEIGHTS_RESIDENT) == bl.BL_ERR_INVALID_ARG
    assert fwd_tq5(bl, K=8) == bl.BL_ERR_UNSUPPORTED_SHAPE
    assert fwd_tq5(bl, K=40960 + 16) == bl.BL_ERR_UNSUPPORTED_SHAPE
    assert fwd_tq5(bl, M=2**31) == bl.BL_ERR_UNSUPPORTED_SHAPE
    assert fwd_tq5(bl, Wt=GOOD + 8) == bl.BL_ERR_MISALIGNED
    assert fwd_tq5(bl, xq=GOOD + 4) == bl.BL_ERR_MISALIGNED
    assert fwd_tq5(bl, y=GOOD + 4) == bl.BL_ERR_MISALIGNED
    assert fwd_tq5(bl, s=GOOD + 2) == bl.BL_ERR_MISALIGNED
    assert fwd_tq5(bl, acc=GOOD + 8) == bl.BL_ERR_MISALIGNED


def test_python_binding_rejects_cpu_tensors(bl):
    import torch

    with pytest.raises(ValueError):
        bl.bitlinear_quant_act(torch.zeros((2, 64), dtype=torch.bfloat16))
    with pytest.raises(ValueError):
        bl.bitlinear_pack_weights(torch.zeros((2, 64), dtype=torch.float32))
