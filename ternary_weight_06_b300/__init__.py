"""BitNet b1.58 BitLinear forward on B300 (sm_103a): Python binding.

A thin ctypes layer over ``libbitlinear.so`` (C ABI in ``include/bitlinear.h``).
Every step of the computation runs in the library's CUDA kernels; this module
only checks tensor metadata, allocates outputs with torch and passes raw
device pointers and the current torch stream.  The library is loaded on first
use; if it is not built (see ``ternary_weight_06_b300.build``) that first call
raises ImportError: there is no fallback.

Functions carry the C names:

* :func:`bitlinear_pack_weights` -- latent fp32 W [N, K] -> (packed uint8 [N, K/4], gamma fp32 [1])
* :func:`bitlinear_quant_act`    -- X bf16/fp32 [M, K]   -> (x_q int8 [M, K], s fp32 [M])
* :func:`bitlinear_forward`      -- packed W, gamma, x_q, s -> y fp32 [M, N] (and int32 acc)
* :func:`bitlinear_forward_ws`, :func:`bitlinear_quant_forward_ws` -- the same with a
  caller workspace (:func:`bitlinear_forward_workspace_bytes`) for the tensor-core path
* :func:`bitlinear_quant_forward_requant_ws` -- the forward with y also quantised to int8 for the next layer
* :func:`bitlinear_rmsnorm_quant_forward_ws` -- the FFN's second BitLinear (RMS norm, quantisation, forward)
* :func:`bitlinear_forward_lut` -- the same product by table lookup (comparison variant)
* :func:`bitlinear_check_device_error`, :func:`bitlinear_status_string`
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "BitLinearError",
    "LIB_PATH",
    "get_lib",
    "bitlinear_pack_weights",
    "bitlinear_pack_workspace_bytes",
    "bitlinear_quant_act",
    "bitlinear_rmsnorm_quant_act",
    "bitlinear_forward",
    "bitlinear_quant_forward",
    "bitlinear_forward_workspace_bytes",
    "bitlinear_forward_ws",
    "bitlinear_quant_forward_ws",
    "bitlinear_rmsnorm_quant_forward_ws",
    "bitlinear_quant_forward_requant_ws",
    "bitlinear_check_device_error",
    "bitlinear_status_string",
    "BITLINEAR_WEIGHTS_RESIDENT",
    "BITLINEAR_TEST_STALL",
    "BITLINEAR_RELU2",
    "bitlinear_tq5_row_bytes",
    "bitlinear_pack_weights_tq5",
    "bitlinear_forward_tq5",
    "bitlinear_forward_lut",
    "EXPORTED_SYMBOLS",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libbitlinear.so")

BL_OK, BL_ERR_INVALID_ARG, BL_ERR_UNSUPPORTED_SHAPE, BL_ERR_MISALIGNED, BL_ERR_WORKSPACE, BL_ERR_CUDA, \
    BL_ERR_TIMEOUT = range(7)
BL_F32, BL_BF16 = 0, 1
BITLINEAR_WEIGHTS_RESIDENT = 1
BITLINEAR_RELU2 = 2  # epilogue writes the squared ReLU of y
BITLINEAR_TEST_STALL = 0x80000000  # test hook: the one-kernel path's bounded waits run out

EXPORTED_SYMBOLS = (
    "bitlinear_pack_workspace_bytes",
    "bitlinear_pack_weights",
    "bitlinear_pack_weights_noalloc",
    "bitlinear_quant_act",
    "bitlinear_rmsnorm_quant_act",
    "bitlinear_forward",
    "bitlinear_quant_forward",
    "bitlinear_forward_workspace_bytes",
    "bitlinear_forward_ws",
    "bitlinear_quant_forward_ws",
    "bitlinear_rmsnorm_quant_forward_ws",
    "bitlinear_quant_forward_requant_ws",
    "bitlinear_tq5_row_bytes",
    "bitlinear_pack_weights_tq5",
    "bitlinear_forward_tq5",
    "bitlinear_forward_lut",
    "bitlinear_check_device_error",
    "bitlinear_status_string",
)


class BitLinearError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {bitlinear_status_string(status)} (status {status})")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with `python -m ternary_weight_06_b300.build` "
                          "(the BitLinear kernels have no non-CUDA fallback)")
    L = ctypes.CDLL(LIB_PATH)
    P, i64, sz, f32, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float, ctypes.c_int
    L.bitlinear_pack_workspace_bytes.argtypes = [i64, i64]
    L.bitlinear_pack_workspace_bytes.restype = sz
    L.bitlinear_pack_weights.argtypes = [P, i64, i64, f32, P, P, P, sz, P]
    L.bitlinear_pack_weights.restype = i32
    L.bitlinear_quant_act.argtypes = [P, i32, i64, i64, P, P, P]
    L.bitlinear_quant_act.restype = i32
    L.bitlinear_rmsnorm_quant_act.argtypes = [P, i32, i64, i64, P, f32, P, P, P]
    L.bitlinear_rmsnorm_quant_act.restype = i32
    L.bitlinear_tq5_row_bytes.argtypes = [i64]
    L.bitlinear_tq5_row_bytes.restype = i64
    L.bitlinear_pack_weights_tq5.argtypes = [P, i64, i64, f32, P, P, P, sz, P]
    L.bitlinear_pack_weights_tq5.restype = i32
    L.bitlinear_forward_tq5.argtypes = [P, P, P, P, i64, i64, i64, P, P, ctypes.c_uint, P]
    L.bitlinear_forward_tq5.restype = i32
    L.bitlinear_forward_lut.argtypes = [P, P, P, P, i64, i64, i64, P, P, ctypes.c_uint, P]
    L.bitlinear_forward_lut.restype = i32
    L.bitlinear_forward.argtypes = [P, P, P, P, i64, i64, i64, P, P, P]
    L.bitlinear_forward.restype = i32
    L.bitlinear_pack_weights_noalloc.argtypes = [P, i64, i64, f32, P, P, P]
    L.bitlinear_pack_weights_noalloc.restype = i32
    L.bitlinear_quant_forward.argtypes = [P, P, P, i32, i64, i64, i64, P, P, P, P, ctypes.c_uint, P]
    L.bitlinear_quant_forward.restype = i32
    L.bitlinear_forward_workspace_bytes.argtypes = [i64, i64, i64]
    L.bitlinear_forward_workspace_bytes.restype = sz
    L.bitlinear_forward_ws.argtypes = [P, P, P, P, i64, i64, i64, P, P, P, sz, P]
    L.bitlinear_forward_ws.restype = i32
    L.bitlinear_quant_forward_ws.argtypes = [P, P, P, i32, i64, i64, i64, P, P, P, P, ctypes.c_uint, P, sz, P]
    L.bitlinear_quant_forward_ws.restype = i32
    L.bitlinear_quant_forward_requant_ws.argtypes = [P, P, P, i32, i64, i64, i64, P, P, P, P, P, ctypes.c_uint, P,
                                                     sz, P]
    L.bitlinear_quant_forward_requant_ws.restype = i32
    L.bitlinear_rmsnorm_quant_forward_ws.argtypes = [P, P, P, i32, i64, i64, i64, P, ctypes.c_float, P, P, P, P,
                                                     ctypes.c_uint, P, sz, P]
    L.bitlinear_rmsnorm_quant_forward_ws.restype = i32
    L.bitlinear_check_device_error.argtypes = [P]
    L.bitlinear_check_device_error.restype = i32
    L.bitlinear_status_string.argtypes = [i32]
    L.bitlinear_status_string.restype = ctypes.c_char_p
    return L


_lib = None


def get_lib() -> ctypes.CDLL:
    """The loaded libbitlinear.so (raises ImportError if it was never built)."""
    global _lib
    if _lib is None:
        _lib = _load()
    return _lib


def bitlinear_status_string(status: int) -> str:
    return get_lib().bitlinear_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != BL_OK:
        raise BitLinearError(status, where)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _dev(t: torch.Tensor, name: str, dtype=None) -> int:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def bitlinear_pack_workspace_bytes(N: int, K: int) -> int:
    return int(get_lib().bitlinear_pack_workspace_bytes(int(N), int(K)))


def bitlinear_pack_weights(W: torch.Tensor, eps: float = 1e-5, W_packed: torch.Tensor | None = None,
                           gamma: torch.Tensor | None = None, workspace: torch.Tensor | None = None, stream=None):
    """Absmean-ternarise and pack latent weights W (fp32 [N, K], K % 4 == 0).
    Returns (W_packed uint8 [N, K/4], gamma fp32 [1]), both on W's device."""
    N, K = W.shape
    if W_packed is None:
        W_packed = torch.empty((N, K // 4), dtype=torch.uint8, device=W.device)
    if gamma is None:
        gamma = torch.empty((1,), dtype=torch.float32, device=W.device)
    ws_bytes = bitlinear_pack_workspace_bytes(N, K)
    if workspace is None:
        workspace = torch.empty((ws_bytes,), dtype=torch.uint8, device=W.device)
    _check(get_lib().bitlinear_pack_weights(_dev(W, "W", torch.float32), N, K, float(eps),
                                      _dev(W_packed, "W_packed", torch.uint8), _dev(gamma, "gamma", torch.float32),
                                      _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
                                      _stream(stream)), "bitlinear_pack_weights")
    return W_packed, gamma


def bitlinear_tq5_row_bytes(K: int) -> int:
    """Bytes per row of the base-3 weight format (five weights per byte)."""
    return int(get_lib().bitlinear_tq5_row_bytes(int(K)))


def bitlinear_pack_weights_tq5(W: torch.Tensor, eps: float = 1e-5, W_tq5: torch.Tensor | None = None,
                               gamma: torch.Tensor | None = None, workspace: torch.Tensor | None = None, stream=None):
    """As :func:`bitlinear_pack_weights`, written five weights per byte in base 3.
    Returns (W_tq5 uint8 [N, bitlinear_tq5_row_bytes(K)], gamma fp32 [1])."""
    N, K = W.shape
    if W_tq5 is None:
        W_tq5 = torch.empty((N, bitlinear_tq5_row_bytes(K)), dtype=torch.uint8, device=W.device)
    if gamma is None:
        gamma = torch.empty((1,), dtype=torch.float32, device=W.device)
    ws_bytes = bitlinear_pack_workspace_bytes(N, K)
    if workspace is None:
        workspace = torch.empty((ws_bytes,), dtype=torch.uint8, device=W.device)
    _check(get_lib().bitlinear_pack_weights_tq5(_dev(W, "W", torch.float32), N, K, float(eps),
                                                _dev(W_tq5, "W_tq5", torch.uint8), _dev(gamma, "gamma", torch.float32),
                                                _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
                                                _stream(stream)), "bitlinear_pack_weights_tq5")
    return W_tq5, gamma


def bitlinear_forward_tq5(W_tq5: torch.Tensor, gamma: torch.Tensor, x_q: torch.Tensor, s: torch.Tensor,
                          y: torch.Tensor | None = None, acc: torch.Tensor | bool | None = None, flags: int = 0,
                          stream=None):
    """:func:`bitlinear_forward` from base-3 packed weights (W_tq5 uint8
    [N, bitlinear_tq5_row_bytes(K)]).  Returns y, or (y, acc) with ``acc``."""
    N, pitch = W_tq5.shape
    M, K = x_q.shape
    if pitch != bitlinear_tq5_row_bytes(K):
        raise ValueError(f"W_tq5 rows have {pitch} bytes but K = {K} needs {bitlinear_tq5_row_bytes(K)}")
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x_q.device)
    want_acc = acc is not None and acc is not False
    if acc is True:
        acc = torch.empty((M, N), dtype=torch.int32, device=x_q.device)
    acc_ptr = _dev(acc, "acc", torch.int32) if want_acc else None
    _check(get_lib().bitlinear_forward_tq5(_dev(W_tq5, "W_tq5", torch.uint8), _dev(gamma, "gamma", torch.float32),
                                           _dev(x_q, "x_q", torch.int8), _dev(s, "s", torch.float32), M, N, K,
                                           _dev(y, "y", torch.float32), acc_ptr, int(flags), _stream(stream)),
           "bitlinear_forward_tq5")
    return (y, acc) if want_acc else y


def bitlinear_forward_lut(W_packed: torch.Tensor, gamma: torch.Tensor, x_q: torch.Tensor, s: torch.Tensor,
                          y: torch.Tensor | None = None, acc: torch.Tensor | bool | None = None, flags: int = 0,
                          stream=None):
    """:func:`bitlinear_forward` computed by table lookup (16-entry tables per
    pair of activations, indexed by nibbles of the packed weights); bit-identical
    results.  Returns y, or (y, acc) with ``acc``."""
    N, kb = W_packed.shape
    M, K = x_q.shape
    if kb * 4 != K:
        raise ValueError(f"W_packed rows have {kb} bytes but K = {K}")
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x_q.device)
    want_acc = acc is not None and acc is not False
    if acc is True:
        acc = torch.empty((M, N), dtype=torch.int32, device=x_q.device)
    acc_ptr = _dev(acc, "acc", torch.int32) if want_acc else None
    _check(get_lib().bitlinear_forward_lut(_dev(W_packed, "W_packed", torch.uint8),
                                           _dev(gamma, "gamma", torch.float32), _dev(x_q, "x_q", torch.int8),
                                           _dev(s, "s", torch.float32), M, N, K, _dev(y, "y", torch.float32), acc_ptr,
                                           int(flags), _stream(stream)), "bitlinear_forward_lut")
    return (y, acc) if want_acc else y


def bitlinear_quant_act(X: torch.Tensor, x_q: torch.Tensor | None = None, s: torch.Tensor | None = None,
                        stream=None):
    """Per-token absmax int8 quantisation of X (bf16 or fp32 [M, K]).
    Returns (x_q int8 [M, K], s fp32 [M])."""
    M, K = X.shape
    if X.dtype == torch.bfloat16:
        dt = BL_BF16
    elif X.dtype == torch.float32:
        dt = BL_F32
    else:
        raise ValueError(f"X must be bf16 or fp32, got {X.dtype}")
    if x_q is None:
        x_q = torch.empty((M, K), dtype=torch.int8, device=X.device)
    if s is None:
        s = torch.empty((M,), dtype=torch.float32, device=X.device)
    _check(get_lib().bitlinear_quant_act(_dev(X, "X"), dt, M, K, _dev(x_q, "x_q", torch.int8),
                                   _dev(s, "s", torch.float32), _stream(stream)), "bitlinear_quant_act")
    return x_q, s


def bitlinear_rmsnorm_quant_act(X: torch.Tensor, gain: torch.Tensor | None = None, eps: float = 1e-5,
                                x_q: torch.Tensor | None = None, s: torch.Tensor | None = None, stream=None):
    """Sub-layer RMS normalisation of X (bf16 or fp32 [M, K]) followed by the
    int8 quantisation of the normalised rows: x_n = fp32(X * gain) /
    fp32(sqrt(mean(X^2) + eps)) with the exact mean of squares, then
    (x_q, s) = bitlinear_quant_act(x_n).  eps > 0.  Returns (x_q int8 [M, K],
    s fp32 [M])."""
    M, K = X.shape
    if X.dtype == torch.bfloat16:
        dt = BL_BF16
    elif X.dtype == torch.float32:
        dt = BL_F32
    else:
        raise ValueError(f"X must be bf16 or fp32, got {X.dtype}")
    if x_q is None:
        x_q = torch.empty((M, K), dtype=torch.int8, device=X.device)
    if s is None:
        s = torch.empty((M,), dtype=torch.float32, device=X.device)
    g_ptr = _dev(gain, "gain", torch.float32) if gain is not None else None
    _check(get_lib().bitlinear_rmsnorm_quant_act(_dev(X, "X"), dt, M, K, g_ptr, float(eps),
                                                 _dev(x_q, "x_q", torch.int8), _dev(s, "s", torch.float32),
                                                 _stream(stream)), "bitlinear_rmsnorm_quant_act")
    return x_q, s


def bitlinear_forward(W_packed: torch.Tensor, gamma: torch.Tensor, x_q: torch.Tensor, s: torch.Tensor,
                      y: torch.Tensor | None = None, acc: torch.Tensor | bool | None = None, stream=None):
    """y = (W_q . x_q) * gamma / s.  W_packed uint8 [N, K/4], x_q int8 [M, K].
    Returns y (fp32 [M, N]); with ``acc=True`` (or an int32 [M, N] tensor)
    returns (y, acc) where acc holds the exact int32 products."""
    N, K4 = W_packed.shape
    M, K = x_q.shape
    if K4 * 4 != K:
        raise ValueError(f"W_packed has K/4 = {K4} but x_q has K = {K}")
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x_q.device)
    want_acc = acc is not None and acc is not False
    if acc is True:
        acc = torch.empty((M, N), dtype=torch.int32, device=x_q.device)
    acc_ptr = _dev(acc, "acc", torch.int32) if want_acc else None
    _check(get_lib().bitlinear_forward(_dev(W_packed, "W_packed", torch.uint8), _dev(gamma, "gamma", torch.float32),
                                 _dev(x_q, "x_q", torch.int8), _dev(s, "s", torch.float32), M, N, K,
                                 _dev(y, "y", torch.float32), acc_ptr, _stream(stream)), "bitlinear_forward")
    return (y, acc) if want_acc else y


def bitlinear_quant_forward(W_packed: torch.Tensor, gamma: torch.Tensor, X: torch.Tensor,
                            y: torch.Tensor | None = None, x_q: torch.Tensor | None = None,
                            s: torch.Tensor | None = None, acc: torch.Tensor | bool | None = None, flags: int = 0,
                            stream=None):
    """Quantise X (bf16/fp32 [M, K]) and apply the BitLinear product in one call
    (one kernel for M <= 4).  Returns (y, x_q, s), or (y, x_q, s, acc) with ``acc``.
    ``flags=BITLINEAR_WEIGHTS_RESIDENT`` lets the kernel stream weights before the
    preceding kernel on the stream finishes; only valid when no pending work on
    the stream writes W_packed or gamma."""
    N, K4 = W_packed.shape
    M, K = X.shape
    if K4 * 4 != K:
        raise ValueError(f"W_packed has K/4 = {K4} but X has K = {K}")
    if X.dtype == torch.bfloat16:
        dt = BL_BF16
    elif X.dtype == torch.float32:
        dt = BL_F32
    else:
        raise ValueError(f"X must be bf16 or fp32, got {X.dtype}")
    dev = X.device
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
    if x_q is None:
        x_q = torch.empty((M, K), dtype=torch.int8, device=dev)
    if s is None:
        s = torch.empty((M,), dtype=torch.float32, device=dev)
    want_acc = acc is not None and acc is not False
    if acc is True:
        acc = torch.empty((M, N), dtype=torch.int32, device=dev)
    acc_ptr = _dev(acc, "acc", torch.int32) if want_acc else None
    _check(get_lib().bitlinear_quant_forward(_dev(W_packed, "W_packed", torch.uint8),
                                             _dev(gamma, "gamma", torch.float32), _dev(X, "X"), dt, M, N, K,
                                             _dev(y, "y", torch.float32), _dev(x_q, "x_q", torch.int8),
                                             _dev(s, "s", torch.float32), acc_ptr, int(flags), _stream(stream)),
           "bitlinear_quant_forward")
    return (y, x_q, s, acc) if want_acc else (y, x_q, s)


def bitlinear_forward_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(get_lib().bitlinear_forward_workspace_bytes(int(M), int(N), int(K)))


def _workspace(M: int, N: int, K: int, workspace, device):
    need = bitlinear_forward_workspace_bytes(M, N, K)
    if workspace is None:
        workspace = torch.empty((max(need, 16),), dtype=torch.uint8, device=device)
    if not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    return workspace.data_ptr(), workspace.numel() * workspace.element_size()


def bitlinear_forward_ws(W_packed: torch.Tensor, gamma: torch.Tensor, x_q: torch.Tensor, s: torch.Tensor,
                         y: torch.Tensor | None = None, acc: torch.Tensor | bool | None = None,
                         workspace: torch.Tensor | None = None, stream=None):
    """:func:`bitlinear_forward` with a workspace of
    ``bitlinear_forward_workspace_bytes(M, N, K)`` bytes (allocated here if not given)."""
    N, K4 = W_packed.shape
    M, K = x_q.shape
    if K4 * 4 != K:
        raise ValueError(f"W_packed has K/4 = {K4} but x_q has K = {K}")
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x_q.device)
    want_acc = acc is not None and acc is not False
    if acc is True:
        acc = torch.empty((M, N), dtype=torch.int32, device=x_q.device)
    acc_ptr = _dev(acc, "acc", torch.int32) if want_acc else None
    ws_ptr, ws_bytes = _workspace(M, N, K, workspace, x_q.device)
    _check(get_lib().bitlinear_forward_ws(_dev(W_packed, "W_packed", torch.uint8), _dev(gamma, "gamma", torch.float32),
                                          _dev(x_q, "x_q", torch.int8), _dev(s, "s", torch.float32), M, N, K,
                                          _dev(y, "y", torch.float32), acc_ptr, ws_ptr, ws_bytes, _stream(stream)),
           "bitlinear_forward_ws")
    return (y, acc) if want_acc else y


def bitlinear_quant_forward_ws(W_packed: torch.Tensor, gamma: torch.Tensor, X: torch.Tensor,
                               y: torch.Tensor | None = None, x_q: torch.Tensor | None = None,
                               s: torch.Tensor | None = None, acc: torch.Tensor | bool | None = None, flags: int = 0,
                               workspace: torch.Tensor | None = None, stream=None):
    """:func:`bitlinear_quant_forward` with a workspace of
    ``bitlinear_forward_workspace_bytes(M, N, K)`` bytes (allocated here if not given)."""
    N, K4 = W_packed.shape
    M, K = X.shape
    if K4 * 4 != K:
        raise ValueError(f"W_packed has K/4 = {K4} but X has K = {K}")
    if X.dtype == torch.bfloat16:
        dt = BL_BF16
    elif X.dtype == torch.float32:
        dt = BL_F32
    else:
        raise ValueError(f"X must be bf16 or fp32, got {X.dtype}")
    dev = X.device
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
    if x_q is None:
        x_q = torch.empty((M, K), dtype=torch.int8, device=dev)
    if s is None:
        s = torch.empty((M,), dtype=torch.float32, device=dev)
    want_acc = acc is not None and acc is not False
    if acc is True:
        acc = torch.empty((M, N), dtype=torch.int32, device=dev)
    acc_ptr = _dev(acc, "acc", torch.int32) if want_acc else None
    ws_ptr, ws_bytes = _workspace(M, N, K, workspace, dev)
    _check(get_lib().bitlinear_quant_forward_ws(_dev(W_packed, "W_packed", torch.uint8),
                                                _dev(gamma, "gamma", torch.float32), _dev(X, "X"), dt, M, N, K,
                                                _dev(y, "y", torch.float32), _dev(x_q, "x_q", torch.int8),
                                                _dev(s, "s", torch.float32), acc_ptr, int(flags), ws_ptr, ws_bytes,
                                                _stream(stream)), "bitlinear_quant_forward_ws")
    return (y, x_q, s, acc) if want_acc else (y, x_q, s)


def bitlinear_quant_forward_requant_ws(W_packed: torch.Tensor, gamma: torch.Tensor, X: torch.Tensor,
                                       y: torch.Tensor | None = None, x_q: torch.Tensor | None = None,
                                       s: torch.Tensor | None = None, y_q: torch.Tensor | None = None,
                                       s_y: torch.Tensor | None = None, flags: int = 0,
                                       workspace: torch.Tensor | None = None, stream=None):
    """:func:`bitlinear_quant_forward_ws` whose output is also quantised for the
    next BitLinear: y_q and s_y are :func:`bitlinear_quant_act` of y, bit for
    bit.  Returns (y, x_q, s, y_q, s_y)."""
    N, K4 = W_packed.shape
    M, K = X.shape
    if K4 * 4 != K:
        raise ValueError(f"W_packed has K/4 = {K4} but X has K = {K}")
    if X.dtype == torch.bfloat16:
        dt = BL_BF16
    elif X.dtype == torch.float32:
        dt = BL_F32
    else:
        raise ValueError(f"X must be bf16 or fp32, got {X.dtype}")
    dev = X.device
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
    if x_q is None:
        x_q = torch.empty((M, K), dtype=torch.int8, device=dev)
    if s is None:
        s = torch.empty((M,), dtype=torch.float32, device=dev)
    if y_q is None:
        y_q = torch.empty((M, N), dtype=torch.int8, device=dev)
    if s_y is None:
        s_y = torch.empty((M,), dtype=torch.float32, device=dev)
    ws_ptr, ws_bytes = _workspace(M, N, K, workspace, dev)
    _check(get_lib().bitlinear_quant_forward_requant_ws(_dev(W_packed, "W_packed", torch.uint8),
                                                        _dev(gamma, "gamma", torch.float32), _dev(X, "X"), dt, M, N,
                                                        K, _dev(y, "y", torch.float32), _dev(x_q, "x_q", torch.int8),
                                                        _dev(s, "s", torch.float32), _dev(y_q, "y_q", torch.int8),
                                                        _dev(s_y, "s_y", torch.float32), int(flags), ws_ptr,
                                                        ws_bytes, _stream(stream)),
           "bitlinear_quant_forward_requant_ws")
    return y, x_q, s, y_q, s_y


def bitlinear_rmsnorm_quant_forward_ws(W_packed: torch.Tensor, gamma: torch.Tensor, X: torch.Tensor,
                                       gain: torch.Tensor | None = None, eps: float = 1e-5,
                                       y: torch.Tensor | None = None, x_q: torch.Tensor | None = None,
                                       s: torch.Tensor | None = None, acc: torch.Tensor | bool | None = None,
                                       flags: int = 0, workspace: torch.Tensor | None = None, stream=None):
    """The FFN's second BitLinear in one call: :func:`bitlinear_rmsnorm_quant_act`
    (sub-layer RMS norm with optional gain, eps > 0) then the forward of
    :func:`bitlinear_forward_ws` on its x_q and s; for more than 4 tokens the
    normalising kernel writes the GEMM's operand itself.  Returns (y, x_q, s)
    or (y, x_q, s, acc)."""
    N, K4 = W_packed.shape
    M, K = X.shape
    if K4 * 4 != K:
        raise ValueError(f"W_packed has K/4 = {K4} but X has K = {K}")
    if X.dtype == torch.bfloat16:
        dt = BL_BF16
    elif X.dtype == torch.float32:
        dt = BL_F32
    else:
        raise ValueError(f"X must be bf16 or fp32, got {X.dtype}")
    if not eps > 0.0:
        raise ValueError("eps must be > 0")
    dev = X.device
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
    if x_q is None:
        x_q = torch.empty((M, K), dtype=torch.int8, device=dev)
    if s is None:
        s = torch.empty((M,), dtype=torch.float32, device=dev)
    want_acc = acc is not None and acc is not False
    if acc is True:
        acc = torch.empty((M, N), dtype=torch.int32, device=dev)
    acc_ptr = _dev(acc, "acc", torch.int32) if want_acc else None
    g_ptr = _dev(gain, "gain", torch.float32) if gain is not None else None
    ws_ptr, ws_bytes = _workspace(M, N, K, workspace, dev)
    _check(get_lib().bitlinear_rmsnorm_quant_forward_ws(_dev(W_packed, "W_packed", torch.uint8),
                                                        _dev(gamma, "gamma", torch.float32), _dev(X, "X"), dt, M, N,
                                                        K, g_ptr, float(eps), _dev(y, "y", torch.float32),
                                                        _dev(x_q, "x_q", torch.int8), _dev(s, "s", torch.float32),
                                                        acc_ptr, int(flags), ws_ptr, ws_bytes, _stream(stream)),
           "bitlinear_rmsnorm_quant_forward_ws")
    return (y, x_q, s, acc) if want_acc else (y, x_q, s)


def bitlinear_check_device_error(stream=None) -> None:
    """Raise BitLinearError if a kernel gave up on a bounded wait (or the stream failed)."""
    _check(get_lib().bitlinear_check_device_error(_stream(stream)), "bitlinear_check_device_error")
