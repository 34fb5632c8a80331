"""Plain CPU oracle for the BitNet b1.58 BitLinear forward.

TEST INFRASTRUCTURE ONLY.  Only the test-suite, ``__graft_entry__.smoke()`` and
the ``cpu_baseline`` / reference leg of ``bench.py`` may import this package.
The CUDA library never calls it, and it never calls the CUDA library: the two
share no code.

The arithmetic lives in ``bitlinear_oracle.c`` (plain C loops, one IEEE fp32
operation per step, exact integer sums); this module compiles it with gcc on
first use and exposes numpy-level wrappers.  Every function states the reading
of the method it follows; see the C file's header for the list.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bitlinear_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_LIB_OMP_PATH = os.path.join(_BUILD_DIR, "liboracle_omp.so")
_lock = threading.Lock()
_libs = {}

# The activation clamp of reading R4 and the eps of the configurations.
ACT_CLAMP_EPS = np.float32(1e-5)
WEIGHT_EPS = np.float32(1e-5)

_CFLAGS = ["-O2", "-std=gnu11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math", "-fno-builtin-rintf"]


def build(force: bool = False, omp: bool = False) -> str:
    """Compile the oracle shared library (idempotent).  Returns its path.
    omp=True builds the same source with -fopenmp (loops over independent
    outputs on several host threads; identical results)."""
    path = _LIB_OMP_PATH if omp else _LIB_PATH
    with _lock:
        stale = (not os.path.exists(path)) or os.path.getmtime(path) < os.path.getmtime(_SRC)
        if force or stale:
            os.makedirs(_BUILD_DIR, exist_ok=True)
            tmp = path + f".tmp{os.getpid()}"
            extra = ["-fopenmp"] if omp else []
            subprocess.run(["gcc", *_CFLAGS, *extra, _SRC, "-o", tmp, "-lm"], check=True)
            os.replace(tmp, path)
    return path


def _load(omp: bool = False):
    if omp not in _libs:
        lib = ctypes.CDLL(build(omp=omp))
        P = ctypes.c_void_p
        u64, i64 = ctypes.c_uint64, ctypes.c_int64
        lib.oracle_absmean.argtypes = [P, u64]
        lib.oracle_absmean.restype = ctypes.c_float
        lib.oracle_ternarize.argtypes = [P, u64, ctypes.c_float, ctypes.c_float, P]
        lib.oracle_pack.argtypes = [P, u64, P]
        lib.oracle_unpack.argtypes = [P, u64, P]
        lib.oracle_unpack.restype = u64
        lib.oracle_bf16_to_f32.argtypes = [P, u64, P]
        lib.oracle_tq5_row_bytes.argtypes = [i64]
        lib.oracle_tq5_row_bytes.restype = i64
        lib.oracle_pack_tq5.argtypes = [P, i64, i64, P]
        lib.oracle_unpack_tq5.argtypes = [P, i64, i64, P]
        lib.oracle_unpack_tq5.restype = u64
        lib.oracle_quant_act.argtypes = [P, i64, i64, ctypes.c_float, P, P]
        lib.oracle_matmul_int.argtypes = [P, P, i64, i64, i64, P]
        lib.oracle_dequant.argtypes = [P, ctypes.c_float, P, i64, i64, P]
        lib.oracle_rmsnorm_quant_act.argtypes = [P, i64, i64, P, ctypes.c_float, ctypes.c_float, P, P]
        lib.oracle_mean_sq.argtypes = [P, i64]
        lib.oracle_mean_sq.restype = ctypes.c_float
        lib.oracle_relu2.argtypes = [P, i64]
        lib.oracle_forward.argtypes = [P, ctypes.c_float, P, P, i64, i64, i64, P, P]
        lib.oracle_forward.restype = i64
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = ctypes.c_int
        _libs[omp] = lib
    return _libs[omp]


def num_threads(omp: bool = True) -> int:
    """Host threads the oracle's loops use in the OpenMP build (1 otherwise)."""
    return int(_load(omp).oracle_num_threads())


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a: np.ndarray) -> int:
    return a.ctypes.data


def absmean(W: np.ndarray) -> np.float32:
    """gamma = mean|W| (reading R1: exact mean, one RNE rounding to fp32)."""
    W = _c(W, np.float32).reshape(-1)
    if W.size == 0 or W.size > 2**32:
        raise ValueError("absmean needs 1..2^32 values")
    return np.float32(_load().oracle_absmean(_p(W), W.size))


def ternarize(W: np.ndarray, gamma, eps=WEIGHT_EPS) -> np.ndarray:
    """W_q = clip(rint(W / fp32(gamma + eps)), -1, 1) (reading R2)."""
    W = _c(W, np.float32)
    q = np.empty(W.shape, dtype=np.int8)
    _load().oracle_ternarize(_p(W), W.size, float(np.float32(gamma)), float(np.float32(eps)), _p(q))
    return q


def pack(q: np.ndarray) -> np.ndarray:
    """Four ternary codes per byte, least significant first (reading R3).
    q is [N, K] with K % 4 == 0; returns uint8 [N, K/4]."""
    q = _c(q, np.int8)
    if q.shape[-1] % 4:
        raise ValueError("K must be a multiple of 4")
    out = np.empty(q.shape[:-1] + (q.shape[-1] // 4,), dtype=np.uint8)
    _load().oracle_pack(_p(q), q.size, _p(out))
    return out


def unpack(packed: np.ndarray, K: int) -> tuple[np.ndarray, int]:
    """Inverse of :func:`pack`; also returns the count of (invalid) code-3 fields."""
    packed = _c(packed, np.uint8)
    n = packed.size * 4
    q = np.empty(packed.shape[:-1] + (K,), dtype=np.int8)
    if q.size != n:
        raise ValueError("packed size does not match K")
    bad = _load().oracle_unpack(_p(packed), n, _p(q))
    return q, int(bad)


def pack_weights(W: np.ndarray, eps=WEIGHT_EPS) -> tuple[np.ndarray, np.float32]:
    """The whole weight path: gamma, ternarise, pack.  Returns (W_packed, gamma)."""
    g = absmean(W)
    return pack(ternarize(W, g, eps)), g


def tq5_row_bytes(K: int) -> int:
    """Bytes per row of the base-3 format (reading R11): ceil(K/5) rounded up to 16."""
    return int(_load().oracle_tq5_row_bytes(int(K)))


def pack_tq5(q: np.ndarray) -> np.ndarray:
    """Five ternary codes per byte as base-3 digits (reading R11).  q is [N, K];
    returns uint8 [N, tq5_row_bytes(K)]."""
    q = _c(q, np.int8)
    N, K = q.shape
    out = np.empty((N, tq5_row_bytes(K)), dtype=np.uint8)
    _load().oracle_pack_tq5(_p(q), N, K, _p(out))
    return out


def unpack_tq5(packed: np.ndarray, K: int) -> tuple[np.ndarray, int]:
    """Inverse of :func:`pack_tq5`; also returns the count of invalid bytes and
    of padding digits that are not zero codes."""
    packed = _c(packed, np.uint8)
    N, pitch = packed.shape
    if pitch != tq5_row_bytes(K):
        raise ValueError("row pitch does not match K")
    q = np.empty((N, K), dtype=np.int8)
    bad = _load().oracle_unpack_tq5(_p(packed), N, K, _p(q))
    return q, int(bad)


def pack_weights_tq5(W: np.ndarray, eps=WEIGHT_EPS) -> tuple[np.ndarray, np.float32]:
    """gamma, ternarise, base-3 pack.  Returns (W_tq5, gamma)."""
    g = absmean(W)
    return pack_tq5(ternarize(W, g, eps)), g


def forward_tq5(W_tq5: np.ndarray, gamma, x_q: np.ndarray, s: np.ndarray, K: int) -> tuple[np.ndarray, np.ndarray]:
    """Forward pass from base-3 packed weights: decode (R11), exact integer
    product, R6 dequantisation.  Returns (y fp32 [M,N], acc int32 [M,N])."""
    q, bad = unpack_tq5(W_tq5, K)
    if bad:
        raise ValueError(f"{bad} invalid base-3 bytes or padding digits")
    acc = matmul_int(q, x_q)
    return dequant(acc, gamma, s), acc


def bf16_bits_to_f32(x_bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 (given as its uint16 bit patterns) to fp32."""
    x_bits = _c(x_bits, np.uint16)
    out = np.empty(x_bits.shape, dtype=np.float32)
    _load().oracle_bf16_to_f32(_p(x_bits), x_bits.size, _p(out))
    return out


def quant_act(X: np.ndarray, clamp_eps=ACT_CLAMP_EPS, omp: bool = False) -> tuple[np.ndarray, np.ndarray]:
    """Per-token absmax int8 quantisation (readings R4, R5).  X is fp32 [M, K].
    omp=True runs the tokens on several host threads (same results)."""
    X = _c(X, np.float32)
    M, K = X.shape
    xq = np.empty((M, K), dtype=np.int8)
    s = np.empty((M,), dtype=np.float32)
    _load(omp).oracle_quant_act(_p(X), M, K, float(np.float32(clamp_eps)), _p(xq), _p(s))
    return xq, s


def mean_sq(x: np.ndarray) -> np.float32:
    """mean(x^2) of one row: the exact mean of the squares of the fp32 values,
    rounded once to fp32 (reading R9, in the manner of R1)."""
    x = _c(x, np.float32).reshape(-1)
    if x.size == 0:
        raise ValueError("mean_sq needs at least one value")
    return np.float32(_load().oracle_mean_sq(_p(x), x.size))


def rmsnorm_quant_act(X: np.ndarray, gain=None, eps=np.float32(1e-5), clamp_eps=ACT_CLAMP_EPS):
    """Sub-layer RMS normalisation, then the absmax quantisation (reading R9):
    x_n = fp32(fp32(X * gain) / fp32(sqrt(fp32(mean(X^2) + eps)))), then
    (x_q, s) = quant_act(x_n).  eps must be > 0."""
    X = _c(X, np.float32)
    M, K = X.shape
    if not (np.isfinite(eps) and np.float32(eps) > 0):
        raise ValueError("eps must be finite and > 0")
    g = None if gain is None else _c(gain, np.float32)
    if g is not None and g.shape != (K,):
        raise ValueError("gain must have K entries")
    xq = np.empty((M, K), dtype=np.int8)
    s = np.empty((M,), dtype=np.float32)
    _load().oracle_rmsnorm_quant_act(_p(X), M, K, None if g is None else _p(g), float(np.float32(eps)),
                                     float(np.float32(clamp_eps)), _p(xq), _p(s))
    return xq, s


def relu2(y: np.ndarray) -> np.ndarray:
    """Squared ReLU, fp32(max(y, 0)^2) (reading R10).  Returns a new array."""
    out = _c(y, np.float32).copy()
    _load().oracle_relu2(_p(out), out.size)
    return out


def matmul_int(q: np.ndarray, x_q: np.ndarray, omp: bool = False) -> np.ndarray:
    """acc[m, n] = sum_k q[n, k] * x_q[m, k] in exact integer arithmetic."""
    q = _c(q, np.int8)
    x_q = _c(x_q, np.int8)
    N, K = q.shape
    M, K2 = x_q.shape
    if K != K2:
        raise ValueError("K mismatch")
    acc = np.empty((M, N), dtype=np.int32)
    _load(omp).oracle_matmul_int(_p(q), _p(x_q), M, N, K, _p(acc))
    return acc


def dequant(acc: np.ndarray, gamma, s: np.ndarray) -> np.ndarray:
    """y = fp32(fp32(acc) * fp32(gamma / s[m])) (reading R6)."""
    acc = _c(acc, np.int32)
    s = _c(s, np.float32)
    M, N = acc.shape
    y = np.empty((M, N), dtype=np.float32)
    _load().oracle_dequant(_p(acc), float(np.float32(gamma)), _p(s), M, N, _p(y))
    return y


def forward(W_packed: np.ndarray, gamma, x_q: np.ndarray, s: np.ndarray, K: int,
            omp: bool = False) -> tuple[np.ndarray, np.ndarray]:
    """Forward pass from packed weights.  Returns (y fp32 [M,N], acc int32 [M,N]).
    omp=True runs the independent outputs on several host threads (same results)."""
    W_packed = _c(W_packed, np.uint8)
    x_q = _c(x_q, np.int8)
    s = _c(s, np.float32)
    N = W_packed.size * 4 // K
    M = x_q.shape[0]
    if W_packed.size * 4 != N * K or x_q.shape[1] != K or s.shape[0] != M:
        raise ValueError("shape mismatch")
    y = np.empty((M, N), dtype=np.float32)
    acc = np.empty((M, N), dtype=np.int32)
    rc = _load(omp).oracle_forward(_p(W_packed), float(np.float32(gamma)), _p(x_q), _p(s), M, N, K, _p(y), _p(acc))
    if rc < 0:
        raise MemoryError("oracle_forward allocation failed")
    if rc > 0:
        raise ValueError(f"packed weights hold {rc} invalid code-3 fields")
    return y, acc
