"""CPU oracle for int4 weight-only quantization and the bf16 x int4 linear
(and the same affine path with 2- and 8-bit codes, and the linear on
dynamically quantized int8 activations).

TEST INFRASTRUCTURE ONLY.  The test-suite, ``__graft_entry__.smoke()`` and
the CPU-baseline / reference leg of ``bench.py`` are the only callers allowed
to import this package.  The product path (the ``bit_weight_quantization_02_b300``
package and its CUDA library) never imports, links or executes it.

The arithmetic lives in ``w4_oracle.c`` (plain C, IEEE fp32 with contraction
off, fp64 for the linear); this module only builds it with gcc and marshals
numpy arrays.  bf16 tensors travel as ``uint16`` bit patterns.

Pins: every function here is checked by ``tests/test_oracle_pins.py`` against
worked examples derived by hand (``tests/golden/``), exact-arithmetic
invariants, brute force over the 16 codes and an independent fp64 matmul.
Parity unpinned (a reading both sides implement, with nothing in the pages to
check it against): the eps value of the scale clamp, the -0.0 < +0.0 order of
the group minimum, the order of the codes inside a packed byte, and the use of
the full 2^b - 1 levels of the affine path at 2 and 8 bits (the pages name the
widths, not their formulas), and for int8 activations the symmetric range
+-127, the eps clamp of their scale and the per-token variant.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "w4_oracle.c")
_LIB = os.path.join(_HERE, "libw4_oracle.so")
_CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-fPIC", "-shared"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no CUDA involved) and return the .so path."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            p = ctypes.c_void_p
            i64 = ctypes.c_int64
            lib.w4_ref_quantize.argtypes = [p, i64, i64, ctypes.c_int, p, p, p]
            lib.w4_ref_quantize.restype = ctypes.c_int
            lib.w4_ref_dequantize.argtypes = [p, p, p, i64, i64, ctypes.c_int, p]
            lib.w4_ref_dequantize.restype = ctypes.c_int
            lib.w4_ref_linear.argtypes = [p, i64, i64, p, p, p, i64, ctypes.c_int, p]
            lib.w4_ref_linear.restype = ctypes.c_int
            lib.w4_ref_quantize_bits.argtypes = [p, i64, i64, ctypes.c_int, ctypes.c_int, p, p, p]
            lib.w4_ref_quantize_bits.restype = ctypes.c_int
            lib.w4_ref_dequantize_bits.argtypes = [p, p, p, i64, i64, ctypes.c_int, ctypes.c_int, p]
            lib.w4_ref_dequantize_bits.restype = ctypes.c_int
            lib.w4_ref_linear_bits.argtypes = [p, i64, i64, p, p, p, i64, ctypes.c_int, ctypes.c_int, p]
            lib.w4_ref_linear_bits.restype = ctypes.c_int
            lib.w4_ref_eps.argtypes = []
            lib.w4_ref_eps.restype = ctypes.c_float
            lib.w4_ref_linear_bias_bits.argtypes = [p, i64, i64, p, p, p, i64, ctypes.c_int, ctypes.c_int, p, p]
            lib.w4_ref_linear_bias_bits.restype = ctypes.c_int
            lib.w4_ref_quantize_activation_i8.argtypes = [p, i64, i64, ctypes.c_int, p, p]
            lib.w4_ref_quantize_activation_i8.restype = ctypes.c_int
            lib.w4_ref_linear_i8.argtypes = [p, p, ctypes.c_int, i64, i64, p, p, p, i64, ctypes.c_int, p, p]
            lib.w4_ref_linear_i8.restype = ctypes.c_int
            lib.w4_ref_threads.argtypes = [ctypes.c_int]
            lib.w4_ref_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"expected uint16 bf16 bit patterns, got {a.dtype}")
    return a


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def set_threads(n: int) -> int:
    """Threads the oracle's row loops use (n <= 0: every core); returns the count in use.
    Results do not depend on it: each row is computed the same way on any thread."""
    return _load().w4_ref_threads(int(n))


def ref_eps() -> float:
    return float(_load().w4_ref_eps())


def _check_bits(bits: int) -> int:
    if bits not in (2, 4, 8):
        raise ValueError("bits must be 2, 4 or 8")
    return 8 // bits  # codes per byte


def ref_quantize(W: np.ndarray, group_size: int, bits: int = 4):
    """W: uint16 [N,K] bf16 bits -> (Wq uint8 [N,K*bits/8], scales uint16 [N,K/g], offsets uint16 [N,K/g])."""
    per_byte = _check_bits(bits)
    W = _u16(W)
    N, K = W.shape
    if group_size not in (32, 64, 128) or K % group_size:
        raise ValueError("unsupported shape / group size")
    Wq = np.zeros((N, K // per_byte), np.uint8)
    sc = np.zeros((N, K // group_size), np.uint16)
    of = np.zeros((N, K // group_size), np.uint16)
    rc = _load().w4_ref_quantize_bits(_ptr(W), N, K, group_size, bits, _ptr(Wq), _ptr(sc), _ptr(of))
    if rc:
        raise RuntimeError(f"w4_ref_quantize_bits failed: {rc}")
    return Wq, sc, of


def ref_dequantize(Wq: np.ndarray, scales: np.ndarray, offsets: np.ndarray, group_size: int,
                   bits: int = 4) -> np.ndarray:
    """Packed codes + qparams -> uint16 [N,K] bf16 bits of W'."""
    per_byte = _check_bits(bits)
    Wq = np.ascontiguousarray(Wq, dtype=np.uint8)
    scales, offsets = _u16(scales), _u16(offsets)
    N, row_bytes = Wq.shape
    K = per_byte * row_bytes
    out = np.zeros((N, K), np.uint16)
    rc = _load().w4_ref_dequantize_bits(_ptr(Wq), _ptr(scales), _ptr(offsets), N, K, group_size, bits, _ptr(out))
    if rc:
        raise RuntimeError(f"w4_ref_dequantize_bits failed: {rc}")
    return out


def ref_linear(X: np.ndarray, Wq: np.ndarray, scales: np.ndarray, offsets: np.ndarray,
               group_size: int, bits: int = 4, bias: np.ndarray | None = None) -> np.ndarray:
    """X uint16 [M,K] bf16 bits, packed weights of [N,K] -> fp64 [M,N] = X . W'^T (+ bias [N], bf16 bits)."""
    per_byte = _check_bits(bits)
    X = _u16(X)
    Wq = np.ascontiguousarray(Wq, dtype=np.uint8)
    scales, offsets = _u16(scales), _u16(offsets)
    M, K = X.shape
    N = Wq.shape[0]
    if Wq.shape[1] * per_byte != K:
        raise ValueError("X and Wq disagree on K")
    Y = np.zeros((M, N), np.float64)
    if bias is not None:
        bias = _u16(bias)
        if bias.shape != (N,):
            raise ValueError("bias must hold N values")
        rc = _load().w4_ref_linear_bias_bits(_ptr(X), M, K, _ptr(Wq), _ptr(scales), _ptr(offsets), N, group_size,
                                             bits, _ptr(bias), _ptr(Y))
    else:
        rc = _load().w4_ref_linear_bits(_ptr(X), M, K, _ptr(Wq), _ptr(scales), _ptr(offsets), N, group_size, bits,
                                        _ptr(Y))
    if rc:
        raise RuntimeError(f"w4_ref_linear failed: {rc}")
    return Y


def ref_quantize_activation_i8(X: np.ndarray, per_token: bool = False):
    """X uint16 [M,K] bf16 bits -> (Xq int8 [M,K], x_scale float32 [1] per tensor or [M] per token):
    s_x = max|x| / 127 (eps-clamped), q_x = clamp(rne(x / s_x), -127, 127), fp32."""
    X = _u16(X)
    M, K = X.shape
    Xq = np.zeros((M, K), np.int8)
    xs = np.zeros((M if per_token else 1,), np.float32)
    rc = _load().w4_ref_quantize_activation_i8(_ptr(X), M, K, int(bool(per_token)), _ptr(Xq), _ptr(xs))
    if rc:
        raise RuntimeError(f"w4_ref_quantize_activation_i8 failed: {rc}")
    return Xq, xs


def ref_linear_i8(Xq: np.ndarray, x_scale: np.ndarray, per_token: bool, Wq: np.ndarray, scales: np.ndarray,
                  offsets: np.ndarray, group_size: int, bias: np.ndarray | None = None) -> np.ndarray:
    """int8 codes [M,K] with their scale(s), 4-bit weights of [N,K] -> fp64 [M,N]
    = s_x * sum_j (s_j I_j + o_j S_j) (+ bias [N], bf16 bits)."""
    Xq = np.ascontiguousarray(Xq, dtype=np.int8)
    x_scale = np.ascontiguousarray(x_scale, dtype=np.float32)
    Wq = np.ascontiguousarray(Wq, dtype=np.uint8)
    scales, offsets = _u16(scales), _u16(offsets)
    M, K = Xq.shape
    N = Wq.shape[0]
    if Wq.shape[1] * 2 != K:
        raise ValueError("Xq and Wq disagree on K")
    if x_scale.shape != ((M,) if per_token else (1,)):
        raise ValueError("x_scale must hold 1 value per tensor or M per token")
    if bias is not None:
        bias = _u16(bias)
        if bias.shape != (N,):
            raise ValueError("bias must hold N values")
    Y = np.zeros((M, N), np.float64)
    rc = _load().w4_ref_linear_i8(_ptr(Xq), _ptr(x_scale), int(bool(per_token)), M, K, _ptr(Wq), _ptr(scales),
                                  _ptr(offsets), N, group_size, _ptr(bias) if bias is not None else None, _ptr(Y))
    if rc:
        raise RuntimeError(f"w4_ref_linear_i8 failed: {rc}")
    return Y


def bf16_bits_to_f64(a: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp64 (bit placement, no arithmetic)."""
    a = _u16(a)
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def within_linear_tolerance(y: np.ndarray, y_ref: np.ndarray):
    """The linear's acceptance test: |y - y_ref| <= 4e-3 |y_ref| + 1e-2 rms(y_ref),
    rms taken over the whole output of one call.  Returns (ok, worst ratio)."""
    y = np.asarray(y, np.float64)
    y_ref = np.asarray(y_ref, np.float64)
    rms = float(np.sqrt(np.mean(y_ref * y_ref))) if y_ref.size else 0.0
    bound = 4e-3 * np.abs(y_ref) + 1e-2 * rms
    err = np.abs(y - y_ref)
    if y_ref.size == 0:
        return True, 0.0
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(bound > 0, err / bound, np.where(err > 0, np.inf, 0.0))
    worst = float(np.max(ratio))
    return bool(np.all(err <= bound)), worst
