"""libw4: int4 weight-only quantization and the bf16 x int4 linear on B300
(and the same affine path with 2- and 8-bit codes: ``w4_*_bits``).

Thin Python binding over the C ABI in ``include/w4.h``.  The functions keep
the C names (``w4_quantize``, ``w4_dequantize``, ``w4_linear`` ...); they only
marshal arguments: torch allocates the outputs and the workspace on the
tensors' device, and every step of the computation runs in the CUDA kernels
of ``libw4.so``.  There is no CPU fallback: if the library is missing or fails
to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = [
    "W4Error", "W4_FORMAT_VERSION", "KERNEL_AUTO", "KERNEL_SKINNY", "KERNEL_GEMM", "KERNEL_SKINNY_CLUSTER",
    "KERNEL_STREAM", "KERNEL_PAIR", "KERNEL_TC_DECODE", "Workspace", "w4_linear_workspace_bytes", "Repacked", "w4_repacked_bytes", "w4_repack",
    "w4_linear_repacked",
    "library_path", "load_library", "w4_quantize", "w4_dequantize", "w4_linear",
    "w4_linear_ex", "w4_packed_bytes", "w4_qparam_bytes", "w4_device_fault", "w4_format_version",
    "w4_linear_static", "w4_linear_bias", "w4_packed_bytes_bits", "w4_quantize_bits", "w4_dequantize_bits", "w4_linear_bits",
    "w4_quantize_activation_i8", "w4_linear_i8", "w4_linear_i8_workspace_bytes", "w4_linear_i8_dynamic",
    "w4_linear_i8_dynamic_workspace_bytes",
]

W4_FORMAT_VERSION = 1
KERNEL_AUTO, KERNEL_SKINNY, KERNEL_GEMM, KERNEL_SKINNY_CLUSTER, KERNEL_STREAM, KERNEL_PAIR, KERNEL_TC_DECODE = (
    0, 1, 2, 3, 4, 5, 6)
_STATUS = {0: "W4_OK", 1: "W4_ERR_INVALID_ARG", 2: "W4_ERR_UNSUPPORTED", 3: "W4_ERR_MISALIGNED",
           4: "W4_ERR_CUDA", 5: "W4_ERR_TIMEOUT"}

_HERE = os.path.dirname(os.path.abspath(__file__))
_lock = threading.Lock()
_lib = None


class W4Error(RuntimeError):
    def __init__(self, status: int, call: str, detail: str):
        self.status = status
        super().__init__(f"{call} failed: {_STATUS.get(status, status)}: {detail}")


def library_path() -> str:
    return os.path.join(_HERE, "libw4.so")


def load_library():
    """Load libw4.so (built in-tree by ``_build.build()``); raise if it is absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"libw4.so not found at {path}: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(path)
        p, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
        sigs = {
            "w4_quantize": ([p, i64, i64, i32, p, p, p, p], i32),
            "w4_dequantize": ([p, p, p, i64, i64, i32, p, p], i32),
            "w4_linear_workspace_bytes": ([i64, i64, i64, i32], sz),
            "w4_linear": ([p, i64, i64, p, p, p, i64, i32, p, p, sz, p], i32),
            "w4_linear_ex": ([p, i64, i64, p, p, p, i64, i32, p, p, sz, i32, p], i32),
            "w4_packed_bytes": ([i64, i64], sz),
            "w4_qparam_bytes": ([i64, i64, i32], sz),
            "w4_device_fault": ([p], i32),
            "w4_status_string": ([i32], ctypes.c_char_p),
            "w4_last_error_detail": ([], ctypes.c_char_p),
            "w4_format_version": ([], i32),
            "w4_linear_static": ([p, i64, i64, p, p, p, i64, i32, p, p], i32),
            "w4_repacked_bytes": ([i64, i64, i32], sz),
            "w4_repack": ([p, p, p, i64, i64, i32, p, p], i32),
            "w4_linear_repacked": ([p, i64, i64, p, i64, i32, p, p, sz, p], i32),
            "w4_packed_bytes_bits": ([i64, i64, i32], sz),
            "w4_quantize_bits": ([p, i64, i64, i32, i32, p, p, p, p], i32),
            "w4_dequantize_bits": ([p, p, p, i64, i64, i32, i32, p, p], i32),
            "w4_linear_bits": ([p, i64, i64, p, p, p, i64, i32, i32, p, p, sz, p], i32),
            "w4_selftest_bounded_waits": ([p, sz, p, ctypes.c_uint64, p], i32),
            "w4_linear_bias": ([p, i64, i64, p, p, p, i64, i32, p, p, p, sz, p], i32),
            "w4_linear_bias_ex": ([p, i64, i64, p, p, p, i64, i32, p, p, p, sz, i32, p], i32),
            "w4_quantize_activation_workspace_bytes": ([i64, i64, i32], sz),
            "w4_quantize_activation_i8": ([p, i64, i64, i32, p, p, p, sz, p], i32),
            "w4_linear_i8_workspace_bytes": ([i64, i64, i64, i32], sz),
            "w4_linear_i8": ([p, p, i32, i64, i64, p, p, p, i64, i32, p, p, p, sz, p], i32),
            "w4_linear_i8_dynamic_workspace_bytes": ([i64, i64, i64, i32], sz),
            "w4_linear_i8_dynamic": ([p, i32, i64, i64, p, p, p, i64, i32, p, p, p, sz, p], i32),
        }
        for name, (args, res) in sigs.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        if lib.w4_format_version() != W4_FORMAT_VERSION:
            raise RuntimeError("libw4.so format version does not match the binding")
        _lib = lib
        return lib


def _check(status: int, call: str):
    if status != 0:
        detail = load_library().w4_last_error_detail()
        raise W4Error(status, call, detail.decode() if detail else "")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(t: torch.Tensor):
    if t.device.type != "cuda":
        raise ValueError("libw4 works on CUDA tensors only (there is no CPU path)")
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _bits16(t: torch.Tensor, name: str) -> torch.Tensor:
    if t.dtype not in (torch.bfloat16, torch.int16, torch.uint16):
        raise TypeError(f"{name} must be bf16 (or its 16-bit pattern), got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def w4_packed_bytes(N: int, K: int) -> int:
    return load_library().w4_packed_bytes(N, K)


def w4_qparam_bytes(N: int, K: int, group_size: int) -> int:
    return load_library().w4_qparam_bytes(N, K, group_size)


def w4_format_version() -> int:
    return load_library().w4_format_version()


def w4_quantize(W: torch.Tensor, group_size: int, out=None):
    """W bf16 [N,K] (CUDA) -> (Wq uint8 [N,K/2], scales bf16 [N,K/g], offsets bf16 [N,K/g])."""
    lib = load_library()
    _bits16(W, "W")
    N, K = W.shape
    if out is None:
        ng = K // group_size if group_size and K % group_size == 0 else 0
        Wq = torch.empty((N, K // 2), dtype=torch.uint8, device=W.device)
        sc = torch.empty((N, ng), dtype=torch.bfloat16, device=W.device)
        of = torch.empty((N, ng), dtype=torch.bfloat16, device=W.device)
    else:
        Wq, sc, of = out
    _check(lib.w4_quantize(_ptr(W), N, K, group_size, _ptr(Wq), _ptr(sc), _ptr(of), _stream(W)), "w4_quantize")
    return Wq, sc, of


def w4_dequantize(Wq: torch.Tensor, scales: torch.Tensor, offsets: torch.Tensor, group_size: int, out=None):
    """Packed int4 weights -> bf16 [N,K]."""
    lib = load_library()
    N, half = Wq.shape
    K = 2 * half
    W = out if out is not None else torch.empty((N, K), dtype=torch.bfloat16, device=Wq.device)
    _check(lib.w4_dequantize(_ptr(Wq), _ptr(scales), _ptr(offsets), N, K, group_size, _ptr(W), _stream(Wq)),
           "w4_dequantize")
    return W


def w4_packed_bytes_bits(N: int, K: int, bits: int) -> int:
    return load_library().w4_packed_bytes_bits(N, K, bits)


def w4_quantize_bits(W: torch.Tensor, group_size: int, bits: int, out=None):
    """W bf16 [N,K] (CUDA) -> (Wq uint8 [N,K*bits/8], scales bf16 [N,K/g], offsets bf16 [N,K/g]),
    codes of 2, 4 or 8 bits (the lowest k in the lowest bits of a byte)."""
    lib = load_library()
    _bits16(W, "W")
    N, K = W.shape
    if out is None:
        ng = K // group_size if group_size and K % group_size == 0 else 0
        row = K * bits // 8 if bits in (2, 4, 8) else 0
        Wq = torch.empty((N, row), dtype=torch.uint8, device=W.device)
        sc = torch.empty((N, ng), dtype=torch.bfloat16, device=W.device)
        of = torch.empty((N, ng), dtype=torch.bfloat16, device=W.device)
    else:
        Wq, sc, of = out
    _check(lib.w4_quantize_bits(_ptr(W), N, K, group_size, bits, _ptr(Wq), _ptr(sc), _ptr(of), _stream(W)),
           "w4_quantize_bits")
    return Wq, sc, of


def w4_dequantize_bits(Wq: torch.Tensor, scales: torch.Tensor, offsets: torch.Tensor, group_size: int, bits: int,
                       out=None):
    """Packed `bits`-bit weights -> bf16 [N,K]."""
    lib = load_library()
    if bits not in (2, 4, 8):
        raise ValueError("bits must be 2, 4 or 8")
    N, row = Wq.shape
    K = row * 8 // bits
    W = out if out is not None else torch.empty((N, K), dtype=torch.bfloat16, device=Wq.device)
    _check(lib.w4_dequantize_bits(_ptr(Wq), _ptr(scales), _ptr(offsets), N, K, group_size, bits, _ptr(W),
                                  _stream(Wq)), "w4_dequantize_bits")
    return W


def w4_linear_bits(X: torch.Tensor, Wq: torch.Tensor, scales: torch.Tensor, offsets: torch.Tensor,
                   group_size: int, bits: int, out=None, workspace=None):
    """Y bf16 [M,N] = X . dequant(Wq)^T for `bits`-bit codes (see include/w4.h)."""
    lib = load_library()
    _bits16(X, "X")
    M, K = X.shape
    N = Wq.shape[0]
    Y = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    ws = _workspace_for(X, M, N, K, group_size, workspace)
    _check(lib.w4_linear_bits(_ptr(X), M, K, _ptr(Wq), _ptr(scales), _ptr(offsets), N, group_size, bits, _ptr(Y),
                              _ptr(ws.buf), ws.nbytes, _stream(X)), "w4_linear_bits")
    return Y


def w4_linear_workspace_bytes(M: int, N: int, K: int, group_size: int) -> int:
    return load_library().w4_linear_workspace_bytes(M, N, K, group_size)


class Workspace:
    """Zero-filled device workspace for w4_linear (the stream kernels' slots for
    the partial sums of row tiles split between warps, and past 16 MiB the
    tensor-core GEMM's partial tiles).  Every call leaves its first 16 MiB
    zeroed, so it can be reused by calls of any shape in sequence; calls that
    can overlap on the GPU need one each.  Growing it allocates (through torch):
    size it before capturing a CUDA graph or timing."""

    def __init__(self, device=None, nbytes: int = 0):
        self.device = torch.device(device or "cuda")
        self.buf = None
        if nbytes:
            self.reserve(nbytes)

    def reserve(self, nbytes: int):
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=self.device)
            # the zero fill ran on the current stream; calls may come on any stream
            torch.cuda.current_stream(self.device).synchronize()
        return self

    def reserve_for(self, M: int, N: int, K: int, group_size: int):
        return self.reserve(w4_linear_workspace_bytes(M, N, K, group_size))

    @property
    def nbytes(self) -> int:
        return 0 if self.buf is None else self.buf.numel()


_default_ws = {}


def _workspace_for(X: torch.Tensor, M, N, K, g, workspace):
    """The caller's workspace as given, or this stream's default one grown to fit."""
    if workspace is not None:
        return workspace
    key = (X.device.index, torch.cuda.current_stream(X.device).cuda_stream)
    ws = _default_ws.get(key)
    if ws is None:
        ws = _default_ws[key] = Workspace(X.device)
    return ws.reserve_for(M, N, K, g)


def w4_linear_ex(X: torch.Tensor, Wq: torch.Tensor, scales: torch.Tensor, offsets: torch.Tensor,
                 group_size: int, kernel: int = KERNEL_AUTO, out=None, workspace: Workspace | None = None):
    """Y bf16 [M,N] = X bf16 [M,K] . dequant(Wq)^T with fp32 accumulation."""
    lib = load_library()
    _bits16(X, "X")
    M, K = X.shape
    N = Wq.shape[0]
    Y = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    ws = _workspace_for(X, M, N, K, group_size, workspace)
    _check(lib.w4_linear_ex(_ptr(X), M, K, _ptr(Wq), _ptr(scales), _ptr(offsets), N, group_size, _ptr(Y),
                            _ptr(ws.buf), ws.nbytes, kernel, _stream(X)), "w4_linear")
    return Y


def w4_linear_bias(X: torch.Tensor, Wq: torch.Tensor, scales: torch.Tensor, offsets: torch.Tensor,
                   group_size: int, bias: torch.Tensor | None, kernel: int = KERNEL_AUTO, out=None,
                   workspace: Workspace | None = None):
    """Y bf16 [M,N] = X . dequant(Wq)^T + bias (bf16 [N], added in fp32 before the rounding; None: no bias)."""
    lib = load_library()
    _bits16(X, "X")
    M, K = X.shape
    N = Wq.shape[0]
    if bias is not None:
        _bits16(bias, "bias")
        if bias.numel() != N:
            raise ValueError("bias must hold N values")
    Y = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    ws = _workspace_for(X, M, N, K, group_size, workspace)
    _check(lib.w4_linear_bias_ex(_ptr(X), M, K, _ptr(Wq), _ptr(scales), _ptr(offsets), N, group_size, _ptr(bias),
                                 _ptr(Y), _ptr(ws.buf), ws.nbytes, kernel, _stream(X)), "w4_linear_bias")
    return Y


def w4_quantize_activation_i8(X: torch.Tensor, per_token: bool = False, out=None, workspace: Workspace | None = None):
    """X bf16 [M,K] -> (Xq int8 [M,K], x_scale fp32 [1] or [M]): s = max|x| / 127 per tensor
    (or per row), Xq = clamp(rne(x / s), -127, 127)."""
    lib = load_library()
    _bits16(X, "X")
    M, K = X.shape
    if out is None:
        Xq = torch.empty((M, K), dtype=torch.int8, device=X.device)
        xs = torch.empty((M if per_token else 1,), dtype=torch.float32, device=X.device)
    else:
        Xq, xs = out
    need = lib.w4_quantize_activation_workspace_bytes(M, K, int(bool(per_token)))
    ws = workspace if workspace is not None else (Workspace(X.device, need) if need else None)
    _check(lib.w4_quantize_activation_i8(_ptr(X), M, K, int(bool(per_token)), _ptr(Xq), _ptr(xs),
                                         _ptr(ws.buf) if ws is not None else None, ws.nbytes if ws is not None else 0,
                                         _stream(X)), "w4_quantize_activation_i8")
    return Xq, xs


def w4_linear_i8_workspace_bytes(M: int, N: int, K: int, group_size: int) -> int:
    return load_library().w4_linear_i8_workspace_bytes(M, N, K, group_size)


def w4_linear_i8(Xq: torch.Tensor, x_scale: torch.Tensor, per_token: bool, Wq: torch.Tensor, scales: torch.Tensor,
                 offsets: torch.Tensor, group_size: int, bias: torch.Tensor | None = None, out=None,
                 workspace: Workspace | None = None):
    """Y bf16 [M,N] = s_x * sum_j (s_j I_j + o_j S_j) (+ bias [N]) on int8 activation codes Xq [M,K]
    (x_scale fp32: [1] per tensor, [M] per token) and 4-bit weights."""
    lib = load_library()
    if Xq.dtype != torch.int8 or not Xq.is_contiguous():
        raise TypeError("Xq must be a contiguous int8 tensor")
    if x_scale.dtype != torch.float32:
        raise TypeError("x_scale must be float32")
    M, K = Xq.shape
    N = Wq.shape[0]
    if x_scale.numel() != (M if per_token else 1):
        raise ValueError("x_scale must hold M values per token, 1 per tensor")
    if bias is not None:
        _bits16(bias, "bias")
        if bias.numel() != N:
            raise ValueError("bias must hold N values")
    Y = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=Xq.device)
    if workspace is None:
        key = ("i8", Xq.device.index, torch.cuda.current_stream(Xq.device).cuda_stream)
        workspace = _default_ws.get(key)
        if workspace is None:
            workspace = _default_ws[key] = Workspace(Xq.device)
        workspace.reserve(lib.w4_linear_i8_workspace_bytes(M, N, K, group_size))
    _check(lib.w4_linear_i8(_ptr(Xq), _ptr(x_scale), int(bool(per_token)), M, K, _ptr(Wq), _ptr(scales), _ptr(offsets),
                            N, group_size, _ptr(bias), _ptr(Y), _ptr(workspace.buf), workspace.nbytes, _stream(Xq)),
           "w4_linear_i8")
    return Y


def w4_linear_i8_dynamic_workspace_bytes(M: int, N: int, K: int, group_size: int) -> int:
    return load_library().w4_linear_i8_dynamic_workspace_bytes(M, N, K, group_size)


def w4_linear_i8_dynamic(X: torch.Tensor, Wq: torch.Tensor, scales: torch.Tensor, offsets: torch.Tensor,
                         group_size: int, per_token: bool = False, bias: torch.Tensor | None = None, out=None,
                         workspace: Workspace | None = None):
    """Y bf16 [M,N]: X bf16 [M,K] quantized to int8 (one scale per tensor, or per token) and the
    int8 linear on the codes, in one call (bit-identical to the two separate calls)."""
    lib = load_library()
    _bits16(X, "X")
    M, K = X.shape
    N = Wq.shape[0]
    if bias is not None:
        _bits16(bias, "bias")
        if bias.numel() != N:
            raise ValueError("bias must hold N values")
    Y = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    if workspace is None:
        key = ("i8", X.device.index, torch.cuda.current_stream(X.device).cuda_stream)
        workspace = _default_ws.get(key)
        if workspace is None:
            workspace = _default_ws[key] = Workspace(X.device)
        workspace.reserve(lib.w4_linear_i8_dynamic_workspace_bytes(M, N, K, group_size))
    _check(lib.w4_linear_i8_dynamic(_ptr(X), int(bool(per_token)), M, K, _ptr(Wq), _ptr(scales), _ptr(offsets), N,
                                    group_size, _ptr(bias), _ptr(Y), _ptr(workspace.buf), workspace.nbytes, _stream(X)),
           "w4_linear_i8_dynamic")
    return Y


def w4_linear(X, Wq, scales, offsets, group_size, out=None, workspace=None):
    """Y bf16 [M,N] = X . dequant(Wq)^T (kernel chosen by M; see include/w4.h)."""
    return w4_linear_ex(X, Wq, scales, offsets, group_size, KERNEL_AUTO, out, workspace)


def w4_repacked_bytes(N: int, K: int, group_size: int) -> int:
    return load_library().w4_repacked_bytes(N, K, group_size)


class Repacked:
    """Weights in the decode layout (include/w4.h): the flat uint8 buffer plus the
    shape it holds."""

    def __init__(self, buf: torch.Tensor, N: int, K: int, group_size: int):
        self.buf, self.N, self.K, self.group_size = buf, N, K, group_size


def w4_repack(Wq: torch.Tensor, scales: torch.Tensor, offsets: torch.Tensor, group_size: int, out=None) -> Repacked:
    """Canonical packed weights -> the decode layout (a load-time conversion)."""
    lib = load_library()
    N, half = Wq.shape
    K = 2 * half
    nbytes = w4_repacked_bytes(N, K, group_size)
    buf = out if out is not None else torch.empty(max(nbytes, 16), dtype=torch.uint8, device=Wq.device)
    _check(lib.w4_repack(_ptr(Wq), _ptr(scales), _ptr(offsets), N, K, group_size, _ptr(buf), _stream(Wq)),
           "w4_repack")
    return Repacked(buf, N, K, group_size)


def w4_linear_repacked(X: torch.Tensor, packed: Repacked, out=None, workspace: Workspace | None = None):
    """Y bf16 [M,N] = X . dequant(W)^T for M <= 32 with W in the decode layout."""
    lib = load_library()
    _bits16(X, "X")
    M, K = X.shape
    N, g = packed.N, packed.group_size
    Y = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    ws = _workspace_for(X, M, N, K, g, workspace)
    _check(lib.w4_linear_repacked(_ptr(X), M, K, _ptr(packed.buf), N, g, _ptr(Y), _ptr(ws.buf), ws.nbytes,
                                  _stream(X)), "w4_linear_repacked")
    return Y


def w4_linear_static(X, Wq, scales, offsets, group_size, out=None):
    """w4_linear for callers that cannot allocate device memory: the library's
    own 4 MiB device array serves as workspace (M <= 8; see include/w4.h).
    Calls that can overlap on the GPU share that array and must be serialized."""
    lib = load_library()
    _bits16(X, "X")
    M, K = X.shape
    N = Wq.shape[0]
    Y = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    # the library finds its array on the current device: make it X's
    with torch.cuda.device(X.device):
        _check(lib.w4_linear_static(_ptr(X), M, K, _ptr(Wq), _ptr(scales), _ptr(offsets), N, group_size, _ptr(Y),
                                    _stream(X)), "w4_linear_static")
    return Y


def w4_device_fault(device=None) -> None:
    """Synchronize the current stream and raise W4Error if a kernel gave up a bounded wait."""
    lib = load_library()
    dev = torch.device(device or "cuda")
    _check(lib.w4_device_fault(ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)), "w4_device_fault")
