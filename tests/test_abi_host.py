"""libw4's C ABI on the host: the library loads, exports every call that
include/w4.h declares, and rejects bad arguments before touching the GPU.
Nothing here launches a kernel, so it runs without a GPU."""
import ctypes
import glob
import os
import re

import pytest
import torch

import bit_weight_quantization_02_b300 as w4

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "w4.h")
HEADERS = sorted(glob.glob(os.path.join(ROOT, "include", "*.h")))

OK, INVALID, UNSUPPORTED, MISALIGNED = 0, 1, 2, 3


def declared_functions():
    text = "\n".join(open(h).read() for h in HEADERS)
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(w4_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from bit_weight_quantization_02_b300 import _build
    _build.build()
    return w4.load_library()


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert {"w4_quantize", "w4_dequantize", "w4_linear", "w4_linear_ex", "w4_linear_workspace_bytes",
            "w4_device_fault"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/*.h but not exported"


def test_only_the_abi_is_exported(lib):
    # the library is built with hidden visibility: no C++ internals leak out
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", w4.library_path()], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert exported, out
    assert {e for e in exported if e.startswith("w4_")} == set(declared_functions())


def test_format_version_and_status_strings(lib):
    assert lib.w4_format_version() == w4.W4_FORMAT_VERSION == 1
    for s, name in [(0, b"W4_OK"), (1, b"W4_ERR_INVALID_ARG"), (2, b"W4_ERR_UNSUPPORTED"),
                    (3, b"W4_ERR_MISALIGNED"), (4, b"W4_ERR_CUDA"), (5, b"W4_ERR_TIMEOUT")]:
        assert lib.w4_status_string(s) == name


def test_sizes(lib):
    assert lib.w4_packed_bytes(14336, 4096) == 14336 * 2048
    assert lib.w4_qparam_bytes(14336, 4096, 32) == 14336 * 128 * 2
    assert lib.w4_qparam_bytes(4096, 14336, 128) == 4096 * 112 * 2
    assert lib.w4_qparam_bytes(10, 100, 32) == 0  # K % g
    assert lib.w4_qparam_bytes(10, 128, 16) == 0  # unsupported g
    assert lib.w4_packed_bytes(-1, 64) == 0


def test_workspace_plan(lib):
    # the stream kernels (M <= 32) need one slot of 16 rows x M 8-byte words per warp of their grid:
    # at most one warp per 16 x 256 unit and at most 4096 warps (8192 with one token)
    assert lib.w4_linear_workspace_bytes(1, 1024, 4096, 32) == 64 * 16 * 128       # 1024 units
    assert lib.w4_linear_workspace_bytes(8, 14336, 4096, 128) == 4096 * 128 * 8    # 14336 units: the cap
    assert lib.w4_linear_workspace_bytes(1, 14336, 4096, 32) == 8192 * 128        # one token: cap 8192
    assert lib.w4_linear_workspace_bytes(8, 10 ** 6, 4096, 32) == 4 << 20          # w4_linear_static's array
    assert lib.w4_linear_workspace_bytes(9, 1024, 4096, 32) == 1024 * 128 * 9
    assert lib.w4_linear_workspace_bytes(32, 1000, 4100 - 4, 32) == 63 * 16 * 128 * 32  # ceil(1000/16) tiles
    assert lib.w4_linear_workspace_bytes(2, 40, 300 - 12, 32) == 3 * 2 * 128 * 2   # ragged: 3 tiles x 2 units
    # M > 32 (the tcgen05 GEMM): its stream-K tail is sized for the current device's SMs (16 MiB of
    # slots, then 128 KB of partial sums a block); without a device there is nothing to size: 0
    gemm_ws = lib.w4_linear_workspace_bytes(33, 1024, 4096, 32)
    if torch.cuda.is_available():
        assert gemm_ws == 0 or (gemm_ws > 16 << 20 and (gemm_ws - (16 << 20)) % (128 << 10) == 0)
    else:
        assert gemm_ws == 0
    assert lib.w4_linear_workspace_bytes(1, 100, 96, 32) == 7 * 128  # K/g odd: the decode layout's need
    assert lib.w4_linear_workspace_bytes(0, 100, 128, 32) == 0


def test_linear_kernel_choice_rules(lib):
    # the stream kernel only takes M <= 32 and needs its workspace; the checks run before any launch
    assert lib.w4_linear_ex(FAKE, 33, 64, FAKE, FAKE, FAKE, 4, 32, FAKE, FAKE, 1 << 20, 4, None) == INVALID
    assert lib.w4_linear_ex(FAKE, 2, 64, FAKE, FAKE, FAKE, 4, 32, FAKE, None, 0, 4, None) == INVALID
    assert b"workspace" in lib.w4_last_error_detail()
    assert lib.w4_linear_ex(FAKE, 33, 64, FAKE, FAKE, FAKE, 4, 32, FAKE, None, 0, 3, None) == INVALID


FAKE = 0x10000  # a 16-byte aligned address that is never dereferenced: every call below fails its checks first


@pytest.mark.parametrize("g,expect", [(16, UNSUPPORTED), (96, UNSUPPORTED), (0, UNSUPPORTED)])
def test_unsupported_group_sizes(lib, g, expect):
    assert lib.w4_quantize(FAKE, 4, 256, g, FAKE, FAKE, FAKE, None) == expect
    assert lib.w4_dequantize(FAKE, FAKE, FAKE, 4, 256, g, FAKE, None) == expect
    assert lib.w4_linear(FAKE, 1, 256, FAKE, FAKE, FAKE, 4, g, FAKE, None, 0, None) == expect


@pytest.mark.parametrize("N,K", [(4, 0), (4, -32), (-1, 64), (4, 96 + 16), (1 << 31, 64), (4, 1 << 31)])
def test_invalid_shapes(lib, N, K):
    assert lib.w4_quantize(FAKE, N, K, 32, FAKE, FAKE, FAKE, None) == INVALID
    assert lib.w4_dequantize(FAKE, FAKE, FAKE, N, K, 32, FAKE, None) == INVALID
    assert lib.w4_linear(FAKE, 1, K, FAKE, FAKE, FAKE, N, 32, FAKE, None, 0, None) == INVALID
    assert lib.w4_last_error_detail()


def test_null_and_misaligned_pointers(lib):
    assert lib.w4_quantize(None, 4, 64, 32, FAKE, FAKE, FAKE, None) == INVALID
    assert lib.w4_quantize(FAKE + 2, 4, 64, 32, FAKE, FAKE, FAKE, None) == MISALIGNED
    assert lib.w4_quantize(FAKE, 4, 64, 32, FAKE + 8, FAKE, FAKE, None) == MISALIGNED
    assert lib.w4_dequantize(FAKE, None, FAKE, 4, 64, 32, FAKE, None) == INVALID
    assert lib.w4_dequantize(FAKE, FAKE, FAKE, 4, 64, 32, FAKE + 4, None) == MISALIGNED
    assert lib.w4_linear(FAKE, 2, 64, FAKE, FAKE, None, 4, 32, FAKE, None, 0, None) == INVALID
    assert lib.w4_linear(FAKE + 2, 2, 64, FAKE, FAKE, FAKE, 4, 32, FAKE, None, 0, None) == MISALIGNED
    assert lib.w4_linear(FAKE, 2, 64, FAKE, FAKE, FAKE, 4, 32, FAKE + 8, None, 0, None) == MISALIGNED
    assert lib.w4_linear(FAKE, 2, 64, FAKE, FAKE, FAKE, 4, 32, FAKE, FAKE + 8, 64, None) == MISALIGNED
    assert b"aligned" in lib.w4_last_error_detail()


def test_empty_problems_succeed_without_launch(lib):
    # N == 0 or M == 0: nothing to do, no pointer is touched, no CUDA call is made
    assert lib.w4_quantize(None, 0, 64, 32, None, None, None, None) == OK
    assert lib.w4_dequantize(None, None, None, 0, 64, 32, None, None) == OK
    assert lib.w4_linear(None, 0, 64, None, None, None, 8, 32, None, None, 0, None) == OK
    assert lib.w4_linear(None, 3, 64, None, None, None, 0, 32, None, None, 0, None) == OK


def test_linear_argument_rules(lib):
    assert lib.w4_linear(FAKE, -1, 64, FAKE, FAKE, FAKE, 4, 32, FAKE, None, 0, None) == INVALID
    # the skinny kernel only takes M <= 32
    assert lib.w4_linear_ex(FAKE, 33, 64, FAKE, FAKE, FAKE, 4, 32, FAKE, None, 0, 1, None) == INVALID
    assert lib.w4_linear_ex(FAKE, 1, 64, FAKE, FAKE, FAKE, 4, 32, FAKE, None, 0, 7, None) == INVALID


def test_binding_refuses_cpu_tensors(lib):
    import torch
    with pytest.raises(ValueError):
        w4.w4_quantize(torch.zeros(4, 64, dtype=torch.bfloat16), 32)


def test_product_package_does_not_touch_the_oracle():
    """The product path never imports, links or runs the oracle."""
    pkg = os.path.join(ROOT, "bit_weight_quantization_02_b300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".c")):
                text = open(os.path.join(dirpath, f)).read()
                for needle in ("import oracle", "from oracle", "w4_ref_", "libw4_oracle", "w4_oracle"):
                    assert needle not in text, (f, needle)


def test_decode_layout_calls(lib):
    # sizes: ceil(N/16) tiles x ceil(K/256) units x (2048 + 16384/g) bytes
    assert lib.w4_repacked_bytes(4096, 4096, 32) == 256 * 16 * 2560
    assert lib.w4_repacked_bytes(17, 300, 64) == 0  # K % g
    assert lib.w4_repacked_bytes(17, 320, 64) == 2 * 2 * 2304
    assert lib.w4_repacked_bytes(1, 128, 128) == 2176
    assert lib.w4_repacked_bytes(4, 256, 48) == 0
    # w4_repack: argument checks before any launch
    assert lib.w4_repack(FAKE, FAKE, FAKE, 4, 256, 48, FAKE, None) == UNSUPPORTED
    assert lib.w4_repack(FAKE, FAKE, FAKE, 4, 100, 32, FAKE, None) == INVALID
    assert lib.w4_repack(FAKE, None, FAKE, 4, 256, 32, FAKE, None) == INVALID
    assert lib.w4_repack(FAKE, FAKE, FAKE, 4, 256, 32, FAKE + 8, None) == MISALIGNED
    assert lib.w4_repack(FAKE, FAKE, FAKE, 0, 256, 32, FAKE, None) == OK  # nothing to do
    # w4_linear_repacked: M <= 8, a workspace of w4_linear_workspace_bytes
    ws = lib.w4_linear_workspace_bytes(2, 64, 512, 32)
    assert lib.w4_linear_repacked(FAKE, 33, 512, FAKE, 64, 32, FAKE, FAKE, 1 << 20, None) == INVALID
    assert lib.w4_linear_repacked(FAKE, -1, 512, FAKE, 64, 32, FAKE, FAKE, ws, None) == INVALID
    assert lib.w4_linear_repacked(FAKE, 2, 512, FAKE, 64, 32, FAKE, None, 0, None) == INVALID
    assert lib.w4_linear_repacked(FAKE, 2, 512, FAKE, 64, 32, FAKE, FAKE, ws - 4, None) == INVALID
    assert lib.w4_linear_repacked(FAKE, 2, 512, FAKE + 4, 64, 32, FAKE, FAKE, ws, None) == MISALIGNED
    assert lib.w4_linear_repacked(FAKE, 2, 512, FAKE, 64, 32, FAKE, FAKE + 8, ws, None) == MISALIGNED
    assert lib.w4_linear_repacked(FAKE, 2, 512, FAKE, 64, 96, FAKE, FAKE, ws, None) == UNSUPPORTED
    assert lib.w4_linear_repacked(FAKE, 0, 512, FAKE, 64, 32, FAKE, None, 0, None) == OK


def test_other_code_widths_host_rules(lib):
    """2- and 8-bit calls: sizes, the width check and the 2-bit row rule, all before any launch."""
    assert lib.w4_packed_bytes_bits(14336, 4096, 2) == 14336 * 1024
    assert lib.w4_packed_bytes_bits(14336, 4096, 4) == lib.w4_packed_bytes(14336, 4096)
    assert lib.w4_packed_bytes_bits(14336, 4096, 8) == 14336 * 4096
    assert lib.w4_packed_bytes_bits(4, 64, 3) == 0
    assert lib.w4_packed_bytes_bits(4, 66, 2) == 0  # K not a whole number of bytes
    for bits in (0, 1, 3, 16):
        assert lib.w4_quantize_bits(FAKE, 4, 256, 32, bits, FAKE, FAKE, FAKE, None) == UNSUPPORTED
        assert lib.w4_dequantize_bits(FAKE, FAKE, FAKE, 4, 256, 32, bits, FAKE, None) == UNSUPPORTED
        assert lib.w4_linear_bits(FAKE, 1, 256, FAKE, FAKE, FAKE, 4, 32, bits, FAKE, None, 0, None) == UNSUPPORTED
        assert b"bits" in lib.w4_last_error_detail()
    for bits in (2, 8):
        assert lib.w4_quantize_bits(FAKE, 4, 256, 16, bits, FAKE, FAKE, FAKE, None) == UNSUPPORTED
        assert lib.w4_quantize_bits(FAKE, 4, 96 + 16, 32, bits, FAKE, FAKE, FAKE, None) == INVALID
        assert lib.w4_quantize_bits(FAKE + 2, 4, 64, 32, bits, FAKE, FAKE, FAKE, None) == MISALIGNED
        assert lib.w4_dequantize_bits(FAKE, FAKE, FAKE, 4, 64, 32, bits, FAKE + 4, None) == MISALIGNED
        assert lib.w4_linear_bits(FAKE, -1, 64, FAKE, FAKE, FAKE, 4, 32, bits, FAKE, None, 0, None) == INVALID
        assert lib.w4_linear_bits(FAKE, 2, 64, FAKE, FAKE, FAKE, 4, 32, bits, FAKE + 8, None, 0, None) == MISALIGNED
        # empty problems: no pointer touched, no launch
        assert lib.w4_quantize_bits(None, 0, 64, 32, bits, None, None, None, None) == OK
        assert lib.w4_linear_bits(None, 0, 64, None, None, None, 8, 32, bits, None, None, 0, None) == OK
    # 2-bit rows must be whole 16-byte pieces for the linear (K % 64), quantize takes any K % g == 0
    assert lib.w4_linear_bits(FAKE, 1, 96, FAKE, FAKE, FAKE, 4, 32, 2, FAKE, None, 0, None) == UNSUPPORTED
    assert b"K % 64" in lib.w4_last_error_detail()


def test_every_exported_python_name_exists_and_covers_the_header():
    """The binding carries the C calls under the same names; the few it does not wrap are
    used inside it (error strings, the workspace-size helper behind the default workspace,
    the _ex form behind keyword arguments, the wait self-test behind its own test)."""
    missing = [n for n in w4.__all__ if not hasattr(w4, n)]
    assert not missing, missing
    internal = {"w4_last_error_detail", "w4_status_string", "w4_linear_bias_ex",
                "w4_quantize_activation_workspace_bytes", "w4_selftest_bounded_waits"}
    unbound = [n for n in declared_functions() if not hasattr(w4, n) and n not in internal]
    assert not unbound, f"declared in include/*.h with no Python binding: {unbound}"
