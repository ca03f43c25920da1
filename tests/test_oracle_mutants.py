"""The oracle's pins catch plausible mistakes.

Each mutant is a temporary copy of oracle/w4_oracle.c with one planted error
(a dropped term, a wrong rounding, a swapped index ...), compiled with gcc and
loaded on the CPU.  The worked examples, invariants and closed forms of
test_oracle_pins.py must reject every one of them.  Nothing here touches a GPU.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle
from tests.test_oracle_pins import GOLDEN_BITS_CASES, GOLDEN_CASES, unpack_codes

SRC = os.path.join(os.path.dirname(oracle.__file__), "w4_oracle.c")

MUTANTS = {
    "round_half_up": ("float r = rintf(t);", "float r = floorf(t + 0.5f);"),
    "truncate_codes": ("float r = rintf(t);", "float r = truncf(t);"),
    "scale_over_2_to_the_b": ("float s32 = range / (float)levels;", "float s32 = range / (float)(levels + 1);"),
    "offset_is_max": ("uint16_t o_bits = ref_float_to_bf16(mn);", "uint16_t o_bits = ref_float_to_bf16(mx);"),
    "code_with_fp32_scale": ("float t = d / s;", "float t = d / s32;"),
    "codes_in_reverse_byte_order": ("int shift = (int)(k % per_byte) * bits;",
                                    "int shift = (int)(per_byte - 1 - k % per_byte) * bits;"),
    "clamp_at_15": ("if (q > levels)\n                    q = levels;", "if (q > 15)\n                    q = 15;"),
    "no_upper_clamp": ("if (q > levels)\n                    q = levels;", ""),
    "dequant_reads_a_nibble": ("& ((1 << bits) - 1);", "& 0x0F;"),
    "dequant_drops_offset": ("float u = t + o;", "float u = t;"),
    "linear_output_transposed": ("Y[m * N + n] = acc;", "Y[n * M + m] = acc;"),
    "no_eps_clamp": ("if (s32 < REF_EPS)\n                s32 = REF_EPS;", ""),
    "bf16_truncates": ("upper += 1u;", "upper += 0u;"),
    "zero_order_ignored": ("return signbit(a) && !signbit(b);", "return 0;"),
    "scale_not_rounded_to_bf16": ("float s = ref_bf16_to_float(s_bits);", "float s = s32;"),
    "bias_dropped": ("Y[m * N + n] += (double)ref_bf16_to_float(bias[n]);", ""),
    "bias_of_the_token": ("Y[m * N + n] += (double)ref_bf16_to_float(bias[n]);",
                          "Y[m * N + n] += (double)ref_bf16_to_float(bias[m]);"),
}


def _build_mutant(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} is not unique"
    c = tmp_path / f"{name}.c"
    c.write_text(src.replace(old, new))
    so = tmp_path / f"{name}.so"
    return _compile(c, so)


def _compile(c, so):
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-fPIC", "-shared",
                    "-o", str(so), str(c), "-lm"], check=True)
    lib = ctypes.CDLL(str(so))
    p, i64 = ctypes.c_void_p, ctypes.c_int64
    lib.w4_ref_quantize.argtypes = [p, i64, i64, ctypes.c_int, p, p, p]
    lib.w4_ref_dequantize.argtypes = [p, p, p, i64, i64, ctypes.c_int, p]
    lib.w4_ref_linear.argtypes = [p, i64, i64, p, p, p, i64, ctypes.c_int, p]
    lib.w4_ref_linear_bias_bits.argtypes = [p, i64, i64, p, p, p, i64, ctypes.c_int, ctypes.c_int, p, p]
    lib.w4_ref_quantize_bits.argtypes = [p, i64, i64, ctypes.c_int, ctypes.c_int, p, p, p]
    lib.w4_ref_dequantize_bits.argtypes = [p, p, p, i64, i64, ctypes.c_int, ctypes.c_int, p]
    return lib


def _pins_reject(lib) -> bool:
    """Run the hand-derived examples and one closed form through a mutant;
    True if any of them disagrees."""
    P = lambda a: ctypes.c_void_p(a.ctypes.data)
    for case in GOLDEN_CASES:
        g = case["g"]
        W = np.ascontiguousarray(case["values"].reshape(1, g))
        Wq = np.zeros((1, g // 2), np.uint8)
        sc = np.zeros((1, 1), np.uint16)
        of = np.zeros((1, 1), np.uint16)
        lib.w4_ref_quantize(P(W), 1, g, g, P(Wq), P(sc), P(of))
        if sc[0, 0] != case["scale"] or of[0, 0] != case["offset"]:
            return True
        if not np.array_equal(unpack_codes(Wq)[0], case["codes"]):
            return True
        if "bytes" in case and not np.array_equal(Wq[0], case["bytes"]):
            return True
        if "deq" in case:
            out = np.zeros((1, g), np.uint16)
            lib.w4_ref_dequantize(P(Wq), P(sc), P(of), 1, g, g, P(out))
            if not np.array_equal(out[0], case["deq"]):
                return True
    for case in GOLDEN_BITS_CASES:
        g, b = case["g"], case["bits"]
        W = np.ascontiguousarray(case["values"].reshape(1, g))
        Wq = np.zeros((1, g * b // 8), np.uint8)
        sc = np.zeros((1, 1), np.uint16)
        of = np.zeros((1, 1), np.uint16)
        lib.w4_ref_quantize_bits(P(W), 1, g, g, b, P(Wq), P(sc), P(of))
        if sc[0, 0] != case["scale"] or of[0, 0] != case["offset"] or not np.array_equal(Wq[0], case["bytes"]):
            return True
        out = np.zeros((1, g), np.uint16)
        lib.w4_ref_dequantize_bits(P(Wq), P(sc), P(of), 1, g, g, b, P(out))
        if not np.array_equal(out[0], case["deq"]):
            return True
    # one-hot closed form of the linear: X = e_k -> Y[k, n] = W'[n, k]
    g, N, K = 32, 3, 32
    case = GOLDEN_CASES[0]
    W = np.ascontiguousarray(np.tile(case["values"], (N, 1)))
    Wq = np.zeros((N, K // 2), np.uint8)
    sc = np.zeros((N, 1), np.uint16)
    of = np.zeros((N, 1), np.uint16)
    lib.w4_ref_quantize(P(W), N, K, g, P(Wq), P(sc), P(of))
    X = np.zeros((K, K), np.uint16)
    X[np.arange(K), np.arange(K)] = 0x3F80
    Y = np.zeros((K, N), np.float64)
    lib.w4_ref_linear(P(X), K, K, P(Wq), P(sc), P(of), N, g, P(Y))
    expect = oracle.bf16_bits_to_f64(case["deq"])
    if not np.array_equal(Y, np.tile(expect[:, None], (1, N))):
        return True
    # the bias closed form: every w' = 0 (codes 0, offsets 0) -> Y[m, n] = bias[n]
    Wz = np.zeros((N, K // 2), np.uint8)
    sz = np.full((N, 1), 0x3C00, np.uint16)
    oz = np.zeros((N, 1), np.uint16)
    bias = np.array([0x3F80, 0xC000, 0x4049], np.uint16)  # 1, -2, 3.140625
    Yb = np.zeros((2, N), np.float64)
    lib.w4_ref_linear_bias_bits(P(X[:2].copy()), 2, K, P(Wz), P(sz), P(oz), N, g, 4, P(bias), P(Yb))
    return not np.array_equal(Yb, np.tile([1.0, -2.0, 3.140625], (2, 1)))


def test_unmutated_oracle_passes(tmp_path):
    src = open(SRC).read()
    c = tmp_path / "clean.c"
    c.write_text(src)
    assert not _pins_reject(_compile(c, tmp_path / "clean.so"))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    assert _pins_reject(_build_mutant(tmp_path, name)), f"pins did not catch mutant {name}"
