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
from tests.test_oracle_pins import ACT_CASES, GOLDEN_BITS_CASES, GOLDEN_CASES, unpack_codes

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
    # int8 activations
    "act_round_half_away": ("float q = rintf(t);", "float q = roundf(t);"),
    "act_scale_over_128": ("float s = a / 127.0f;", "float s = a / 128.0f;"),
    "act_signed_maximum": ("float v = fabsf(ref_bf16_to_float(X[m * K + k]));",
                           "float v = ref_bf16_to_float(X[m * K + k]);"),
    "act_no_eps_clamp": ("if (s < REF_EPS)\n            s = REF_EPS;", ""),
    "act_truncating_quotient": ("float q = rintf(t);", "float q = truncf(t);"),
    "act_one_scale_for_every_token": ("double y = (double)x_scale[per_token ? m : 0] * acc;",
                                      "double y = (double)x_scale[0] * acc;"),
    "act_offset_term_dropped": ("\n                     + (double)ref_bf16_to_float(offsets[n * ng + j]) * (double)S;", ";"),
    "act_scale_not_applied": ("double y = (double)x_scale[per_token ? m : 0] * acc;", "double y = acc;"),
    "act_weight_codes_high_nibble_first": ("int q = (Wq[n * (K / 2) + k / 2] >> ((int)(k % 2) * 4)) & 0xF;",
                                           "int q = (Wq[n * (K / 2) + k / 2] >> ((int)(1 - k % 2) * 4)) & 0xF;"),
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
    lib.w4_ref_quantize_activation_i8.argtypes = [p, i64, i64, ctypes.c_int, p, p]
    lib.w4_ref_linear_i8.argtypes = [p, p, ctypes.c_int, i64, i64, p, p, p, i64, ctypes.c_int, p, p]
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
    if not np.array_equal(Yb, np.tile([1.0, -2.0, 3.140625], (2, 1))):
        return True
    return _activation_pins_reject(lib)


def _activation_pins_reject(lib) -> bool:
    """The int8-activation pins: the hand-derived activation cases, the int8 linear
    against the bf16 linear on exact inputs (per tensor and per token), and the
    offset closed form."""
    P = lambda a: ctypes.c_void_p(a.ctypes.data)
    for c in ACT_CASES.values():
        M, K = c["X"].shape
        X = np.ascontiguousarray(c["X"])
        Xq = np.zeros((M, K), np.int8)
        xs = np.zeros(c["scale"].shape, np.float32)
        lib.w4_ref_quantize_activation_i8(P(X), M, K, int(c["per_token"]), P(Xq), P(xs))
        if not np.array_equal(xs.view(np.uint32), c["scale"]) or not np.array_equal(Xq, c["codes"]):
            return True
    M, N, K, g = 2, 8, 64, 32
    rng = np.random.default_rng(7)
    ints = rng.integers(-127, 128, size=(M, K))
    ints[0, 3], ints[1, 4] = 127, -127
    X = ((ints.astype(np.float32) * np.float32(0.125)).view(np.uint32) >> 16).astype(np.uint16)
    X[1] = ((ints[1].astype(np.float32) * np.float32(0.25)).view(np.uint32) >> 16).astype(np.uint16)  # row 1: 2^-2
    q = rng.integers(0, 16, size=(N, K), dtype=np.uint8)
    Wq = np.ascontiguousarray((q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8))
    sc = np.full((N, K // g), 0x3C00, np.uint16)  # 2^-7
    of = np.full((N, K // g), 0xBD80, np.uint16)  # -2^-4: w' = (q - 8) 2^-7, exact in bf16
    y16 = np.zeros((M, N), np.float64)
    lib.w4_ref_linear(P(X), M, K, P(Wq), P(sc), P(of), N, g, P(y16))
    Xq = np.zeros((M, K), np.int8)
    xs = np.zeros((M,), np.float32)
    lib.w4_ref_quantize_activation_i8(P(X), M, K, 1, P(Xq), P(xs))
    y8 = np.zeros((M, N), np.float64)
    lib.w4_ref_linear_i8(P(Xq), P(xs), 1, M, K, P(Wq), P(sc), P(of), N, g, None, P(y8))
    if not np.array_equal(y8, y16):
        return True
    # per tensor the shared scale is row 1's, 2^-2: row 0 (2^-3 multiples) codes to half its integers
    Xqt = np.zeros((M, K), np.int8)
    xst = np.zeros((1,), np.float32)
    lib.w4_ref_quantize_activation_i8(P(X), M, K, 0, P(Xqt), P(xst))
    if xst[0] != np.float32(0.25) or not np.array_equal(Xqt[1], ints[1].astype(np.int8)):
        return True
    # offset closed form: codes 0, every activation code 5, scale 1/4
    Wz = np.zeros((N, K // 2), np.uint8)
    oz = np.tile(np.array([[0x3F80, 0xBF00]], np.uint16), (N, 1))  # 1, -0.5
    Xc = np.full((M, K), 5, np.int8)
    x4 = np.array([0.25], np.float32)
    yo = np.zeros((M, N), np.float64)
    lib.w4_ref_linear_i8(P(Xc), P(x4), 0, M, K, P(Wz), P(sc), P(oz), N, g, None, P(yo))
    return not np.array_equal(yo, np.full((M, N), 0.25 * 5 * 32 * (1 - 0.5)))


def test_unmutated_oracle_passes(tmp_path):
    src = open(SRC).read()
    c = tmp_path / "clean.c"
    c.write_text(src)
    assert not _pins_reject(_compile(c, tmp_path / "clean.so"))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    assert _pins_reject(_build_mutant(tmp_path, name)), f"pins did not catch mutant {name}"
