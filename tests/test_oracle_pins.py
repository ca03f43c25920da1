"""Pins for the CPU oracle: checks against things other than the oracle itself.

* hand-derived worked examples (tests/golden/quantize_worked_examples.txt, and
  tests/golden/quantize_bits_worked_examples.txt for 2- and 8-bit codes);
* exact-arithmetic invariants of the affine group projection (Optimum Quanto,
  "Design overview / Tensors"): codes in [0, 15], |w - w'| <= s/2, the group
  minimum codes to 0 and the maximum to 15, the scale is range/15 up to bf16
  rounding, constant groups come back exactly;
* brute force over all 16 codes for the half-to-even rounding (torch.round);
* the memory ratio "about float bits / integer bits" (Optimum Quanto,
  "Performance");
* smaller groups are at least as accurate (torchao guide, section 3.1 tip);
* the fp64 linear against one-hot closed forms, a pure-Python triple loop and
  numpy's float64 matmul;
* at 2 and 8 bits (Optimum Quanto's int2 / int8 weights, torchao's int8
  weight-only per group): the same invariants with 2^b - 1 levels, brute
  force over all 2^b codes, and more bits never less accurate.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from bit_weight_quantization_02_b300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "quantize_worked_examples.txt")
GOLDEN_BITS = os.path.join(os.path.dirname(__file__), "golden", "quantize_bits_worked_examples.txt")


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _expand(tokens):
    out = []
    for t in tokens:
        if "*" in t:
            v, n = t.split("*")
            out.extend([v] * int(n))
        else:
            out.append(t)
    return out


def load_golden(path=GOLDEN):
    cases, cur = [], None
    for raw in open(path):
        line = raw.strip()
        if not line or line.startswith("#"):
            continue
        key, *rest = line.split()
        if key == "case":
            cur = {"name": rest[0], "bits": 4}
        elif key == "end":
            cases.append(cur)
            cur = None
        elif key == "g":
            cur["g"] = int(rest[0])
        elif key == "bits":
            cur["bits"] = int(rest[0])
        elif key in ("values", "deq"):
            cur[key] = np.array([int(v, 16) for v in _expand(rest)], np.uint16)
        elif key in ("scale", "offset"):
            cur[key] = int(rest[0], 16)
        elif key == "codes":
            cur[key] = np.array([int(v) for v in _expand(rest)], np.int64)
        elif key == "bytes":
            cur[key] = np.array([int(v, 16) for v in _expand(rest)], np.uint8)
        else:
            raise ValueError(f"bad golden line: {line}")
    return cases


GOLDEN_CASES = load_golden()
GOLDEN_BITS_CASES = load_golden(GOLDEN_BITS)


def unpack_codes(Wq: np.ndarray, bits: int = 4) -> np.ndarray:
    """Packed bytes [N, K*bits/8] -> codes [N, K]; the code of the lowest k in
    the lowest bits of its byte (at 4 bits: even k in the low nibble)."""
    per = 8 // bits
    parts = [((Wq >> (bits * i)) & ((1 << bits) - 1)).astype(np.int64) for i in range(per)]
    return np.stack(parts, axis=-1).reshape(Wq.shape[0], -1)


def bits_f64(a):
    return oracle.bf16_bits_to_f64(np.ascontiguousarray(a, np.uint16))


def test_golden_file_is_complete():
    assert len(GOLDEN_CASES) >= 9
    for c in GOLDEN_CASES:
        assert len(c["values"]) == c["g"], c["name"]
        assert len(c["codes"]) == c["g"], c["name"]
        if "deq" in c:
            assert len(c["deq"]) == c["g"], c["name"]


@pytest.mark.parametrize("case", GOLDEN_CASES, ids=[c["name"] for c in GOLDEN_CASES])
def test_golden_single_group(case):
    g = case["g"]
    W = case["values"].reshape(1, g)
    Wq, sc, of = oracle.ref_quantize(W, g)
    assert sc[0, 0] == case["scale"], f"scale {sc[0,0]:04X} != {case['scale']:04X}"
    assert of[0, 0] == case["offset"], f"offset {of[0,0]:04X} != {case['offset']:04X}"
    np.testing.assert_array_equal(unpack_codes(Wq)[0], case["codes"])
    if "bytes" in case:
        np.testing.assert_array_equal(Wq[0], case["bytes"])
    if "deq" in case:
        np.testing.assert_array_equal(oracle.ref_dequantize(Wq, sc, of, g)[0], case["deq"])


@pytest.mark.parametrize("case", GOLDEN_CASES, ids=[c["name"] for c in GOLDEN_CASES])
def test_golden_group_embedded_in_matrix(case):
    """The worked group placed at row 2, group 3 of a random 4 x 5g matrix: the
    oracle must put its outputs at that position (pins row/group indexing)."""
    g = case["g"]
    rng = np.random.default_rng(7)
    W = _bits(torch.from_numpy(rng.normal(0, 0.02, (4, 5 * g)).astype(np.float32)).to(torch.bfloat16)).copy()
    W[2, 3 * g:4 * g] = case["values"]
    Wq, sc, of = oracle.ref_quantize(W, g)
    assert sc[2, 3] == case["scale"]
    assert of[2, 3] == case["offset"]
    np.testing.assert_array_equal(unpack_codes(Wq)[2, 3 * g:4 * g], case["codes"])
    if "deq" in case:
        np.testing.assert_array_equal(oracle.ref_dequantize(Wq, sc, of, g)[2, 3 * g:4 * g], case["deq"])


def test_bits_golden_file_is_complete():
    assert {c["bits"] for c in GOLDEN_BITS_CASES} == {2, 8}
    assert len(GOLDEN_BITS_CASES) >= 9
    for c in GOLDEN_BITS_CASES:
        for key in ("values", "codes", "deq"):
            assert len(c[key]) == c["g"], (c["name"], key)
        assert len(c["bytes"]) == c["g"] * c["bits"] // 8, c["name"]


@pytest.mark.parametrize("case", GOLDEN_BITS_CASES, ids=[c["name"] for c in GOLDEN_BITS_CASES])
def test_bits_golden_single_group(case):
    g, b = case["g"], case["bits"]
    W = case["values"].reshape(1, g)
    Wq, sc, of = oracle.ref_quantize(W, g, bits=b)
    assert Wq.shape == (1, g * b // 8)
    assert sc[0, 0] == case["scale"], f"scale {sc[0,0]:04X} != {case['scale']:04X}"
    assert of[0, 0] == case["offset"], f"offset {of[0,0]:04X} != {case['offset']:04X}"
    np.testing.assert_array_equal(Wq[0], case["bytes"])
    np.testing.assert_array_equal(unpack_codes(Wq, b)[0], case["codes"])
    np.testing.assert_array_equal(oracle.ref_dequantize(Wq, sc, of, g, bits=b)[0], case["deq"])


@pytest.mark.parametrize("case", GOLDEN_BITS_CASES, ids=[c["name"] for c in GOLDEN_BITS_CASES])
def test_bits_golden_group_embedded_in_matrix(case):
    """The worked group at row 1, group 2 of a random 3 x 4g matrix."""
    g, b = case["g"], case["bits"]
    rng = np.random.default_rng(8)
    W = _bits(torch.from_numpy(rng.normal(0, 0.02, (3, 4 * g)).astype(np.float32)).to(torch.bfloat16)).copy()
    W[1, 2 * g:3 * g] = case["values"]
    Wq, sc, of = oracle.ref_quantize(W, g, bits=b)
    assert sc[1, 2] == case["scale"] and of[1, 2] == case["offset"]
    np.testing.assert_array_equal(unpack_codes(Wq, b)[1, 2 * g:3 * g], case["codes"])
    np.testing.assert_array_equal(oracle.ref_dequantize(Wq, sc, of, g, bits=b)[1, 2 * g:3 * g], case["deq"])


def adversarial_matrix(g: int, seed: int = 3) -> np.ndarray:
    """Rows of random groups plus hand-picked awkward ones: constant, two-valued,
    signed zeros, tiny (subnormal-range) values, a huge range, exact half-steps."""
    rng = np.random.default_rng(seed)
    rows = []
    base = rng.normal(0, 0.02, (24, 4 * g)).astype(np.float32)
    base[5] *= 100.0
    base[6] *= 1e-37  # bf16 subnormal range (|w| ~ 2e-39)
    base[7] = rng.choice([-1.0, 3.0], size=4 * g)
    base[8] = 0.0
    base[8, ::3] = -0.0
    base[9] = 0.123
    base[10] = rng.normal(0, 1e37, 4 * g)  # large but finite range
    base[11] = (rng.integers(0, 31, 4 * g) * 0.5 - 3.0)  # many exact half-steps
    rows.append(base)
    W = torch.from_numpy(np.concatenate(rows)).to(torch.bfloat16)
    return _bits(W).copy()


@pytest.mark.parametrize("g", [32, 64, 128])
@pytest.mark.parametrize("src", ["normal_outliers", "adversarial"])
def test_affine_projection_invariants(g, src):
    if src == "normal_outliers":
        W = _bits(workloads.gen_weight(64, 8 * g, seed=11, outliers=True))
    else:
        W = adversarial_matrix(g)
    N, K = W.shape
    Wq, sc, of = oracle.ref_quantize(W, g)
    q = unpack_codes(Wq)
    assert q.min() >= 0 and q.max() <= 15
    w = bits_f64(W).reshape(N, K // g, g)
    s = bits_f64(sc)[..., None]
    o = bits_f64(of)[..., None]
    qg = q.reshape(N, K // g, g).astype(np.float64)
    # |w - (q s + o)| <= s/2, up to the fp32 rounding of the subtract and the divide
    err = np.abs(w - (qg * s + o))
    assert np.all(err <= s / 2 * (1 + 2.0 ** -16)), float(np.max(err / s))
    # the offset is the group minimum and codes to 0
    np.testing.assert_array_equal(o[..., 0], w.min(axis=-1))
    amin = w.argmin(axis=-1)
    assert np.all(np.take_along_axis(qg, amin[..., None], -1) == 0)
    # the scale is (max - min)/15 up to bf16 rounding, unless the eps clamp is active
    rng_ = w.max(axis=-1) - w.min(axis=-1)
    ideal = rng_ / 15.0
    eps = oracle.ref_eps()
    unclamped = ideal > eps * (1 + 2.0 ** -8)
    rel = np.abs(s[..., 0] - ideal) / np.where(ideal > 0, ideal, 1.0)
    assert np.all(rel[unclamped] <= 2.0 ** -8)
    assert np.all(s[..., 0][~unclamped] >= eps * (1 - 2.0 ** -8))
    # and the group maximum then codes to 15
    amax = w.argmax(axis=-1)
    qmax = np.take_along_axis(qg, amax[..., None], -1)[..., 0]
    assert np.all(qmax[unclamped] == 15)


def _nearest_even_code(t: np.float32) -> int:
    """Brute force: the code in [0, 15] nearest to t, ties to the even code."""
    best, best_d = None, None
    for c in range(16):
        d = abs(float(t) - c)
        if best is None or d < best_d or (d == best_d and c % 2 == 0):
            best, best_d = c, d
    return best


@pytest.mark.parametrize("g", [32, 64, 128])
def test_rounding_by_brute_force(g):
    """Every code is the nearest of the 16 codes to the fp32 quotient
    (w - o)/s, ties to even (torch.round), saturating at 0 and 15."""
    W = np.concatenate([_bits(workloads.gen_weight(6, 2 * g, seed=21 + g)), adversarial_matrix(g)[:12, :2 * g]])
    Wq, sc, of = oracle.ref_quantize(W, g)
    q = unpack_codes(Wq)
    N, K = W.shape
    wf = (W.astype(np.uint32) << 16).view(np.float32)
    sf = (sc.astype(np.uint32) << 16).view(np.float32)
    of_ = (of.astype(np.uint32) << 16).view(np.float32)
    for n in range(N):
        for k in range(K):
            j = k // g
            t = np.float32(np.float32(wf[n, k]) - of_[n, j]) / sf[n, j]
            assert q[n, k] == _nearest_even_code(t), (n, k, float(t))


@pytest.mark.parametrize("g", [32, 64, 128])
def test_dequantize_is_q_times_s_plus_o(g):
    W = _bits(workloads.gen_weight(32, 4 * g, seed=5, outliers=True))
    Wq, sc, of = oracle.ref_quantize(W, g)
    Wd = oracle.ref_dequantize(Wq, sc, of, g)
    q = unpack_codes(Wq).astype(np.float64)
    s = np.repeat(bits_f64(sc), g, axis=1)
    o = np.repeat(bits_f64(of), g, axis=1)
    exact = q * s + o
    wd = bits_f64(Wd)
    # one fp32 rounding then one bf16 rounding: within half a bf16 ulp plus half an fp32 ulp
    ulp_bf16 = np.spacing(np.abs(wd).astype(np.float32)).astype(np.float64) * 2 ** 16
    assert np.all(np.abs(wd - exact) <= ulp_bf16 / 2 + ulp_bf16 / 2 ** 17)


@pytest.mark.parametrize("g", [32, 64, 128])
def test_memory_ratio(g):
    """Device memory ~ float bits / integer bits: 4/16 for the codes plus two
    bf16 qparams per group, i.e. exactly (4 + 32/g)/16 of the bf16 weights."""
    W = _bits(workloads.gen_weight(16, 2 * g, seed=1))
    Wq, sc, of = oracle.ref_quantize(W, g)
    ratio = (Wq.nbytes + sc.nbytes + of.nbytes) / W.nbytes
    assert ratio == pytest.approx((4 + 32 / g) / 16, abs=0)
    assert abs(ratio - 4 / 16) <= 32 / g / 16 + 1e-12


def test_smaller_groups_are_at_least_as_accurate():
    W = _bits(workloads.gen_weight(256, 1024, seed=9, outliers=True))
    errs = []
    for g in (32, 64, 128):
        Wq, sc, of = oracle.ref_quantize(W, g)
        errs.append(float(np.mean(np.abs(bits_f64(oracle.ref_dequantize(Wq, sc, of, g)) - bits_f64(W)))))
    assert errs[0] <= errs[1] <= errs[2], errs


def test_rows_quantize_independently():
    W = _bits(workloads.gen_weight(40, 256, seed=2, outliers=True))
    full = oracle.ref_quantize(W, 64)
    part = oracle.ref_quantize(W[13:29], 64)
    for a, b in zip(full, part):
        np.testing.assert_array_equal(a[13:29], b)


def test_unsupported_shapes_rejected():
    W = np.zeros((2, 96), np.uint16)
    with pytest.raises(ValueError):
        oracle.ref_quantize(W, 64)
    with pytest.raises(ValueError):
        oracle.ref_quantize(np.zeros((2, 64), np.uint16), 16)


# ---- 2 and 8 bits ----------------------------------------------------------

@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("g", [32, 128])
@pytest.mark.parametrize("src", ["normal_outliers", "adversarial"])
def test_bits_affine_projection_invariants(bits, g, src):
    """With L = 2^b - 1 levels: codes in [0, L], |w - (q s + o)| <= s/2, the
    minimum codes to 0 and is the offset, s = range/L up to bf16 rounding, and
    the maximum codes to L whenever the eps clamp is inactive."""
    L = (1 << bits) - 1
    if src == "normal_outliers":
        W = _bits(workloads.gen_weight(48, 4 * g, seed=13 + bits, outliers=True))
    else:
        W = adversarial_matrix(g, seed=4 + bits)
    N, K = W.shape
    Wq, sc, of = oracle.ref_quantize(W, g, bits=bits)
    assert Wq.shape == (N, K * bits // 8)
    q = unpack_codes(Wq, bits)
    assert q.min() >= 0 and q.max() <= L
    w = bits_f64(W).reshape(N, K // g, g)
    s = bits_f64(sc)[..., None]
    o = bits_f64(of)[..., None]
    qg = q.reshape(N, K // g, g).astype(np.float64)
    # fp32 rounding of the subtract and the divide: t carries up to ~2^-23 * L relative slack.
    # Codes below L are the nearest level: |w - (q s + o)| <= s/2.  A code at L may be a clamped
    # one: the stored scale can be up to 2^-8 (relative) below range/L, which leaves
    # t <= L / (1 - 2^-8); at 2 and 4 bits that is below L + 1/2, at 8 bits up to L + 1.
    err = np.abs(w - (qg * s + o))
    slack = 1 + L * 2.0 ** -20
    top = L / (1 - 2.0 ** -8) - L
    bound = np.where(qg == L, np.maximum(0.5, top) * s * slack, s / 2 * slack)
    assert np.all(err <= bound), float(np.max(err / s))
    if bits < 8:
        assert np.all(err <= s / 2 * slack)
    np.testing.assert_array_equal(o[..., 0], w.min(axis=-1))
    amin = w.argmin(axis=-1)
    assert np.all(np.take_along_axis(qg, amin[..., None], -1) == 0)
    rng_ = w.max(axis=-1) - w.min(axis=-1)
    ideal = rng_ / L
    unclamped = ideal > oracle.ref_eps() * (1 + 2.0 ** -8)
    rel = np.abs(s[..., 0] - ideal) / np.where(ideal > 0, ideal, 1.0)
    assert np.all(rel[unclamped] <= 2.0 ** -8)
    amax = w.argmax(axis=-1)
    qmax = np.take_along_axis(qg, amax[..., None], -1)[..., 0]
    # the stored scale may exceed range/L by up to 2^-9 relative: the maximum codes to L,
    # or (8 bits: L 2^-9 > 1/2 can move it) to L - 1
    if bits < 8:
        assert np.all(qmax[unclamped] == L)
    else:
        assert np.all(qmax[unclamped] >= L - 1)


def _nearest_even_code_upto(t, L):
    best, best_d = None, None
    for c in range(L + 1):
        d = abs(float(t) - c)
        if best is None or d < best_d or (d == best_d and c % 2 == 0):
            best, best_d = c, d
    return best


@pytest.mark.parametrize("bits", [2, 8])
def test_bits_rounding_by_brute_force(bits):
    """Every code is the nearest of the 2^b codes to the fp32 quotient, ties to even."""
    g = 32
    L = (1 << bits) - 1
    W = np.concatenate([_bits(workloads.gen_weight(4, 2 * g, seed=71 + bits)), adversarial_matrix(g)[:12, :2 * g]])
    Wq, sc, of = oracle.ref_quantize(W, g, bits=bits)
    q = unpack_codes(Wq, bits)
    N, K = W.shape
    wf = (W.astype(np.uint32) << 16).view(np.float32)
    sf = (sc.astype(np.uint32) << 16).view(np.float32)
    of_ = (of.astype(np.uint32) << 16).view(np.float32)
    for n in range(N):
        for k in range(K):
            j = k // g
            t = np.float32(np.float32(wf[n, k]) - of_[n, j]) / sf[n, j]
            assert q[n, k] == _nearest_even_code_upto(t, L), (n, k, float(t))


@pytest.mark.parametrize("bits", [2, 8])
def test_bits_dequantize_is_q_times_s_plus_o(bits):
    g = 64
    W = _bits(workloads.gen_weight(16, 4 * g, seed=15, outliers=True))
    Wq, sc, of = oracle.ref_quantize(W, g, bits=bits)
    Wd = oracle.ref_dequantize(Wq, sc, of, g, bits=bits)
    exact = (unpack_codes(Wq, bits).astype(np.float64) * np.repeat(bits_f64(sc), g, axis=1)
             + np.repeat(bits_f64(of), g, axis=1))
    wd = bits_f64(Wd)
    ulp_bf16 = np.spacing(np.abs(wd).astype(np.float32)).astype(np.float64) * 2 ** 16
    assert np.all(np.abs(wd - exact) <= ulp_bf16 / 2 + ulp_bf16 / 2 ** 17)


@pytest.mark.parametrize("bits", [2, 8])
@pytest.mark.parametrize("g", [32, 64, 128])
def test_bits_memory_ratio(bits, g):
    """Codes take bits/16 of the bf16 weights, plus two bf16 qparams per group."""
    W = _bits(workloads.gen_weight(8, 2 * g, seed=1))
    Wq, sc, of = oracle.ref_quantize(W, g, bits=bits)
    assert (Wq.nbytes + sc.nbytes + of.nbytes) / W.nbytes == pytest.approx((bits + 32 / g) / 16, abs=0)


def test_more_bits_are_at_least_as_accurate():
    """Mean |w - w'| falls from 2 to 4 to 8 bits on the same weights, by about
    the factor the level counts (3, 15, 255) predict."""
    W = _bits(workloads.gen_weight(128, 1024, seed=19, outliers=True))
    errs = {}
    for b in (2, 4, 8):
        Wq, sc, of = oracle.ref_quantize(W, 128, bits=b)
        errs[b] = float(np.mean(np.abs(bits_f64(oracle.ref_dequantize(Wq, sc, of, 128, bits=b)) - bits_f64(W))))
    assert errs[2] > errs[4] > errs[8], errs
    assert 3.0 < errs[2] / errs[4] < 7.0, errs


@pytest.mark.parametrize("bits", [2, 8])
def test_bits_smaller_groups_are_at_least_as_accurate(bits):
    W = _bits(workloads.gen_weight(128, 1024, seed=9, outliers=True))
    errs = []
    for g in (32, 64, 128):
        Wq, sc, of = oracle.ref_quantize(W, g, bits=bits)
        errs.append(float(np.mean(np.abs(bits_f64(oracle.ref_dequantize(Wq, sc, of, g, bits=bits)) - bits_f64(W)))))
    assert errs[0] <= errs[1] <= errs[2], errs


def test_bits_rejected():
    W = np.zeros((2, 64), np.uint16)
    for b in (1, 3, 16):
        with pytest.raises(ValueError):
            oracle.ref_quantize(W, 32, bits=b)


# ---- the fp64 linear -------------------------------------------------------

def _packed(N, K, g, seed):
    W = _bits(workloads.gen_weight(N, K, seed=seed, outliers=True))
    return oracle.ref_quantize(W, g)


@pytest.mark.parametrize("g", [32, 128])
def test_linear_one_hot_picks_a_column(g):
    """X = e_k gives y[n] = W'[n, k] exactly: pins which operand is transposed."""
    N, K = 24, 2 * g
    Wq, sc, of = _packed(N, K, g, 31)
    Wd = bits_f64(oracle.ref_dequantize(Wq, sc, of, g))
    X = np.zeros((K, K), np.uint16)
    X[np.arange(K), np.arange(K)] = 0x3F80  # 1.0
    Y = oracle.ref_linear(X, Wq, sc, of, g)
    np.testing.assert_array_equal(Y, Wd.T)


def test_linear_brute_force_triple_loop():
    g, M, N, K = 32, 3, 5, 64
    Wq, sc, of = _packed(N, K, g, 41)
    X = _bits(workloads.gen_activation(M, K, seed=42))
    Wd = bits_f64(oracle.ref_dequantize(Wq, sc, of, g))
    Xd = bits_f64(X)
    Y = oracle.ref_linear(X, Wq, sc, of, g)
    for m in range(M):
        for n in range(N):
            acc = 0.0
            for k in range(K):
                acc += Xd[m, k] * Wd[n, k]
            assert Y[m, n] == acc


@pytest.mark.parametrize("shape", [(1, 7, 32), (4, 33, 96), (9, 64, 256)])
def test_linear_matches_numpy_float64(shape):
    M, N, K = shape
    g = 32
    Wq, sc, of = _packed(N, K, g, 51 + N)
    X = _bits(workloads.gen_activation(M, K, seed=52 + N))
    Y = oracle.ref_linear(X, Wq, sc, of, g)
    ref = bits_f64(X) @ bits_f64(oracle.ref_dequantize(Wq, sc, of, g)).T
    np.testing.assert_allclose(Y, ref, rtol=1e-12, atol=1e-12)


def test_linear_scales_exactly_with_powers_of_two():
    g, M, N, K = 64, 2, 8, 128
    Wq, sc, of = _packed(N, K, g, 61)
    X = _bits(workloads.gen_activation(M, K, seed=62))
    X4 = _bits((torch.from_numpy(bits_f64(X)).to(torch.float32) * 4).to(torch.bfloat16))
    np.testing.assert_array_equal(oracle.ref_linear(X4, Wq, sc, of, g), 4 * oracle.ref_linear(X, Wq, sc, of, g))


def test_tolerance_rule():
    """|y - y_ref| <= 4e-3 |y_ref| + 1e-2 rms(y_ref), rms over the whole output."""
    y_ref = np.array([3.0, -4.0, 0.0, 0.0])  # rms = 2.5
    ok, _ = oracle.within_linear_tolerance(y_ref + np.array([0.012 + 0.025, 0, 0.025, -0.025]), y_ref)
    assert ok
    ok, worst = oracle.within_linear_tolerance(y_ref + np.array([0, 0, 0.0251, 0]), y_ref)
    assert not ok and worst > 1.0


@pytest.mark.parametrize("bits", [2, 8])
def test_bits_linear_one_hot_and_numpy(bits):
    """X = e_k picks column k of W' exactly; a random X matches numpy's fp64 matmul."""
    g, N, K = 32, 10, 96
    W = _bits(workloads.gen_weight(N, K, seed=81 + bits, outliers=True))
    Wq, sc, of = oracle.ref_quantize(W, g, bits=bits)
    Wd = bits_f64(oracle.ref_dequantize(Wq, sc, of, g, bits=bits))
    X = np.zeros((K, K), np.uint16)
    X[np.arange(K), np.arange(K)] = 0x3F80
    np.testing.assert_array_equal(oracle.ref_linear(X, Wq, sc, of, g, bits=bits), Wd.T)
    Xr = _bits(workloads.gen_activation(5, K, seed=82))
    np.testing.assert_allclose(oracle.ref_linear(Xr, Wq, sc, of, g, bits=bits), bits_f64(Xr) @ Wd.T,
                               rtol=1e-12, atol=1e-12)


def test_results_do_not_depend_on_the_thread_count():
    """The oracle's row loops may run on several threads: each row is computed the
    same way on any of them, so codes, qparams and the fp64 products are identical."""
    import torch
    from bit_weight_quantization_02_b300 import workloads as wl
    W = wl.gen_weight(300, 1024, seed=17, outliers=True).view(torch.int16).numpy().view(np.uint16)
    X = wl.gen_activation(3, 1024, seed=18).view(torch.int16).numpy().view(np.uint16)
    results = []
    for n in (1, 0):
        oracle.set_threads(n)
        q = oracle.ref_quantize(W, 64)
        results.append((q, oracle.ref_dequantize(*q, 64), oracle.ref_linear(X, *q, 64)))
    (qa, da, ya), (qb, db, yb) = results
    assert all(np.array_equal(a, b) for a, b in zip(qa, qb))
    assert np.array_equal(da, db) and np.array_equal(ya, yb)


# ---------------------------------------------------------------- bias

def test_bias_alone_when_every_weight_is_zero():
    """Codes 0 with zero offsets make every w' = 0: the linear is the bias, exactly."""
    N, K, g = 5, 64, 32
    Wq = np.zeros((N, K // 2), np.uint8)
    sc = np.full((N, K // g), 0x3C00, np.uint16)  # scale 2^-7, unused (q = 0)
    of = np.zeros((N, K // g), np.uint16)
    X = workloads.gen_activation(3, K, seed=5).view(torch.int16).numpy().view(np.uint16)
    bias = np.array([0x3F80, 0xC000, 0x0000, 0x4049, 0xBE00], np.uint16)  # 1, -2, 0, 3.140625, -0.125
    y = oracle.ref_linear(X, Wq, sc, of, g, bias=bias)
    np.testing.assert_array_equal(y, np.tile([1.0, -2.0, 0.0, 3.140625, -0.125], (3, 1)))


def test_bias_adds_its_value_to_the_product():
    """y(bias) - y(no bias) is the bias, up to the one fp64 rounding of the addition; a
    worked case: X = (1, 2, 0 ...), w' = 2^-7 q with q = (1, 3, 0 ...), bias 0.5 gives
    1 * 2^-7 + 2 * 3 * 2^-7 + 0.5 = 7/128 + 0.5 = 0.5546875."""
    W = workloads.gen_weight(64, 256, seed=21, outliers=True).view(torch.int16).numpy().view(np.uint16)
    X = workloads.gen_activation(4, 256, seed=22).view(torch.int16).numpy().view(np.uint16)
    q = oracle.ref_quantize(W, 32)
    bias = workloads.gen_activation(1, 64, seed=23).view(torch.int16).numpy().view(np.uint16)[0]
    yb = oracle.ref_linear(X, *q, 32, bias=bias)
    y0 = oracle.ref_linear(X, *q, 32)
    bf = oracle.bf16_bits_to_f64(bias)
    np.testing.assert_allclose(yb - y0, np.tile(bf, (4, 1)), rtol=0, atol=4 * np.finfo(np.float64).eps * np.abs(yb).max())
    # the worked case
    Wq = np.zeros((1, 16), np.uint8)
    Wq[0, 0] = 1 | (3 << 4)  # k = 0: q = 1, k = 1: q = 3
    sc = np.array([[0x3C00]], np.uint16)  # 2^-7
    of = np.zeros((1, 1), np.uint16)
    Xw = np.zeros((1, 32), np.uint16)
    Xw[0, 0], Xw[0, 1] = 0x3F80, 0x4000  # 1, 2
    y = oracle.ref_linear(Xw, Wq, sc, of, 32, bias=np.array([0x3F00], np.uint16))  # bias 0.5
    assert y[0, 0] == 7 / 128 + 0.5


# ---------------------------------------------------------------- int8 activations

GOLDEN_ACT = os.path.join(os.path.dirname(__file__), "golden", "activation_i8_worked_examples.txt")


def load_activation_golden(path=GOLDEN_ACT):
    """Cases of the activation file: name -> {per_token, X uint16 [M,K], scale uint32 [.], codes int8 [M,K]}."""
    cases, cur = {}, None
    for raw in open(path):
        line = raw.split("#", 1)[0].strip()
        if not line:
            continue
        key, *vals = line.split()
        if key == "case":
            cur = {"name": vals[0], "rows": [], "codes": []}
        elif key == "granularity":
            cur["per_token"] = vals[0] == "token"
        elif key == "row":
            cur["rows"].append([int(v, 16) for v in vals])
        elif key == "scale":
            cur["scale"] = np.array([int(v, 16) for v in vals], np.uint32)
        elif key == "codes":
            cur["codes"].append([int(v) for v in vals])
        elif key == "end":
            cases[cur["name"]] = {"per_token": cur["per_token"], "X": np.array(cur["rows"], np.uint16),
                                  "scale": cur["scale"], "codes": np.array(cur["codes"], np.int8)}
    return cases


ACT_CASES = load_activation_golden()


def test_activation_golden_file_is_complete():
    assert set(ACT_CASES) == {"unit_scale_half_even", "scale_two_ties", "inexact_scale", "negative_extreme",
                              "all_zero_eps",
                              "tiny_values_eps_binds", "two_rows_per_tensor", "two_rows_per_token"}
    for c in ACT_CASES.values():
        assert c["X"].shape == c["codes"].shape
        assert c["scale"].shape == ((c["X"].shape[0],) if c["per_token"] else (1,))


@pytest.mark.parametrize("name", sorted(ACT_CASES))
def test_activation_golden(name):
    c = ACT_CASES[name]
    Xq, xs = oracle.ref_quantize_activation_i8(c["X"], per_token=c["per_token"])
    np.testing.assert_array_equal(xs.view(np.uint32), c["scale"])
    np.testing.assert_array_equal(Xq, c["codes"])


@pytest.mark.parametrize("per_token", [False, True])
def test_activation_invariants(per_token):
    """|x - s_x q_x| <= s_x / 2 plus the fp32 quotient's rounding (at most 2^-24 |t| <= 128 2^-24
    code units, which can carry a value just inside a tie across it), |q| <= 127, the
    largest magnitude codes to +-127, q(-x) = -q(x), and zeros code to 0."""
    X = workloads.gen_activation(6, 512, seed=41)
    X[2] *= 1e-3  # a row far below the others (per tensor: coarse codes there)
    X[3, 7] = 0.0
    Xb = _bits(X)
    Xq, xs = oracle.ref_quantize_activation_i8(Xb, per_token=per_token)
    x = bits_f64(Xb)
    s = xs.astype(np.float64)[:, None] if per_token else np.float64(xs[0])
    assert np.abs(Xq.astype(np.int32)).max() <= 127
    assert np.all(np.abs(x - s * Xq) <= s * (0.5 + 128 * 2.0 ** -24))
    rows = range(6) if per_token else [int(np.argmax(np.abs(x).max(axis=1)))]
    for m in rows:
        k = int(np.argmax(np.abs(x[m])))
        assert abs(int(Xq[m, k])) == 127
    assert Xq[3, 7] == 0
    Xn = (Xb ^ np.uint16(0x8000))  # -x, bit for bit
    Xqn, xsn = oracle.ref_quantize_activation_i8(Xn, per_token=per_token)
    np.testing.assert_array_equal(xsn, xs)
    np.testing.assert_array_equal(Xqn, -Xq)


def test_activation_rounding_by_brute_force():
    """Each code is the integer nearest to the fp32 quotient x / s_x, ties to the even one."""
    X = workloads.gen_activation(4, 256, seed=42)
    Xb = _bits(X)
    Xq, xs = oracle.ref_quantize_activation_i8(Xb, per_token=True)
    for m in range(4):
        t = (bits_f64(Xb[m]).astype(np.float32) / xs[m]).astype(np.float64)  # the fp32 quotient
        cand = np.arange(-127, 128)[None, :]
        d = np.abs(t[:, None] - cand)
        best = d.min(axis=1, keepdims=True)
        ties = (d == best)
        for k in range(256):
            opts = cand[0][ties[k]]
            want = opts[0] if len(opts) == 1 else opts[opts % 2 == 0][0]
            assert Xq[m, k] == want


def test_activation_powers_of_two_scale_exactly():
    """X * 2^e gives s_x * 2^e and the same codes (no clamp active)."""
    Xb = _bits(workloads.gen_activation(3, 256, seed=43))
    Xq, xs = oracle.ref_quantize_activation_i8(Xb)
    X4 = (bits_f64(Xb) * 16).astype(np.float32).view(np.uint32) >> 16  # exact: bf16 * 16 is bf16
    Xq4, xs4 = oracle.ref_quantize_activation_i8(X4.astype(np.uint16))
    assert xs4[0] == np.float32(xs[0] * 16)
    np.testing.assert_array_equal(Xq4, Xq)


def _exact_weights(N, K, g, seed):
    """4-bit codes with s = 2^-7 and o = -2^-4 in every group: w' = (q - 8) 2^-7 is
    exact in bf16, so the bf16 linear and the int8 linear see the same real weights."""
    rng = np.random.default_rng(seed)
    q = rng.integers(0, 16, size=(N, K), dtype=np.uint8)
    Wq = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
    sc = np.full((N, K // g), 0x3C00, np.uint16)  # 2^-7
    of = np.full((N, K // g), 0xBD80, np.uint16)  # -2^-4
    return Wq, sc, of


@pytest.mark.parametrize("g", [32, 64, 128])
@pytest.mark.parametrize("per_token", [False, True])
def test_linear_i8_matches_the_bf16_linear_on_exact_inputs(g, per_token):
    """X = 2^-3 * integers in [-127, 127] with one +-127 per row: s_x = 2^-3 exactly and
    q_x = the integers, so the int8 linear must equal the bf16 oracle linear (pinned
    separately against a triple loop and numpy) exactly: every product and sum is exact."""
    M, N, K = 3, 40, 256
    rng = np.random.default_rng(g + per_token)
    ints = rng.integers(-127, 128, size=(M, K))
    ints[:, 5] = 127
    ints[1, 9] = -127
    X = (ints.astype(np.float32) * np.float32(0.125)).view(np.uint32) >> 16  # exact in bf16 (8 significant bits)
    X = X.astype(np.uint16)
    Wq, sc, of = _exact_weights(N, K, g, seed=g)
    Xq, xs = oracle.ref_quantize_activation_i8(X, per_token=per_token)
    assert np.all(xs == np.float32(0.125))
    np.testing.assert_array_equal(Xq, ints.astype(np.int8))
    y8 = oracle.ref_linear_i8(Xq, xs, per_token, Wq, sc, of, g)
    y16 = oracle.ref_linear(X, Wq, sc, of, g)
    np.testing.assert_array_equal(y8, y16)


def test_linear_i8_uses_each_tokens_scale():
    """Row 1 = 2 x row 0 per token: the same codes, scale 2x, so y[1] = 2 y[0] exactly;
    per tensor the shared scale is row 1's."""
    K, N, g = 128, 24, 32
    X0 = workloads.gen_activation(1, K, seed=44)
    Xb = _bits(torch.cat([X0, X0 * 2]))
    W = _bits(workloads.gen_weight(N, K, seed=45))
    Wq, sc, of = oracle.ref_quantize(W, g)
    Xq, xs = oracle.ref_quantize_activation_i8(Xb, per_token=True)
    np.testing.assert_array_equal(Xq[0], Xq[1])
    assert xs[1] == 2 * xs[0]
    y = oracle.ref_linear_i8(Xq, xs, True, Wq, sc, of, g)
    np.testing.assert_array_equal(y[1], 2 * y[0])
    Xqt, xst = oracle.ref_quantize_activation_i8(Xb, per_token=False)
    assert xst[0] == xs[1]
    np.testing.assert_array_equal(Xqt[1], Xq[1])


def test_linear_i8_offset_term_closed_form():
    """Codes q = 0 everywhere leave only the offsets: with every activation code c,
    y = s_x * c * g * sum_j o_j (exact: small integers times bf16 values)."""
    N, K, g = 6, 128, 32
    Wq = np.zeros((N, K // 2), np.uint8)
    sc = np.full((N, K // g), 0x3C00, np.uint16)
    of = np.array([[0x3F80, 0xBF00, 0x3E80, 0x4000]] * N, np.uint16)  # 1, -0.5, 0.25, 2
    Xq = np.full((2, K), 5, np.int8)
    xs = np.array([0.25], np.float32)
    y = oracle.ref_linear_i8(Xq, xs, False, Wq, sc, of, g)
    np.testing.assert_array_equal(y, np.full((2, N), 0.25 * 5 * 32 * (1 - 0.5 + 0.25 + 2)))


def test_linear_i8_bias():
    N, K, g = 16, 256, 64
    Xb = _bits(workloads.gen_activation(2, K, seed=46))
    Wq, sc, of = oracle.ref_quantize(_bits(workloads.gen_weight(N, K, seed=47)), g)
    bias = _bits(workloads.gen_activation(1, N, seed=48))[0]
    Xq, xs = oracle.ref_quantize_activation_i8(Xb)
    y0 = oracle.ref_linear_i8(Xq, xs, False, Wq, sc, of, g)
    yb = oracle.ref_linear_i8(Xq, xs, False, Wq, sc, of, g, bias=bias)
    np.testing.assert_allclose(yb - y0, np.tile(bits_f64(bias), (2, 1)), rtol=0,
                               atol=4 * np.finfo(np.float64).eps * np.abs(yb).max())
