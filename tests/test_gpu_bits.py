"""GPU parity for 2- and 8-bit codes (the same affine group quantizer with
2^b - 1 levels: Optimum Quanto's int2 / int8 weights, torchao's int8
weight-only per group of 128), through the C ABI, against the CPU oracle:

* w4_quantize_bits / w4_dequantize_bits: bit-exact, on the hand-derived
  worked groups, ragged shapes and adversarial groups, outputs between guard
  bytes;
* w4_linear_bits on both kernels (the stream-K batched decode kernel for
  M <= 32 with a workspace, the tcgen05 GEMM otherwise): within
  |y - y_ref| <= 4e-3 |y_ref| + 1e-2 rms(y_ref), y_ref the oracle's fp64
  product with the dequantized weights; deterministic;
* full-size Llama-3-8B shapes on sampled rows and columns.
"""
import numpy as np
import pytest
import torch

import oracle
import bit_weight_quantization_02_b300 as w4
from bit_weight_quantization_02_b300 import workloads as wl
from tests.test_gpu_parity import DEV, Guarded, assert_linear_ok, bits, f64
from tests.test_oracle_pins import GOLDEN_BITS_CASES, adversarial_matrix

pytestmark = pytest.mark.gpu


def gpu_quantize_bits(W, g, b):
    N, K = W.shape
    out = (Guarded((N, K * b // 8), torch.uint8), Guarded((N, K // g), torch.bfloat16),
           Guarded((N, K // g), torch.bfloat16))
    w4.w4_quantize_bits(W, g, b, out=tuple(o.t for o in out))
    for o in out:
        o.check()
    return tuple(o.t for o in out)


def gpu_linear_bits(X, Wq, sc, of, g, b, workspace=None):
    M, N = X.shape[0], Wq.shape[0]
    Y = Guarded((M, N), torch.bfloat16)
    w4.w4_linear_bits(X, Wq, sc, of, g, b, out=Y.t, workspace=workspace)
    Y.check()
    return Y.t


def _w(N, K, seed):
    return wl.gen_weight(N, K, seed=seed, outliers=True).to(DEV)


@pytest.mark.parametrize("case", GOLDEN_BITS_CASES, ids=[c["name"] for c in GOLDEN_BITS_CASES])
def test_worked_groups_on_the_gpu(case):
    """The hand-derived groups: codes, bytes, scale, offset and w' bit for bit."""
    g, b = case["g"], case["bits"]
    W = torch.from_numpy(case["values"].reshape(1, g).view(np.int16).copy()).view(torch.bfloat16).to(DEV)
    Wq, sc, of = gpu_quantize_bits(W, g, b)
    assert int(bits(sc)[0, 0]) == case["scale"] and int(bits(of)[0, 0]) == case["offset"]
    np.testing.assert_array_equal(Wq.cpu().numpy()[0], case["bytes"])
    np.testing.assert_array_equal(bits(w4.w4_dequantize_bits(Wq, sc, of, g, b))[0], case["deq"])


@pytest.mark.parametrize("b", [2, 8])
@pytest.mark.parametrize("N,K,g", [(512, 512, 32), (300, 4224, 64), (7, 128, 128), (64, 14336, 32), (33, 2112, 32)])
def test_quantize_dequantize_bit_exact(b, N, K, g):
    W = _w(N, K, seed=900 + N)
    Wq, sc, of = gpu_quantize_bits(W, g, b)
    rq, rs, ro = oracle.ref_quantize(bits(W), g, bits=b)
    np.testing.assert_array_equal(Wq.cpu().numpy(), rq)
    np.testing.assert_array_equal(bits(sc), rs)
    np.testing.assert_array_equal(bits(of), ro)
    Wd = Guarded((N, K), torch.bfloat16)
    w4.w4_dequantize_bits(Wq, sc, of, g, b, out=Wd.t)
    Wd.check()
    np.testing.assert_array_equal(bits(Wd.t), oracle.ref_dequantize(rq, rs, ro, g, bits=b))


@pytest.mark.parametrize("b", [2, 8])
@pytest.mark.parametrize("g", [32, 128])
def test_quantize_adversarial_groups(b, g):
    """Constant, two-valued, signed-zero, subnormal, huge-range and half-step groups."""
    Wb = adversarial_matrix(g, seed=11 + b)
    W = torch.from_numpy(Wb.view(np.int16).copy()).view(torch.bfloat16).to(DEV)
    Wq, sc, of = gpu_quantize_bits(W, g, b)
    rq, rs, ro = oracle.ref_quantize(Wb, g, bits=b)
    np.testing.assert_array_equal(Wq.cpu().numpy(), rq)
    np.testing.assert_array_equal(bits(sc), rs)
    np.testing.assert_array_equal(bits(of), ro)


@pytest.mark.parametrize("b", [2, 8])
@pytest.mark.parametrize("M", [1, 3, 8, 13, 32])
@pytest.mark.parametrize("N,K,g", [(512, 512, 32), (300, 4224, 64), (1000, 1024, 128), (200, 1024, 64)])
def test_linear_batched_decode(b, M, N, K, g):
    """M <= 32 with a workspace: the stream-K kernel with 64-row units (ragged N, ragged K tail;
    qparams by TMA boxes of 8 groups where K/g is a multiple of 8, by cp.async otherwise)."""
    W = _w(N, K, seed=1000 + N + M)
    X = wl.gen_activation(M, K, seed=1100 + M).to(DEV)
    Wq, sc, of = gpu_quantize_bits(W, g, b)
    y = gpu_linear_bits(X, Wq, sc, of, g, b)
    y_ref = oracle.ref_linear(bits(X), Wq.cpu().numpy(), bits(sc), bits(of), g, bits=b)
    assert_linear_ok(y, y_ref, f"w{b} batched M={M} N={N} K={K} g={g}")


@pytest.mark.parametrize("b", [2, 8])
@pytest.mark.parametrize("M", [2, 33, 300])
@pytest.mark.parametrize("N,K,g", [(256, 512, 32), (300, 4224, 64)])
def test_linear_tensor_core_gemm(b, M, N, K, g):
    """The tcgen05 GEMM: M > 32, or M <= 32 without a workspace."""
    W = _w(N, K, seed=1200 + N + M)
    X = wl.gen_activation(M, K, seed=1300 + M).to(DEV)
    Wq, sc, of = gpu_quantize_bits(W, g, b)
    ws = w4.Workspace(DEV)  # empty: M <= 32 falls back to the GEMM
    y = gpu_linear_bits(X, Wq, sc, of, g, b, workspace=ws)
    y_ref = oracle.ref_linear(bits(X), Wq.cpu().numpy(), bits(sc), bits(of), g, bits=b)
    assert_linear_ok(y, y_ref, f"w{b} gemm M={M} N={N} K={K} g={g}")


@pytest.mark.parametrize("b", [2, 8])
def test_eight_bit_gemm_products_use_the_dequantized_weights(b):
    """X = I picks columns of W' exactly through the GEMM at 8 bits (w' = bf16(fp32(q s + o))
    bit for bit); at 2 bits the single-rounding w' may differ from w4_dequantize_bits by one ulp."""
    N, K, g = 128, 256, 32
    Wq, sc, of = gpu_quantize_bits(_w(N, K, seed=77), g, b)
    X = torch.eye(K, dtype=torch.bfloat16, device=DEV)
    y = gpu_linear_bits(X, Wq, sc, of, g, b, workspace=w4.Workspace(DEV))
    Wd = w4.w4_dequantize_bits(Wq, sc, of, g, b)
    if b == 8:
        np.testing.assert_array_equal(bits(y), bits(Wd.t().contiguous()))
    else:
        ulp = np.spacing(np.abs(f64(Wd)).astype(np.float32)).astype(np.float64) * 2 ** 16
        assert np.all(np.abs(f64(y) - f64(Wd).T) <= ulp.T + 1e-30)


@pytest.mark.parametrize("b", [2, 8])
def test_linear_is_deterministic(b):
    N, K, g = 4096, 4096, 128
    Wq, sc, of = gpu_quantize_bits(_w(N, K, seed=5), g, b)
    for M in (1, 16):
        X = wl.gen_activation(M, K, seed=6).to(DEV)
        y1 = gpu_linear_bits(X, Wq, sc, of, g, b)
        y2 = gpu_linear_bits(X, Wq, sc, of, g, b)
        np.testing.assert_array_equal(bits(y1), bits(y2))


@pytest.mark.parametrize("b,g", [(8, 128), (2, 32)])
@pytest.mark.parametrize("N,K", [(14336, 4096), (4096, 14336)])
def test_full_size_sampled(b, g, N, K):
    """Llama-3-8B gate/up and down shapes at M = 1, 16 (decode) and 2048 (GEMM), on 48 sampled
    output columns (and 24 sampled tokens at M = 2048) that the oracle computes one by one."""
    W = wl.gen_weight(N, K, seed=wl.weight_seed(6, 0, b), outliers=True, device=DEV)
    Wq, sc, of = gpu_quantize_bits(W, g, b)
    rng = np.random.default_rng(N + b)
    cols = np.sort(rng.choice(N, 48, replace=False))
    rq, rs, ro = oracle.ref_quantize(bits(W[torch.from_numpy(cols).to(DEV)]), g, bits=b)
    np.testing.assert_array_equal(Wq[torch.from_numpy(cols).to(DEV)].cpu().numpy(), rq)
    del W
    for M in (1, 16, 2048):
        X = wl.gen_activation(M, K, seed=7 + M, device=DEV)
        y = w4.w4_linear_bits(X, Wq, sc, of, g, b)
        rows = np.arange(M) if M <= 16 else np.sort(rng.choice(M, 24, replace=False))
        y_ref = oracle.ref_linear(bits(X[torch.from_numpy(rows).to(DEV)]), rq, rs, ro, g, bits=b)
        ys = y[torch.from_numpy(rows).to(DEV)][:, torch.from_numpy(cols).to(DEV)]
        assert_linear_ok(ys, y_ref, f"w{b} full size M={M} N={N} K={K}")
