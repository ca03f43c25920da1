"""GPU parity of the tensor-core batched-decode kernel (w4_linear_ex with
KERNEL_TC_DECODE), through the C ABI, against the CPU oracle: |y - y_ref| <=
4e-3 |y_ref| + 1e-2 rms(y_ref), y_ref the fp64 product with the dequantized
weights.

The shapes cover: tiles split between blocks (the owner adds the later blocks'
shares) and tiles a block covers whole, N not a multiple of 128, K not a
multiple of 64 (a last unit half past K), both qparam paths (TMA boxes when
K / g is a multiple of 8, per-thread loads otherwise), every group size, both
token tiles (16 and 32) and M = 1 .. 32.  Each output sits between guard
bytes, repeated calls are bit-identical and leave the workspace at zero; a bias
and the int8 activation scale go through the same epilogue.
"""
import numpy as np
import pytest
import torch

import oracle
import bit_weight_quantization_02_b300 as w4
from tests.test_gpu_parity import DEV, _problem, assert_linear_ok, gpu_linear, bits

pytestmark = pytest.mark.gpu

TC_M = [1, 2, 5, 8, 13, 16, 17, 24, 32]
TC_NK = [(520, 512), (1030, 1024), (200, 4160), (4096, 1536), (96, 96), (128, 14336)]


@pytest.mark.parametrize("g", [32, 64, 128])
@pytest.mark.parametrize("nk", TC_NK, ids=[f"{n}x{k}" for n, k in TC_NK])
def test_tc_decode_matches_oracle(nk, g):
    N, K = nk
    if K % g:
        pytest.skip("K % g != 0")
    ws = w4.Workspace(DEV, max(w4.w4_linear_workspace_bytes(M, N, K, g) for M in TC_M))
    for M in TC_M:
        (X, Wq, sc, of), y_ref = _problem(M, N, K, g, seed=M * 31 + N + K + g)
        y = gpu_linear(X, Wq, sc, of, g, w4.KERNEL_TC_DECODE, workspace=ws)
        assert_linear_ok(y, y_ref, f"tc decode M={M} N={N} K={K} g={g}")
    assert int(ws.buf.count_nonzero()) == 0, "the workspace did not come back to zero"
    w4.w4_device_fault(DEV)


@pytest.mark.parametrize("M", [8, 32])
def test_tc_decode_full_size_and_deterministic(M):
    """The down projection of the batched workloads (4096 x 14336, g = 64): rows sampled
    against the oracle; three calls bit-identical."""
    N, K, g = 4096, 14336, 64
    from bit_weight_quantization_02_b300 import workloads as wl
    W = wl.gen_weight(N, K, seed=11, outliers=True)
    Wq, sc, of = w4.w4_quantize(W.to(DEV), g)
    X = wl.gen_activation(M, K, seed=12).to(DEV)
    ws = w4.Workspace(DEV, w4.w4_linear_workspace_bytes(M, N, K, g))
    y = gpu_linear(X, Wq, sc, of, g, w4.KERNEL_TC_DECODE, workspace=ws)
    for _ in range(2):
        again = gpu_linear(X, Wq, sc, of, g, w4.KERNEL_TC_DECODE, workspace=ws)
        assert torch.equal(y.view(torch.int16), again.view(torch.int16)), "not deterministic"
    rows = np.random.default_rng(M).choice(N, 64, replace=False)
    y_ref = oracle.ref_linear(bits(X.cpu()), Wq.cpu().numpy()[rows], bits(sc)[rows], bits(of)[rows], g)
    ok, worst = oracle.within_linear_tolerance(oracle.bf16_bits_to_f64(bits(y))[:, rows], y_ref)
    assert ok, f"full size M={M}: worst ratio {worst:.3f}"
    w4.w4_device_fault(DEV)


def test_tc_decode_with_bias():
    N, K, g, M = 1030, 1024, 32, 9
    from bit_weight_quantization_02_b300 import workloads as wl
    (X, Wq, sc, of), _ = _problem(M, N, K, g, seed=5)
    bias = wl.gen_activation(1, N, seed=6)[0]
    y_ref = oracle.ref_linear(bits(X.cpu()), Wq.cpu().numpy(), bits(sc), bits(of), g, bias=bits(bias))
    ws = w4.Workspace(DEV, w4.w4_linear_workspace_bytes(M, N, K, g))
    y = w4.w4_linear_bias(X, Wq, sc, of, g, bias.to(DEV), kernel=w4.KERNEL_TC_DECODE, workspace=ws)
    assert_linear_ok(y, y_ref, "tc decode with a bias")


def test_tc_decode_refuses_more_than_32_tokens_and_no_workspace():
    (X, Wq, sc, of), _ = _problem(33, 256, 512, 32, seed=7)
    with pytest.raises(w4.W4Error, match="INVALID_ARG"):
        gpu_linear(X, Wq, sc, of, 32, w4.KERNEL_TC_DECODE)
    (X, Wq, sc, of), _ = _problem(8, 256, 512, 32, seed=8)
    with pytest.raises(w4.W4Error, match="INVALID_ARG"):
        gpu_linear(X, Wq, sc, of, 32, w4.KERNEL_TC_DECODE, workspace=w4.Workspace(DEV))
