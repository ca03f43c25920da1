"""The tensor-core GEMM's stream-K tail on the GPU, against the oracle.

With a workspace (w4_linear_workspace_bytes > 16 MiB for the shape), the tiles of
a part-empty last round are split by k blocks over the persistent blocks: a
block that shares a tile publishes its fp32 partial sums and a flag, and the
block holding the tile's first k block adds them in block order.  Checked here:

* the split result is within the linear tolerance of the oracle, on shapes with
  ragged N and M, many sharers per tile (few tiles) and one or two (a full round
  split), every group size and both qparam paths;
* the same call without a workspace (whole tiles) is within tolerance too;
* the split result is the same bits on every run (fixed summation order);
* the workspace's flag region is zero again afterwards, and no wait timed out.
"""
import numpy as np
import pytest
import torch

import oracle
import bit_weight_quantization_02_b300 as w4
from bit_weight_quantization_02_b300 import workloads as wl
from tests.test_gpu_parity import DEV, Guarded, _problem, f64

pytestmark = pytest.mark.gpu

# (M, N, K, g): 10 tiles split 8 ways; 18 tiles split 8 ways at g=128; ragged M and N; qparams by
# TMA (K/g a multiple of 8) and per thread (4160/32 = 130 groups); 32 tiles split ~4.6 ways at g=64.
# SAMPLED (oracle on sampled rows): 168 tiles (a full round split), and 297 tiles (a round of
# whole tiles before the split ones).
SPLIT_SHAPES = [(300, 520, 4096, 32), (257, 1030, 8192, 128), (40, 2056, 4160, 32), (300, 2048, 14336, 64)]
SAMPLED = [(600, 7168, 8192, 32), (256, 38016, 4096, 32)]


def _u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _linear(X, Wq, sc, of, g, ws, bits=4):
    M, N = X.shape[0], Wq.shape[0]
    Y = Guarded((M, N), torch.bfloat16)
    if bits == 4:
        w4.w4_linear_ex(X, Wq, sc, of, g, w4.KERNEL_GEMM, out=Y.t, workspace=ws)
    else:
        w4.w4_linear_bits(X, Wq, sc, of, g, bits, out=Y.t, workspace=ws)
    Y.check()
    return Y.t.clone()


@pytest.mark.parametrize("shape", SPLIT_SHAPES, ids=[f"m{m}_{n}x{k}g{g}" for m, n, k, g in SPLIT_SHAPES])
def test_split_tail_matches_oracle_and_whole_tiles(shape):
    M, N, K, g = shape
    need = w4.w4_linear_workspace_bytes(M, N, K, g)
    assert need > 16 << 20, "this shape is meant to split its last round"
    (X, Wq, sc, of), y_ref = _problem(M, N, K, g, seed=M + N + K)
    ws = w4.Workspace(DEV, need)
    y_split = _linear(X, Wq, sc, of, g, ws)
    ok, worst = oracle.within_linear_tolerance(f64(y_split), y_ref)
    assert ok, f"split M={M} N={N} K={K} g={g}: worst ratio {worst:.3f}"
    y_whole = _linear(X, Wq, sc, of, g, w4.Workspace(DEV))  # no workspace: whole tiles
    ok, worst = oracle.within_linear_tolerance(f64(y_whole), y_ref)
    assert ok, f"whole tiles M={M} N={N} K={K} g={g}: worst ratio {worst:.3f}"
    for _ in range(3):  # deterministic: the sharers' sums are added in block order
        assert torch.equal(_linear(X, Wq, sc, of, g, ws).view(torch.int16), y_split.view(torch.int16))
    assert int(ws.buf[: 16 << 20].count_nonzero()) == 0, "split-tile flags left set"
    w4.w4_device_fault(DEV)


def test_split_tail_with_bias_and_other_code_widths():
    M, N, K, g = 300, 520, 4096, 32
    ws = w4.Workspace(DEV, w4.w4_linear_workspace_bytes(M, N, K, g))
    (X, Wq, sc, of), _ = _problem(M, N, K, g, seed=7)
    bias = torch.randn(N, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16).to(DEV)
    Y = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    w4.w4_linear_bias(X, Wq, sc, of, g, bias, out=Y, workspace=ws)
    Xb = _u16(X)
    y_ref = oracle.ref_linear(Xb, Wq.cpu().numpy(), _u16(sc), _u16(of), g, bias=_u16(bias))
    ok, worst = oracle.within_linear_tolerance(f64(Y), y_ref)
    assert ok, f"split with bias: worst ratio {worst:.3f}"
    for bits in (2, 8):
        W = torch.randn(N, K, generator=torch.Generator().manual_seed(bits)) * 0.02
        Wq_b, sc_b, of_b = w4.w4_quantize_bits(W.to(torch.bfloat16).to(DEV), g, bits)
        y_b = _linear(X, Wq_b, sc_b, of_b, g, ws, bits=bits)
        y_ref = oracle.ref_linear(Xb, Wq_b.cpu().numpy(), _u16(sc_b), _u16(of_b), g, bits=bits)
        ok, worst = oracle.within_linear_tolerance(f64(y_b), y_ref)
        assert ok, f"split {bits}-bit: worst ratio {worst:.3f}"
    assert int(ws.buf[: 16 << 20].count_nonzero()) == 0
    w4.w4_device_fault(DEV)


@pytest.mark.parametrize("shape", SAMPLED, ids=[f"m{m}_{n}x{k}g{g}" for m, n, k, g in SAMPLED])
def test_split_tail_large_sampled(shape):
    """A full round split, and a round of whole tiles before the split ones (oracle on sampled rows)."""
    M, N, K, g = shape
    need = w4.w4_linear_workspace_bytes(M, N, K, g)
    assert need > 16 << 20, "this shape is meant to split its last round"
    W = wl.gen_weight(N, K, seed=21, device=DEV)
    Wq, sc, of = w4.w4_quantize(W, g)
    X = wl.gen_activation(M, K, seed=22, device=DEV)
    ws = w4.Workspace(DEV, need)
    Y = _linear(X, Wq, sc, of, g, ws)
    rows = np.unique(np.concatenate([np.arange(0, N, 97), np.arange(N - 128, N)]))  # every tile region, the last tile
    y_ref = oracle.ref_linear(_u16(X), Wq.cpu().numpy()[rows], _u16(sc)[rows], _u16(of)[rows], g)
    ok, worst = oracle.within_linear_tolerance(f64(Y[:, rows]), y_ref)
    assert ok, f"split M={M} N={N} K={K} g={g}: worst ratio {worst:.3f}"
    assert torch.equal(_linear(X, Wq, sc, of, g, ws).view(torch.int16), Y.view(torch.int16))
    assert int(ws.buf[: 16 << 20].count_nonzero()) == 0
    w4.w4_device_fault(DEV)


@pytest.mark.parametrize("split", [False, True], ids=["whole", "split"])
def test_gemm_rows_not_16_byte_multiples(split):
    """N = 1030 (Y's rows are not 16-byte multiples, so no TMA store): the GEMM writes Y with plain
    stores, whole tiles and split ones, within tolerance of the oracle and inside Y only."""
    M, N, K, g = 300, 1030, 4096, 32
    (X, Wq, sc, of), y_ref = _problem(M, N, K, g, seed=41)
    if split:
        need = w4.w4_linear_workspace_bytes(M, N, K, g)
        assert need > 16 << 20, "this shape is meant to split its last round"
        ws = w4.Workspace(DEV, need)
    else:
        ws = w4.Workspace(DEV)
    Y = Guarded((M, N), torch.bfloat16)
    w4.w4_linear_ex(X, Wq, sc, of, g, w4.KERNEL_GEMM, out=Y.t, workspace=ws)
    Y.check()
    ok, worst = oracle.within_linear_tolerance(f64(Y.t), y_ref)
    assert ok, f"N={N} ({'split' if split else 'whole'}): worst ratio {worst:.3f}"
    w4.w4_device_fault(DEV)
