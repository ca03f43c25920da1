"""GPU parity of the one-token SM-pair kernel (w4_linear_ex with KERNEL_PAIR,
and w4_linear's automatic choice at M = 1), through the C ABI, against the CPU
oracle: |y - y_ref| <= 4e-3 |y_ref| + 1e-2 rms(y_ref), y_ref the fp64 product
with the dequantized weights.

The shapes cover: several 64-row stages and 256-row passes per cluster, row
ranges whose last group is cut into 32/16/8-row boxes, N not a multiple of 8,
fewer 8-row groups than clusters, an odd number of 512-k stages (the two
blocks of a pair take unequal halves of K), K below one stage (the second
block has no k at all) and every group size.  Each output sits between guard
bytes, repeated calls must be bit-identical, and the kernel needs no
workspace.
"""
import numpy as np
import pytest
import torch

import oracle
import bit_weight_quantization_02_b300 as w4
from tests.test_gpu_parity import DEV, _problem, assert_linear_ok, gpu_linear, bits

pytestmark = pytest.mark.gpu

PAIR_CASES = [
    (512, 512, 32), (4096, 4096, 32), (1024, 4096, 32), (4096, 4096, 128), (1024, 4096, 128),
    (1000, 1024, 32), (1037, 1536, 32), (8, 256, 32), (16, 512, 64), (24, 1024, 128), (3, 256, 32),
    (777, 3072, 32), (592, 768, 32), (129, 256, 32), (600, 16384, 32), (40000, 2048, 32), (2056, 2048, 64),
    (4096, 14336, 64),
]


@pytest.mark.parametrize("case", PAIR_CASES, ids=[f"{n}x{k}g{g}" for n, k, g in PAIR_CASES])
def test_pair_kernel_matches_oracle_and_is_deterministic(case):
    N, K, g = case
    (X, Wq, sc, of), y_ref = _problem(1, N, K, g, seed=N + 3 * K + g)
    no_ws = w4.Workspace(DEV)  # an empty workspace: the pair kernel needs none
    y = gpu_linear(X, Wq, sc, of, g, w4.KERNEL_PAIR, workspace=no_ws)
    assert_linear_ok(y, y_ref, f"pair N={N} K={K} g={g}")
    for _ in range(2):
        again = gpu_linear(X, Wq, sc, of, g, w4.KERNEL_PAIR, workspace=no_ws)
        assert torch.equal(y.view(torch.int16), again.view(torch.int16)), "pair kernel not deterministic"
    w4.w4_device_fault(DEV)


def test_auto_picks_the_pair_kernel_for_one_token_without_a_workspace():
    (X, Wq, sc, of), y_ref = _problem(1, 2048, 4096, 32, seed=91)
    no_ws = w4.Workspace(DEV)
    y_auto = gpu_linear(X, Wq, sc, of, 32, w4.KERNEL_AUTO, workspace=no_ws)
    y_pair = gpu_linear(X, Wq, sc, of, 32, w4.KERNEL_PAIR, workspace=no_ws)
    assert torch.equal(y_auto.view(torch.int16), y_pair.view(torch.int16))
    assert_linear_ok(y_auto, y_ref, "auto M=1")


def test_pair_kernel_refuses_what_it_cannot_run():
    (X, Wq, sc, of), _ = _problem(2, 64, 512, 32, seed=5)
    with pytest.raises(w4.W4Error, match="INVALID_ARG"):
        gpu_linear(X, Wq, sc, of, 32, w4.KERNEL_PAIR)
    (X, Wq, sc, of), _ = _problem(1, 64, 96, 32, seed=6)  # K / g = 3: qparam rows not whole 16-byte pieces
    with pytest.raises(w4.W4Error, match="INVALID_ARG"):
        gpu_linear(X, Wq, sc, of, 32, w4.KERNEL_PAIR)
    (X, Wq, sc, of), y_ref = _problem(1, 64, 96, 32, seed=6)  # auto falls back to another kernel
    assert_linear_ok(gpu_linear(X, Wq, sc, of, 32), y_ref, "auto M=1 K=96")


def test_pair_chain_reads_each_previous_output():
    """Each call's X is the previous call's Y: the next launch streams its
    weights early but must read X only once the previous launch is complete."""
    K = 2048
    probs = [_problem(1, K, K, 64, seed=300 + i) for i in range(8)]
    y = probs[0][0][0]
    outs = []
    for (X, Wq, sc, of), _ in probs:
        y = w4.w4_linear_ex(y, Wq, sc, of, 64, w4.KERNEL_PAIR)
        outs.append(y)
    torch.cuda.synchronize()
    y = probs[0][0][0]
    for ((X, Wq, sc, of), _), got in zip(probs, outs):
        q = Wq.cpu().numpy()
        s = bits(sc)
        o = bits(of)
        y_ref = oracle.ref_linear(bits(y), q, s, o, 64)
        assert_linear_ok(got, y_ref, "pair chain")
        y = got
