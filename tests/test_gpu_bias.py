"""GPU parity of the fused bias epilogue (w4_linear_bias): every linear kernel
adds bias[n] to its fp32 sum before the one rounding to bf16, checked against
the oracle's fp64 product plus the bias, |y - y_ref| <= 4e-3 |y_ref| + 1e-2
rms(y_ref); a NULL bias gives w4_linear's result bit for bit.  Shapes span
split row tiles (stream-K owners and sharers), ragged N and every kernel:
the stream kernels (1-4 tokens, with a workspace), the batched decode kernel
(5-32), the SM-pair kernel (one token, no workspace), the cluster kernel
(2-32 tokens, no workspace) and the tcgen05 GEMM."""
import numpy as np
import pytest
import torch

import oracle
import bit_weight_quantization_02_b300 as w4
from bit_weight_quantization_02_b300 import workloads as wl
from tests.test_gpu_parity import DEV, Guarded, assert_linear_ok, bits

pytestmark = pytest.mark.gpu

CASES = [  # M, N, K, g, kernel, workspace
    (1, 4104, 4096, 32, w4.KERNEL_STREAM, True),
    (3, 1030, 1024, 64, w4.KERNEL_STREAM, True),
    (16, 520, 2048, 32, w4.KERNEL_STREAM, True),
    (1, 1037, 2048, 32, w4.KERNEL_PAIR, False),
    (5, 200, 4160, 32, w4.KERNEL_SKINNY_CLUSTER, False),
    (160, 300, 1024, 128, w4.KERNEL_GEMM, False),
    (1, 777, 3072, 32, w4.KERNEL_AUTO, True),
    (33, 129, 512, 32, w4.KERNEL_AUTO, True),
]


def _problem(M, N, K, g, seed):
    W = wl.gen_weight(N, K, seed=seed, outliers=True)
    X = wl.gen_activation(M, K, seed=seed + wl.ACT_SEED_OFFSET)
    bias = wl.gen_activation(1, N, seed=seed + 7)[0]  # bf16 ~ N(0, 1)
    q = oracle.ref_quantize(bits(W), g)
    dev = (X.to(DEV), torch.from_numpy(q[0]).to(DEV),
           torch.from_numpy(q[1].view(np.int16)).view(torch.bfloat16).to(DEV),
           torch.from_numpy(q[2].view(np.int16)).view(torch.bfloat16).to(DEV))
    return dev, bias.to(DEV), oracle.ref_linear(bits(X), *q, g, bias=bits(bias))


@pytest.mark.parametrize("case", CASES, ids=[f"M{c[0]}_{c[1]}x{c[2]}_g{c[3]}_k{c[4]}" for c in CASES])
def test_bias_epilogue_matches_oracle(case):
    M, N, K, g, kernel, with_ws = case
    (X, Wq, sc, of), bias, y_ref = _problem(M, N, K, g, seed=M + N + K)
    ws = w4.Workspace(DEV).reserve_for(M, N, K, g) if with_ws else w4.Workspace(DEV)
    Y = Guarded((M, N), torch.bfloat16)
    w4.w4_linear_bias(X, Wq, sc, of, g, bias, kernel=kernel, out=Y.t, workspace=ws)
    Y.check()
    assert_linear_ok(Y.t, y_ref, f"bias M={M} N={N} K={K} g={g} kernel={kernel}")
    # NULL bias: exactly the plain linear
    y0 = w4.w4_linear_bias(X, Wq, sc, of, g, None, kernel=kernel, workspace=ws)
    y1 = w4.w4_linear_ex(X, Wq, sc, of, g, kernel, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))
    w4.w4_device_fault(DEV)
