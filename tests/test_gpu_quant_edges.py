"""Quantize edge cases on the GPU, bit-exact against the oracle, at 2, 4 and 8 bits.

The quantize kernel gives each lane a segment of 64 consecutive weights: two groups at
g = 32, one at g = 64, half of one at g = 128. Two paths of that design get their own cases:

* A g = 32 tensor with an odd number of groups leaves the last segment with one group. Only
  that group's codes and qparams may be written. The outputs are canary-guarded, so a store
  for the missing second group shows.
* The group min / max comes from the hardware's bf16 min / max, which does not order -0.0
  against +0.0. A group whose min or max is a zero is redone on order keys, where -0.0 ranks
  below +0.0 (the header's reading). The cases cover a non-positive group with and without
  +0.0 (max +0.0 or -0.0), a non-negative group with and without -0.0 (min -0.0 or +0.0), an
  all -0.0 group, an all +0.0 group, and a control group without zeros.
"""
import numpy as np
import pytest
import torch

import oracle
import bit_weight_quantization_02_b300 as w4
from tests.test_gpu_parity import DEV, Guarded, bits

pytestmark = pytest.mark.gpu


def _bf16_bits(a: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _check(Wb: np.ndarray, g: int, b: int):
    N, K = Wb.shape
    W = torch.from_numpy(Wb.view(np.int16).copy()).view(torch.bfloat16).to(DEV)
    out = (Guarded((N, K * b // 8), torch.uint8), Guarded((N, K // g), torch.bfloat16),
           Guarded((N, K // g), torch.bfloat16))
    w4.w4_quantize_bits(W, g, b, out=tuple(o.t for o in out))
    for o in out:
        o.check()
    rq, rs, ro = oracle.ref_quantize(Wb, g, bits=b)
    np.testing.assert_array_equal(out[0].t.cpu().numpy(), rq)
    np.testing.assert_array_equal(bits(out[1].t), rs)
    np.testing.assert_array_equal(bits(out[2].t), ro)
    w4.w4_device_fault(DEV)


# (N, K) with an odd number of g = 32 groups: 1, 3, 21, 25 and 33 * 129 of them
ODD = [(1, 32), (3, 32), (7, 96), (5, 160), (33, 4128)]


@pytest.mark.parametrize("b", [2, 4, 8])
@pytest.mark.parametrize("shape", ODD, ids=[f"{n}x{k}" for n, k in ODD])
def test_odd_number_of_g32_groups(shape, b):
    N, K = shape
    rng = np.random.default_rng(N * 1000 + K + b)
    _check(_bf16_bits(rng.normal(0, 0.02, (N, K))), 32, b)


def _zero_rows(g: int, seed: int) -> np.ndarray:
    """Rows of four groups each; every group of a row follows the row's recipe."""
    rng = np.random.default_rng(seed)
    K = 4 * g
    neg = -rng.uniform(0.05, 1.0, (K,))
    pos = rng.uniform(0.05, 1.0, (K,))
    rows = []
    r = neg.copy(); r[3::g // 4] = 0.0; r[5::g // 4] = -0.0; rows.append(r)    # max must be +0.0
    r = neg.copy(); r[5::g // 4] = -0.0; rows.append(r)                        # max must be -0.0
    r = pos.copy(); r[3::g // 4] = 0.0; r[5::g // 4] = -0.0; rows.append(r)    # min must be -0.0
    r = pos.copy(); r[3::g // 4] = 0.0; rows.append(r)                         # min must be +0.0
    rows.append(np.full(K, -0.0))                                              # all -0.0
    rows.append(np.zeros(K))                                                   # all +0.0
    r = np.zeros(K); r[1::2] = -0.0; rows.append(r)                            # +0.0 and -0.0 only
    rows.append(rng.normal(0, 0.5, (K,)))                                      # control, no zeros
    return _bf16_bits(np.stack(rows))


@pytest.mark.parametrize("b", [2, 4, 8])
@pytest.mark.parametrize("g", [32, 64, 128])
def test_signed_zero_group_bounds(g, b):
    Wb = _zero_rows(g, seed=17 * g + b)
    # the recipes above need the zeros' signs to survive the bf16 conversion
    assert (Wb[1] == 0x8000).any() and (Wb[2] == 0x0000).any() and (Wb[4] == 0x8000).all()
    _check(Wb, g, b)
    # the same rows inside a larger tensor, so the warp that meets them also holds ordinary groups
    rng = np.random.default_rng(5 + g + b)
    big = _bf16_bits(rng.normal(0, 0.02, (40, 4 * g)))
    big[7:7 + Wb.shape[0]] = Wb
    _check(big, g, b)
