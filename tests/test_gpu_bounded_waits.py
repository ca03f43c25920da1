"""The bounded-wait path on the GPU, without a fault or a hang.

w4_selftest_bounded_waits runs the kernels' own wait helpers against an mbarrier
that nothing completes and a split-tile sharer that never publishes, with a
1 ms limit.  Checked here:
* the call is enqueued with W4_OK, and only w4_device_fault reports the timeout
  (W4_ERR_TIMEOUT, naming the self-test in the detail), once: the flag clears;
* the owner that gave up still finished its tile, counting the missing share as
  zero (Y[r] = r + 0.5), and left the workspace at zero;
* the context stays usable: a linear right after is within tolerance and
  w4_device_fault is clean.
"""
import ctypes

import numpy as np
import pytest
import torch

import bit_weight_quantization_02_b300 as w4
from tests.test_gpu_parity import DEV, _problem, assert_linear_ok

pytestmark = pytest.mark.gpu


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream)


def test_waits_that_run_out_are_reported_and_the_context_stays_usable():
    lib = w4.load_library()
    w4.w4_device_fault(DEV)  # start clean
    ws = torch.zeros(512, dtype=torch.uint8, device=DEV)
    Y = torch.zeros(16, dtype=torch.bfloat16, device=DEV)
    st = lib.w4_selftest_bounded_waits(ctypes.c_void_p(ws.data_ptr()), ws.numel(), ctypes.c_void_p(Y.data_ptr()),
                                       1_000_000, _stream())
    assert st == 0, lib.w4_last_error_detail()
    st = lib.w4_device_fault(_stream())
    assert st == 5, f"expected W4_ERR_TIMEOUT, got {st}"
    detail = lib.w4_last_error_detail().decode()
    assert "self-test 0x3" in detail, detail  # both waits gave up: the mbarrier (1) and the owner collect (2)
    assert lib.w4_device_fault(_stream()) == 0  # cleared
    # the owner wrote its own sums, the missing share counted as zero
    np.testing.assert_array_equal(Y.float().cpu().numpy(), np.arange(16, dtype=np.float32) + 0.5)
    assert int(ws.count_nonzero()) == 0
    # the context is still usable
    (X, Wq, sc, of), y_ref = _problem(1, 1024, 2048, 32, seed=61)
    assert_linear_ok(w4.w4_linear(X, Wq, sc, of, 32), y_ref, "linear after a timed-out self-test")
    w4.w4_device_fault(DEV)


def test_self_test_refuses_bad_arguments():
    lib = w4.load_library()
    ws = torch.zeros(512, dtype=torch.uint8, device=DEV)
    Y = torch.zeros(16, dtype=torch.bfloat16, device=DEV)
    p = ctypes.c_void_p
    assert lib.w4_selftest_bounded_waits(p(ws.data_ptr()), 128, p(Y.data_ptr()), 1_000_000, _stream()) == 1
    assert lib.w4_selftest_bounded_waits(p(ws.data_ptr()), 512, p(Y.data_ptr()), 10, _stream()) == 1
    assert lib.w4_selftest_bounded_waits(p(ws.data_ptr()), 512, p(Y.data_ptr()), 10_000_000_000, _stream()) == 1
    assert lib.w4_selftest_bounded_waits(None, 512, p(Y.data_ptr()), 1_000_000, _stream()) == 1
    assert lib.w4_selftest_bounded_waits(p(ws.data_ptr() + 8), 504, p(Y.data_ptr()), 1_000_000, _stream()) == 3
    assert lib.w4_device_fault(_stream()) == 0  # nothing was launched
