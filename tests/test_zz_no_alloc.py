"""w4_linear_static: the linear for callers that cannot allocate device memory.

Some callers may not call cudaMalloc or any allocating routine (a plugin inside
another framework that owns every device allocation, a service with a fixed
device-memory budget), so w4_linear_static runs the stream-K decode kernel with
a device array that the library itself holds as workspace.  This file checks,
through the C ABI, that two calls in a row give what w4_linear (with a
caller-provided workspace) gives on the same inputs, bit for bit (both run the
same plan), that the first result is within the linear's tolerance of the
oracle, and that once the first call has set the array aside, later calls
leave the device's free memory unchanged.  It is collected last so that a run stopping at the first failure
has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import bit_weight_quantization_02_b300 as w4
from bit_weight_quantization_02_b300 import workloads as wl

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _static_fn():
    fn = w4.load_library().w4_linear_static
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                   ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn


def _problem(M, N, K, g, seed, dev):
    W = wl.gen_weight(N, K, seed=seed, outliers=True, device=dev)
    X = wl.gen_activation(M, K, seed=seed + wl.ACT_SEED_OFFSET, device=dev)
    Wq, sc, of = w4.w4_quantize(W, g)
    return X, Wq, sc, of


def test_static_scratch_entry_matches_w4_linear_on_two_calls_in_a_row():
    dev = torch.device("cuda:0")
    fn = _static_fn()
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    cases = [(1, 4096, 4096, 32, 71), (5, 1536, 2048, 64, 72)]
    probs = [(_problem(M, N, K, g, seed, dev), M, N, K, g) for M, N, K, g, seed in cases]
    rounds = [[torch.empty((M, N), dtype=torch.bfloat16, device=dev) for _, M, N, K, g in probs] for _ in range(2)]

    def call_all(outs):  # the two cases in a row, no synchronization between them
        for ((X, Wq, sc, of), M, N, K, g), Y in zip(probs, outs):
            st = fn(X.data_ptr(), M, K, Wq.data_ptr(), sc.data_ptr(), of.data_ptr(), N, g, Y.data_ptr(), stream)
            assert st == 0, w4.load_library().w4_last_error_detail()

    call_all(rounds[0])  # the first calls: the array (and each kernel's code) may be loaded here
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info(dev)[0]
    call_all(rounds[1])  # later calls allocate nothing
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info(dev)[0] == free_before
    for a, b in zip(*rounds):  # calls that share the array one after another give the same bits
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    outs = rounds[1]
    for i, (((X, Wq, sc, of), M, N, K, g), Y) in enumerate(zip(probs, outs)):
        # the same plan and launch as w4_linear's stream kernel with a caller workspace: the same bits
        ws = w4.Workspace(dev).reserve_for(M, N, K, g)
        Y_ws = w4.w4_linear_ex(X, Wq, sc, of, g, w4.KERNEL_STREAM, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(Y.view(torch.int16), Y_ws.view(torch.int16)), \
            f"w4_linear_static differs from w4_linear (M={M} N={N} K={K} g={g})"
        if i == 0:  # and against the oracle's fp64 product
            y_ref = oracle.ref_linear(_bits(X), Wq.cpu().numpy(), _bits(sc), _bits(of), g)
            ok, worst = oracle.within_linear_tolerance(oracle.bf16_bits_to_f64(_bits(Y)), y_ref)
            assert ok, f"w4_linear_static outside the linear tolerance: worst ratio {worst:.3f}"


def test_static_scratch_entry_rejects_what_it_cannot_run():
    # every M <= 8 problem's workspace fits the array (tests/test_abi_host.py checks the size rule on
    # the CPU); M > 8 and an odd K / group_size are refused before any launch
    dev = torch.device("cuda:0")
    fn = _static_fn()
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    X = torch.zeros((9, 256), dtype=torch.bfloat16, device=dev)
    Wq = torch.zeros((16, 128), dtype=torch.uint8, device=dev)
    sc = torch.zeros((16, 8), dtype=torch.bfloat16, device=dev)
    Y = torch.zeros((9, 16), dtype=torch.bfloat16, device=dev)
    st = fn(X.data_ptr(), 9, 256, Wq.data_ptr(), sc.data_ptr(), sc.data_ptr(), 16, 32, Y.data_ptr(), stream)
    assert st == 1 and b"M <= 8" in w4.load_library().w4_last_error_detail()
    st = fn(X.data_ptr(), 1, 96, Wq.data_ptr(), sc.data_ptr(), sc.data_ptr(), 16, 32, Y.data_ptr(), stream)
    assert st == 1 and b"even" in w4.load_library().w4_last_error_detail()
