"""GPU parity of the int8-activation path, through the C ABI, against the CPU
oracle.

* w4_quantize_activation_i8: codes and scales bit-exact (per tensor and per
  token), on the hand-derived cases, seeded activations of several shapes,
  rows of zeros, rows far below the others and exact ties; outputs between
  guard bytes.
* w4_linear_i8: within |y - y_ref| <= 4e-3 |y_ref| + 1e-2 rms(y_ref) of the
  oracle's integer-accumulated linear, for M = 1 .. 256 (the direct int8 stream
  kernel up to 4 tokens; the widened codes on the batch kernel up to 32 and
  the tensor-core kernel above), every group size, both granularities, with
  and without a bias, odd group counts (the widened path at any M); repeated
  calls bit-identical (the workspace comes back clean).
"""
import numpy as np
import pytest
import torch

import oracle
import bit_weight_quantization_02_b300 as w4
from bit_weight_quantization_02_b300 import workloads as wl
from tests.test_gpu_parity import DEV, Guarded, bits, f64
from tests.test_oracle_pins import ACT_CASES

pytestmark = pytest.mark.gpu


def gpu_act(X: torch.Tensor, per_token: bool):
    M, K = X.shape
    Xq = Guarded((M, K), torch.int8)
    xs = Guarded((M if per_token else 1,), torch.float32)
    w4.w4_quantize_activation_i8(X, per_token, out=(Xq.t, xs.t))
    Xq.check()
    xs.check()
    return Xq.t, xs.t


def _x16(X_bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(X_bits).view(np.int16)).view(torch.bfloat16).to(DEV)


@pytest.mark.parametrize("name", sorted(ACT_CASES))
def test_activation_golden_cases(name):
    c = ACT_CASES[name]
    M, K = c["X"].shape
    X = np.zeros((M, 32), np.uint16)  # K a multiple of 32: pad with zeros (they change no maximum, code to 0)
    X[:, :K] = c["X"]
    Xq, xs = gpu_act(_x16(X), c["per_token"])
    np.testing.assert_array_equal(xs.cpu().numpy().view(np.uint32), c["scale"])
    np.testing.assert_array_equal(Xq.cpu().numpy()[:, :K], c["codes"])
    assert not Xq.cpu().numpy()[:, K:].any()


ACT_SHAPES = [(1, 4096), (1, 14336), (3, 512), (16, 4096), (33, 1024), (300, 2048), (2048, 4096)]


@pytest.mark.parametrize("per_token", [False, True], ids=["tensor", "token"])
@pytest.mark.parametrize("shape", ACT_SHAPES, ids=[f"{m}x{k}" for m, k in ACT_SHAPES])
def test_activation_quantize_bit_exact(shape, per_token):
    M, K = shape
    X = wl.gen_activation(M, K, seed=M * 7 + K)
    if M > 2:
        X[1] = 0.0          # a zero row
        X[2] *= 1e-4        # a row far below the others
    Xb = bits(X)
    rq, rs = oracle.ref_quantize_activation_i8(Xb, per_token=per_token)
    Xq, xs = gpu_act(X.to(DEV), per_token)
    np.testing.assert_array_equal(xs.cpu().numpy().view(np.uint32), rs.view(np.uint32))
    np.testing.assert_array_equal(Xq.cpu().numpy(), rq)


def test_activation_quantize_exact_ties():
    """max |x| = 63.5: s = 0.5 exactly and every x = 0.25 i sits on a half-integer or an
    integer of x / s; half-integers go to the even code."""
    K = 256
    i = np.arange(K) - 127
    x = (i.astype(np.float32) * np.float32(0.25)).view(np.uint32) >> 16
    X = np.tile(x.astype(np.uint16), (2, 1))
    X[:, 0] = 0x427E  # 63.5
    X[1, 1] = 0xC27E  # -63.5
    rq, rs = oracle.ref_quantize_activation_i8(X)
    assert rs[0] == np.float32(0.5)
    Xq, xs = gpu_act(_x16(X), False)
    np.testing.assert_array_equal(Xq.cpu().numpy(), rq)


def _near_half_integer_rows(R, K, seed, common=False):
    """R rows of K bf16 values, each row led by its own maximum m (one m for all rows when
    common, for one scale per tensor), the rest mostly values x
    for which the fp32 quotient x / s (s = m / 127) lies within 2^-13 of a half-integer: the
    codes there come from the kernels' division fallback, or from their multiply path right at
    its threshold.  Found by scanning every positive bf16 value below m on the host (IEEE fp32
    division in numpy, as the method states it)."""
    rng = np.random.default_rng(seed)
    pos = np.arange(1, 0x7F80, dtype=np.uint32)          # positive finite bf16 bit patterns
    vals = (pos << 16).view(np.float32)
    X = np.zeros((R, K), np.uint16)
    near_total = 0
    for r in range(R):
        if not common:
            mb = int(rng.integers(0x3F80, 0x42C8))  # m in [1, 100)
        elif r == 0:  # the m in [1, 100) with the most quotients near, but not on, a half-integer
            best = -1
            for cb in range(0x3F80, 0x42C8):
                cm = np.array([cb << 16], np.uint32).view(np.float32)[0]
                cs = np.float32(cm / np.float32(127.0))
                cq = (vals[vals <= cm] / cs).astype(np.float32)
                cd = np.abs(np.abs(cq - np.rint(cq)) - np.float32(0.5))
                n = int(((cd > 0) & (cd < np.float32(2.0 ** -13))).sum())
                if n > best:
                    best, mb = n, cb
        m = np.float32(np.array([mb << 16], np.uint32).view(np.float32)[0])
        s = np.float32(m / np.float32(127.0))
        below = vals <= m
        q = (vals[below] / s).astype(np.float32)
        d = np.abs(q - np.rint(q))
        near = pos[below][np.abs(d - np.float32(0.5)) < np.float32(2.0 ** -13)]
        rng.shuffle(near)
        near = near[: K - 1 - K // 4]
        near_total += len(near)
        fill = rng.choice(pos[below], size=K - 1 - len(near))
        row = np.concatenate([near, fill]).astype(np.uint16)
        row |= (rng.integers(0, 2, size=row.size) << 15).astype(np.uint16)  # random signs
        X[r, 0] = mb
        X[r, 1:] = row
    return X, near_total


@pytest.mark.parametrize("per_token", [False, True], ids=["tensor", "token"])
def test_activation_codes_near_half_integers(per_token):
    """Codes of quotients within 2^-13 of a half-integer are bit-exact against the oracle, in the
    activation kernels and in the stream kernel that quantizes X itself."""
    R, K = 256, 512
    X, near = _near_half_integer_rows(R, K, seed=11, common=not per_token)
    assert near >= 200, near  # enough values on the fallback side of the threshold
    rq, rs = oracle.ref_quantize_activation_i8(X, per_token=per_token)
    Xq, xs = gpu_act(_x16(X), per_token)
    np.testing.assert_array_equal(xs.cpu().numpy().view(np.uint32), rs.view(np.uint32))
    np.testing.assert_array_equal(Xq.cpu().numpy(), rq)
    W = wl.gen_weight(136, K, seed=5, outliers=False)
    Wq, sc, of = w4.w4_quantize(W.to(DEV), 32)
    for r0 in range(0, 16, 4):  # the one-call path (one kernel for up to 4 tokens) on the same rows
        x4 = _x16(X[r0:r0 + 4])
        y1 = w4.w4_linear_i8_dynamic(x4, Wq, sc, of, 32, per_token=per_token)
        q4, s4 = w4.w4_quantize_activation_i8(x4, per_token)
        y2 = w4.w4_linear_i8(q4, s4, per_token, Wq, sc, of, 32)
        assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
        rq4, rs4 = oracle.ref_quantize_activation_i8(X[r0:r0 + 4], per_token=per_token)
        np.testing.assert_array_equal(q4.cpu().numpy(), rq4)


def _int8_problem(M, N, K, g, seed, per_token, with_bias):
    W = wl.gen_weight(N, K, seed=seed, outliers=True)
    X = wl.gen_activation(M, K, seed=seed + wl.ACT_SEED_OFFSET)
    rq, rs, ro = oracle.ref_quantize(bits(W), g)
    xq, xs = oracle.ref_quantize_activation_i8(bits(X), per_token=per_token)
    bias = bits(wl.gen_activation(1, N, seed=seed + 5))[0] if with_bias else None
    y_ref = oracle.ref_linear_i8(xq, xs, per_token, rq, rs, ro, g, bias=bias)
    to16 = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(DEV)
    dev = dict(Xq=torch.from_numpy(xq).to(DEV), xs=torch.from_numpy(xs).to(DEV), Wq=torch.from_numpy(rq).to(DEV),
               sc=to16(rs), of=to16(ro), bias=to16(bias) if bias is not None else None)
    return dev, y_ref


def gpu_linear_i8(d, per_token, g, workspace=None):
    M, N = d["Xq"].shape[0], d["Wq"].shape[0]
    Y = Guarded((M, N), torch.bfloat16)
    w4.w4_linear_i8(d["Xq"], d["xs"], per_token, d["Wq"], d["sc"], d["of"], g, bias=d["bias"], out=Y.t,
                    workspace=workspace)
    Y.check()
    return Y.t


I8_M = [1, 2, 3, 4, 5, 8, 16, 32, 33, 256]
I8_NK = [(520, 512), (1030, 1024), (200, 4160)]


@pytest.mark.parametrize("per_token", [False, True], ids=["tensor", "token"])
@pytest.mark.parametrize("g", [32, 64, 128])
@pytest.mark.parametrize("nk", I8_NK, ids=[f"{n}x{k}" for n, k in I8_NK])
def test_linear_i8_matches_oracle(nk, g, per_token):
    N, K = nk
    if K % g:
        pytest.skip("K % g != 0")
    for M in I8_M:
        d, y_ref = _int8_problem(M, N, K, g, seed=M + N + g, per_token=per_token, with_bias=(M % 2 == 1))
        y = gpu_linear_i8(d, per_token, g)
        ok, worst = oracle.within_linear_tolerance(f64(y), y_ref)
        assert ok, f"int8 linear M={M} N={N} K={K} g={g} per_token={per_token}: worst ratio {worst:.3f}"
    w4.w4_device_fault(DEV)


@pytest.mark.parametrize("M", [1, 4, 8, 64])
def test_linear_i8_odd_group_count_and_repeats(M):
    """K / g = 3 (odd): the stream kernels do not take it, the codes are widened for the
    tensor-core kernel; repeated calls on one workspace are bit-identical."""
    N, K, g = 136, 96, 32
    d, y_ref = _int8_problem(M, N, K, g, seed=3 + M, per_token=True, with_bias=True)
    ws = w4.Workspace(DEV, w4.w4_linear_i8_workspace_bytes(M, N, K, g))
    y = gpu_linear_i8(d, True, g, workspace=ws)
    ok, worst = oracle.within_linear_tolerance(f64(y), y_ref)
    assert ok, f"odd group count M={M}: worst ratio {worst:.3f}"
    again = gpu_linear_i8(d, True, g, workspace=ws)
    assert torch.equal(y.view(torch.int16), again.view(torch.int16))


@pytest.mark.parametrize("M", [1, 3, 16])
def test_linear_i8_full_size_sampled(M):
    """The down projection of the decode workloads (4096 x 14336, g = 32), rows sampled."""
    N, K, g = 4096, 14336, 32
    W = wl.gen_weight(N, K, seed=77, outliers=True)
    Wq, sc, of = w4.w4_quantize(W.to(DEV), g)
    X = wl.gen_activation(M, K, seed=78)
    Xq, xs = w4.w4_quantize_activation_i8(X.to(DEV), per_token=True)
    y = w4.w4_linear_i8(Xq, xs, True, Wq, sc, of, g)
    rows = np.random.default_rng(M).choice(N, 96, replace=False)
    rq = Wq.cpu().numpy()[rows]
    rs, ro = bits(sc)[rows], bits(of)[rows]
    y_ref = oracle.ref_linear_i8(Xq.cpu().numpy(), xs.cpu().numpy(), True, rq, rs, ro, g)
    ok, worst = oracle.within_linear_tolerance(f64(y)[:, rows], y_ref)
    assert ok, f"full-size int8 linear M={M}: worst ratio {worst:.3f}"


def test_direct_and_widened_paths_agree():
    """The same four tokens through the direct int8 stream kernel and (as rows of a
    five-token call) through the widened codes on the batch kernel."""
    N, K, g = 1024, 2048, 64
    d5, y_ref = _int8_problem(5, N, K, g, seed=9, per_token=True, with_bias=False)
    y5 = gpu_linear_i8(d5, True, g)
    d4 = dict(d5, Xq=d5["Xq"][:4].contiguous(), xs=d5["xs"][:4].contiguous())
    y4 = gpu_linear_i8(d4, True, g)
    ok, worst = oracle.within_linear_tolerance(f64(y4), y_ref[:4])
    assert ok, worst
    np.testing.assert_allclose(f64(y4), f64(y5)[:4], rtol=8e-3, atol=1e-2 * np.sqrt(np.mean(y_ref ** 2)))


def test_int8_calls_refuse_bad_arguments():
    lib = w4.load_library()
    d, _ = _int8_problem(1, 64, 256, 32, seed=1, per_token=False, with_bias=False)
    Y = torch.empty((1, 64), dtype=torch.bfloat16, device=DEV)
    s = w4._stream(Y)
    p = lambda t: w4._ptr(t)
    # workspace missing
    assert lib.w4_linear_i8(p(d["Xq"]), p(d["xs"]), 0, 1, 256, p(d["Wq"]), p(d["sc"]), p(d["of"]), 64, 32, None, p(Y),
                            None, 0, s) == 1
    ws = w4.Workspace(DEV, w4.w4_linear_i8_workspace_bytes(1, 64, 256, 32))
    # granularity must be 0 or 1
    assert lib.w4_linear_i8(p(d["Xq"]), p(d["xs"]), 2, 1, 256, p(d["Wq"]), p(d["sc"]), p(d["of"]), 64, 32, None, p(Y),
                            p(ws.buf), ws.nbytes, s) == 1
    # misaligned scale pointer
    xs_raw = torch.zeros(4, dtype=torch.uint8, device=DEV)
    bad = torch.ones(8, dtype=torch.uint8, device=DEV)
    import ctypes
    assert lib.w4_linear_i8(p(d["Xq"]), ctypes.c_void_p(bad.data_ptr() + 1), 0, 1, 256, p(d["Wq"]), p(d["sc"]),
                            p(d["of"]), 64, 32, None, p(Y), p(ws.buf), ws.nbytes, s) == 3
    # activation quantize: K not a multiple of 32, per tensor over rows without a workspace
    X = torch.zeros((2, 48), dtype=torch.bfloat16, device=DEV)
    Xq = torch.empty((2, 48), dtype=torch.int8, device=DEV)
    xs = torch.empty((1,), dtype=torch.float32, device=DEV)
    assert lib.w4_quantize_activation_i8(p(X), 2, 48, 0, p(Xq), p(xs), None, 0, s) == 1
    X = torch.zeros((2, 64), dtype=torch.bfloat16, device=DEV)
    Xq = torch.empty((2, 64), dtype=torch.int8, device=DEV)
    assert lib.w4_quantize_activation_i8(p(X), 2, 64, 0, p(Xq), p(xs), None, 0, s) == 1
    assert lib.w4_quantize_activation_i8(p(X), 2, 64, 1, p(Xq), None, None, 0, s) == 1
    del xs_raw
    assert lib.w4_device_fault(s) == 0  # nothing bad was launched


def test_one_workspace_serves_every_shape_in_sequence():
    """The widened codes of a large-M call are scratch past the 16 MiB of split-tile
    slots: later int8 and bf16 calls on the same workspace still find their slots at zero."""
    N, K, g = 1030, 1024, 32
    sizes = [w4.w4_linear_i8_workspace_bytes(M, N, K, g) for M in (256, 33, 5, 2, 1)]
    ws = w4.Workspace(DEV, max(sizes + [w4.w4_linear_workspace_bytes(5, N, K, g)]))
    for M, per_token in ((256, False), (33, True), (5, True), (2, False), (1, True), (5, False)):
        d, y_ref = _int8_problem(M, N, K, g, seed=100 + M, per_token=per_token, with_bias=False)
        y = gpu_linear_i8(d, per_token, g, workspace=ws)
        ok, worst = oracle.within_linear_tolerance(f64(y), y_ref)
        assert ok, f"M={M} after other shapes on one workspace: worst ratio {worst:.3f}"
    from tests.test_gpu_parity import _problem, gpu_linear
    (X, Wq, sc, of), y_ref = _problem(5, N, K, g, seed=5)
    assert_ok = oracle.within_linear_tolerance(f64(gpu_linear(X, Wq, sc, of, g, workspace=ws)), y_ref)
    assert assert_ok[0], f"bf16 linear on the shared workspace: worst ratio {assert_ok[1]:.3f}"
    assert int(ws.buf[: 16 << 20].count_nonzero()) == 0  # the slots came back to zero


DYN_SHAPES = [(1, 520, 512, 32), (2, 1030, 1024, 64), (3, 200, 4160, 32), (4, 4096, 4096, 128), (1, 8, 256, 32),
              (1, 14336, 4096, 32), (1, 4096, 14336, 32), (5, 1030, 1024, 32), (33, 520, 512, 64), (4, 136, 96, 32)]


@pytest.mark.parametrize("per_token", [False, True], ids=["tensor", "token"])
@pytest.mark.parametrize("shape", DYN_SHAPES, ids=[f"m{m}_{n}x{k}g{g}" for m, n, k, g in DYN_SHAPES])
def test_dynamic_call_is_the_two_calls_bit_for_bit(shape, per_token):
    """w4_linear_i8_dynamic (one kernel up to 4 tokens, the two steps in turn beyond, or for
    an odd group count) equals w4_quantize_activation_i8 + w4_linear_i8 bit for bit, and is
    within the tolerance of the oracle; the workspace's slots come back to zero."""
    M, N, K, g = shape
    W = wl.gen_weight(N, K, seed=N + K, outliers=True)
    Wq, sc, of = w4.w4_quantize(W.to(DEV), g)
    X = wl.gen_activation(M, K, seed=M + 3).to(DEV)
    bias = wl.gen_activation(1, N, seed=9)[0].to(DEV) if M % 2 else None
    ws = w4.Workspace(DEV, w4.w4_linear_i8_dynamic_workspace_bytes(M, N, K, g))
    Y = Guarded((M, N), torch.bfloat16)
    w4.w4_linear_i8_dynamic(X, Wq, sc, of, g, per_token=per_token, bias=bias, out=Y.t, workspace=ws)
    Y.check()
    Xq, xs = w4.w4_quantize_activation_i8(X, per_token)
    y2 = w4.w4_linear_i8(Xq, xs, per_token, Wq, sc, of, g, bias=bias)
    assert torch.equal(Y.t.view(torch.int16), y2.view(torch.int16)), "one call and two calls differ"
    y_ref = oracle.ref_linear_i8(Xq.cpu().numpy(), xs.cpu().numpy(), per_token, Wq.cpu().numpy(), bits(sc), bits(of),
                                 g, bias=bits(bias.cpu()) if bias is not None else None)
    ok, worst = oracle.within_linear_tolerance(f64(Y.t), y_ref)
    assert ok, f"dynamic int8 M={M} N={N} K={K} g={g}: worst ratio {worst:.3f}"
    assert int(ws.buf[: 16 << 20].count_nonzero()) == 0
    w4.w4_device_fault(DEV)
