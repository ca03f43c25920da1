"""GPU parity: libw4's kernels (through the C ABI) against the CPU oracle.

* w4_quantize / w4_dequantize: bit-exact, including ragged shapes and
  adversarial groups;
* w4_linear (skinny decode kernel and tcgen05 GEMM): within
  |y - y_ref| <= 4e-3 |y_ref| + 1e-2 rms(y_ref), y_ref the oracle's fp64
  product with the dequantized weights; rms over the whole output of the call,
  or over the sampled outputs where only a sample is computed;
* every output buffer sits between guard bytes that must survive the call
  (out-of-bounds writes would show there);
* the full-size workloads, in the launch configuration the benchmark times,
  on sampled rows and columns that the oracle computes one by one.
"""
import numpy as np
import pytest
import torch

import oracle
import bit_weight_quantization_02_b300 as w4
from bit_weight_quantization_02_b300 import workloads as wl
from tests.test_oracle_pins import adversarial_matrix
from tests.decode_layout import repack_ref

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
CANARY = 0x5A


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def f64(t: torch.Tensor) -> np.ndarray:
    return oracle.bf16_bits_to_f64(bits(t))


class Guarded:
    """A device tensor with 256 canary bytes on both sides."""
    PAD = 256

    def __init__(self, shape, dtype):
        n = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
        self.raw = torch.full((n + 2 * self.PAD,), CANARY, dtype=torch.uint8, device=DEV)
        self.n = n
        self.t = self.raw[self.PAD:self.PAD + n].view(dtype).view(shape)

    def check(self):
        torch.cuda.synchronize()
        head = self.raw[:self.PAD]
        tail = self.raw[self.PAD + self.n:]
        assert bool((head == CANARY).all()) and bool((tail == CANARY).all()), "write outside the output buffer"


def gpu_quantize(W, g):
    N, K = W.shape
    out = (Guarded((N, K // 2), torch.uint8), Guarded((N, K // g), torch.bfloat16),
           Guarded((N, K // g), torch.bfloat16))
    w4.w4_quantize(W, g, out=tuple(o.t for o in out))
    for o in out:
        o.check()
    return tuple(o.t for o in out)


def gpu_linear(X, Wq, sc, of, g, kernel=w4.KERNEL_AUTO, workspace=None):
    M, N = X.shape[0], Wq.shape[0]
    Y = Guarded((M, N), torch.bfloat16)
    w4.w4_linear_ex(X, Wq, sc, of, g, kernel, out=Y.t, workspace=workspace)
    Y.check()
    return Y.t


def assert_linear_ok(y_gpu: torch.Tensor, y_ref: np.ndarray, what: str):
    ok, worst = oracle.within_linear_tolerance(f64(y_gpu), y_ref)
    assert ok, f"{what}: outside |y-y_ref| <= 4e-3|y_ref| + 1e-2 rms, worst ratio {worst:.3f}"


# ----------------------------------------------------------------- quantize

QUANT_SHAPES = [(512, 512), (300, 4224), (7, 128), (64, 14336), (1, 4096)]


@pytest.mark.parametrize("g", [32, 64, 128])
@pytest.mark.parametrize("shape", QUANT_SHAPES, ids=[f"{n}x{k}" for n, k in QUANT_SHAPES])
def test_quantize_bit_exact(g, shape):
    N, K = shape
    W = wl.gen_weight(N, K, seed=100 + N + g, outliers=True)
    Wq, sc, of = gpu_quantize(W.to(DEV), g)
    rq, rs, ro = oracle.ref_quantize(bits(W), g)
    np.testing.assert_array_equal(Wq.cpu().numpy(), rq)
    np.testing.assert_array_equal(bits(sc), rs)
    np.testing.assert_array_equal(bits(of), ro)


@pytest.mark.parametrize("g", [32, 64, 128])
def test_quantize_adversarial_groups_bit_exact(g):
    Wb = adversarial_matrix(g)
    W = torch.from_numpy(Wb.view(np.int16)).view(torch.bfloat16).to(DEV)
    Wq, sc, of = gpu_quantize(W, g)
    rq, rs, ro = oracle.ref_quantize(Wb, g)
    np.testing.assert_array_equal(Wq.cpu().numpy(), rq)
    np.testing.assert_array_equal(bits(sc), rs)
    np.testing.assert_array_equal(bits(of), ro)


def test_quantize_golden_cases():
    from tests.test_oracle_pins import GOLDEN_CASES, unpack_codes
    for case in GOLDEN_CASES:
        g = case["g"]
        W = torch.from_numpy(case["values"].reshape(1, g).view(np.int16)).view(torch.bfloat16).to(DEV)
        Wq, sc, of = gpu_quantize(W, g)
        assert bits(sc)[0, 0] == case["scale"] and bits(of)[0, 0] == case["offset"], case["name"]
        np.testing.assert_array_equal(unpack_codes(Wq.cpu().numpy())[0], case["codes"])


# --------------------------------------------------------------- dequantize

@pytest.mark.parametrize("g", [32, 64, 128])
@pytest.mark.parametrize("shape", [(300, 4224), (64, 128), (3, 14336)])
def test_dequantize_bit_exact_on_arbitrary_codes(g, shape):
    """Random code bytes and random finite qparams, independent of w4_quantize."""
    N, K = shape
    rng = np.random.default_rng(N * K + g)
    rq = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    rs = bits(torch.from_numpy(np.abs(rng.normal(0, 0.01, (N, K // g))).astype(np.float32) + 1e-6).to(torch.bfloat16))
    ro = bits(torch.from_numpy(rng.normal(0, 0.05, (N, K // g)).astype(np.float32)).to(torch.bfloat16))
    Wq = torch.from_numpy(rq).to(DEV)
    sc = torch.from_numpy(rs.view(np.int16)).view(torch.bfloat16).to(DEV)
    of = torch.from_numpy(ro.view(np.int16)).view(torch.bfloat16).to(DEV)
    out = Guarded((N, K), torch.bfloat16)
    w4.w4_dequantize(Wq, sc, of, g, out=out.t)
    out.check()
    np.testing.assert_array_equal(bits(out.t), oracle.ref_dequantize(rq, rs, ro, g))


# ------------------------------------------------------------------- linear

def _problem(M, N, K, g, seed, outliers=True):
    W = wl.gen_weight(N, K, seed=seed, outliers=outliers)
    X = wl.gen_activation(M, K, seed=seed + wl.ACT_SEED_OFFSET)
    rq, rs, ro = oracle.ref_quantize(bits(W), g)
    dev = (X.to(DEV), torch.from_numpy(rq).to(DEV),
           torch.from_numpy(rs.view(np.int16)).view(torch.bfloat16).to(DEV),
           torch.from_numpy(ro.view(np.int16)).view(torch.bfloat16).to(DEV))
    y_ref = oracle.ref_linear(bits(X), rq, rs, ro, g)
    return dev, y_ref


SKINNY_M = [1, 2, 3, 5, 8, 9, 16, 17, 24, 31, 32]
SKINNY_NK = [(200, 4160), (520, 512), (64, 96), (1030, 1024)]


@pytest.mark.parametrize("g", [32, 64, 128])
@pytest.mark.parametrize("nk", SKINNY_NK, ids=[f"{n}x{k}" for n, k in SKINNY_NK])
def test_linear_skinny_cluster(g, nk):
    N, K = nk
    if K % g:
        pytest.skip("K not a multiple of g")
    for M in SKINNY_M:
        (X, Wq, sc, of), y_ref = _problem(M, N, K, g, seed=7 * M + N + g)
        assert_linear_ok(gpu_linear(X, Wq, sc, of, g, w4.KERNEL_SKINNY_CLUSTER), y_ref,
                         f"skinny cluster M={M} N={N} K={K} g={g}")


STREAM_NK = [(200, 4160), (520, 512), (64, 256), (1030, 1024), (4096, 1536), (48, 14336)]


@pytest.mark.parametrize("g", [32, 64, 128])
@pytest.mark.parametrize("nk", STREAM_NK, ids=[f"{n}x{k}" for n, k in STREAM_NK])
def test_linear_stream(g, nk):
    N, K = nk
    if K % g or (K // g) % 2:
        pytest.skip("the stream kernel needs an even K/g")
    ws = w4.Workspace(DEV).reserve_for(32, N, K, g)
    for M in (1, 2, 3, 5, 8, 9, 16, 17, 31, 32):
        (X, Wq, sc, of), y_ref = _problem(M, N, K, g, seed=13 * M + N + g)
        assert_linear_ok(gpu_linear(X, Wq, sc, of, g, w4.KERNEL_STREAM, workspace=ws), y_ref,
                         f"stream M={M} N={N} K={K} g={g}")
        torch.cuda.synchronize()
        assert int(ws.buf.count_nonzero()) == 0, "the stream kernel must leave its workspace zeroed"


# one token on problems large enough for 32-row units (two row tiles per unit), ragged row tails;
# the last three give between half and all of the resident warps a 32-row unit (1312, 1615 and
# 2048 units against about 2400 warps), with ragged tails in the first two
ONE_TOKEN_NK = [(4104, 6144), (4120, 6144), (4096, 6080), (8192, 4096), (2600, 4096), (3016, 4160), (4096, 4096)]


@pytest.mark.parametrize("g", [32, 64, 128])
@pytest.mark.parametrize("nk", ONE_TOKEN_NK, ids=[f"{n}x{k}" for n, k in ONE_TOKEN_NK])
def test_linear_stream_one_token_large(g, nk):
    N, K = nk
    if K % g or (K // g) % 2:
        pytest.skip("the stream kernel needs an even K/g")
    ws = w4.Workspace(DEV).reserve_for(1, N, K, g)
    (X, Wq, sc, of), y_ref = _problem(1, N, K, g, seed=N + K + g)
    y = gpu_linear(X, Wq, sc, of, g, w4.KERNEL_STREAM, workspace=ws)
    assert_linear_ok(y, y_ref, f"stream M=1 N={N} K={K} g={g}")
    for _ in range(3):  # deterministic
        assert torch.equal(y.view(torch.int16), gpu_linear(X, Wq, sc, of, g, w4.KERNEL_STREAM, workspace=ws).view(torch.int16))
    torch.cuda.synchronize()
    assert int(ws.buf.count_nonzero()) == 0, "the stream kernel must leave its workspace zeroed"
    w4.w4_device_fault(DEV)


REPACK_NK = [(200, 4160), (520, 512), (64, 96), (1030, 1024), (48, 14336), (16, 256), (33, 1152)]


def _repacked(Wq, sc, of, g):
    """w4_repack into a canary-guarded buffer."""
    N, K = Wq.shape[0], 2 * Wq.shape[1]
    out = Guarded((w4.w4_repacked_bytes(N, K, g),), torch.uint8)
    rp = w4.w4_repack(Wq, sc, of, g, out=out.t)
    out.check()
    return rp


@pytest.mark.parametrize("g", [32, 64, 128])
@pytest.mark.parametrize("nk", REPACK_NK, ids=[f"{n}x{k}" for n, k in REPACK_NK])
def test_repack_bit_exact(g, nk):
    """w4_repack equals the layout reference byte for byte (ragged tiles and units)."""
    N, K = nk
    if K % g:
        pytest.skip("K not a multiple of g")
    W = wl.gen_weight(N, K, seed=N + K + g)
    rq, rs, ro = oracle.ref_quantize(bits(W), g)
    Wq = torch.from_numpy(rq).to(DEV)
    sc = torch.from_numpy(rs.view(np.int16)).view(torch.bfloat16).to(DEV)
    of = torch.from_numpy(ro.view(np.int16)).view(torch.bfloat16).to(DEV)
    rp = _repacked(Wq, sc, of, g)
    assert np.array_equal(rp.buf.cpu().numpy(), repack_ref(rq, rs, ro, N, K, g))


@pytest.mark.parametrize("g", [32, 64, 128])
@pytest.mark.parametrize("nk", REPACK_NK, ids=[f"{n}x{k}" for n, k in REPACK_NK])
def test_linear_repacked(g, nk):
    """The decode-layout kernel (one to four groups of 8 tokens), against the oracle."""
    N, K = nk
    if K % g:
        pytest.skip("K not a multiple of g")
    for M in (1, 2, 3, 5, 8, 9, 16, 17, 31, 32):
        (X, Wq, sc, of), y_ref = _problem(M, N, K, g, seed=19 * M + N + g)
        rp = _repacked(Wq, sc, of, g)
        Y = Guarded((M, N), torch.bfloat16)
        w4.w4_linear_repacked(X, rp, out=Y.t)
        Y.check()
        assert_linear_ok(Y.t, y_ref, f"repacked M={M} N={N} K={K} g={g}")
    w4.w4_device_fault(DEV)
    ws = w4._workspace_for(X, 32, N, K, g, None)  # the stream's default workspace, shared with other calls
    torch.cuda.synchronize()
    # its slot region (the first 16 MiB) comes back to zero; past it, the tensor-core GEMM keeps
    # partial sums that it always writes before reading
    assert int(ws.buf[: 16 << 20].count_nonzero()) == 0, "the decode-layout kernel must leave its slots zeroed"


GEMM_M = [1, 33, 127, 129, 300]
GEMM_NK = [(200, 4160), (520, 512), (256, 64), (1000, 96), (136, 3072), (384, 4096)]


@pytest.mark.parametrize("g", [32, 64, 128])
@pytest.mark.parametrize("nk", GEMM_NK, ids=[f"{n}x{k}" for n, k in GEMM_NK])
def test_linear_gemm(g, nk):
    N, K = nk
    if K % g:
        pytest.skip("K not a multiple of g")
    for M in GEMM_M:
        (X, Wq, sc, of), y_ref = _problem(M, N, K, g, seed=11 * M + N + g)
        assert_linear_ok(gpu_linear(X, Wq, sc, of, g, w4.KERNEL_GEMM), y_ref, f"gemm M={M} N={N} K={K} g={g}")
    w4.w4_device_fault(DEV)


def test_linear_auto_dispatch_and_both_kernels_agree():
    (X, Wq, sc, of), y_ref = _problem(32, 768, 2048, 32, seed=5)
    ys = gpu_linear(X, Wq, sc, of, 32, w4.KERNEL_SKINNY_CLUSTER)
    yg = gpu_linear(X, Wq, sc, of, 32, w4.KERNEL_GEMM)
    yt = gpu_linear(X, Wq, sc, of, 32, w4.KERNEL_STREAM)
    ya = gpu_linear(X, Wq, sc, of, 32)  # M <= 32 with the default workspace: the stream kernel
    y0 = gpu_linear(X, Wq, sc, of, 32, w4.KERNEL_AUTO, workspace=w4.Workspace(DEV))  # no workspace: cluster
    assert torch.equal(ys.view(torch.int16), y0.view(torch.int16))
    for y, what in ((ys, "skinny"), (yg, "gemm"), (yt, "stream"), (ya, "auto")):
        assert_linear_ok(y, y_ref, what)
    # the kernels round differently but agree to bf16 precision
    for y in (ys, yt, ya):
        assert float((y.float() - yg.float()).abs().max()) <= 2e-2 * float(yg.float().abs().max())


def test_workspace_shared_by_calls_of_different_shapes():
    """One workspace, stream-kernel calls of different shapes in turn: each
    leaves it zeroed for the next."""
    a = _problem(8, 1030, 1024, 32, seed=31)
    b = _problem(1, 14336, 1024, 32, seed=32)
    c = _problem(3, 200, 4160, 32, seed=33)
    ws = w4.Workspace(DEV).reserve(max(w4.w4_linear_workspace_bytes(8, 1030, 1024, 32),
                                       w4.w4_linear_workspace_bytes(1, 14336, 1024, 32),
                                       w4.w4_linear_workspace_bytes(3, 200, 4160, 32)))
    for (dev, y_ref) in (a, b, c, a, c, b):
        assert_linear_ok(gpu_linear(*dev, 32, w4.KERNEL_STREAM, workspace=ws), y_ref, "shared workspace")
    torch.cuda.synchronize()
    assert int(ws.buf.count_nonzero()) == 0


def test_auto_uses_the_stream_kernel_only_with_a_workspace():
    (X, Wq, sc, of), y_ref = _problem(2, 2048, 2048, 64, seed=34)
    no_ws = w4.Workspace(DEV)  # zero bytes: the cluster kernel runs
    y0 = gpu_linear(X, Wq, sc, of, 64, w4.KERNEL_AUTO, workspace=no_ws)
    y1 = gpu_linear(X, Wq, sc, of, 64, w4.KERNEL_SKINNY_CLUSTER)
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))
    assert_linear_ok(gpu_linear(X, Wq, sc, of, 64), y_ref, "auto with workspace")


def test_linear_is_deterministic():
    (X, Wq, sc, of), y_ref = _problem(3, 2048, 4096, 64, seed=9)
    first = gpu_linear(X, Wq, sc, of, 64, w4.KERNEL_SKINNY_CLUSTER)
    for _ in range(5):
        again = gpu_linear(X, Wq, sc, of, 64, w4.KERNEL_SKINNY_CLUSTER)
        assert torch.equal(first.view(torch.int16), again.view(torch.int16))
    assert_linear_ok(first, y_ref, "repeat")


@pytest.mark.parametrize("M", [1, 3, 8, 17, 32])
def test_stream_kernels_are_deterministic(M):
    """Row tiles split between warps are summed in a fixed order: repeated calls
    agree bit for bit (canonical and decode layouts; k/v-like shape, where every
    tile is split between 16 warps, and a ragged one)."""
    for (N, K, g) in [(1024, 4096, 32), (520, 4608, 64)]:
        (X, Wq, sc, of), y_ref = _problem(M, N, K, g, seed=70 + M + N)
        ws = w4.Workspace(DEV).reserve_for(M, N, K, g)
        first = gpu_linear(X, Wq, sc, of, g, w4.KERNEL_STREAM, workspace=ws)
        rp = w4.w4_repack(Wq, sc, of, g)
        rfirst = w4.w4_linear_repacked(X, rp, workspace=ws)
        for _ in range(4):
            again = gpu_linear(X, Wq, sc, of, g, w4.KERNEL_STREAM, workspace=ws)
            assert torch.equal(first.view(torch.int16), again.view(torch.int16))
            ragain = w4.w4_linear_repacked(X, rp, workspace=ws)
            assert torch.equal(rfirst.view(torch.int16), ragain.view(torch.int16))
        assert_linear_ok(first, y_ref, f"stream M={M} N={N}")
        assert_linear_ok(rfirst, y_ref, f"repacked M={M} N={N}")
        torch.cuda.synchronize()
        assert int(ws.buf.count_nonzero()) == 0
    w4.w4_device_fault(DEV)


def test_consecutive_linears_overlap_safely():
    """Back-to-back skinny launches on one stream may overlap (programmatic
    dependent launch): a chain where each call reads the previous call's output
    must still see it complete."""
    K = 1024
    Ws = [wl.gen_weight(K, K, seed=40 + i) for i in range(6)]
    packed = [oracle.ref_quantize(bits(W), 32) for W in Ws]
    dev = [(torch.from_numpy(q).to(DEV), torch.from_numpy(s.view(np.int16)).view(torch.bfloat16).to(DEV),
            torch.from_numpy(o.view(np.int16)).view(torch.bfloat16).to(DEV)) for q, s, o in packed]
    x = wl.gen_activation(1, K, seed=47)
    y = x.to(DEV)
    for d in dev:
        y = w4.w4_linear(y, *d, 32)
    torch.cuda.synchronize()
    # the same chain, one linear at a time against the oracle's fp64 product of the previous GPU output
    y = x.to(DEV)
    for (q, s, o), d in zip(packed, dev):
        y_ref = oracle.ref_linear(bits(y), q, s, o, 32)
        y = w4.w4_linear(y, *d, 32)
        torch.cuda.synchronize()
        assert_linear_ok(y, y_ref, "chain")


def test_linear_edge_shapes():
    for M, N, K, g in [(1, 1, 32, 32), (1, 7, 64, 64), (2, 65, 128, 128), (32, 257, 32, 32), (129, 9, 128, 32),
                       (1, 4096, 128, 128), (5, 3, 14336, 32)]:
        (X, Wq, sc, of), y_ref = _problem(M, N, K, g, seed=M + N + K)
        assert_linear_ok(gpu_linear(X, Wq, sc, of, g), y_ref, f"edge M={M} N={N} K={K} g={g}")
        assert_linear_ok(gpu_linear(X, Wq, sc, of, g, w4.KERNEL_GEMM), y_ref, f"edge gemm M={M} N={N} K={K}")


def test_empty_problems():
    X = torch.zeros((0, 64), dtype=torch.bfloat16, device=DEV)
    Wq = torch.zeros((8, 32), dtype=torch.uint8, device=DEV)
    sc = torch.zeros((8, 2), dtype=torch.bfloat16, device=DEV)
    Y = w4.w4_linear(X, Wq, sc, sc, 32)
    assert Y.shape == (0, 8)
    W = torch.zeros((0, 64), dtype=torch.bfloat16, device=DEV)
    q, s, o = w4.w4_quantize(W, 32)
    assert q.shape == (0, 32)


def test_cuda_graph_capture_matches_eager():
    probs = [_problem(1, N, K, 32, seed=20 + i) for i, (N, K) in enumerate([(1024, 4096), (4096, 1024), (768, 2048)])]
    outs = [torch.empty((1, p[0][1].shape[0]), dtype=torch.bfloat16, device=DEV) for p in probs]
    ws = w4.Workspace(DEV).reserve(max(w4.w4_linear_workspace_bytes(1, p[0][1].shape[0], p[0][0].shape[1], 32)
                                       for p in probs))
    eager = [gpu_linear(*p[0], 32, workspace=ws).clone() for p in probs]
    s = torch.cuda.Stream(DEV)
    s.wait_stream(torch.cuda.current_stream(DEV))
    with torch.cuda.stream(s):
        for (dev, _), out in zip(probs, outs):  # warm up on the capture stream
            w4.w4_linear(*dev, 32, out=out, workspace=ws)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            for (dev, _), out in zip(probs, outs):
                w4.w4_linear(*dev, 32, out=out, workspace=ws)
    torch.cuda.current_stream(DEV).wait_stream(s)
    for out in outs:
        out.zero_()
    graph.replay()
    torch.cuda.synchronize()
    for (dev, y_ref), o in zip(probs, outs):
        assert_linear_ok(o, y_ref, "graph replay")


def test_no_device_fault_pending():
    w4.w4_device_fault(DEV)


# ------------------------------------------ full-size workloads, sampled

def _sampled_quantize_check(W_dev, g, rows):
    Wq, sc, of = w4.w4_quantize(W_dev, g)
    Wr = bits(W_dev[rows])
    rq, rs, ro = oracle.ref_quantize(Wr, g)
    np.testing.assert_array_equal(Wq[rows].cpu().numpy(), rq)
    np.testing.assert_array_equal(bits(sc[rows]), rs)
    np.testing.assert_array_equal(bits(of[rows]), ro)
    return Wq, sc, of, (rq, rs, ro)


def _rows(N, n=48, seed=0):
    rng = np.random.default_rng(seed)
    r = np.unique(np.concatenate([rng.choice(N, size=min(n, N), replace=False), [0, N - 1]]))
    return torch.from_numpy(r).to(DEV)


@pytest.mark.parametrize("case", wl.config2(), ids=[c.name for c in wl.config2()])
def test_full_size_decode_config2(case):
    """Llama-3-8B decode linears, M=1, g=32, 0.1 % x10 outliers."""
    W = wl.gen_weight(case.N, case.K, case.w_seed, outliers=True, device=DEV)
    rows = _rows(case.N, seed=case.w_seed)
    Wq, sc, of, (rq, rs, ro) = _sampled_quantize_check(W, case.group_size, rows)
    X = wl.gen_activation(case.M, case.K, case.x_seed, device=DEV)
    Y = gpu_linear(X, Wq, sc, of, case.group_size)
    y_ref = oracle.ref_linear(bits(X), rq, rs, ro, case.group_size)
    assert_linear_ok(Y[:, rows], y_ref, f"config2 {case.name}")
    # the same weights in the decode layout (the benchmark's headline path)
    Yr = w4.w4_linear_repacked(X, w4.w4_repack(Wq, sc, of, case.group_size))
    assert_linear_ok(Yr[:, rows], y_ref, f"config2 {case.name} (decode layout)")


def test_full_size_batched_decode_config3():
    for case in wl.config3():
        W = wl.gen_weight(case.N, case.K, case.w_seed, device=DEV)
        rows = _rows(case.N, n=24, seed=case.w_seed + case.M)
        Wq, sc, of, (rq, rs, ro) = _sampled_quantize_check(W, case.group_size, rows)
        X = wl.gen_activation(case.M, case.K, case.x_seed + case.M, device=DEV)
        Y = gpu_linear(X, Wq, sc, of, case.group_size)
        y_ref = oracle.ref_linear(bits(X), rq, rs, ro, case.group_size)
        assert_linear_ok(Y[:, rows], y_ref, f"config3 {case.name}")


def test_full_size_prefill_config4():
    for case in wl.config4():
        W = wl.gen_weight(case.N, case.K, case.w_seed, device=DEV)
        rows = _rows(case.N, n=24, seed=case.w_seed)
        Wq, sc, of, (rq, rs, ro) = _sampled_quantize_check(W, case.group_size, rows)
        X = wl.gen_activation(case.M, case.K, case.x_seed + case.M, device=DEV)
        Y = gpu_linear(X, Wq, sc, of, case.group_size)
        toks = _rows(case.M, n=40, seed=case.M)
        y_ref = oracle.ref_linear(bits(X[toks]), rq, rs, ro, case.group_size)
        assert_linear_ok(Y[toks][:, rows], y_ref, f"config4 {case.name}")
        del W, Wq, sc, of, X, Y
    w4.w4_device_fault(DEV)


@pytest.mark.parametrize("layer", [0, 31])
def test_full_size_stack_config5_layers(layer):
    """Two blocks of the 32-layer g=128 stack: every linear, M=1 and M=16."""
    for i, (name, N, K) in enumerate(wl.LLAMA3_8B_LINEARS):
        seed = wl.weight_seed(5, layer, i)
        W = wl.gen_weight(N, K, seed, device=DEV)
        rows = _rows(N, n=16, seed=seed)
        Wq, sc, of, (rq, rs, ro) = _sampled_quantize_check(W, 128, rows)
        del W
        for M in (1, 16):
            X = wl.gen_activation(M, K, seed + wl.ACT_SEED_OFFSET + M, device=DEV)
            Y = gpu_linear(X, Wq, sc, of, 128)
            y_ref = oracle.ref_linear(bits(X), rq, rs, ro, 128)
            assert_linear_ok(Y[:, rows], y_ref, f"config5 L{layer}.{name} M={M}")
