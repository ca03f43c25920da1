"""Host-side check of the stream-K partition the decode kernels share (no GPU).

Worker w (a warp, or a block in the batched kernel) owns the contiguous units
[U w / W, U (w + 1) / W).  A row tile split between workers is finished by the
worker holding its first unit, which must find every later sharer; it looks
them up with split_warp_of(u) = ((u + 1) W - 1) / U.  If that ever named a
worker whose range does not hold u, the owner would wait for a share that never
arrives (a bounded wait that ends in W4_ERR_TIMEOUT).  The formulas are read
from the CUDA sources so that this test follows them.
"""
import os
import re

import numpy as np

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "bit_weight_quantization_02_b300", "csrc")


def _src(name):
    with open(os.path.join(CSRC, name)) as f:
        return f.read()


def test_the_sources_use_the_checked_formulas():
    dev = _src("w4_device.cuh")
    assert re.search(r"split_warp_of\(long long u, long long units, int workers\)\s*\{\s*"
                     r"return \(int\)\(\(\(u \+ 1\) \* workers - 1\) / units\);", dev)
    for name, who, count in (("w4_stream.cu", "worker", "workers"), ("w4_decode.cu", "worker", "workers"),
                             ("w4_batch.cu", "cta", "ctas")):
        s = _src(name)
        assert f"p.units * {who} / p.{count}" in s, name
        assert f"p.units * ({who} + 1) / p.{count}" in s, name


def test_owner_lookup_names_the_range_holding_each_unit():
    """Every unit u of every (U, W) with W <= U: floor(((u+1) W - 1) / U) = w with
    floor(U w / W) <= u < floor(U (w+1) / W), and the ranges tile [0, U) without gaps."""
    for U in list(range(1, 120)) + [1024, 4096, 7168, 14336]:
        Ws = sorted({1, 2, 3, 7, U // 3 or 1, U // 2 or 1, U - 1 or 1, U} | set(range(1, min(U, 40) + 1)))
        u = np.arange(U, dtype=np.int64)
        for W in Ws:
            if W > U:
                continue
            w = ((u + 1) * W - 1) // U
            lo, hi = U * w // W, U * (w + 1) // W
            assert np.all((lo <= u) & (u < hi)), (U, W)
            starts = U * np.arange(W + 1, dtype=np.int64) // W
            assert starts[0] == 0 and starts[-1] == U and np.all(np.diff(starts) >= 1), (U, W)


def test_split_tiles_have_one_owner_and_contiguous_sharers():
    """For a row of nkc units per tile, the tile's first unit's worker owns it and the workers of
    its later units are consecutive after the owner (the owner reads their slots in order)."""
    for nkc in (1, 2, 7, 16, 56):
        for tiles in (1, 3, 64, 448):
            U = tiles * nkc
            for W in {1, 5, 148 * 4, 2368, 3552} - {0}:
                if W > U:
                    W = U
                u = np.arange(U, dtype=np.int64)
                w = ((u + 1) * W - 1) // U
                per_tile = w.reshape(tiles, nkc)
                assert np.all(np.diff(per_tile, axis=1) >= 0)
                assert np.all(np.diff(per_tile, axis=1) <= 1)  # no worker skipped inside a tile
