"""The decode layout (include/w4.h): its reference round-trips the canonical
arrays, and a few bytes are checked against hand-worked offsets.  CPU only."""
import numpy as np
import pytest

from tests.decode_layout import SIGMA, _reorder, repack_ref, repacked_bytes, unit_bytes, unpack_ref


def _random(N, K, g, seed):
    rng = np.random.default_rng(seed)
    Wq = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    sc = rng.integers(1, 65535, size=(N, K // g), dtype=np.uint16)
    of = rng.integers(1, 65535, size=(N, K // g), dtype=np.uint16)
    return Wq, sc, of


@pytest.mark.parametrize("g", [32, 64, 128])
@pytest.mark.parametrize("N,K", [(16, 256), (37, 384), (8, 128), (33, 1152), (5, 4224)])
def test_round_trip(g, N, K):
    if K % g:
        pytest.skip("K not a multiple of g")
    Wq, sc, of = _random(N, K, g, seed=N * 1000 + K + g)
    packed = repack_ref(Wq, sc, of, N, K, g)
    assert packed.size == repacked_bytes(N, K, g)
    Wq2, sc2, of2, seen = unpack_ref(packed, N, K, g)
    assert np.array_equal(Wq, Wq2)
    assert np.array_equal(sc, sc2) and np.array_equal(of, of2)
    # every (row, group) appears g/32 times... once per lane group that reads it
    assert seen.min() >= 1


def test_unit_sizes():
    assert [unit_bytes(g) for g in (32, 64, 128)] == [2560, 2304, 2176]
    # 4096 x 4096 at g=32: 256 tiles x 16 units x 2560 B = exactly codes + qparams
    assert repacked_bytes(4096, 4096, 32) == 4096 * 4096 // 2 + 4 * 4096 * 4096 // 32


def test_hand_worked_offsets():
    """N=16, K=256, g=32: one unit.  Byte 512*1 + 16*5 is fragment j=1 of lane 5
    (r=1, q=1): row 1+8 = 9, k from 32 -> canonical bytes Wq[9, 16:32].  Qparam
    piece 6 serves lane 6 (r=1, q0=2): groups (64)/32 = 2 and (128+64)/32 = 6 of
    rows 1 and 9."""
    N, K, g = 16, 256, 32
    Wq = np.arange(N * K // 2, dtype=np.uint32).astype(np.uint8).reshape(N, K // 2)
    sc = (np.arange(N * 8, dtype=np.uint16) + 100).reshape(N, 8)
    of = (np.arange(N * 8, dtype=np.uint16) + 5000).reshape(N, 8)
    packed = repack_ref(Wq, sc, of, N, K, g)

    def codes(frag):  # 16 bytes -> the 32 codes in k order, undoing the nibble order by hand
        out = []
        for w in range(4):
            word = int.from_bytes(bytes(frag[4 * w: 4 * w + 4]), "little")
            nib = [(word >> (4 * i)) & 0xF for i in range(8)]
            out += [nib[0], nib[4], nib[1], nib[5], nib[2], nib[6], nib[3], nib[7]]
        return out

    def canon(row, b0):  # the 32 canonical codes of 16 bytes from byte b0 of a row
        return [int(Wq[row, b0 + i // 2]) >> (4 * (i % 2)) & 0xF for i in range(32)]

    assert codes(packed[512 + 80: 512 + 96]) == canon(9, 16)
    assert codes(packed[0:16]) == canon(0, 0)                          # j=0, lane 0: row 0, k 0..31
    assert codes(packed[1024 + 16 * 31: 1024 + 16 * 32]) == canon(7, 112)  # j=2, lane 31: row 7, k 224..255
    # one word by hand: canonical bytes 0x10 0x32 0x54 0x76 (codes 0..7 in k order)
    # -> nibbles k0 k2 k4 k6 k1 k3 k5 k7 = 0x75316420
    assert SIGMA == (0, 2, 4, 6, 1, 3, 5, 7)
    word = _reorder(np.array([0x10, 0x32, 0x54, 0x76] * 4, dtype=np.uint8))
    assert int(word.view("<u4")[0]) == 0x75316420
    q = packed[2048 + 16 * 6: 2048 + 16 * 7].view("<u2")
    assert list(q) == [sc[1, 2], of[1, 2], sc[9, 2], of[9, 2], sc[1, 6], of[1, 6], sc[9, 6], of[9, 6]]


def test_ragged_edges_are_zero():
    N, K, g = 3, 160, 32  # one tile with 13 missing rows, one unit with 96 missing k
    Wq, sc, of = _random(N, K, g, seed=7)
    packed = repack_ref(Wq, sc, of, N, K, g)
    # lane 16 is row 4 (>= N): its fragments are zero
    assert not packed[16 * 16: 16 * 17].any()
    # j = 2 covers k from 128 + 32q: only q = 0 (k 128..159) lies inside K = 160
    for lane in range(32):
        frag = packed[1024 + 16 * lane: 1024 + 16 * lane + 16]
        r, q = lane // 4, lane % 4
        if q == 0 and r < N:
            assert frag.any() or not Wq[r, 64:80].any()
        else:
            assert not frag.any()
    # j = 1 and 3 are rows 8.. (all >= N): zero
    assert not packed[512:1024].any() and not packed[1536:2048].any()
