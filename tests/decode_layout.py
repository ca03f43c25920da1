"""Reference of libw4's decode layout, written from the byte-exact description in
include/w4.h (a rearrangement of the canonical arrays, no arithmetic of the
method): used by the tests to check w4_repack bit for bit and, through its
inverse, that the layout holds exactly the canonical numbers.

Canonical arrays: Wq uint8 [N, K/2], scales / offsets uint16 (bf16 bits) [N, K/g].
"""
import numpy as np


# nibble i of a decode-layout word holds canonical nibble (k offset) SIGMA[i]
SIGMA = (0, 2, 4, 6, 1, 3, 5, 7)


def _reorder(frag: np.ndarray) -> np.ndarray:
    """16 canonical code bytes -> the decode layout's nibble order (per 32-bit word)."""
    words = frag.view("<u4").astype(np.uint64)
    out = np.zeros_like(words)
    for i, src in enumerate(SIGMA):
        out |= ((words >> (4 * src)) & 0xF) << (4 * i)
    return out.astype("<u4").view(np.uint8)


def _restore(frag: np.ndarray) -> np.ndarray:
    """The inverse of _reorder."""
    words = frag.view("<u4").astype(np.uint64)
    out = np.zeros_like(words)
    for i, src in enumerate(SIGMA):
        out |= ((words >> (4 * i)) & 0xF) << (4 * src)
    return out.astype("<u4").view(np.uint8)


def unit_bytes(g: int) -> int:
    return 2048 + 16 * 32 * 32 // g


def repacked_bytes(N: int, K: int, g: int) -> int:
    return -(-N // 16) * -(-K // 256) * unit_bytes(g)


def repack_ref(Wq: np.ndarray, scales: np.ndarray, offsets: np.ndarray, N: int, K: int, g: int) -> np.ndarray:
    """Canonical -> decode layout, one unit at a time with plain loops."""
    tiles, nkc, ng, U = -(-N // 16), -(-K // 256), K // g, unit_bytes(g)
    out = np.zeros(tiles * nkc * U, dtype=np.uint8)
    lanes_per_piece = g // 32
    for t in range(tiles):
        for c in range(nkc):
            base = (t * nkc + c) * U
            for j in range(4):
                for lane in range(32):
                    r, q = lane // 4, lane % 4
                    row = 16 * t + r + 8 * (j % 2)
                    k0 = 256 * c + 128 * (j // 2) + 32 * q
                    if row < N and k0 < K:
                        out[base + 512 * j + 16 * lane: base + 512 * j + 16 * lane + 16] = \
                            _reorder(np.ascontiguousarray(Wq[row, k0 // 2: k0 // 2 + 16]))
            for p in range(1024 // g):
                l0 = p * lanes_per_piece
                r, q0 = l0 // 4, l0 % 4
                vals = []
                for h in range(2):
                    grp = (256 * c + 128 * h + 32 * q0) // g
                    for row in (16 * t + r, 16 * t + r + 8):
                        ok = row < N and grp < ng
                        vals += [int(scales[row, grp]) if ok else 0, int(offsets[row, grp]) if ok else 0]
                out[base + 2048 + 16 * p: base + 2048 + 16 * p + 16] = np.array(vals, dtype="<u2").view(np.uint8)
    return out


def unpack_ref(packed: np.ndarray, N: int, K: int, g: int):
    """Decode layout -> canonical arrays (the inverse of repack_ref)."""
    tiles, nkc, ng, U = -(-N // 16), -(-K // 256), K // g, unit_bytes(g)
    Wq = np.zeros((N, K // 2), dtype=np.uint8)
    sc = np.zeros((N, ng), dtype=np.uint16)
    of = np.zeros((N, ng), dtype=np.uint16)
    seen = np.zeros((N, ng), dtype=np.int32)
    for t in range(tiles):
        for c in range(nkc):
            base = (t * nkc + c) * U
            for j in range(4):
                for lane in range(32):
                    r, q = lane // 4, lane % 4
                    row = 16 * t + r + 8 * (j % 2)
                    k0 = 256 * c + 128 * (j // 2) + 32 * q
                    if row < N and k0 < K:
                        Wq[row, k0 // 2: k0 // 2 + 16] = \
                            _restore(np.ascontiguousarray(packed[base + 512 * j + 16 * lane: base + 512 * j + 16 * lane + 16]))
            for p in range(1024 // g):
                l0 = p * (g // 32)
                r, q0 = l0 // 4, l0 % 4
                vals = packed[base + 2048 + 16 * p: base + 2048 + 16 * p + 16].view("<u2")
                i = 0
                for h in range(2):
                    grp = (256 * c + 128 * h + 32 * q0) // g
                    for row in (16 * t + r, 16 * t + r + 8):
                        if row < N and grp < ng:
                            sc[row, grp], of[row, grp] = vals[i], vals[i + 1]
                            seen[row, grp] += 1
                        i += 2
    return Wq, sc, of, seen
