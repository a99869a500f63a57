"""Packed int4 byte layout (KMR4 v1), written from its specification.

TEST INFRASTRUCTURE ONLY (see the package docstring).  The layout is the
library's own; this module restates its specification — given in words in
the C header of the library — as a direct address computation, so that the
library's packer can be checked bit for bit against it.  Nothing here is
shared with the CUDA path.

Specification, restated:
  W_ks = largest multiple of 128 dividing K with W_ks <= 1024; KSL = K / W_ks.
  Rows in tiles of 8 (padding rows: q = 8, s = z = 0).  Gate/up packing puts
  gate rows 4t..4t+3 then up rows 4t..4t+3 into tile t.
  Unit (t, j) at byte (t * KSL + j) * UB, UB = 4 * W_ks + W_ks / 4:
    nibble of (row r of tile, input k = j*W_ks + 8i + e) lives in the 32-bit
    little-endian word at byte r * W_ks/2 + 4i, bit offset BITOFF[e];
    (s, z) of (row r, group gl) are the two little-endian uint16 at byte
    4*W_ks + (r * (W_ks/128) + gl) * 4.
"""
from __future__ import annotations

import numpy as np

BITOFF = (0, 16, 4, 20, 8, 24, 12, 28)


def slice_width(K: int) -> int:
    for w in range(1024, 0, -128):
        if K % w == 0:
            return w
    raise ValueError(f"K={K} is not a multiple of 128")


def packed_size(N: int, K: int, group: int = 128) -> int:
    assert group == 128 and K % 128 == 0
    W = slice_width(K)
    return ((N + 7) // 8) * (K // W) * (4 * W + W // 4)


def canonical_row_of_packed_row(N: int, gate_up: bool) -> np.ndarray:
    """For each packed row index p (N padded to 8), the canonical row or -1 (padding)."""
    Np = (N + 7) // 8 * 8
    out = np.full(Np, -1, dtype=np.int64)
    if not gate_up:
        out[:N] = np.arange(N)
        return out
    assert N % 8 == 0, "gate/up packing needs N/2 a multiple of 4"
    half = N // 2
    for p in range(Np):
        t, r = divmod(p, 8)
        out[p] = 4 * t + r if r < 4 else half + 4 * t + (r - 4)
    return out


def pack_int4_spec(q: np.ndarray, s_bits: np.ndarray, z_bits: np.ndarray,
                   group: int = 128, gate_up: bool = False) -> np.ndarray:
    """Packed bytes (uint8 array of packed_size) of canonical q [N,K], s/z bf16 bits [N,K/128]."""
    q = np.asarray(q, dtype=np.uint8)
    N, K = q.shape
    W = slice_width(K)
    KSL = K // W
    UB = 4 * W + W // 4
    out = np.zeros(packed_size(N, K, group), dtype=np.uint8)
    src = canonical_row_of_packed_row(N, gate_up)
    for p, n in enumerate(src):
        t, r = divmod(p, 8)
        qrow = np.full(K, 8, np.uint8) if n < 0 else q[n]
        srow = np.zeros(K // 128, np.uint16) if n < 0 else np.asarray(s_bits[n], np.uint16)
        zrow = np.zeros(K // 128, np.uint16) if n < 0 else np.asarray(z_bits[n], np.uint16)
        for j in range(KSL):
            base = (t * KSL + j) * UB
            ks = qrow[j * W:(j + 1) * W].reshape(W // 8, 8).astype(np.uint32)   # [word i, e]
            words = np.zeros(W // 8, dtype=np.uint32)
            for e in range(8):
                words |= ks[:, e] << np.uint32(BITOFF[e])
            o = base + r * (W // 2)
            out[o:o + W // 2] = words.astype("<u4").view(np.uint8)
            G = W // 128
            sz = np.empty(2 * G, dtype="<u2")
            sz[0::2] = srow[j * G:(j + 1) * G]
            sz[1::2] = zrow[j * G:(j + 1) * G]
            o = base + 4 * W + r * G * 4
            out[o:o + 4 * G] = sz.view(np.uint8)
    return out
