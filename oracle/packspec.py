"""Packed int4 byte layout (KMR4 v2), written from its specification.

TEST INFRASTRUCTURE ONLY (see the package docstring).  The layout is the
library's own; this module restates its specification — given in words in
the C header of the library — as a direct address computation, so that the
library's packer can be checked bit for bit against it.  Nothing here is
shared with the CUDA path.

Specification, restated:
  Rows in tiles of 16 (padding rows: q = 8, s = z = 0).  Gate/up packing puts
  gate rows 8t..8t+7 then up rows 8t..8t+7 into tile t.
  Group gr (128 inputs) of tile T occupies 1088 bytes at (T * K/128 + gr) * 1088.
  For k-step ks (k0 = 128 gr + 16 ks) and lane l (g = l // 4, t = l % 4) the
  little-endian 32-bit word at (ks // 4) * 512 + l * 16 + (ks % 4) * 4 holds the
  codes of (tile row, input) at these bit offsets:
      0: (g, k0+2t)    16: (g, k0+2t+1)    4: (g+8, k0+2t)    20: (g+8, k0+2t+1)
      8: (g, k0+2t+8)  24: (g, k0+2t+9)   12: (g+8, k0+2t+8)  28: (g+8, k0+2t+9)
  Bytes 1024 + 4 r hold (s, z) of tile row r for that group, little-endian uint16.
"""
from __future__ import annotations

import numpy as np

GROUP_BYTES = 1088
# (row offset within the 16x16 block, input offset relative to k0 + 2t, bit offset)
NIBBLES = ((0, 0, 0), (0, 1, 16), (8, 0, 4), (8, 1, 20), (0, 8, 8), (0, 9, 24), (8, 8, 12), (8, 9, 28))


def packed_size(N: int, K: int, group: int = 128) -> int:
    assert group == 128 and K % 128 == 0
    return ((N + 15) // 16) * (K // 128) * GROUP_BYTES


def canonical_row_of_packed_row(N: int, gate_up: bool) -> np.ndarray:
    """For each packed row index p (N padded to 16), the canonical row or -1 (padding)."""
    Np = (N + 15) // 16 * 16
    out = np.full(Np, -1, dtype=np.int64)
    if not gate_up:
        out[:N] = np.arange(N)
        return out
    assert N % 16 == 0, "gate/up packing needs N/2 a multiple of 8"
    half = N // 2
    for p in range(Np):
        t, r = divmod(p, 16)
        out[p] = 8 * t + r if r < 8 else half + 8 * t + (r - 8)
    return out


def pack_int4_spec(q: np.ndarray, s_bits: np.ndarray, z_bits: np.ndarray,
                   group: int = 128, gate_up: bool = False) -> np.ndarray:
    """Packed bytes (uint8 array of packed_size) of canonical q [N,K], s/z bf16 bits [N,K/128]."""
    q = np.asarray(q, dtype=np.uint8)
    N, K = q.shape
    G = K // 128
    src = canonical_row_of_packed_row(N, gate_up)
    Np = src.size
    # canonical arrays re-indexed by packed row (padding: code 8, s = z = 0)
    qp = np.full((Np, K), 8, np.uint32)
    sp = np.zeros((Np, G), np.uint16)
    zp = np.zeros((Np, G), np.uint16)
    have = src >= 0
    qp[have] = q[src[have]]
    sp[have] = np.asarray(s_bits, np.uint16)[src[have]]
    zp[have] = np.asarray(z_bits, np.uint16)[src[have]]
    out = np.zeros(packed_size(N, K, group), dtype=np.uint8)
    lanes = np.arange(32)
    g_l, t_l = lanes // 4, lanes % 4
    for T in range(Np // 16):
        for gr in range(G):
            base = (T * G + gr) * GROUP_BYTES
            for ks in range(8):
                k0 = 128 * gr + 16 * ks
                words = np.zeros(32, np.uint32)
                for dr, dk, bit in NIBBLES:
                    words |= qp[16 * T + g_l + dr, k0 + 2 * t_l + dk] << np.uint32(bit)
                for l in range(32):
                    o = base + (ks // 4) * 512 + l * 16 + (ks % 4) * 4
                    out[o:o + 4] = np.array([words[l]], "<u4").view(np.uint8)
            for r in range(16):
                o = base + 1024 + 4 * r
                out[o:o + 4] = np.array([sp[16 * T + r, gr], zp[16 * T + r, gr]], "<u2").view(np.uint8)
    return out
