"""Plain CPU oracle of KV row migration between static caches.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, links or
executes this file; only tests do.  It shares no code with the CUDA path.

Source: "kaminari — a single-GPU Qwen3-VL inference engine, explained",
§08 The serving layer (the continuous scheduler's slot pool owns one static
cache with a physical row per slot; copy_row_from moves a row's KV state into
it) and §03 State model (the cache buffers mutate in place; everything else is
replaced, not mutated).

A cache is a pair of arrays K, V of shape [L][slots][n_kv][max_len][d] (bf16
bit patterns, compared as integers).  Moving row r of a source cache into row
s of a destination cache for the first `length` positions means: for every
layer, head and position p < length, destination[l][s][h][p] = source[l][r][h][p],
for K and for V; nothing else of the destination changes.  The reading of
"migrates a row's KV state" as "the filled prefix [0, length) of the row" is
ours (the pages give no signature); positions at or past `length` are not part
of the row's state.

Pinned in tests/test_oracle_slots.py against an element-by-element loop on
tiny caches and against invariants (a copy and its inverse restore the row,
untouched slots and positions keep their bits, length 0 and a copy of a row
onto itself change nothing).
"""
from __future__ import annotations

import numpy as np

__all__ = ["copy_row_from", "copy_row_from_loops"]


def copy_row_from(dst_k: np.ndarray, dst_v: np.ndarray, dst_slot: int, src_k: np.ndarray, src_v: np.ndarray,
                  src_row: int, length: int) -> None:
    """Write positions [0, length) of row src_row of (src_k, src_v) into row dst_slot of
    (dst_k, dst_v), every layer and head, in place (arrays [L][slots][n_kv][max_len][d])."""
    for dst, src in ((dst_k, src_k), (dst_v, src_v)):
        if dst.shape[0] != src.shape[0] or dst.shape[2:3] != src.shape[2:3] or dst.shape[4] != src.shape[4]:
            raise ValueError("caches differ in layers, KV heads or head size")
        if not (0 <= length <= min(dst.shape[3], src.shape[3])):
            raise ValueError("length outside both caches")
        dst[:, dst_slot, :, :length, :] = src[:, src_row, :, :length, :].copy()


def copy_row_from_loops(dst_k, dst_v, dst_slot: int, src_k, src_v, src_row: int, length: int) -> None:
    """The same, one element at a time (tiny caches only: the brute-force pin)."""
    L, _, nkv, _, d = dst_k.shape
    for dst, src in ((dst_k, src_k), (dst_v, src_v)):
        for l in range(L):
            for h in range(nkv):
                for p in range(length):
                    for e in range(d):
                        dst[l, dst_slot, h, p, e] = src[l, src_row, h, p, e]
