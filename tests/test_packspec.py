"""Pins of the packed-layout restatement (oracle/packspec.py) on hand-placed values."""
import numpy as np

from oracle import packspec as ps


def _canon(N, K, fill=8):
    return (np.full((N, K), fill, np.uint8), np.zeros((N, K // 128), np.uint16),
            np.zeros((N, K // 128), np.uint16))


def test_slice_width_and_size():
    assert ps.slice_width(2048) == 1024 and ps.slice_width(6144) == 1024
    assert ps.slice_width(256) == 256 and ps.slice_width(768) == 768 and ps.slice_width(640) == 640
    # K/2 nibble bytes + 4 bytes (s, z) per group, per row, rows padded to 8
    assert ps.packed_size(4096, 2048) == 4096 * (1024 + 64) == 4456448
    assert ps.packed_size(2048, 6144) == 2048 * (3072 + 192) == 6684672
    assert ps.packed_size(5, 256) == 8 * (128 + 8)


def test_hand_placed_nibbles():
    N, K = 8, 256
    q, s, z = _canon(N, K)
    q[0, 1] = 3        # word 0, e = 1 -> bit 16 -> byte 2, low nibble
    q[0, 2] = 5        # e = 2 -> bit 4 -> byte 0, high nibble
    q[1, 15] = 0       # row 1 word 1, e = 7 -> bit 28 -> byte 128 + 4 + 3, high nibble
    q[0, 255] = 15     # last word (31) of row 0, e = 7 -> byte 124 + 3, high nibble
    p = ps.pack_int4_spec(q, s, z)
    assert p.size == 8 * 136
    assert p[0] == 0x58 and p[2] == 0x83
    assert p[128 + 7] == 0x08
    assert p[127] == 0xF8
    untouched = np.ones(1024, bool)
    untouched[[0, 2, 135, 127]] = False
    assert np.all(p[:1024][untouched] == 0x88)


def test_scale_zero_placement_and_padding():
    N, K = 3, 256       # padded to 8 rows
    q, s, z = _canon(N, K, fill=1)
    s[2, 1] = 0x1234
    z[2, 1] = 0xABCD
    p = ps.pack_int4_spec(q, s, z)
    base = 4 * 256 + (2 * 2 + 1) * 4      # row 2, group 1
    assert p[base:base + 4].tolist() == [0x34, 0x12, 0xCD, 0xAB]
    # padding rows 3..7 hold code 8 everywhere (zero weights)
    assert np.all(p[3 * 128:8 * 128] == 0x88) and np.all(p[:3 * 128] == 0x11)


def test_gate_up_row_order():
    N, K = 16, 128
    q = np.tile(np.arange(N, dtype=np.uint8)[:, None], (1, K))   # row n holds code n
    s = np.zeros((N, 1), np.uint16)
    p = ps.pack_int4_spec(q, s, s, gate_up=True)
    UB = 4 * 128 + 32
    got = [p[t * UB + r * 64] & 0xF for t in range(2) for r in range(8)]
    # tile 0: gate 0..3 then up 0..3 (= canonical 8..11); tile 1: gate 4..7, up 12..15
    assert got == [0, 1, 2, 3, 8, 9, 10, 11, 4, 5, 6, 7, 12, 13, 14, 15]
