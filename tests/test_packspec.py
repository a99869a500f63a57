"""Pins of the packed-layout restatement (oracle/packspec.py) on hand-placed values."""
import numpy as np

from oracle import packspec as ps


def _canon(N, K, fill=8):
    return (np.full((N, K), fill, np.uint8), np.zeros((N, K // 128), np.uint16),
            np.zeros((N, K // 128), np.uint16))


def test_size():
    # K/2 nibble bytes + 4 bytes (s, z) per group, per row, rows padded to 16
    assert ps.packed_size(4096, 2048) == 4096 * (1024 + 64) == 4456448
    assert ps.packed_size(2048, 6144) == 2048 * (3072 + 192) == 6684672
    assert ps.packed_size(5, 256) == 16 * (128 + 8)


def test_hand_placed_nibbles():
    N, K = 16, 128
    q, s, z = _canon(N, K)
    q[0, 1] = 3        # (g=0, k0+2t+1) of lane 0, k-step 0 -> word at 0, bit 16 -> byte 2 low nibble
    q[8, 0] = 5        # row g+8 of lane 0, k 0 -> bit 4 -> byte 0 high nibble
    q[9, 27] = 0       # k-step 1 (k0=16), k 27 = k0 + 2*1 + 9 -> lane 4*1+1=5, row g+8 (g=1), bit 28
    q[15, 127] = 15    # k-step 7 (k0=112), k = 112 + 2*3 + 9 -> lane 4*7+3=31, row g+8 (g=7), bit 28
    p = ps.pack_int4_spec(q, s, z)
    assert p.size == 1088
    assert p[0] == 0x58 and p[2] == 0x83
    # lane 5, k-step 1: byte offset 5*16 + 1*4 = 84, bit 28 -> byte 87 high nibble
    assert p[87] == 0x08
    # lane 31, k-step 7: (7 // 4) * 512 + 31 * 16 + 3 * 4 = 1020, bit 28 -> byte 1023 high nibble
    assert p[1023] == 0xF8
    untouched = np.ones(1024, bool)
    untouched[[0, 2, 87, 1023]] = False
    assert np.all(p[:1024][untouched] == 0x88)


def test_scale_zero_placement_and_padding():
    N, K = 3, 256       # padded to 16 rows
    q, s, z = _canon(N, K, fill=1)
    s[2, 1] = 0x1234
    z[2, 1] = 0xABCD
    p = ps.pack_int4_spec(q, s, z)
    base = 1 * 1088 + 1024 + 2 * 4      # group 1, row 2
    assert p[base:base + 4].tolist() == [0x34, 0x12, 0xCD, 0xAB]
    # lanes with g >= 3 and rows g+8 hold padding code 8; lane 0 word 0 mixes row 0 (code 1) and row 8 (code 8)
    w = int(np.frombuffer(p[0:4].tobytes(), "<u4")[0])
    assert (w >> 0) & 15 == 1 and (w >> 4) & 15 == 8 and (w >> 16) & 15 == 1 and (w >> 20) & 15 == 8
    w12 = int(np.frombuffer(p[12 * 16:12 * 16 + 4].tobytes(), "<u4")[0])   # lane 12: g = 3 (padding)
    assert w12 == 0x88888888


def test_gate_up_row_order():
    N, K = 32, 128
    q = np.tile((np.arange(N) % 16).astype(np.uint8)[:, None], (1, K))   # row n holds code n % 16
    s = np.zeros((N, 1), np.uint16)
    p = ps.pack_int4_spec(q, s, s, gate_up=True)
    got = []
    for T in range(2):
        for g in range(8):
            w = int(np.frombuffer(p[T * 1088 + 4 * g * 16:T * 1088 + 4 * g * 16 + 4].tobytes(), "<u4")[0])
            got.append((w & 15, (w >> 4) & 15))     # (tile row g, tile row g + 8)
    # tile 0: rows g = gate g (codes 0..7), rows g+8 = up g (canonical 16+g -> code g)
    # tile 1: rows g = gate 8+g (codes 8..15), rows g+8 = up 8+g (canonical 24+g -> code 8+g)
    assert got == [(g, g) for g in range(8)] + [(8 + g, 8 + g) for g in range(8)]
