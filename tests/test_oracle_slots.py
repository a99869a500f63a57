"""Pins of the KV row migration oracle (oracle/slots.py) — CPU only.

The oracle's slicing form is checked against an element-by-element loop on
tiny caches and against the invariants that define a row move ("kaminari",
§08 The serving layer: copy_row_from moves a row's KV state into a slot of the
pool's static cache)."""
import numpy as np
import pytest

from oracle.slots import copy_row_from, copy_row_from_loops


def _cache(rng, L=2, slots=3, nkv=2, S=5, d=4):
    k = rng.integers(0, 1 << 16, size=(L, slots, nkv, S, d), dtype=np.uint16)
    v = rng.integers(0, 1 << 16, size=(L, slots, nkv, S, d), dtype=np.uint16)
    return k, v


@pytest.mark.parametrize("length", [0, 1, 3, 5])
def test_matches_element_loop(length):
    rng = np.random.default_rng(1)
    dk, dv = _cache(rng)
    sk, sv = _cache(rng, slots=2, S=6)
    a = (dk.copy(), dv.copy())
    b = (dk.copy(), dv.copy())
    copy_row_from(a[0], a[1], 2, sk, sv, 1, length)
    copy_row_from_loops(b[0], b[1], 2, sk, sv, 1, length)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_only_the_prefix_of_the_destination_row_changes():
    rng = np.random.default_rng(2)
    dk, dv = _cache(rng)
    sk, sv = _cache(rng)
    k0, v0 = dk.copy(), dv.copy()
    copy_row_from(dk, dv, 0, sk, sv, 2, 3)
    assert np.array_equal(dk[:, 0, :, :3], sk[:, 2, :, :3]) and np.array_equal(dv[:, 0, :, :3], sv[:, 2, :, :3])
    assert np.array_equal(dk[:, 0, :, 3:], k0[:, 0, :, 3:]) and np.array_equal(dv[:, 0, :, 3:], v0[:, 0, :, 3:])
    assert np.array_equal(dk[:, 1:], k0[:, 1:]) and np.array_equal(dv[:, 1:], v0[:, 1:])


def test_move_and_move_back_restore_the_row():
    rng = np.random.default_rng(3)
    k, v = _cache(rng)
    k0, v0 = k.copy(), v.copy()
    copy_row_from(k, v, 2, k, v, 0, 5)          # row 0 -> row 2 (same cache)
    copy_row_from(k, v, 0, k, v, 2, 5)          # and back
    assert np.array_equal(k[:, 0], k0[:, 0]) and np.array_equal(v[:, 0], v0[:, 0])
    assert np.array_equal(k[:, 1], k0[:, 1])


def test_self_copy_and_empty_copy_change_nothing():
    rng = np.random.default_rng(4)
    k, v = _cache(rng)
    k0, v0 = k.copy(), v.copy()
    copy_row_from(k, v, 1, k, v, 1, 5)
    copy_row_from(k, v, 0, k, v, 2, 0)
    assert np.array_equal(k, k0) and np.array_equal(v, v0)


def test_shape_and_length_checks():
    rng = np.random.default_rng(5)
    dk, dv = _cache(rng)
    sk, sv = _cache(rng, nkv=1)
    with pytest.raises(ValueError):
        copy_row_from(dk, dv, 0, sk, sv, 0, 1)
    sk, sv = _cache(rng, S=2)
    with pytest.raises(ValueError):
        copy_row_from(dk, dv, 0, sk, sv, 0, 3)
