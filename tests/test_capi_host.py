"""Host-side checks of the C ABI: the library loads, exports every symbol the
header declares, packs bit-exactly on the host against the layout
specification, and rejects bad arguments before touching a GPU."""
import ctypes
import os
import re

import numpy as np
import pytest

import int4_weight_only_group_gb300 as kmr
from oracle import packspec
from workloads import f32_to_bf16_bits

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(kmr.library_path()):
        from int4_weight_only_group_gb300.build import build
        build()
    return kmr.lib()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "kmr.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kmr_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported_and_bound(L):
    declared = _declared_functions()
    assert len(declared) >= 20
    for name in declared:
        assert hasattr(L, name), name                      # dlsym succeeds
        assert name in kmr.EXPORTED_SYMBOLS, name          # the binding declares its signature
    assert sorted(kmr.EXPORTED_SYMBOLS) == declared


def test_status_strings_and_version(L):
    assert kmr.kmr_layout_version() == 2
    assert kmr.kmr_status_string(0) == "ok"
    for code in range(-9, 0):
        assert kmr.kmr_status_string(code) != "unknown status"


def _canon(r, N, K):
    q = r.integers(0, 16, (N, K), dtype=np.uint8)
    s = f32_to_bf16_bits(r.uniform(0.002, 0.02, (N, K // 128)).astype(np.float32))
    z = f32_to_bf16_bits((r.standard_normal((N, K // 128)) * 0.005).astype(np.float32))
    return q, s, z


@pytest.mark.parametrize("N,K,flags", [(8, 128, 0), (13, 256, 0), (40, 768, 0), (64, 2048, 0), (24, 6144, 0),
                                       (16, 640, 1), (48, 2048, 1), (32, 384, 1)])
def test_host_pack_matches_spec_and_roundtrips(L, N, K, flags):
    r = np.random.default_rng(N * 7 + K)
    q, s, z = _canon(r, N, K)
    size = kmr.kmr_packed_size(N, K, 128)
    assert size == packspec.packed_size(N, K)
    out = np.zeros(size, np.uint8)
    kmr.kmr_pack_int4(q, s, z, N, K, 128, flags, out, size, 0)
    assert np.array_equal(out, packspec.pack_int4_spec(q, s, z, gate_up=bool(flags)))
    q2, s2, z2 = np.zeros_like(q), np.zeros_like(s), np.zeros_like(z)
    kmr.kmr_unpack_int4(out, size, N, K, 128, flags, q2, s2, z2, 0)
    assert np.array_equal(q, q2) and np.array_equal(s, s2) and np.array_equal(z, z2)


def test_every_code_value_roundtrips(L):
    # every code at every nibble position, every byte pattern, and extreme s/z bit patterns
    N, K = 64, 1024
    r = np.random.default_rng(99)
    q = r.integers(0, 16, (N, K), dtype=np.uint8)
    s = r.integers(0, 65536, (N, K // 128), dtype=np.uint16)
    z = r.integers(0, 65536, (N, K // 128), dtype=np.uint16)
    s[0, 0], z[0, 0] = 0xFFFF, 0x8000
    size = kmr.kmr_packed_size(N, K, 128)
    out = np.zeros(size, np.uint8)
    kmr.kmr_pack_int4(q, s, z, N, K, 128, 0, out, size, 0)
    nib = out.reshape(-1, 1088)[:, :1024].reshape(-1)
    assert set(np.unique(nib)) == set(range(256))
    q2, s2, z2 = np.zeros_like(q), np.zeros_like(s), np.zeros_like(z)
    kmr.kmr_unpack_int4(out, size, N, K, 128, 0, q2, s2, z2, 0)
    assert np.array_equal(q, q2) and np.array_equal(s, s2) and np.array_equal(z, z2)


def test_host_pack_rejects_bad_input(L):
    q = np.full((8, 128), 8, np.uint8)
    s = np.zeros((8, 1), np.uint16)
    out = np.zeros(kmr.kmr_packed_size(8, 128, 128), np.uint8)
    with pytest.raises(kmr.KmrError) as e:
        kmr.kmr_pack_int4(q, s, s, 8, 100, 128, 0, out, out.size, 0)
    assert e.value.code == kmr.KMR_ERR_SHAPE
    with pytest.raises(kmr.KmrError) as e:
        kmr.kmr_pack_int4(q, s, s, 8, 128, 64, 0, out, out.size, 0)
    assert e.value.code == kmr.KMR_ERR_SHAPE
    with pytest.raises(kmr.KmrError) as e:
        kmr.kmr_pack_int4(q, s, s, 8, 128, 128, 0, out, out.size - 16, 0)
    assert e.value.code == kmr.KMR_ERR_BUFFER_SIZE
    bad = q.copy()
    bad[3, 5] = 16
    with pytest.raises(kmr.KmrError) as e:
        kmr.kmr_pack_int4(bad, s, s, 8, 128, 128, 0, out, out.size, 0)
    assert e.value.code == kmr.KMR_ERR_INVALID_ARG
    with pytest.raises(kmr.KmrError) as e:
        kmr.kmr_pack_int4(q, s, s, 8, 128, 128, 4, out, out.size, 0)
    assert e.value.code == kmr.KMR_ERR_INVALID_ARG
    assert kmr.kmr_packed_size(8, 100, 128) == 0


def test_entry_points_reject_bad_arguments_without_a_gpu(L):
    # every check below runs on the host before any CUDA call
    assert L.kmr_int4_gemv(None, 8, 128, 128, 0, None, 1, None, 0, None) == kmr.KMR_ERR_INVALID_ARG
    assert L.kmr_int4_gemv(1, 8, 100, 128, 0, 1, 1, 1, 0, None) == kmr.KMR_ERR_SHAPE
    assert L.kmr_int4_gemv(1, 8, 128, 64, 0, 1, 1, 1, 0, None) == kmr.KMR_ERR_SHAPE
    assert L.kmr_int4_gemv(1, 8, 8320, 128, 0, 1, 1, 1, 0, None) == kmr.KMR_ERR_SHAPE
    assert L.kmr_int4_gemv(1, 8, 128, 128, 0, 1, 0, 1, 0, None) == kmr.KMR_ERR_BATCH
    assert L.kmr_int4_gemv(1, 8, 128, 128, 0, 1, 17, 1, 0, None) == kmr.KMR_ERR_BATCH
    assert L.kmr_int4_gemv(1, 16, 128, 128, 0, 1, 1, 1, 2, None) == kmr.KMR_ERR_INVALID_ARG   # SiLU needs gate/up packing
    assert L.kmr_int4_gemv(1, 8, 128, 128, 1, 1, 1, 1, 2, None) == kmr.KMR_ERR_INVALID_ARG    # N not a multiple of 16
    assert L.kmr_int4_gemv(1, 8, 128, 128, 0, 1, 1, 1, 7, None) == kmr.KMR_ERR_INVALID_ARG
    assert L.kmr_int4_gemv(1, 8, 128, 128, 2, 1, 1, 1, 0, None) == kmr.KMR_ERR_INVALID_ARG
    assert L.kmr_decode_attn(None, 1, 1, 1, 1, 1, 16, 8, 128, 64, 1, 0.1, 1, 1, 1 << 30, None) == kmr.KMR_ERR_INVALID_ARG
    assert L.kmr_decode_attn(1, 1, 1, 1, 1, 1, 16, 8, 96, 64, 1, 0.1, 1, 1, 1 << 30, None) == kmr.KMR_ERR_SHAPE
    assert L.kmr_decode_attn(1, 1, 1, 1, 1, 1, 16, 5, 128, 64, 1, 0.1, 1, 1, 1 << 30, None) == kmr.KMR_ERR_SHAPE
    assert L.kmr_decode_attn(1, 1, 1, 1, 1, 0, 16, 8, 128, 64, 1, 0.1, 1, 1, 1 << 30, None) == kmr.KMR_ERR_BATCH
    assert L.kmr_decode_attn(1, 1, 1, 1, 1, 2, 16, 8, 128, 64, 1, 0.1, 1, 1, 16, None) == kmr.KMR_ERR_BUFFER_SIZE
    # shared-prefix attention: (q, k, v, slots, cpos, prefix_slot, prefix_len, B, nq, nkv, d, S, slots, scale, out, ws, n)
    C = L.kmr_decode_attn_cascade
    assert C(None, 1, 1, 1, 1, 0, 8, 2, 16, 8, 128, 64, 4, 0.1, 1, 1, 1 << 30, None) == kmr.KMR_ERR_INVALID_ARG
    assert C(1, 1, 1, 1, 1, 0, 8, 0, 16, 8, 128, 64, 4, 0.1, 1, 1, 1 << 30, None) == kmr.KMR_ERR_BATCH
    assert C(1, 1, 1, 1, 1, 0, 8, 2, 16, 8, 96, 64, 4, 0.1, 1, 1, 1 << 30, None) == kmr.KMR_ERR_SHAPE
    assert C(1, 1, 1, 1, 1, 0, 8, 2, 16, 6, 128, 64, 4, 0.1, 1, 1, 1 << 30, None) == kmr.KMR_ERR_SHAPE
    assert C(1, 1, 1, 1, 1, 4, 8, 2, 16, 8, 128, 64, 4, 0.1, 1, 1, 1 << 30, None) == kmr.KMR_ERR_SLOT_RANGE
    assert C(1, 1, 1, 1, 1, 0, 64, 2, 16, 8, 128, 64, 4, 0.1, 1, 1, 1 << 30, None) == kmr.KMR_ERR_CACHE_FULL
    assert C(1, 1, 1, 1, 1, 0, -1, 2, 16, 8, 128, 64, 4, 0.1, 1, 1, 1 << 30, None) == kmr.KMR_ERR_INVALID_ARG
    assert C(1, 1, 1, 1, 1, 0, 8, 2, 16, 8, 128, 64, 4, 0.1, 1, None, 1 << 30, None) == kmr.KMR_ERR_INVALID_ARG
    assert C(1, 1, 1, 1, 1, 0, 8, 2, 16, 8, 128, 64, 4, 0.1, 1, 1, 16, None) == kmr.KMR_ERR_BUFFER_SIZE
    assert C(1, 1, 1, 1, 1, 0, 8, 2, 16, 8, 128, 64, 4, float("nan"), 1, 1, 1 << 30, None) == kmr.KMR_ERR_INVALID_ARG
    W = L.kmr_decode_attn_cascade_workspace_size
    assert W(2, 16, 8, 128, 400) > 0 and W(2, 16, 8, 96, 400) == 0 and W(0, 16, 8, 128, 400) == 0
    assert W(2, 16, 8, 128, 400) == 2 * W(1, 16, 8, 128, 400)
    assert L.kmr_model_copy_row_from(None, 0, None, None, 0, 0, 0, 1, None) == kmr.KMR_ERR_INVALID_ARG
    assert L.kmr_decode_step(None, 1, 1, 1, 1, 1, 1, None, None) == kmr.KMR_ERR_INVALID_ARG
    assert L.kmr_decode_step_host(None, 1, 1, 1, 1, 1, 1, None, None) == kmr.KMR_ERR_INVALID_ARG
    assert L.kmr_model_destroy(None) == kmr.KMR_ERR_INVALID_ARG
    assert L.kmr_model_sync_status(None, None) == kmr.KMR_ERR_INVALID_ARG
    assert L.kmr_model_set_prefill_tcgen05(None, 1) == kmr.KMR_ERR_INVALID_ARG
    assert L.kmr_model_set_prefill_plan(None, 0, 0) == kmr.KMR_ERR_INVALID_ARG
    assert L.kmr_selftest_wait_timeout(999, None) == kmr.KMR_ERR_INVALID_ARG          # below 1 us
    assert L.kmr_selftest_wait_timeout(2_000_000_001, None) == kmr.KMR_ERR_INVALID_ARG  # above 2 s
    assert L.kmr_model_kernels_per_step(None, 1) == 0
    assert L.kmr_model_device_bytes(None, None, None, None) == 0
    assert L.kmr_model_set_persistent_step(None, 1) == kmr.KMR_ERR_INVALID_ARG


def test_model_create_rejects_bad_config_on_host(L):
    from workloads import tiny_config
    cfg = tiny_config()
    bad_cases = [dict(head_dim=96), dict(group=64), dict(n_kv_heads=3), dict(mrope_sections=(8, 12, 11)),
                 dict(hidden=200), dict(max_len=0), dict(eos_id=5000)]
    for kw in bad_cases:
        c = kmr.ModelConfig()
        base = dict(cfg.__dict__)
        base.update(kw)
        for f, _ in kmr.ModelConfig._fields_:
            if f == "mrope_sections":
                c.mrope_sections = (ctypes.c_int * 3)(*base["mrope_sections"])
            elif f == "max_batch":
                c.max_batch = 1
            elif f == "qk_norm":
                c.qk_norm = int(base["qk_norm"])
            else:
                setattr(c, f, base[f])
        h = ctypes.c_void_p()
        assert L.kmr_model_create(ctypes.byref(c), ctypes.byref(h)) == kmr.KMR_ERR_SHAPE, kw
        assert not h.value


def test_prefill_plan_split_depends_on_the_shape_only(L):
    """The tcgen05 prefill plan on the host: the K split of each 2B projection is the same for
    every prompt length (so chunked and one-chunk prefill sum each output in the same order), the
    tile width is one of 64/128/256, the split never exceeds K / 128, and at 512 tokens on 152 SMs
    the plans are the fastest ones a GB300 sweep measured for each projection."""
    shapes = {"qkv": (4096, 2048), "o": (2048, 2048), "gate_up": (12288, 2048), "down": (2048, 6144),
              "tiny_qkv": (512, 256), "tiny_down": (256, 768)}
    for name, (N, K) in shapes.items():
        splits = set()
        for M in (1, 7, 16, 100, 128, 200, 256, 300, 512, 777, 1024, 2048):
            nt, ks = kmr.kmr_prefill_plan(N, K, M, 152)
            assert nt in (64, 128, 256) and ks in (1, 2, 4) and ks <= K // 128, (name, M, nt, ks)
            splits.add(ks)
        assert len(splits) == 1, (name, splits)
    assert kmr.kmr_prefill_plan(4096, 2048, 512, 152) == (128, 1)
    assert kmr.kmr_prefill_plan(2048, 2048, 512, 152) == (128, 2)
    assert kmr.kmr_prefill_plan(12288, 2048, 512, 152) == (256, 1)
    assert kmr.kmr_prefill_plan(2048, 6144, 512, 152) == (256, 4)
    nt, ks = ctypes.c_int(), ctypes.c_int()
    for args in ((100, 2048, 512, 152), (4096, 100, 512, 152), (4096, 16384, 512, 152), (4096, 2048, 0, 152),
                 (4096, 2048, 512, 0)):
        assert L.kmr_prefill_plan(*args, ctypes.byref(nt), ctypes.byref(ks)) == kmr.KMR_ERR_INVALID_ARG, args
    assert L.kmr_prefill_plan(4096, 2048, 512, 152, None, None) == kmr.KMR_ERR_INVALID_ARG
