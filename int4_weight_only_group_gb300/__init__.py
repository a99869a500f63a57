"""GB300 int4 weight-only, group-wise decode step — Python binding of libkmr.

Argument marshalling only: every step of the decode path runs in the CUDA
kernels of ``_lib/libkmr.so`` behind the C ABI declared in ``include/kmr.h``.
PyTorch is used only for device memory and streams.  There is no fallback:
if the library has not been built, every call raises ``KmrLibraryMissing``.

Names follow the C ABI (``kmr_pack_int4``, ``kmr_int4_gemv``,
``kmr_decode_attn``, ``kmr_decode_step`` ...).  Arrays may be numpy arrays
(host memory), torch tensors (host or device; their data pointer is passed)
or raw integer addresses.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence, Tuple

__all__ = [
    "KmrError", "KmrLibraryMissing", "lib", "library_path", "EXPORTED_SYMBOLS",
    "KMR_OK", "KMR_ERR_INVALID_ARG", "KMR_ERR_SHAPE", "KMR_ERR_SLOT_RANGE", "KMR_ERR_CACHE_FULL",
    "KMR_ERR_NO_PACK", "KMR_ERR_CUDA", "KMR_ERR_DEVICE_TIMEOUT", "KMR_ERR_BUFFER_SIZE", "KMR_ERR_BATCH",
    "KMR_PACK_GATE_UP", "KMR_EPI_NONE", "KMR_EPI_RESIDUAL", "KMR_EPI_SILU_MUL",
    "KMR_W_QKV", "KMR_W_O", "KMR_W_GATE_UP", "KMR_W_DOWN", "KMR_N_INPUT", "KMR_N_POST", "KMR_N_Q", "KMR_N_K",
    "ModelConfig", "kmr_status_string", "kmr_layout_version", "kmr_packed_size", "kmr_pack_int4",
    "kmr_unpack_int4", "kmr_int4_gemv", "kmr_decode_attn_workspace_size",
    "kmr_decode_attn", "kmr_decode_attn_noalloc", "kmr_decode_attn_cascade_workspace_size",
    "kmr_decode_attn_cascade", "kmr_last_device_error", "kmr_smem_poison", "kmr_selftest_wait_timeout", "Model",
]

KMR_OK = 0
KMR_ERR_INVALID_ARG = -1
KMR_ERR_SHAPE = -2
KMR_ERR_SLOT_RANGE = -3
KMR_ERR_CACHE_FULL = -4
KMR_ERR_NO_PACK = -5
KMR_ERR_CUDA = -6
KMR_ERR_DEVICE_TIMEOUT = -7
KMR_ERR_BUFFER_SIZE = -8
KMR_ERR_BATCH = -9
KMR_PACK_GATE_UP = 1
KMR_EPI_NONE, KMR_EPI_RESIDUAL, KMR_EPI_SILU_MUL = 0, 1, 2
KMR_W_QKV, KMR_W_O, KMR_W_GATE_UP, KMR_W_DOWN = 0, 1, 2, 3
KMR_N_INPUT, KMR_N_POST, KMR_N_Q, KMR_N_K = 0, 1, 2, 3

_HERE = os.path.dirname(os.path.abspath(__file__))


def library_path() -> str:
    return os.path.join(_HERE, "_lib", "libkmr.so")


class KmrError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {kmr_status_string(code)} ({code})")


class KmrLibraryMissing(ImportError):
    pass


class ModelConfig(ctypes.Structure):
    """Mirror of kmr_model_config."""
    _fields_ = [
        ("hidden", ctypes.c_int), ("n_q_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int),
        ("head_dim", ctypes.c_int), ("intermediate", ctypes.c_int), ("vocab", ctypes.c_int),
        ("n_layers", ctypes.c_int), ("group", ctypes.c_int), ("eps", ctypes.c_float),
        ("rope_theta", ctypes.c_float), ("mrope_sections", ctypes.c_int * 3), ("qk_norm", ctypes.c_int),
        ("eos_id", ctypes.c_int), ("pad_id", ctypes.c_int), ("max_len", ctypes.c_int), ("slots", ctypes.c_int),
        ("max_batch", ctypes.c_int),
    ]


_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t
# name -> (restype, argtypes); every symbol include/kmr.h declares
_SIGNATURES = {
    "kmr_status_string": (ctypes.c_char_p, [_I]),
    "kmr_layout_version": (_I, []),
    "kmr_packed_size": (_SZ, [_I, _I, _I]),
    "kmr_pack_int4": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _SZ, _I, _P]),
    "kmr_unpack_int4": (_I, [_P, _SZ, _I, _I, _I, _I, _P, _P, _P, _I, _P]),
    "kmr_int4_gemv": (_I, [_P, _I, _I, _I, _I, _P, _I, _P, _I, _P]),
    "kmr_decode_attn_workspace_size": (_SZ, [_I, _I, _I, _I]),
    "kmr_decode_attn": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, ctypes.c_float, _P, _P, _SZ, _P]),
    "kmr_decode_attn_noalloc": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, ctypes.c_float, _P, _P]),
    "kmr_decode_attn_cascade_workspace_size": (_SZ, [_I, _I, _I, _I, _I]),
    "kmr_decode_attn_cascade": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, ctypes.c_float, _P, _P, _SZ,
                                     _P]),
    "kmr_last_device_error": (_I, []),
    "kmr_model_create": (_I, [ctypes.POINTER(ModelConfig), ctypes.POINTER(_P)]),
    "kmr_model_destroy": (_I, [_P]),
    "kmr_model_set_linear": (_I, [_P, _I, _I, _P, _P, _P]),
    "kmr_model_set_norm": (_I, [_P, _I, _I, _P]),
    "kmr_model_set_embedding": (_I, [_P, _P]),
    "kmr_model_set_kv": (_I, [_P, _I, _I, _I, _P, _P]),
    "kmr_model_kv_pointers": (_I, [_P, _I, ctypes.POINTER(_P), ctypes.POINTER(_P)]),
    "kmr_model_reserve_prefill": (_I, [_P, _I]),
    "kmr_prefill": (_I, [_P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P, _P]),
    "kmr_model_copy_row_from": (_I, [_P, _I, _P, _P, _I, _I, _I, _I, _P]),
    "kmr_decode_step": (_I, [_P, _P, _P, _P, _P, _P, _I, _P, _P]),
    "kmr_decode_step_host": (_I, [_P, _P, _P, _P, _P, _P, _I, _P, _P]),
    "kmr_model_sync_status": (_I, [_P, _P]),
    "kmr_model_kernels_per_step": (_I, [_P, _I]),
    "kmr_model_device_bytes": (_SZ, [_P, ctypes.POINTER(_SZ), ctypes.POINTER(_SZ), ctypes.POINTER(_SZ)]),
    "kmr_smem_poison": (_I, [ctypes.c_uint32, _P]),
    "kmr_selftest_wait_timeout": (_I, [ctypes.c_ulonglong, _P]),
    "kmr_model_set_smem_poison": (_I, [_P, _I, ctypes.c_uint32]),
    "kmr_model_set_prefill_tcgen05": (_I, [_P, _I]),
    "kmr_model_set_prefill_plan": (_I, [_P, _I, _I]),
    "kmr_prefill_plan": (_I, [_I, _I, _I, _I, _P, _P]),
    "kmr_model_set_persistent_step": (_I, [_P, _I]),
}
EXPORTED_SYMBOLS = tuple(_SIGNATURES)

_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libkmr (raises KmrLibraryMissing if it was never built)."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise KmrLibraryMissing(f"{path} is missing: build it with int4_weight_only_group_gb300.build.build()")
        L = ctypes.CDLL(path)
        for name, (res, args) in _SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


# ------------------------------------------------------------------ marshalling
def _ptr(a) -> Optional[int]:
    if a is None:
        return None
    if isinstance(a, int):
        return a
    if hasattr(a, "data_ptr"):           # torch.Tensor
        if not a.is_contiguous():
            raise ValueError("tensor must be contiguous")
        return a.data_ptr()
    if hasattr(a, "ctypes"):             # numpy.ndarray
        if not a.flags["C_CONTIGUOUS"]:
            raise ValueError("array must be C-contiguous")
        return a.ctypes.data
    raise TypeError(f"cannot pass {type(a).__name__} as a pointer")


def _stream(s) -> Optional[int]:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream                  # torch.cuda.Stream


def _check(code: int, where: str) -> None:
    if code != KMR_OK:
        raise KmrError(code, where)


# ------------------------------------------------------------------ C ABI wrappers
def kmr_status_string(code: int) -> str:
    try:
        return lib().kmr_status_string(code).decode()
    except KmrLibraryMissing:
        return f"status {code}"


def kmr_layout_version() -> int:
    return lib().kmr_layout_version()


def kmr_packed_size(N: int, K: int, group: int = 128) -> int:
    return lib().kmr_packed_size(N, K, group)


def kmr_pack_int4(q, s, z, N, K, group, flags, packed, packed_bytes, on_device, stream=None) -> None:
    _check(lib().kmr_pack_int4(_ptr(q), _ptr(s), _ptr(z), N, K, group, flags, _ptr(packed), packed_bytes,
                               int(on_device), _stream(stream)), "kmr_pack_int4")


def kmr_unpack_int4(packed, packed_bytes, N, K, group, flags, q, s, z, on_device, stream=None) -> None:
    _check(lib().kmr_unpack_int4(_ptr(packed), packed_bytes, N, K, group, flags, _ptr(q), _ptr(s), _ptr(z),
                                 int(on_device), _stream(stream)), "kmr_unpack_int4")


def kmr_int4_gemv(packed, N, K, group, flags, x, M, y, epilogue, stream=None) -> None:
    _check(lib().kmr_int4_gemv(_ptr(packed), N, K, group, flags, _ptr(x), M, _ptr(y), epilogue, _stream(stream)),
           "kmr_int4_gemv")


def kmr_decode_attn_workspace_size(B, nq, nkv, d) -> int:
    return lib().kmr_decode_attn_workspace_size(B, nq, nkv, d)


def kmr_decode_attn(q, k_cache, v_cache, slot_ids, cache_position, B, nq, nkv, d, max_len, slots, scale, out,
                    workspace, workspace_bytes, stream=None) -> None:
    _check(lib().kmr_decode_attn(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(slot_ids), _ptr(cache_position), B,
                                 nq, nkv, d, max_len, slots, float(scale), _ptr(out), _ptr(workspace),
                                 workspace_bytes, _stream(stream)), "kmr_decode_attn")


def kmr_decode_attn_noalloc(q, k_cache, v_cache, slot_ids, cache_position, B, nq, nkv, d, max_len, slots, scale,
                            out, stream=None) -> None:
    """kmr_decode_attn for callers that cannot allocate device memory: no workspace argument,
    the library's fixed device scratch is used instead (see include/kmr.h for its limit)."""
    _check(lib().kmr_decode_attn_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(slot_ids),
                                         _ptr(cache_position), B, nq, nkv, d, max_len, slots, float(scale),
                                         _ptr(out), _stream(stream)), "kmr_decode_attn_noalloc")


def kmr_decode_attn_cascade_workspace_size(B, nq, nkv, d, prefix_len) -> int:
    return lib().kmr_decode_attn_cascade_workspace_size(B, nq, nkv, d, prefix_len)


def kmr_decode_attn_cascade(q, k_cache, v_cache, slot_ids, cache_position, prefix_slot, prefix_len, B, nq, nkv, d,
                            max_len, slots, scale, out, workspace, workspace_bytes, stream=None) -> None:
    """Shared-prefix decode attention: row b attends [0, prefix_len) of cache row prefix_slot,
    then [prefix_len, cache_position[b]] of its own row (see include/kmr.h)."""
    _check(lib().kmr_decode_attn_cascade(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(slot_ids),
                                         _ptr(cache_position), prefix_slot, prefix_len, B, nq, nkv, d, max_len,
                                         slots, float(scale), _ptr(out), _ptr(workspace), workspace_bytes,
                                         _stream(stream)), "kmr_decode_attn_cascade")


def kmr_prefill_plan(N: int, K: int, M: int, sms: int) -> Tuple[int, int]:
    """kmr_prefill_plan: (tokens per CTA, K split) of a tcgen05 prefill projection (host only)."""
    nt, ks = ctypes.c_int(0), ctypes.c_int(0)
    _check(lib().kmr_prefill_plan(int(N), int(K), int(M), int(sms), ctypes.byref(nt), ctypes.byref(ks)),
           "kmr_prefill_plan")
    return nt.value, ks.value


def kmr_last_device_error() -> int:
    return lib().kmr_last_device_error()


def kmr_selftest_wait_timeout(limit_ns: int, stream=None) -> None:
    """Launch the bounded-wait self-test (a wait nothing completes gives up after limit_ns);
    kmr_last_device_error() then reads KMR_ERR_DEVICE_TIMEOUT."""
    _check(lib().kmr_selftest_wait_timeout(int(limit_ns), _stream(stream)), "kmr_selftest_wait_timeout")


def kmr_smem_poison(pattern: int, stream=None) -> None:
    """Fill every SM's shared memory with the 32-bit `pattern` (diagnostic; see include/kmr.h)."""
    _check(lib().kmr_smem_poison(pattern & 0xFFFFFFFF, _stream(stream)), "kmr_smem_poison")


# ------------------------------------------------------------------ model handle
class Model:
    """Owner of one kmr_model (packed weights, static KV cache, step scratch)."""

    def __init__(self, hidden, n_q_heads, n_kv_heads, head_dim, intermediate, vocab, n_layers, group=128,
                 eps=1e-6, rope_theta=1e6, mrope_sections: Sequence[int] = (16, 24, 24), qk_norm=True,
                 eos_id=-1, pad_id=0, max_len=1024, slots=1, max_batch=1):
        c = ModelConfig()
        c.hidden, c.n_q_heads, c.n_kv_heads, c.head_dim = hidden, n_q_heads, n_kv_heads, head_dim
        c.intermediate, c.vocab, c.n_layers, c.group = intermediate, vocab, n_layers, group
        c.eps, c.rope_theta = eps, rope_theta
        c.mrope_sections = (ctypes.c_int * 3)(*mrope_sections)
        c.qk_norm, c.eos_id, c.pad_id = int(bool(qk_norm)), eos_id, pad_id
        c.max_len, c.slots, c.max_batch = max_len, slots, max_batch
        self.config = c
        h = _P()
        _check(lib().kmr_model_create(ctypes.byref(c), ctypes.byref(h)), "kmr_model_create")
        self._h = h

    @classmethod
    def from_config(cls, cfg, max_batch: int = 1) -> "Model":
        """From any object with the ModelConfig field names (e.g. workloads.ModelConfig)."""
        return cls(cfg.hidden, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.intermediate, cfg.vocab,
                   cfg.n_layers, cfg.group, cfg.eps, cfg.rope_theta, tuple(cfg.mrope_sections), cfg.qk_norm,
                   cfg.eos_id, cfg.pad_id, cfg.max_len, cfg.slots, max_batch)

    @property
    def handle(self) -> int:
        return self._h.value

    def close(self) -> None:
        if getattr(self, "_h", None) is not None and self._h.value:
            lib().kmr_model_destroy(self._h)
            self._h = _P()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_linear(self, layer: int, which: int, q, s, z) -> None:
        _check(lib().kmr_model_set_linear(self._h, layer, which, _ptr(q), _ptr(s), _ptr(z)), "kmr_model_set_linear")

    def set_norm(self, layer: int, which: int, w) -> None:
        _check(lib().kmr_model_set_norm(self._h, layer, which, _ptr(w)), "kmr_model_set_norm")

    def set_embedding(self, e) -> None:
        _check(lib().kmr_model_set_embedding(self._h, _ptr(e)), "kmr_model_set_embedding")

    def set_kv(self, layer: int, slot: int, length: int, k, v) -> None:
        _check(lib().kmr_model_set_kv(self._h, layer, slot, length, _ptr(k), _ptr(v)), "kmr_model_set_kv")

    def kv_pointers(self, layer: int):
        k, v = _P(), _P()
        _check(lib().kmr_model_kv_pointers(self._h, layer, ctypes.byref(k), ctypes.byref(v)), "kmr_model_kv_pointers")
        return k.value, v.value

    def reserve_prefill(self, max_tokens: int) -> None:
        """kmr_model_reserve_prefill: scratch for prefill chunks of up to max_tokens positions."""
        _check(lib().kmr_model_reserve_prefill(self._h, max_tokens), "kmr_model_reserve_prefill")

    def prefill(self, token_ids, positions, T: int, slot: int, start_pos: int, state_token, state_positions,
                state_cache_position, state_finished, logits=None, stream=None) -> None:
        """kmr_prefill on device tensors: one prompt chunk into cache row `slot` at
        [start_pos, start_pos + T); the one-row state tensors receive the first decode step's state."""
        _check(lib().kmr_prefill(self._h, _ptr(token_ids), _ptr(positions), T, slot, start_pos, _ptr(state_token),
                                 _ptr(state_positions), _ptr(state_cache_position), _ptr(state_finished),
                                 _ptr(logits), _stream(stream)), "kmr_prefill")

    def copy_row_from(self, dst_slot: int, length: int, src_row: int, src_k=None, src_v=None, src_slots: int = 0,
                      src_max_len: int = 0, stream=None) -> None:
        """kmr_model_copy_row_from: positions [0, length) of row src_row of a source cache (device
        tensors or addresses of its layer 0, laid out like the model's cache; None: the model's own
        cache) into cache row dst_slot, every layer, K and V.  Queued on `stream`."""
        _check(lib().kmr_model_copy_row_from(self._h, dst_slot, _ptr(src_k), _ptr(src_v), src_slots, src_max_len,
                                             src_row, length, _stream(stream)), "kmr_model_copy_row_from")

    def decode_step(self, token_ids, positions, cache_position, slot_ids, finished, B: int, logits=None,
                    stream=None) -> None:
        """kmr_decode_step on device tensors (state advanced in place)."""
        _check(lib().kmr_decode_step(self._h, _ptr(token_ids), _ptr(positions), _ptr(cache_position),
                                     _ptr(slot_ids), _ptr(finished), B, _ptr(logits), _stream(stream)),
               "kmr_decode_step")

    def decode_step_host(self, token_ids, positions, cache_position, slot_ids, finished, B: int, logits=None,
                         stream=None) -> None:
        """kmr_decode_step_host on host arrays (copies in, steps, copies back, synchronises)."""
        _check(lib().kmr_decode_step_host(self._h, _ptr(token_ids), _ptr(positions), _ptr(cache_position),
                                          _ptr(slot_ids), _ptr(finished), B, _ptr(logits), _stream(stream)),
               "kmr_decode_step_host")

    def sync_status(self, stream=None) -> int:
        return lib().kmr_model_sync_status(self._h, _stream(stream))

    def kernels_per_step(self, B: int) -> int:
        return lib().kmr_model_kernels_per_step(self._h, B)

    def device_bytes(self) -> dict:
        """kmr_model_device_bytes: device memory the model holds, total and split."""
        w, kv, sc = _SZ(0), _SZ(0), _SZ(0)
        total = lib().kmr_model_device_bytes(self._h, ctypes.byref(w), ctypes.byref(kv), ctypes.byref(sc))
        return {"total": int(total), "weights": int(w.value), "kv_cache": int(kv.value), "scratch": int(sc.value)}

    def set_prefill_tcgen05(self, enable: bool) -> None:
        """kmr_model_set_prefill_tcgen05: run prefill projections on the tcgen05 kernel."""
        _check(lib().kmr_model_set_prefill_tcgen05(self._h, int(bool(enable))), "kmr_model_set_prefill_tcgen05")

    def set_prefill_plan(self, nt: int = 0, ksplit: int = 0) -> None:
        """kmr_model_set_prefill_plan: force the tcgen05 tile width / K split (0, 0: planned)."""
        _check(lib().kmr_model_set_prefill_plan(self._h, int(nt), int(ksplit)), "kmr_model_set_prefill_plan")

    def set_persistent_step(self, enable: bool) -> None:
        """kmr_model_set_persistent_step: run the step's layers as one persistent kernel."""
        _check(lib().kmr_model_set_persistent_step(self._h, int(bool(enable))), "kmr_model_set_persistent_step")

    def set_smem_poison(self, enable: bool, pattern: int = 0xFFFFFFFF) -> None:
        """Precede every kernel of the step with a shared-memory fill of `pattern` (diagnostic)."""
        _check(lib().kmr_model_set_smem_poison(self._h, int(bool(enable)), pattern & 0xFFFFFFFF),
               "kmr_model_set_smem_poison")
