"""Shared helpers of the GPU parity tests (imported by tests only)."""
import os

import numpy as np
import pytest

import int4_weight_only_group_gb300 as kmr
from int4_weight_only_group_gb300 import driver

REL_L2_TOL = 1e-2          # projection / attention / logits tolerance (relative L2 vs the fp64 oracle)
GAP_RULE = 1e-2            # greedy tokens must agree where top-2 gap > GAP_RULE * |max logit|


def require_gpu():
    torch = pytest.importorskip("torch")
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    if not os.path.exists(kmr.library_path()):
        from int4_weight_only_group_gb300.build import build
        build()
    kmr.lib()
    return torch


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def greedy_agrees(gpu_id: int, ref_logits: np.ndarray) -> bool:
    """True if gpu_id is the oracle's argmax, or the oracle's top-2 gap is within the gap rule
    and gpu_id is one of the tied-within-gap candidates."""
    v = np.where(np.isnan(ref_logits), -np.inf, ref_logits)
    top = int(np.argmax(v))
    if gpu_id == top:
        return True
    gap = v[top] - v[gpu_id]
    return gap <= GAP_RULE * abs(v[top])


def build_model(wl, fill: int = 0, max_batch: int = None, layers: int = None):
    cfg = wl.cfg
    from workloads import SyntheticModel
    syn = SyntheticModel(cfg, wl.seed)
    m = kmr.Model.from_config(cfg, max_batch=max_batch or wl.batch)
    driver.load_weights(m, syn, cfg.n_layers, cfg.qk_norm)
    for b in range(wl.batch):
        # with a non-zero fill the whole row is written, so unfilled positions hold `fill` on the GPU too
        length = wl.prefill[b] if fill == 0 else cfg.max_len
        for l in range(cfg.n_layers):
            k = syn.kv_prefill(l, wl.slot_ids[b], wl.prefill[b], "k", fill)[:, :length]
            v = syn.kv_prefill(l, wl.slot_ids[b], wl.prefill[b], "v", fill)[:, :length]
            m.set_kv(l, wl.slot_ids[b], length, np.ascontiguousarray(k), np.ascontiguousarray(v))
    return m, syn


def d2h_bytes(ptr: int, nbytes: int) -> np.ndarray:
    """Copy nbytes of device memory at a raw address to a host uint8 array."""
    import ctypes
    rt = ctypes.CDLL("libcudart.so.13")
    out = np.empty(nbytes, np.uint8)
    rc = rt.cudaMemcpy(ctypes.c_void_p(out.ctypes.data), ctypes.c_void_p(ptr), ctypes.c_size_t(nbytes), 2)
    assert rc == 0, rc
    return out
