"""Host step-loop driver around the C ABI (the decode loop of "kaminari — a
single-GPU Qwen3-VL inference engine, explained", §04: step until every row is
finished or max_new_tokens is reached, then trim each row at its first EOS).

Plumbing only: weights are handed to the library in canonical form (it packs
them on the device), state lives in torch device tensors, and every step is
one ``kmr_decode_step`` call.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence

import numpy as np

from . import (KMR_N_INPUT, KMR_N_K, KMR_N_POST, KMR_N_Q, KMR_W_DOWN, KMR_W_GATE_UP, KMR_W_O, KMR_W_QKV, Model)

_LINEARS = {"qkv": KMR_W_QKV, "o": KMR_W_O, "gate_up": KMR_W_GATE_UP, "down": KMR_W_DOWN}
_NORMS = {"in": KMR_N_INPUT, "post": KMR_N_POST, "q": KMR_N_Q, "k": KMR_N_K}


def load_weights(model: Model, source, n_layers: int, qk_norm: bool = True) -> None:
    """Load every layer from `source`, an object with linear(layer, name) -> (q, s, z),
    norm(layer, name) -> bf16 bits and embedding() -> bf16 bits (canonical arrays)."""
    for l in range(n_layers):
        for name, which in _LINEARS.items():
            q, s, z = source.linear(l, name)
            model.set_linear(l, which, np.ascontiguousarray(q), np.ascontiguousarray(s), np.ascontiguousarray(z))
        for name, which in _NORMS.items():
            if name in ("q", "k") and not qk_norm:
                continue
            model.set_norm(l, which, np.ascontiguousarray(source.norm(l, name)))
    model.set_norm(-1, KMR_N_INPUT, np.ascontiguousarray(source.norm(-1, "final")))
    model.set_embedding(np.ascontiguousarray(source.embedding()))


def load_kv(model: Model, source, n_layers: int, slot: int, length: int, fill: int = 0) -> None:
    """Write positions [0, length) of every layer's cache row `slot` from source.kv_prefill."""
    for l in range(n_layers):
        k = source.kv_prefill(l, slot, length, "k", fill)[:, :length, :]
        v = source.kv_prefill(l, slot, length, "v", fill)[:, :length, :]
        model.set_kv(l, slot, length, np.ascontiguousarray(k), np.ascontiguousarray(v))


class DeviceState:
    """Step state of B rows as device tensors: token ids (B), positions (3, B),
    cache_position (B), slot ids (B), finished (B)."""

    def __init__(self, tokens, positions, cache_position, slot_ids, finished=None, device="cuda"):
        import torch
        B = len(tokens)
        self.B = B
        self.tokens = torch.tensor(np.asarray(tokens, np.int32), device=device)
        self.positions = torch.tensor(np.asarray(positions, np.int32).reshape(3, B), device=device)
        self.cache_position = torch.tensor(np.asarray(cache_position, np.int32), device=device)
        self.slot_ids = torch.tensor(np.asarray(slot_ids, np.int32), device=device)
        fin = np.zeros(B, np.uint8) if finished is None else np.asarray(finished, np.uint8)
        self.finished = torch.tensor(fin, device=device)

    def step(self, model: Model, logits=None, stream=None) -> None:
        model.decode_step(self.tokens, self.positions, self.cache_position, self.slot_ids, self.finished, self.B,
                          logits, stream)


def generate(model: Model, state: DeviceState, max_new_tokens: int, eos_id: int = -1,
             finish_at: Optional[Dict[int, int]] = None) -> List[List[int]]:
    """Greedy decode up to max_new_tokens; rows stop at EOS (or are marked finished by
    `finish_at[row] = step`, the scheduler retiring a row); returns each row's tokens
    trimmed at its first EOS."""
    import torch
    hist = torch.empty((max_new_tokens, state.B), dtype=torch.int32, device=state.tokens.device)
    steps = 0
    for t in range(max_new_tokens):
        if finish_at:
            for row, at in finish_at.items():
                if at == t:
                    state.finished[row] = 1
        state.step(model)
        hist[t].copy_(state.tokens)
        steps += 1
        if t % 32 == 31 and bool(state.finished.all()):
            break
    out = hist[:steps].t().cpu().numpy()
    fin_rows = []
    for b in range(state.B):
        row = []
        for tok in out[b]:
            row.append(int(tok))
            if eos_id >= 0 and tok == eos_id:
                break
        fin_rows.append(row)
    return fin_rows
