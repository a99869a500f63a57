"""Host step-loop driver around the C ABI (the decode loop of "kaminari — a
single-GPU Qwen3-VL inference engine, explained", §04: step until every row is
finished or max_new_tokens is reached, then trim each row at its first EOS).

Plumbing only: weights are handed to the library in canonical form (it packs
them on the device), state lives in torch device tensors, and every step is
one ``kmr_decode_step`` call.
"""
from __future__ import annotations

import collections
import dataclasses
from typing import Any, Callable, Dict, List, Optional, Sequence

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


# ------------------------------------------------------------------ continuous batching
class SlotPool:
    """Fixed pool of physical cache rows ("kaminari", §03 State model: a DecodeSlot pins a
    live row to a physical cache row; the DecodeSlotPool is sized once and never grows).
    Free rows are handed out lowest first; a released row is free again at once."""

    def __init__(self, n_slots: int):
        if n_slots <= 0:
            raise ValueError("a pool needs at least one slot")
        self.n_slots = n_slots
        self._free = list(range(n_slots))
        self._owner: Dict[int, Any] = {}

    @property
    def n_free(self) -> int:
        return len(self._free)

    @property
    def active(self) -> Dict[int, Any]:
        return dict(self._owner)

    def admit(self, key: Any) -> int:
        if not self._free:
            raise RuntimeError("slot pool is full")
        slot = self._free.pop(0)
        self._owner[slot] = key
        return slot

    def release(self, slot: int) -> Any:
        if slot not in self._owner:
            raise KeyError(f"slot {slot} is not in use")
        key = self._owner.pop(slot)
        self._free.append(slot)
        self._free.sort()
        return key


@dataclasses.dataclass
class Request:
    """One generation.  Either its prompt's KV state is already prefilled elsewhere and
    `load_kv(model, slot, stream)` writes it into the slot it gets (for instance a
    copy_row_from of a prefilled row; decoding starts from `first_token` at cache position
    `length`), or `prompt` holds the prompt's token ids and the slot is prefilled on
    admission (kmr_prefill; the prefill's greedy token is the first generated token, and
    `first_token` / `length` / `load_kv` are ignored).  Text M-RoPE ids are the cache position
    plus `rope_delta` on all three axes."""
    rid: Any
    first_token: int
    length: int
    rope_delta: int
    max_new_tokens: int
    load_kv: Optional[Callable[..., None]] = None
    prompt: Optional[Sequence[int]] = None


def generate_continuous(model: Model, requests: Sequence[Request], n_slots: int, eos_id: int = -1,
                        stream=None, device: str = "cuda") -> Dict[Any, List[int]]:
    """Continuous batching over a fixed slot pool ("kaminari", §08 ContinuousBatchScheduler:
    requests are admitted into free slots, active slots advance one token per tick, and a row
    is finalised the moment it finishes instead of waiting for the whole batch).

    Batch row b always uses cache row b, so every tick is the same captured step (B = n_slots);
    an empty row is a finished row, which reads and writes no KV.  Before each tick waiting
    requests take the free slots (their KV state loaded, their row state written); after it,
    rows that emitted EOS, hit the cache cap or spent max_new_tokens are finalised (trimmed
    at the first EOS) and their slots released.  Returns rid -> generated tokens.  `stream`
    (a torch stream or None) is made current for the whole loop, so the row-state writes,
    the steps and the reads are ordered on it."""
    import contextlib
    import torch
    for req in requests:
        if req.prompt is not None and len(req.prompt) == 0:
            raise ValueError(f"request {req.rid!r}: empty prompt")
        if req.prompt is None and req.load_kv is None and req.max_new_tokens > 0:
            raise ValueError(f"request {req.rid!r}: needs a prompt or a load_kv callback")
    with torch.cuda.stream(stream) if stream is not None else contextlib.nullcontext():
        return _continuous(model, requests, n_slots, eos_id, stream, device)


def _continuous(model, requests, n_slots, eos_id, stream, device):
    import torch
    B = n_slots
    pool = SlotPool(n_slots)
    tok = torch.zeros(B, dtype=torch.int32, device=device)
    pos = torch.zeros((3, B), dtype=torch.int32, device=device)
    cpos = torch.zeros(B, dtype=torch.int32, device=device)
    slots = torch.arange(B, dtype=torch.int32, device=device)
    fin = torch.ones(B, dtype=torch.uint8, device=device)
    queue = collections.deque(requests)
    live: Dict[int, List[Any]] = {}               # row -> [request, produced tokens]
    out: Dict[Any, List[int]] = {}

    def finalize(row, req, got):
        if eos_id >= 0 and eos_id in got:
            got = got[:got.index(eos_id) + 1]
        out[req.rid] = got
        fin[row] = 1
        pool.release(row)

    while queue or live:
        while queue and pool.n_free:
            req = queue.popleft()
            if req.max_new_tokens <= 0:
                out[req.rid] = []
                continue
            row = pool.admit(req.rid)
            if req.prompt is not None:
                # prefill the prompt into the slot; the row's state becomes the first decode step's
                T = len(req.prompt)
                ptok = torch.tensor(np.asarray(req.prompt, np.int32), device=device)
                ppos = (torch.arange(T, dtype=torch.int32, device=device) + req.rope_delta).repeat(3, 1).contiguous()
                spos = torch.empty(3, dtype=torch.int32, device=device)
                model.reserve_prefill(T)
                model.prefill(ptok, ppos, T, row, 0, tok[row:row + 1], spos, cpos[row:row + 1], fin[row:row + 1],
                              None, stream)
                pos[:, row] = spos
                first = int(tok[row].item())
                if bool(fin[row].item()) or req.max_new_tokens == 1:
                    finalize(row, req, [first])
                    continue
                live[row] = [req, [first]]
                continue
            req.load_kv(model, row, stream)
            p = req.length + req.rope_delta
            tok[row] = req.first_token
            pos[:, row] = p
            cpos[row] = req.length
            fin[row] = 0
            live[row] = [req, []]
        if not live:
            continue
        model.decode_step(tok, pos, cpos, slots, fin, B, None, stream)
        t_h = tok.cpu().numpy()
        f_h = fin.cpu().numpy()
        for row in sorted(live):
            req, got = live[row]
            got.append(int(t_h[row]))
            if f_h[row] or len(got) >= req.max_new_tokens:
                del live[row]
                finalize(row, req, got)
    return out
