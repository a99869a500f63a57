"""Seeded synthetic inputs for the int4 decode step.

This module is shared by the CPU oracle (``oracle/``) and by the CUDA path's
tests and benchmark.  It holds shapes, seeds and random-number draws only:
nothing here computes any part of the decode step.  Every tensor is drawn from
its own ``numpy.random.Generator(PCG64(SeedSequence([seed, tag])))`` stream, so
one layer can be regenerated without drawing every tensor before it.

Distributions (the workload recipe):
  * int4 codes q ~ U{0..15}, scales s ~ U(0.002, 0.02), zeros z ~ N(0, 0.005),
    group 128 along K, dequantised as w = (q - 8) * s + z;
  * tied embedding / LM head ~ N(0, 0.02), stored bf16;
  * RMSNorm weights (input, post-attention, final, per-head q/k) 1 + N(0, 0.1);
  * prefilled KV cache entries ~ N(0, 1), stored bf16.
Model dimensions follow a Qwen3-style 2B text decoder (hidden 2048, 16 query /
8 key-value heads of 128, intermediate 6144, vocab 151936, 28 layers) and a
tiny 2-layer variant of the same structure.
"""
from __future__ import annotations

import dataclasses
import zlib
from typing import Dict, List, Optional, Tuple

import numpy as np

__all__ = [
    "ModelConfig", "tiny_config", "layer2b_config", "full2b_config",
    "f32_to_bf16_bits", "bf16_bits_to_f32", "SyntheticModel", "Workload",
    "tiny_workload", "layer2b_workload", "full2b_b1_workload", "full2b_b4_workload",
    "BF16_NAN", "initial_state",
]

BF16_NAN = np.uint16(0x7FC0)


@dataclasses.dataclass(frozen=True)
class ModelConfig:
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    intermediate: int
    vocab: int
    n_layers: int
    group: int = 128
    eps: float = 1e-6
    rope_theta: float = 1e6
    mrope_sections: Tuple[int, int, int] = (16, 24, 24)
    qk_norm: bool = True
    eos_id: int = -1          # -1: no token ever ends a row
    pad_id: int = 0
    max_len: int = 1024       # static cache length per slot (S)
    slots: int = 1            # physical cache rows

    @property
    def q_dim(self) -> int:
        return self.n_q_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    @property
    def qkv_rows(self) -> int:
        return self.q_dim + 2 * self.kv_dim

    def linear_shapes(self) -> Dict[str, Tuple[int, int]]:
        """(N, K) of each quantised linear: rows = outputs, cols = inputs."""
        return {
            "qkv": (self.qkv_rows, self.hidden),
            "o": (self.hidden, self.q_dim),
            "gate_up": (2 * self.intermediate, self.hidden),
            "down": (self.hidden, self.intermediate),
        }


def tiny_config(**kw) -> ModelConfig:
    base = dict(hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64, intermediate=768,
                vocab=1024, n_layers=2, mrope_sections=(8, 12, 12), eos_id=1023,
                max_len=128, slots=1)
    base.update(kw)
    return ModelConfig(**base)


def layer2b_config(**kw) -> ModelConfig:
    base = dict(hidden=2048, n_q_heads=16, n_kv_heads=8, head_dim=128, intermediate=6144,
                vocab=151936, n_layers=1, max_len=1024, slots=1)
    base.update(kw)
    return ModelConfig(**base)


def full2b_config(**kw) -> ModelConfig:
    base = dict(hidden=2048, n_q_heads=16, n_kv_heads=8, head_dim=128, intermediate=6144,
                vocab=151936, n_layers=28, max_len=1024, slots=1)
    base.update(kw)
    return ModelConfig(**base)


# --------------------------------------------------------------------------- bf16 storage
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    nan = np.isnan(np.ascontiguousarray(x, dtype=np.float32))
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    if nan.any():
        r[nan] = BF16_NAN
    return r


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------- generators
def _rng(seed: int, tag: str) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, zlib.crc32(tag.encode())])))


class SyntheticModel:
    """Lazily drawn weights of one seeded synthetic model.

    int4 linears come back in the canonical unpacked form: q uint8 [N, K] with
    values 0..15 (row = output feature, column = input feature), and bf16 bit
    patterns s, z of shape [N, K / group].  Fused matrices are row
    concatenations: qkv = [q; k; v], gate_up = [gate; up].
    """

    def __init__(self, cfg: ModelConfig, seed: int = 0, memo: bool = False):
        self.cfg = cfg
        self.seed = seed
        self.memo = memo              # keep drawn linears (several consumers of one model)
        self._cache: Dict[str, object] = {}

    def linear(self, layer: int, name: str):
        key = f"L{layer}.{name}"
        if self.memo and key in self._cache:
            return self._cache[key]
        out = self._draw_linear(key, name)
        if self.memo:
            self._cache[key] = out
        return out

    def _draw_linear(self, key: str, name: str):
        N, K = self.cfg.linear_shapes()[name]
        g = self.cfg.group
        assert K % g == 0
        q = _rng(self.seed, key + ".q").integers(0, 16, size=(N, K), dtype=np.uint8)
        s = _rng(self.seed, key + ".s").uniform(0.002, 0.02, size=(N, K // g)).astype(np.float32)
        z = (_rng(self.seed, key + ".z").standard_normal(size=(N, K // g)) * 0.005).astype(np.float32)
        return q, f32_to_bf16_bits(s), f32_to_bf16_bits(z)

    def norm(self, layer: int, name: str) -> np.ndarray:
        """bf16 bits of an RMSNorm weight: name in {in, post, q, k}; layer -1 = final norm."""
        n = self.cfg.head_dim if name in ("q", "k") else self.cfg.hidden
        w = 1.0 + 0.1 * _rng(self.seed, f"L{layer}.norm_{name}").standard_normal(size=n)
        return f32_to_bf16_bits(w.astype(np.float32))

    def embedding(self) -> np.ndarray:
        """bf16 bits [vocab, hidden] of the tied embedding / LM head."""
        if "embed" not in self._cache:
            cfg = self.cfg
            e = _rng(self.seed, "embed").standard_normal(size=(cfg.vocab, cfg.hidden), dtype=np.float32)
            e *= np.float32(0.02)
            self._cache["embed"] = f32_to_bf16_bits(e)
        return self._cache["embed"]

    def kv_prefill(self, layer: int, slot: int, length: int, which: str,
                   fill: Optional[int] = 0) -> np.ndarray:
        """bf16 bits [n_kv_heads, max_len, head_dim] of one slot's K or V cache row.

        Positions [0, length) hold N(0, 1) draws; the rest hold `fill` (a bf16
        bit pattern; BF16_NAN lets tests prove unfilled positions are never read).
        """
        cfg = self.cfg
        out = np.full((cfg.n_kv_heads, cfg.max_len, cfg.head_dim), fill, dtype=np.uint16)
        if length > 0:
            r = _rng(self.seed, f"L{layer}.slot{slot}.{which}")
            out[:, :length, :] = f32_to_bf16_bits(
                r.standard_normal(size=(cfg.n_kv_heads, length, cfg.head_dim), dtype=np.float32))
        return out


# --------------------------------------------------------------------------- workloads
@dataclasses.dataclass
class Workload:
    """One decode workload: model, batch rows, their cache rows and schedules."""
    name: str
    cfg: ModelConfig
    seed: int
    batch: int
    prefill: List[int]                 # filled positions per batch row
    rope_delta: List[int]              # per-row M-RoPE delta (positions = cache_position + delta)
    slot_ids: List[int]                # physical cache row per batch row
    first_tokens: List[int]            # input token per row at the first decode step
    steps: int                         # greedy decode steps
    finish_at: Dict[int, int] = dataclasses.field(default_factory=dict)  # row -> step it is marked finished

    def describe(self) -> dict:
        c = self.cfg
        return {"workload": self.name, "layers": c.n_layers, "hidden": c.hidden,
                "heads": f"{c.n_q_heads}q/{c.n_kv_heads}kv x {c.head_dim}",
                "intermediate": c.intermediate, "vocab": c.vocab, "group": c.group,
                "batch": self.batch, "kv_max_len": c.max_len, "prefill": list(self.prefill),
                "steps": self.steps}


def _first_tokens(seed: int, batch: int, vocab: int, eos: int) -> List[int]:
    r = _rng(seed, "first_tokens")
    toks = r.integers(1, vocab - 1, size=batch)
    return [int(t) if t != eos else 1 for t in toks]


def tiny_workload(seed: int = 0) -> Workload:
    cfg = tiny_config()
    return Workload("tiny decode (2 layers, hidden 256, 4q/2kv x 64, vocab 1024)", cfg, seed,
                    batch=1, prefill=[32], rope_delta=[0], slot_ids=[0],
                    first_tokens=_first_tokens(seed, 1, cfg.vocab, cfg.eos_id), steps=16)


def layer2b_workload(seed: int = 0) -> Workload:
    cfg = layer2b_config()
    return Workload("single 2B-shaped layer (hidden 2048, 16q/8kv x 128, 600 cached)", cfg, seed,
                    batch=1, prefill=[600], rope_delta=[-40], slot_ids=[0],
                    first_tokens=_first_tokens(seed, 1, cfg.vocab, cfg.eos_id), steps=1)


def full2b_b1_workload(seed: int = 0) -> Workload:
    cfg = full2b_config()
    return Workload("28-layer 2B-shaped decoder, batch 1, 512 prefilled, 256 steps", cfg, seed,
                    batch=1, prefill=[512], rope_delta=[0], slot_ids=[0],
                    first_tokens=_first_tokens(seed, 1, cfg.vocab, cfg.eos_id), steps=256)


def full2b_b4_workload(seed: int = 0) -> Workload:
    cfg = full2b_config(slots=4)
    r = _rng(seed, "rope_delta_b4")
    deltas = [int(v) for v in r.integers(-60, 1, size=4)]
    return Workload("28-layer 2B-shaped decoder, batch 4 continuous slots (300/512/700/900 prefilled), 128 steps",
                    cfg, seed, batch=4, prefill=[300, 512, 700, 900], rope_delta=deltas,
                    slot_ids=[0, 1, 2, 3], first_tokens=_first_tokens(seed, 4, cfg.vocab, cfg.eos_id),
                    steps=128, finish_at={2: 64})


def full2b_b16_workload(seed: int = 0) -> Workload:
    """Sixteen continuous slots of the 28-layer model (prefilled lengths spread over 256..896,
    deltas in [-60, 0], 128 steps, no row finishes early): the batch 8-16 case."""
    cfg = full2b_config(slots=16)
    r = _rng(seed, "b16")
    prefill = [int(v) for v in r.integers(256, 897, size=16)]
    deltas = [int(v) for v in r.integers(-60, 1, size=16)]
    return Workload("28-layer 2B-shaped decoder, batch 16 continuous slots (256..896 prefilled), 128 steps",
                    cfg, seed, batch=16, prefill=prefill, rope_delta=deltas, slot_ids=list(range(16)),
                    first_tokens=_first_tokens(seed, 16, cfg.vocab, cfg.eos_id), steps=128)


def initial_state(wl: Workload):
    """(tokens [B], positions [3, B], cache_position [B], slot_ids [B], finished [B]) at the
    first decode step: the new token is written at the prefilled length and rotated at
    that length plus the row's M-RoPE delta on all three axes."""
    B = wl.batch
    cpos = np.array(wl.prefill, dtype=np.int32)
    pos = np.tile(cpos + np.array(wl.rope_delta, dtype=np.int32), (3, 1)).astype(np.int32)
    return (np.array(wl.first_tokens, dtype=np.int32), pos, cpos,
            np.array(wl.slot_ids, dtype=np.int32), np.zeros(B, dtype=np.uint8))
