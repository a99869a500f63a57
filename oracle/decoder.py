"""Plain CPU oracle of the int4 weight-only, group-wise greedy decode step.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, links or
executes this file; only tests, the smoke check and the benchmark's CPU
baseline do.  It shares no code with the CUDA path: it reads the canonical
(unpacked) synthetic inputs from ``workloads`` and computes everything in
numpy float64 (the KV cache is bf16 storage by definition, so values written
to it are rounded to bf16 here).

Sources (page titles and sections):
  [K] "kaminari — a single-GPU Qwen3-VL inference engine, explained":
      §03 Architecture overview (TextModel, DecoderLayer, TextAttention with
      fused QKV, MLP, Mrope, StaticKVCache; Live state with 3-D M-RoPE
      positions, cache_position and per-row finished flags; the cache mutates
      in place), §04 Request lifecycle / decode (one-token step on token ids
      (B,1), positions (3,B,1), cache_position; greedy argmax on device; EOS
      flips finished; finished rows padded), §07 int4 sidecar quantization
      (decoder attention/MLP linears weight-only int4; embeddings, lm_head and
      norms stay bf16).
  [G] "The Ghost in the Batch: How vLLM Silently Switches Algorithms":
      "What Attention Does" (softmax(Q K^T / sqrt(d)) V) and the LSE-weighted
      merge of partial attention results.
Readings where the pages are silent (each also listed in the design notes):
  group 128 along K with w = (q - 8) * s + z, s and z bf16 per (row, group);
  RMSNorm eps 1e-6; per-head q/k RMSNorm before the rotary embedding;
  contiguous 3-section M-RoPE, NeoX rotate-half pairing (i, i + d/2),
  inv_freq_i = theta^(-2i/d); fused rows qkv = [q; k; v], gate_up = [gate; up];
  query head i reads KV head i // (n_q / n_kv); argmax ties go to the lowest
  index and NaN never wins; a finished row writes and reads no KV, emits pad
  and does not advance; a row that has written position max_len - 1 is
  finished (length cap).
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence

import numpy as np

from workloads import ModelConfig, SyntheticModel, Workload

__all__ = [
    "bf16_to_f64", "f64_to_bf16_bits", "dequant_int4", "rmsnorm", "mrope_axis_of_freq",
    "mrope_inv_freq", "mrope", "decode_attention", "merge_partials", "attention_with_lse", "cascade_attention",
    "silu", "argmax_lowest",
    "OracleDecoder", "StepResult",
]


# --------------------------------------------------------------------------- storage formats
def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Value of bf16 bit patterns (the top 16 bits of an IEEE float32)."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round to bf16: 8 significant bits, nearest, ties to even (normal range)."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                          # x = m * 2**e, 0.5 <= |m| < 1
    r = np.ldexp(np.rint(m * 256.0), e - 8)     # keep 8 significant bits
    return (r.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


# --------------------------------------------------------------------------- int4 linear [K §07]
def dequant_int4(q: np.ndarray, s_bits: np.ndarray, z_bits: np.ndarray, group: int) -> np.ndarray:
    """Dense weight W[n, k] = (q[n, k] - 8) * s[n, k // group] + z[n, k // group]."""
    q = np.asarray(q)
    N, K = q.shape
    assert K % group == 0 and s_bits.shape == (N, K // group) == z_bits.shape
    s = np.repeat(bf16_to_f64(s_bits), group, axis=1)
    z = np.repeat(bf16_to_f64(z_bits), group, axis=1)
    return (q.astype(np.float64) - 8.0) * s + z


def int4_linear(x: np.ndarray, q, s_bits, z_bits, group: int) -> np.ndarray:
    """y[m, n] = sum_k x[m, k] * W[n, k] with W dequantised as above."""
    return np.asarray(x, dtype=np.float64) @ dequant_int4(q, s_bits, z_bits, group).T


# --------------------------------------------------------------------------- RMSNorm [K §03, §07]
def rmsnorm(x: np.ndarray, w_bits: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2 over the last axis) + eps) * w."""
    x = np.asarray(x, dtype=np.float64)
    r = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return x * r * bf16_to_f64(w_bits)


# --------------------------------------------------------------------------- M-RoPE [K §03, §04]
def mrope_axis_of_freq(head_dim: int, sections: Sequence[int]) -> np.ndarray:
    """Position axis (0 = T, 1 = H, 2 = W) that drives each of the head_dim/2 frequencies.

    Sections are contiguous: the first sections[0] frequencies follow T, the
    next sections[1] follow H, the last sections[2] follow W.
    """
    assert sum(sections) == head_dim // 2
    return np.repeat(np.arange(3), sections)


def mrope_inv_freq(head_dim: int, theta: float) -> np.ndarray:
    i = np.arange(head_dim // 2, dtype=np.float64)
    return theta ** (-2.0 * i / head_dim)


def mrope(x: np.ndarray, pos3: Sequence[int], head_dim: int, theta: float,
          sections: Sequence[int]) -> np.ndarray:
    """Rotate every head of x[..., head_dim] by the 3-section M-RoPE angles.

    Frequency i turns the pair (x[i], x[i + d/2]) by pos[axis(i)] * inv_freq[i].
    """
    x = np.asarray(x, dtype=np.float64)
    half = head_dim // 2
    pos = np.asarray(pos3, dtype=np.float64)[mrope_axis_of_freq(head_dim, sections)]
    ang = pos * mrope_inv_freq(head_dim, theta)
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


# --------------------------------------------------------------------------- attention [G]
def decode_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray) -> np.ndarray:
    """GQA decode attention of one token.

    q [n_q, d]; K, V [n_kv, T, d] hold the T attended positions.  Query head i
    reads KV head i // (n_q / n_kv); out_i = softmax(q_i K^T / sqrt(d)) V.
    """
    n_q, d = q.shape
    n_kv = K.shape[0]
    rep = n_q // n_kv
    out = np.empty((n_q, d), dtype=np.float64)
    for i in range(n_q):
        h = i // rep
        sc = K[h] @ q[i] / np.sqrt(d)
        p = np.exp(sc - sc.max())
        p /= p.sum()
        out[i] = p @ V[h]
    return out


def merge_partials(outs: Sequence[np.ndarray], lses: Sequence[np.ndarray]) -> np.ndarray:
    """LSE-weighted merge of normalised partial attention outputs [G].

    Weights exp(lse_j - max lse) per part; output = sum_j w_j o_j / sum_j w_j.
    """
    lse = np.stack([np.asarray(l, dtype=np.float64) for l in lses])
    m = lse.max(axis=0)
    w = np.exp(lse - m)
    o = np.stack([np.asarray(o, dtype=np.float64) for o in outs])
    return (w[..., None] * o).sum(axis=0) / w.sum(axis=0)[..., None]


def attention_with_lse(q: np.ndarray, K: np.ndarray, V: np.ndarray):
    """Decode attention of one token over T positions returning, per query head, the
    normalised output and the log-sum-exp of its scaled scores [G] (the statistic the
    LSE-weighted merge needs).  q [n_q, d]; K, V [n_kv, T, d], T >= 1."""
    n_q, d = q.shape
    rep = n_q // K.shape[0]
    out = np.empty((n_q, d), dtype=np.float64)
    lse = np.empty(n_q, dtype=np.float64)
    for i in range(n_q):
        sc = K[i // rep] @ q[i] / np.sqrt(d)
        mx = sc.max()
        e = np.exp(sc - mx)
        lse[i] = mx + np.log(e.sum())
        out[i] = (e / e.sum()) @ V[i // rep]
    return out, lse


def cascade_attention(q: np.ndarray, K_prefix: np.ndarray, V_prefix: np.ndarray, K_suffix: np.ndarray,
                      V_suffix: np.ndarray) -> np.ndarray:
    """Shared-prefix decode attention in the pages' three steps [G, The Optimization That
    Changes Everything]: attention over the shared prefix (output and LSE), attention over
    the row's own suffix (output and LSE), then the LSE-weighted merge.  K_prefix, V_prefix
    [n_kv, P, d] (P may be 0: the suffix alone); K_suffix, V_suffix [n_kv, T, d], T >= 1."""
    suf_out, suf_lse = attention_with_lse(q, K_suffix, V_suffix)
    if K_prefix.shape[1] == 0:
        return suf_out
    pre_out, pre_lse = attention_with_lse(q, K_prefix, V_prefix)
    return merge_partials([pre_out, suf_out], [pre_lse, suf_lse])


# --------------------------------------------------------------------------- MLP, head, argmax
def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def argmax_lowest(logits: np.ndarray) -> int:
    """Index of the largest finite-or-inf value; lowest index on ties; NaN never wins."""
    v = np.where(np.isnan(logits), -np.inf, logits)
    return int(np.argmax(v))     # numpy returns the first maximal index


# --------------------------------------------------------------------------- the decode step
@dataclasses.dataclass
class StepResult:
    logits: np.ndarray        # [B, V] float64 (NaN for rows finished before the step)
    next_ids: np.ndarray      # [B] int32 token emitted this step (pad for finished rows)
    positions: np.ndarray     # [3, B] int32 after the step
    cache_position: np.ndarray  # [B] int32 after the step
    finished: np.ndarray      # [B] uint8 after the step


class OracleDecoder:
    """The decoder of one synthetic model plus its static bf16 KV cache.

    KV cache layout: K[layer][slot, kv_head, position, dim] as bf16 bits
    (the static, slot-addressable cache of [K §03]); the step writes the new
    token's K and V in place at cache_position.
    """

    def __init__(self, cfg: ModelConfig, seed: int = 0, layers: Optional[int] = None,
                 head_rows: Optional[slice] = None, syn: Optional[SyntheticModel] = None):
        self.cfg = cfg
        self.syn = syn if syn is not None else SyntheticModel(cfg, seed)
        self.n_layers = cfg.n_layers if layers is None else layers
        self.head_rows = head_rows      # restrict the LM head to a vocab slice (bounded CPU samples)
        shape = (cfg.slots, cfg.n_kv_heads, cfg.max_len, cfg.head_dim)
        self.K = [np.zeros(shape, np.uint16) for _ in range(self.n_layers)]
        self.V = [np.zeros(shape, np.uint16) for _ in range(self.n_layers)]

    def prefill_cache(self, slot: int, length: int, fill: int = 0):
        for l in range(self.n_layers):
            self.K[l][slot] = self.syn.kv_prefill(l, slot, length, "k", fill)
            self.V[l][slot] = self.syn.kv_prefill(l, slot, length, "v", fill)

    @classmethod
    def for_workload(cls, wl: Workload, fill: int = 0, **kw) -> "OracleDecoder":
        o = cls(wl.cfg, wl.seed, **kw)
        for b in range(wl.batch):
            o.prefill_cache(wl.slot_ids[b], wl.prefill[b], fill)
        return o

    # -- one layer over the active rows -------------------------------------------------
    def _layer(self, l: int, x: np.ndarray, pos: np.ndarray, cpos: np.ndarray,
               slots: np.ndarray, active: np.ndarray) -> np.ndarray:
        cfg, syn = self.cfg, self.syn
        g, d = cfg.group, cfg.head_dim
        qd, kvd = cfg.q_dim, cfg.kv_dim
        h = rmsnorm(x, syn.norm(l, "in"), cfg.eps)
        qkv = int4_linear(h, *syn.linear(l, "qkv"), g)
        o = np.zeros((x.shape[0], qd))
        for b in np.nonzero(active)[0]:
            q = qkv[b, :qd].reshape(cfg.n_q_heads, d)
            k = qkv[b, qd:qd + kvd].reshape(cfg.n_kv_heads, d)
            v = qkv[b, qd + kvd:].reshape(cfg.n_kv_heads, d)
            if cfg.qk_norm:
                q = rmsnorm(q, syn.norm(l, "q"), cfg.eps)
                k = rmsnorm(k, syn.norm(l, "k"), cfg.eps)
            q = mrope(q, pos[:, b], d, cfg.rope_theta, cfg.mrope_sections)
            k = mrope(k, pos[:, b], d, cfg.rope_theta, cfg.mrope_sections)
            t = int(cpos[b])
            self.K[l][slots[b], :, t, :] = f64_to_bf16_bits(k)
            self.V[l][slots[b], :, t, :] = f64_to_bf16_bits(v)
            Kf = bf16_to_f64(self.K[l][slots[b], :, :t + 1, :])
            Vf = bf16_to_f64(self.V[l][slots[b], :, :t + 1, :])
            o[b] = decode_attention(q, Kf, Vf).reshape(-1)
        x = x + int4_linear(o, *syn.linear(l, "o"), g)
        h = rmsnorm(x, syn.norm(l, "post"), cfg.eps)
        gu = int4_linear(h, *syn.linear(l, "gate_up"), g)
        a = silu(gu[:, :cfg.intermediate]) * gu[:, cfg.intermediate:]
        return x + int4_linear(a, *syn.linear(l, "down"), g)

    def hidden(self, tokens, positions, cache_position, slot_ids, finished) -> np.ndarray:
        """Final-norm input x after all layers, [B, hidden]; advances nothing."""
        cfg = self.cfg
        tokens = np.asarray(tokens).reshape(-1)
        B = tokens.shape[0]
        pos = np.asarray(positions).reshape(3, B)
        cpos = np.asarray(cache_position).reshape(B)
        slots = np.asarray(slot_ids).reshape(B)
        active = np.asarray(finished).reshape(B) == 0
        for b in np.nonzero(active)[0]:
            if not (0 <= cpos[b] < cfg.max_len):
                raise ValueError(f"row {b}: cache_position {cpos[b]} outside [0, {cfg.max_len})")
        x = bf16_to_f64(self.syn.embedding()[tokens])
        for l in range(self.n_layers):
            x = self._layer(l, x, pos, cpos, slots, active)
        return x

    def logits_of(self, x: np.ndarray, chunk: int = 8192) -> np.ndarray:
        cfg = self.cfg
        h = rmsnorm(x, self.syn.norm(-1, "final"), cfg.eps)
        E = self.syn.embedding()
        rows = range(cfg.vocab) if self.head_rows is None else range(cfg.vocab)[self.head_rows]
        lo, hi = rows.start, rows.stop
        out = np.full((x.shape[0], cfg.vocab), np.nan)
        for c0 in range(lo, hi, chunk):
            c1 = min(hi, c0 + chunk)
            out[:, c0:c1] = h @ bf16_to_f64(E[c0:c1]).T
        return out

    def prefill(self, tokens, positions, slot: int, start: int) -> "StepResult":
        """Prefill [K §04] by its definition: the decode step applied to each prompt token in
        order — token i at cache position start + i of row `slot`, attending 0..start + i.
        Returns the last token's step: its logits, the greedy next token and the advanced
        state (positions + 1, cache position start + T)."""
        positions = np.asarray(positions, dtype=np.int64).reshape(3, -1)
        res = None
        for i, tok in enumerate(np.asarray(tokens).reshape(-1)):
            res = self.step([int(tok)], positions[:, i:i + 1], [start + i], [slot], [0])
        return res

    def step(self, tokens, positions, cache_position, slot_ids, finished) -> StepResult:
        """One greedy decode step [K §04]: logits, argmax, finished/pad masking, advance."""
        cfg = self.cfg
        tokens = np.asarray(tokens, dtype=np.int64).reshape(-1)
        B = tokens.shape[0]
        fin0 = np.asarray(finished, dtype=np.uint8).reshape(B).copy()
        pos = np.asarray(positions, dtype=np.int64).reshape(3, B).copy()
        cpos = np.asarray(cache_position, dtype=np.int64).reshape(B).copy()
        logits = self.logits_of(self.hidden(tokens, pos, cpos, slot_ids, fin0))
        nxt = np.full(B, cfg.pad_id, dtype=np.int64)
        fin = fin0.copy()
        for b in range(B):
            if fin0[b]:
                logits[b] = np.nan
                continue
            nxt[b] = argmax_lowest(logits[b])
            cpos[b] += 1
            pos[:, b] += 1
            if nxt[b] == cfg.eos_id or cpos[b] >= cfg.max_len:
                fin[b] = 1
        return StepResult(logits, nxt.astype(np.int32), pos.astype(np.int32),
                          cpos.astype(np.int32), fin)


def initial_state(wl: Workload):
    """The workload's first-step state (see workloads.initial_state)."""
    from workloads import initial_state as _init
    return _init(wl)
