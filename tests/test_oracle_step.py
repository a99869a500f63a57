"""Invariants and special cases of the oracle's whole decode step (tiny model)."""
import numpy as np
import pytest

from oracle import decoder as od
from workloads import BF16_NAN, tiny_config, tiny_workload


def _state(B=1, cpos=32, delta=0, tok=5, slot=0):
    return (np.full(B, tok, np.int32), np.full((3, B), cpos + delta, np.int32),
            np.full(B, cpos, np.int32), np.full(B, slot, np.int32), np.zeros(B, np.uint8))


def test_zero_weights_reduce_to_embedding_dot():
    """With every int4 linear zero (q=8, z=0) the residual stream stays E[tok]:
    logits = E . rmsnorm(E[tok]) * w_final — a closed form of the tiny model."""
    cfg = tiny_config()
    o = od.OracleDecoder(cfg, seed=0)
    zero = {}
    for name, (N, K) in cfg.linear_shapes().items():
        zero[name] = (np.full((N, K), 8, np.uint8), np.zeros((N, K // 128), np.uint16),
                      np.zeros((N, K // 128), np.uint16))
    o.syn.linear = lambda layer, name: zero[name]
    o.prefill_cache(0, 32)
    res = o.step(*_state(tok=77))
    E = od.bf16_to_f64(o.syn.embedding())
    x = E[77]
    wf = od.bf16_to_f64(o.syn.norm(-1, "final"))
    h = x / np.sqrt(np.mean(x * x) + cfg.eps) * wf
    assert np.allclose(res.logits[0], E @ h, rtol=1e-12, atol=1e-15)


def test_rows_are_independent_batch_invariance():
    cfg = tiny_config(slots=3)
    a = od.OracleDecoder(cfg, seed=0)
    b = od.OracleDecoder(cfg, seed=0)
    for s in range(3):
        a.prefill_cache(s, 20 + 5 * s)
        b.prefill_cache(s, 20 + 5 * s)
    toks = np.array([3, 9, 100], np.int32)
    cp = np.array([20, 25, 30], np.int32)
    pos = np.stack([cp - 2, cp, cp + 1]).astype(np.int32)
    full = a.step(toks, pos, cp, np.arange(3, dtype=np.int32), np.zeros(3, np.uint8))
    one = b.step(toks[1:2], pos[:, 1:2], cp[1:2], np.array([1], np.int32), np.zeros(1, np.uint8))
    assert np.allclose(full.logits[1], one.logits[0], rtol=1e-12, atol=1e-14)
    assert full.next_ids[1] == one.next_ids[0]


def test_step_writes_kv_only_at_cache_position_and_ignores_unfilled():
    cfg = tiny_config()
    clean = od.OracleDecoder(cfg, seed=0)
    clean.prefill_cache(0, 32, fill=0)
    nanfill = od.OracleDecoder(cfg, seed=0)
    nanfill.prefill_cache(0, 32, fill=int(BF16_NAN))
    before = [k.copy() for k in clean.K]
    r1 = clean.step(*_state())
    r2 = nanfill.step(*_state())
    assert np.all(np.isfinite(r2.logits))
    assert np.array_equal(r1.logits, r2.logits)       # positions > cache_position never read
    for l in range(cfg.n_layers):
        diff = np.argwhere(clean.K[l] != before[l])
        assert diff.size and np.all(diff[:, 2] == 32)   # only position 32 changed


def test_finished_row_emits_pad_and_does_not_advance():
    cfg = tiny_config()
    o = od.OracleDecoder(cfg, seed=0)
    o.prefill_cache(0, 32)
    kb = [k.copy() for k in o.K]
    t, p, c, s, f = _state()
    f[:] = 1
    r = o.step(t, p, c, s, f)
    assert r.next_ids[0] == cfg.pad_id and r.cache_position[0] == 32 and r.positions[0, 0] == 32
    assert r.finished[0] == 1 and np.all(np.isnan(r.logits[0]))
    assert all(np.array_equal(a, b) for a, b in zip(o.K, kb))


def test_advance_eos_and_length_cap():
    cfg = tiny_config()
    o = od.OracleDecoder(cfg, seed=0)
    o.prefill_cache(0, 32)
    r = o.step(*_state())
    assert r.cache_position[0] == 33 and np.all(r.positions[:, 0] == 33) and r.finished[0] == 0
    assert r.next_ids[0] == od.argmax_lowest(r.logits[0])
    # the same step with eos = the emitted token finishes the row
    cfg2 = tiny_config(eos_id=int(r.next_ids[0]))
    o2 = od.OracleDecoder(cfg2, seed=0)
    o2.prefill_cache(0, 32)
    assert o2.step(*_state()).finished[0] == 1
    # writing the last cache position finishes the row (length cap)
    o3 = od.OracleDecoder(cfg, seed=0)
    o3.prefill_cache(0, cfg.max_len - 1)
    r3 = o3.step(*_state(cpos=cfg.max_len - 1))
    assert r3.finished[0] == 1 and r3.cache_position[0] == cfg.max_len
    with pytest.raises(ValueError):
        o3.step(*_state(cpos=cfg.max_len))


def test_slot_indirection():
    cfg = tiny_config(slots=4)
    a = od.OracleDecoder(cfg, seed=0)
    b = od.OracleDecoder(cfg, seed=0)
    a.prefill_cache(0, 32)
    # the same cache contents placed in physical slot 3
    b.prefill_cache(3, 0)
    for l in range(cfg.n_layers):
        b.K[l][3] = a.K[l][0]
        b.V[l][3] = a.V[l][0]
    ra = a.step(*_state(slot=0))
    rb = b.step(*_state(slot=3))
    assert np.array_equal(ra.logits, rb.logits)


def test_tiny_workload_greedy_16_steps_runs():
    wl = tiny_workload()
    o = od.OracleDecoder.for_workload(wl)
    st = od.initial_state(wl)
    toks = []
    for _ in range(wl.steps):
        r = o.step(*st)
        toks.append(int(r.next_ids[0]))
        st = (r.next_ids, r.positions, r.cache_position, st[3], r.finished)
    assert len(toks) == 16 and all(0 <= t < wl.cfg.vocab for t in toks)
    assert st[2][0] == 32 + 16


def test_oracle_prefill_is_causal_and_chunkable():
    """Prefill [K §04] as the step applied to each prompt token: a chunked prefill equals one
    prefill, and a later prompt token changes neither the K/V nor the hidden state of the
    earlier positions (causal attention)."""
    from workloads import tiny_config
    cfg = tiny_config(slots=2)
    toks = [5, 77, 300, 12, 999, 64]
    pos = np.array([list(range(3, 9))] * 3)
    a = od.OracleDecoder(cfg, 0)
    ra = a.prefill(toks, pos, 1, 3)
    b = od.OracleDecoder(cfg, 0)
    b.prefill(toks[:4], pos[:, :4], 1, 3)
    rb = b.prefill(toks[4:], pos[:, 4:], 1, 7)
    assert np.array_equal(ra.logits, rb.logits) and ra.next_ids[0] == rb.next_ids[0]
    for l in range(cfg.n_layers):
        assert np.array_equal(a.K[l], b.K[l]) and np.array_equal(a.V[l], b.V[l])
    assert int(ra.cache_position[0]) == 9 and np.array_equal(ra.positions[:, 0], [9, 9, 9])
    c = od.OracleDecoder(cfg, 0)
    c.prefill(toks[:-1] + [1], pos, 1, 3)                      # only the last token differs
    for l in range(cfg.n_layers):
        assert np.array_equal(a.K[l][1, :, :8], c.K[l][1, :, :8]) and not np.array_equal(a.K[l][1, :, 8], c.K[l][1, :, 8])


def _one_layer_with(cfg, edit):
    """Oracle over layer 0 only, with its int4 linears replaced by edit(name, (q, s, z))."""
    o = od.OracleDecoder(cfg, seed=0, layers=1)
    lin = {n: edit(n, tuple(a.copy() for a in o.syn.linear(0, n))) for n in cfg.linear_shapes()}
    o.syn.linear = lambda layer, name: lin[name]
    return o, {n: od.dequant_int4(*lin[n], cfg.group) for n in lin}


def _zero_rows(qsz, rows):
    q, s, z = qsz
    q[rows] = 8                          # (8 - 8) s + 0 = 0 exactly
    z[rows] = 0
    return q, s, z


def _rms(x, w_bits, eps):
    return x / np.sqrt(np.mean(x * x) + eps) * od.bf16_to_f64(w_bits)


def test_layer_with_zero_q_and_k_attends_uniformly():
    """W_q = W_k = 0 make every score 0, so each query head's attention is the plain mean of
    its KV head's cached V rows and the new token's v (bf16, as the cache holds it); with
    gate_up = 0 the MLP adds nothing.  The layer then has a closed form that fixes how the
    pieces compose: v from the normed input, the new position included, the query-to-KV-head
    map, the O projection's head order and the residual."""
    cfg = tiny_config()
    qd, kvd, d = cfg.q_dim, cfg.kv_dim, cfg.head_dim
    rep = cfg.n_q_heads // cfg.n_kv_heads
    o, W = _one_layer_with(cfg, lambda n, qsz: _zero_rows(qsz, slice(0, qd + kvd)) if n == "qkv"
                           else (_zero_rows(qsz, slice(None)) if n == "gate_up" else qsz))
    t, tok = 20, 41
    o.prefill_cache(0, t)
    res = o.step(*_state(cpos=t, tok=tok))
    syn = o.syn
    E = od.bf16_to_f64(syn.embedding())
    x0 = E[tok]
    h = _rms(x0, syn.norm(0, "in"), cfg.eps)
    v_new = od.bf16_to_f64(od.f64_to_bf16_bits((W["qkv"][qd + kvd:] @ h).reshape(cfg.n_kv_heads, d)))
    V = np.concatenate([od.bf16_to_f64(syn.kv_prefill(0, 0, t, "v")[:, :t]), v_new[:, None, :]], axis=1)
    per_kv = V.sum(axis=1) / (t + 1)
    attn = np.concatenate([per_kv[i // rep] for i in range(cfg.n_q_heads)])
    x1 = x0 + W["o"] @ attn
    logits = E @ _rms(x1, syn.norm(-1, "final"), cfg.eps)
    assert np.allclose(res.logits[0], logits, rtol=1e-11, atol=1e-14)
    assert np.array_equal(od.bf16_to_f64(o.V[0][0][:, t]), v_new)
    assert not od.bf16_to_f64(o.K[0][0][:, t]).any()


def test_layer_with_zero_attention_is_the_mlp_block():
    """W_qkv = 0 on an empty row (cache position 0: the new token attends itself, v = 0) leaves
    the attention block adding 0; the layer is then x + W_down (silu(gate) * up) of the
    post-attention RMSNorm, gate the first half of gate_up's rows."""
    cfg = tiny_config()
    o, W = _one_layer_with(cfg, lambda n, qsz: _zero_rows(qsz, slice(None)) if n == "qkv" else qsz)
    tok = 300
    res = o.step(*_state(cpos=0, tok=tok))
    syn = o.syn
    E = od.bf16_to_f64(syn.embedding())
    x0 = E[tok]
    h2 = _rms(x0, syn.norm(0, "post"), cfg.eps)
    gu = W["gate_up"] @ h2
    g, u = gu[:cfg.intermediate], gu[cfg.intermediate:]
    x2 = x0 + W["down"] @ (g / (1.0 + np.exp(-g)) * u)
    logits = E @ _rms(x2, syn.norm(-1, "final"), cfg.eps)
    assert np.allclose(res.logits[0], logits, rtol=1e-11, atol=1e-14)


def _rot_complex(x, pos3, d, theta, sections):
    """M-RoPE written independently of the oracle: the pair (x_i, x_{i+d/2}) as one complex
    number turned by exp(j * pos[axis(i)] * theta^(-2i/d)), axis(i) from contiguous sections."""
    axes = [0] * sections[0] + [1] * sections[1] + [2] * sections[2]
    out = np.empty(d)
    for i in range(d // 2):
        zc = complex(x[i], x[i + d // 2]) * np.exp(1j * pos3[axes[i]] * theta ** (-2.0 * i / d))
        out[i], out[i + d // 2] = zc.real, zc.imag
    return out


def _two_position_layer(cfg, syn, W, tok, pos3, cpos, norm_after_rope=False, swap_qk_norm=False,
                        rotate_at_cache_position=False):
    """Closed form of one layer on a row holding one cached position (cache position 1): q and k
    from the normed input, per-head RMSNorm with the q and k weights, the rotation at the row's
    positions, then a two-way softmax per query head over the cached k and the new (bf16) k.
    The keyword flags build the same closed form with one plausible mistake in it."""
    d, qd, kvd = cfg.head_dim, cfg.q_dim, cfg.kv_dim
    rep = cfg.n_q_heads // cfg.n_kv_heads
    E = od.bf16_to_f64(syn.embedding())
    x0 = E[tok]
    h = _rms(x0, syn.norm(0, "in"), cfg.eps)
    qkv = W["qkv"] @ h
    q = qkv[:qd].reshape(cfg.n_q_heads, d)
    k = qkv[qd:qd + kvd].reshape(cfg.n_kv_heads, d)
    v = qkv[qd + kvd:].reshape(cfg.n_kv_heads, d)
    wq, wk = syn.norm(0, "q"), syn.norm(0, "k")
    if swap_qk_norm:
        wq, wk = wk, wq
    p = [cpos] * 3 if rotate_at_cache_position else list(pos3)
    rot = lambda a: _rot_complex(a, p, d, cfg.rope_theta, cfg.mrope_sections)
    if norm_after_rope:
        qr = np.stack([_rms(rot(a), wq, cfg.eps) for a in q])
        kr = np.stack([_rms(rot(a), wk, cfg.eps) for a in k])
    else:
        qr = np.stack([rot(_rms(a, wq, cfg.eps)) for a in q])
        kr = np.stack([rot(_rms(a, wk, cfg.eps)) for a in k])
    k_new = od.bf16_to_f64(od.f64_to_bf16_bits(kr))
    v_new = od.bf16_to_f64(od.f64_to_bf16_bits(v))
    K0 = od.bf16_to_f64(syn.kv_prefill(0, 0, 1, "k")[:, 0])
    V0 = od.bf16_to_f64(syn.kv_prefill(0, 0, 1, "v")[:, 0])
    attn = np.empty((cfg.n_q_heads, d))
    for i in range(cfg.n_q_heads):
        hk = i // rep
        s0 = qr[i] @ K0[hk] / np.sqrt(d)
        s1 = qr[i] @ k_new[hk] / np.sqrt(d)
        p1 = 1.0 / (1.0 + np.exp(s0 - s1))           # softmax over the two positions
        attn[i] = (1.0 - p1) * V0[hk] + p1 * v_new[hk]
    x1 = x0 + W["o"] @ attn.reshape(-1)
    return E @ _rms(x1, syn.norm(-1, "final"), cfg.eps), k_new


def test_layer_qk_norm_then_mrope_at_positions_closed_form():
    """How the attention prologue composes ("kaminari", §03 Architecture overview: TextAttention
    with fused QKV and Mrope; §04 Request lifecycle: positions (3, B, 1) and cache_position):
    per-head RMSNorm of q and k with their own weights, then the 3-section rotation at the row's
    positions (distinct T/H/W ids, none equal to the cache position), then attention over the
    cached position and the new one.  Non-zero W_q and W_k, gate_up = 0 (the MLP adds nothing).
    The same closed form built with the norm after the rotation, with the q and k norm weights
    swapped, or with the rotation at cache_position differs from the correct one by far more than
    the tolerance, so an oracle making any of those mistakes fails this test."""
    cfg = tiny_config()
    o, W = _one_layer_with(cfg, lambda n, qsz: _zero_rows(qsz, slice(None)) if n == "gate_up" else qsz)
    tok, cp, pos3 = 211, 1, (57, 23, 9)
    o.prefill_cache(0, cp)
    state = (np.array([tok], np.int32), np.array(pos3, np.int32).reshape(3, 1), np.array([cp], np.int32),
             np.array([0], np.int32), np.zeros(1, np.uint8))
    res = o.step(*state)
    want, k_new = _two_position_layer(cfg, o.syn, W, tok, pos3, cp)
    assert np.allclose(res.logits[0], want, rtol=1e-11, atol=1e-14)
    assert np.array_equal(od.bf16_to_f64(o.K[0][0][:, cp]), k_new)     # the cache holds the rotated k
    scale = np.linalg.norm(want)
    for mistake in ("norm_after_rope", "swap_qk_norm", "rotate_at_cache_position"):
        wrong, _ = _two_position_layer(cfg, o.syn, W, tok, pos3, cp, **{mistake: True})
        assert np.linalg.norm(wrong - want) > 1e-6 * scale, mistake
