"""GPU parity of KV row migration and of continuous batching over a slot pool.

kmr_model_copy_row_from must reproduce the oracle's row move (oracle/slots.py) bit for
bit — it is a copy — at Tiny sizes and at the 2B cache shape; a continuous run whose
rows are admitted by copy_row_from must emit, per request, the tokens of that request
decoded alone ("kaminari", §08 ContinuousBatchScheduler; §03 the static cache mutated in
place)."""
import numpy as np
import pytest

from gpu_helpers import build_model, d2h_bytes, greedy_agrees, require_gpu
import int4_weight_only_group_gb300 as kmr
from int4_weight_only_group_gb300 import driver
from oracle import decoder as od
from oracle.slots import copy_row_from
from workloads import SyntheticModel, layer2b_config, tiny_config, tiny_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return require_gpu()


def _cache_host(m, cfg):
    """The model's whole K and V caches as [L][slots][n_kv][max_len][d] uint16 arrays."""
    n = cfg.slots * cfg.n_kv_heads * cfg.max_len * cfg.head_dim
    ks, vs = [], []
    for l in range(cfg.n_layers):
        kp, vp = m.kv_pointers(l)
        ks.append(d2h_bytes(kp, n * 2).view(np.uint16).reshape(cfg.slots, cfg.n_kv_heads, cfg.max_len, cfg.head_dim))
        vs.append(d2h_bytes(vp, n * 2).view(np.uint16).reshape(cfg.slots, cfg.n_kv_heads, cfg.max_len, cfg.head_dim))
    return np.stack(ks), np.stack(vs)


def _random_cache(torch, rng, L, slots, nkv, S, d):
    k = rng.integers(0, 1 << 16, size=(L, slots, nkv, S, d), dtype=np.uint16)
    v = rng.integers(0, 1 << 16, size=(L, slots, nkv, S, d), dtype=np.uint16)
    dk = torch.from_numpy(k.view(np.int16)).cuda()
    dv = torch.from_numpy(v.view(np.int16)).cuda()
    return k, v, dk, dv


def _fill_model(m, cfg, rng):
    for l in range(cfg.n_layers):
        for s in range(cfg.slots):
            k = rng.integers(0, 1 << 16, size=(cfg.n_kv_heads, cfg.max_len, cfg.head_dim), dtype=np.uint16)
            v = rng.integers(0, 1 << 16, size=(cfg.n_kv_heads, cfg.max_len, cfg.head_dim), dtype=np.uint16)
            m.set_kv(l, s, cfg.max_len, k, v)


@pytest.mark.parametrize("src_row,dst,length", [(0, 2, 17), (3, 1, 128), (1, 0, 1), (2, 3, 0), (1, 1, 50)])
def test_copy_row_within_the_pool(torch, src_row, dst, length):
    cfg = tiny_config(slots=4)
    m = kmr.Model.from_config(cfg)
    _fill_model(m, cfg, np.random.default_rng(7))
    k, v = _cache_host(m, cfg)
    m.copy_row_from(dst, length, src_row)
    torch.cuda.synchronize()
    copy_row_from(k, v, dst, k, v, src_row, length)
    k2, v2 = _cache_host(m, cfg)
    assert np.array_equal(k2, k) and np.array_equal(v2, v)
    m.close()


@pytest.mark.parametrize("src_S,length", [(96, 96), (200, 128), (128, 33)])
def test_copy_row_from_an_external_cache(torch, src_S, length):
    cfg = tiny_config(slots=3)
    m = kmr.Model.from_config(cfg)
    rng = np.random.default_rng(11)
    _fill_model(m, cfg, rng)
    k, v = _cache_host(m, cfg)
    sk, sv, dk, dv = _random_cache(torch, rng, cfg.n_layers, 5, cfg.n_kv_heads, src_S, cfg.head_dim)
    m.copy_row_from(1, length, 4, dk, dv, 5, src_S)
    torch.cuda.synchronize()
    copy_row_from(k, v, 1, sk, sv, 4, length)
    k2, v2 = _cache_host(m, cfg)
    assert np.array_equal(k2, k) and np.array_equal(v2, v)
    m.close()


def test_copy_row_errors(torch):
    cfg = tiny_config(slots=2)
    m = kmr.Model.from_config(cfg)
    _, _, dk, dv = _random_cache(torch, np.random.default_rng(1), cfg.n_layers, 2, cfg.n_kv_heads, 64, cfg.head_dim)
    L = kmr.lib()
    h = m.handle
    cases = [
        (dict(dst=2, src_k=None, src_v=None, slots=0, S=0, row=0, n=4), kmr.KMR_ERR_SLOT_RANGE),
        (dict(dst=-1, src_k=None, src_v=None, slots=0, S=0, row=0, n=4), kmr.KMR_ERR_SLOT_RANGE),
        (dict(dst=0, src_k=None, src_v=None, slots=0, S=0, row=5, n=4), kmr.KMR_ERR_SLOT_RANGE),
        (dict(dst=0, src_k=None, src_v=None, slots=0, S=0, row=1, n=cfg.max_len + 1), kmr.KMR_ERR_CACHE_FULL),
        (dict(dst=0, src_k=dk.data_ptr(), src_v=dv.data_ptr(), slots=2, S=64, row=0, n=65), kmr.KMR_ERR_CACHE_FULL),
        (dict(dst=0, src_k=dk.data_ptr(), src_v=dv.data_ptr(), slots=2, S=64, row=2, n=4), kmr.KMR_ERR_INVALID_ARG),
        (dict(dst=0, src_k=dk.data_ptr(), src_v=None, slots=2, S=64, row=0, n=4), kmr.KMR_ERR_INVALID_ARG),
        (dict(dst=0, src_k=dk.data_ptr() + 2, src_v=dv.data_ptr(), slots=2, S=64, row=0, n=4), kmr.KMR_ERR_INVALID_ARG),
        (dict(dst=0, src_k=dk.data_ptr(), src_v=dv.data_ptr(), slots=0, S=64, row=0, n=4), kmr.KMR_ERR_INVALID_ARG),
        (dict(dst=0, src_k=None, src_v=None, slots=0, S=0, row=1, n=-1), kmr.KMR_ERR_INVALID_ARG),
    ]
    for a, want in cases:
        got = L.kmr_model_copy_row_from(h, a["dst"], a["src_k"], a["src_v"], a["slots"], a["S"], a["row"], a["n"], None)
        assert got == want, (a, got)
    assert L.kmr_model_copy_row_from(None, 0, None, None, 0, 0, 0, 1, None) == kmr.KMR_ERR_INVALID_ARG
    m.close()


def test_copy_full_row_at_2b_cache_shape(torch):
    """A whole 1024-position row of the 2B cache (28 layers x 8 heads x K/V: 117 MB)."""
    cfg = layer2b_config(n_layers=28, slots=3)
    m = kmr.Model.from_config(cfg)
    rng = np.random.default_rng(5)
    S = cfg.max_len
    sk, sv, dk, dv = _random_cache(torch, rng, cfg.n_layers, 2, cfg.n_kv_heads, S, cfg.head_dim)
    m.copy_row_from(2, S, 1, dk, dv, 2, S)                       # external row 1 -> slot 2
    m.copy_row_from(0, 700, 2)                                   # slot 2 -> slot 0, first 700 positions
    torch.cuda.synchronize()
    assert m.sync_status() == 0
    k, v = _cache_host(m, cfg)
    assert np.array_equal(k[:, 2], sk[:, 1]) and np.array_equal(v[:, 2], sv[:, 1])
    assert np.array_equal(k[:, 0, :, :700], sk[:, 1, :, :700]) and np.array_equal(v[:, 0, :, :700], sv[:, 1, :, :700])
    assert not k[:, 0, :, 700:].any() and not v[:, 1].any()      # untouched rows stay zero-filled
    m.close()


def test_continuous_batching_matches_each_request_alone(torch):
    """Five requests through a two-slot pool, each admitted by copy_row_from of its prefilled
    row in a separate prefill cache: every request's tokens equal that request decoded alone
    on the GPU (batch invariance), and agree with the oracle under the gap rule."""
    R = 5
    cfg = tiny_config(slots=max(R, 2))
    seed = 2
    syn = SyntheticModel(cfg, seed)
    lengths = [9, 40, 3, 77, 20]
    deltas = [0, -3, 5, 0, -10]
    budgets = [6, 3, 9, 4, 1]
    firsts = [17, 300, 5, 1000, 64]
    # the prefill stand-in: row r of an external cache holds request r's prompt K/V
    L, nkv, S, d = cfg.n_layers, cfg.n_kv_heads, cfg.max_len, cfg.head_dim
    pk = np.zeros((L, R, nkv, S, d), np.uint16)
    pv = np.zeros((L, R, nkv, S, d), np.uint16)
    for r in range(R):
        for l in range(L):
            pk[l, r] = syn.kv_prefill(l, r, lengths[r], "k")
            pv[l, r] = syn.kv_prefill(l, r, lengths[r], "v")
    dpk = torch.from_numpy(pk.view(np.int16)).cuda()
    dpv = torch.from_numpy(pv.view(np.int16)).cuda()

    pool_cfg = tiny_config(slots=2)
    m = kmr.Model.from_config(pool_cfg, max_batch=2)
    driver.load_weights(m, syn, L, cfg.qk_norm)

    def loader(r):
        return lambda model, slot, stream: model.copy_row_from(slot, lengths[r], r, dpk, dpv, R, S, stream)

    reqs = [driver.Request(r, firsts[r], lengths[r], deltas[r], budgets[r], loader(r)) for r in range(R)]
    out = driver.generate_continuous(m, reqs, n_slots=2, eos_id=cfg.eos_id)
    assert sorted(out) == list(range(R))

    # each request alone, B = 1, on its own model: the same tokens bit for bit
    solo = kmr.Model.from_config(pool_cfg, max_batch=1)
    driver.load_weights(solo, syn, L, cfg.qk_norm)
    for r in range(R):
        solo.copy_row_from(0, lengths[r], r, dpk, dpv, R, S)
        st = driver.DeviceState([firsts[r]], [[lengths[r] + deltas[r]]] * 3, [lengths[r]], [0])
        toks = driver.generate(solo, st, budgets[r], eos_id=cfg.eos_id)[0]
        assert toks == out[r], (r, toks, out[r])

    # and the oracle, free running per request, until a near tie may legitimately diverge
    for r in range(R):
        o = od.OracleDecoder(cfg, seed)
        o.prefill_cache(r, lengths[r])
        st = (np.array([firsts[r]], np.int32), np.full((3, 1), lengths[r] + deltas[r], np.int32),
              np.array([lengths[r]], np.int32), np.array([r], np.int32), np.zeros(1, np.uint8))
        for t, tok in enumerate(out[r]):
            res = o.step(*st)
            if tok != int(res.next_ids[0]):
                assert greedy_agrees(tok, res.logits[0]), (r, t)
                break
            st = (res.next_ids, res.positions, res.cache_position, st[3], res.finished)
    m.close()
    solo.close()


def test_continuous_batching_prefills_prompts_on_admission(torch):
    """Requests that carry their prompt: each is prefilled into its slot on admission and
    decoded in the shared batch.  Every request's tokens equal that request prefilled and
    decoded alone on the GPU, and agree with the oracle's prefill + steps under the gap rule."""
    cfg = tiny_config(slots=2)
    seed = 3
    syn = SyntheticModel(cfg, seed)
    rng = np.random.default_rng(11)
    lengths = [12, 1, 57, 30, 128]
    deltas = [0, 4, -7, 0, 2]
    budgets = [5, 3, 1, 7, 4]
    prompts = [rng.integers(1, cfg.vocab - 1, size=n).astype(np.int32) for n in lengths]
    m = kmr.Model.from_config(cfg, max_batch=2)
    driver.load_weights(m, syn, cfg.n_layers, cfg.qk_norm)
    reqs = [driver.Request(r, 0, 0, deltas[r], budgets[r], prompt=prompts[r].tolist()) for r in range(len(lengths))]
    out = driver.generate_continuous(m, reqs, n_slots=2, eos_id=cfg.eos_id)
    assert sorted(out) == list(range(len(lengths)))

    solo = kmr.Model.from_config(cfg, max_batch=1)
    driver.load_weights(solo, syn, cfg.n_layers, cfg.qk_norm)
    solo.reserve_prefill(max(lengths))
    for r, T in enumerate(lengths):
        tok = torch.zeros(1, dtype=torch.int32, device="cuda")
        spos = torch.zeros(3, dtype=torch.int32, device="cuda")
        cpos = torch.zeros(1, dtype=torch.int32, device="cuda")
        fin = torch.zeros(1, dtype=torch.uint8, device="cuda")
        p = np.arange(T, dtype=np.int32) + deltas[r]
        solo.prefill(torch.from_numpy(prompts[r]).cuda(), torch.from_numpy(np.stack([p, p, p])).cuda(), T, 0, 0,
                     tok, spos, cpos, fin, None)
        first = int(tok.cpu()[0])
        got = [first]
        if budgets[r] > 1 and not int(fin.cpu()[0]):
            st = driver.DeviceState([first], spos.cpu().numpy().reshape(3, 1), [T], [0])
            got += driver.generate(solo, st, budgets[r] - 1, eos_id=cfg.eos_id)[0]
        if cfg.eos_id in got:
            got = got[:got.index(cfg.eos_id) + 1]
        assert got == out[r], (r, got, out[r])

    for r, T in enumerate(lengths):
        o = od.OracleDecoder(cfg, seed)
        p = np.arange(T, dtype=np.int32) + deltas[r]
        res = o.prefill(prompts[r], np.stack([p, p, p]), 0, 0)
        for t, tok in enumerate(out[r]):
            if tok != int(res.next_ids[0]):
                assert greedy_agrees(tok, res.logits[0]), (r, t)
                break
            st = (res.next_ids, res.positions, res.cache_position, np.array([0], np.int32), res.finished)
            res = o.step(*st)
    m.close()
    solo.close()
