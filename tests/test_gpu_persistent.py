"""The persistent decode step (every layer in one kernel, kmr_model_set_persistent_step)
against the multi-kernel step, bit for bit: logits, emitted tokens, the advanced state and
the whole KV cache after several free-running steps, from identical models.  Both paths run
the same per-row arithmetic in the same order, so nothing may differ; parity of either path
with the oracle is covered by the step tests, which run the persistent step by default."""
import numpy as np
import pytest

from gpu_helpers import build_model, d2h_bytes, require_gpu
from oracle import decoder as od
from workloads import Workload, layer2b_config, tiny_config

pytestmark = pytest.mark.gpu


class _State:
    def __init__(self, torch, st, V):
        self.t = torch
        tok, pos, cpos, slot, fin = st
        self.B = len(tok)
        self.tok = torch.tensor(np.asarray(tok, np.int32), device="cuda")
        self.pos = torch.tensor(np.asarray(pos, np.int32).reshape(3, self.B), device="cuda")
        self.cpos = torch.tensor(np.asarray(cpos, np.int32), device="cuda")
        self.slot = torch.tensor(np.asarray(slot, np.int32), device="cuda")
        self.fin = torch.tensor(np.asarray(fin, np.uint8), device="cuda")
        self.logits = torch.zeros((self.B, V), dtype=torch.float32, device="cuda")

    def step(self, m):
        m.decode_step(self.tok, self.pos, self.cpos, self.slot, self.fin, self.B, self.logits)
        self.t.cuda.synchronize()
        assert m.sync_status() == 0
        return [a.cpu().numpy().copy() for a in (self.tok, self.pos, self.cpos, self.fin, self.logits)]


def _kv(m, cfg):
    n = cfg.slots * cfg.n_kv_heads * cfg.max_len * cfg.head_dim * 2
    out = []
    for l in range(cfg.n_layers):
        k, v = m.kv_pointers(l)
        out.append((d2h_bytes(k, n), d2h_bytes(v, n)))
    return out


def _compare_paths(torch, wl, steps, finish=None):
    cfg = wl.cfg
    models = {}
    for persistent in (True, False):
        m, _ = build_model(wl, max_batch=wl.batch)
        m.set_persistent_step(persistent)
        models[persistent] = m
    assert models[True].kernels_per_step(wl.batch) == 2, "the persistent step does not serve this shape"
    assert models[False].kernels_per_step(wl.batch) > 2
    st = od.initial_state(wl)
    devs = {k: _State(torch, st, cfg.vocab) for k in models}
    for t in range(steps):
        if finish and t in finish:
            for d in devs.values():
                d.fin[finish[t]] = 1
        outs = {k: devs[k].step(models[k]) for k in models}
        for name, a, b in zip(("tok", "pos", "cpos", "fin", "logits"), outs[True], outs[False]):
            assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), (t, name)
    assert models[True].kernels_per_step(wl.batch) == 2, "the persistent step fell back to the multi-kernel step"
    for l, ((ka, va), (kb, vb)) in enumerate(zip(_kv(models[True], cfg), _kv(models[False], cfg))):
        assert np.array_equal(ka, kb) and np.array_equal(va, vb), l
    for m in models.values():
        m.close()


@pytest.mark.parametrize("B", [1, 2, 4])
def test_tiny_persistent_equals_multi_kernel(B):
    torch = require_gpu()
    cfg = tiny_config(slots=4)
    r = np.random.default_rng(40 + B)
    wl = Workload(f"tiny b{B}", cfg, 3, batch=B, prefill=[int(v) for v in r.integers(1, 100, B)],
                  rope_delta=[int(v) for v in r.integers(-9, 1, B)], slot_ids=[int(v) for v in r.permutation(4)[:B]],
                  first_tokens=[int(v) for v in r.integers(0, 1000, B)], steps=6)
    _compare_paths(torch, wl, 6, finish={3: B - 1} if B > 1 else None)


def test_2b_layers_persistent_equals_multi_kernel_b1():
    torch = require_gpu()
    cfg = layer2b_config(n_layers=3, vocab=8192)
    wl = Workload("2b 3 layers b1", cfg, 0, batch=1, prefill=[600], rope_delta=[-40], slot_ids=[0],
                  first_tokens=[17], steps=3)
    _compare_paths(torch, wl, 3)


def test_2b_layers_persistent_equals_multi_kernel_b4_slots():
    torch = require_gpu()
    cfg = layer2b_config(n_layers=2, vocab=8192, slots=4)
    wl = Workload("2b 2 layers b4", cfg, 1, batch=4, prefill=[300, 512, 700, 1020], rope_delta=[0, -17, -60, -3],
                  slot_ids=[2, 0, 3, 1], first_tokens=[5, 77, 300, 1000], steps=3)
    # row 3 writes positions 1020..1022; row 2 retires at step 1
    _compare_paths(torch, wl, 3, finish={1: 2})


def test_persistent_step_reports_bad_row_state_without_faulting():
    """An unfinished row with cache_position = max_len: the persistent step records
    KMR_ERR_CACHE_FULL and leaves the other rows' results intact (equal to the multi-kernel
    step's)."""
    torch = require_gpu()
    import int4_weight_only_group_gb300 as kmr
    cfg = tiny_config(slots=2)
    wl = Workload("tiny bad", cfg, 2, batch=2, prefill=[20, 30], rope_delta=[0, 0], slot_ids=[0, 1],
                  first_tokens=[5, 6], steps=1)
    res = {}
    for persistent in (True, False):
        m, _ = build_model(wl, max_batch=2)
        m.set_persistent_step(persistent)
        st = list(od.initial_state(wl))
        st[2] = np.array([20, cfg.max_len], np.int32)
        d = _State(torch, st, cfg.vocab)
        m.decode_step(d.tok, d.pos, d.cpos, d.slot, d.fin, 2, d.logits)
        torch.cuda.synchronize()
        assert m.sync_status() == kmr.KMR_ERR_CACHE_FULL
        res[persistent] = d.logits.cpu().numpy()[0].copy()
        m.close()
    assert np.array_equal(res[True].view(np.uint32), res[False].view(np.uint32))
