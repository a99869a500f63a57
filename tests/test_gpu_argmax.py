"""Greedy argmax on the device, checked bit for bit ("kaminari", §04 Request lifecycle: the
greedy argmax stays on the device; reading c10: the lowest vocabulary index wins a tie and NaN
never wins, an all-NaN row yields 0).

The ties and NaNs are planted in the tied embedding, so they reach the logits through the real
LM head: after a first step, each row's winning vocabulary row a_b is copied onto a lower
index l_b (two bit-identical logits at the row's maximum), and one whole 8-row tile of the table
plus a single row just below the lowest winner are set to bf16 NaN.  The step is then re-run
from the same state.  Every row's token must equal the lowest-index argmax of the logits the
GPU itself returned (NaN read as -inf), must be the lowest copy of its winner, and must agree with the oracle run on the
same edited table, beside the usual relative-L2 and gap-rule checks."""
import numpy as np
import pytest

from gpu_helpers import GAP_RULE, REL_L2_TOL, build_model, greedy_agrees, rel_l2, require_gpu
from oracle import decoder as od
from workloads import BF16_NAN, Workload, tiny_config

pytestmark = pytest.mark.gpu


class _State:
    def __init__(self, torch, st, V):
        self.t = torch
        self.st = st
        self.B = len(st[0])
        self.logits = torch.zeros((self.B, V), dtype=torch.float32, device="cuda")
        self.reset()

    def reset(self):
        tok, pos, cpos, slot, fin = self.st
        t = self.t
        self.tok = t.tensor(np.asarray(tok, np.int32), device="cuda")
        self.pos = t.tensor(np.asarray(pos, np.int32).reshape(3, self.B), device="cuda")
        self.cpos = t.tensor(np.asarray(cpos, np.int32), device="cuda")
        self.slot = t.tensor(np.asarray(slot, np.int32), device="cuda")
        self.fin = t.tensor(np.asarray(fin, np.uint8), device="cuda")

    def step(self, m):
        m.decode_step(self.tok, self.pos, self.cpos, self.slot, self.fin, self.B, self.logits)
        self.t.cuda.synchronize()
        assert m.sync_status() == 0
        return self.tok.cpu().numpy().copy(), self.logits.cpu().numpy().copy()


def _workload(B):
    cfg = tiny_config(slots=B)
    r = np.random.default_rng(100 + B)
    prefill = [int(v) for v in r.integers(1, cfg.max_len - 8, B)]
    return Workload(f"tiny argmax b{B}", cfg, 5, batch=B, prefill=prefill,
                    rope_delta=[int(v) for v in r.integers(-9, 1, B)], slot_ids=[int(v) for v in r.permutation(B)],
                    first_tokens=[int(v) for v in r.integers(0, 1000, B)], steps=1)


def _lowest_argmax_bits(logits):
    v = np.where(np.isnan(logits), -np.inf, logits)
    return int(np.flatnonzero(v == v.max())[0])


@pytest.mark.parametrize("B", [1, 16])
def test_argmax_ties_and_nan_rows_bit_exact(B):
    torch = require_gpu()
    wl = _workload(B)
    cfg = wl.cfg
    m, syn = build_model(wl, max_batch=B)
    st = od.initial_state(wl)
    dev = _State(torch, st, cfg.vocab)
    tok1, log1 = dev.step(m)
    win = [_lowest_argmax_bits(log1[b]) for b in range(B)]
    assert [int(t) for t in tok1] == win                 # unedited table: token = own lowest argmax

    # plant: a tie below every winner that has room, an all-NaN tile and one NaN row
    taken = set(int(t) for t in st[0]) | set(win)
    free = [v for v in range(cfg.vocab) if v not in taken]
    E = syn.embedding().copy()
    E2 = E.copy()
    tile = next(t for t in range(0, cfg.vocab // 8) if all(8 * t + i in free for i in range(8)))
    nan_rows = set(range(8 * tile, 8 * tile + 8))
    lone = max(v for v in free if v < min(win) and v not in nan_rows) if any(
        v < min(win) and v not in nan_rows for v in free) else None
    if lone is not None:
        nan_rows.add(lone)
    low = {}
    for b, a in enumerate(win):
        cands = [v for v in free if v < a and v not in nan_rows and v not in low.values()]
        if cands:
            low[b] = cands[0]
            E2[cands[0]] = E[a]
    for v in nan_rows:
        E2[v] = BF16_NAN
    assert low, "no row had room for a lower duplicate"
    m.set_embedding(np.ascontiguousarray(E2))
    dev.reset()
    tok2, log2 = dev.step(m)

    o = od.OracleDecoder.for_workload(wl)
    o.syn.embedding = lambda: E2
    res = o.step(*st)
    bits = log2.view(np.uint32)
    nan_idx = sorted(nan_rows)
    for b in range(B):
        assert np.isnan(log2[b, nan_idx]).all(), b
        assert int(tok2[b]) == _lowest_argmax_bits(log2[b]), (b, int(tok2[b]))
        assert int(tok2[b]) not in nan_rows
        if b in low:
            assert bits[b, low[b]] == bits[b, win[b]], b          # the planted tie is exact
            # every copy of row b's winner ties with it (rows may share a winner)
            copies = [low[k] for k in low if win[k] == win[b]] + [win[b]]
            assert int(tok2[b]) == min(copies), (b, int(tok2[b]), copies)
        ok = ~np.isnan(res.logits[b])
        assert rel_l2(log2[b][ok], res.logits[b][ok]) <= REL_L2_TOL, b
        assert greedy_agrees(int(tok2[b]), res.logits[b]), b
        v = np.where(np.isnan(res.logits[b]), -np.inf, res.logits[b])
        top = v.max()
        below = v[v < top]
        if below.size and top - below.max() > GAP_RULE * abs(top):
            assert int(tok2[b]) == int(res.next_ids[b]), b         # exact ties resolve alike
    m.close()


def test_all_nan_logits_yield_token_zero():
    torch = require_gpu()
    wl = _workload(1)
    cfg = wl.cfg
    m, syn = build_model(wl, max_batch=1)
    E = np.full_like(syn.embedding(), BF16_NAN)
    m.set_embedding(np.ascontiguousarray(E))
    st = od.initial_state(wl)
    dev = _State(torch, st, cfg.vocab)
    tok, logits = dev.step(m)
    assert np.isnan(logits[0]).all()
    assert int(tok[0]) == 0
    assert int(dev.cpos.cpu()[0]) == int(st[2][0]) + 1        # the row still advances
    m.close()
