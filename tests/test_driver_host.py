"""Host logic of the continuous-batching driver (slot pool, admission, eviction) — CPU only.

A fake model stands in for the library: its decode step emits, for each unfinished row,
the next token of a per-slot script and applies the same finished / advance rules the
step documents (EOS or the cache cap finish a row; finished rows emit pad and stay put)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from int4_weight_only_group_gb300.driver import Request, SlotPool, generate_continuous


def test_slot_pool_lowest_first_and_reuse():
    p = SlotPool(3)
    assert [p.admit(k) for k in "abc"] == [0, 1, 2] and p.n_free == 0
    with pytest.raises(RuntimeError):
        p.admit("d")
    assert p.release(1) == "b" and p.n_free == 1
    assert p.admit("d") == 1 and p.active == {0: "a", 1: "d", 2: "c"}
    with pytest.raises(KeyError):
        p.release(7)
    with pytest.raises(ValueError):
        SlotPool(0)


class FakeModel:
    """Scripted stand-in for Model.decode_step on CPU tensors."""

    def __init__(self, scripts, eos, pad, max_len):
        self.scripts = scripts          # slot -> callable(step index within the row's life) -> token
        self.eos, self.pad, self.max_len = eos, pad, max_len
        self.loaded = []                # (rid, slot) in load order
        self.age = {}
        self.ticks = 0

    def load(self, rid):
        def f(model, slot, stream):
            assert model is self
            self.loaded.append((rid, slot))
            self.age[slot] = 0
        return f

    def decode_step(self, tok, pos, cpos, slots, fin, B, logits, stream):
        self.ticks += 1
        for b in range(B):
            if fin[b]:
                tok[b] = self.pad
                continue
            s = int(slots[b])
            t = self.scripts[s](self.age[s])
            self.age[s] += 1
            tok[b] = t
            cpos[b] += 1
            pos[:, b] += 1
            if t == self.eos or int(cpos[b]) >= self.max_len:
                fin[b] = 1


def test_continuous_admits_finalises_and_reuses_slots():
    eos, pad, S = 99, 0, 64
    # every slot emits 10, 11, 12, ... ; request "e" will meet EOS through its script below
    scripts = {s: (lambda a: 10 + a) for s in range(2)}
    m = FakeModel(scripts, eos, pad, S)
    reqs = [Request("a", 5, 4, 0, 3, m.load("a")),
            Request("b", 5, 4, 0, 5, m.load("b")),
            Request("c", 5, 4, 0, 2, m.load("c")),
            Request("z", 5, 4, 0, 0, m.load("z")),          # nothing to generate: never takes a slot
            Request("d", 5, 62, 0, 10, m.load("d"))]        # meets the cache cap after 2 tokens
    out = generate_continuous(m, reqs, n_slots=2, eos_id=eos, device="cpu")
    assert out == {"a": [10, 11, 12], "b": [10, 11, 12, 13, 14], "c": [10, 11], "z": [], "d": [10, 11]}
    # a frees slot 0 after 3 ticks and c takes it; b frees slot 1, d takes the lowest free slot
    assert m.loaded == [("a", 0), ("b", 1), ("c", 0), ("d", 0)]
    assert m.ticks == 7


def test_continuous_trims_at_eos():
    eos, pad = 99, 0
    scripts = {0: (lambda a: [7, 8, eos, 5][a])}
    m = FakeModel(scripts, eos, pad, 64)
    out = generate_continuous(m, [Request("x", 1, 3, -2, 8, m.load("x"))], n_slots=1, eos_id=eos, device="cpu")
    assert out == {"x": [7, 8, eos]} and m.ticks == 3


def test_continuous_row_state_written_at_admission():
    seen = {}

    class Probe(FakeModel):
        def decode_step(self, tok, pos, cpos, slots, fin, B, logits, stream):
            if self.ticks == 0:
                seen.update(tok=tok.clone(), pos=pos.clone(), cpos=cpos.clone(), fin=fin.clone())
            super().decode_step(tok, pos, cpos, slots, fin, B, logits, stream)

    m = Probe({0: (lambda a: 3), 1: (lambda a: 3), 2: (lambda a: 3)}, 99, 0, 64)
    reqs = [Request("p", 11, 20, -5, 1, m.load("p")), Request("q", 12, 30, 2, 1, m.load("q"))]
    generate_continuous(m, reqs, n_slots=3, device="cpu")
    assert seen["tok"].tolist() == [11, 12, 0]
    assert seen["cpos"].tolist() == [20, 30, 0]
    assert np.array_equal(seen["pos"].numpy(), np.array([[15, 32, 0]] * 3))
    assert seen["fin"].tolist() == [0, 0, 1]                 # the empty row is a finished row


class FakePrefillModel(FakeModel):
    """FakeModel plus a scripted prefill: the first token of slot s is 50 + s, the row state
    advances to the first decode step's (cache position T, ids last + 1)."""

    def __init__(self, *a, **kw):
        super().__init__(*a, **kw)
        self.prefilled = []

    def reserve_prefill(self, T):
        pass

    def prefill(self, ptok, ppos, T, slot, start, st_tok, st_pos, st_cpos, st_fin, logits, stream):
        self.prefilled.append((slot, T, ptok.tolist(), ppos[:, -1].tolist()))
        self.age[slot] = 0
        st_tok[0] = 50 + slot
        st_pos.copy_(ppos[:, -1] + 1)
        st_cpos[0] = start + T
        st_fin[0] = 1 if start + T >= self.max_len else 0


def test_continuous_prefills_prompts_on_admission():
    eos, pad = 99, 0
    m = FakePrefillModel({s: (lambda a: 10 + a) for s in range(2)}, eos, pad, 64)
    reqs = [Request("p", 0, 0, 2, 3, prompt=[7, 8, 9]),
            Request("q", 0, 0, -1, 1, prompt=[4]),                  # one token: the prefill's alone
            Request("r", 0, 0, 0, 2, prompt=list(range(64))),      # fills the row: finished at once
            Request("s", 0, 0, 0, 2, prompt=[5, 6])]
    out = generate_continuous(m, reqs, n_slots=2, eos_id=eos, device="cpu")
    # p: prefill token 50 (slot 0), then decode 10, 11; q: 51 alone (slot 1); r: slot 1, full;
    # s: slot 1 after r, 51 then 10
    assert out == {"p": [50, 10, 11], "q": [51], "r": [51], "s": [51, 10]}
    assert m.prefilled[0] == (0, 3, [7, 8, 9], [4, 4, 4])      # ids = position + rope_delta
    assert [x[0] for x in m.prefilled] == [0, 1, 1, 1]


def test_continuous_rejects_requests_without_a_kv_source():
    m = FakePrefillModel({0: (lambda a: 10)}, 99, 0, 64)
    with pytest.raises(ValueError, match="empty prompt"):
        generate_continuous(m, [Request("e", 0, 0, 0, 2, prompt=[])], n_slots=1, device="cpu")
    with pytest.raises(ValueError, match="prompt or a load_kv"):
        generate_continuous(m, [Request("n", 0, 0, 0, 2)], n_slots=1, device="cpu")
    assert m.prefilled == [] and m.ticks == 0                 # nothing ran
