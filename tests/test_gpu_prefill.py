"""GPU parity of text prefill (kmr_prefill) against the oracle's definition — the decode step
applied to each prompt token in order ("kaminari", §04 Request lifecycle: prefill fills the
static cache and yields the first token from the last position's logits).

Besides the oracle: chunked prefill must equal one-chunk prefill bit for bit (a row's result
depends only on that row), and prefill must agree with the GPU's own decode step run token by
token (the prefill GEMM sums the 128-input groups in order where the decode GEMV uses a
pairwise tree, so the two differ by rounding only).

The oracle cases run on both projection kernels: the default warp-level one and the opt-in
tcgen05 one (fp16-dequantised weights, fp32 accumulation in tensor memory)."""
import numpy as np
import pytest

from gpu_helpers import REL_L2_TOL, d2h_bytes, greedy_agrees, rel_l2, require_gpu
import int4_weight_only_group_gb300 as kmr
from int4_weight_only_group_gb300 import driver
from oracle import decoder as od
from workloads import SyntheticModel, layer2b_config, tiny_config

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return require_gpu()


def _model(cfg, seed=0, cap=None, max_batch=1, tc=False):
    """tc: False (warp-level kernel), True (tcgen05, planned tiles) or (nt, ksplit) forced."""
    syn = SyntheticModel(cfg, seed)
    m = kmr.Model.from_config(cfg, max_batch=max_batch)
    driver.load_weights(m, syn, cfg.n_layers, cfg.qk_norm)
    m.set_prefill_tcgen05(bool(tc))
    if isinstance(tc, tuple):
        m.set_prefill_plan(*tc)
    if cap:
        m.reserve_prefill(cap)
    return m, syn


def _prompt(cfg, T, seed, start=0, delta=0):
    r = np.random.default_rng(seed)
    toks = r.integers(1, cfg.vocab - 1, size=T).astype(np.int32)
    p = np.arange(start, start + T, dtype=np.int32) + delta
    return toks, np.stack([p, p, p]).astype(np.int32)


class State:
    def __init__(self, torch, V):
        self.t = torch
        self.tok = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.pos = torch.zeros(3, dtype=torch.int32, device="cuda")
        self.cpos = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.fin = torch.ones(1, dtype=torch.uint8, device="cuda")
        self.logits = torch.zeros(V, dtype=torch.float32, device="cuda")


def _prefill(torch, m, toks, pos, slot, start, st):
    T = len(toks)
    dt = torch.from_numpy(toks).cuda()
    dp = torch.from_numpy(np.ascontiguousarray(pos)).cuda()
    m.prefill(dt, dp, T, slot, start, st.tok, st.pos, st.cpos, st.fin, st.logits)
    torch.cuda.synchronize()
    assert m.sync_status() == 0


def _cache(m, cfg, slot):
    n = cfg.slots * cfg.n_kv_heads * cfg.max_len * cfg.head_dim
    out = []
    for l in range(cfg.n_layers):
        for p in m.kv_pointers(l):
            a = d2h_bytes(p, n * 2).view(np.uint16).reshape(cfg.slots, cfg.n_kv_heads, cfg.max_len, cfg.head_dim)
            out.append(a[slot].copy())
    return out


TC = pytest.mark.parametrize("tc", [False, True, (256, 2), (64, 4)], ids=["mma", "tcgen05", "tc256x2", "tc64x4"])


@TC
@pytest.mark.parametrize("T,start,slot", [(40, 0, 1), (1, 0, 0), (23, 17, 1), (128, 0, 0), (16, 112, 1)])
def test_tiny_prefill_matches_oracle(torch, T, start, slot, tc):
    cfg = tiny_config(slots=2)
    m, syn = _model(cfg, cap=128, tc=tc)
    o = od.OracleDecoder(cfg, 0)
    if start:
        # earlier chunk already in the row (same on both sides)
        for l in range(cfg.n_layers):
            k = syn.kv_prefill(l, slot, start, "k")[:, :start]
            v = syn.kv_prefill(l, slot, start, "v")[:, :start]
            m.set_kv(l, slot, start, np.ascontiguousarray(k), np.ascontiguousarray(v))
        o.prefill_cache(slot, start)
    toks, pos = _prompt(cfg, T, seed=T + start, start=start, delta=-3)
    st = State(torch, cfg.vocab)
    _prefill(torch, m, toks, pos, slot, start, st)
    res = o.prefill(toks, pos, slot, start)
    logits = st.logits.cpu().numpy()
    assert rel_l2(logits, res.logits[0]) <= REL_L2_TOL
    tok = int(st.tok.cpu()[0])
    assert greedy_agrees(tok, res.logits[0])
    assert int(st.cpos.cpu()[0]) == start + T and np.array_equal(st.pos.cpu().numpy(), pos[:, -1] + 1)
    assert int(st.fin.cpu()[0]) == int(res.finished[0])
    gpu = _cache(m, cfg, slot)
    for l in range(cfg.n_layers):
        for j, ref in enumerate((o.K[l][slot], o.V[l][slot])):
            got = gpu[2 * l + j]
            sl = slice(start, start + T)
            assert rel_l2(od.bf16_to_f64(got[:, sl]), od.bf16_to_f64(ref[:, sl])) <= REL_L2_TOL, (l, j)
            if start:
                assert np.array_equal(got[:, :start], ref[:, :start])     # earlier positions untouched
    m.close()


@TC
def test_chunked_prefill_equals_one_chunk_bitwise(torch, tc):
    cfg = tiny_config(slots=2)
    toks, pos = _prompt(cfg, 70, seed=9)
    a, _ = _model(cfg, cap=70, tc=tc)
    b, _ = _model(cfg, cap=32, tc=tc)
    sa, sb = State(torch, cfg.vocab), State(torch, cfg.vocab)
    _prefill(torch, a, toks, pos, 1, 0, sa)
    for c0, c1 in ((0, 32), (32, 40), (40, 70)):
        _prefill(torch, b, toks[c0:c1], pos[:, c0:c1], 1, c0, sb)
    assert np.array_equal(sa.logits.cpu().numpy(), sb.logits.cpu().numpy())
    assert int(sa.tok.cpu()[0]) == int(sb.tok.cpu()[0])
    for x, y in zip(_cache(a, cfg, 1), _cache(b, cfg, 1)):
        assert np.array_equal(x, y)
    a.close()
    b.close()


def test_prefill_agrees_with_decode_steps_and_decoding_continues(torch):
    """Prefill of T tokens = the decode step fed the same T tokens one at a time, up to the
    order of fp32 sums: a sum that lands on the other side of a bf16 rounding boundary changes
    one cached value by a bf16 step, and the last logits move by ~1e-3 (relative L2) — within
    the parity bar both paths keep against the oracle; the same token unless the decode logits
    have a near tie.  Then decoding from the prefill's state follows the oracle under the gap
    rule."""
    cfg = tiny_config(slots=2)
    T = 37
    toks, pos = _prompt(cfg, T, seed=4, delta=5)
    a, _ = _model(cfg, cap=T)
    sa = State(torch, cfg.vocab)
    _prefill(torch, a, toks, pos, 0, 0, sa)
    b, _ = _model(cfg)
    d = driver.DeviceState([int(toks[0])], pos[:, :1], [0], [0])
    lg = torch.zeros((1, cfg.vocab), dtype=torch.float32, device="cuda")
    for i in range(T):
        d.tokens[0] = int(toks[i])                       # teacher forcing with the prompt
        d.step(b, logits=lg)
    torch.cuda.synchronize()
    dec = lg[0].cpu().numpy()
    assert rel_l2(sa.logits.cpu().numpy(), dec) <= REL_L2_TOL
    assert greedy_agrees(int(sa.tok.cpu()[0]), dec)
    assert int(sa.cpos.cpu()[0]) == int(d.cache_position.cpu()[0]) == T
    for x, y in zip(_cache(a, cfg, 0), _cache(b, cfg, 0)):
        assert rel_l2(od.bf16_to_f64(x[:, :T]), od.bf16_to_f64(y[:, :T])) <= REL_L2_TOL
    # decode on from the prefill's state, against the oracle
    o = od.OracleDecoder(cfg, 0)
    res = o.prefill(toks, pos, 0, 0)
    st = (res.next_ids, res.positions, res.cache_position, np.array([0], np.int32), res.finished)
    dev = driver.DeviceState([int(sa.tok.cpu()[0])], sa.pos.cpu().numpy().reshape(3, 1), [T], [0])
    for t in range(8):
        res = o.step(*st)
        dev.step(a, logits=lg)
        tok = int(dev.tokens.cpu()[0])
        assert rel_l2(lg[0].cpu().numpy(), res.logits[0]) <= REL_L2_TOL
        if tok != int(res.next_ids[0]):
            assert greedy_agrees(tok, res.logits[0])
            break
        st = (res.next_ids, res.positions, res.cache_position, st[3], res.finished)
    a.close()
    b.close()


@TC
def test_prefill_single_2b_layer_matches_oracle(torch, tc):
    cfg = layer2b_config(slots=1)
    T = 48
    m, _ = _model(cfg, cap=64, tc=tc)
    o = od.OracleDecoder(cfg, 0)
    toks, pos = _prompt(cfg, T, seed=2, delta=-40)
    st = State(torch, cfg.vocab)
    _prefill(torch, m, toks, pos, 0, 0, st)
    res = o.prefill(toks, pos, 0, 0)
    assert rel_l2(st.logits.cpu().numpy(), res.logits[0]) <= REL_L2_TOL
    assert greedy_agrees(int(st.tok.cpu()[0]), res.logits[0])
    gpu = _cache(m, cfg, 0)
    assert rel_l2(od.bf16_to_f64(gpu[0][:, :T]), od.bf16_to_f64(o.K[0][0][:, :T])) <= REL_L2_TOL
    assert rel_l2(od.bf16_to_f64(gpu[1][:, :T]), od.bf16_to_f64(o.V[0][0][:, :T])) <= REL_L2_TOL
    m.close()


def test_tcgen05_prefill_agrees_with_the_default_kernel(torch):
    """The tensor-core (tcgen05) projections against the default ones on the same prompt:
    logits and every cached K/V within the parity bar (fp16-dequantised weights and per-row
    scaled fp16 tokens against per-group folded integer products), the same greedy token
    unless the logits have a near tie, the same row state."""
    cfg = layer2b_config(slots=1, n_layers=2)
    T = 200
    toks, pos = _prompt(cfg, T, seed=12, delta=3)
    outs = []
    for tc in (False, True):
        m, _ = _model(cfg, cap=T, tc=tc)
        st = State(torch, cfg.vocab)
        _prefill(torch, m, toks, pos, 0, 0, st)
        outs.append((st.logits.cpu().numpy(), int(st.tok.cpu()[0]), st.pos.cpu().numpy(), int(st.cpos.cpu()[0]),
                     _cache(m, cfg, 0)))
        m.close()
    (la, ta, pa, ca, ka), (lb, tb, pb, cb, kb) = outs
    assert rel_l2(lb, la) <= REL_L2_TOL
    assert ta == tb or greedy_agrees(tb, la.astype(np.float64))
    assert np.array_equal(pa, pb) and ca == cb == T
    for x, y in zip(ka, kb):
        assert rel_l2(od.bf16_to_f64(y[:, :T]), od.bf16_to_f64(x[:, :T])) <= REL_L2_TOL


def test_tcgen05_chunked_prefill_2b_bitwise(torch):
    """On 2B-shaped projections, where the chunk sizes take different tcgen05 tile widths, a
    chunked prefill equals the one-chunk prefill bit for bit: the K split (the only plan choice
    that changes an output's sums) depends on the projection's shape alone."""
    cfg = layer2b_config(slots=1, n_layers=2)
    T = 300
    toks, pos = _prompt(cfg, T, seed=21)
    a, _ = _model(cfg, cap=T, tc=True)
    sa = State(torch, cfg.vocab)
    _prefill(torch, a, toks, pos, 0, 0, sa)
    la, ka = sa.logits.cpu().numpy(), _cache(a, cfg, 0)
    a.close()
    b, _ = _model(cfg, cap=256, tc=True)
    sb = State(torch, cfg.vocab)
    for c0, c1 in ((0, 256), (256, 264), (264, T)):
        _prefill(torch, b, toks[c0:c1], pos[:, c0:c1], 0, c0, sb)
    assert np.array_equal(la, sb.logits.cpu().numpy())
    for x, y in zip(ka, _cache(b, cfg, 0)):
        assert np.array_equal(x[:, :T], y[:, :T])
    b.close()


_PLAN_REF = {}


@pytest.mark.parametrize("plan", [(64, 1), (128, 2), (256, 1), (256, 4), (64, 4), (128, 4)],
                         ids=lambda p: f"nt{p[0]}_ks{p[1]}")
def test_tcgen05_tile_plans_agree(torch, plan):
    """Every tcgen05 tile width (64, 128, 256 tokens per CTA) and K split (1, 2, 4 CTAs of one
    cluster, partials summed in rank order) on a 200-token prompt (a ragged last tile for each
    width) of two 2B-shaped layers: within the parity bar of the default kernel, and the same
    plan run twice gives the same bits."""
    cfg = layer2b_config(slots=1, n_layers=2)
    T = 200
    toks, pos = _prompt(cfg, T, seed=12, delta=3)
    if "ref" not in _PLAN_REF:
        m, _ = _model(cfg, cap=T, tc=False)
        st = State(torch, cfg.vocab)
        _prefill(torch, m, toks, pos, 0, 0, st)
        _PLAN_REF["ref"] = (st.logits.cpu().numpy(), _cache(m, cfg, 0))
        m.close()
    la, ka = _PLAN_REF["ref"]
    m, _ = _model(cfg, cap=T, tc=plan)
    runs = []
    for _ in range(2):
        st = State(torch, cfg.vocab)
        _prefill(torch, m, toks, pos, 0, 0, st)
        runs.append((st.logits.cpu().numpy(), _cache(m, cfg, 0)))
    m.close()
    (lb, kb), (lc, kc) = runs
    assert rel_l2(lb, la) <= REL_L2_TOL
    for x, y in zip(ka, kb):
        assert rel_l2(od.bf16_to_f64(y[:, :T]), od.bf16_to_f64(x[:, :T])) <= REL_L2_TOL
    assert np.array_equal(lb, lc) and all(np.array_equal(x, y) for x, y in zip(kb, kc))


def test_prefill_plan_argument_errors(torch):
    """kmr_model_set_prefill_plan takes nt in {64, 128, 256} with ksplit in {1, 2, 4}, or (0, 0)
    for the planned tiles; anything else is rejected and leaves the plan as it was."""
    cfg = tiny_config(slots=2)
    m, _ = _model(cfg)
    L, h = kmr.lib(), m.handle
    for nt, ks in ((32, 1), (256, 3), (0, 1), (128, 0), (512, 2), (-64, 1)):
        assert L.kmr_model_set_prefill_plan(h, nt, ks) == kmr.KMR_ERR_INVALID_ARG, (nt, ks)
    for nt, ks in ((64, 1), (128, 2), (256, 4), (0, 0)):
        assert L.kmr_model_set_prefill_plan(h, nt, ks) == kmr.KMR_OK, (nt, ks)
    m.close()


def test_prefill_argument_errors(torch):
    cfg = tiny_config(slots=2)
    m, _ = _model(cfg)
    st = State(torch, cfg.vocab)
    toks, pos = _prompt(cfg, 8, seed=1)
    dt, dp = torch.from_numpy(toks).cuda(), torch.from_numpy(pos).cuda()
    L, h = kmr.lib(), m.handle
    call = lambda T, slot, start: L.kmr_prefill(h, dt.data_ptr(), dp.data_ptr(), T, slot, start, st.tok.data_ptr(),
                                               st.pos.data_ptr(), st.cpos.data_ptr(), st.fin.data_ptr(), None, None)
    assert call(8, 0, 0) == kmr.KMR_ERR_BUFFER_SIZE                 # nothing reserved yet
    assert L.kmr_model_reserve_prefill(h, 0) == kmr.KMR_ERR_INVALID_ARG
    assert L.kmr_model_reserve_prefill(h, cfg.max_len + 1) == kmr.KMR_ERR_CACHE_FULL
    m.reserve_prefill(8)
    assert call(0, 0, 0) == kmr.KMR_ERR_INVALID_ARG
    assert call(9, 0, 0) == kmr.KMR_ERR_BUFFER_SIZE
    assert call(8, 2, 0) == kmr.KMR_ERR_SLOT_RANGE
    assert call(8, 0, cfg.max_len - 7) == kmr.KMR_ERR_CACHE_FULL
    assert call(8, 0, -1) == kmr.KMR_ERR_CACHE_FULL
    assert L.kmr_prefill(h, None, dp.data_ptr(), 8, 0, 0, st.tok.data_ptr(), st.pos.data_ptr(),
                         st.cpos.data_ptr(), st.fin.data_ptr(), None, None) == kmr.KMR_ERR_INVALID_ARG
    empty = kmr.Model.from_config(cfg)
    empty.reserve_prefill(8)
    assert L.kmr_prefill(empty.handle, dt.data_ptr(), dp.data_ptr(), 8, 0, 0, st.tok.data_ptr(), st.pos.data_ptr(),
                         st.cpos.data_ptr(), st.fin.data_ptr(), None, None) == kmr.KMR_ERR_NO_PACK
    # a full row: the next token is emitted and the row is finished (cache cap)
    m.reserve_prefill(cfg.max_len)
    toks, pos = _prompt(cfg, cfg.max_len, seed=3)
    _prefill(torch, m, toks, pos, 1, 0, st)
    assert int(st.fin.cpu()[0]) == 1 and int(st.cpos.cpu()[0]) == cfg.max_len
    empty.close()
    m.close()
