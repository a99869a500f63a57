"""GPU parity of the shared-prefix (cascade) decode attention against the oracle's three
steps ("The Ghost in the Batch", The Optimization That Changes Everything: prefix once,
each suffix separately, LSE-weighted merge) and against plain decode attention over the
concatenated context."""
import math

import numpy as np
import pytest

from gpu_helpers import REL_L2_TOL, rel_l2, require_gpu
import int4_weight_only_group_gb300 as kmr
from oracle import decoder as od
from workloads import BF16_NAN, f32_to_bf16_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return require_gpu()


def _setup(r, B, nq, nkv, d, S, slots, pslot, P, cpos, slot_ids):
    """A one-layer cache with NaN wherever the cascade must not read: the prefix row past P,
    each row's own positions below P and past cache_position."""
    q = r.standard_normal((B, nq, d)).astype(np.float32)
    kc = np.full((slots, nkv, S, d), BF16_NAN, np.uint16)
    vc = np.full((slots, nkv, S, d), BF16_NAN, np.uint16)
    kc[pslot, :, :P] = f32_to_bf16_bits(r.standard_normal((nkv, P, d)).astype(np.float32))
    vc[pslot, :, :P] = f32_to_bf16_bits(r.standard_normal((nkv, P, d)).astype(np.float32))
    for b in range(B):
        n = cpos[b] + 1 - P
        kc[slot_ids[b], :, P:cpos[b] + 1] = f32_to_bf16_bits(r.standard_normal((nkv, n, d)).astype(np.float32))
        vc[slot_ids[b], :, P:cpos[b] + 1] = f32_to_bf16_bits(r.standard_normal((nkv, n, d)).astype(np.float32))
    return q, kc, vc


def _run(torch, q, kc, vc, slot_ids, cpos, pslot, P, nq, nkv, d, S, slots):
    B = q.shape[0]
    ws_bytes = kmr.kmr_decode_attn_cascade_workspace_size(B, nq, nkv, d, P)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    out = torch.full((B, nq, d), float("nan"), dtype=torch.float32, device="cuda")
    kmr.kmr_decode_attn_cascade(torch.from_numpy(q).cuda(), torch.from_numpy(kc.view(np.int16)).cuda(),
                                torch.from_numpy(vc.view(np.int16)).cuda(),
                                torch.tensor(slot_ids, dtype=torch.int32, device="cuda"),
                                torch.tensor(cpos, dtype=torch.int32, device="cuda"), pslot, P, B, nq, nkv, d, S, slots,
                                1.0 / math.sqrt(d), out, ws, ws_bytes, torch.cuda.current_stream())
    torch.cuda.synchronize()
    return out.cpu().numpy(), kmr.kmr_last_device_error()


def _oracle(q, kc, vc, slot_ids, cpos, pslot, P):
    out = []
    for b in range(q.shape[0]):
        Kp, Vp = od.bf16_to_f64(kc[pslot, :, :P]), od.bf16_to_f64(vc[pslot, :, :P])
        Ks = od.bf16_to_f64(kc[slot_ids[b], :, P:cpos[b] + 1])
        Vs = od.bf16_to_f64(vc[slot_ids[b], :, P:cpos[b] + 1])
        out.append(od.cascade_attention(q[b].astype(np.float64), Kp, Vp, Ks, Vs))
    return np.stack(out)


@pytest.mark.parametrize("d,nq,nkv", [(128, 16, 8), (64, 4, 2), (128, 8, 8), (64, 16, 4)])
@pytest.mark.parametrize("P", [0, 1, 16, 400, 700])
def test_cascade_matches_oracle(torch, d, nq, nkv, P):
    r = np.random.default_rng(P + d + nq)
    S = 1024
    B = 6
    cpos = [P, P + 1, P + 7, P + 63, P + 64, min(S - 1, P + 200)]     # own suffixes of 1 .. 201 positions
    slots = B + 2
    pslot = B + 1
    slot_ids = list(range(B))
    q, kc, vc = _setup(r, B, nq, nkv, d, S, slots, pslot, P, cpos, slot_ids)
    out, err = _run(torch, q, kc, vc, slot_ids, cpos, pslot, P, nq, nkv, d, S, slots)
    assert err == 0 and np.all(np.isfinite(out))           # NaN where nothing may be read
    ref = _oracle(q, kc, vc, slot_ids, cpos, pslot, P)
    for b in range(B):
        assert rel_l2(out[b], ref[b]) <= 1e-4, (b, rel_l2(out[b], ref[b]))


def test_cascade_equals_plain_attention_over_the_concatenation(torch):
    """16 rows sharing a 400-position prefix with 100 own positions each (the pages'
    example): the cascade equals kmr_decode_attn over rows that hold [prefix; own]."""
    r = np.random.default_rng(3)
    B, nq, nkv, d, S, P = 16, 16, 8, 128, 1024, 400
    cpos = [P + 99 - (b % 5) for b in range(B)]
    slots = B + 1
    q, kc, vc = _setup(r, B, nq, nkv, d, S, slots, B, P, cpos, list(range(B)))
    out, err = _run(torch, q, kc, vc, list(range(B)), cpos, B, P, nq, nkv, d, S, slots)
    assert err == 0
    full_k, full_v = kc.copy(), vc.copy()
    full_k[:B, :, :P] = kc[B, :, :P]
    full_v[:B, :, :P] = vc[B, :, :P]
    ws_bytes = kmr.kmr_decode_attn_workspace_size(B, nq, nkv, d)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    plain = torch.zeros((B, nq, d), dtype=torch.float32, device="cuda")
    kmr.kmr_decode_attn(torch.from_numpy(q).cuda(), torch.from_numpy(full_k.view(np.int16)).cuda(),
                        torch.from_numpy(full_v.view(np.int16)).cuda(),
                        torch.arange(B, dtype=torch.int32, device="cuda"),
                        torch.tensor(cpos, dtype=torch.int32, device="cuda"), B, nq, nkv, d, S, slots,
                        1.0 / math.sqrt(d), plain, ws, ws_bytes, torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert kmr.kmr_last_device_error() == 0
    assert rel_l2(out, plain.cpu().numpy()) <= 1e-5
    ref = _oracle(q, kc, vc, list(range(B)), cpos, B, P)
    assert rel_l2(out, ref) <= 1e-4


def test_cascade_row_result_independent_of_the_other_rows(torch):
    r = np.random.default_rng(4)
    B, nq, nkv, d, S, P = 5, 16, 8, 128, 512, 300
    cpos = [300, 333, 400, 511, 301]
    slots = B + 1
    q, kc, vc = _setup(r, B, nq, nkv, d, S, slots, B, P, cpos, list(range(B)))
    out, err = _run(torch, q, kc, vc, list(range(B)), cpos, B, P, nq, nkv, d, S, slots)
    assert err == 0
    again, _ = _run(torch, q, kc, vc, list(range(B)), cpos, B, P, nq, nkv, d, S, slots)
    assert np.array_equal(out, again)                       # run to run
    for b in (0, 3):
        one, _ = _run(torch, q[b:b + 1], kc, vc, [b], [cpos[b]], B, P, nq, nkv, d, S, slots)
        assert np.array_equal(one[0], out[b])               # bitwise, alone or with others


def test_cascade_bad_rows_get_zeros_and_an_error(torch):
    r = np.random.default_rng(5)
    B, nq, nkv, d, S, P = 3, 4, 2, 64, 128, 40
    slots = 4
    q, kc, vc = _setup(r, B, nq, nkv, d, S, slots, 3, P, [40, 50, 60], [0, 1, 2])
    # row 1: own slot out of range; row 2: cache_position below the prefix
    out, err = _run(torch, q, kc, vc, [0, 9, 2], [40, 50, 39], 3, P, nq, nkv, d, S, slots)
    assert err in (kmr.KMR_ERR_SLOT_RANGE, kmr.KMR_ERR_CACHE_FULL)
    assert not out[1].any() and not out[2].any() and np.all(np.isfinite(out[0])) and out[0].any()
    ref = _oracle(q[:1], kc, vc, [0], [40], 3, P)
    assert rel_l2(out[0], ref[0]) <= 1e-4
