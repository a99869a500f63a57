"""kmr_decode_attn_noalloc: the decode attention for callers that cannot allocate
device memory (graph capture in global mode, engines that own the whole device
heap, loops that cannot afford cudaMalloc's implicit synchronisation).

Its scratch is one fixed array shared by every call, so these tests check it call
after call: against kmr_decode_attn with a caller workspace (the attention
tolerance: the two merge the splits in different forms), against the oracle's
plain definition element by element, at both head sizes, at the largest batch
that fits the array and one row beyond it.  This file is collected last so a
failure here never hides the rest of the suite."""
import math

import numpy as np
import pytest

import int4_weight_only_group_gb300 as kmr
from gpu_helpers import REL_L2_TOL, rel_l2, require_gpu
from oracle import decoder as od
from workloads import f32_to_bf16_bits

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 4 << 20          # KMR_NOALLOC_ATTN_SCRATCH_BYTES
ATTN_TOL = 1e-4                  # fp32 attention against the fp64 definition


def _inputs(torch, seed, B, nq, nkv, d, S):
    r = np.random.default_rng(seed)
    cpos = r.integers(0, S, size=B).astype(np.int32)
    slot_ids = r.permutation(B).astype(np.int32)
    qh = r.standard_normal((B, nq, d)).astype(np.float32)
    kc = f32_to_bf16_bits(r.standard_normal((B, nkv, S, d)).astype(np.float32))
    vc = f32_to_bf16_bits(r.standard_normal((B, nkv, S, d)).astype(np.float32))
    dev = (torch.from_numpy(qh).cuda(), torch.from_numpy(kc.view(np.int16)).cuda(),
           torch.from_numpy(vc.view(np.int16)).cuda(), torch.from_numpy(slot_ids).cuda(),
           torch.from_numpy(cpos).cuda())
    return dev, (qh, kc, vc, slot_ids, cpos)


def _oracle(host, B):
    qh, kc, vc, slot_ids, cpos = host
    out = []
    for b in range(B):
        t = int(cpos[b]) + 1
        out.append(od.decode_attention(qh[b].astype(np.float64), od.bf16_to_f64(kc[slot_ids[b], :, :t]),
                                       od.bf16_to_f64(vc[slot_ids[b], :, :t])))
    return np.stack(out)


def _max_batch(torch, nq, nkv, d):
    """Largest B whose split partials and arrival counters fit the fixed array (the limit the
    header states: splits = ceil(SMs / n_kv) capped at 32)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    splits = min(32, max(1, -(-sms // nkv)))
    B = 1
    while True:
        nb = B + 1
        part = (nb * nq * splits * (d + 2) * 4 + 15) & ~15
        if part + nb * nkv * 4 > SCRATCH_BYTES:
            return B
        B = nb


def test_noalloc_attention_matches_workspace_attention_two_calls_in_a_row():
    torch = require_gpu()
    B, nq, nkv, d, S = 4, 16, 8, 128, 1024
    scale = 1.0 / math.sqrt(d)
    ws_bytes = kmr.kmr_decode_attn_workspace_size(B, nq, nkv, d)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    for call, seed in enumerate((11, 12)):        # two calls in a row, different inputs
        (q, kc, vc, slots, cpos), _ = _inputs(torch, seed, B, nq, nkv, d, S)
        ref = torch.zeros((B, nq, d), dtype=torch.float32, device="cuda")
        kmr.kmr_decode_attn(q, kc, vc, slots, cpos, B, nq, nkv, d, S, B, scale, ref, ws, ws_bytes)
        out = torch.full((B, nq, d), float("nan"), dtype=torch.float32, device="cuda")
        kmr.kmr_decode_attn_noalloc(q, kc, vc, slots, cpos, B, nq, nkv, d, S, B, scale, out)
        torch.cuda.synchronize()
        assert kmr.kmr_last_device_error() == 0
        o, r = out.cpu().numpy(), ref.cpu().numpy()
        assert np.all(np.isfinite(o)), f"call {call}"
        assert rel_l2(o, r) <= REL_L2_TOL, f"call {call}: {rel_l2(o, r)}"


@pytest.mark.parametrize("nq,nkv,d,S", [(16, 8, 128, 1024), (8, 4, 64, 512)])
def test_noalloc_attention_matches_oracle_at_the_largest_batch_that_fits(nq, nkv, d, S):
    torch = require_gpu()
    B = _max_batch(torch, nq, nkv, d)
    scale = 1.0 / math.sqrt(d)
    for call, seed in enumerate((21, 22)):        # two calls in a row on the shared array
        (q, kc, vc, slots, cpos), host = _inputs(torch, seed + d, B, nq, nkv, d, S)
        out = torch.full((B, nq, d), float("nan"), dtype=torch.float32, device="cuda")
        kmr.kmr_decode_attn_noalloc(q, kc, vc, slots, cpos, B, nq, nkv, d, S, B, scale, out)
        torch.cuda.synchronize()
        assert kmr.kmr_last_device_error() == 0
        o = out.cpu().numpy().astype(np.float64)
        want = _oracle(host, B)
        for b in range(B):
            assert rel_l2(o[b], want[b]) <= ATTN_TOL, f"call {call} row {b}: {rel_l2(o[b], want[b])}"
    # one row more than the array holds: rejected before any launch
    rc = kmr.lib().kmr_decode_attn_noalloc(1, 1, 1, 1, 1, B + 1, nq, nkv, d, S, B + 1, scale, 1, None)
    assert rc == kmr.KMR_ERR_SHAPE


def test_noalloc_attention_rejects_problems_beyond_its_scratch():
    require_gpu()
    # 4096 rows x 16 heads x (128 + 2) floats x >= 1 split is far beyond the fixed scratch
    rc = kmr.lib().kmr_decode_attn_noalloc(1, 1, 1, 1, 1, 4096, 16, 8, 128, 64, 1, 0.1, 1, None)
    assert rc == kmr.KMR_ERR_SHAPE
