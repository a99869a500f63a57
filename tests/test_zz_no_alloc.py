"""kmr_decode_attn_noalloc: the decode attention for callers that cannot allocate
device memory (graph capture in global mode, engines that own the whole device
heap, loops that cannot afford cudaMalloc's implicit synchronisation).

It must give the same results as kmr_decode_attn with a caller workspace, call
after call, although its scratch is one fixed array shared by every call.  This
file is collected last so a failure here never hides the rest of the suite."""
import math

import numpy as np
import pytest

import int4_weight_only_group_gb300 as kmr
from gpu_helpers import REL_L2_TOL, rel_l2, require_gpu
from workloads import f32_to_bf16_bits

pytestmark = pytest.mark.gpu


def _inputs(torch, seed, B, nq, nkv, d, S):
    r = np.random.default_rng(seed)
    cpos = r.integers(0, S, size=B).astype(np.int32)
    slot_ids = r.permutation(B).astype(np.int32)
    q = torch.from_numpy(r.standard_normal((B, nq, d)).astype(np.float32)).cuda()
    kc = f32_to_bf16_bits(r.standard_normal((B, nkv, S, d)).astype(np.float32))
    vc = f32_to_bf16_bits(r.standard_normal((B, nkv, S, d)).astype(np.float32))
    return (q, torch.from_numpy(kc.view(np.int16)).cuda(), torch.from_numpy(vc.view(np.int16)).cuda(),
            torch.from_numpy(slot_ids).cuda(), torch.from_numpy(cpos).cuda())


def test_noalloc_attention_matches_workspace_attention_two_calls_in_a_row():
    torch = require_gpu()
    B, nq, nkv, d, S = 4, 16, 8, 128, 1024
    scale = 1.0 / math.sqrt(d)
    ws_bytes = kmr.kmr_decode_attn_workspace_size(B, nq, nkv, d)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    for call, seed in enumerate((11, 12)):        # two calls in a row, different inputs
        q, kc, vc, slots, cpos = _inputs(torch, seed, B, nq, nkv, d, S)
        ref = torch.zeros((B, nq, d), dtype=torch.float32, device="cuda")
        kmr.kmr_decode_attn(q, kc, vc, slots, cpos, B, nq, nkv, d, S, B, scale, ref, ws, ws_bytes)
        out = torch.full((B, nq, d), float("nan"), dtype=torch.float32, device="cuda")
        kmr.kmr_decode_attn_noalloc(q, kc, vc, slots, cpos, B, nq, nkv, d, S, B, scale, out)
        torch.cuda.synchronize()
        assert kmr.kmr_last_device_error() == 0
        o, r = out.cpu().numpy(), ref.cpu().numpy()
        assert np.all(np.isfinite(o)), f"call {call}"
        assert rel_l2(o, r) <= REL_L2_TOL, f"call {call}: {rel_l2(o, r)}"


def test_noalloc_attention_rejects_problems_beyond_its_scratch():
    require_gpu()
    # 4096 rows x 16 heads x (128 + 2) floats x >= 1 split is far beyond the fixed scratch
    rc = kmr.lib().kmr_decode_attn_noalloc(1, 1, 1, 1, 1, 4096, 16, 8, 128, 64, 1, 0.1, 1, None)
    assert rc == kmr.KMR_ERR_SHAPE
