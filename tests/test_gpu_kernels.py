"""GPU parity of the packing, int4 GEMV and decode-attention kernels against the
CPU oracle, through the C ABI."""
import math

import numpy as np
import pytest

import int4_weight_only_group_gb300 as kmr
from oracle import decoder as od
from oracle import packspec
from gpu_helpers import REL_L2_TOL, rel_l2, require_gpu
from workloads import BF16_NAN, f32_to_bf16_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return require_gpu()


def _canon(seed, N, K):
    r = np.random.default_rng(seed)
    q = r.integers(0, 16, (N, K), dtype=np.uint8)
    s = f32_to_bf16_bits(r.uniform(0.002, 0.02, (N, K // 128)).astype(np.float32))
    z = f32_to_bf16_bits((r.standard_normal((N, K // 128)) * 0.005).astype(np.float32))
    return q, s, z


def _device_pack(torch, q, s, z, flags=0):
    N, K = q.shape
    size = kmr.kmr_packed_size(N, K, 128)
    dq, ds, dz = (torch.from_numpy(a).cuda() for a in (q, s.view(np.int16), z.view(np.int16)))
    out = torch.zeros(size, dtype=torch.uint8, device="cuda")
    kmr.kmr_pack_int4(dq, ds, dz, N, K, 128, flags, out, size, 1, torch.cuda.current_stream())
    torch.cuda.synchronize()
    return out


# ------------------------------------------------------------------ packing (bit-exact)
@pytest.mark.parametrize("N,K,flags", [(13, 256, 0), (64, 768, 0), (4096, 2048, 0), (2048, 6144, 0),
                                       (12288, 2048, 1), (32, 640, 1)])
def test_device_pack_bit_exact(torch, N, K, flags):
    q, s, z = _canon(N + K, N, K)
    dev = _device_pack(torch, q, s, z, flags).cpu().numpy()
    host = np.zeros_like(dev)
    kmr.kmr_pack_int4(q, s, z, N, K, 128, flags, host, host.size, 0)
    assert np.array_equal(dev, host)
    if N * K <= 2048 * 64:
        assert np.array_equal(dev, packspec.pack_int4_spec(q, s, z, gate_up=bool(flags)))
    dq = torch.zeros((N, K), dtype=torch.uint8, device="cuda")
    ds = torch.zeros((N, K // 128), dtype=torch.int16, device="cuda")
    dz = torch.zeros_like(ds)
    kmr.kmr_unpack_int4(torch.from_numpy(dev).cuda(), dev.size, N, K, 128, flags, dq, ds, dz, 1)
    torch.cuda.synchronize()
    assert np.array_equal(dq.cpu().numpy(), q)
    assert np.array_equal(ds.cpu().numpy().view(np.uint16), s)
    assert np.array_equal(dz.cpu().numpy().view(np.uint16), z)


# ------------------------------------------------------------------ int4 GEMV
def _gemv(torch, packed, N, K, x, epi=kmr.KMR_EPI_NONE, flags=0, y0=None, poison=None):
    M = x.shape[0]
    ncol = N // 2 if epi == kmr.KMR_EPI_SILU_MUL else N
    y = torch.from_numpy(y0).cuda() if y0 is not None else torch.zeros((M, ncol), dtype=torch.float32, device="cuda")
    xd = torch.from_numpy(np.ascontiguousarray(x, np.float32)).cuda()
    if poison is not None:
        kmr.kmr_smem_poison(poison, torch.cuda.current_stream())
    kmr.kmr_int4_gemv(packed, N, K, 128, flags, xd, M, y, epi, torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert kmr.kmr_last_device_error() == 0
    return y.cpu().numpy()


def _rows(N, limit=768):
    if N <= limit:
        return np.arange(N)
    r = np.random.default_rng(N)
    return np.unique(np.concatenate([np.arange(8), np.arange(N - 8, N), r.choice(N, limit - 16, replace=False)]))


SHAPES = [(8, 128), (13, 256), (512, 256), (768, 768), (4096, 2048), (2048, 2048), (12288, 2048), (2048, 6144),
          (24, 8192)]


@pytest.mark.parametrize("N,K", SHAPES)
@pytest.mark.parametrize("M", [1, 2, 4, 8, 16])
def test_int4_gemv_matches_oracle(torch, N, K, M):
    q, s, z = _canon(7 * N + K, N, K)
    packed = _device_pack(torch, q, s, z)
    x = np.random.default_rng(M).standard_normal((M, K)).astype(np.float32)
    y = _gemv(torch, packed, N, K, x)
    rows = _rows(N)
    ref = od.int4_linear(x.astype(np.float64), q[rows], s[rows], z[rows], 128)
    err = rel_l2(y[:, rows], ref)
    assert err <= REL_L2_TOL, err
    assert err <= 2e-3, f"unexpectedly large error {err}"


def test_int4_gemv_full_vocab_shape_sampled(torch):
    N, K = 151936, 2048
    q, s, z = _canon(5, N, K)
    packed = _device_pack(torch, q, s, z)
    for M in (1, 16):
        x = np.random.default_rng(M).standard_normal((M, K)).astype(np.float32)
        y = _gemv(torch, packed, N, K, x)
        rows = _rows(N, 1024)
        assert rel_l2(y[:, rows], od.int4_linear(x.astype(np.float64), q[rows], s[rows], z[rows], 128)) <= REL_L2_TOL


def test_int4_gemv_epilogues(torch):
    N, K, M = 2048, 6144, 4
    q, s, z = _canon(11, N, K)
    packed = _device_pack(torch, q, s, z)
    r = np.random.default_rng(3)
    x = r.standard_normal((M, K)).astype(np.float32)
    y0 = r.standard_normal((M, N)).astype(np.float32)
    y = _gemv(torch, packed, N, K, x, kmr.KMR_EPI_RESIDUAL, y0=y0)
    assert rel_l2(y, y0 + od.int4_linear(x.astype(np.float64), q, s, z, 128)) <= REL_L2_TOL
    # gate/up with SiLU(gate) * up
    I = 1536
    q, s, z = _canon(12, 2 * I, 2048)
    packed = _device_pack(torch, q, s, z, kmr.KMR_PACK_GATE_UP)
    x = r.standard_normal((M, 2048)).astype(np.float32)
    y = _gemv(torch, packed, 2 * I, 2048, x, kmr.KMR_EPI_SILU_MUL, flags=kmr.KMR_PACK_GATE_UP)
    gu = od.int4_linear(x.astype(np.float64), q, s, z, 128)
    assert rel_l2(y, od.silu(gu[:, :I]) * gu[:, I:]) <= REL_L2_TOL


def test_int4_gemv_special_cases(torch):
    # The tensor cores accumulate (1024 + c q) x' in float32 and the 1024 offset is removed
    # once per group (y = s (D - 1024 X) / c + (z - 8 s) X), so an all-zero weight row leaves
    # a cancellation residue of order (k-steps per group) * 2^-24 * 1032 * |x| per group:
    # bounded here by 2^-14 * s * ||x||_1, four orders of magnitude below a wrong term.
    N, K = 64, 1024
    q = np.full((N, K), 8, np.uint8)
    s = f32_to_bf16_bits(np.full((N, K // 128), 0.5, np.float32))
    z = np.zeros((N, K // 128), np.uint16)
    x = np.random.default_rng(0).standard_normal((3, K)).astype(np.float32)
    bound = 2.0 ** -14 * 0.5 * np.abs(x).sum(axis=1, keepdims=True)
    y = _gemv(torch, _device_pack(torch, q, s, z), N, K, x)
    assert np.all(np.abs(y) <= bound)                                                     # W = 0
    q[5, 777] = 9                                                                         # one code 9
    y = _gemv(torch, _device_pack(torch, q, s, z), N, K, x)
    assert np.allclose(y[:, 5], 0.5 * x[:, 777], rtol=1e-3, atol=bound[:, 0].max())
    assert np.all(np.abs(y[:, np.arange(N) != 5]) <= bound)
    assert np.all(_gemv(torch, _device_pack(torch, q, s, z), N, K, np.zeros((2, K), np.float32)) == 0.0)


def test_int4_gemv_deterministic_and_batch_invariant(torch):
    N, K = 4096, 2048
    q, s, z = _canon(21, N, K)
    packed = _device_pack(torch, q, s, z)
    x = np.random.default_rng(9).standard_normal((16, K)).astype(np.float32)
    y16 = _gemv(torch, packed, N, K, x)
    assert np.array_equal(y16, _gemv(torch, packed, N, K, x))
    for m in range(0, 16, 5):
        assert np.array_equal(_gemv(torch, packed, N, K, x[m:m + 1])[0], y16[m])
    assert np.array_equal(_gemv(torch, packed, N, K, x[4:8]), y16[4:8])


# Shared memory filled with NaN / Inf / large-value bits before the launch must not change a
# single output bit: no kernel may read shared memory it did not write in the same launch.
POISON_PATTERNS = (0xFFFFFFFF, 0x7F807F80, 0x7BFF7BFF)


@pytest.mark.parametrize("N,K,M,epi", [(13, 256, 3, kmr.KMR_EPI_NONE), (768, 768, 1, kmr.KMR_EPI_NONE),
                                       (4096, 2048, 4, kmr.KMR_EPI_RESIDUAL), (2048, 6144, 8, kmr.KMR_EPI_NONE),
                                       (512, 256, 5, kmr.KMR_EPI_SILU_MUL), (12288, 2048, 2, kmr.KMR_EPI_SILU_MUL)])
def test_int4_gemv_ignores_stale_shared_memory(torch, N, K, M, epi):
    flags = kmr.KMR_PACK_GATE_UP if epi == kmr.KMR_EPI_SILU_MUL else 0
    q, s, z = _canon(3 * N + K, N, K)
    packed = _device_pack(torch, q, s, z, flags)
    x = np.random.default_rng(N + M).standard_normal((M, K)).astype(np.float32)
    y0 = np.random.default_rng(1).standard_normal((M, N)).astype(np.float32) if epi == kmr.KMR_EPI_RESIDUAL else None
    clean = _gemv(torch, packed, N, K, x, epi, flags, y0)
    assert np.all(np.isfinite(clean))
    for pat in POISON_PATTERNS:
        assert np.array_equal(_gemv(torch, packed, N, K, x, epi, flags, y0, poison=pat), clean), hex(pat)


# ------------------------------------------------------------------ decode attention
def _attn_case(torch, B, nq, nkv, d, S, slots, cpos, slot_ids, seed=0, poison=None):
    r = np.random.default_rng(seed)
    q = r.standard_normal((B, nq, d)).astype(np.float32)
    kc = np.full((slots, nkv, S, d), BF16_NAN, np.uint16)
    vc = np.full((slots, nkv, S, d), BF16_NAN, np.uint16)
    for b in range(B):
        n = cpos[b] + 1
        kc[slot_ids[b], :, :n] = f32_to_bf16_bits(r.standard_normal((nkv, n, d)).astype(np.float32))
        vc[slot_ids[b], :, :n] = f32_to_bf16_bits(r.standard_normal((nkv, n, d)).astype(np.float32))
    ws_bytes = kmr.kmr_decode_attn_workspace_size(B, nq, nkv, d)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    out = torch.zeros((B, nq, d), dtype=torch.float32, device="cuda")
    dk = torch.from_numpy(kc.view(np.int16)).cuda()
    dv = torch.from_numpy(vc.view(np.int16)).cuda()
    if poison is not None:
        kmr.kmr_smem_poison(poison, torch.cuda.current_stream())
    kmr.kmr_decode_attn(torch.from_numpy(q).cuda(), dk, dv, torch.tensor(slot_ids, dtype=torch.int32, device="cuda"),
                        torch.tensor(cpos, dtype=torch.int32, device="cuda"), B, nq, nkv, d, S, slots,
                        1.0 / math.sqrt(d), out, ws, ws_bytes, torch.cuda.current_stream())
    torch.cuda.synchronize()
    err = kmr.kmr_last_device_error()
    cnt_bytes = (B * nkv * 4 + 15) // 16 * 16
    assert int(ws[-cnt_bytes:].sum().item()) == 0      # arrival counters left zeroed
    ref = np.stack([od.decode_attention(q[b].astype(np.float64),
                                        od.bf16_to_f64(kc[slot_ids[b], :, :cpos[b] + 1]),
                                        od.bf16_to_f64(vc[slot_ids[b], :, :cpos[b] + 1])) for b in range(B)])
    return out.cpu().numpy(), ref, err


@pytest.mark.parametrize("d,nq,nkv", [(128, 16, 8), (64, 4, 2), (128, 8, 8), (64, 16, 4)])
def test_decode_attn_matches_oracle(torch, d, nq, nkv):
    cpos = [0, 1, 15, 16, 31, 32, 33, 255, 599, 1023]
    B = len(cpos)
    slots = B + 2
    slot_ids = list(np.random.default_rng(1).permutation(slots)[:B])
    out, ref, err = _attn_case(torch, B, nq, nkv, d, 1024, slots, cpos, slot_ids)
    assert err == 0
    assert np.all(np.isfinite(out))                   # NaN-filled unfilled positions never read
    assert rel_l2(out, ref) <= 1e-4                     # well inside the 1e-2 bar
    for b in range(B):
        assert rel_l2(out[b], ref[b]) <= 1e-4


@pytest.mark.parametrize("L", [256, 1024, 4096, 8192])
@pytest.mark.parametrize("B", [1, 4, 16])
def test_decode_attn_sweep_shapes(torch, B, L):
    cpos = [L - 1 - 7 * b for b in range(B)]
    out, ref, err = _attn_case(torch, B, 16, 8, 128, L, B, cpos, list(range(B)), seed=L + B)
    assert err == 0 and rel_l2(out, ref) <= REL_L2_TOL


def test_decode_attn_single_token_and_determinism(torch):
    out, ref, _ = _attn_case(torch, 3, 16, 8, 128, 64, 3, [0, 40, 63], [2, 0, 1], seed=5)
    assert rel_l2(out, ref) <= 1e-5
    again, _, _ = _attn_case(torch, 3, 16, 8, 128, 64, 3, [0, 40, 63], [2, 0, 1], seed=5)
    assert np.array_equal(out, again)


@pytest.mark.parametrize("nkv,S", [(4, 1024), (8, 4096), (8, 8192)])   # 8-/16-position chunks; 8192: global merge
def test_decode_attn_ignores_stale_shared_memory(torch, nkv, S):
    cpos = [0, 6, 15, 16, 70, 127, 1000, S - 1]   # lone last positions, exact splits, ragged tails
    args = (torch, len(cpos), 16, nkv, 128, S, len(cpos), cpos, list(range(len(cpos))))
    clean, ref, err = _attn_case(*args, seed=11)
    assert err == 0 and np.all(np.isfinite(clean)) and rel_l2(clean, ref) <= 1e-4
    for pat in POISON_PATTERNS:
        out, _, err = _attn_case(*args, seed=11, poison=pat)
        assert err == 0 and np.array_equal(out, clean), hex(pat)


@pytest.mark.parametrize("S", [1024, 8192])        # cluster-merged splits; workspace-merged splits
def test_decode_attn_batch_invariant(torch, S):
    """A row's output is bitwise the same alone (B = 1) and inside a batch of 5, whatever the
    other rows hold: the split plan depends on the row's length, n_kv and max_len only."""
    nq, nkv, d, B = 16, 8, 128, 5
    r = np.random.default_rng(S)
    cpos = [S - 1, 3, S // 2 + 5, 70, S - 300]
    kc = f32_to_bf16_bits(r.standard_normal((B, nkv, S, d)).astype(np.float32))
    vc = f32_to_bf16_bits(r.standard_normal((B, nkv, S, d)).astype(np.float32))
    q = torch.from_numpy(r.standard_normal((B, nq, d)).astype(np.float32)).cuda()
    dk = torch.from_numpy(kc.view(np.int16)).cuda()
    dv = torch.from_numpy(vc.view(np.int16)).cuda()

    def run(rows):
        n = len(rows)
        ws_bytes = kmr.kmr_decode_attn_workspace_size(n, nq, nkv, d)
        ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
        out = torch.zeros((n, nq, d), dtype=torch.float32, device="cuda")
        kmr.kmr_decode_attn(q[rows].contiguous(), dk, dv, torch.tensor(rows, dtype=torch.int32, device="cuda"),
                            torch.tensor([cpos[i] for i in rows], dtype=torch.int32, device="cuda"), n, nq, nkv, d,
                            S, B, 1.0 / math.sqrt(d), out, ws, ws_bytes, torch.cuda.current_stream())
        torch.cuda.synchronize()
        assert kmr.kmr_last_device_error() == 0
        return out.cpu().numpy()

    full = run(list(range(B)))
    for i in range(B):
        assert np.array_equal(run([i])[0], full[i]), i
    assert np.array_equal(run([3, 0])[1], full[0])


def test_decode_attn_bad_rows_flag_errors(torch):
    out, _, err = _attn_case(torch, 2, 16, 8, 128, 64, 2, [10, 20], [0, 1])
    assert err == 0
    torch_ = torch
    ws_bytes = kmr.kmr_decode_attn_workspace_size(2, 16, 8, 128)
    ws = torch_.zeros(ws_bytes, dtype=torch_.uint8, device="cuda")
    q = torch_.ones((2, 16, 128), device="cuda")
    cache = torch_.zeros((2, 8, 64, 128), dtype=torch_.int16, device="cuda")
    res = torch_.full((2, 16, 128), 7.0, device="cuda")
    for slot, pos, code in (([0, 5], [3, 3], kmr.KMR_ERR_SLOT_RANGE), ([0, 1], [3, 64], kmr.KMR_ERR_CACHE_FULL)):
        kmr.kmr_decode_attn(q, cache, cache, torch_.tensor(slot, dtype=torch_.int32, device="cuda"),
                            torch_.tensor(pos, dtype=torch_.int32, device="cuda"), 2, 16, 8, 128, 64, 2, 0.1, res,
                            ws, ws_bytes)
        assert kmr.kmr_last_device_error() == code
        assert float(res[1].abs().sum()) == 0.0         # the bad row is zeroed, not read


def test_bounded_wait_gives_up_with_a_status(torch):
    """Failure detection without a fault: a device wait that nothing completes gives up after
    its limit and reports KMR_ERR_DEVICE_TIMEOUT through the error word; the context stays
    usable (a GEMV afterwards still matches the oracle)."""
    import time
    assert kmr.kmr_last_device_error() == 0
    t0 = time.perf_counter()
    kmr.kmr_selftest_wait_timeout(2_000_000)                       # 2 ms
    assert kmr.kmr_last_device_error() == kmr.KMR_ERR_DEVICE_TIMEOUT
    assert time.perf_counter() - t0 < 10.0
    assert kmr.kmr_last_device_error() == 0                        # reading clears the word
    with pytest.raises(kmr.KmrError):
        kmr.kmr_selftest_wait_timeout(10)                          # limit below 1 us: refused on the host
    q, s, z = _canon(3, 64, 256)
    x = np.random.default_rng(3).standard_normal((2, 256)).astype(np.float32)
    y = _gemv(torch, _device_pack(torch, q, s, z), 64, 256, x)
    assert rel_l2(y, od.int4_linear(x.astype(np.float64), q, s, z, 128)) <= REL_L2_TOL
    assert kmr.kmr_last_device_error() == 0
