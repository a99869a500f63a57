/*
 * kmr.h — C ABI of the GB300 int4 weight-only, group-wise decode-step library.
 *
 * The method: one greedy decode step of a Qwen3-style text decoder whose
 * attention and MLP linears are stored as int4 codes with a bf16 scale and
 * zero per group of 128 inputs, while embeddings, the tied LM head and the
 * norms stay bf16 ("kaminari — a single-GPU Qwen3-VL inference engine,
 * explained", §07 int4 sidecar quantization; §04 Request lifecycle, decode).
 *
 * Conventions for every entry point
 *   - Return value: KMR_OK (0) or a negative KMR_ERR_* code; arguments are
 *     checked on the host before anything is launched, and a failed check
 *     launches nothing.
 *   - Device pointers are raw CUDA device addresses on the current device;
 *     host pointers are ordinary process memory.  The library never frees or
 *     keeps a pointer the caller passes, except where stated.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Device work is asynchronous on that stream unless the entry
 *     point says it synchronises.
 *   - Kernels that detect bad per-row state at run time (a slot id out of
 *     range, an unfinished row whose cache_position is outside [0, max_len))
 *     skip that row and record the first such error in a device error word
 *     that kmr_model_sync_status() / kmr_last_device_error() return.
 *   - No kernel traps; every device wait is bounded and reports
 *     KMR_ERR_DEVICE_TIMEOUT instead of hanging.
 *
 * Packed int4 layout ("KMR4", version 2; the library's own, not torchao's)
 *   Canonical input: q uint8 [N, K] row-major with values 0..15 (row n =
 *   output feature, column k = input feature), s and z bf16 [N, K / 128].
 *   The dense weight is W[n, k] = (q[n, k] - 8) * s[n, k/128] + z[n, k/128].
 *   Packing (one 32-bit word per lane per 16x16 block: the A fragment of a
 *   16x8x16 tensor-core product):
 *     Rows are grouped in tiles of 16 (N is padded to a multiple of 16 with
 *     q = 8, s = z = 0, i.e. zero weights).  With KMR_PACK_GATE_UP (N a
 *     multiple of 16) the canonical rows [gate (N/2); up (N/2)] are reordered
 *     so that packed tile t holds gate rows 8t..8t+7 then up rows 8t..8t+7.
 *     A tile is K/128 consecutive groups of 1088 bytes; group gr of tile T
 *     starts at T * (K/128) * 1088 + gr * 1088 and holds
 *       bytes [0, 1024): for k-step ks = 0..7 (inputs k0 = 128 gr + 16 ks)
 *         and lane l = 0..31 (g = l / 4, t = l % 4), the little-endian
 *         32-bit word at (ks / 4) * 512 + l * 16 + (ks % 4) * 4 whose
 *         nibbles are, by bit offset (row r of the tile, input k):
 *            0: (g, k0+2t)     16: (g, k0+2t+1)
 *            4: (g+8, k0+2t)   20: (g+8, k0+2t+1)
 *            8: (g, k0+2t+8)   24: (g, k0+2t+9)
 *           12: (g+8, k0+2t+8) 28: (g+8, k0+2t+9)
 *       bytes [1024, 1088): for rows r = 0..15 of the tile, (s bf16, z bf16)
 *         of group gr, little-endian, at 1024 + 4 r.
 *   kmr_packed_size() = ceil(N/16) * (K/128) * 1088
 *                     = ceil(N/16)*16 * (K/2 + 4*K/128) bytes.
 */
#ifndef KMR_H_
#define KMR_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------------ status */
#define KMR_OK                   0
#define KMR_ERR_INVALID_ARG     -1   /* null pointer, bad flag, bad scalar        */
#define KMR_ERR_SHAPE           -2   /* unsupported or inconsistent dimensions    */
#define KMR_ERR_SLOT_RANGE      -3   /* slot id outside [0, slots)                */
#define KMR_ERR_CACHE_FULL      -4   /* unfinished row with cache_position >= max_len */
#define KMR_ERR_NO_PACK         -5   /* a layer's int4 weights were never loaded  */
#define KMR_ERR_CUDA            -6   /* a CUDA runtime call failed                */
#define KMR_ERR_DEVICE_TIMEOUT  -7   /* a bounded device wait gave up             */
#define KMR_ERR_BUFFER_SIZE     -8   /* a caller buffer is smaller than required  */
#define KMR_ERR_BATCH           -9   /* batch outside [1, max_batch]              */

/* Human-readable name of a status code (static string, never NULL). */
const char* kmr_status_string(int status);

/* Library / layout version: returns 2 for the KMR4 v2 packed layout. */
int kmr_layout_version(void);

/* ------------------------------------------------------------------ packing */
#define KMR_PACK_GATE_UP  1   /* interleave [gate; up] halves in blocks of 8 rows */

/* Bytes of the packed form of an [N, K] int4 matrix with the given group
 * (group must be 128; K a multiple of 128).  Returns 0 for unsupported shapes. */
size_t kmr_packed_size(int N, int K, int group);

/* Pack canonical q/s/z (layout above) into `packed` (packed_bytes >=
 * kmr_packed_size).  on_device = 0: all pointers are host memory and the call
 * is synchronous on the host.  on_device = 1: all pointers are device memory
 * and the work is queued on `stream`.  Codes above 15 are rejected on the
 * host path (KMR_ERR_INVALID_ARG); the device path masks them to 4 bits.
 * Bit-exact: kmr_unpack_int4(kmr_pack_int4(x)) == x. */
int kmr_pack_int4(const uint8_t* q, const uint16_t* s_bf16, const uint16_t* z_bf16,
                  int N, int K, int group, int flags,
                  void* packed, size_t packed_bytes, int on_device, void* stream);

/* Inverse of kmr_pack_int4 (same flags, same pointer placement rules). */
int kmr_unpack_int4(const void* packed, size_t packed_bytes, int N, int K, int group, int flags,
                    uint8_t* q, uint16_t* s_bf16, uint16_t* z_bf16, int on_device, void* stream);

/* ------------------------------------------------------------------ int4 GEMV */
#define KMR_EPI_NONE      0   /* y[m, n]  = sum_k x[m, k] W[n, k]                       */
#define KMR_EPI_RESIDUAL  1   /* y[m, n] += sum_k x[m, k] W[n, k]                       */
#define KMR_EPI_SILU_MUL  2   /* packed with KMR_PACK_GATE_UP: y[m, j] = silu(g_j) * u_j,
                                 j < N/2, g = rows [0, N/2), u = rows [N/2, N)         */

/* Dequant-fused int4 GEMV / skinny GEMM ("kaminari", §07 int4 sidecar
 * quantization: decoder linears weight-only int4; §06 The optimization
 * ladder: decode is memory-bandwidth-bound, so the packed weights are
 * streamed once and dequantised in registers).
 *   packed  device, KMR4 layout of W [N, K] (flags as packed)
 *   x       device fp32 [M, K] row-major, 1 <= M <= 16
 *   y       device fp32 [M, N] (or [M, N/2] for KMR_EPI_SILU_MUL), row-major
 *   K <= 8192.  No workspace: each CTA owns whole 16-row tiles.  The
 *   reduction order is fixed (no float atomics): results are bitwise
 *   reproducible and a row's result does not depend on M. */
int kmr_int4_gemv(const void* packed, int N, int K, int group, int flags,
                  const float* x, int M, float* y, int epilogue, void* stream);

/* ------------------------------------------------------------------ attention */
/* Workspace bytes kmr_decode_attn needs (device memory).  The caller
 * zero-fills it once before its first use; its last B*n_kv_heads*4 bytes
 * (rounded up to 16) are arrival counters that every successful call leaves
 * zeroed, the rest is scratch.  Calls sharing one workspace must not overlap. */
size_t kmr_decode_attn_workspace_size(int B, int n_q_heads, int n_kv_heads, int head_dim);

/* GQA decode attention of one token per row over a static, slot-addressable
 * bf16 KV cache ("The Ghost in the Batch", What Attention Does:
 * out = softmax(q K^T / sqrt(d)) V, and the LSE-weighted merge of partial
 * results; "kaminari", §03 StaticKVCache).  Split-KV: each (row, KV head)
 * is cut into position chunks whose partial softmax states are merged in a
 * fixed order; the split plan depends only on the row's own length and on
 * n_kv_heads and max_len (which choose between 8 splits merged inside a
 * thread-block cluster and up to 32 splits merged through the workspace),
 * never on B: a row's result does not depend on the other rows.
 *   q        device fp32 [B, n_q, d]
 *   k_cache, v_cache  device bf16 [slots, n_kv, max_len, d] (one layer)
 *   slot_ids device int32 [B]; cache_position device int32 [B]: row b attends
 *            positions 0..cache_position[b] inclusive of slot slot_ids[b]
 *   scale    softmax scale (1/sqrt(d) for the plain definition)
 *   out      device fp32 [B, n_q, d]
 *   Query head i reads KV head i / (n_q / n_kv).  head_dim must be 64 or 128.
 *   Rows with a slot or position out of range are skipped (output zeros) and
 *   set the error word read by kmr_last_device_error(). */
int kmr_decode_attn(const float* q, const uint16_t* k_cache, const uint16_t* v_cache,
                    const int32_t* slot_ids, const int32_t* cache_position,
                    int B, int n_q_heads, int n_kv_heads, int head_dim, int max_len, int slots,
                    float scale, float* out, void* workspace, size_t workspace_bytes, void* stream);

/* Shared-prefix (cascade) decode attention ("The Ghost in the Batch", The
 * Optimization That Changes Everything: the shared prefix is attended once
 * for all queries, each request's own suffix separately, and the two partial
 * results merged with their log-sum-exp weights).  Row b attends positions
 * [0, prefix_len) of cache row prefix_slot followed by positions
 * [prefix_len, cache_position[b]] of its own row slot_ids[b] (its own
 * positions below prefix_len are not read); the result equals kmr_decode_attn
 * over that concatenated context up to the order of the sums.  The prefix's K
 * and V are read from memory once per call, not once per row.
 *   q, out, slot_ids, cache_position, k_cache, v_cache, scale, head shapes:
 *            as kmr_decode_attn
 *   prefix_slot  cache row holding the shared prefix, 0 <= prefix_slot < slots
 *   prefix_len   shared positions, 0 <= prefix_len < max_len (0: no prefix,
 *                plain attention over each row's own positions)
 *   workspace    device scratch of kmr_decode_attn_cascade_workspace_size()
 *                bytes (same B, heads, head_dim and prefix_len; may be NULL
 *                when prefix_len is 0); no initialisation needed
 * Two kernel launches queued on `stream`, no synchronisation; the split plan
 * of the prefix depends only on prefix_len, n_kv_heads and the GPU, so a row's
 * result does not depend on the other rows of the call.  Host errors:
 * KMR_ERR_INVALID_ARG, KMR_ERR_BATCH, KMR_ERR_SHAPE (as kmr_decode_attn),
 * KMR_ERR_SLOT_RANGE (prefix_slot), KMR_ERR_CACHE_FULL (prefix_len >= max_len),
 * KMR_ERR_BUFFER_SIZE.  Rows whose slot is out of range or whose
 * cache_position lies outside [prefix_len, max_len) get zeros and set the
 * error word read by kmr_last_device_error(). */
size_t kmr_decode_attn_cascade_workspace_size(int B, int n_q_heads, int n_kv_heads, int head_dim, int prefix_len);
int kmr_decode_attn_cascade(const float* q, const uint16_t* k_cache, const uint16_t* v_cache,
                            const int32_t* slot_ids, const int32_t* cache_position, int prefix_slot,
                            int prefix_len, int B, int n_q_heads, int n_kv_heads, int head_dim, int max_len,
                            int slots, float scale, float* out, void* workspace, size_t workspace_bytes,
                            void* stream);

/* Fixed device scratch of kmr_decode_attn_noalloc, in bytes (4 MiB). */
#define KMR_NOALLOC_ATTN_SCRATCH_BYTES (4u << 20)

/* kmr_decode_attn without a workspace argument, for callers that cannot
 * allocate device memory: code running while a CUDA graph is captured in
 * global mode, engines whose memory planner owns the whole device heap, and
 * latency-critical loops that cannot afford cudaMalloc's implicit device
 * synchronisation.  The pages this library follows have no counterpart of
 * this entry point; it exists only for such callers.
 *   Same arguments and layouts as kmr_decode_attn, minus the workspace.  It
 *   always runs the global-merge form (splits = ceil(SM count / n_kv_heads),
 *   capped at 32, each writing its partial state to the array, the last CTA
 *   of a (row, KV head) to arrive merging them in split order), whereas
 *   kmr_decode_attn takes the cluster-merged form for most shapes: the two
 *   agree within the attention tolerance, not bit for bit, and both match the
 *   plain definition (relative L2 <= 1e-4 in the tests).  The split partials
 *   live in one fixed array inside the
 *   library's device image (KMR_NOALLOC_ATTN_SCRATCH_BYTES, held by every GPU
 *   that loads the library until the process exits); the call allocates
 *   nothing, and clears the array's arrival counters with cudaMemsetAsync on
 *   `stream` before launching.
 *   Limit: B * n_q_heads * splits * (head_dim + 2) * 4 bytes (rounded up to
 *   16) + B * n_kv_heads * 4 bytes must fit the array, where splits =
 *   ceil(SM count / n_kv_heads) capped at 32 (19 for 8 KV heads on a 152-SM
 *   GB300); larger problems return KMR_ERR_SHAPE and launch nothing.
 *   Every call on a device shares the array and it keeps the last call's
 *   contents, so calls that overlap on the GPU race: order them on one stream.
 *   The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current) and caches it; make that
 *   first call before any stream capture. */
int kmr_decode_attn_noalloc(const float* q, const uint16_t* k_cache, const uint16_t* v_cache,
                            const int32_t* slot_ids, const int32_t* cache_position,
                            int B, int n_q_heads, int n_kv_heads, int head_dim, int max_len, int slots,
                            float scale, float* out, void* stream);

/* Error word of the standalone kernels (kmr_int4_gemv, kmr_decode_attn) on the
 * current device: synchronises the device, returns the first recorded
 * KMR_ERR_* (or KMR_OK) and clears it. */
int kmr_last_device_error(void);

/* ------------------------------------------------------------------ model */
typedef struct kmr_model_config {
    int hidden;            /* H                                    */
    int n_q_heads;         /* query heads                          */
    int n_kv_heads;        /* key/value heads (GQA)                */
    int head_dim;          /* d: 64 or 128                         */
    int intermediate;      /* I (MLP)                              */
    int vocab;             /* V (tied embedding / LM head rows)    */
    int n_layers;          /* L                                    */
    int group;             /* int4 group along K: 128              */
    float eps;             /* RMSNorm epsilon                      */
    float rope_theta;      /* M-RoPE base                          */
    int mrope_sections[3]; /* frequencies driven by T, H, W; sum = d/2 */
    int qk_norm;           /* 1: per-head RMSNorm of q and k before the rotary embedding */
    int eos_id;            /* token that finishes a row; -1: none  */
    int pad_id;            /* token emitted by finished rows       */
    int max_len;           /* static KV cache positions per slot   */
    int slots;             /* physical cache rows                  */
    int max_batch;         /* largest B a step may use (<= 16)     */
} kmr_model_config;

typedef struct kmr_model kmr_model;

/* Create a model on the current device: allocates (once) the packed weights,
 * the bf16 KV cache [L][slots][n_kv][max_len][d] for K and for V (zero-filled),
 * and all step scratch.  No allocation happens per step ("kaminari", §03: the
 * static cache is preallocated and mutated in place). */
int kmr_model_create(const kmr_model_config* cfg, kmr_model** out);
int kmr_model_destroy(kmr_model* m);

/* Load one int4 linear of one layer from canonical host arrays (layout above).
 * which: 0 = qkv [(nq+2nkv)d, H], 1 = o [H, nq d], 2 = gate_up [2I, H],
 * 3 = down [H, I].  Fused rows follow qkv = [q; k; v], gate_up = [gate; up].
 * Synchronous. */
#define KMR_W_QKV 0
#define KMR_W_O 1
#define KMR_W_GATE_UP 2
#define KMR_W_DOWN 3
int kmr_model_set_linear(kmr_model* m, int layer, int which,
                         const uint8_t* q, const uint16_t* s_bf16, const uint16_t* z_bf16);

/* Load an RMSNorm weight (bf16 host array).  which: 0 = input [H],
 * 1 = post-attention [H], 2 = q-norm [d], 3 = k-norm [d]; layer = -1 with
 * which = 0 loads the final norm [H].  Synchronous. */
#define KMR_N_INPUT 0
#define KMR_N_POST 1
#define KMR_N_Q 2
#define KMR_N_K 3
int kmr_model_set_norm(kmr_model* m, int layer, int which, const uint16_t* w_bf16);

/* Load the tied bf16 embedding / LM head [V, H] from host memory.  Synchronous. */
int kmr_model_set_embedding(kmr_model* m, const uint16_t* e_bf16);

/* Write positions [0, length) of one layer's K and V cache rows of a slot
 * from host bf16 arrays [n_kv, length, d] (a prefill stand-in).  Synchronous. */
int kmr_model_set_kv(kmr_model* m, int layer, int slot, int length,
                     const uint16_t* k_bf16, const uint16_t* v_bf16);

/* Prefill scratch: device memory for chunks of up to max_tokens prompt
 * positions (residual, QKV, attention and MLP rows of the chunk), allocated
 * once here, synchronously (a larger request replaces the scratch; a smaller
 * one keeps it).  No counterpart in the pages' API: it keeps kmr_prefill free of
 * allocation.  Errors: KMR_ERR_INVALID_ARG (max_tokens < 1),
 * KMR_ERR_CACHE_FULL (max_tokens > max_len), KMR_ERR_CUDA. */
int kmr_model_reserve_prefill(kmr_model* m, int max_tokens);

/* Text prefill of one chunk of one sequence ("kaminari", §04 Request
 * lifecycle: prefill runs the prompt through the decoder once, fills the static
 * cache and yields the first generated token from the last prompt position's
 * logits — logits_to_keep = 1).  Token i of the chunk is written to cache row
 * `slot` at position start_pos + i in every layer and attends positions
 * [0, start_pos + i] of that row, so a prompt can be fed in chunks of
 * increasing start_pos (the earlier positions must already be in the row).
 * Every prompt position computes exactly what a decode step would compute for
 * that token at that cache position; prefill is that step applied to all of
 * them at once.
 *   token_ids     device int32 [T], 1 <= T <= the reserved chunk size
 *   positions     device int32 [3, T]: M-RoPE (T, H, W) ids of each position
 *   state_token, state_positions [3], state_cache_position, state_finished:
 *                 device (one row each): receive the first decode step's state
 *                 of this sequence — the greedy token after the chunk (lowest
 *                 index on ties), the last position's ids + 1, start_pos + T,
 *                 and finished = 1 if that token is eos_id or the row is full
 *   logits        device fp32 [V]: the last position's logits, or NULL
 * Queued on `stream` without synchronisation (about 4 launches per layer and
 * 16 positions, plus the LM head).  Errors: KMR_ERR_INVALID_ARG (NULL
 * pointer, T < 1), KMR_ERR_BUFFER_SIZE (T above the reserved size),
 * KMR_ERR_SLOT_RANGE, KMR_ERR_CACHE_FULL (start_pos < 0 or start_pos + T >
 * max_len), KMR_ERR_NO_PACK (weights not loaded), KMR_ERR_CUDA; a token id
 * out of range sets the device error word (kmr_model_sync_status). */
int kmr_prefill(kmr_model* m, const int32_t* token_ids, const int32_t* positions, int T, int slot, int start_pos,
                int32_t* state_token, int32_t* state_positions, int32_t* state_cache_position,
                uint8_t* state_finished, float* logits, void* stream);

/* Device pointers of one layer's K and V cache ([slots][n_kv][max_len][d] bf16). */
int kmr_model_kv_pointers(kmr_model* m, int layer, void** k_cache, void** v_cache);

/* Row migration into the model's static cache ("kaminari", §08 The serving
 * layer: the continuous scheduler's slot pool owns one static cache with a
 * physical row per slot, and copy_row_from moves a row's KV state into it;
 * §03 State model: the cache is mutated in place).
 * Copies positions [0, length) of row src_row of a source cache into cache row
 * dst_slot of the model, for every layer, K and V:
 *   src_k, src_v   device pointers to layer 0 of a source cache laid out like
 *                  the model's: [L][src_slots][n_kv][src_max_len][d] bf16 with
 *                  the model's L, n_kv and d, 16-byte aligned, not overlapping
 *                  the destination row.  Both NULL: the model's own cache
 *                  (src_slots and src_max_len are then ignored), i.e. a slot to
 *                  slot migration.
 *   length         positions copied, 0 <= length <= min(src_max_len, max_len)
 * Positions >= length of the destination row keep their contents.  One kernel
 * launch queued on `stream`, no synchronisation; the source row must not be
 * written nor the destination row used by a step until it has run.  Copying a
 * row of the model's cache onto itself, or length 0, launches nothing.
 * Errors: KMR_ERR_INVALID_ARG (NULL model, one source pointer NULL and not the
 * other, misaligned source, src_slots or src_max_len <= 0, src_row outside an
 * external source, negative length), KMR_ERR_SLOT_RANGE (dst_slot, or src_row
 * of the model's own cache, outside [0, slots)), KMR_ERR_CACHE_FULL (length
 * above either cache's max_len), KMR_ERR_CUDA. */
int kmr_model_copy_row_from(kmr_model* m, int dst_slot, const uint16_t* src_k, const uint16_t* src_v,
                            int src_slots, int src_max_len, int src_row, int length, void* stream);

/* One greedy decode step for B rows ("kaminari", §04 Request lifecycle,
 * decode; §08 ContinuousBatchScheduler slots).  All pointers are device
 * memory; the step state is read and advanced in place:
 *   token_ids      int32 [B]    in: this step's token; out: the emitted token
 *                               (argmax, lowest index on ties, or pad_id for
 *                               rows finished before the step)
 *   positions      int32 [3, B] in: M-RoPE (T, H, W) ids of this token;
 *                               out: +1 for rows not finished before the step
 *   cache_position int32 [B]    in: where this token's K/V are written (the row
 *                               attends 0..cache_position); out: +1 likewise
 *   slot_ids       int32 [B]    physical cache row of each batch row
 *   finished       uint8 [B]    in/out: set when the emitted token is eos_id or
 *                               the row has written position max_len - 1
 *   logits         fp32 [B, V] or NULL: the final logits of every row
 * A row finished before the step reads and writes no KV and does not advance.
 * The step is a cached CUDA graph of the whole layer stack (captured on first
 * use per pointer set and B); it is queued on `stream` without synchronising.
 * Returns KMR_ERR_NO_PACK if any weight was never loaded. */
int kmr_decode_step(kmr_model* m, int32_t* token_ids, int32_t* positions, int32_t* cache_position,
                    const int32_t* slot_ids, uint8_t* finished, int B, float* logits, void* stream);

/* The same step on HOST state arrays (same shapes and meaning): copies the
 * state in, runs the step, copies the updated state back and synchronises
 * `stream`.  logits (host fp32 [B, V]) may be NULL.  Per-row state is checked
 * on the host first (KMR_ERR_SLOT_RANGE, KMR_ERR_CACHE_FULL). */
int kmr_decode_step_host(kmr_model* m, int32_t* token_ids, int32_t* positions, int32_t* cache_position,
                         const int32_t* slot_ids, uint8_t* finished, int B, float* logits, void* stream);

/* Synchronise `stream`, then return and clear the model's device error word. */
int kmr_model_sync_status(kmr_model* m, void* stream);

/* ---- Diagnostics (no counterpart in the method's description) ----------------
 * Shared-memory poisoning.  kmr_smem_poison fills the shared memory of every SM
 * of the current device with the 32-bit `pattern`, asynchronously on `stream`
 * (one CTA per SM holding 227 KB).  With kmr_model_set_smem_poison(m, 1, pattern)
 * every kernel of the model's decode step is preceded by such a fill, so a
 * kernel that reads shared memory it did not write sees `pattern` (choose NaN
 * or Inf bits) rather than leftovers; a poisoned step must equal a clean one
 * bit for bit.  Enabling or disabling synchronises the device and drops the
 * model's captured step graphs.  Off by default; costs one extra launch per
 * kernel.  Returns KMR_OK, KMR_ERR_INVALID_ARG (null model) or KMR_ERR_CUDA. */
int kmr_smem_poison(uint32_t pattern, void* stream);

/* Self-test of the bounded device waits (failure detection without a fault):
 * launches one warp that waits on a shared-memory mbarrier nothing completes.
 * The wait gives up after limit_ns nanoseconds (1 us .. 2 s), the kernel
 * returns, and kmr_last_device_error() then reads KMR_ERR_DEVICE_TIMEOUT; the
 * context stays usable.  Asynchronous on `stream`.  Returns KMR_OK,
 * KMR_ERR_INVALID_ARG (limit out of range) or KMR_ERR_CUDA. */
int kmr_selftest_wait_timeout(unsigned long long limit_ns, void* stream);
int kmr_model_set_smem_poison(kmr_model* m, int enable, uint32_t pattern);

/* Prefill projections on the 5th-generation tensor cores (the prefill of
 * "kaminari", §04 Request lifecycle; the projections of §07).  With enable = 1
 * (the default), kmr_prefill runs every projection whose output rows are a
 * multiple of 128 as a tcgen05.mma kernel: each 128-input group's int4 weights
 * dequantised to fp16 in tensor memory, the staged tokens as fp16 scaled by a
 * per-row power of two, fp32 accumulation in tensor memory across the CTA's K
 * range.  enable = 0 selects the warp-level mma kernel.  The two agree within
 * rounding and are parity-tested against the oracle the same way; on either,
 * a token's result does not depend on the prompt length or chunking.  Takes
 * effect from the next kmr_prefill call.  Returns KMR_OK or
 * KMR_ERR_INVALID_ARG (null model). */
int kmr_model_set_prefill_tcgen05(kmr_model* m, int enable);

/* Tile shape of the tcgen05 prefill projections: nt tokens per CTA (64, 128
 * or 256; the MMA's N) and the K range split over ksplit CTAs of one
 * thread-block cluster (1, 2 or 4; a projection with fewer 128-input groups
 * takes the largest power of two that fits), whose fp32 partials are summed
 * in rank order through distributed shared memory.  nt = ksplit = 0 (the
 * default) plans each projection from its shape: N x K, the prompt length and
 * the SM count.  The result does not depend on the K split beyond fp32
 * rounding, and the same plan always gives the same bits.  Takes effect from
 * the next kmr_prefill call.  Returns KMR_OK or KMR_ERR_INVALID_ARG (null
 * model, or a value outside those sets). */
int kmr_model_set_prefill_plan(kmr_model* m, int nt, int ksplit);

/* The tile plan kmr_prefill chooses for a tcgen05 projection with N output
 * rows (a multiple of 128), K inputs (a multiple of 128, at most 8192) and M
 * prompt tokens on a GPU with `sms` SMs: *nt tokens per CTA and *ksplit CTAs
 * along K.  The split depends on (N, K, sms) only, never on M, so a token's
 * result does not change with the prompt length or chunking.  Host-only (no
 * GPU needed).  Returns KMR_OK or KMR_ERR_INVALID_ARG (unsupported shape, M or
 * sms < 1, null output). */
int kmr_prefill_plan(int N, int K, int M, int sms, int* nt, int* ksplit);

/* Whether the decode step runs its layers as one persistent kernel (default
 * off: on GB300 it measured slower than the multi-kernel step, whose
 * programmatic-dependent-launch hand-off between kernels costs less than the
 * persistent kernel's grid-wide phase barriers; it stays selectable and is
 * parity-tested).  The persistent kernel keeps one CTA per SM for the whole step: each
 * CTA streams its share of every layer's int4 weights and its attention
 * splits' K/V rows through a ring of shared-memory slots (cp.async.bulk),
 * phases (QKV, attention, O, gate_up, down of each layer) start when every CTA
 * has finished the previous one (bounded waits on global counters; a wait that
 * runs out records KMR_ERR_DEVICE_TIMEOUT), and the LM head follows as its own
 * kernel.  It serves up to 4 rows for head sizes 64 and 128 with 2 query heads
 * per KV head; other shapes and larger batches keep the multi-kernel step.
 * Both give the same bits ("kaminari — a single-GPU Qwen3-VL inference engine,
 * explained", §06 The optimization ladder: decode is memory-bandwidth bound
 * and per-step launch overhead was the next cost removed).  Takes effect from
 * the next kmr_decode_step.  Returns KMR_OK or KMR_ERR_INVALID_ARG (null
 * model) / KMR_ERR_CUDA. */
int kmr_model_set_persistent_step(kmr_model* m, int enable);

/* Launches one step makes (kernels per step) for the given B, for accounting
 * (twice as many while shared-memory poisoning is on). */
int kmr_model_kernels_per_step(const kmr_model* m, int B);

/* Device memory the model holds ("kaminari — a single-GPU Qwen3-VL inference
 * engine, explained", §01 TL;DR and §02: int4 weights with a static
 * 1024-token cache brought peak VRAM from 4.2 GB to 2.3 GB).  Returns the
 * bytes of every device allocation the handle owns (packed int4 weights,
 * bf16 embedding and norms, the static KV cache, step and prefill scratch,
 * the host-state step's logits buffer once allocated) and, where the pointers
 * are not null, splits it into weights (packed linears, embedding, norms),
 * kv_cache (K and V of every layer and slot) and scratch (the rest).  No
 * CUDA call; 0 for a null model. */
size_t kmr_model_device_bytes(const kmr_model* m, size_t* weights, size_t* kv_cache, size_t* scratch);

#ifdef __cplusplus
}
#endif
#endif /* KMR_H_ */
