/*
 * pka.h -- C ABI of the paged-KV attention forward for GB300 (sm_103a).
 *
 * One serving-engine attention step over a paged KV pool:
 *   pka_reshape_and_cache   write this step's K/V rows into the pool
 *                           (_ex: NHD or HND pool; _fp8: an fp8 e4m3 pool),
 *   pka_paged_attn_forward  attention of a mixed, decode-first batch over
 *                           the pool (split-KV decode, causal / chunked
 *                           prefill, optional shared-prefix cascade; bf16
 *                           or fp8 e4m3 pool, NHD or HND),
 *   pka_paged_attn_forward_fused  the two above in one call, the write done
 *                           inside the decode launch,
 *   pka_paged_attn_forward_noalloc  the forward without a caller workspace,
 *   pka_cascade_merge       log-sum-exp merge of two partial attentions,
 *   pka_merge_partials      the N-way merge with an explicit lse base (the
 *                           combine of a decode context-parallel step).
 *
 * Sources, cited by page title and section:
 *  [FA/FI]   "FlashAttention y FlashInfer: los dos grandes backends de atencion
 *            en GPU" (vllm-arch-zh.pages.dev/es/attention/flash)
 *  [blog]    "El especialista del plato estrella: el backend de atencion de
 *            vLLM (FlashAttention, FlashInfer y la asimetria prefill/decode)"
 *            (blog.lo0.es)
 *  [backend] "AttentionBackend: capa de abstraccion de backends de atencion"
 *            (vllm-arch-zh.pages.dev/es/attention/backend)
 *
 * Common rules for every entry point
 *  - Device buffers are owned by the caller; the library never allocates or
 *    frees device memory and never synchronises the stream, except
 *    pka_check_status, which synchronises on purpose.
 *  - Work is enqueued on `stream` (a cudaStream_t / CUstream passed as
 *    void*; NULL is the legacy default stream) and runs asynchronously.
 *  - Tensors are dense, row-major, with 16-byte aligned base addresses.
 *  - bf16 means IEEE bfloat16 (the upper half of a binary32).
 *  - Every call returns a pka_status; on a non-OK status nothing was
 *    enqueued and pka_last_error() describes the reason.  No C++ exception
 *    crosses this boundary.
 *  - A device-side check that fails (an out-of-pool slot or block id, or a
 *    pipeline wait that exceeded its time limit) never traps: the access is
 *    skipped, a sticky error word is set, and the next pka_check_status
 *    returns PKA_ERR_DEVICE_CHECK.
 */
#ifndef PKA_H
#define PKA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PKA_OK = 0,
    PKA_ERR_INVALID_ARG = -1,  /* a bad argument (null pointer, size, alignment, block size) */
    PKA_ERR_UNSUPPORTED = -2,  /* valid, but not a shape this build serves */
    PKA_ERR_WORKSPACE = -3,    /* workspace missing, too small or misaligned */
    PKA_ERR_CUDA = -4,         /* a CUDA runtime/driver call failed */
    PKA_ERR_DEVICE_CHECK = -5  /* a device-side check failed (see pka_check_status) */
} pka_status;

/*
 * Batch metadata, the per-step fields of CommonAttentionMetadata
 * ([backend] "Archivos clave": query_start_loc, seq_lens, block_table_tensor;
 * [FA/FI] "Responsabilidades": decode-first order; [backend] "Flujo de datos":
 * build(common_prefix_len, ...)).  The struct itself lives in host memory;
 * the three array pointers are device pointers.
 *
 *  query_start_loc  int32 [num_seqs+1]; qsl[0] = 0, nondecreasing,
 *                   qsl[num_seqs] = num_tokens.  Sequence s owns query
 *                   tokens [qsl[s], qsl[s+1]).
 *  seq_lens         int32 [num_seqs]; L_s >= 1, the whole KV length of s
 *                   including this step's tokens (already written by
 *                   pka_reshape_and_cache).  Prior context c_s = L_s - q_s.
 *                   A decode may have L_s = 0 (no keys, e.g. a context-
 *                   parallel rank's empty shard): its rows get out = 0 and
 *                   lse = -inf.
 *  block_table      int32 [num_seqs, block_table_stride]; entry n of row s
 *                   is the physical block holding keys [n*bs, (n+1)*bs) of
 *                   s.  Entries past ceil(L_s/bs) are never read.
 *  num_decodes      the first num_decodes sequences are decodes: exactly one
 *                   query token each ([FA/FI] "Responsabilidades": decode
 *                   first, then prefill).
 *  max_query_len    host upper bound on q_s over the prefill sequences.
 *  max_seq_len      host upper bound on L_s over all sequences (0 only in a
 *                   batch of decodes that all have L_s = 0).
 *  common_prefix_len  0, or a multiple of block_size P such that the first
 *                   P/bs block-table entries of every sequence are the same
 *                   blocks and P <= c_s for every s ([blog] "Que aporta
 *                   FlashInfer: JIT y cascade attention").
 *  split_kv_tokens  0 = automatic (the decode work is divided evenly over one
 *                   CTA per SM); else a target number of keys per CTA, which
 *                   uses fewer CTAs when the batch is small (a tuning and
 *                   test knob; results are the same either way).
 *  kv_layout        physical order of the pool (pka_kv_layout): PKA_LAYOUT_NHD
 *                   (0, the default of a zero-initialised struct) or
 *                   PKA_LAYOUT_HND.
 *  kv_dtype         element type of the pool (pka_kv_dtype): PKA_KV_BF16 (0,
 *                   the default) or PKA_KV_FP8_E4M3.
 *  k_scale, v_scale fp8 pools only: the per-tensor dequantisation scales of
 *                   K and V (element value = e4m3 code value x scale);
 *                   positive and finite.  Ignored for bf16.
 */

/*
 * Physical layouts of the pool ([FA/FI] "Resumen en una frase": the two
 * layouts NHD / HND, chosen by get_kv_cache_stride_order).  The logical shape
 * is always [num_blocks, 2, block_size, num_kv_heads, head_size]; the layout
 * says which of block_size and num_kv_heads varies faster in memory:
 *  NHD  [num_blocks, 2, block_size, num_kv_heads, head_size] -- the K (or V)
 *       rows of one slot, all heads, are contiguous;
 *  HND  [num_blocks, 2, num_kv_heads, block_size, head_size] -- the page of
 *       one head (block_size rows) is contiguous.
 */
typedef enum { PKA_LAYOUT_NHD = 0, PKA_LAYOUT_HND = 1 } pka_kv_layout;

/*
 * Element type of the pool ([FA/FI] "Resumen en una frase" and "Limites y
 * fallos": an fp8 e4m3 KV cache).  The pages fix no quantisation rule; this
 * library uses one fp32 scale per tensor for K and one for V:
 *     code  = e4m3(x / scale)   (x/scale in binary32, rounded to the nearest
 *                                e4m3 value, ties to the even code, clamped
 *                                to +-448: the OCP E4M3 format, no infinity)
 *     value = e4m3_value(code) * scale
 * An fp8 pool has the bf16 pool's logical shape with one byte per element.
 */
typedef enum { PKA_KV_BF16 = 0, PKA_KV_FP8_E4M3 = 1 } pka_kv_dtype;

typedef struct {
    const int32_t *query_start_loc;
    const int32_t *seq_lens;
    const int32_t *block_table;
    int32_t block_table_stride;
    int32_t num_seqs;
    int32_t num_decodes;
    int32_t max_query_len;
    int32_t max_seq_len;
    int32_t common_prefix_len;
    int32_t split_kv_tokens;
    int32_t kv_layout;
    int32_t kv_dtype;
    float k_scale;
    float v_scale;
} pka_meta;

/*
 * Write this step's K/V rows into the paged pool (the cache-update op of
 * [FA/FI] "Responsabilidades", unified_kv_cache_update).
 *
 *  key, value     device bf16 [num_tokens, num_kv_heads, head_size]
 *  kv_cache       device bf16 [num_blocks, 2, block_size, num_kv_heads,
 *                 head_size] ([FA/FI] "Flujo de datos", get_kv_cache_shape;
 *                 index 0 of the second axis is K, 1 is V), written in place
 *  slot_mapping   device int64 [num_tokens]; slot = block*block_size +
 *                 offset; a negative slot is padding and is skipped
 *
 * For every token t with slot >= 0 the K row and the V row land byte for
 * byte at (slot/block_size, slot%block_size); nothing else is written.
 * A slot >= num_blocks*block_size is skipped and flagged on the device.
 * Duplicate slots in one call are a caller error (the winner is undefined).
 * Errors: PKA_ERR_INVALID_ARG for null pointers, num_tokens < 0,
 * block_size not a multiple of 16 ([FA/FI] "Flujo de datos": "Block size must
 * be a multiple of 16"), head_size not a multiple of 8.
 */
pka_status pka_reshape_and_cache(const void *key, const void *value, void *kv_cache,
                                 const int64_t *slot_mapping, int32_t num_tokens,
                                 int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                                 int64_t num_blocks, void *stream);

/*
 * pka_reshape_and_cache for a pool in the physical layout `kv_layout`
 * (pka_kv_layout); PKA_LAYOUT_NHD is exactly pka_reshape_and_cache.  In HND
 * the row of head k of slot (b, o) is at [b][kv][k][o].  Errors as
 * pka_reshape_and_cache, plus PKA_ERR_INVALID_ARG for an unknown layout.
 */
pka_status pka_reshape_and_cache_ex(const void *key, const void *value, void *kv_cache,
                                    const int64_t *slot_mapping, int32_t num_tokens,
                                    int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                                    int64_t num_blocks, int32_t kv_layout, void *stream);

/*
 * pka_reshape_and_cache_ex into an fp8 e4m3 pool (pka_kv_dtype): every element
 * of the token's K row is stored as e4m3(k / k_scale), of its V row as
 * e4m3(v / v_scale), by the rule stated at pka_kv_dtype.
 *
 *  kv_cache       device uint8 pool, the bf16 pool's shape in the layout
 *                 kv_layout, one byte per element, written in place
 *  k_scale, v_scale  positive finite fp32 scales (host values)
 *
 * Errors as pka_reshape_and_cache_ex, plus PKA_ERR_INVALID_ARG for a scale
 * that is not positive and finite and PKA_ERR_UNSUPPORTED for head_size not
 * a multiple of 16.
 */
pka_status pka_reshape_and_cache_fp8(const void *key, const void *value, void *kv_cache,
                                     const int64_t *slot_mapping, int32_t num_tokens,
                                     int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                                     int64_t num_blocks, int32_t kv_layout, float k_scale,
                                     float v_scale, void *stream);

/*
 * Bytes of device workspace pka_paged_attn_forward needs for this batch
 * (split-KV and cascade partial results, fp32).  Same shape arguments as the
 * forward; depends only on host-side fields of `meta`.  Returns 0 when the
 * arguments are invalid.
 */
size_t pka_workspace_size(const pka_meta *meta, int32_t num_tokens, int32_t num_heads,
                          int32_t num_kv_heads, int32_t head_size, int32_t block_size);

/*
 * The smallest workspace pka_paged_attn_forward accepts for this batch (same
 * arguments; 0 when they are invalid).  pka_workspace_size can be larger: with
 * a bf16 pool of 16-key pages and query-heavy prefills (at least 256 query
 * tokens per prefill sequence on average) it adds room for a copy of the
 * prefill sequences' keys in 128-key blocks, which the tensor-core prefill
 * then reads with one TMA box per tile half instead of one per page.  Given a
 * workspace of at least this size but below pka_workspace_size, the forward
 * reads the pages as they are; the results are the same bit for bit.  The
 * pages have no counterpart of this call.
 */
size_t pka_workspace_size_min(const pka_meta *meta, int32_t num_tokens, int32_t num_heads,
                              int32_t num_kv_heads, int32_t head_size, int32_t block_size);

/*
 * Attention forward of one layer over the paged pool ([backend] "Archivos
 * clave": AttentionImpl.forward(layer, query, key, value, kv_cache,
 * attn_metadata, output); [FA/FI] "Responsabilidades": Q/K/V reshaped to
 * [num_tokens, num_heads, head_size]; [blog] "Como lee el backend el KV
 * paginado": the kernel gathers the physical blocks through the block table).
 *
 * For query token t of sequence s (t = qsl[s] + i), head h, kv head
 * k = h / (num_heads/num_kv_heads), key j admitted iff !causal || j <= c_s+i:
 *     x_j  = scale * <q[t,h], K_j>,        K_j = kv_cache[bt[s][j/bs], 0, j%bs, k]
 *     lse  = ln sum_j exp(x_j)
 *     out  = sum_j exp(x_j - lse) * V_j,   V_j = kv_cache[bt[s][j/bs], 1, j%bs, k]
 * With common_prefix_len P > 0 the result is the same, computed as the
 * cascade of [blog] "Que aporta FlashInfer": the shared prefix keys [0, P)
 * are attended once for all queries and merged with each sequence's own
 * suffix [P, L_s) by log-sum-exp.
 *
 *  query      device bf16 [num_tokens, num_heads, head_size]
 *  kv_cache   device bf16 [num_blocks, 2, block_size, num_kv_heads, head_size]
 *             (uint8 codes of that shape for an fp8 pool; the order of the
 *             middle axes is meta->kv_layout)
 *  meta       host pointer to the batch metadata above
 *  out        device bf16 [num_tokens, num_heads, head_size]; must not alias
 *             query; every row of every query token is written
 *  lse        device fp32 [num_tokens, num_heads], natural-log units
 *             ([backend] "Limites y fallos": the lse base must be known),
 *             or NULL
 *  scale      softmax scale (1/sqrt(head_size) in the usual case)
 *  causal     1: bottom-right causal mask; 0: every key [0, L_s) admitted
 *  workspace  device buffer of pka_workspace_size(...) bytes (at least
 *             pka_workspace_size_min(...): see there), 256-byte aligned (may be
 *             NULL when that size is 0)
 *
 * Served shapes: head_size 64 or 128; num_kv_heads in {1, 2, 4, 8};
 * num_heads/num_kv_heads <= 8 for decodes; block_size a multiple of 16
 * (PKA_ERR_INVALID_ARG otherwise, as [FA/FI] "Limites y fallos" and
 * [backend] "Limites y fallos" require); other shapes PKA_ERR_UNSUPPORTED.
 * An fp8 pool (meta->kv_dtype = PKA_KV_FP8_E4M3) is served at head_size 128
 * (other head sizes: PKA_ERR_UNSUPPORTED): K_j and V_j above are then the
 * dequantised values code x k_scale and code x v_scale.  Decodes read the
 * codes directly; the tensor-core passes (prefill sequences, a cascade's
 * shared prefix) run on copies of the blocks they read, made in the workspace
 * as bf16 code values (ceil(max_seq_len / block_size) blocks per prefill
 * sequence, plus common_prefix_len / block_size when decodes share a prefix),
 * which pka_workspace_size counts.
 */
pka_status pka_paged_attn_forward(const void *query, const void *kv_cache, const pka_meta *meta,
                                  void *out, float *lse, int32_t num_tokens, int32_t num_heads,
                                  int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                                  int64_t num_blocks, float scale, int32_t causal,
                                  void *workspace, size_t workspace_bytes, void *stream);

/*
 * pka_reshape_and_cache followed by pka_paged_attn_forward, with the cache
 * write folded into the forward's launches ([FA/FI] "Responsabilidades": the
 * FlashAttention kernel writes the KV cache itself,
 * forward_includes_kv_cache_update).  Same results, bit for bit in the pool,
 * as the two calls.  Each decode's new K/V row is written by the decode
 * kernel itself: copied from `key`/`value` into the tile its attention reads
 * (the pool need not hold it yet) and stored at its slot.  The prefill
 * tokens' rows are written by the cache-write kernel before the forward's
 * other launches (one warp per token over the whole GPU; written by the
 * decode CTAs they would hold back the decode's first copies).  A batch of
 * decodes only is thus one launch for write and attention.  Over a bf16 pool
 * the prefill pass reads a 128-key tile that holds only this step's keys
 * (one that starts at or after its sequence's prior context) from
 * `key`/`value` rather than from the pool, the same values.
 *
 *  key, value     device bf16 [num_tokens, num_kv_heads, head_size], as in
 *                 pka_reshape_and_cache; 16-byte aligned, read until the
 *                 forward's last launch
 *  slot_mapping   device int64 [num_tokens]; the slot of each token's key
 *                 through block_table: token qsl[s] + i is key
 *                 L_s - q_s + i of sequence s (for a decode, key L_s - 1),
 *                 which is what makes the fused and the two-call results agree
 *  kv_cache       device pool, written in place (layout meta->kv_layout);
 *                 for an fp8 pool the rows are stored as pka_reshape_and_cache_fp8
 *                 stores them, with meta->k_scale and meta->v_scale, and the
 *                 attention reads the stored codes
 *  other arguments as pka_paged_attn_forward.
 * Errors: those of the two calls; a batch the forward does not serve returns
 * before anything is written.
 */
pka_status pka_paged_attn_forward_fused(const void *query, const void *key, const void *value,
                                        const int64_t *slot_mapping, void *kv_cache,
                                        const pka_meta *meta, void *out, float *lse,
                                        int32_t num_tokens, int32_t num_heads,
                                        int32_t num_kv_heads, int32_t head_size,
                                        int32_t block_size, int64_t num_blocks, float scale,
                                        int32_t causal, void *workspace, size_t workspace_bytes,
                                        void *stream);

/*
 * pka_paged_attn_forward for callers that cannot allocate device memory.
 * The pages have no counterpart of this entry point.
 *
 * Some callers cannot provide a workspace: an engine that reserved almost
 * all of HBM for its KV pool at start-up, a plugin host that only passes
 * input and output pointers, or a serving loop that must not call cudaMalloc
 * because it can synchronise the device.  This entry point takes the same
 * arguments as pka_paged_attn_forward minus the workspace; its scratch (the
 * fp32 split-KV and cascade partials) is a 16 MiB buffer built into the
 * library's device image, which every GPU that loads the library holds until
 * the process exits.  It allocates and frees nothing.
 *
 *  - A batch whose pka_workspace_size is above 16 MiB is rejected with
 *    PKA_ERR_WORKSPACE (and a message naming both sizes); nothing is enqueued.
 *  - The first call on a device looks up the buffer's device address once
 *    (cudaGetSymbolAddress, with that device current); make that first call
 *    before any stream capture.  The address is kept with the CUDA context it
 *    belongs to: the first call after the device's context was torn down and
 *    made anew (cudaDeviceReset, say) looks it up again, so that call too
 *    belongs before any capture.
 *  - Every call shares the one buffer and leaves its contents behind; each
 *    call clears what must start at zero (its per-sequence counters) and
 *    writes all the rest before reading it.  Calls that overlap on the GPU
 *    (other streams, other host threads) race on it: serialise them.
 */
pka_status pka_paged_attn_forward_noalloc(const void *query, const void *kv_cache,
                                          const pka_meta *meta, void *out, float *lse,
                                          int32_t num_tokens, int32_t num_heads,
                                          int32_t num_kv_heads, int32_t head_size,
                                          int32_t block_size, int64_t num_blocks, float scale,
                                          int32_t causal, void *stream);

/*
 * Log-sum-exp merge of two partial attentions of the same queries over
 * disjoint key sets ([blog] "Que aporta FlashInfer: JIT y cascade attention":
 * the prefix result is combined with each request's suffix; [FA/FI] "Limites
 * y fallos": the softmax combine across shards; [backend] "Limites y fallos":
 * natural-log lse).  Per row r = t*num_heads + h:
 *     lse = ln(exp(lse_a) + exp(lse_b))
 *     out = exp(lse_a - lse) * out_a + exp(lse_b - lse) * out_b
 * A side with lse = -inf holds no keys and is the identity.
 *
 *  out_a, out_b  device bf16 [num_tokens, num_heads, head_size]
 *  lse_a, lse_b  device fp32 [num_tokens, num_heads], natural log
 *  out           device bf16, same shape (may alias out_a or out_b)
 *  lse_out       device fp32 [num_tokens, num_heads] or NULL (may alias)
 */
pka_status pka_cascade_merge(const void *out_a, const float *lse_a, const void *out_b,
                             const float *lse_b, void *out, float *lse_out, int32_t num_tokens,
                             int32_t num_heads, int32_t head_size, void *stream);

/* Units of a log-sum-exp: natural log or log base 2. */
typedef enum { PKA_LSE_BASE_E = 0, PKA_LSE_BASE_2 = 1 } pka_lse_base;

/*
 * Log-sum-exp merge of num_parts partial attentions of the same queries over
 * disjoint key sets: the combine step of decode context parallelism, where
 * each rank attends over its shard of every sequence's keys ([FA/FI] "Limites
 * y fallos": the DCP combine branch; [backend] "Limites y fallos": the lse
 * base, ln or log2, has to be the one the partials carry -- a wrong base
 * silently breaks the softmax denominator across shards).  Per row
 * r = t*num_heads + h, with b = e (PKA_LSE_BASE_E) or 2 (PKA_LSE_BASE_2):
 *     lse = log_b(sum_p b^lse_p),   out = sum_p b^(lse_p - lse) * out_p
 * A part with lse = -inf holds no keys and adds nothing; a row with no keys in
 * any part gets out = 0, lse = -inf.
 *
 *  outs      device bf16 [num_parts, num_tokens, num_heads, head_size]
 *  lses      device fp32 [num_parts, num_tokens, num_heads], base lse_base
 *  out       device bf16 [num_tokens, num_heads, head_size]; must not alias outs
 *  lse_out   device fp32 [num_tokens, num_heads] in base lse_base, or NULL
 * Errors: PKA_ERR_INVALID_ARG for num_parts < 1, bad shapes (head_size a
 * multiple of 8), an unknown base, null or misaligned pointers, out aliasing
 * outs.  Asynchronous on `stream`.
 */
pka_status pka_merge_partials(const void *outs, const float *lses, int32_t num_parts, void *out,
                              float *lse_out, int32_t num_tokens, int32_t num_heads,
                              int32_t head_size, int32_t lse_base, void *stream);

/*
 * Synchronise `stream`, then read and clear the sticky device error word.
 * Returns PKA_OK, PKA_ERR_DEVICE_CHECK (with the failing check named by
 * pka_last_error), or PKA_ERR_CUDA when the stream itself reports an error.
 */
pka_status pka_check_status(void *stream);

/*
 * Instrumentation for timing one kernel with CUDA events.  With start/stop
 * non-NULL (cudaEvent_t passed as void*), every later pka_paged_attn_forward
 * on this thread records `start` on its stream right before it launches the
 * kernel named by `kernel` (PKA_KERNEL_DECODE: the split-KV decode kernel;
 * PKA_KERNEL_PREFILL: the prefill kernel) and `stop` right after it.  NULL
 * start/stop turns the recording off.  The events stay owned by the caller.
 * Errors: PKA_ERR_INVALID_ARG for an unknown kernel id.
 */
enum { PKA_KERNEL_DECODE = 0, PKA_KERNEL_PREFILL = 1 };
pka_status pka_set_kernel_events(int32_t kernel, void *start, void *stop);

/*
 * Test hook of the failure path (bounded waits).  With on != 0, the decode and
 * prefill kernels that later pka_paged_attn_forward calls on this thread
 * launch issue no TMA copy and publish no work: the first bounded wait of
 * every CTA runs out after its time limit (2 s), the CTA raises the abort flag,
 * winds down with nothing in flight (no copy issued, no MMA issued, its TMEM
 * freed) and returns; no output row is written, and the next pka_check_status
 * returns PKA_ERR_DEVICE_CHECK ("pipeline wait timed out").  The GPU context
 * stays usable.  on = 0 turns the hook off.  For tests only; never set it in
 * production.  The pages have no counterpart of this call.
 */
pka_status pka_test_skip_copies(int32_t on);

/* Number of kernels the library has launched from this thread so far
 * (instrumentation; counts every launch of every entry point). */
uint64_t pka_kernel_launches(void);

/* Thread-local description of the last non-OK status on this thread. */
const char *pka_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* PKA_H */
