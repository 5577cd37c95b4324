// internal.h -- host-side interface between the C ABI (api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pka.h"

namespace pka {

// Everything one forward launch needs, validated by api.cu.
struct Fwd {
    const void *query;
    const void *kv_cache;
    const int32_t *qsl;
    const int32_t *seq_lens;
    const int32_t *block_table;
    int32_t bt_stride;
    int32_t num_seqs;
    int32_t num_decodes;
    int32_t max_query_len;
    int32_t max_seq_len;
    int32_t common_prefix_len;
    void *out;
    float *lse;
    int32_t num_tokens;
    int32_t num_heads;
    int32_t num_kv_heads;
    int32_t head_size;
    int32_t block_size;
    int64_t num_blocks;
    int32_t kv_hnd;  // 1: pool in HND order, 0: NHD
    int32_t kv_fp8 = 0;  // 1: pool of e4m3 codes, 0: bf16
    float k_scale = 1.f;
    float v_scale = 1.f;
    float out_scale = 1.f;  // prefill: output multiplier (v_scale over a dequantised copy)
    // fused cache write: the decode launch also writes this step's K/V rows
    int32_t fuse_write = 0;
    const void *new_key = nullptr;
    const void *new_value = nullptr;
    const int64_t *slots = nullptr;
    void *kv_cache_w = nullptr;
    float scale;
    int32_t causal;
    cudaStream_t stream;
    int num_sms;
    // test hook of the failure path (pka_test_skip_copies): the kernels' TMA
    // producers issue nothing, so the first bounded wait of every CTA runs out
    int32_t test_skip_copies = 0;
};

// Plan of the decode part of a batch (persistent stream-K grid).
struct DecodePlan {
    int32_t stage_keys;     // keys per pipeline stage (16 * 8/num_kv_heads)
    int32_t grid;           // CTAs of the persistent grid (SM count)
    int32_t chunk;          // decodes per launch (at most 4096)
    int32_t target_keys;    // 0, or keys per CTA to aim for (fewer CTAs)
    int32_t rows_per_slot;  // partial rows per (CTA, sequence) piece and head: 8/num_kv_heads
};

// Workspace carve-up (byte offsets from the workspace base, 256-aligned).
struct Workspace {
    size_t o_part, lse_part;   // decode piece partials
    size_t counters;           // pieces finished per decode (int32)
    size_t o_pre, lse_pre;     // cascade: shared-prefix partials of every token, one per
                               // key chunk of the prefix ([pre_splits][T, H, D])
    int32_t pre_splits;        // cascade: key chunks of the shared-prefix pass
    size_t o_suf, lse_suf;     // cascade: suffix partial of every prefill token
    size_t pf_counters;        // prefill work-queue counters (int32 x 2)
    // fp8 pool with prefills or a cascade: the prefill sequences' blocks as bf16
    // code values (fp8_blocks_per_seq = ceil(max_seq_len / bs) blocks per prefill
    // sequence), then (cascade with decodes) the shared prefix's fp8_prefix_blocks
    // blocks of block-table row 0, and their block table ([num_seqs,
    // fp8_blocks_per_seq] int32)
    size_t fp8_scratch, fp8_table;
    int32_t fp8_blocks_per_seq;
    int32_t fp8_prefix_blocks;
    int64_t fp8_scratch_blocks;
    // bf16 pool of small pages: the prefill sequences' keys re-blocked into
    // 128-key NHD blocks (reblock_blocks_per_seq = ceil(max_seq_len / 128) per
    // prefill sequence) and their block table ([num_seqs, blocks_per_seq])
    size_t reblock_scratch, reblock_table;
    int32_t reblock_blocks_per_seq;
    int64_t reblock_blocks;
    size_t total;
};

DecodePlan plan_decode(int32_t split_kv_tokens, int32_t num_decodes, int32_t num_kv_heads,
                       int num_sms);
// Cascade (the shared-prefix pass and the suffix passes): how many key chunks
// the prefix is cut into (each chunk's partial is merged later), and whether
// the prefix pass runs on pre_ctas SMs beside the suffix decode on the other
// SMs (overlap: the decode is a dependent launch that starts at once) or on
// every SM before it.  Chosen on a cost model of both passes; host sizes only.
struct CascadePlan {
    int32_t pre_splits = 1;
    int32_t pre_ctas = 0;  // 0: every SM
    bool overlap = false;
};
// Decodes and prefills of one batch (no cascade) side by side: the
// decode on dec_ctas SMs, the prefill pass as its programmatic dependent on the
// others, taking over the decode's SMs as they free up.
struct MixedPlan {
    bool overlap = false;
    int32_t dec_ctas = 0;
};
MixedPlan plan_mixed(int32_t num_tokens, int32_t num_heads, int32_t num_kv_heads,
                     int32_t head_size, int32_t num_decodes, int32_t num_seqs,
                     int32_t max_seq_len, bool kv_fp8, bool single_decode_launch, int num_sms);
CascadePlan plan_cascade(int32_t num_tokens, int32_t num_heads, int32_t num_kv_heads,
                         int32_t head_size, int32_t prefix_len, int32_t num_decodes,
                         int32_t max_seq_len, bool kv_fp8, bool single_decode_launch,
                         int num_sms);
Workspace plan_workspace(const DecodePlan &dp, int32_t num_tokens, int32_t num_decodes,
                         int32_t num_heads, int32_t head_size, bool cascade,
                         int32_t pre_splits);
// A bf16 pool of small pages read by a query-heavy prefill pass: the 128-key
// re-blocking of the prefill sequences' keys (none otherwise), appended.
void plan_reblock(Workspace &w, bool kv_fp8, int32_t num_tokens, int32_t num_seqs,
                  int32_t num_decodes, int32_t max_seq_len, int32_t block_size,
                  int32_t num_kv_heads, int32_t head_size);
// The smallest workspace a forward accepts (without the re-blocking copy);
// 0 when the arguments are invalid.
size_t workspace_size_min(const pka_meta *m, int32_t num_tokens, int32_t num_heads,
                          int32_t num_kv_heads, int32_t head_size, int32_t block_size);
// The fp8 prefill copy: blocks per prefill sequence and bytes of the bf16 scratch pool
// (0 when the pool is bf16 or there are no prefills); appended to a planned workspace.
void plan_fp8_prefill(Workspace &w, bool kv_fp8, int32_t num_seqs, int32_t num_decodes,
                      int32_t max_seq_len, int32_t common_prefix_len, int32_t block_size,
                      int32_t num_kv_heads, int32_t head_size);

// kv_write.cu
cudaError_t launch_reshape_and_cache(const void *key, const void *value, void *cache,
                                     const int64_t *slots, int32_t num_tokens,
                                     int32_t num_kv_heads, int32_t head_size,
                                     int32_t block_size, int64_t num_blocks, int32_t hnd,
                                     cudaStream_t st);
cudaError_t launch_reshape_and_cache_fp8(const void *key, const void *value, void *cache,
                                         const int64_t *slots, int32_t num_tokens,
                                         int32_t num_kv_heads, int32_t head_size,
                                         int32_t block_size, int64_t num_blocks, int32_t hnd,
                                         float k_scale, float v_scale, cudaStream_t st);
// Blocks of an fp8 pool (f.kv_cache, layout f.kv_hnd) as bf16 code values in a
// dense NHD scratch pool and its block table: block-table rows [first_row,
// first_row + num_rows), columns below min(ceil(L/bs), col_limit), row p at
// scratch blocks dst_base + p*row_blocks + n, table rows of stride table_stride.
// dependent_follows: the next launch is its programmatic dependent (started at
// once; it waits for this grid before it reads the copy).
cudaError_t launch_dequant_blocks(const Fwd &f, void *scratch, int32_t *table, int32_t first_row,
                                  int32_t num_rows, int32_t row_blocks, int32_t col_limit,
                                  int64_t dst_base, int32_t table_stride,
                                  bool dependent_follows = false);
// The prefill sequences' keys of a bf16 pool of small pages (block_size a
// divisor of 32) copied into 128-key NHD blocks of a scratch pool: block-table
// rows [first_row, first_row + num_rows), destination block dst_base +
// p * row_blocks + n of row p, table rows of stride table_stride.  With
// context_lo >= 0 only the blocks that a pass starting at key context_lo still
// reads from the pool when it takes the tiles of this step's keys from the
// step's rows (those below a sequence's context, plus one) are copied.
cudaError_t launch_reblock(const Fwd &f, void *scratch, int32_t *table, int32_t first_row,
                           int32_t num_rows, int32_t row_blocks, int64_t dst_base,
                           int32_t table_stride, int32_t context_lo = -1);
uint32_t kv_write_take_error();

// Most key chunks of a cascade's shared-prefix pass (partials per row).
constexpr int32_t kMaxPrefixSplits = 8;
// A decode batch of at most one stage per SM whose longest sequence has at most
// this many stages is divided one sequence per CTA instead of evenly: no
// sequence is split over CTAs, so none waits on a cross-CTA merge (a fence, an
// atomic count and an L2 round trip of partials, several microseconds), while
// one CTA streams a few stages in well under that.
constexpr int kAlignedMaxStages = 8;

// Where the decode launch puts its rows.
struct DecodeOut {
    // nullptr: bf16 out / ln lse.  Else (cascade suffix) fp32 normalised
    // partials [T, H, D] and log2 lse [T, H], merged with the prefix later.
    float *o_suf = nullptr;
    float *lse_suf = nullptr;
    // the launch is the dependent of the shared-prefix pass enqueued just
    // before it (programmatic stream serialisation: it starts on the SMs that
    // pass leaves free, and its grid completes after that pass)
    bool after_prefix = false;
    // the first launch's per-sequence counters were zeroed by the caller
    // (before the prefix pass, so that nothing stands between the two kernels)
    bool counters_zeroed = false;
    // a programmatic dependent launch follows (the cascade's combine, or the
    // prefill pass beside this decode): let it be scheduled as this grid drains
    bool dependent_follows = false;
    // the batch is small enough, by max_seq_len, for the kernel to divide it
    // one sequence per CTA (kAlignedMaxStages): no piece is merged across
    // CTAs, so the per-decode counters are not reset (a batch longer than
    // max_seq_len says is flagged by the kernel, which then computes nothing)
    bool expect_aligned = false;
    // a decode-only batch of a few long decodes: the pieces of a decode split
    // over several CTAs are merged by a launch over the whole GPU after the
    // decode's (its programmatic dependent), not by the decode's last CTA
    bool defer_merge = false;
};

// decode.cu: paged decode of sequences [0, num_decodes) over keys
// [kv_begin, L_s), stream-K over a persistent grid of dp.grid CTAs with the
// split combine fused in.
cudaError_t launch_decode(const Fwd &f, const DecodePlan &dp, const Workspace &ws, char *wsp,
                          const CUtensorMap &kv_map, int32_t kv_begin, const DecodeOut &dout);
// Cascade: merge every token's suffix partial with its shared-prefix partials.
cudaError_t launch_cascade_combine(const Fwd &f, const Workspace &ws, char *wsp);
uint32_t decode_take_error();

// merge.cu
cudaError_t launch_cascade_merge(const void *out_a, const float *lse_a, const void *out_b,
                                 const float *lse_b, void *out, float *lse_out,
                                 int32_t num_tokens, int32_t num_heads, int32_t head_size,
                                 cudaStream_t st);

cudaError_t launch_merge_partials(const void *outs, const float *lses, int32_t num_parts,
                                  void *out, float *lse_out, int32_t num_tokens,
                                  int32_t num_heads, int32_t head_size, int32_t base2,
                                  cudaStream_t st);
uint32_t merge_take_error();

// Set the thread-local message pka_last_error() returns (api.cu).
void set_last_error(const char *fmt, ...);

// Per-thread count of kernel launches (api.cu), bumped by every launcher.
void count_launch();

// prefill.cu: one pass of the tensor-core kernel.
//  shared_prefix = false: the prefill sequences [num_decodes, num_seqs), keys
//    [kv_lo, min(kv_cap, L_s)), causal or not;
//  shared_prefix = true: every token of the batch against keys [0, kv_cap) of
//    the prefix all sequences share (block-table row 0), no mask; the keys are
//    cut into kv_splits chunks, chunk c's partial at rows c*T*H + t*H + h.
//  o_part == nullptr: write bf16 out / ln lse; else fp32 partials (normalised)
//    and log2 lse at rows (t - token_base) * num_heads + h.
struct PrefillPass {
    int32_t kv_lo;
    int32_t kv_cap;
    int32_t causal;
    bool shared_prefix;
    float *o_part;
    float *lse_part;
    int32_t token_base;
    int32_t *item_counter;  // device int32 for the dynamic work queue (zeroed per launch)
    int32_t kv_splits = 1;  // shared_prefix: key chunks
    int32_t max_ctas = 0;   // 0: one CTA per SM; else at most this many CTAs
    // let a dependent launch (the cascade's suffix decode) start as soon as
    // every CTA of this pass is resident
    bool trigger_dependents = false;
    // a bf16 pool written this step (the fused call): key tiles that hold only
    // this step's keys are read from its key/value rows, not from the pool
    bool new_from_input = false;
    // launched as the programmatic dependent of the decode just before it
    // (beside it on the SMs it leaves); the pass completes after the decode
    bool after_decode = false;
    // item_counter was zeroed by the caller (nothing may stand between the
    // decode and this launch)
    bool counter_zeroed = false;
    // launched as the programmatic dependent of the fp8 block copy just before
    // it: the pass waits for the copy's grid before it reads anything the copy
    // writes (its blocks and block table)
    bool after_copy = false;
};
cudaError_t launch_prefill(const Fwd &f, const PrefillPass &pass);
uint32_t prefill_take_error();
constexpr int kMaxPrefillSeqsPerCall = 4096;

// tensor maps (api.cu): a 3-D bf16 tensor (d0 contiguous), 128-byte swizzle
CUresult encode_3d_bf16(CUtensorMap *map, const void *base, uint64_t d0, uint64_t d1,
                        uint64_t d2, uint64_t stride1_bytes, uint64_t stride2_bytes,
                        uint32_t box0, uint32_t box1, uint32_t box2);
// The pool as a 3-D tensor whose box {128 bytes, 1, rows} (NHD) / {128 bytes,
// rows, 1} (HND) -- 64 bf16 dims, or 128 e4m3 dims of an fp8 pool
// (elem_bytes 1) -- reads `rows` consecutive keys of one head of one page
// (page = block*2 + kv), 128-byte swizzled, in the same shared-memory layout
// either way:
//   NHD  (head_size, num_kv_heads, pages*block_size), coordinates
//        (dim, head, page*block_size + offset);
//   HND  (head_size, block_size, pages*num_kv_heads), coordinates
//        (dim, offset, page*num_kv_heads + head).
CUresult encode_kv_map(CUtensorMap *map, const void *cache, int32_t head_size,
                       int32_t num_kv_heads, int32_t block_size, int64_t num_blocks, int32_t hnd,
                       uint32_t box_rows, int32_t elem_bytes = 2);
// The pool as a 3-D tensor whose outermost dimension is the kv head, box
// {128 bytes, 16 keys, num_kv_heads}: one box reads 16 consecutive keys of one
// page for every head, head after head (2 KB each), 128-byte swizzled -- the
// decode kernel's view:
//   NHD  (head_size, pages*block_size, num_kv_heads), coordinates
//        (dim, page*block_size + offset, 0); the head stride is one row;
//   HND  (head_size, block_size, pages*num_kv_heads), coordinates
//        (dim, offset, page*num_kv_heads).
CUresult encode_kv_map_heads(CUtensorMap *map, const void *cache, int32_t head_size,
                             int32_t num_kv_heads, int32_t block_size, int64_t num_blocks,
                             int32_t hnd, int32_t elem_bytes);

}  // namespace pka
