// api.cu -- the C ABI (include/pka.h): argument checks, the host-side plan of
// one forward (decode/prefill partition, split-KV size, workspace carve-up),
// TMA descriptor encoding and the launch sequence on the caller's stream.
//
// The plan uses host-side sizes only (the metadata arrays stay on the device),
// so a forward enqueues kernels and never waits on the GPU; this is the
// analogue of the metadata builder's ahead-of-time schedule on the
// "FlashAttention y FlashInfer" page ("Responsabilidades").
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"
#include "pka.h"

namespace pka {

static thread_local char g_msg[512] = "";
// Optional timing events per kernel kind (pka_set_kernel_events).
static thread_local cudaEvent_t g_ev_start[2] = {nullptr, nullptr};
static thread_local cudaEvent_t g_ev_stop[2] = {nullptr, nullptr};

static thread_local uint64_t g_launches = 0;
// Failure-path test hook (pka_test_skip_copies).
static thread_local int32_t g_test_skip_copies = 0;
void count_launch() { ++g_launches; }

static void record_start(int which, cudaStream_t st)
{
    if (g_ev_start[which])
        cudaEventRecord(g_ev_start[which], st);
}

static void record_stop(int which, cudaStream_t st)
{
    if (g_ev_stop[which])
        cudaEventRecord(g_ev_stop[which], st);
}

static pka_status fail(pka_status st, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof g_msg, fmt, ap);
    va_end(ap);
    return st;
}

void set_last_error(const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof g_msg, fmt, ap);
    va_end(ap);
}

static pka_status cuda_fail(cudaError_t e, const char *what)
{
    return fail(PKA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

static bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

static size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// ------------------------------------------------------------ device facts
static int sm_count()
{
    static std::mutex mu;
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return 148;
    std::lock_guard<std::mutex> lock(mu);
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
        cached[dev] = n;
    }
    return cached[dev];
}

// ------------------------------------------------------------ tensor maps
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

static CUresult encode_3d(CUtensorMap *map, CUtensorMapDataType dtype, const void *base,
                          uint64_t d0, uint64_t d1, uint64_t d2, uint64_t stride1_bytes,
                          uint64_t stride2_bytes, uint32_t box0, uint32_t box1, uint32_t box2)
{
    auto fn = encode_fn();
    if (!fn)
        return CUDA_ERROR_NOT_FOUND;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
    cuuint32_t box[3] = {box0, box1, box2};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, dtype, 3, const_cast<void *>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

CUresult encode_3d_bf16(CUtensorMap *map, const void *base, uint64_t d0, uint64_t d1,
                        uint64_t d2, uint64_t stride1_bytes, uint64_t stride2_bytes,
                        uint32_t box0, uint32_t box1, uint32_t box2)
{
    return encode_3d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, d0, d1, d2, stride1_bytes,
                     stride2_bytes, box0, box1, box2);
}

CUresult encode_kv_map(CUtensorMap *map, const void *cache, int32_t head_size,
                       int32_t num_kv_heads, int32_t block_size, int64_t num_blocks, int32_t hnd,
                       uint32_t box_rows, int32_t elem_bytes)
{
    const uint64_t D = uint64_t(head_size), Hkv = uint64_t(num_kv_heads),
                   bs = uint64_t(block_size), pages = uint64_t(num_blocks) * 2;
    const uint64_t row = D * uint64_t(elem_bytes);  // bytes of one (slot, head) row
    const CUtensorMapDataType dt =
        elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const uint32_t box0 = 128u / uint32_t(elem_bytes);  // one 128-byte swizzle row
    if (hnd)  // (dim, offset, page*Hkv + head): a head's page is bs contiguous rows
        return encode_3d(map, dt, cache, D, bs, pages * Hkv, row, row * bs, box0, box_rows, 1);
    // (dim, head, page*bs + offset): a slot's heads are Hkv contiguous rows
    return encode_3d(map, dt, cache, D, Hkv, pages * bs, row, row * Hkv, box0, 1, box_rows);
}

CUresult encode_kv_map_heads(CUtensorMap *map, const void *cache, int32_t head_size,
                             int32_t num_kv_heads, int32_t block_size, int64_t num_blocks,
                             int32_t hnd, int32_t elem_bytes)
{
    const uint64_t D = uint64_t(head_size), Hkv = uint64_t(num_kv_heads),
                   bs = uint64_t(block_size), pages = uint64_t(num_blocks) * 2;
    const uint64_t row = D * uint64_t(elem_bytes);  // bytes of one (slot, head) row
    const CUtensorMapDataType dt =
        elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const uint32_t box0 = 128u / uint32_t(elem_bytes);  // one 128-byte swizzle row
    if (hnd)  // (dim, offset, page*Hkv + head): a head's page is bs contiguous rows
        return encode_3d(map, dt, cache, D, bs, pages * Hkv, row, row * bs, box0, 16,
                         uint32_t(Hkv));
    // (dim, page*bs + offset, head): the head is the outer dimension, one row apart
    return encode_3d(map, dt, cache, D, pages * bs, Hkv, row * Hkv, row, box0, 16,
                     uint32_t(Hkv));
}

// ------------------------------------------------------------ planning
CascadePlan plan_cascade(int32_t num_tokens, int32_t num_heads, int32_t num_kv_heads,
                         int32_t head_size, int32_t prefix_len, int32_t num_decodes,
                         int32_t max_seq_len, bool kv_fp8, bool single_decode_launch,
                         int num_sms)
{
    CascadePlan c;
    if (prefix_len <= 0 || num_tokens <= 0)
        return c;
    // the search below runs once per distinct batch shape (a serving loop
    // repeats the same shapes): the last plan of this thread is kept
    struct Key {
        int32_t v[8];
        int sms;
        bool fp8, single;
        bool operator==(const Key &o) const
        {
            return memcmp(v, o.v, sizeof v) == 0 && sms == o.sms && fp8 == o.fp8 &&
                   single == o.single;
        }
    };
    const Key key{{num_tokens, num_heads, num_kv_heads, head_size, prefix_len, num_decodes,
                   max_seq_len, 0},
                  num_sms, kv_fp8, single_decode_launch};
    static thread_local Key last_key{{-1, -1, -1, -1, -1, -1, -1, -1}, -1, false, false};
    static thread_local CascadePlan last_plan;
    if (key == last_key)
        return last_plan;
    const int64_t base_items = (int64_t(num_tokens) + 255) / 256 * num_heads;
    const int64_t tiles = (int64_t(prefix_len) + 127) / 128;
    // Cost model in cycles.  A prefix work item of n key tiles costs about
    // n + 1 tile pairs (one pair of start-up) of kPairCycles each; the suffix
    // decode streams its KV at kSmBytesPerCycle per SM, at most
    // kHbmBytesPerCycle over the chip, after a fixed start-up and tail.  The
    // suffix length is not known on the host: half of max_seq_len - prefix_len
    // per decode is taken (lengths spread evenly).  (Measured on GB300: the
    // decode kernel streams ~80 GB/s per SM when HBM is not the limit and
    // saturates HBM on about 100 SMs; a tile pair of the tensor-core pass takes
    // ~4,250 cycles.  The per-SM rates below are the ones that gave the
    // fastest steps on the 256-decode, 4096-token-prefix batch: 39 B/cycle of
    // bf16 K/V (a 64-CTA prefix pass beside an 88-CTA decode, 0.122 ms), 28 of
    // fp8 codes (the same split, 0.103 ms; 34 picked 5 key chunks on 80 CTAs
    // and took 0.122 ms).)
    constexpr double kPairCycles = 4250.0;
    constexpr double kPrefixStartCycles = 8000.0;
    constexpr double kDecodeStartCycles = 30000.0;
    const double kSmBytesPerCycle = kv_fp8 ? 28.0 : 39.0;
    constexpr double kHbmBytesPerCycle = 3250.0;  // ~6.7 TB/s at ~2.07 GHz
    const double suffix_keys =
        double(num_decodes) * std::max(1.0, 0.5 * double(max_seq_len - prefix_len + 1));
    const double dec_bytes = suffix_keys * num_kv_heads * head_size * 2.0 * (kv_fp8 ? 1.0 : 2.0);
    auto t_dec = [&](int ctas) {
        return ctas <= 0 ? 1e30
                         : kDecodeStartCycles +
                               dec_bytes / std::min(kHbmBytesPerCycle, ctas * kSmBytesPerCycle);
    };
    auto t_pre = [&](int64_t chunks, int ctas) {
        const int64_t items = base_items * chunks;
        const int64_t per = (tiles + chunks - 1) / chunks;
        const int64_t waves = (items + ctas - 1) / ctas;
        return kPrefixStartCycles + double(waves) * double(per + 1) * kPairCycles;
    };
    // serial: the prefix pass on every SM, then the decode on every SM
    double best = 1e30;
    for (int64_t s = 1; s <= kMaxPrefixSplits && tiles / s >= 2; ++s) {
        const double t = t_pre(s, num_sms) + (num_decodes > 0 ? t_dec(num_sms) : 0.0);
        if (t < best) {
            best = t;
            c.pre_splits = int32_t(s);
            c.pre_ctas = num_sms;
            c.overlap = false;
        }
    }
    // side by side: the prefix pass on pre_ctas SMs, the decode on the rest
    if (num_decodes > 0 && single_decode_launch && num_sms >= 16) {
        for (int64_t s = 1; s <= kMaxPrefixSplits && tiles / s >= 2; ++s)
            for (int x = 8; x <= num_sms - 8; ++x) {
                const double t = std::max(t_pre(s, x), t_dec(num_sms - x));
                if (t < best * 0.999) {
                    best = t;
                    c.pre_splits = int32_t(s);
                    c.pre_ctas = x;
                    c.overlap = true;
                }
            }
    }
    last_key = key;
    last_plan = c;
    return c;
}

// Decodes and prefills of one batch (no cascade).  The decode is bound by HBM
// and the prefill pass by its SMs (tensor cores and shared memory), and one SM
// of the decode streams ~39 B/cycle (~80 GB/s; 28 of fp8 codes) while HBM
// takes ~3,250 B/cycle: on every SM the decode holds 152 SMs for its bytes at
// the chip's rate, on x SMs only x.  So the decode may run on x SMs beside the
// prefill pass on the others, the pass (its programmatic dependent, one CTA per
// SM, work items claimed from a counter) taking over the decode's SMs as they
// free up: the step then costs about the pass's SM-time plus the decode's bytes
// at the per-SM rate, over the chip.  The host does not see the lengths: every
// sequence's keys are taken as half of max_seq_len, the decode's bytes with a
// 25% margin (a decode that ends after the pass holds the whole step, one that
// ends before it only lends its SMs to the pass later).  A tile pair of the
// pass (two 128-query tiles against a 128-key tile) takes ~4,250 cycles:
// ~3,950 flops per SM and cycle at head_size 128.  Chosen only when the model
// saves at least 5%.  (Measured on the mixed batch of 64 decodes and four
// 2,048-query chunks: 1.426 ms one after the other; side by side with the
// decode on 16 / 24 / 31 / 40 / 48 / 64 / 80 SMs 1.612 / 1.132 / 1.149 / 1.147
// / 1.145 / 1.160 / 1.232 ms; the model picks 31.)
MixedPlan plan_mixed(int32_t num_tokens, int32_t num_heads, int32_t num_kv_heads,
                     int32_t head_size, int32_t num_decodes, int32_t num_seqs,
                     int32_t max_seq_len, bool kv_fp8, bool single_decode_launch, int num_sms)
{
    MixedPlan mp;
    const int64_t prefill_tokens = int64_t(num_tokens) - num_decodes;
    if (num_decodes <= 0 || num_seqs <= num_decodes || prefill_tokens <= 0 ||
        !single_decode_launch || num_sms < 32)
        return mp;
    constexpr double kPassFlopsPerSmCycle = 3950.0;
    constexpr double kPassStartCycles = 8000.0;
    constexpr double kDecodeStartCycles = 30000.0;
    const double kSmBytesPerCycle = kv_fp8 ? 28.0 : 39.0;
    constexpr double kHbmBytesPerCycle = 3250.0;
    const double half = std::max(1.0, 0.5 * double(max_seq_len));
    const double dec_bytes = 1.25 * double(num_decodes) * half * num_kv_heads * head_size *
                             (kv_fp8 ? 2.0 : 4.0);
    const double pass_sm_cycles =
        double(prefill_tokens) * half * 4.0 * head_size * num_heads / kPassFlopsPerSmCycle;
    auto t_dec = [&](int ctas) {
        return kDecodeStartCycles + dec_bytes / std::min(kHbmBytesPerCycle, ctas * kSmBytesPerCycle);
    };
    const double t_serial = t_dec(num_sms) + kPassStartCycles + pass_sm_cycles / num_sms;
    double best = 0.95 * t_serial;
    for (int x = 16; x <= num_sms - 16; ++x) {
        const double td = t_dec(x);
        const double beside = double(num_sms - x) * std::max(0.0, td - kPassStartCycles);
        const double t = pass_sm_cycles <= beside
                             ? td
                             : td + (pass_sm_cycles - beside) / num_sms;
        if (t < best) {
            best = t;
            mp.overlap = true;
            mp.dec_ctas = x;
        }
    }
    return mp;
}

Workspace plan_workspace(const DecodePlan &dp, int32_t num_tokens, int32_t num_decodes,
                         int32_t num_heads, int32_t head_size, bool cascade,
                         int32_t pre_splits)
{
    // (a cascade: pre_splits shared-prefix partials and one suffix partial
    // for every token, decodes included)
    Workspace w;
    size_t off = 0;
    // one partial per (CTA, sequence) piece: slot ids b + s < grid + chunk
    const size_t slots = num_decodes > 0 ? size_t(dp.grid) + dp.chunk : 0;
    const size_t rows_part = slots * dp.rows_per_slot * num_heads;
    w.o_part = off;
    off = round256(off + rows_part * head_size * 4);
    w.lse_part = off;
    off = round256(off + rows_part * 4);
    w.counters = off;
    off = round256(off + size_t(dp.chunk) * 4);
    w.pre_splits = cascade ? pre_splits : 0;
    const size_t rows_all = cascade ? size_t(pre_splits) * num_tokens * num_heads : 0;
    w.o_pre = off;
    off = round256(off + rows_all * head_size * 4);
    w.lse_pre = off;
    off = round256(off + rows_all * 4);
    const size_t rows_pf = cascade ? size_t(num_tokens) * num_heads : 0;
    w.o_suf = off;
    off = round256(off + rows_pf * head_size * 4);
    w.lse_suf = off;
    off = round256(off + rows_pf * 4);
    w.pf_counters = off;
    if (cascade || num_tokens > num_decodes)
        off = round256(off + 2 * sizeof(int32_t));
    w.fp8_table = w.fp8_scratch = off;
    w.fp8_blocks_per_seq = w.fp8_prefix_blocks = 0;
    w.fp8_scratch_blocks = 0;
    w.total = off;
    return w;
}

void plan_fp8_prefill(Workspace &w, bool kv_fp8, int32_t num_seqs, int32_t num_decodes,
                      int32_t max_seq_len, int32_t common_prefix_len, int32_t block_size,
                      int32_t num_kv_heads, int32_t head_size)
{
    const int32_t nprefill = num_seqs - num_decodes;
    const bool cascade = common_prefix_len > 0;
    if (!kv_fp8 || (nprefill <= 0 && !cascade))
        return;
    const int32_t mb = (max_seq_len + block_size - 1) / block_size;
    // the shared prefix is read through row 0; a decode there has no copy of
    // its own, so its first P/bs blocks get one
    const int32_t pb = cascade && num_decodes > 0 ? common_prefix_len / block_size : 0;
    size_t off = w.total;
    // the table first: a read past its last row (a length above max_seq_len,
    // flagged) stays inside the workspace
    w.fp8_table = off;
    off = round256(off + size_t(num_seqs) * mb * 4);
    w.fp8_scratch = off;
    w.fp8_scratch_blocks = int64_t(nprefill) * mb + pb;
    off = round256(off + size_t(w.fp8_scratch_blocks) * 2 * block_size * num_kv_heads *
                             head_size * 2);
    w.fp8_blocks_per_seq = mb;
    w.fp8_prefix_blocks = pb;
    w.total = off;
}

// A bf16 pool of small pages (16 keys) read by a prefill pass that is mostly
// queries (at least 256 query tokens per prefill sequence on average): the
// prefill sequences' keys are first copied into 128-key blocks, so that the
// tensor-core pass reads one TMA box per tile half instead of one per page
// (measured on GB300: 55% of the bf16 peak at 16-key pages, 66% at 32 and
// above).  Decode-like chunks (few queries over a long context) would pay the
// copy for little work, so they read the pages as they are.
void plan_reblock(Workspace &w, bool kv_fp8, int32_t num_tokens, int32_t num_seqs,
                  int32_t num_decodes, int32_t max_seq_len, int32_t block_size,
                  int32_t num_kv_heads, int32_t head_size)
{
    w.reblock_table = w.reblock_scratch = w.total;
    w.reblock_blocks_per_seq = 0;
    w.reblock_blocks = 0;
    const int32_t nprefill = num_seqs - num_decodes;
    if (kv_fp8 || nprefill <= 0 || block_size >= 32 || 32 % block_size != 0)
        return;
    if (int64_t(num_tokens) - num_decodes < int64_t(256) * nprefill)
        return;
    const int32_t mb = (max_seq_len + 127) / 128;
    size_t off = w.total;
    // the table first (as for the fp8 copy): a read past its last row stays
    // inside the workspace
    w.reblock_table = off;
    off = round256(off + size_t(num_seqs) * mb * 4);
    w.reblock_scratch = off;
    w.reblock_blocks = int64_t(nprefill) * mb;
    off = round256(off + size_t(w.reblock_blocks) * 2 * 128 * num_kv_heads * head_size * 2);
    w.reblock_blocks_per_seq = mb;
    w.total = off;
}

static bool scale_ok(float s) { return s > 0.f && s <= 3.4e38f; }

// Checks shared by pka_workspace_size and pka_paged_attn_forward.
static pka_status check_shape(const pka_meta *m, int32_t num_tokens, int32_t num_heads,
                              int32_t num_kv_heads, int32_t head_size, int32_t block_size)
{
    if (!m)
        return fail(PKA_ERR_INVALID_ARG, "meta is NULL");
    if (m->kv_layout != PKA_LAYOUT_NHD && m->kv_layout != PKA_LAYOUT_HND)
        return fail(PKA_ERR_INVALID_ARG, "unknown kv_layout %d", m->kv_layout);
    if (m->kv_dtype != PKA_KV_BF16 && m->kv_dtype != PKA_KV_FP8_E4M3)
        return fail(PKA_ERR_INVALID_ARG, "unknown kv_dtype %d", m->kv_dtype);
    if (m->kv_dtype == PKA_KV_FP8_E4M3 && !(scale_ok(m->k_scale) && scale_ok(m->v_scale)))
        return fail(PKA_ERR_INVALID_ARG, "k_scale / v_scale must be positive and finite");
    if (block_size <= 0 || block_size % 16 != 0)
        return fail(PKA_ERR_INVALID_ARG, "Block size must be a multiple of 16 (got %d).",
                    block_size);
    if (head_size <= 0 || head_size % 8 != 0 || head_size > 256)
        return fail(PKA_ERR_INVALID_ARG,
                    "head_size must be a positive multiple of 8 not above 256 (got %d)",
                    head_size);
    if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0)
        return fail(PKA_ERR_INVALID_ARG,
                    "num_heads (%d) must be a positive multiple of num_kv_heads (%d)", num_heads,
                    num_kv_heads);
    if (num_tokens < 0 || m->num_seqs < 0 || m->num_decodes < 0 ||
        m->num_decodes > m->num_seqs || m->num_decodes > num_tokens)
        return fail(PKA_ERR_INVALID_ARG,
                    "inconsistent sizes: num_tokens %d, num_seqs %d, num_decodes %d", num_tokens,
                    m->num_seqs, m->num_decodes);
    // a decode may hold no key (L_s = 0: a context-parallel rank's empty
    // shard), so max_seq_len 0 is a valid bound for a decode-only batch
    if (m->max_seq_len < 0 || (m->num_seqs > m->num_decodes && m->max_seq_len < 1))
        return fail(PKA_ERR_INVALID_ARG,
                    "max_seq_len must be >= 0, and >= 1 when prefills are present");
    if (m->num_seqs > m->num_decodes && m->max_query_len < 1)
        return fail(PKA_ERR_INVALID_ARG, "max_query_len must be >= 1 when prefills are present");
    if (m->common_prefix_len < 0 || m->common_prefix_len % block_size != 0 ||
        (m->common_prefix_len > 0 && m->common_prefix_len >= m->max_seq_len))
        return fail(PKA_ERR_INVALID_ARG,
                    "common_prefix_len (%d) must be a multiple of block_size below max_seq_len",
                    m->common_prefix_len);
    if (m->split_kv_tokens < 0)
        return fail(PKA_ERR_INVALID_ARG, "split_kv_tokens must be >= 0");
    if (m->num_seqs > 0 &&
        int64_t(m->block_table_stride) * block_size < int64_t(m->max_seq_len))
        return fail(PKA_ERR_INVALID_ARG,
                    "block_table_stride %d too small for max_seq_len %d at block_size %d",
                    m->block_table_stride, m->max_seq_len, block_size);
    if (head_size != 64 && head_size != 128)
        return fail(PKA_ERR_UNSUPPORTED, "head_size %d is not built (64, 128)", head_size);
    if (num_kv_heads != 1 && num_kv_heads != 2 && num_kv_heads != 4 && num_kv_heads != 8)
        return fail(PKA_ERR_UNSUPPORTED, "num_kv_heads %d is not built (1, 2, 4, 8)",
                    num_kv_heads);
    if (m->num_decodes > 0 && num_heads / num_kv_heads > 8)
        return fail(PKA_ERR_UNSUPPORTED, "decode query-head group %d above 8",
                    num_heads / num_kv_heads);
    if (m->num_decodes > 65535)
        return fail(PKA_ERR_UNSUPPORTED, "more than 65535 decodes in one call");
    if (m->kv_dtype == PKA_KV_FP8_E4M3) {
        if (head_size != 128)
            return fail(PKA_ERR_UNSUPPORTED, "fp8 pool: head_size %d is not built (128)",
                        head_size);
    }
    return PKA_OK;
}

// The whole host plan of one forward (pka_workspace_size and the forward
// itself make the same one): decode grid, cascade split, workspace carve-up.
struct ForwardPlan {
    DecodePlan dp;
    CascadePlan cp;
    MixedPlan mp;
    Workspace ws;
};

static ForwardPlan plan_forward(const pka_meta *m, int32_t num_tokens, int32_t num_heads,
                                int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                                int sms, bool allow_reblock = true)
{
    ForwardPlan fp;
    const bool cascade = m->common_prefix_len > 0;
    const bool fp8 = m->kv_dtype == PKA_KV_FP8_E4M3;
    fp.dp = plan_decode(m->split_kv_tokens, m->num_decodes, num_kv_heads, sms);
    if (cascade) {
        fp.cp = plan_cascade(num_tokens, num_heads, num_kv_heads, head_size,
                             m->common_prefix_len, m->num_decodes, m->max_seq_len, fp8,
                             fp.dp.chunk == m->num_decodes, sms);
        if (fp.cp.overlap)
            fp.dp.grid = sms - fp.cp.pre_ctas;  // the decode takes the SMs the prefix leaves
    } else {
        fp.mp = plan_mixed(num_tokens, num_heads, num_kv_heads, head_size, m->num_decodes,
                           m->num_seqs, m->max_seq_len, fp8, fp.dp.chunk == m->num_decodes, sms);
        if (fp.mp.overlap)
            fp.dp.grid = fp.mp.dec_ctas;
    }
    fp.ws = plan_workspace(fp.dp, num_tokens, m->num_decodes, num_heads, head_size, cascade,
                           fp.cp.pre_splits);
    plan_fp8_prefill(fp.ws, fp8, m->num_seqs, m->num_decodes, m->max_seq_len,
                     m->common_prefix_len, block_size, num_kv_heads, head_size);
    if (allow_reblock)
        plan_reblock(fp.ws, fp8, num_tokens, m->num_seqs, m->num_decodes, m->max_seq_len,
                     block_size, num_kv_heads, head_size);
    else
        plan_reblock(fp.ws, true, 0, 0, 0, 0, block_size, 0, 0);  // none: offsets only
    return fp;
}

// Smallest workspace of a forward (its plan without the prefill re-blocking).
size_t workspace_size_min(const pka_meta *m, int32_t num_tokens, int32_t num_heads,
                          int32_t num_kv_heads, int32_t head_size, int32_t block_size)
{
    if (check_shape(m, num_tokens, num_heads, num_kv_heads, head_size, block_size) != PKA_OK)
        return 0;
    return plan_forward(m, num_tokens, num_heads, num_kv_heads, head_size, block_size,
                        sm_count(), false)
        .ws.total;
}

}  // namespace pka

using namespace pka;

extern "C" {

const char *pka_last_error(void) { return g_msg; }

uint64_t pka_kernel_launches(void) { return g_launches; }

pka_status pka_set_kernel_events(int32_t kernel, void *start, void *stop)
{
    if (kernel != PKA_KERNEL_DECODE && kernel != PKA_KERNEL_PREFILL)
        return fail(PKA_ERR_INVALID_ARG, "unknown kernel id %d", kernel);
    g_ev_start[kernel] = static_cast<cudaEvent_t>(start);
    g_ev_stop[kernel] = static_cast<cudaEvent_t>(stop);
    return PKA_OK;
}

pka_status pka_test_skip_copies(int32_t on)
{
    g_test_skip_copies = on ? 1 : 0;
    return PKA_OK;
}

pka_status pka_reshape_and_cache(const void *key, const void *value, void *kv_cache,
                                 const int64_t *slot_mapping, int32_t num_tokens,
                                 int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                                 int64_t num_blocks, void *stream)
{
    return pka_reshape_and_cache_ex(key, value, kv_cache, slot_mapping, num_tokens, num_kv_heads,
                                    head_size, block_size, num_blocks, PKA_LAYOUT_NHD, stream);
}

pka_status pka_reshape_and_cache_ex(const void *key, const void *value, void *kv_cache,
                                    const int64_t *slot_mapping, int32_t num_tokens,
                                    int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                                    int64_t num_blocks, int32_t kv_layout, void *stream)
{
    if (kv_layout != PKA_LAYOUT_NHD && kv_layout != PKA_LAYOUT_HND)
        return fail(PKA_ERR_INVALID_ARG, "unknown kv_layout %d", kv_layout);
    if (num_tokens < 0)
        return fail(PKA_ERR_INVALID_ARG, "num_tokens < 0");
    if (block_size <= 0 || block_size % 16 != 0)
        return fail(PKA_ERR_INVALID_ARG, "Block size must be a multiple of 16 (got %d).",
                    block_size);
    if (head_size <= 0 || head_size % 8 != 0 || num_kv_heads <= 0 || num_blocks <= 0)
        return fail(PKA_ERR_INVALID_ARG,
                    "bad shape: head_size %d (multiple of 8), num_kv_heads %d, num_blocks %lld",
                    head_size, num_kv_heads, static_cast<long long>(num_blocks));
    if (num_tokens == 0)
        return PKA_OK;
    if (!key || !value || !kv_cache || !slot_mapping)
        return fail(PKA_ERR_INVALID_ARG, "null pointer argument");
    if (!aligned(key, 16) || !aligned(value, 16) || !aligned(kv_cache, 16) ||
        !aligned(slot_mapping, 8))
        return fail(PKA_ERR_INVALID_ARG, "misaligned pointer (16 bytes required)");
    cudaError_t e = launch_reshape_and_cache(key, value, kv_cache, slot_mapping, num_tokens,
                                             num_kv_heads, head_size, block_size, num_blocks,
                                             kv_layout == PKA_LAYOUT_HND ? 1 : 0,
                                             static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "reshape_and_cache launch");
    return PKA_OK;
}

pka_status pka_reshape_and_cache_fp8(const void *key, const void *value, void *kv_cache,
                                     const int64_t *slot_mapping, int32_t num_tokens,
                                     int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                                     int64_t num_blocks, int32_t kv_layout, float k_scale,
                                     float v_scale, void *stream)
{
    if (kv_layout != PKA_LAYOUT_NHD && kv_layout != PKA_LAYOUT_HND)
        return fail(PKA_ERR_INVALID_ARG, "unknown kv_layout %d", kv_layout);
    if (num_tokens < 0)
        return fail(PKA_ERR_INVALID_ARG, "num_tokens < 0");
    if (block_size <= 0 || block_size % 16 != 0)
        return fail(PKA_ERR_INVALID_ARG, "Block size must be a multiple of 16 (got %d).",
                    block_size);
    if (head_size <= 0 || head_size % 8 != 0 || num_kv_heads <= 0 || num_blocks <= 0)
        return fail(PKA_ERR_INVALID_ARG,
                    "bad shape: head_size %d (multiple of 8), num_kv_heads %d, num_blocks %lld",
                    head_size, num_kv_heads, static_cast<long long>(num_blocks));
    if (!scale_ok(k_scale) || !scale_ok(v_scale))
        return fail(PKA_ERR_INVALID_ARG, "k_scale / v_scale must be positive and finite");
    if (head_size % 16 != 0)
        return fail(PKA_ERR_UNSUPPORTED, "fp8 pool: head_size %d not a multiple of 16",
                    head_size);
    if (num_tokens == 0)
        return PKA_OK;
    if (!key || !value || !kv_cache || !slot_mapping)
        return fail(PKA_ERR_INVALID_ARG, "null pointer argument");
    if (!aligned(key, 16) || !aligned(value, 16) || !aligned(kv_cache, 16) ||
        !aligned(slot_mapping, 8))
        return fail(PKA_ERR_INVALID_ARG, "misaligned pointer (16 bytes required)");
    cudaError_t e = launch_reshape_and_cache_fp8(
        key, value, kv_cache, slot_mapping, num_tokens, num_kv_heads, head_size, block_size,
        num_blocks, kv_layout == PKA_LAYOUT_HND ? 1 : 0, k_scale, v_scale,
        static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "reshape_and_cache_fp8 launch");
    return PKA_OK;
}

size_t pka_workspace_size(const pka_meta *meta, int32_t num_tokens, int32_t num_heads,
                          int32_t num_kv_heads, int32_t head_size, int32_t block_size)
{
    if (check_shape(meta, num_tokens, num_heads, num_kv_heads, head_size, block_size) != PKA_OK)
        return 0;
    return plan_forward(meta, num_tokens, num_heads, num_kv_heads, head_size, block_size,
                        sm_count())
        .ws.total;
}

size_t pka_workspace_size_min(const pka_meta *meta, int32_t num_tokens, int32_t num_heads,
                              int32_t num_kv_heads, int32_t head_size, int32_t block_size)
{
    return workspace_size_min(meta, num_tokens, num_heads, num_kv_heads, head_size, block_size);
}

// This step's new K/V rows for pka_paged_attn_forward_fused.
struct FuseArgs {
    const void *key;
    const void *value;
    const int64_t *slots;
    void *kv_cache;
};

static pka_status forward_impl(const void *query, const void *kv_cache, const pka_meta *meta,
                               void *out, float *lse, int32_t num_tokens, int32_t num_heads,
                               int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                               int64_t num_blocks, float scale, int32_t causal, void *workspace,
                               size_t workspace_bytes, void *stream, const FuseArgs *fuse)
{
    pka_status st = check_shape(meta, num_tokens, num_heads, num_kv_heads, head_size, block_size);
    if (st != PKA_OK)
        return st;
    if (num_tokens == 0 || meta->num_seqs == 0)
        return PKA_OK;
    if (!query || !kv_cache || !out || !meta->query_start_loc || !meta->seq_lens ||
        !meta->block_table)
        return fail(PKA_ERR_INVALID_ARG, "null pointer argument");
    if (!aligned(query, 16) || !aligned(kv_cache, 16) || !aligned(out, 16) ||
        (lse && !aligned(lse, 4)))
        return fail(PKA_ERR_INVALID_ARG, "misaligned pointer (16 bytes required)");
    if (query == out)
        return fail(PKA_ERR_INVALID_ARG, "out must not alias query");
    if (num_blocks <= 0)
        return fail(PKA_ERR_INVALID_ARG, "num_blocks must be positive");
    // the TMA row coordinate (page*block_size + offset, or page*num_kv_heads
    // + head in HND) is a 32-bit integer
    if (num_blocks * 2 * int64_t(meta->kv_layout == PKA_LAYOUT_HND ? num_kv_heads : block_size) >=
        (int64_t(1) << 31))
        return fail(PKA_ERR_UNSUPPORTED, "pool has more than 2^31 rows");
    if (!(scale > 0.f) || scale != scale || scale > 1e30f)
        return fail(PKA_ERR_INVALID_ARG, "scale must be a positive finite number");

    const bool cascade = meta->common_prefix_len > 0;
    const int32_t kv_begin = meta->common_prefix_len;
    const int num_prefills = meta->num_seqs - meta->num_decodes;
    if (num_prefills > kMaxPrefillSeqsPerCall)
        return fail(PKA_ERR_UNSUPPORTED, "more than %d prefill sequences in one call",
                    kMaxPrefillSeqsPerCall);

    Fwd f;
    f.query = query;
    f.kv_cache = kv_cache;
    f.qsl = meta->query_start_loc;
    f.seq_lens = meta->seq_lens;
    f.block_table = meta->block_table;
    f.bt_stride = meta->block_table_stride;
    f.num_seqs = meta->num_seqs;
    f.num_decodes = meta->num_decodes;
    f.max_query_len = meta->max_query_len;
    f.max_seq_len = meta->max_seq_len;
    f.common_prefix_len = meta->common_prefix_len;
    f.out = out;
    f.lse = lse;
    f.num_tokens = num_tokens;
    f.num_heads = num_heads;
    f.num_kv_heads = num_kv_heads;
    f.head_size = head_size;
    f.block_size = block_size;
    f.num_blocks = num_blocks;
    f.kv_hnd = meta->kv_layout == PKA_LAYOUT_HND ? 1 : 0;
    f.kv_fp8 = meta->kv_dtype == PKA_KV_FP8_E4M3 ? 1 : 0;
    f.k_scale = meta->k_scale;
    f.v_scale = meta->v_scale;
    f.scale = scale;
    f.causal = causal;
    f.stream = static_cast<cudaStream_t>(stream);
    f.num_sms = sm_count();
    f.test_skip_copies = g_test_skip_copies;
    if (fuse) {
        f.fuse_write = 1;
        f.new_key = fuse->key;
        f.new_value = fuse->value;
        f.slots = fuse->slots;
        f.kv_cache_w = fuse->kv_cache;
    }
    const bool fuse_prefill_rows = fuse && num_tokens > meta->num_decodes;

    ForwardPlan plan = plan_forward(meta, num_tokens, num_heads, num_kv_heads, head_size,
                                    block_size, f.num_sms);
    // the re-blocking copy is an optimisation: with a workspace sized for the
    // plan without it, the prefill reads the pages as they are
    if (plan.ws.reblock_blocks > 0 && workspace_bytes < plan.ws.total)
        plan = plan_forward(meta, num_tokens, num_heads, num_kv_heads, head_size, block_size,
                            f.num_sms, false);
    const DecodePlan &dp = plan.dp;
    const CascadePlan &cp = plan.cp;
    const MixedPlan &mp = plan.mp;
    const Workspace &ws = plan.ws;
    if (ws.fp8_scratch_blocks * 2 * block_size >= (int64_t(1) << 31) ||
        ws.reblock_blocks * 2 * 128 >= (int64_t(1) << 31))
        return fail(PKA_ERR_UNSUPPORTED, "prefill copy has more than 2^31 rows");
    if (ws.total > 0 && (!workspace || workspace_bytes < ws.total || !aligned(workspace, 256)))
        return fail(PKA_ERR_WORKSPACE, "workspace needs %zu bytes, 256-byte aligned (got %zu)",
                    ws.total, workspace_bytes);
    char *wsp = static_cast<char *>(workspace);

    CUtensorMap kv_map;
    CUresult cr = encode_kv_map_heads(&kv_map, kv_cache, head_size, num_kv_heads, block_size,
                                      num_blocks, f.kv_hnd, f.kv_fp8 ? 1 : 2);
    if (cr != CUDA_SUCCESS)
        return fail(PKA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", int(cr));

    cudaError_t e;
    if (fuse_prefill_rows) {
        // The prefill tokens' new rows go first, through the cache-write
        // kernel (one warp per token over the whole GPU); the decode launch
        // writes only each decode's own row, into the tile it attends over and
        // into the pool.  Written inside the decode launch, those rows held
        // back its first copies (measured: the decode of a batch with 8,192
        // prefill tokens ran 4% slower over a bf16 pool, 19% over fp8).
        const size_t row = size_t(num_kv_heads) * head_size * 2;  // bytes of a bf16 row
        const int32_t nd = meta->num_decodes;
        const char *k = static_cast<const char *>(fuse->key) + size_t(nd) * row;
        const char *v = static_cast<const char *>(fuse->value) + size_t(nd) * row;
        e = f.kv_fp8 ? launch_reshape_and_cache_fp8(k, v, fuse->kv_cache, fuse->slots + nd,
                                                     num_tokens - nd, num_kv_heads, head_size,
                                                     block_size, num_blocks, f.kv_hnd, f.k_scale,
                                                     f.v_scale, f.stream)
                     : launch_reshape_and_cache(k, v, fuse->kv_cache, fuse->slots + nd,
                                                num_tokens - nd, num_kv_heads, head_size,
                                                block_size, num_blocks, f.kv_hnd, f.stream);
        if (e != cudaSuccess)
            return cuda_fail(e, "cache write launch");
    }
    // An fp8 pool: the tensor-core prefill (prefill sequences, the cascade's
    // shared prefix) runs on bf16 copies of the blocks it reads, made in the
    // workspace as exact code values, with k_scale in the score scale and
    // v_scale on the output; the decodes read the codes themselves.
    Fwd fp = f;
    int32_t *fp8_table = reinterpret_cast<int32_t *>(wsp + ws.fp8_table);
    void *fp8_scratch = wsp + ws.fp8_scratch;
    const int32_t mb = ws.fp8_blocks_per_seq;
    // A cascade over an fp8 pool whose passes run side by side: the prefix
    // pass is the copy's programmatic dependent (it waits for the copy before
    // it reads the blocks), so the suffix decode, the pass's own dependent,
    // starts beside the copy instead of after it.  Nothing may stand between
    // the launches: both work counters are zeroed and the timing brackets
    // (instrumentation) opened before the copy.
    const bool copy_chained = cascade && cp.overlap && f.kv_fp8 && ws.fp8_scratch_blocks > 0 &&
                              meta->num_decodes > 0;
    if (copy_chained) {
        e = cudaMemsetAsync(wsp + ws.counters, 0, size_t(dp.chunk) * 4, f.stream);
        if (e == cudaSuccess)
            e = cudaMemsetAsync(reinterpret_cast<int32_t *>(wsp + ws.pf_counters) + 1, 0,
                                sizeof(int32_t), f.stream);
        if (e != cudaSuccess)
            return cuda_fail(e, "counter reset");
        record_start(PKA_KERNEL_PREFILL, f.stream);
        record_start(PKA_KERNEL_DECODE, f.stream);
    }
    if (f.kv_fp8 && ws.fp8_scratch_blocks > 0) {
        fp.kv_cache = fp8_scratch;
        fp.block_table = fp8_table;
        fp.bt_stride = mb;
        fp.num_blocks = ws.fp8_scratch_blocks;
        fp.kv_hnd = 0;
        fp.kv_fp8 = 0;
        fp.scale = f.scale * f.k_scale;
        fp.out_scale = f.v_scale;
        // before any pass: the prefill rows' copies when no decode launch writes
        // new rows first (the prefix is then row 0's own copy), else the prefix
        // blocks of row 0 (no new row lies in the prefix)
        if (meta->num_decodes == 0)
            e = launch_dequant_blocks(f, fp8_scratch, fp8_table, 0, num_prefills, mb, mb, 0, mb);
        else
            e = launch_dequant_blocks(f, fp8_scratch, fp8_table, 0, 1, 0, ws.fp8_prefix_blocks,
                                      int64_t(num_prefills) * mb, mb, copy_chained);
        if (e != cudaSuccess)
            return cuda_fail(e, "fp8 block copy launch");
    }
    // [blog] "Que aporta FlashInfer: JIT y cascade attention": with a shared
    // prefix P, the prefix keys [0, P) are attended once for every query (a
    // tensor-core pass with no mask), each sequence's own suffix [P, L_s) by
    // the decode / prefill passes, and the parts are merged by log-sum-exp.
    // The prefix pass is bound by the tensor cores and the suffix decode by
    // HBM, so when the plan says so they run side by side on disjoint SMs: the
    // decode is launched as the prefix pass's dependent (it starts on the SMs
    // the pass leaves free and completes after it), its rows go out as fp32
    // partials, and one combine kernel merges every token's parts at the end.
    DecodeOut dout;
    if (cascade) {
        dout.o_suf = reinterpret_cast<float *>(wsp + ws.o_suf);
        dout.lse_suf = reinterpret_cast<float *>(wsp + ws.lse_suf);
        dout.after_prefix = cp.overlap;
        dout.dependent_follows = true;  // the combine
        if (cp.overlap) {
            // nothing may stand between the two launches: zero the decode's
            // counters first (before the copy when it is chained)
            if (!copy_chained) {
                e = cudaMemsetAsync(wsp + ws.counters, 0, size_t(dp.chunk) * 4, f.stream);
                if (e != cudaSuccess)
                    return cuda_fail(e, "counter reset");
                // the two passes run at the same time: both timing brackets
                // (instrumentation) cover the pair
                record_start(PKA_KERNEL_PREFILL, f.stream);
                record_start(PKA_KERNEL_DECODE, f.stream);
            }
            dout.counters_zeroed = true;
        }
        PrefillPass pre{0, kv_begin, 0, true, reinterpret_cast<float *>(wsp + ws.o_pre),
                        reinterpret_cast<float *>(wsp + ws.lse_pre), 0,
                        reinterpret_cast<int32_t *>(wsp + ws.pf_counters) + 1, cp.pre_splits};
        pre.max_ctas = cp.overlap ? cp.pre_ctas : 0;
        pre.trigger_dependents = cp.overlap;
        pre.after_copy = copy_chained;
        pre.counter_zeroed = copy_chained;
        if (!cp.overlap)
            record_start(PKA_KERNEL_PREFILL, f.stream);
        e = launch_prefill(fp, pre);
        if (!cp.overlap)
            record_stop(PKA_KERNEL_PREFILL, f.stream);
        if (e != cudaSuccess)
            return cuda_fail(e, "cascade prefix launch");
    }
    // The prefill pass of the sequences [num_decodes, S).  With decodes beside it
    // (the mixed plan) it is the decode's programmatic dependent: it starts on
    // the SMs the decode leaves and takes the decode's SMs as they free up, so
    // its counter, the re-blocking copy and the timing brackets go first --
    // nothing may stand between the two launches.
    PrefillPass pf{kv_begin, INT32_MAX, causal ? 1 : 0, false,
                   cascade ? reinterpret_cast<float *>(wsp + ws.o_suf) : nullptr,
                   cascade ? reinterpret_cast<float *>(wsp + ws.lse_suf) : nullptr, 0,
                   reinterpret_cast<int32_t *>(wsp + ws.pf_counters)};
    // the fused call over a bf16 pool: key tiles of this step's keys only are
    // read from its key/value rows (identical to what was just written into
    // the pool)
    pf.new_from_input = f.fuse_write && !f.kv_fp8;
    // a bf16 pool of small pages: the pass reads the re-blocked copy (of the
    // tiles it still reads from the pool)
    Fwd fr = fp;
    auto reblock = [&]() -> cudaError_t {
        int32_t *rtable = reinterpret_cast<int32_t *>(wsp + ws.reblock_table);
        void *rscratch = wsp + ws.reblock_scratch;
        const int32_t rb = ws.reblock_blocks_per_seq;
        const cudaError_t re = launch_reblock(f, rscratch, rtable, meta->num_decodes,
                                              num_prefills, rb, 0, rb,
                                              pf.new_from_input ? kv_begin : -1);
        fr.kv_cache = rscratch;
        fr.block_table = rtable;
        fr.bt_stride = rb;
        fr.num_blocks = ws.reblock_blocks;
        fr.block_size = 128;
        fr.kv_hnd = 0;
        return re;
    };
    const bool beside = mp.overlap && num_prefills > 0 && !cascade;
    if (beside) {
        e = cudaMemsetAsync(pf.item_counter, 0, sizeof(int32_t), f.stream);
        if (e != cudaSuccess)
            return cuda_fail(e, "counter reset");
        pf.counter_zeroed = true;
        pf.after_decode = true;
        if (ws.reblock_blocks > 0 && (e = reblock()) != cudaSuccess)
            return cuda_fail(e, "prefill re-block launch");
        // an fp8 pool: the prefill sequences' blocks as bf16 (the decode writes
        // only its own sequences' new rows, into their last blocks)
        if (f.kv_fp8 &&
            (e = launch_dequant_blocks(f, fp8_scratch, fp8_table, meta->num_decodes,
                                       num_prefills, mb, mb, 0, mb)) != cudaSuccess)
            return cuda_fail(e, "fp8 block copy launch");
        dout.dependent_follows = true;
        // the two passes run at the same time: both timing brackets
        // (instrumentation) cover the pair
        record_start(PKA_KERNEL_PREFILL, f.stream);
    }
    // A decode-only batch of a few long decodes (at least 4 SMs per decode, more
    // stages than SMs by the longest length): each decode spreads over many
    // CTAs, and their pieces are merged by a launch over the whole GPU after the
    // decode's rather than each by the decode's last CTA (measured on 8 of
    // decode_heavy's decodes: that merge folds ~19 parts, 2 per L2 round trip,
    // and ended ~12 us after the rest of the grid).
    if (!cascade && num_prefills == 0 && meta->num_decodes > 0 &&
        dp.chunk >= meta->num_decodes && dp.target_keys == 0) {
        const int64_t sk = int64_t(f.kv_fp8 ? 32 : 16) * (8 / num_kv_heads);  // keys per stage
        const int64_t longest = (int64_t(meta->max_seq_len) + sk - 1) / sk;
        if (int64_t(dp.grid) >= 4 * int64_t(meta->num_decodes) &&
            int64_t(meta->num_decodes) * longest > dp.grid)
            dout.defer_merge = true;
    }
    // A small decode-only batch that the kernel divides one sequence per CTA
    // (at most kAlignedMaxStages stages per decode and at most one stage per
    // CTA in all, by max_seq_len) merges no pieces across CTAs: its counters
    // are not reset (one launch less; the kernel checks the lengths).
    if (!cascade && num_prefills == 0 && meta->num_decodes > 0 && dp.target_keys == 0 &&
        dp.chunk >= meta->num_decodes) {
        const int64_t sk = int64_t(f.kv_fp8 ? 32 : 16) * (8 / num_kv_heads);  // keys per stage
        const int64_t longest = std::max<int64_t>(1, (int64_t(meta->max_seq_len) + sk - 1) / sk);
        if (longest <= kAlignedMaxStages && int64_t(meta->num_decodes) * longest <= dp.grid)
            dout.expect_aligned = true;
    }
    if (!cp.overlap)
        record_start(PKA_KERNEL_DECODE, f.stream);
    e = launch_decode(f, dp, ws, wsp, kv_map, kv_begin, dout);
    if (!beside)
        record_stop(PKA_KERNEL_DECODE, f.stream);
    if (cp.overlap)
        record_stop(PKA_KERNEL_PREFILL, f.stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "decode launch");
    if (num_prefills > 0) {
        // fp8 after the decode launch (which wrote this step's rows): the
        // prefill sequences' blocks (beside the decode: copied before it)
        if (f.kv_fp8 && meta->num_decodes > 0 && !beside) {
            e = launch_dequant_blocks(f, fp8_scratch, fp8_table, meta->num_decodes, num_prefills,
                                      mb, mb, 0, mb);
            if (e != cudaSuccess)
                return cuda_fail(e, "fp8 block copy launch");
        }
        if (!beside && ws.reblock_blocks > 0 && (e = reblock()) != cudaSuccess)
            return cuda_fail(e, "prefill re-block launch");
        if (!cascade && !beside)
            record_start(PKA_KERNEL_PREFILL, f.stream);
        e = launch_prefill(fr, pf);
        if (beside)
            record_stop(PKA_KERNEL_DECODE, f.stream);
        if (!cascade)
            record_stop(PKA_KERNEL_PREFILL, f.stream);
        if (e != cudaSuccess)
            return cuda_fail(e, "prefill launch");
    }
    if (cascade) {
        e = launch_cascade_combine(f, ws, wsp);
        if (e != cudaSuccess)
            return cuda_fail(e, "cascade combine launch");
    }
    return PKA_OK;
}

pka_status pka_paged_attn_forward(const void *query, const void *kv_cache, const pka_meta *meta,
                                  void *out, float *lse, int32_t num_tokens, int32_t num_heads,
                                  int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                                  int64_t num_blocks, float scale, int32_t causal,
                                  void *workspace, size_t workspace_bytes, void *stream)
{
    return forward_impl(query, kv_cache, meta, out, lse, num_tokens, num_heads, num_kv_heads,
                        head_size, block_size, num_blocks, scale, causal, workspace,
                        workspace_bytes, stream, nullptr);
}

pka_status pka_paged_attn_forward_fused(const void *query, const void *key, const void *value,
                                        const int64_t *slot_mapping, void *kv_cache,
                                        const pka_meta *meta, void *out, float *lse,
                                        int32_t num_tokens, int32_t num_heads,
                                        int32_t num_kv_heads, int32_t head_size,
                                        int32_t block_size, int64_t num_blocks, float scale,
                                        int32_t causal, void *workspace, size_t workspace_bytes,
                                        void *stream)
{
    pka_status st = check_shape(meta, num_tokens, num_heads, num_kv_heads, head_size, block_size);
    if (st != PKA_OK)
        return st;
    if (num_tokens == 0 || meta->num_seqs == 0)
        return PKA_OK;
    if (!key || !value || !slot_mapping)
        return fail(PKA_ERR_INVALID_ARG, "null pointer argument");
    if (!aligned(key, 16) || !aligned(value, 16) || !aligned(slot_mapping, 8))
        return fail(PKA_ERR_INVALID_ARG, "misaligned pointer (16 bytes required)");
    // the prefill tokens' rows are written by the cache-write kernel first,
    // each decode's by the decode launch
    const FuseArgs fa{key, value, slot_mapping, kv_cache};
    return forward_impl(query, kv_cache, meta, out, lse, num_tokens, num_heads, num_kv_heads,
                        head_size, block_size, num_blocks, scale, causal, workspace,
                        workspace_bytes, stream, &fa);
}

pka_status pka_merge_partials(const void *outs, const float *lses, int32_t num_parts, void *out,
                              float *lse_out, int32_t num_tokens, int32_t num_heads,
                              int32_t head_size, int32_t lse_base, void *stream)
{
    if (num_parts < 1 || num_tokens < 0 || num_heads <= 0 || head_size <= 0 ||
        head_size % 8 != 0)
        return fail(PKA_ERR_INVALID_ARG, "bad shape: parts %d tokens %d heads %d head_size %d",
                    num_parts, num_tokens, num_heads, head_size);
    if (lse_base != PKA_LSE_BASE_E && lse_base != PKA_LSE_BASE_2)
        return fail(PKA_ERR_INVALID_ARG, "unknown lse base %d", lse_base);
    if (num_tokens == 0)
        return PKA_OK;
    if (!outs || !lses || !out)
        return fail(PKA_ERR_INVALID_ARG, "null pointer argument");
    if (!aligned(outs, 16) || !aligned(out, 16) || !aligned(lses, 4) ||
        (lse_out && !aligned(lse_out, 4)))
        return fail(PKA_ERR_INVALID_ARG, "misaligned pointer (16 bytes required)");
    const size_t part_bytes = size_t(num_tokens) * num_heads * head_size * 2;
    const char *o0 = static_cast<const char *>(outs);
    const char *o1 = o0 + part_bytes * size_t(num_parts);
    const char *d0 = static_cast<const char *>(out);
    if (d0 < o1 && o0 < d0 + part_bytes)
        return fail(PKA_ERR_INVALID_ARG, "out must not alias outs");
    cudaError_t e = launch_merge_partials(outs, lses, num_parts, out, lse_out, num_tokens,
                                          num_heads, head_size, lse_base == PKA_LSE_BASE_2 ? 1 : 0,
                                          static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "merge_partials launch");
    return PKA_OK;
}

pka_status pka_cascade_merge(const void *out_a, const float *lse_a, const void *out_b,
                             const float *lse_b, void *out, float *lse_out, int32_t num_tokens,
                             int32_t num_heads, int32_t head_size, void *stream)
{
    if (num_tokens < 0 || num_heads <= 0 || head_size <= 0 || head_size % 8 != 0)
        return fail(PKA_ERR_INVALID_ARG, "bad shape: tokens %d heads %d head_size %d",
                    num_tokens, num_heads, head_size);
    if (num_tokens == 0)
        return PKA_OK;
    if (!out_a || !lse_a || !out_b || !lse_b || !out)
        return fail(PKA_ERR_INVALID_ARG, "null pointer argument");
    if (!aligned(out_a, 16) || !aligned(out_b, 16) || !aligned(out, 16) || !aligned(lse_a, 4) ||
        !aligned(lse_b, 4) || (lse_out && !aligned(lse_out, 4)))
        return fail(PKA_ERR_INVALID_ARG, "misaligned pointer (16 bytes required)");
    cudaError_t e = launch_cascade_merge(out_a, lse_a, out_b, lse_b, out, lse_out, num_tokens,
                                         num_heads, head_size, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "cascade_merge launch");
    return PKA_OK;
}

pka_status pka_check_status(void *stream)
{
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "stream synchronize");
    const uint32_t bits =
        kv_write_take_error() | decode_take_error() | prefill_take_error() | merge_take_error();
    if (bits == 0)
        return PKA_OK;
    char buf[256] = "";
    if (bits & kErrSlotOutOfPool)
        strcat(buf, " slot_mapping entry outside the pool;");
    if (bits & kErrBlockOutOfPool)
        strcat(buf, " block_table entry outside the pool;");
    if (bits & kErrWaitTimeout)
        strcat(buf, " pipeline wait timed out;");
    if (bits & kErrTmemAlloc)
        strcat(buf, " tensor-memory allocation failed;");
    if (bits & kErrBadMetadata)
        strcat(buf, " seq_lens/query_start_loc outside the stated bounds;");
    if (bits & kErrBadPartial)
        strcat(buf, " a merge input's lse is +inf or NaN;");
    return fail(PKA_ERR_DEVICE_CHECK, "device check failed:%s", buf);
}

}  // extern "C"
