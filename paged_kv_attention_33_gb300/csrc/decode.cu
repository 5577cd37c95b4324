// decode.cu -- paged decode (split-KV, stream-K) with the split combine fused in.
//
// What it computes (the "El especialista del plato estrella" blog,
// "Por que prefill y decode son problemas opuestos"): one query token per
// sequence against all of that sequence's keys.  The work is memory bound,
// so the kernel is built to keep HBM busy: every byte of K and V is read once,
// for all query heads of its kv head at the same time (GQA packing), and is
// staged into shared memory by TMA ahead of use.
//
// Grid: persistent, one CTA per SM (or, beside a cascade's shared-prefix pass,
// one per SM that pass leaves), stream-K.  The decodes' keys
// [kv_begin, L_s) are cut into stages of 16*(8/Hkv) keys; the flattened list
// of all stages (sequence after sequence) is divided into equal, contiguous
// ranges, one per CTA, so every CTA streams the same number of bytes and its
// TMA ring never drains between sequences.  A CTA's range covers one or more
// "pieces" (the part of one sequence inside the range).  A sequence covered by
// one piece is finished by that CTA; otherwise each piece writes an fp32
// partial and the last CTA to finish a piece of that sequence (an atomic
// counter per sequence) merges them -- the split combine fused into the kernel.
//
// CTA: 8 consumer warps + 1 producer warp.  A pipeline stage holds 8 "units";
// unit u is 16 consecutive keys of kv head k = u % Hkv, slice r = u / Hkv of the
// stage's 16*(8/Hkv) keys (so every warp works in every stage).  The producer
// issues, per slice and 64-dim half (fp8: per 16-key half of a slice), one TMA
// box {128 bytes, 16 keys, Hkv heads} for K and one for V: the pool is viewed
// as a 3-D tensor whose outermost
// dimension is the kv head (NHD: (head_size, num_blocks*2*block_size,
// num_kv_heads), the head stride being one row; HND: (head_size, block_size,
// num_blocks*2*num_kv_heads)) -- the "FlashAttention y FlashInfer" page's
// cache shape with (block, kv, offset) flattened.  One box thus lands every
// head's 16-key tile of the slice, head after head, 128-byte swizzled so that
// the ldmatrix reads below are conflict free; a few large boxes per stage let
// one SM stream almost twice the bytes that one small box per unit and half
// did, so HBM is saturated long before every SM decodes.
// Pages are found through the block table ("Como lee el backend el KV
// paginado": the kernel gathers physical blocks, no contiguous KV).
//
// Consumer warp u owns kv head k and keeps, for the g = H/Hkv query heads of
// k, a transposed accumulator O^T[D x 8] in registers:
//   S^T[16 keys x 8 heads] = K[16 x D] * Q^T[D x 8]        (mma m16n8k16)
//   online softmax per head (column), P^T moved into B-fragment order with
//   movmatrix, then O^T[D x 8] += V^T[D x 16] * P^T[16 x 8] (mma m16n8k16).
// The tensor work is g FLOP per byte of KV, far below the ridge point, so the
// warp-level mma is ample; the kernel is bound by HBM.
//
// An fp8 e4m3 pool (the "FlashAttention y FlashInfer" page, "Resumen en una
// frase" and "Limites y fallos": an fp8 KV cache; one scale per tensor for K
// and V) halves the bytes, so the same stage carries 32 keys per unit, loaded
// as two 16-row boxes of 128-byte code rows.  The codes are converted to f16
// once each (exact: every e4m3 value is an f16 normal), K from 16-byte row
// reads and V from ldmatrix.m16n16.trans.b8 (a byte transpose), and meet
// f16 Q (each head prescaled by a power of two into f16 range, exact for bf16
// values) and f16 P in mma m16n8k16; k_scale is folded into the score scale
// and v_scale into the output scale.  The keys of a unit are taken in an
// order that keeps both the K row reads and the V row gathers free of bank
// conflicts.  (On this GPU an fp8 mma.sync converts both operands itself on
// every call, which would convert each code once per Q or P term.)
//
// At the end of a piece every warp writes its rows straight from registers:
// the final bf16 rows and lse (a cascade's suffix: fp32 rows and log2-sum-exp,
// merged with the shared prefix by a later kernel), or (several pieces, or
// Hkv < 8 where several warps share a kv head) a normalised fp32 partial and
// its log2-sum-exp.
// Fused cache write: the stage holding a decode's new key (key L-1) gets that
// row from the step's K/V rows, and the row is stored at the token's slot, so
// the pool need not hold it before the launch.
// Failure path: every wait is bounded; a warp whose wait gives up raises a
// CTA-wide abort flag, stops computing and writing, but still walks the same
// stage and piece sequence so that every named barrier is reached by all.
#include <math.h>

#include <algorithm>
#include <atomic>
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace pka {

struct DecodeParams {
    const uint32_t *query;  // bf16 pairs, [T, H, D]
    const int32_t *qsl;
    const int32_t *seq_lens;
    const int32_t *block_table;
    int32_t bt_stride;
    int32_t num_tokens;
    int32_t num_heads;
    int32_t num_kv_heads;
    int32_t group;
    int32_t block_size;
    int32_t num_blocks;
    int32_t seq0;         // first decode sequence of this launch
    int32_t nseq;         // decodes in this launch (<= kMaxDecodeChunk)
    int32_t kv_begin;     // first key (cascade suffix: the shared prefix length)
    int32_t target_keys;  // 0, or keys per CTA to aim for (fewer CTAs)
    float scale_log2;     // softmax scale * log2(e)
    __nv_bfloat16 *out;
    float *lse;
    // cascade suffix: each decode row's result over keys [kv_begin, L) goes to
    // o_suf [T, H, D] as a normalised fp32 partial with its log2-sum-exp in
    // lse_suf [T, H] (merged with the shared prefix later), not to out / lse
    float *o_suf;
    float *lse_suf;
    // launched as the dependent of the cascade's shared-prefix pass, which
    // runs on the other SMs at the same time: the grid completes only after
    // that pass completed (griddepcontrol.wait before every CTA exits)
    int32_t after_prefix;
    int32_t trigger_dependents;  // a programmatic dependent launch follows
    // the host did not reset the counters, expecting the one-sequence-per-CTA
    // division (kAlignedMaxStages); a batch that does not allow it is flagged
    int32_t expect_aligned;
    float *o_part;        // [slots, R, H, D] normalised partials
    float *lse_part;      // [slots, R, H], log2 units
    int32_t *counters;    // [nseq] pieces finished per sequence (zeroed before the launch)
    // 1: a sequence split over several CTAs is not merged here; its pieces'
    // partials are left for the merge launch that follows (counters[s] then
    // holds its first CTA | pieces << 16, or 0 when it was not split)
    int32_t defer_merge;
    // fused cache write (pka_paged_attn_forward_fused): this step's K/V rows
    // [T, Hkv, D] and their slots; each decode's own row is written through
    // `pool` (the prefill tokens' rows are written before this launch)
    int32_t fuse_write;
    const uint4 *new_key;
    const uint4 *new_value;
    const int64_t *slots;
    uint4 *pool;
    // fp8 pool: element value = code value x scale (K, V)
    float k_scale;
    float v_scale;
    int32_t test_skip_copies;  // failure-path test: the producer issues nothing
};

constexpr int kConsumerWarps = 8;
constexpr int kDecodeThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxDecodeChunk = 4096;
constexpr float kNegInf = -INFINITY;
constexpr float kLn2 = 0.69314718055994530942f;

// kFp8: the pool holds e4m3 codes (one byte per element) and a unit is 32
// keys (the k extent of an fp8 mma), loaded as two 16-row boxes, so that a
// stage moves as many bytes as a bf16 one.
template <int D, bool kFp8 = false>
struct DecodeCfg {
    static constexpr int kUnitKeys = kFp8 ? 32 : 16;               // keys of one unit
    static constexpr int kRowBytes = D * (kFp8 ? 1 : 2);           // one key of one head
    static constexpr int kHalves = kRowBytes / 128;                // 128-byte TMA boxes per row
    static constexpr int kBoxes = kHalves * kUnitKeys / 16;        // 2 KB tiles of a unit
    // Shared-memory layout of K (and of V) in a stage: for each slice r, box b
    // (a 64-dim half, or an fp8 unit's 16-key half) and head k, the 16-key
    // tile of 2 KB at ((r * kBoxes + b) * Hkv + k) * 2048; unit (k, r) starts
    // at r * Hkv * kUnitBytes + k * 2048 and its box b is Hkv * 2048 further.
    static constexpr int kUnitBytes = kUnitKeys * kRowBytes;
    static constexpr int kKvBytes = kConsumerWarps * kUnitBytes;   // all units of K (or V)
    static constexpr int kStageBytes = 2 * kKvBytes;
    static constexpr int kStages = kStageBytes >= 65536 ? 3 : 6;
    static constexpr int kBarOff = kStages * kStageBytes;
    static constexpr int kMiscOff = kBarOff + 2 * kStages * 8;    // last-piece flag, abort flag
    static constexpr int kPrefixOff = kMiscOff + 16;
    static constexpr size_t kSmemBytes = kPrefixOff + (kMaxDecodeChunk + 1) * 4 + 1024;
    static_assert(kSmemBytes <= 232448, "shared memory");
};

__device__ __forceinline__ float warp_max_heads(float v)
{
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
    return v;
}

__device__ __forceinline__ float warp_sum_heads(float v)
{
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    v += __shfl_xor_sync(0xffffffffu, v, 8);
    v += __shfl_xor_sync(0xffffffffu, v, 16);
    return v;
}

__device__ __forceinline__ void consumer_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

// Bounded wait that also gives up at once when another warp of the CTA gave up.
__device__ __forceinline__ bool dec_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag)
{
    if (mbar_test(bar, parity))
        return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1; it < kWaitIterCap; ++it) {
        if (mbar_test(bar, parity))
            return true;
        if ((it & 127u) == 0) {
            if (*abort_flag)
                return false;
            if (global_timer_ns() - t0 > kWaitLimitNs)
                break;
        }
    }
    flag_error(kErrWaitTimeout);
    *abort_flag = 1;
    return false;
}

// Stages of decode s (at least one, so every decode owns a piece).
__device__ __forceinline__ int dec_stages(const DecodeParams &p, int s, int stage_keys)
{
    const int n = p.seq_lens[p.seq0 + s] - p.kv_begin;
    return n > 0 ? (n + stage_keys - 1) / stage_keys : 1;
}

// CTA whose range [floor(b*TS/G), floor((b+1)*TS/G)) holds stage x.
__device__ __forceinline__ int cta_of_stage(int64_t x, int64_t total, int grid)
{
    return static_cast<int>(((x + 1) * grid + total - 1) / total - 1);
}

__device__ __forceinline__ float warp_max32(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum32(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Merge the partials of decode s (token t): its nparts pieces -- part q lives
// in slot (bf + q / R + s), sub-row q % R.  Warp w takes heads w, w+8, ..., kHB
// of them at a time, lanes along head_size.  The parts are folded in rounds of
// kQB: every load of a round (kQB x kHB log2-sum-exps and rows) is issued
// before any is used, so a merge costs about one L2 round trip per round -- it
// runs at the end of a CTA's range, while the other SMs still stream, where
// each round trip is long.  The merged row goes to out / lse (bf16, ln), or in
// a cascade suffix to o_suf / lse_suf (fp32, log2).
template <int D, int kQB = 2, int kHB = 4>  // kQB: parts per round, kHB: heads per batch
__device__ __forceinline__ void merge_pieces(const DecodeParams &p, int t, int s, int bf,
                                             int nparts, int R, int warp, int lane)
{
    constexpr int kPer = D / 32;  // dims per lane
    using Vec = typename std::conditional<kPer == 4, float4, float2>::type;
    const int H = p.num_heads;
    for (int h0 = warp; h0 < H; h0 += kHB * kConsumerWarps) {
        float M[kHB], W[kHB], acc[kHB][kPer];
#pragma unroll
        for (int j = 0; j < kHB; ++j) {
            M[j] = kNegInf;
            W[j] = 0.f;
#pragma unroll
            for (int e = 0; e < kPer; ++e)
                acc[j][e] = 0.f;
        }
        for (int q0 = 0; q0 < nparts; q0 += kQB) {
            float lq[kQB][kHB];
            Vec v[kQB][kHB];
#pragma unroll
            for (int i = 0; i < kQB; ++i) {
                const int q = q0 + i < nparts ? q0 + i : 0;
                // the kHB heads of part q are rows row0 + 8j: one base address
                const int64_t row0 = (int64_t(bf + q / R + s) * R + q % R) * H + h0;
                const float *lq_p = p.lse_part + row0;
                const Vec *v_p = reinterpret_cast<const Vec *>(p.o_part + row0 * D) + lane;
#pragma unroll
                for (int j = 0; j < kHB; ++j) {
                    if (q0 + i < nparts && h0 + j * kConsumerWarps < H) {
                        lq[i][j] = __ldcg(lq_p + j * kConsumerWarps);
                        v[i][j] = __ldcg(v_p + j * kConsumerWarps * (D / kPer));
                    } else {
                        lq[i][j] = kNegInf;
                        v[i][j] = Vec{};
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < kHB; ++j) {
                float mr = M[j];
#pragma unroll
                for (int i = 0; i < kQB; ++i)
                    mr = fmaxf(mr, lq[i][j]);
                if (mr == kNegInf)
                    continue;  // every part so far is empty
                const float a = exp2f(M[j] - mr);
                W[j] *= a;
#pragma unroll
                for (int e = 0; e < kPer; ++e)
                    acc[j][e] *= a;
#pragma unroll
                for (int i = 0; i < kQB; ++i) {
                    // an empty part adds nothing, whatever its row holds
                    const float w = lq[i][j] == kNegInf ? 0.f : exp2f(lq[i][j] - mr);
                    W[j] += w;
                    const float *x = reinterpret_cast<const float *>(&v[i][j]);
#pragma unroll
                    for (int e = 0; e < kPer; ++e)
                        acc[j][e] += w * x[e];
                }
                M[j] = mr;
            }
        }
#pragma unroll
        for (int j = 0; j < kHB; ++j) {
            const int h = h0 + j * kConsumerWarps;
            if (h >= H)
                continue;
            const int64_t row_out = int64_t(t) * H + h;
            const float inv = W[j] > 0.f ? 1.f / W[j] : 0.f;
            const float lse2 = W[j] > 0.f ? M[j] + log2f(W[j]) : kNegInf;
            if (p.o_suf) {
                float *dst = p.o_suf + row_out * D + lane * kPer;
                Vec r;
                float *rr = reinterpret_cast<float *>(&r);
#pragma unroll
                for (int e = 0; e < kPer; ++e)
                    rr[e] = acc[j][e] * inv;
                *reinterpret_cast<Vec *>(dst) = r;
                if (lane == 0)
                    p.lse_suf[row_out] = lse2;
                continue;
            }
            __nv_bfloat16 *dst = p.out + row_out * D + lane * kPer;
#pragma unroll
            for (int e = 0; e < kPer; e += 2)
                *reinterpret_cast<__nv_bfloat162 *>(dst + e) =
                    __floats2bfloat162_rn(acc[j][e] * inv, acc[j][e + 1] * inv);
            if (lane == 0 && p.lse)
                p.lse[row_out] = lse2 * kLn2;
        }
    }
}

// 16 e4m3 codes of chunk c (elements 16c..16c+15) of token tk's row of kv
// head h: the fp8 pool's quantisation of two 16-byte bf16 vectors.
template <int D>
__device__ __noinline__ uint4 quantized_chunk(const DecodeParams &p, int64_t tk, int h, int c,
                                                 int kv)
{
    const uint4 *src = (kv ? p.new_value : p.new_key) + (tk * p.num_kv_heads + h) * (D / 8) + 2 * c;
    const float sc = kv ? p.v_scale : p.k_scale;
    const uint2 lo = quantize8_e4m3(__ldg(src), sc), hi = quantize8_e4m3(__ldg(src + 1), sc);
    return make_uint4(lo.x, lo.y, hi.x, hi.y);
}

// 16-byte chunk c of kv head h's K (kv 0) or V (kv 1) row of slot sl (block
// sl / bs, offset sl % bs) in a pool of kChunks chunks per row, NHD or HND.
template <bool kHnd>
__device__ __forceinline__ int64_t pool_chunk(const DecodeParams &p, int64_t sl, int kv, int h,
                                              int c, int kChunks)
{
    const int64_t blk = sl / p.block_size, off = sl % p.block_size;
    const int Hkv = p.num_kv_heads;
    const int64_t row = kHnd ? ((blk * 2 + kv) * Hkv + h) * p.block_size + off
                             : ((blk * 2 + kv) * p.block_size + off) * Hkv + h;
    return row * kChunks + c;
}

// The work of one CTA (the kernel below adds the wait of a dependent launch).
template <int D, bool kHnd, bool kFp8>
__device__ __forceinline__ void decode_cta(const CUtensorMap &kv_map, const DecodeParams &p)
{
    static_assert(!kFp8 || D == 128, "the fp8 tile addressing assumes 128-byte rows");
    using Cfg = DecodeCfg<D, kFp8>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Cfg::kBarOff);
    uint64_t *empty = full + Cfg::kStages;
    volatile int *last_flag = reinterpret_cast<volatile int *>(smem + Cfg::kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + Cfg::kMiscOff + 4);
    int32_t *prefix = reinterpret_cast<int32_t *>(smem + Cfg::kPrefixOff);

    const int Hkv = p.num_kv_heads;
    const int R = kConsumerWarps / Hkv;
    const int stage_keys = Cfg::kUnitKeys * R;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nseq = p.nseq;

    // ---- stage prefix sums over the decodes of this launch: each thread sums a
    // run of decodes, then a block-wide exclusive scan of the run sums
    {
        const int per = (nseq + kDecodeThreads - 1) / kDecodeThreads;
        const int a = min(nseq, int(threadIdx.x) * per);
        const int e = min(nseq, a + per);
        int sum = 0;
        for (int k = a; k < e; ++k)
            sum += dec_stages(p, k, stage_keys);
        int run = block_exclusive_scan<kDecodeThreads>(sum, prefix + nseq);
        for (int k = a; k < e; ++k) {
            prefix[k] = run;
            run += dec_stages(p, k, stage_keys);
        }
        __syncthreads();
    }
    const int64_t total = prefix[nseq];
    int grid = gridDim.x;
    // a small batch (at most one stage per SM, so at most one sequence per
    // thread here): one sequence per CTA unless one of them is long; the same
    // choice in every CTA
    bool aligned = false;
    if (p.target_keys == 0 && total <= grid) {
        const int k = threadIdx.x;
        aligned = !__syncthreads_or(k < nseq && prefix[k + 1] - prefix[k] > kAlignedMaxStages);
    }
    if (p.expect_aligned && !aligned) {
        // (the same in every CTA) a decode longer than max_seq_len: the
        // counters hold leftovers, so nothing is computed
        if (blockIdx.x == 0 && threadIdx.x == 0)
            flag_error(kErrBadMetadata);
        return;
    }
    if (aligned)
        grid = nseq;
    if (p.target_keys > 0) {
        const int64_t per_cta = (int64_t(p.target_keys) + stage_keys - 1) / stage_keys;
        const int64_t want = (total + per_cta - 1) / per_cta;
        grid = want < 1 ? 1 : (want < grid ? static_cast<int>(want) : grid);
    }
    // every CTA of the effective grid must own at least one stage, so that the
    // CTAs [bf, bl] of a sequence are exactly its pieces
    if (total < grid)
        grid = static_cast<int>(total);
    if (p.defer_merge && blockIdx.x == 0) {
        // where the merge launch finds each split sequence's pieces
        for (int k = threadIdx.x; k < nseq; k += kDecodeThreads) {
            const int kf = aligned ? k : cta_of_stage(prefix[k], total, grid);
            const int kl = aligned ? k : cta_of_stage(prefix[k + 1] - 1, total, grid);
            p.counters[k] = kl > kf ? kf | ((kl - kf + 1) << 16) : 0;
        }
    }
    const int b = blockIdx.x;
    if (b >= grid)
        return;  // whole CTA (uniform): not needed for this batch
    const int64_t lo = aligned ? prefix[b] : int64_t(b) * total / grid;
    const int64_t hi = aligned ? prefix[b + 1] : int64_t(b + 1) * total / grid;
    if (lo >= hi)
        return;  // whole CTA (uniform): no stage falls in its range
    // first sequence of the range: the largest s with prefix[s] <= lo
    int s_first = b;
    if (!aligned) {
        int a = 0, e = nseq;
        while (e - a > 1) {
            const int mid = (a + e) >> 1;
            if (prefix[mid] <= lo)
                a = mid;
            else
                e = mid;
        }
        s_first = a;
    }

    if (threadIdx.x == 0) {
        for (int i = 0; i < Cfg::kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kConsumerWarps);
        }
        *abort_flag = 0;
        *last_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        // lane = one box of every stage: (slice r, K|V, box b), box = the
        // 128-byte half of a bf16 row, or the 16-key half of an fp8 unit, over
        // all Hkv heads (2 KB per head); its block id is looked up for the next
        // stage before waiting for a free slot
        if (lane == 0)
            tma_prefetch_desc(&kv_map);
        const uint64_t policy = l2_policy_evict_first();
        const int ops = R * 2 * Cfg::kBoxes;  // <= 8 * 2 * 2
        const int r = lane / (2 * Cfg::kBoxes);
        const int kv = (lane / Cfg::kBoxes) & 1;
        const int box = lane % Cfg::kBoxes;
        const int half = kFp8 ? 0 : box;          // 128-byte half of the row
        const int key_off = kFp8 ? 16 * box : 0;  // first key of the box in the unit
        int s = s_first;
        // TMA coordinates of the box's 16 keys in the pool map: NHD (page*bs +
        // offset, head 0), HND (offset, page*Hkv + head 0), page = block*2 +
        // (K|V); row = -1: no keys (a box whose first key is past the end is not
        // loaded, its block-table entry is not valid); live16 = loaded 16-key
        // blocks of each kv head, the same for all lanes
        auto lookup = [&](int64_t x, int seq, int &row, int &c1, int &live16) {
            // the table entry is read before the length is known (the row of
            // the table is in bounds), so that both loads are in flight at once
            const int k0 = p.kv_begin + int(x - prefix[seq]) * stage_keys;
            const int ks = k0 + Cfg::kUnitKeys * r + key_off;
            const int col = ks / p.block_size;
            const int32_t *bt = p.block_table + int64_t(p.seq0 + seq) * p.bt_stride;
            const int blk_raw = lane < ops && col < p.bt_stride ? bt[col] : -1;
            const int L = p.seq_lens[p.seq0 + seq];
            live16 = max(0, min(R * Cfg::kUnitKeys / 16, (L - k0 + 15) / 16));
            row = -1;
            c1 = 0;
            if (lane < ops && ks < L) {
                int blk = blk_raw;
                if (blk < 0 || blk >= p.num_blocks) {
                    flag_error(kErrBlockOutOfPool);
                    blk = 0;  // keep the transaction count whole; result is flagged
                }
                if (kHnd) {
                    c1 = ks % p.block_size;
                    row = (blk * 2 + kv) * Hkv;
                } else {
                    c1 = (blk * 2 + kv) * p.block_size + (ks % p.block_size);
                    row = 0;
                }
            }
        };
        // stages [lo, armed) have been armed (expect_tx) and their copies issued
        int64_t armed = lo;
        int row_next, c1_next, live_next;
        lookup(lo, s, row_next, c1_next, live_next);
        for (int64_t x = p.test_skip_copies ? hi : lo; x < hi; ++x) {
            const int i = int(x - lo);
            const int row = row_next, c1 = c1_next, live16 = live_next;
            const int slot = i % Cfg::kStages;
            const int round = i / Cfg::kStages;
            if (round > 0 && !dec_wait(&empty[slot], (round - 1) & 1, abort_flag))
                break;
            if (lane == 0)  // boxes of 2 KB: live 16-key blocks x heads x K|V (x halves)
                mbar_arrive_expect_tx(&full[slot],
                                      static_cast<uint32_t>(live16 * (kFp8 ? 1 : Cfg::kHalves) *
                                                            Hkv * 2 * 2048));
            __syncwarp();
            if (row >= 0) {
                uint8_t *dst = smem + slot * Cfg::kStageBytes + kv * Cfg::kKvBytes +
                               (r * Cfg::kBoxes + box) * Hkv * 2048;
                tma_load_3d(dst, &kv_map, &full[slot], half * (128 / (kFp8 ? 1 : 2)), c1, row,
                            policy);
            }
            armed = x + 1;
            // the next stage's blocks are looked up after this one is issued
            if (x + 1 < hi) {
                while (prefix[s + 1] <= x + 1)
                    ++s;
                lookup(x + 1, s, row_next, c1_next, live_next);
            }
        }
        // Wind-down: the CTA must not exit while a copy it issued still writes
        // its shared memory.  A stage is refilled only after the consumers
        // freed it, which they do after its copies landed, so only the last
        // kStages armed stages can still be in flight: wait for their full
        // barriers (bounded, whatever the abort flag says).  On the normal
        // path they completed long ago and each test succeeds at once.
        for (int64_t x = armed - Cfg::kStages > lo ? armed - Cfg::kStages : lo; x < armed; ++x) {
            const int i = int(x - lo);
            mbar_wait(&full[i % Cfg::kStages], (i / Cfg::kStages) & 1);
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int u = warp;
    const int k = u % Hkv;
    const int r = u / Hkv;
    const int g = p.group;
    const int tq = lane & 3;   // thread-in-quad
    const int gq = lane >> 2;  // quad index
    const int H = p.num_heads;
    const uint32_t bstride = uint32_t(Hkv) * 2048;  // from one box of a unit to the next

    // ldmatrix lane addressing (rows = keys of the unit tile)
    const uint32_t k_row = (lane & 7) + ((lane >> 3) & 1) * 8;  // K: non-transposed A
    const uint32_t k_chunk = lane >> 4;
    const uint32_t v_row = (lane & 7) + (lane >> 4) * 8;  // V: transposed A
    const uint32_t v_chunk = (lane >> 3) & 1;

    // Q^T as B fragments: bf16 pairs, or (fp8 pool) prescaled f16 pairs
    uint32_t qf[D / 16][2];
    float o[D / 16][4];
    float m0, m1, l0, l1;
    // log2-domain multipliers of the raw scores of heads n0 = 2tq and n1 = 2tq+1
    float mul0 = p.scale_log2, mul1 = p.scale_log2;
    int s = s_first;
    int t = 0, L = 0;
    bool ok = true;
    // the next piece's token and length are loaded one piece ahead
    int t_nx = p.qsl[p.seq0 + s], L_nx = p.seq_lens[p.seq0 + s];
    auto begin_piece = [&]() {
        t = t_nx;
        L = L_nx;
        if (s + 1 < nseq) {
            t_nx = p.qsl[p.seq0 + s + 1];
            L_nx = p.seq_lens[p.seq0 + s + 1];
        }
        if (t < 0 || t >= p.num_tokens) {
            flag_error(kErrBadMetadata);
            t = 0;
        }
        if (p.kv_begin > 0 && L <= p.kv_begin)
            flag_error(kErrBadMetadata);  // a cascade decode must come after the prefix
        // Q^T as B fragments: column n = query head k*g + gq, rows = dims
        const bool live = gq < g;
        const uint32_t *qrow =
            p.query + ((static_cast<int64_t>(t) * H + k * g + (live ? gq : 0)) * D) / 2;
        if constexpr (kFp8) {
            // f16 fragments (the K and V codes are converted to f16, exactly),
            // each head prescaled by the power of two 2^(14-E) that puts its
            // largest |q| (in [2^E, 2^(E+1))) into [2^14, 2^15): bf16 has a
            // wider range than f16, and normal bf16 values are exact in f16.
            // Step kk = 4*hh + m takes rows (2tq, 2tq+1 | 2tq+8, 2tq+9) from
            // dims 64*hh + 16*tq + 4*m + (0, 1 | 2, 3): the dims one 16-byte
            // read of a K row gives this lane (below).
            const uint4 *qv = reinterpret_cast<const uint4 *>(qrow);
            uint4 raw[D / 64][2];
            float amax = 0.f;
#pragma unroll
            for (int hh = 0; hh < D / 64; ++hh)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    raw[hh][j] = live ? __ldg(qv + (64 * hh + 16 * tq) / 8 + j) : make_uint4(0, 0, 0, 0);
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const uint32_t x = u4_word(raw[hh][j], w);
                        amax = fmax3(amax, fabsf(__uint_as_float(x << 16)),
                                     fabsf(__uint_as_float(x & 0xffff0000u)));
                    }
                }
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
            const int e =
                amax > 0.f ? max(int((__float_as_uint(amax) >> 23) & 0xffu) - 127, -112) : 0;
            const float pre = __uint_as_float(uint32_t(127 + 14 - e) << 23);
            const float mul = p.scale_log2 * p.k_scale * __uint_as_float(uint32_t(127 - 14 + e) << 23);
#pragma unroll
            for (int hh = 0; hh < D / 64; ++hh)
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const uint32_t w0 = u4_word(raw[hh][m >> 1], 2 * (m & 1));
                    const uint32_t w1 = u4_word(raw[hh][m >> 1], 2 * (m & 1) + 1);
                    qf[4 * hh + m][0] = pack_f16x2(__uint_as_float(w0 << 16) * pre,
                                                   __uint_as_float(w0 & 0xffff0000u) * pre);
                    qf[4 * hh + m][1] = pack_f16x2(__uint_as_float(w1 << 16) * pre,
                                                   __uint_as_float(w1 & 0xffff0000u) * pre);
                }
            // head n is prescaled in the lanes with gq = n (lane 4n)
            mul0 = __shfl_sync(0xffffffffu, mul, 8 * tq);
            mul1 = __shfl_sync(0xffffffffu, mul, 8 * tq + 4);
        } else {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                qf[kk][0] = live ? __ldg(qrow + (16 * kk + 2 * tq) / 2) : 0u;
                qf[kk][1] = live ? __ldg(qrow + (16 * kk + 8 + 2 * tq) / 2) : 0u;
            }
        }
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt)
            o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
        m0 = m1 = kNegInf;
        l0 = l1 = 0.f;
    };
    begin_piece();

    // Running max of the two heads with a lazy rescale: it moves only when a
    // unit's max (cand, log2 units) exceeds it by more than 8, so every p is
    // at most 2^8 and the rescale of O and l (warp-uniform) is rare after a
    // piece's first unit; the result is the same up to rounding.
    auto update_max = [&](float cand0, float cand1) {
        const bool up0 = cand0 > m0 + 8.f, up1 = cand1 > m1 + 8.f;
        if (__any_sync(0xffffffffu, up0 || up1)) {
            const float al0 = up0 ? fast_exp2(m0 - cand0) : 1.f;
            const float al1 = up1 ? fast_exp2(m1 - cand1) : 1.f;
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
                o[mt][0] *= al0;
                o[mt][1] *= al1;
                o[mt][2] *= al0;
                o[mt][3] *= al1;
            }
            l0 *= al0;
            l1 *= al1;
            m0 = up0 ? cand0 : m0;
            m1 = up1 ? cand1 : m1;
        }
    };

    for (int64_t x = lo; x < hi; ++x) {
        const int i = int(x - lo);
        const int slot = i % Cfg::kStages;
        if (ok && !dec_wait(&full[slot], (i / Cfg::kStages) & 1, abort_flag))
            ok = false;
        const int ks = p.kv_begin + int(x - prefix[s]) * stage_keys + Cfg::kUnitKeys * r;
        const int valid = min(Cfg::kUnitKeys, L - ks);
        if (ok && valid > 0) {
            // this unit's first 16-key tile of K; its box b lies b * bstride on
            const uint32_t kbase = smem_addr(smem + slot * Cfg::kStageBytes +
                                             r * Hkv * Cfg::kUnitBytes + k * 2048);
            const uint32_t vbase = kbase + Cfg::kKvBytes;
            if (p.fuse_write && L - 1 < ks + Cfg::kUnitKeys) {
                // this stage holds the decode's new key (key L-1): the pool may
                // not have it yet, so it is taken from the step's K/V rows into
                // the staged tile, and written to the pool at the token's slot
                // (the same registers both times: lanes [0, kChunks) cover head
                // k's row)
                const int64_t sl = p.slots[t];
                if (sl >= 0 && sl < int64_t(p.num_blocks) * p.block_size) {
                    constexpr int kChunks = Cfg::kRowBytes / 16;  // 16-byte chunks of a row
                    // lanes [0, kChunks) take the K row, the next kChunks the V row
                    // (an fp8 pool: 8 + 8 lanes; bf16 D=128: 16 + 16)
                    static_assert(2 * kChunks <= 32, "one chunk per lane");
                    if (lane < 2 * kChunks) {
                        const int kv = lane / kChunks, c = lane % kChunks;
                        uint4 nr;
                        if constexpr (kFp8)
                            nr = quantized_chunk<D>(p, t, k, c, kv);
                        else
                            nr = __ldg((kv ? p.new_value : p.new_key) +
                                       (int64_t(t) * Hkv + k) * kChunks + c);
                        // the row's 16-byte chunk c: box = its half (bf16) or its
                        // 16-key half (fp8), then row and chunk in that tile
                        const int kr = L - 1 - ks;
                        const uint32_t o = (kFp8 ? kr >> 4 : c >> 3) * bstride +
                                           swz128(kr & 15, c & 7);
                        uint8_t *tile = smem + slot * Cfg::kStageBytes + kv * Cfg::kKvBytes +
                                        r * Hkv * Cfg::kUnitBytes + k * 2048;
                        *reinterpret_cast<uint4 *>(tile + o) = nr;
                        // the stage is refilled by TMA later: order this generic
                        // write before the async proxy's
                        fence_proxy_async_smem();
                        p.pool[pool_chunk<kHnd>(p, sl, kv, k, c, kChunks)] = nr;
                    }
                    __syncwarp();
                } else if (sl >= 0 && lane == 0) {
                    flag_error(kErrSlotOutOfPool);
                }
            }
            if constexpr (kFp8) {
                // ---- S^T = K Q^T over the unit's 32 keys, two 16-key row tiles.
                // Each K code is converted to f16 once (exact) and meets the f16
                // Q in mma m16n8k16.  Row gq (gq+8) of tile t2 is key 16*t2 + ka
                // (+2), ka = 8*(gq>>2) + 4*(gq&1) + ((gq>>1)&1): the two rows of
                // a quarter-warp differ in swizzle bit 2 (conflict-free 16-byte
                // reads) and the V rows gathered below are conflict free too.
                const int ka = 8 * (gq >> 2) + 4 * (gq & 1) + ((gq >> 1) & 1);
                float sc[2][4];
#pragma unroll
                for (int t2 = 0; t2 < 2; ++t2) {
                    float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int hh = 0; hh < D / 64; ++hh) {
                        const uint4 kr0 = lds128(kbase + t2 * bstride + swz128(ka, 4 * hh + tq));
                        const uint4 kr1 =
                            lds128(kbase + t2 * bstride + swz128(ka + 2, 4 * hh + tq));
#pragma unroll
                        for (int m = 0; m < 4; ++m) {
                            uint32_t a0, a1, a2, a3;
                            e4m3x4_to_f16x2x2(u4_word(kr0, m), a0, a2);
                            e4m3x4_to_f16x2x2(u4_word(kr1, m), a1, a3);
                            mma_f16_16816(c, a0, a1, a2, a3, qf[4 * hh + m][0], qf[4 * hh + m][1]);
                        }
                    }
                    const bool va = 16 * t2 + ka < valid, vb = 16 * t2 + ka + 2 < valid;
                    sc[t2][0] = va ? c[0] * mul0 : kNegInf;
                    sc[t2][1] = va ? c[1] * mul1 : kNegInf;
                    sc[t2][2] = vb ? c[2] * mul0 : kNegInf;
                    sc[t2][3] = vb ? c[3] * mul1 : kNegInf;
                }
                update_max(warp_max_heads(fmax3(fmaxf(sc[0][0], sc[0][2]), sc[1][0], sc[1][2])),
                           warp_max_heads(fmax3(fmaxf(sc[0][1], sc[0][3]), sc[1][1], sc[1][3])));
                float pv[2][4];
#pragma unroll
                for (int t2 = 0; t2 < 2; ++t2)
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        pv[t2][i] = fast_exp2(sc[t2][i] - ((i & 1) ? m1 : m0));
                l0 += (pv[0][0] + pv[0][2]) + (pv[1][0] + pv[1][2]);
                l1 += (pv[0][1] + pv[0][3]) + (pv[1][1] + pv[1][3]);
                // ---- P^T as f16 B fragments: movmatrix turns S^T rows (keys)
                // into columns, so the lane holds keys (2tq, 2tq+1) and (2tq+8,
                // 2tq+9) of tile t2 for head gq: k = (2tq, 2tq+1 | 2tq+8, 2tq+9)
                // of a 16-key mma, in the order the V rows are gathered below.
                uint32_t b0[2], b1[2];
#pragma unroll
                for (int t2 = 0; t2 < 2; ++t2) {
                    b0[t2] = movmatrix_trans(pack_f16x2(pv[t2][0], pv[t2][1]));
                    b1[t2] = movmatrix_trans(pack_f16x2(pv[t2][2], pv[t2][3]));
                }
                // ---- O^T += V^T P^T, 16 dims per step: ldmatrix row j is key
                // vkey(j) of the tile (rows 4tq..4tq+3 of a register = S^T rows
                // 2tq, 2tq+1, 2tq+8, 2tq+9); lanes 16-31 give the rows of keys
                // 16-31.  Each register's four codes become the (2tq, 2tq+1)
                // and (2tq+8, 2tq+9) f16 pairs of one dim.
                const int jl = lane & 15, tj = jl >> 2, ij = jl & 3;
                const int vrow = 16 * (lane >> 4) + 8 * (tj >> 1) + 4 * (ij & 1) +
                                 2 * (ij >> 1) + (tj & 1);
                auto pv_pass = [&](auto masked) {
                    // keys past the end may hold anything (e4m3 NaN codes too):
                    // zero their bytes; this lane's bytes are keys vkey(4tq + i)
                    uint32_t mk0 = 0xffffffffu, mk1 = 0xffffffffu;
                    if constexpr (decltype(masked)::value) {
                        mk0 = mk1 = 0u;
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int kk = 8 * (tq >> 1) + 4 * (i & 1) + 2 * (i >> 1) + (tq & 1);
                            mk0 |= kk < valid ? 0xffu << (8 * i) : 0u;
                            mk1 |= kk + 16 < valid ? 0xffu << (8 * i) : 0u;
                        }
                    }
#pragma unroll
                    for (int mt = 0; mt < D / 16; ++mt) {
                        uint32_t v[4];  // [tile 0: dim gq, dim gq+8, tile 1: dim gq, dim gq+8]
                        ldsm_x2_trans_b8(vbase + (vrow >> 4) * bstride + swz128(vrow & 15, mt),
                                         v[0], v[1], v[2], v[3]);
                        if constexpr (decltype(masked)::value) {
                            v[0] &= mk0;
                            v[1] &= mk0;
                            v[2] &= mk1;
                            v[3] &= mk1;
                        }
#pragma unroll
                        for (int t2 = 0; t2 < 2; ++t2) {
                            uint32_t a0, a1, a2, a3;
                            e4m3x4_to_f16x2x2(v[2 * t2], a0, a2);
                            e4m3x4_to_f16x2x2(v[2 * t2 + 1], a1, a3);
                            mma_f16_16816(o[mt], a0, a1, a2, a3, b0[t2], b1[t2]);
                        }
                    }
                };
                if (valid < 32)
                    pv_pass(std::true_type{});
                else
                    pv_pass(std::false_type{});
            } else {
                // S^T = K Q^T
                float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t ch = 2 * kk + k_chunk;
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(kbase + (ch >> 3) * bstride + swz128(k_row, ch & 7), a0, a1, a2, a3);
                    mma_bf16_16816(c, a0, a1, a2, a3, qf[kk][0], qf[kk][1]);
                }
                const bool va = gq < valid, vb = gq + 8 < valid;
                const float s0 = va ? c[0] * mul0 : kNegInf;
                const float s1 = va ? c[1] * mul1 : kNegInf;
                const float s2 = vb ? c[2] * mul0 : kNegInf;
                const float s3 = vb ? c[3] * mul1 : kNegInf;
                update_max(warp_max_heads(fmaxf(s0, s2)), warp_max_heads(fmaxf(s1, s3)));
                const float p0 = fast_exp2(s0 - m0), p1 = fast_exp2(s1 - m1);
                const float p2 = fast_exp2(s2 - m0), p3 = fast_exp2(s3 - m1);
                l0 += p0 + p2;
                l1 += p1 + p3;
                // P^T as B fragments: rows 0-7 and 8-15 of S^T
                const uint32_t b0 = movmatrix_trans(pack_bf16x2(p0, p1));
                const uint32_t b1 = movmatrix_trans(pack_bf16x2(p2, p3));
                auto pv_pass = [&](auto masked) {
                    // rows of V past the end of the sequence may hold anything:
                    // zero them (only a sequence's last unit has such rows)
                    uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
                    if constexpr (decltype(masked)::value) {
                        mlo = (2 * tq < valid ? 0x0000ffffu : 0u) |
                              (2 * tq + 1 < valid ? 0xffff0000u : 0u);
                        mhi = (2 * tq + 8 < valid ? 0x0000ffffu : 0u) |
                              (2 * tq + 9 < valid ? 0xffff0000u : 0u);
                    }
#pragma unroll
                    for (int mt = 0; mt < D / 16; ++mt) {
                        const uint32_t ch = 2 * mt + v_chunk;
                        uint32_t a0, a1, a2, a3;
                        ldsm_x4_trans(vbase + (ch >> 3) * bstride + swz128(v_row, ch & 7), a0, a1,
                                      a2, a3);
                        if constexpr (decltype(masked)::value) {
                            a0 &= mlo;
                            a1 &= mlo;
                            a2 &= mhi;
                            a3 &= mhi;
                        }
                        mma_bf16_16816(o[mt], a0, a1, a2, a3, b0, b1);
                    }
                };
                if (valid < 16)
                    pv_pass(std::true_type{});
                else
                    pv_pass(std::false_type{});
            }
        }
        __syncwarp();
        if (ok && lane == 0)
            mbar_arrive(&empty[slot]);

        if (x + 1 < hi && x + 1 < prefix[s + 1])
            continue;  // the piece goes on
        // ------------------------------------------------------------ end of a piece
        const float lr0 = warp_sum_heads(l0);
        const float lr1 = warp_sum_heads(l1);
        const int bf = aligned ? s : cta_of_stage(prefix[s], total, grid);
        const int bl = aligned ? s : cta_of_stage(prefix[s + 1] - 1, total, grid);
        const int np = bl - bf + 1;
        // a sequence inside one CTA (and one warp per kv head) is finished from
        // registers
        const bool direct = np == 1 && R == 1;
        const int n0 = 2 * tq, n1 = 2 * tq + 1;  // the two heads of this thread
        // row scales of the output (an fp8 pool's V dequantisation folded in)
        const float vsc = kFp8 ? p.v_scale : 1.f;
        const float i0 = lr0 > 0.f ? vsc / lr0 : 0.f;
        const float i1 = lr1 > 0.f ? vsc / lr1 : 0.f;
        if (direct) {
            if (ok) {
                // log2-sum-exp of the two heads (-inf: no key)
                const float ls0 = lr0 > 0.f ? m0 + log2f(lr0) : kNegInf;
                const float ls1 = lr1 > 0.f ? m1 + log2f(lr1) : kNegInf;
                const int64_t r0 = int64_t(t) * H + k * g + n0;
                const int64_t r1 = r0 + 1;
#pragma unroll
                for (int mt = 0; mt < D / 16; ++mt) {  // dims 16*mt + gq and +8
                    const int d = 16 * mt + gq;
                    if (p.o_suf) {  // cascade suffix: fp32 partial rows
                        if (n0 < g) {
                            p.o_suf[r0 * D + d] = o[mt][0] * i0;
                            p.o_suf[r0 * D + d + 8] = o[mt][2] * i0;
                        }
                        if (n1 < g) {
                            p.o_suf[r1 * D + d] = o[mt][1] * i1;
                            p.o_suf[r1 * D + d + 8] = o[mt][3] * i1;
                        }
                        continue;
                    }
                    if (n0 < g) {
                        p.out[r0 * D + d] = __float2bfloat16_rn(o[mt][0] * i0);
                        p.out[r0 * D + d + 8] = __float2bfloat16_rn(o[mt][2] * i0);
                    }
                    if (n1 < g) {
                        p.out[r1 * D + d] = __float2bfloat16_rn(o[mt][1] * i1);
                        p.out[r1 * D + d + 8] = __float2bfloat16_rn(o[mt][3] * i1);
                    }
                }
                if (gq == 0) {
                    float *dst = p.o_suf ? p.lse_suf : p.lse;
                    const float u = p.o_suf ? 1.f : kLn2;  // log2 partial, or ln
                    if (dst && n0 < g)
                        dst[r0] = ls0 * u;
                    if (dst && n1 < g)
                        dst[r1] = ls1 * u;
                }
            }
        } else {
            const int slot_id = b + s;  // unique per (CTA, sequence) piece
            const int64_t prow = (int64_t(slot_id) * R + r) * H + k * g;
            if (ok) {
#pragma unroll
                for (int mt = 0; mt < D / 16; ++mt) {
                    const int d = 16 * mt + gq;
                    if (n0 < g) {
                        float *dst = p.o_part + (prow + n0) * D;
                        dst[d] = o[mt][0] * i0;
                        dst[d + 8] = o[mt][2] * i0;
                    }
                    if (n1 < g) {
                        float *dst = p.o_part + (prow + n1) * D;
                        dst[d] = o[mt][1] * i1;
                        dst[d + 8] = o[mt][3] * i1;
                    }
                }
                if (gq == 0) {
                    if (n0 < g)
                        p.lse_part[prow + n0] = lr0 > 0.f ? m0 + log2f(lr0) : kNegInf;
                    if (n1 < g)
                        p.lse_part[prow + n1] = lr1 > 0.f ? m1 + log2f(lr1) : kNegInf;
                }
            }
            // The piece's rows are written (the barrier orders every consumer's
            // writes before thread 0's); thread 0 releases them to the GPU
            // with one fence before it counts the piece, and the last piece's
            // thread 0 acquires the others' rows with one fence after it: the
            // barrier then orders those before every consumer's reads.  A
            // sequence inside this CTA (its parts are the warps' rows) needs
            // only the barrier: no count, no fence.
            // (a split sequence's pieces are left for the merge launch after
            // this grid when it defers them)
            if (np == 1 || !p.defer_merge) {
                consumer_sync();  // all eight warps reach it, failed or not
                if (np > 1) {
                    if (threadIdx.x == 0) {
                        __threadfence();
                        *last_flag = (atomicAdd(&p.counters[s], 1) == np - 1) ? 1 : 0;
                        __threadfence();
                    }
                    consumer_sync();
                }
                if ((np == 1 || *last_flag) && !*abort_flag) {
                    // every piece of this sequence is written: merge them, one warp
                    // per head (warp-shuffle max/sum of the parts' log2-sum-exp,
                    // then the weighted sum of their rows, lanes along head_size).
                    // A round of a merge holds kQB x kHB rows in registers: with one
                    // head per warp (H <= 8) the rounds take more parts instead of
                    // more heads, so that the np x R parts of a short batch cost
                    // one or two L2 round trips.  (The fp8 stage loop leaves fewer
                    // registers: two rows per round with one head per warp, four
                    // with more.)
                    if (H <= kConsumerWarps)
                        merge_pieces<D, kFp8 ? 2 : 8, 1>(p, t, s, bf, np * R, R, warp, lane);
                    else
                        merge_pieces<D, 2, kFp8 ? 2 : 4>(p, t, s, bf, np * R, R,
                                                                     warp, lane);
                }
            }
        }
        if (x + 1 < hi) {
            ++s;
            begin_piece();
        }
    }
}

template <int D, bool kHnd, bool kFp8>
__global__ void __launch_bounds__(kDecodeThreads, 1)
    paged_decode_kernel(const __grid_constant__ CUtensorMap kv_map, const DecodeParams p)
{
    // The launch after this grid, its programmatic dependent (the cascade's
    // combine, or a prefill pass beside this decode), may be scheduled on SMs
    // as they free up; it waits for this grid to complete before it reads this
    // grid's results or exits.
    if (p.trigger_dependents)
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    decode_cta<D, kHnd, kFp8>(kv_map, p);
    // A cascade's suffix pass runs beside the shared-prefix pass (a dependent
    // launch that starts while the prefix pass holds its SMs); its CTAs wait
    // here for that grid to complete, so that the kernels after this one see
    // both passes' partials.  The prefix pass never waits on this grid.
    if (p.after_prefix)
        asm volatile("griddepcontrol.wait;" ::: "memory");
}

// --------------------------------------------------------------------- combine
// Cascade: every token's suffix partial (over keys [P, L), from the decode
// kernel or the prefill kernel) merged with its pre_splits shared-prefix
// partials (keys [0, P), one per key chunk) -- the log-sum-exp merge of the
// "El especialista del plato estrella" blog ("Que aporta FlashInfer: JIT y
// cascade attention").  One warp per (token, head) row, lanes along
// head_size; every log2-sum-exp of a row is loaded before any is used, then
// every part's row, so a row costs about two memory round trips.
struct CombineParams {
    int32_t num_tokens;
    int32_t num_heads;
    int32_t pre_splits;   // <= kMaxPrefixSplits
    const float *o_pre;   // [pre_splits][T, H, D]
    const float *lse_pre; // [pre_splits][T, H], log2 units
    const float *o_suf;   // [T, H, D]
    const float *lse_suf; // [T, H], log2 units
    __nv_bfloat16 *out;
    float *lse;
};

template <int D>
__global__ void __launch_bounds__(256) cascade_combine_kernel(const CombineParams p)
{
    constexpr int kPer = D / 32;
    constexpr int kParts = 1 + kMaxPrefixSplits;  // part 0: the suffix, 1 + c: prefix chunk c
    using Vec = typename std::conditional<kPer == 4, float4, float2>::type;
    // a dependent launch: the passes that write the partials may still run
    // (this grid's CTAs start as theirs finish); wait until they completed
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t row = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t rows = int64_t(p.num_tokens) * p.num_heads;
    if (row >= rows)
        return;
    const int nparts = 1 + p.pre_splits;
    float l[kParts];
#pragma unroll
    for (int q = 0; q < kParts; ++q)
        l[q] = q >= nparts ? kNegInf
                           : q == 0 ? __ldcg(p.lse_suf + row)
                                    : __ldcg(p.lse_pre + (q - 1) * rows + row);
    float mx = kNegInf;
#pragma unroll
    for (int q = 0; q < kParts; ++q)
        mx = fmaxf(mx, l[q]);
    Vec v[kParts];
#pragma unroll
    for (int q = 0; q < kParts; ++q) {
        // an empty part (lse = -inf) adds nothing: its row is not read
        const float *src = q == 0 ? p.o_suf + row * D : p.o_pre + ((q - 1) * rows + row) * D;
        v[q] = l[q] != kNegInf ? __ldcg(reinterpret_cast<const Vec *>(src) + lane) : Vec{};
    }
    float acc[kPer];
#pragma unroll
    for (int e = 0; e < kPer; ++e)
        acc[e] = 0.f;
    float ws = 0.f;
    if (mx != kNegInf) {
#pragma unroll
        for (int q = 0; q < kParts; ++q) {
            const float w = l[q] == kNegInf ? 0.f : exp2f(l[q] - mx);
            ws += w;
            const float *x = reinterpret_cast<const float *>(&v[q]);
#pragma unroll
            for (int e = 0; e < kPer; ++e)
                acc[e] += w * x[e];
        }
    }
    const float inv = ws > 0.f ? 1.f / ws : 0.f;
    __nv_bfloat16 *dst = p.out + row * D + lane * kPer;
#pragma unroll
    for (int e = 0; e < kPer; e += 2)
        *reinterpret_cast<__nv_bfloat162 *>(dst + e) =
            __floats2bfloat162_rn(acc[e] * inv, acc[e + 1] * inv);
    if (lane == 0 && p.lse)
        p.lse[row] = ws > 0.f ? (mx + log2f(ws)) * kLn2 : kNegInf;
}

// --------------------------------------------------------------------- host
DecodePlan plan_decode(int32_t split_kv_tokens, int32_t num_decodes, int32_t num_kv_heads,
                       int num_sms)
{
    DecodePlan dp;
    dp.stage_keys = 16 * (kConsumerWarps / num_kv_heads);
    dp.grid = std::max(1, num_sms);
    dp.chunk = std::min(num_decodes, kMaxDecodeChunk);
    dp.target_keys = split_kv_tokens;
    dp.rows_per_slot = kConsumerWarps / num_kv_heads;
    return dp;
}

// The pieces of every decode that the launch before split over several CTAs
// (a batch of a few long decodes: each spreads over many SMs), merged by one
// warp per (decode, head) over the whole GPU instead of by the decode's last
// CTA, which would fold its many parts a few per L2 round trip while the rest
// of the GPU idles.  A programmatic dependent of that launch: its CTAs start
// as the decode's finish and wait for the whole grid before reading.
struct PieceMergeParams {
    const float *o_part;    // [slots, R, H, D] normalised partials
    const float *lse_part;  // [slots, R, H], log2 units
    const int32_t *table;   // [nseq]: first CTA | pieces << 16, or 0 (not split)
    const int32_t *qsl;
    int32_t seq0, nseq, num_heads, R;
    __nv_bfloat16 *out;
    float *lse;
};

template <int D>
__global__ void __launch_bounds__(256) decode_merge_kernel(const PieceMergeParams p)
{
    constexpr int kPer = D / 32;  // dims per lane
    constexpr int kQB = 8;        // parts per round: every load of a round in flight at once
    using Vec = typename std::conditional<kPer == 4, float4, float2>::type;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t unit = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int H = p.num_heads;
    if (unit >= int64_t(p.nseq) * H)
        return;
    const int s = static_cast<int>(unit / H), h = static_cast<int>(unit % H);
    const int32_t e = __ldcg(p.table + s);
    if (e == 0)
        return;  // finished by the decode launch
    const int bf = e & 0xFFFF, nparts = (e >> 16) * p.R;
    float M = kNegInf, W = 0.f, acc[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k)
        acc[k] = 0.f;
    for (int q0 = 0; q0 < nparts; q0 += kQB) {
        float lq[kQB];
        Vec v[kQB];
#pragma unroll
        for (int i = 0; i < kQB; ++i) {
            const int q = q0 + i;
            if (q < nparts) {
                // part q: slot bf + q / R + s, sub-row q % R
                const int64_t row = (int64_t(bf + q / p.R + s) * p.R + q % p.R) * H + h;
                lq[i] = __ldcg(p.lse_part + row);
                v[i] = __ldcg(reinterpret_cast<const Vec *>(p.o_part + row * D) + lane);
            } else {
                lq[i] = kNegInf;
                v[i] = Vec{};
            }
        }
        float mr = M;
#pragma unroll
        for (int i = 0; i < kQB; ++i)
            mr = fmaxf(mr, lq[i]);
        if (mr == kNegInf)
            continue;  // every part so far is empty
        const float a = exp2f(M - mr);
        W *= a;
#pragma unroll
        for (int k = 0; k < kPer; ++k)
            acc[k] *= a;
#pragma unroll
        for (int i = 0; i < kQB; ++i) {
            // an empty part adds nothing, whatever its row holds
            const float w = lq[i] == kNegInf ? 0.f : exp2f(lq[i] - mr);
            W += w;
            const float *x = reinterpret_cast<const float *>(&v[i]);
#pragma unroll
            for (int k = 0; k < kPer; ++k)
                acc[k] += w * x[k];
        }
        M = mr;
    }
    const int64_t row_out = int64_t(p.qsl[p.seq0 + s]) * H + h;
    const float inv = W > 0.f ? 1.f / W : 0.f;
    __nv_bfloat16 *dst = p.out + row_out * D + lane * kPer;
#pragma unroll
    for (int k = 0; k < kPer; k += 2)
        *reinterpret_cast<__nv_bfloat162 *>(dst + k) =
            __floats2bfloat162_rn(acc[k] * inv, acc[k + 1] * inv);
    if (lane == 0 && p.lse)
        p.lse[row_out] = W > 0.f ? (M + log2f(W)) * kLn2 : kNegInf;
}

template <int D, bool kHnd, bool kFp8>
static cudaError_t launch_decode_d(const Fwd &f, const DecodePlan &dp, const Workspace &ws,
                                   char *wsp, const CUtensorMap &kv_map, int32_t kv_begin,
                                   const DecodeOut &dout)
{
    using Cfg = DecodeCfg<D, kFp8>;
    // devices (bit d for device d < 64) on which this instantiation's launch
    // attribute is set; atomic, since several host threads may launch
    static std::atomic<uint64_t> configured{0};
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t dev_bit = (dev >= 0 && dev < 64) ? (uint64_t(1) << dev) : 0;
    if (dev_bit == 0 || (configured.load(std::memory_order_acquire) & dev_bit) == 0) {
        cudaError_t e = cudaFuncSetAttribute(paged_decode_kernel<D, kHnd, kFp8>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(Cfg::kSmemBytes));
        if (e != cudaSuccess)
            return e;
        configured.fetch_or(dev_bit, std::memory_order_release);
    }
    DecodeParams p;
    p.query = static_cast<const uint32_t *>(f.query);
    p.qsl = f.qsl;
    p.seq_lens = f.seq_lens;
    p.block_table = f.block_table;
    p.bt_stride = f.bt_stride;
    p.num_tokens = f.num_tokens;
    p.num_heads = f.num_heads;
    p.num_kv_heads = f.num_kv_heads;
    p.group = f.num_heads / f.num_kv_heads;
    p.block_size = f.block_size;
    p.num_blocks = static_cast<int32_t>(f.num_blocks);
    p.kv_begin = kv_begin;
    p.target_keys = dp.target_keys;
    p.scale_log2 = f.scale * 1.4426950408889634f;
    p.out = static_cast<__nv_bfloat16 *>(f.out);
    p.lse = f.lse;
    p.o_part = reinterpret_cast<float *>(wsp + ws.o_part);
    p.lse_part = reinterpret_cast<float *>(wsp + ws.lse_part);
    p.counters = reinterpret_cast<int32_t *>(wsp + ws.counters);
    p.o_suf = dout.o_suf;
    p.lse_suf = dout.lse_suf;
    p.fuse_write = f.fuse_write;
    p.new_key = static_cast<const uint4 *>(f.new_key);
    p.new_value = static_cast<const uint4 *>(f.new_value);
    p.slots = f.slots;
    p.pool = static_cast<uint4 *>(f.kv_cache_w);
    p.k_scale = f.k_scale;
    p.v_scale = f.v_scale;
    p.test_skip_copies = f.test_skip_copies;
    p.trigger_dependents = dout.dependent_follows || dout.defer_merge ? 1 : 0;
    p.defer_merge = dout.defer_merge ? 1 : 0;
    p.expect_aligned = dout.expect_aligned ? 1 : 0;
    // one launch per chunk of at most kMaxDecodeChunk decodes (stream ordered,
    // so chunks reuse the same partial slots and counters)
    for (int32_t seq0 = 0; seq0 < f.num_decodes; seq0 += dp.chunk) {
        p.seq0 = seq0;
        p.nseq = std::min(dp.chunk, f.num_decodes - seq0);
        cudaError_t e = cudaSuccess;
        if (seq0 > 0 || !(dout.counters_zeroed || dout.expect_aligned))
            e = cudaMemsetAsync(p.counters, 0, size_t(p.nseq) * 4, f.stream);
        if (e != cudaSuccess)
            return e;
        // the first launch may be the dependent of the shared-prefix pass
        // enqueued just before it (it then starts on the SMs that pass leaves)
        p.after_prefix = seq0 == 0 && dout.after_prefix ? 1 : 0;
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        cfg.gridDim = dim3(dp.grid);
        cfg.blockDim = dim3(kDecodeThreads);
        cfg.dynamicSmemBytes = Cfg::kSmemBytes;
        cfg.stream = f.stream;
        if (p.after_prefix) {
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[0].val.programmaticStreamSerializationAllowed = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
        }
        count_launch();
        e = cudaLaunchKernelEx(&cfg, paged_decode_kernel<D, kHnd, kFp8>, kv_map, p);
        if (e != cudaSuccess)
            return e;
        if (p.defer_merge) {
            // the split decodes' pieces, merged over the whole GPU as the
            // decode's programmatic dependent (nothing may stand between them)
            PieceMergeParams m;
            m.o_part = p.o_part;
            m.lse_part = p.lse_part;
            m.table = p.counters;
            m.qsl = p.qsl;
            m.seq0 = p.seq0;
            m.nseq = p.nseq;
            m.num_heads = p.num_heads;
            m.R = kConsumerWarps / p.num_kv_heads;
            m.out = p.out;
            m.lse = p.lse;
            const int64_t warps = int64_t(p.nseq) * p.num_heads;
            cudaLaunchConfig_t mc = {};
            cudaLaunchAttribute ma[1];
            mc.gridDim = dim3(static_cast<unsigned>((warps * 32 + 255) / 256));
            mc.blockDim = dim3(256);
            mc.stream = f.stream;
            ma[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            ma[0].val.programmaticStreamSerializationAllowed = 1;
            mc.attrs = ma;
            mc.numAttrs = 1;
            count_launch();
            e = cudaLaunchKernelEx(&mc, decode_merge_kernel<D>, m);
            if (e != cudaSuccess)
                return e;
        }
    }
    return cudaSuccess;
}

cudaError_t launch_decode(const Fwd &f, const DecodePlan &dp, const Workspace &ws, char *wsp,
                          const CUtensorMap &kv_map, int32_t kv_begin, const DecodeOut &dout)
{
    if (f.num_decodes == 0)
        return cudaSuccess;
    if (f.kv_fp8) {  // head_size 128 only (checked by the caller)
        if (f.head_size != 128)
            return cudaErrorInvalidValue;
        return f.kv_hnd
                   ? launch_decode_d<128, true, true>(f, dp, ws, wsp, kv_map, kv_begin, dout)
                   : launch_decode_d<128, false, true>(f, dp, ws, wsp, kv_map, kv_begin, dout);
    }
    if (f.head_size == 128)
        return f.kv_hnd
                   ? launch_decode_d<128, true, false>(f, dp, ws, wsp, kv_map, kv_begin, dout)
                   : launch_decode_d<128, false, false>(f, dp, ws, wsp, kv_map, kv_begin, dout);
    return f.kv_hnd ? launch_decode_d<64, true, false>(f, dp, ws, wsp, kv_map, kv_begin, dout)
                    : launch_decode_d<64, false, false>(f, dp, ws, wsp, kv_map, kv_begin, dout);
}

cudaError_t launch_cascade_combine(const Fwd &f, const Workspace &ws, char *wsp)
{
    const int64_t warps = int64_t(f.num_tokens) * f.num_heads;
    if (warps == 0)
        return cudaSuccess;
    if (ws.pre_splits < 1 || ws.pre_splits > kMaxPrefixSplits)
        return cudaErrorInvalidValue;
    CombineParams p;
    p.num_tokens = f.num_tokens;
    p.num_heads = f.num_heads;
    p.pre_splits = ws.pre_splits;
    p.o_pre = reinterpret_cast<const float *>(wsp + ws.o_pre);
    p.lse_pre = reinterpret_cast<const float *>(wsp + ws.lse_pre);
    p.o_suf = reinterpret_cast<const float *>(wsp + ws.o_suf);
    p.lse_suf = reinterpret_cast<const float *>(wsp + ws.lse_suf);
    p.out = static_cast<__nv_bfloat16 *>(f.out);
    p.lse = f.lse;
    // launched as the dependent of the kernel before it (the suffix decode or
    // the prefill pass), so that its CTAs take SMs as that grid drains
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(static_cast<unsigned>((warps * 32 + 255) / 256));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = f.stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    count_launch();
    if (f.head_size == 128)
        return cudaLaunchKernelEx(&cfg, cascade_combine_kernel<128>, p);
    return cudaLaunchKernelEx(&cfg, cascade_combine_kernel<64>, p);
}

uint32_t decode_take_error() { return take_device_error(); }

}  // namespace pka
