// decode.cu -- split-KV paged decode and its log-sum-exp combine.
//
// What it computes (the "El especialista del plato estrella" blog,
// "Por que prefill y decode son problemas opuestos"): one query token per
// sequence against all of that sequence's keys.  The work is memory bound,
// so the kernel is built to keep HBM busy: every byte of K and V is read once,
// for all query heads of its kv head at the same time (GQA packing), and is
// staged into shared memory by TMA ahead of use.
//
// Grid: one CTA per (decode sequence s, split j).  Split j covers keys
// [kv_begin + j*C, min(kv_begin + (j+1)*C, L_s)), C = split_tokens.  CTAs of
// splits past the end of their sequence exit at once.
//
// CTA: 8 consumer warps + 1 producer warp.  A pipeline stage holds 8 "units";
// unit u is 16 consecutive keys of kv head k = u % Hkv, slice r = u / Hkv of the
// stage's 16*(8/Hkv) keys (so every warp works in every stage).  The producer
// issues, per unit, one TMA box {64 dims, 1 head, 16 rows} per 64-dim half for
// K and for V out of the pool viewed as a 3-D tensor
// (head_size, num_kv_heads, num_blocks*2*block_size) -- the "FlashAttention y
// FlashInfer" page's cache shape with (block, kv, offset) flattened -- with
// 128-byte swizzling so that the ldmatrix reads below are conflict free.
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
// At the end the warps of the same kv head (when Hkv < 8) are merged through
// shared memory and the CTA writes either the final bf16 row and lse (single
// split) or a normalised fp32 partial and its log2-sum-exp for the combine.
#include <math.h>

#include <algorithm>

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
    int32_t split_tokens;
    int32_t max_splits;
    int32_t kv_begin;
    int32_t partial_only;
    float scale_log2;  // softmax scale * log2(e)
    __nv_bfloat16 *out;
    float *lse;
    float *o_part;    // [num_decodes, max_splits, H, D]
    float *lse_part;  // [num_decodes, max_splits, H], log2 units
};

constexpr int kConsumerWarps = 8;
constexpr int kDecodeThreads = (kConsumerWarps + 1) * 32;
constexpr float kNegInf = -INFINITY;
constexpr float kLn2 = 0.69314718055994530942f;

template <int D>
struct DecodeCfg {
    static constexpr int kHalves = D / 64;
    static constexpr int kUnitBytes = 16 * D * 2;                  // 16 rows x D bf16
    static constexpr int kKvBytes = kConsumerWarps * kUnitBytes;   // all units of K (or V)
    static constexpr int kStageBytes = 2 * kKvBytes;
    static constexpr int kStages = (D == 128) ? 3 : 6;
    static constexpr int kScratchFloats = 16 + 8 * D;              // per warp: m, l, O^T
    static constexpr size_t kSmemBytes =
        size_t(kStages) * kStageBytes + 2 * kStages * sizeof(uint64_t) + 1024;
    static_assert(kConsumerWarps * kScratchFloats * 4 <= kStages * kStageBytes, "scratch");
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

template <int D>
__global__ void __launch_bounds__(kDecodeThreads, 1)
    paged_decode_kernel(const __grid_constant__ CUtensorMap kv_map, const DecodeParams p)
{
    using Cfg = DecodeCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Cfg::kStages * Cfg::kStageBytes);
    uint64_t *empty = full + Cfg::kStages;

    const int s = blockIdx.y;
    const int split = blockIdx.x;
    const int L = p.seq_lens[s];
    if (p.kv_begin > 0 && L <= p.kv_begin) {
        // cascade suffix pass: the decode's query must come after the shared prefix
        if (threadIdx.x == 0 && split == 0)
            flag_error(kErrBadMetadata);
        return;
    }
    const int key_begin = p.kv_begin + split * p.split_tokens;
    if (key_begin >= L)
        return;  // whole CTA: this split lies past the end of the sequence
    const int key_end = min(L, key_begin + p.split_tokens);
    const int nsplit = (L - p.kv_begin + p.split_tokens - 1) / p.split_tokens;
    const int t = p.qsl[s];
    if (nsplit > p.max_splits || t < 0 || t >= p.num_tokens) {
        // seq_lens above the stated max_seq_len, or a token index outside the
        // batch: nothing is read or written for this sequence
        if (threadIdx.x == 0 && split == 0)
            flag_error(kErrBadMetadata);
        return;
    }
    const int Hkv = p.num_kv_heads;
    const int R = kConsumerWarps / Hkv;
    const int stage_keys = 16 * R;
    const int nstage = (key_end - key_begin + stage_keys - 1) / stage_keys;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < Cfg::kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kConsumerWarps);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        if (lane == 0)
            tma_prefetch_desc(&kv_map);
        const uint64_t policy = l2_policy_evict_first();
        const int32_t *bt = p.block_table + static_cast<int64_t>(s) * p.bt_stride;
        constexpr int kOps = kConsumerWarps * 2 * Cfg::kHalves;  // (unit, K|V, half)
        for (int i = 0; i < nstage; ++i) {
            const int slot = i % Cfg::kStages;
            const int round = i / Cfg::kStages;
            if (round > 0 && !mbar_wait(&empty[slot], (round - 1) & 1))
                break;
            const int k0 = key_begin + i * stage_keys;
            const int slices = min(R, (key_end - k0 + 15) / 16);
            if (lane == 0)
                mbar_arrive_expect_tx(&full[slot],
                                      static_cast<uint32_t>(slices * Hkv * 2 * Cfg::kUnitBytes));
            __syncwarp();
            uint8_t *stage = smem + slot * Cfg::kStageBytes;
            for (int op = lane; op < kOps; op += 32) {
                const int u = op % kConsumerWarps;
                const int kv = (op / kConsumerWarps) & 1;
                const int half = op / (2 * kConsumerWarps);
                const int r = u / Hkv;
                const int k = u % Hkv;
                const int ks = k0 + 16 * r;
                if (r >= slices)
                    continue;
                const int col = ks / p.block_size;
                int blk = col < p.bt_stride ? bt[col] : -1;
                if (blk < 0 || blk >= p.num_blocks) {
                    flag_error(kErrBlockOutOfPool);
                    blk = 0;  // keep the transaction count whole; result is flagged
                }
                const int row = (blk * 2 + kv) * p.block_size + (ks % p.block_size);
                uint8_t *dst = stage + kv * Cfg::kKvBytes + u * Cfg::kUnitBytes + half * 2048;
                tma_load_3d(dst, &kv_map, &full[slot], half * 64, k, row, policy);
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int u = warp;
    const int k = u % Hkv;
    const int r = u / Hkv;
    const int g = p.group;
    const int tq = lane & 3;  // thread-in-quad
    const int gq = lane >> 2;  // quad index

    // Q^T as B fragments: column n = query head k*g + gq, rows = dims.
    uint32_t qf[D / 16][2];
    {
        const bool live = gq < g;
        const uint32_t *qrow =
            p.query + ((static_cast<int64_t>(t) * p.num_heads + k * g + (live ? gq : 0)) * D) / 2;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            qf[kk][0] = live ? __ldg(qrow + (16 * kk + 2 * tq) / 2) : 0u;
            qf[kk][1] = live ? __ldg(qrow + (16 * kk + 8 + 2 * tq) / 2) : 0u;
        }
    }

    float o[D / 16][4];
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt)
        o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    float m0 = kNegInf, m1 = kNegInf, l0 = 0.f, l1 = 0.f;
    bool ok = true;

    // ldmatrix lane addressing (rows = keys of the unit tile)
    const uint32_t k_row = (lane & 7) + ((lane >> 3) & 1) * 8;  // K: non-transposed A
    const uint32_t k_chunk = lane >> 4;
    const uint32_t v_row = (lane & 7) + (lane >> 4) * 8;  // V: transposed A
    const uint32_t v_chunk = (lane >> 3) & 1;

    for (int i = 0; i < nstage; ++i) {
        const int slot = i % Cfg::kStages;
        if (!mbar_wait(&full[slot], (i / Cfg::kStages) & 1)) {
            ok = false;
            break;
        }
        const int ks = key_begin + i * stage_keys + 16 * r;
        const int valid = min(16, key_end - ks);
        if (valid > 0) {
            const uint32_t kbase =
                smem_addr(smem + slot * Cfg::kStageBytes + u * Cfg::kUnitBytes);
            const uint32_t vbase = kbase + Cfg::kKvBytes;
            // S^T = K Q^T
            float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t ch = 2 * kk + k_chunk;
                uint32_t a0, a1, a2, a3;
                ldsm_x4(kbase + (ch >> 3) * 2048 + swz128(k_row, ch & 7), a0, a1, a2, a3);
                mma_bf16_16816(c, a0, a1, a2, a3, qf[kk][0], qf[kk][1]);
            }
            const bool va = gq < valid, vb = gq + 8 < valid;
            const float s0 = va ? c[0] * p.scale_log2 : kNegInf;
            const float s1 = va ? c[1] * p.scale_log2 : kNegInf;
            const float s2 = vb ? c[2] * p.scale_log2 : kNegInf;
            const float s3 = vb ? c[3] * p.scale_log2 : kNegInf;
            const float mn0 = fmaxf(m0, warp_max_heads(fmaxf(s0, s2)));
            const float mn1 = fmaxf(m1, warp_max_heads(fmaxf(s1, s3)));
            const float al0 = fast_exp2(m0 - mn0), al1 = fast_exp2(m1 - mn1);
            const float p0 = fast_exp2(s0 - mn0), p1 = fast_exp2(s1 - mn1);
            const float p2 = fast_exp2(s2 - mn0), p3 = fast_exp2(s3 - mn1);
            l0 = l0 * al0 + (p0 + p2);
            l1 = l1 * al1 + (p1 + p3);
            m0 = mn0;
            m1 = mn1;
            const uint32_t b0 = movmatrix_trans(pack_bf16x2(p0, p1));  // keys 0-7
            const uint32_t b1 = movmatrix_trans(pack_bf16x2(p2, p3));  // keys 8-15
            // rows of V past the end of the sequence may hold anything: zero them
            const uint32_t mlo = (2 * tq < valid ? 0x0000ffffu : 0u) |
                                 (2 * tq + 1 < valid ? 0xffff0000u : 0u);
            const uint32_t mhi = (2 * tq + 8 < valid ? 0x0000ffffu : 0u) |
                                 (2 * tq + 9 < valid ? 0xffff0000u : 0u);
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
                const uint32_t ch = 2 * mt + v_chunk;
                uint32_t a0, a1, a2, a3;
                ldsm_x4_trans(vbase + (ch >> 3) * 2048 + swz128(v_row, ch & 7), a0, a1, a2, a3);
                o[mt][0] *= al0;
                o[mt][1] *= al1;
                o[mt][2] *= al0;
                o[mt][3] *= al1;
                mma_bf16_16816(o[mt], a0 & mlo, a1 & mlo, a2 & mhi, a3 & mhi, b0, b1);
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[slot]);
    }

    l0 = warp_sum_heads(l0);
    l1 = warp_sum_heads(l1);

    // ------------------------------------------------------------ finalise
    consumer_sync();  // every warp is done with the stage buffers
    float *scr = reinterpret_cast<float *>(smem) + warp * Cfg::kScratchFloats;
    if (gq == 0) {
        scr[2 * tq] = m0;
        scr[2 * tq + 1] = m1;
        scr[8 + 2 * tq] = l0;
        scr[8 + 2 * tq + 1] = l1;
    }
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
        const int d = 16 * mt + gq;
        scr[16 + d * 8 + 2 * tq] = o[mt][0];
        scr[16 + d * 8 + 2 * tq + 1] = o[mt][1];
        scr[16 + (d + 8) * 8 + 2 * tq] = o[mt][2];
        scr[16 + (d + 8) * 8 + 2 * tq + 1] = o[mt][3];
    }
    consumer_sync();
    if (!ok)
        return;

    const bool direct = (nsplit == 1) && !p.partial_only;
    const float *all = reinterpret_cast<const float *>(smem);
    const int total = Hkv * g * D;
    for (int idx = threadIdx.x; idx < total; idx += kConsumerWarps * 32) {
        const int d = idx % D;
        const int hn = idx / D;
        const int kh = hn / g;
        const int n = hn - kh * g;
        float M = kNegInf;
        for (int rr = 0; rr < R; ++rr)
            M = fmaxf(M, all[(rr * Hkv + kh) * Cfg::kScratchFloats + n]);
        float W = 0.f, acc = 0.f;
        for (int rr = 0; rr < R; ++rr) {
            const float *w = all + (rr * Hkv + kh) * Cfg::kScratchFloats;
            const float e = (w[n] == kNegInf) ? 0.f : exp2f(w[n] - M);
            W += e * w[8 + n];
            acc += e * w[16 + d * 8 + n];
        }
        const int h = kh * g + n;
        const float val = acc / W;
        const float lse2 = M + log2f(W);
        if (direct) {
            p.out[(static_cast<int64_t>(t) * p.num_heads + h) * D + d] = __float2bfloat16_rn(val);
            if (d == 0 && p.lse)
                p.lse[static_cast<int64_t>(t) * p.num_heads + h] = lse2 * kLn2;
        } else {
            const int64_t row = (static_cast<int64_t>(s) * p.max_splits + split) * p.num_heads + h;
            p.o_part[row * D + d] = val;
            if (d == 0)
                p.lse_part[row] = lse2;
        }
    }
}

// --------------------------------------------------------------------- combine
struct CombineParams {
    const int32_t *qsl;
    const int32_t *seq_lens;
    int32_t num_tokens;
    int32_t num_decodes;
    int32_t num_heads;
    int32_t split_tokens;
    int32_t max_splits;
    int32_t kv_begin;
    int32_t with_prefix;
    const float *o_part;   // decode split partials
    const float *lse_part;
    const float *o_pre;    // cascade: shared-prefix partial of every token [T, H, D]
    const float *lse_pre;
    const float *o_suf;    // cascade: suffix partial of every prefill token
    const float *lse_suf;
    __nv_bfloat16 *out;
    float *lse;
};

// One warp per (token, head) row: warp-shuffle max and sum of the parts'
// log2-sum-exp values, then the weighted sum of their normalised partial
// outputs -- the cascade merge, over n parts.  Parts of a decode token: its
// splits (and the shared prefix in a cascade); of a prefill token in a
// cascade: its suffix and the shared prefix.
template <int D>
__global__ void __launch_bounds__(256) decode_combine_kernel(const CombineParams p)
{
    constexpr int kPer = D / 32;
    const int64_t gw = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t nrows = int64_t(p.with_prefix ? p.num_tokens : p.num_decodes) * p.num_heads;
    if (gw >= nrows)
        return;
    const int t = static_cast<int>(gw / p.num_heads);  // decode s owns token s
    const int h = static_cast<int>(gw - int64_t(t) * p.num_heads);
    const int64_t row = int64_t(t) * p.num_heads + h;
    const float *parts_o[2];
    float parts_l[2];
    int nextra = 0;
    if (p.with_prefix) {
        parts_o[nextra] = p.o_pre + row * D;
        parts_l[nextra++] = p.lse_pre[row];
    }
    int n = 0;
    int64_t base = 0;
    if (t < p.num_decodes) {
        const int L = p.seq_lens[t];
        n = max(0, (L - p.kv_begin + p.split_tokens - 1) / p.split_tokens);
        if (n <= 1 && !p.with_prefix)
            return;  // finished by the decode kernel itself
        if (n > p.max_splits || p.qsl[t] != t)
            return;  // flagged by the decode kernel
        base = int64_t(t) * p.max_splits * p.num_heads + h;
    } else {
        const int64_t srow = int64_t(t - p.num_decodes) * p.num_heads + h;
        parts_o[nextra] = p.o_suf + srow * D;
        parts_l[nextra++] = p.lse_suf[srow];
    }
    float mx = kNegInf;
    for (int e = 0; e < nextra; ++e)
        mx = fmaxf(mx, parts_l[e]);
    for (int j = lane; j < n; j += 32)
        mx = fmaxf(mx, p.lse_part[base + int64_t(j) * p.num_heads]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float acc[kPer];
#pragma unroll
    for (int e = 0; e < kPer; ++e)
        acc[e] = 0.f;
    float ws = 0.f;
    if (mx != kNegInf) {
        for (int j = lane; j < n; j += 32)
            ws += exp2f(p.lse_part[base + int64_t(j) * p.num_heads] - mx);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            ws += __shfl_xor_sync(0xffffffffu, ws, o);
        for (int j = 0; j < n; ++j) {
            const int64_t prow = base + int64_t(j) * p.num_heads;
            const float w = exp2f(p.lse_part[prow] - mx);
            const float *src = p.o_part + prow * D + lane * kPer;
#pragma unroll
            for (int e = 0; e < kPer; ++e)
                acc[e] += w * src[e];
        }
        for (int x = 0; x < nextra; ++x) {
            if (parts_l[x] == kNegInf)
                continue;  // an empty part contributes nothing, whatever it holds
            const float w = exp2f(parts_l[x] - mx);
            ws += w;
            const float *src = parts_o[x] + lane * kPer;
#pragma unroll
            for (int e = 0; e < kPer; ++e)
                acc[e] += w * src[e];
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
DecodePlan plan_decode(int32_t requested_split, int32_t num_decodes, int32_t max_seq_len,
                       int32_t kv_begin, int32_t num_kv_heads, int num_sms)
{
    DecodePlan dp;
    dp.stage_keys = 16 * (kConsumerWarps / num_kv_heads);
    const int64_t span = std::max<int64_t>(1, int64_t(max_seq_len) - kv_begin);
    int64_t split;
    if (requested_split > 0) {
        split = requested_split;
    } else {
        // About eight CTAs per SM over the batch, taking the mean decode length
        // as 60% of the longest; at least four stages per CTA.
        const double total = 0.6 * double(num_decodes) * double(span);
        split = static_cast<int64_t>(total / (8.0 * std::max(1, num_sms))) + 1;
        split = std::max<int64_t>(split, 4 * dp.stage_keys);
    }
    split = (split + dp.stage_keys - 1) / dp.stage_keys * dp.stage_keys;
    split = std::min<int64_t>(split, (span + dp.stage_keys - 1) / dp.stage_keys * dp.stage_keys);
    dp.split_tokens = static_cast<int32_t>(split);
    dp.max_splits = static_cast<int32_t>((span + split - 1) / split);
    return dp;
}

template <int D>
static cudaError_t launch_decode_d(const Fwd &f, const DecodePlan &dp, const Workspace &ws,
                                   char *wsp, const CUtensorMap &kv_map, int32_t kv_begin,
                                   bool partial_only)
{
    using Cfg = DecodeCfg<D>;
    static int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(paged_decode_kernel<D>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(Cfg::kSmemBytes));
        if (e != cudaSuccess)
            return e;
        configured_device = dev;
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
    p.split_tokens = dp.split_tokens;
    p.max_splits = dp.max_splits;
    p.kv_begin = kv_begin;
    p.partial_only = partial_only ? 1 : 0;
    p.scale_log2 = f.scale * 1.4426950408889634f;
    p.out = static_cast<__nv_bfloat16 *>(f.out);
    p.lse = f.lse;
    p.o_part = reinterpret_cast<float *>(wsp + ws.o_part);
    p.lse_part = reinterpret_cast<float *>(wsp + ws.lse_part);
    dim3 grid(dp.max_splits, f.num_decodes);
    count_launch();
    paged_decode_kernel<D><<<grid, kDecodeThreads, Cfg::kSmemBytes, f.stream>>>(kv_map, p);
    return cudaGetLastError();
}

cudaError_t launch_decode(const Fwd &f, const DecodePlan &dp, const Workspace &ws, char *wsp,
                          const CUtensorMap &kv_map, int32_t kv_begin, bool partial_only)
{
    if (f.num_decodes == 0)
        return cudaSuccess;
    if (f.head_size == 128)
        return launch_decode_d<128>(f, dp, ws, wsp, kv_map, kv_begin, partial_only);
    return launch_decode_d<64>(f, dp, ws, wsp, kv_map, kv_begin, partial_only);
}

cudaError_t launch_decode_combine(const Fwd &f, const DecodePlan &dp, const Workspace &ws,
                                  char *wsp, int32_t kv_begin, bool with_prefix)
{
    if (!with_prefix && (f.num_decodes == 0 || dp.max_splits <= 1))
        return cudaSuccess;
    CombineParams p;
    p.qsl = f.qsl;
    p.seq_lens = f.seq_lens;
    p.num_tokens = f.num_tokens;
    p.num_decodes = f.num_decodes;
    p.num_heads = f.num_heads;
    p.split_tokens = dp.split_tokens;
    p.max_splits = dp.max_splits;
    p.kv_begin = kv_begin;
    p.with_prefix = with_prefix ? 1 : 0;
    p.o_part = reinterpret_cast<const float *>(wsp + ws.o_part);
    p.lse_part = reinterpret_cast<const float *>(wsp + ws.lse_part);
    p.o_pre = reinterpret_cast<const float *>(wsp + ws.o_pre);
    p.lse_pre = reinterpret_cast<const float *>(wsp + ws.lse_pre);
    p.o_suf = reinterpret_cast<const float *>(wsp + ws.o_suf);
    p.lse_suf = reinterpret_cast<const float *>(wsp + ws.lse_suf);
    p.out = static_cast<__nv_bfloat16 *>(f.out);
    p.lse = f.lse;
    const int64_t warps = int64_t(with_prefix ? f.num_tokens : f.num_decodes) * f.num_heads;
    const unsigned grid = static_cast<unsigned>((warps * 32 + 255) / 256);
    count_launch();
    if (f.head_size == 128)
        decode_combine_kernel<128><<<grid, 256, 0, f.stream>>>(p);
    else
        decode_combine_kernel<64><<<grid, 256, 0, f.stream>>>(p);
    return cudaGetLastError();
}

uint32_t decode_take_error() { return take_device_error(); }

}  // namespace pka
