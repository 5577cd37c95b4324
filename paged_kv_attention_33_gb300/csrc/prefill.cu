// prefill.cu -- varlen causal prefill / chunked prefill on the fifth-generation
// tensor cores (tcgen05) with accumulators in tensor memory (TMEM).
//
// What it computes (the "El especialista del plato estrella" blog, "Por que
// prefill y decode son problemas opuestos"): N queries against N (+ prior
// context) keys, N^2 d flops over N d bytes, so it is bound by the tensor
// cores.  For sequence s with q_s queries after c_s cached tokens, query i
// admits keys j <= c_s + i (bottom-right causal alignment), keys read through
// the block table (the blog's "Como lee el backend el KV paginado").
//
// Work item: (sequence s, 256-query super-tile, query head h) = two 128-row
// tiles A and B that share every K/V tile, in a persistent grid (one CTA per
// SM, or a cascade prefix pass's share of the SMs).  Items are claimed
// dynamically from a global counter (the heaviest causal tiles of each
// sequence first), so CTAs that draw light items take more.  The pool it reads
// may be the forward's 128-key re-blocking of a 16-key-page pool (one box per
// tile half instead of one per page: at 16-key pages one SM's TMA box rate,
// not the MMAs, bounded this kernel).
// Roles (384 threads, three warpgroups):
//   warp 0      TMA producer: Q tiles once per item, K and V tiles of 128 keys
//               into two-stage rings (K one tile ahead of V, each freed by its
//               own barrier), one TMA box per page straight from the pool
//               (128-byte swizzled), block ids looked up one per lane;
//   warp 1      MMA issuer (one thread).  Per K/V tile j it issues
//                 PV_A(j-1), S_A(j), PV_B(j-1), S_B(j)
//               so that while one softmax warpgroup works on its S tile the
//               tensor core runs the other tile's MMAs;
//               S = Q K^T: M=128, N=128, K=head_size, both operands in smem;
//               O += P V: M=128, N=head_size, K=128 keys, P read from TMEM;
//   warp 2      TMEM allocator;
//   warps 4-7   softmax of tile A, warps 8-11 softmax of tile B: thread r owns
//               query row r; it reads its S row from TMEM, masks (only on
//               tiles that need it), runs the base-2 online softmax with the
//               scale folded into one FFMA per element, writes P back over S
//               as bf16, rescales its O row in TMEM when its reference max
//               moved by more than 8, and at the end writes out = O / l and lse.
// Registers: the producer warpgroup gives registers back (setmaxnreg) to the
// two softmax warpgroups: 128 x 104 + 256 x 200 = 64512 = 384 x 168 at launch.
// TMEM columns: S_A [0,128), S_B [128,256), O_A [256, 256+D), O_B [256+D, 256+2D).
#include <math.h>

#include <atomic>
#include <algorithm>
#include <numeric>

#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace pka {

constexpr int kBM = 128;             // query rows per tile
constexpr int kBN = 128;             // keys per tile
constexpr int kSuper = 2 * kBM;      // query rows per work item (tiles A and B)
constexpr int kPfThreads = 384;
// Register split by setmaxnreg: warps 0-3 (TMA producer, MMA issuer, TMEM
// allocator, spare) drop to kPfRegsLow, the eight softmax warps rise to
// kPfRegsHigh.  setmaxnreg.inc draws on the registers the block was launched
// with, so the split has to fit in kPfThreads x (registers per thread at
// launch), or the softmax warps would wait for registers forever: 168 under
// __launch_bounds__(384, 1), checked again at launch against the compiled kernel.
constexpr uint32_t kPfRegsLow = 104, kPfRegsHigh = 200;
constexpr uint32_t kPfRegsSplit = 4 * 32 * kPfRegsLow + 8 * 32 * kPfRegsHigh;
static_assert(kPfRegsSplit <= uint32_t(kPfThreads) * 168, "setmaxnreg split");
constexpr int kPfStages = 2;
constexpr int kMaxPrefillSeqs = 4096;
constexpr uint32_t kTmemCols = 512;
constexpr float kPfNegInf = -INFINITY;
constexpr float kPfLn2 = 0.69314718055994530942f;
constexpr float kRescaleThreshold = 8.f;  // log2 units: p stays <= 256

struct PrefillParams {
    const int32_t *qsl;
    const int32_t *seq_lens;
    const int32_t *block_table;
    int32_t bt_stride;
    int32_t first_seq;  // prefill sequences are [first_seq, num_seqs)
    int32_t num_seqs;
    int32_t num_tokens;
    int32_t num_heads;
    int32_t group;
    int32_t block_size;
    int32_t box_rows;  // rows per K/V TMA box: gcd(block_size, 128)
    int32_t num_blocks;
    int32_t num_kv_heads;
    int32_t kv_lo;     // first key attended
    int32_t kv_cap;    // keys >= kv_cap are not attended
    int32_t causal;
    float scale_log2;
    float out_scale;     // output multiplier (the V scale of a dequantised fp8 copy)
    int32_t partial;     // 0: bf16 out + ln lse; 1: fp32 partial + log2 lse
    int32_t token_base;  // partial rows are (t - token_base) * H + h
    int32_t shared_prefix;  // 1: every token of the batch against keys [0, kv_cap) of
                            //    block-table row 0 (the cascade's shared prefix)
    __nv_bfloat16 *out;
    float *lse;
    float *o_part;
    float *lse_part;
    int32_t *item_counter;  // work items claimed so far (zeroed before each launch)
    int32_t kv_splits;      // shared_prefix: key chunks, split_tiles key tiles each
    int32_t split_tiles;
    int32_t test_skip_copies;  // failure-path test: the producer issues nothing
    // 1: a K/V tile that starts at or after its sequence's context (all its
    // keys are this step's) is read from the step's key/value rows
    // ([num_tokens, Hkv, D], one box of 128 tokens per half) instead of the pool
    int32_t new_from_input;
    int32_t trigger_dependents;  // the cascade's suffix decode may start beside this pass
    int32_t after_decode;        // the dependent of the decode just before it: wait for it at the end
    int32_t after_copy;          // the dependent of the block copy just before it: wait for it first
};

template <int D>
struct PfCfg {
    static constexpr int kHalves = D / 64;
    static constexpr int kHalfBytes = 128 * 128;             // 128 rows x 128 B
    static constexpr int kTileBytes = kHalves * kHalfBytes;  // one Q, K or V tile
    static constexpr int kQOff = 0;                          // Q_A, then Q_B
    static constexpr int kKOff = 2 * kTileBytes;
    static constexpr int kVOff = kKOff + kPfStages * kTileBytes;
    static constexpr int kBarOff = kVOff + kPfStages * kTileBytes;
    static constexpr int kNumBars = 24;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;  // tmem base, abort flag
    static constexpr int kPrefixOff = kMiscOff + 16;
    static constexpr size_t kSmemBytes = kPrefixOff + (kMaxPrefillSeqs + 1) * 4 + 1024;
    static constexpr uint32_t kIdescS = idesc_bf16_f32(kBM, kBN, 0, 0);
    static constexpr uint32_t kIdescPV = idesc_bf16_f32(kBM, D, 0, 1);
    static_assert(kSmemBytes <= 232448, "shared memory");
};

// One work item: two query tiles (A = rows [0,128), B = rows [128,256) of the
// super-tile) of one head against the K/V tiles of one sequence.
struct PfItem {
    int s, h, t0, ctx, L, qidx0;
    int rows[2];   // valid query rows of tile A / B (0: tile absent)
    int n_kv[2];   // K/V tiles tile A / B attends
    int n_kv_all;  // K/V tiles the item loads (max of the two)
    int kv_lo;     // first key of the item (a multiple of the key tile)
    int kv_hi;     // keys [kv_lo, kv_hi) are loaded
    int split;     // shared_prefix: key chunk of the item (its partial's slice)
};

__device__ __forceinline__ int pf_tiles_of(int kv_lo, int hi)
{
    return hi > kv_lo ? (hi - kv_lo + kBN - 1) / kBN : 0;
}

__device__ __forceinline__ bool pf_item(const PrefillParams &p, const int32_t *prefix, int nseq,
                                        int item, PfItem &it)
{
    int qlen;
    if (p.shared_prefix) {
        // one pseudo-sequence: all tokens of the batch, keys [0, kv_cap) of the
        // prefix every sequence shares, no mask (the prefix precedes every query)
        // (keys of chunk `split` only; the chunks' partials are merged later)
        const int tiles = (p.num_tokens + kSuper - 1) / kSuper;
        const int per_split = tiles * p.num_heads;
        if (item >= per_split * p.kv_splits)
            return false;
        it.split = item / per_split;
        const int rem = item - it.split * per_split;
        it.h = rem % p.num_heads;
        const int st_idx = tiles - 1 - rem / p.num_heads;
        it.s = 0;
        qlen = p.num_tokens;
        it.t0 = st_idx * kSuper;
        it.qidx0 = it.t0;
        it.kv_lo = p.kv_lo + it.split * p.split_tiles * kBN;
        it.L = min(p.kv_cap, it.kv_lo + p.split_tiles * kBN);
        it.ctx = it.L;
    } else {
        const int tiles = prefix[nseq];
        if (item >= tiles * p.num_heads)
            return false;
        it.h = item % p.num_heads;
        const int r = item / p.num_heads;
        int lo = 0, hi = nseq;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (prefix[mid] <= r)
                lo = mid;
            else
                hi = mid;
        }
        it.s = p.first_seq + lo;
        const int ntile = prefix[lo + 1] - prefix[lo];
        const int st_idx = ntile - 1 - (r - prefix[lo]);  // heaviest super-tile first
        const int q0 = p.qsl[it.s];
        qlen = p.qsl[it.s + 1] - q0;
        it.L = p.seq_lens[it.s];
        it.ctx = it.L - qlen;
        it.qidx0 = st_idx * kSuper;
        it.t0 = q0 + it.qidx0;
        it.kv_lo = p.kv_lo;
        it.split = 0;
    }
    it.rows[0] = max(0, min(kBM, qlen - it.qidx0));
    it.rows[1] = max(0, min(kBM, qlen - it.qidx0 - kBM));
    int all_hi = 0;
    for (int tl = 0; tl < 2; ++tl) {
        int hi = 0;
        if (it.rows[tl] > 0) {
            if (p.shared_prefix || !p.causal)
                hi = it.L;
            else
                hi = min(it.L, it.ctx + it.qidx0 + tl * kBM + it.rows[tl]);
            hi = min(hi, p.kv_cap);
        }
        it.n_kv[tl] = it.rows[tl] > 0 ? pf_tiles_of(it.kv_lo, hi) : 0;
        all_hi = max(all_hi, hi);
    }
    it.kv_hi = all_hi;
    it.n_kv_all = max(it.n_kv[0], it.n_kv[1]);
    if (!p.shared_prefix && p.kv_lo > 0 && it.ctx < p.kv_lo) {
        // a cascade suffix pass needs every query after the shared prefix
        flag_error(kErrBadMetadata);
        it.n_kv[0] = it.n_kv[1] = it.n_kv_all = 0;
    }
    return true;
}

// Bounded wait that also gives up once another role has given up.
__device__ __forceinline__ bool pf_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag)
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

template <uint32_t N>
__device__ __forceinline__ void reg_dealloc()
{
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

template <uint32_t N>
__device__ __forceinline__ void reg_alloc()
{
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

struct PfBars {
    uint64_t *q_full, *q_empty, *k_full, *v_full, *k_empty, *v_empty;
    uint64_t *s_full, *p_full, *o_done, *o_free;  // [2] each: tile A, tile B
    uint64_t *drain;
    uint64_t *item_full, *item_empty;  // [2] each: the work-item hand-off ring
    volatile int32_t *item_slot;       // [2]
};

// Number of consumer warps of the item ring: the MMA warp and 8 softmax warps.
constexpr uint32_t kItemReaders = 9;

// The n-th work item the producer handed to this CTA (-1: no more work).
__device__ __forceinline__ int pf_next_item(const PfBars &bars, uint32_t n,
                                            volatile int *abort_flag)
{
    const int slot = n & 1;
    if (!pf_wait(&bars.item_full[slot], (n >> 1) & 1, abort_flag))
        return -1;
    const int item = bars.item_slot[slot];
    __syncwarp();
    if ((threadIdx.x & 31) == 0)
        mbar_arrive(&bars.item_empty[slot]);
    return item;
}

// ---------------------------------------------------------------- softmax role
template <int D>
__device__ __forceinline__ void pf_softmax(const PrefillParams &p, const int32_t *prefix,
                                           int nseq, const PfBars &bars, int tl, uint32_t tS,
                                           uint32_t tO, volatile int *abort_flag)
{
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int wq = warp & 3;  // TMEM lane quarter of this warp
    const int r = wq * 32 + lane;
    const uint32_t lane_off = uint32_t(wq * 32) << 16;
    const uint32_t ts = tS + lane_off;
    uint32_t s_n = 0, pv_n = 0, n_got = 0;
    PfItem it;
    for (;;) {
        const int item = pf_next_item(bars, n_got++, abort_flag);
        if (item < 0 || !pf_item(p, prefix, nseq, item, it))
            break;
        const int rows = it.rows[tl];
        const int nkv = it.n_kv[tl];
        const bool valid = r < rows;
        const int t = it.t0 + tl * kBM + r;
        if (rows == 0)
            continue;
        if (nkv == 0) {
            // no admitted key at all: an empty part (cascade partial mode only)
            if (valid && p.partial) {
                const int64_t row =
                    (int64_t(it.split) * p.num_tokens + t - p.token_base) * p.num_heads + it.h;
                for (int d = 0; d < D; ++d)
                    p.o_part[row * D + d] = 0.f;
                p.lse_part[row] = kPfNegInf;
            }
            continue;
        }
        int hi_row;
        if (p.shared_prefix || !p.causal)
            hi_row = it.L;
        else
            hi_row = min(it.L, it.ctx + it.qidx0 + tl * kBM + r + 1);
        hi_row = min(hi_row, p.kv_cap);
        float m = kPfNegInf, l = 0.f;
        for (int jt = 0; jt < nkv; ++jt, ++s_n) {
            if (!pf_wait(&bars.s_full[tl], s_n & 1, abort_flag))
                return;
            tc_fence_after();
            uint32_t x[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c)
                tmem_ld32(ts + c * 32, x[c]);
            tmem_wait_ld();
            const int lim = hi_row - (it.kv_lo + jt * kBN);  // columns c < lim admitted
            const bool full_tile = __all_sync(0xffffffffu, lim >= kBN);
            // row max of the raw logits: three-input max, four chains; the scale
            // is positive so max and scaling commute
            float mx4[4] = {kPfNegInf, kPfNegInf, kPfNegInf, kPfNegInf};
            if (!full_tile) {
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (c * 32 + i >= lim)
                            x[c][i] = __float_as_uint(kPfNegInf);
            }
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int i = 0; i < 32; i += 2)
                    mx4[(i >> 1) & 3] = fmax3(mx4[(i >> 1) & 3], __uint_as_float(x[c][i]),
                                              __uint_as_float(x[c][i + 1]));
            const float mx = fmax3(fmaxf(mx4[0], mx4[1]), mx4[2], mx4[3]) * p.scale_log2;
            // The reference max m moves only when the row max passes it by more
            // than the threshold: every p stays <= 2^8 and the O rescale in TMEM
            // is rare.  Exact either way: lse and 1/l use the same reference.
            const float m_new = mx > m + kRescaleThreshold ? mx : m;
            const float base = m_new == kPfNegInf ? 0.f : m_new;
            // p = 2^(x*scale - base): the argument two elements at a time
            // (fma.f32x2), the row sum likewise (add.f32x2), P packed to bf16
            const uint64_t sl2 = pack_f32x2(p.scale_log2, p.scale_log2);
            const uint64_t nb2 = pack_f32x2(-base, -base);
            uint64_t sum2[2] = {pack_f32x2(0.f, 0.f), pack_f32x2(0.f, 0.f)};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const uint64_t arg = fma_f32x2(
                        pack_f32x2(__uint_as_float(x[c][2 * i]), __uint_as_float(x[c][2 * i + 1])),
                        sl2, nb2);
                    float a0, a1;
                    unpack_f32x2(arg, a0, a1);
                    const float p0 = fast_exp2(a0);
                    const float p1 = fast_exp2(a1);
                    sum2[i & 1] = add_f32x2(sum2[i & 1], pack_f32x2(p0, p1));
                    pk[i] = pack_bf16x2(p0, p1);
                }
                tmem_st16(ts + c * 16, pk);
            }
            tmem_wait_st();
            float s0, s1, s2, s3;
            unpack_f32x2(sum2[0], s0, s1);
            unpack_f32x2(sum2[1], s2, s3);
            const float alpha = fast_exp2(m - base);  // exactly 1 when m did not move
            l = l * alpha + ((s0 + s1) + (s2 + s3));
            const bool moved = m_new != m;
            m = m_new;
            if (jt > 0) {
                // O holds PV of the previous tiles: wait for the last one, then
                // rescale the rows whose reference moved
                if (!pf_wait(&bars.o_done[tl], pv_n & 1, abort_flag))
                    return;
                ++pv_n;
                tc_fence_after();
                if (__any_sync(0xffffffffu, moved)) {
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        tmem_ld32(tO + lane_off + c * 32, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tmem_st32(tO + lane_off + c * 32, o);
                    }
                    tmem_wait_st();
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&bars.p_full[tl]);
        }
        // ---- epilogue: out = O / l, lse
        if (!pf_wait(&bars.o_done[tl], pv_n & 1, abort_flag))
            return;
        ++pv_n;
        tc_fence_after();
        {
            const float inv = l > 0.f ? p.out_scale / l : 0.f;
            const float lse2 = m + log2f(l);
            const int64_t orow = int64_t(t) * p.num_heads + it.h;
            const int64_t prow =
                (int64_t(it.split) * p.num_tokens + t - p.token_base) * p.num_heads + it.h;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(tO + lane_off + c * 32, o);
                tmem_wait_ld();
                if (valid) {
                    if (p.partial) {
                        float4 *dst = reinterpret_cast<float4 *>(p.o_part + prow * D + c * 32);
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            dst[i] = make_float4(__uint_as_float(o[4 * i]) * inv,
                                                 __uint_as_float(o[4 * i + 1]) * inv,
                                                 __uint_as_float(o[4 * i + 2]) * inv,
                                                 __uint_as_float(o[4 * i + 3]) * inv);
                    } else {
                        uint4 *dst = reinterpret_cast<uint4 *>(p.out + orow * D + c * 32);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            dst[i] = make_uint4(pack_bf16x2(__uint_as_float(o[8 * i]) * inv,
                                                            __uint_as_float(o[8 * i + 1]) * inv),
                                                pack_bf16x2(__uint_as_float(o[8 * i + 2]) * inv,
                                                            __uint_as_float(o[8 * i + 3]) * inv),
                                                pack_bf16x2(__uint_as_float(o[8 * i + 4]) * inv,
                                                            __uint_as_float(o[8 * i + 5]) * inv),
                                                pack_bf16x2(__uint_as_float(o[8 * i + 6]) * inv,
                                                            __uint_as_float(o[8 * i + 7]) * inv));
                    }
                }
            }
            if (valid) {
                if (p.partial)
                    p.lse_part[prow] = lse2;
                else if (p.lse)
                    p.lse[orow] = lse2 * kPfLn2;
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&bars.o_free[tl]);
    }
}

template <int D, bool kHnd>
__global__ void __launch_bounds__(kPfThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap q_map,
                      const __grid_constant__ CUtensorMap kv_map,
                      const __grid_constant__ CUtensorMap kin_map,
                      const __grid_constant__ CUtensorMap vin_map, const PrefillParams p)
{
    using Cfg = PfCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *b = reinterpret_cast<uint64_t *>(smem + Cfg::kBarOff);
    PfBars bars;
    bars.q_full = b + 0;
    bars.q_empty = b + 1;
    bars.k_full = b + 2;     // [kPfStages]
    bars.v_full = b + 4;     // [kPfStages]
    bars.k_empty = b + 6;    // [kPfStages]: K tile free once the S MMAs read it
    bars.v_empty = b + 18;   // [kPfStages]: V tile free once the PV MMAs read it
    bars.s_full = b + 8;     // [2]
    bars.p_full = b + 10;    // [2]
    bars.o_done = b + 12;    // [2]
    bars.o_free = b + 14;    // [2]
    bars.drain = b + 16;
    bars.item_full = b + 20;   // [2]
    bars.item_empty = b + 22;  // [2]
    bars.item_slot = reinterpret_cast<volatile int32_t *>(smem + Cfg::kMiscOff + 8);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + Cfg::kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + Cfg::kMiscOff + 4);
    int32_t *prefix = reinterpret_cast<int32_t *>(smem + Cfg::kPrefixOff);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nseq = p.shared_prefix ? 0 : p.num_seqs - p.first_seq;

    // The dependent launch (a cascade's suffix decode, which never reads what
    // this pass writes) may be scheduled on the free SMs right away.
    if (p.trigger_dependents)
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // ---- prefix sums of 256-query super-tiles per prefill sequence
    {
        const int per = (nseq + kPfThreads - 1) / kPfThreads;
        const int a = min(nseq, int(threadIdx.x) * per);
        const int e = min(nseq, a + per);
        int sum = 0;
        for (int k = a; k < e; ++k) {
            const int s = p.first_seq + k;
            const int ql = p.qsl[s + 1] - p.qsl[s];
            sum += ql > 0 ? (ql + kSuper - 1) / kSuper : 0;
        }
        int run = block_exclusive_scan<kPfThreads>(sum, prefix + nseq);
        for (int k = a; k < e; ++k) {
            prefix[k] = run;
            const int s = p.first_seq + k;
            const int ql = p.qsl[s + 1] - p.qsl[s];
            run += ql > 0 ? (ql + kSuper - 1) / kSuper : 0;
        }
    }

    if (threadIdx.x == 0) {
        mbar_init(bars.q_full, 1);
        mbar_init(bars.q_empty, 1);
        for (int i = 0; i < kPfStages; ++i) {
            mbar_init(&bars.k_full[i], 1);
            mbar_init(&bars.v_full[i], 1);
            mbar_init(&bars.k_empty[i], 1);
            mbar_init(&bars.v_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars.s_full[i], 1);
            mbar_init(&bars.p_full[i], 4);
            mbar_init(&bars.o_done[i], 1);
            mbar_init(&bars.o_free[i], 4);
        }
        mbar_init(bars.drain, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars.item_full[i], 1);
            mbar_init(&bars.item_empty[i], kItemReaders);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 2) {
        tmem_alloc(tmem_holder, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_holder;

    // The programmatic dependent of the fp8 block copy: everything above
    // overlapped the copy; its blocks and block table are read from here on.
    if (p.after_copy)
        asm volatile("griddepcontrol.wait;" ::: "memory");

    // All 512 columns belong to this CTA, so the allocation starts at lane 0,
    // column 0: the MMA issuer's TMEM addresses are compile-time constants.
    if (tbase != 0) {
        if (threadIdx.x == 0)
            flag_error(kErrTmemAlloc);
    } else if (warp < 4) {
        reg_dealloc<kPfRegsLow>();
        if (warp == 0) {
            // ============================================================ producer
            if (lane == 0) {
                tma_prefetch_desc(&q_map);
                tma_prefetch_desc(&kv_map);
                if (p.new_from_input) {
                    tma_prefetch_desc(&kin_map);
                    tma_prefetch_desc(&vin_map);
                }
            }
            const uint64_t pol_kv = l2_policy_evict_last();
            const uint64_t pol_q = l2_policy_evict_first();
            uint32_t li = 0, kv_it = 0, n_pub = 0;
            // copies armed so far: Q loads, K and V stages (for the wind-down)
            uint32_t q_armed = 0, k_armed = 0, v_armed = 0;
            PfItem it;
            for (;;) {
                if (p.test_skip_copies)
                    break;  // publish no item: the other roles' first wait runs out
                // claim the next work item (dynamic: a CTA that finishes early
                // takes more) and hand its index to the MMA and softmax warps
                int item = 0;
                if (lane == 0)
                    item = atomicAdd(p.item_counter, 1);
                item = __shfl_sync(0xffffffffu, item, 0);
                const bool have = pf_item(p, prefix, nseq, item, it);
                const int slot = n_pub & 1;
                if (n_pub >= 2 &&
                    !pf_wait(&bars.item_empty[slot], ((n_pub >> 1) - 1) & 1, abort_flag))
                    break;
                if (lane == 0) {
                    bars.item_slot[slot] = have ? item : -1;
                    mbar_arrive(&bars.item_full[slot]);
                }
                __syncwarp();
                ++n_pub;
                if (!have)
                    break;
                if (it.n_kv_all == 0)
                    continue;
                const int kvh = it.h / p.group;
                const int32_t *bt = p.block_table + int64_t(it.s) * p.bt_stride;
                const int kv_hi = it.kv_hi;
                // lane b owns TMA box b of every K/V tile; its block id is looked
                // up for the next tile before waiting for a free stage
                // a tile of this step's keys only: read from the step's rows
                auto from_input = [&](int key0) { return p.new_from_input && key0 >= it.ctx; };
                auto lane_block = [&](int jt) -> int {
                    const int key0 = it.kv_lo + jt * kBN;
                    const int nbox = (min(kBN, kv_hi - key0) + p.box_rows - 1) / p.box_rows;
                    if (lane >= nbox || from_input(key0))
                        return -1;
                    const int col = (key0 + lane * p.box_rows) / p.block_size;
                    int blk = col < p.bt_stride ? bt[col] : -1;
                    if (blk < 0 || blk >= p.num_blocks) {
                        flag_error(kErrBlockOutOfPool);
                        blk = 0;  // keep the byte count whole; the result is flagged
                    }
                    return blk;
                };
                int blk_next = lane_block(0);
                if (li > 0 && !pf_wait(bars.q_empty, (li - 1) & 1, abort_flag))
                    break;
                ++q_armed;
                if (lane == 0) {
                    const int ntiles = it.rows[1] > 0 ? 2 : 1;
                    mbar_arrive_expect_tx(bars.q_full, ntiles * Cfg::kTileBytes);
                    for (int tl = 0; tl < ntiles; ++tl)
                        for (int hf = 0; hf < Cfg::kHalves; ++hf)
                            tma_load_3d(smem + Cfg::kQOff + tl * Cfg::kTileBytes +
                                            hf * Cfg::kHalfBytes,
                                        &q_map, bars.q_full, hf * 64, it.h, it.t0 + tl * kBM,
                                        pol_q);
                }
                // K runs one tile ahead of V: K(j+1) is issued before V(j), and
                // each has its own free barrier, so the next K tile streams in
                // while the PV MMAs of the current tile still hold V
                const uint32_t kv_base = kv_it;
                auto issue = [&](int which, int jt, int blk) -> bool {
                    const uint32_t n = kv_base + jt;
                    const int st = n % kPfStages;
                    const uint32_t rnd = n / kPfStages;
                    uint64_t *emp = which ? &bars.v_empty[st] : &bars.k_empty[st];
                    if (rnd > 0 && !pf_wait(emp, (rnd - 1) & 1, abort_flag))
                        return false;
                    const int key0 = it.kv_lo + jt * kBN;
                    uint64_t *bar = which ? &bars.v_full[st] : &bars.k_full[st];
                    uint8_t *tile = smem + (which ? Cfg::kVOff : Cfg::kKOff) + st * Cfg::kTileBytes;
                    if (from_input(key0)) {
                        // token of key key0: the sequence's first query token is
                        // the step row of its first new key (key ctx); rows past
                        // the sequence's end are masked, V's zeroed by the MMA warp
                        const int tok = it.t0 - it.qidx0 + (key0 - it.ctx);
                        if (lane == 0) {
                            mbar_arrive_expect_tx(bar, kBN * 128 * Cfg::kHalves);
                            for (int hf = 0; hf < Cfg::kHalves; ++hf)
                                tma_load_3d(tile + hf * Cfg::kHalfBytes, which ? &vin_map : &kin_map,
                                            bar, hf * 64, kvh, tok, pol_kv);
                        }
                        __syncwarp();
                        (which ? v_armed : k_armed) = n + 1;
                        return true;
                    }
                    const int nbox = (min(kBN, kv_hi - key0) + p.box_rows - 1) / p.box_rows;
                    const uint32_t bytes = nbox * p.box_rows * 128 * Cfg::kHalves;
                    if (lane == 0)
                        mbar_arrive_expect_tx(bar, bytes);
                    __syncwarp();
                    (which ? v_armed : k_armed) = n + 1;
                    if (lane < nbox) {
                        // coordinates in the pool map: NHD (head, page*bs + offset),
                        // HND (offset, page*Hkv + head), page = block*2 + (K|V)
                        const int key = key0 + lane * p.box_rows;
                        const int c1 = kHnd ? key % p.block_size : kvh;
                        const int row = kHnd ? (blk * 2 + which) * p.num_kv_heads + kvh
                                             : (blk * 2 + which) * p.block_size + key % p.block_size;
                        uint8_t *dst = tile + lane * p.box_rows * 128;
                        for (int hf = 0; hf < Cfg::kHalves; ++hf)
                            tma_load_3d(dst + hf * Cfg::kHalfBytes, &kv_map, bar, hf * 64, c1,
                                        row, pol_kv);
                    }
                    return true;
                };
                bool stop = !issue(0, 0, blk_next);
                for (int jt = 0; jt < it.n_kv_all && !stop; ++jt) {
                    const int blk_v = blk_next;
                    if (jt + 1 < it.n_kv_all) {
                        blk_next = lane_block(jt + 1);
                        if (!issue(0, jt + 1, blk_next)) {
                            stop = true;
                            break;
                        }
                    }
                    if (!issue(1, jt, blk_v))
                        stop = true;
                }
                kv_it += it.n_kv_all;
                if (stop)
                    break;
                ++li;
            }
            // Wind-down: the CTA must not exit (nor free its TMEM) while a copy
            // this warp issued still writes shared memory.  A K or V stage is
            // refilled only after the MMAs that read it completed, and a Q tile
            // only after the last S of its item, so only the last kPfStages K
            // and V stages and the last Q load can still be in flight: wait for
            // their full barriers (bounded, whatever the abort flag says).  On
            // the normal path each test succeeds at once.
            for (uint32_t n = k_armed > kPfStages ? k_armed - kPfStages : 0; n < k_armed; ++n)
                mbar_wait(&bars.k_full[n % kPfStages], (n / kPfStages) & 1);
            for (uint32_t n = v_armed > kPfStages ? v_armed - kPfStages : 0; n < v_armed; ++n)
                mbar_wait(&bars.v_full[n % kPfStages], (n / kPfStages) & 1);
            if (q_armed > 0)
                mbar_wait(bars.q_full, (q_armed - 1) & 1);
        } else if (warp == 1) {
            // ============================================================ MMA issuer
            // One elected lane issues every MMA and commit.  At N = 128 an MMA
            // runs 64 cycles, so the issue has to keep up while the softmax warps
            // of the same sub-partitions compete for the scheduler: TMEM addresses
            // are constants (the allocation starts at 0) and a shared-memory
            // descriptor is its low word alone (start address and LBO; the high
            // word is common to all operands), so that a k-step or a stage costs
            // one 32-bit add.  Every tile lies below 256 KB of shared memory, so
            // the add never carries out of the 14-bit start-address field.
            const uint32_t q_lo0 = smem_desc_lo(smem_addr(smem + Cfg::kQOff), 16);
            const uint32_t k_lo0 = smem_desc_lo(smem_addr(smem + Cfg::kKOff), 16);
            const uint32_t v_lo0 = smem_desc_lo(smem_addr(smem + Cfg::kVOff), Cfg::kHalfBytes);
            constexpr uint32_t kTileStep = Cfg::kTileBytes >> 4;
            uint32_t li = 0, kv_it = 0;
            // per Q tile: P tiles consumed, items that used the tile (registers:
            // the tile loop below is unrolled, so every index is a constant)
            uint32_t p_cnt[2] = {0, 0}, item_cnt[2] = {0, 0};
            PfItem it;
            bool ok = true;
            uint32_t n_got = 0;
            while (ok) {
                const int item = pf_next_item(bars, n_got++, abort_flag);
                if (item < 0 || !pf_item(p, prefix, nseq, item, it))
                    break;
                if (it.n_kv_all == 0)
                    continue;
                if (!pf_wait(bars.q_full, li & 1, abort_flag))
                    break;
                tc_fence_after();
                const int n = it.n_kv_all;
                const int nk[2] = {it.n_kv[0], it.n_kv[1]};
                const int kv_lo = it.kv_lo, kv_hi = it.kv_hi;
                for (int jt = 0; jt <= n && ok; ++jt) {
                    const uint32_t kn = kv_it + jt;
                    const int st = kn % kPfStages;
                    if (jt < n) {
                        if (!pf_wait(&bars.k_full[st], (kn / kPfStages) & 1, abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                    }
#pragma unroll
                    for (int tl = 0; tl < 2; ++tl) {
                        // ---- O_tl += P_tl V of the previous K/V tile
                        if (jt > 0 && jt - 1 < nk[tl]) {
                            const int jp = jt - 1;
                            const uint32_t pn = kv_it + jp;
                            const int pst = pn % kPfStages;
                            // tile B reads the V tile that tile A has just waited for
                            // when both attend it
                            const bool first_reader = tl == 0 || jp >= nk[0];
                            if (!pf_wait(&bars.p_full[tl], p_cnt[tl] & 1, abort_flag) ||
                                (first_reader &&
                                 !pf_wait(&bars.v_full[pst], (pn / kPfStages) & 1, abort_flag))) {
                                ok = false;
                                break;
                            }
                            ++p_cnt[tl];
                            const int nvalid = kv_hi - (kv_lo + jp * kBN);
                            if (jp == n - 1 && nvalid < kBN && first_reader) {
                                // rows past the last key may hold anything (or nothing
                                // was loaded there): zero them once, before the first
                                // PV that reads this tile, so that P = 0 meets finite V
                                uint8_t *vt = smem + Cfg::kVOff + pst * Cfg::kTileBytes;
                                for (int hf = 0; hf < Cfg::kHalves; ++hf) {
                                    uint4 *zb = reinterpret_cast<uint4 *>(
                                        vt + hf * Cfg::kHalfBytes + nvalid * 128);
                                    const int n16 = (kBN - nvalid) * 8;
                                    for (int i = lane; i < n16; i += 32)
                                        zb[i] = make_uint4(0, 0, 0, 0);
                                }
                                fence_proxy_async_smem();
                                __syncwarp();
                            }
                            if (jp == 0 && item_cnt[tl] > 0 &&
                                !pf_wait(&bars.o_free[tl], (item_cnt[tl] - 1) & 1, abort_flag)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            const uint32_t v_lo = v_lo0 + pst * kTileStep;
                            const uint32_t tO_ = 256 + tl * D;
                            const uint32_t tP_ = tl * 128;
                            const uint32_t acc0 = jp > 0 ? 1u : 0u;
                            const bool last_v = tl == (jp < nk[1] ? 1 : 0);
                            if (elect_one()) {
                                mma_ts(tO_, tP_, v_lo, Cfg::kIdescPV, acc0);
#pragma unroll
                                for (int k = 1; k < kBN / 16; ++k)
                                    mma_ts(tO_, tP_ + k * 8, v_lo + uint32_t(k * 2048 >> 4),
                                           Cfg::kIdescPV, 1u);
                                mma_commit(&bars.o_done[tl]);
                                if (last_v)
                                    mma_commit(&bars.v_empty[pst]);  // last reader of V(jp)
                            }
                            __syncwarp();
                        }
                        // ---- S_tl = Q_tl K^T of this K/V tile
                        if (jt < nk[tl]) {
                            const uint32_t k_lo = k_lo0 + st * kTileStep;
                            const uint32_t tS_ = tl * 128;
                            const uint32_t q_lo = q_lo0 + tl * kTileStep;
                            const bool last_k = tl == (jt < nk[1] ? 1 : 0);
                            if (elect_one()) {
#pragma unroll
                                for (int k = 0; k < D / 16; ++k) {
                                    const uint32_t off =
                                        ((k >> 2) * Cfg::kHalfBytes + (k & 3) * 32) >> 4;
                                    mma_ss(tS_, q_lo + off, k_lo + off, Cfg::kIdescS,
                                           k > 0 ? 1u : 0u);
                                }
                                mma_commit(&bars.s_full[tl]);
                                if (last_k)
                                    mma_commit(&bars.k_empty[st]);  // last reader of K(jt)
                            }
                            __syncwarp();
                        }
                    }
                    if (!ok)
                        break;
                    if (jt == n - 1 && elect_one())
                        mma_commit(bars.q_empty);  // Q is free once the last S is done
                    __syncwarp();
                }
                if (!ok)
                    break;
#pragma unroll
                for (int tl = 0; tl < 2; ++tl)
                    if (nk[tl] > 0)
                        ++item_cnt[tl];
                kv_it += n;
                ++li;
            }
            if (elect_one()) {
                // the issuing lane's commit fires once every MMA it issued has finished
                mma_commit(bars.drain);
                mbar_wait(bars.drain, 0);
            }
            __syncwarp();
        }
    } else {
        reg_alloc<kPfRegsHigh>();
        const int tl = (warp - 4) / 4;  // warps 4-7: tile A, warps 8-11: tile B
        pf_softmax<D>(p, prefix, nseq, bars, tl, tbase + tl * 128, tbase + 256 + tl * D,
                      abort_flag);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 2)
        tmem_dealloc(tbase, kTmemCols);
    // Beside a decode (this pass is its programmatic dependent, started on the
    // SMs the decode left free): the grid completes only after the decode's,
    // so that the launches after it see both passes' rows.
    if (p.after_decode)
        asm volatile("griddepcontrol.wait;" ::: "memory");
}

// --------------------------------------------------------------------- host
template <int D, bool kHnd>
static cudaError_t launch_prefill_d(const Fwd &f, const PrefillParams &p, int grid)
{
    using Cfg = PfCfg<D>;
    // devices (bit d for device d < 64) on which this instantiation's launch
    // attributes are set; atomic, since several host threads may launch
    static std::atomic<uint64_t> configured{0};
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t dev_bit = (dev >= 0 && dev < 64) ? (uint64_t(1) << dev) : 0;
    if (dev_bit == 0 || (configured.load(std::memory_order_acquire) & dev_bit) == 0) {
        cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<D, kHnd>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(Cfg::kSmemBytes));
        if (e != cudaSuccess)
            return e;
        cudaFuncAttributes attr;
        e = cudaFuncGetAttributes(&attr, prefill_tc_kernel<D, kHnd>);
        if (e != cudaSuccess)
            return e;
        if (uint32_t(attr.numRegs) * kPfThreads < kPfRegsSplit)
            return cudaErrorInvalidConfiguration;  // the register split would never be granted
        configured.fetch_or(dev_bit, std::memory_order_release);
    }
    CUtensorMap q_map, kv_map;
    if (encode_3d_bf16(&q_map, f.query, D, f.num_heads, f.num_tokens, uint64_t(D) * 2,
                       uint64_t(f.num_heads) * D * 2, 64, 1, kBM) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    if (encode_kv_map(&kv_map, f.kv_cache, D, f.num_kv_heads, f.block_size, f.num_blocks,
                      f.kv_hnd, uint32_t(p.box_rows)) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    count_launch();
    // the step's key and value rows as (dim, head, token), one box of 128
    // tokens per 64-dim half (unused unless p.new_from_input)
    CUtensorMap kin_map = kv_map, vin_map = kv_map;
    if (p.new_from_input) {
        const uint64_t row = uint64_t(D) * 2;
        if (encode_3d_bf16(&kin_map, f.new_key, D, f.num_kv_heads, f.num_tokens, row,
                           row * f.num_kv_heads, 64, 1, kBN) != CUDA_SUCCESS ||
            encode_3d_bf16(&vin_map, f.new_value, D, f.num_kv_heads, f.num_tokens, row,
                           row * f.num_kv_heads, 64, 1, kBN) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kPfThreads);
    cfg.dynamicSmemBytes = Cfg::kSmemBytes;
    cfg.stream = f.stream;
    if (p.after_decode || p.after_copy) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, prefill_tc_kernel<D, kHnd>, q_map, kv_map, kin_map, vin_map,
                              p);
}

cudaError_t launch_prefill(const Fwd &f, const PrefillPass &pass)
{
    const int nseq = f.num_seqs - f.num_decodes;
    if (!pass.shared_prefix && nseq <= 0)
        return cudaSuccess;
    PrefillParams p;
    p.qsl = f.qsl;
    p.seq_lens = f.seq_lens;
    p.block_table = f.block_table;
    p.bt_stride = f.bt_stride;
    p.first_seq = f.num_decodes;
    p.num_seqs = f.num_seqs;
    p.num_tokens = f.num_tokens;
    p.num_heads = f.num_heads;
    p.group = f.num_heads / f.num_kv_heads;
    p.block_size = f.block_size;
    // boxes never straddle a block: key offsets are multiples of block_size,
    // of 128 (tile) and of the first key kv_lo (a cascade suffix starts at the
    // prefix length, a multiple of the pool's block size, which a re-blocked
    // copy of 128-key blocks need not share), so use their gcd
    p.box_rows = std::gcd(std::gcd(f.block_size, 128), pass.kv_lo);
    p.num_blocks = static_cast<int32_t>(f.num_blocks);
    p.num_kv_heads = f.num_kv_heads;
    p.kv_lo = pass.kv_lo;
    p.kv_cap = pass.kv_cap;
    p.causal = pass.causal;
    p.scale_log2 = f.scale * 1.4426950408889634f;
    p.out_scale = f.out_scale;
    p.partial = pass.o_part != nullptr ? 1 : 0;
    p.token_base = pass.token_base;
    p.shared_prefix = pass.shared_prefix ? 1 : 0;
    p.out = static_cast<__nv_bfloat16 *>(f.out);
    p.lse = f.lse;
    p.o_part = pass.o_part;
    p.lse_part = pass.lse_part;
    p.item_counter = pass.item_counter;
    p.kv_splits = 1;
    p.split_tiles = 0;
    p.test_skip_copies = f.test_skip_copies;
    p.trigger_dependents = pass.trigger_dependents ? 1 : 0;
    p.new_from_input = pass.new_from_input && !pass.shared_prefix && f.new_key && f.new_value ? 1 : 0;
    p.after_decode = pass.after_decode ? 1 : 0;
    p.after_copy = pass.after_copy ? 1 : 0;
    if (pass.shared_prefix) {
        const int tiles = (pass.kv_cap - pass.kv_lo + kBN - 1) / kBN;
        p.kv_splits = std::max(1, pass.kv_splits);
        p.split_tiles = (tiles + p.kv_splits - 1) / p.kv_splits;
    }
    if (!pass.counter_zeroed)
        if (cudaError_t e = cudaMemsetAsync(p.item_counter, 0, sizeof(int32_t), f.stream))
            return e;
    int64_t items;
    if (pass.shared_prefix)
        items = int64_t((f.num_tokens + kSuper - 1) / kSuper) * f.num_heads * p.kv_splits;
    else
        items = (int64_t(f.num_tokens - f.num_decodes) + int64_t(nseq) * (kSuper - 1)) /
                kSuper * f.num_heads;
    // persistent grid: one CTA per SM (or the pass's share of the SMs), but no
    // more CTAs than work items
    const int ctas = pass.max_ctas > 0 ? std::min(pass.max_ctas, f.num_sms) : f.num_sms;
    const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(ctas, items)));
    if (f.head_size == 128)
        return f.kv_hnd ? launch_prefill_d<128, true>(f, p, grid)
                        : launch_prefill_d<128, false>(f, p, grid);
    return f.kv_hnd ? launch_prefill_d<64, true>(f, p, grid) : launch_prefill_d<64, false>(f, p, grid);
}

uint32_t prefill_take_error() { return take_device_error(); }

}  // namespace pka
