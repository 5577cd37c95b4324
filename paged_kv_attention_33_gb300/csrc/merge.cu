// merge.cu -- cascade_merge: log-sum-exp merge of two partial attentions.
//
// The blog post "El especialista del plato estrella" ("Que aporta FlashInfer:
// JIT y cascade attention") computes attention over a shared prefix once and
// combines it with each request's own suffix; the "FlashAttention y
// FlashInfer" page ("Limites y fallos") names the same softmax combine across
// shards, and the "AttentionBackend" page ("Limites y fallos") requires the
// lse base to be known -- here the natural log.  Per row:
//     lse = ln(e^lse_a + e^lse_b),  out = e^(lse_a-lse) out_a + e^(lse_b-lse) out_b.
// One warp per (token, head) row, 16-byte vectors along head_size.
// An lse of +inf or NaN is no partial attention at all (a corrupt input, say
// from a remote rank): the row is still computed, and the kernel raises the
// sticky device error (pka_check_status reports it) instead of letting the
// NaN pass unnoticed.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace pka {

__global__ void __launch_bounds__(256)
    cascade_merge_kernel(const uint4 *out_a, const float *lse_a, const uint4 *out_b,
                         const float *lse_b, uint4 *out, float *lse_out, int64_t rows,
                         int32_t vecs_per_row)
{
    const int64_t r = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (r >= rows)
        return;
    const float la = lse_a[r], lb = lse_b[r];
    // -inf (an empty side) and finite values pass; +inf and NaN do not
    if (lane == 0 && !(la < INFINITY && lb < INFINITY))
        flag_error(kErrBadPartial);
    const float m = fmaxf(la, lb);
    float ca = 0.f, cb = 0.f, l = -INFINITY;
    if (m != -INFINITY) {
        const float wa = expf(la - m), wb = expf(lb - m);
        l = m + logf(wa + wb);
        ca = expf(la - l);
        cb = expf(lb - l);
    }
    for (int v = lane; v < vecs_per_row; v += 32) {
        const int64_t i = r * vecs_per_row + v;
        const uint4 a = out_a[i], b = out_b[i];
        const __nv_bfloat162 *pa = reinterpret_cast<const __nv_bfloat162 *>(&a);
        const __nv_bfloat162 *pb = reinterpret_cast<const __nv_bfloat162 *>(&b);
        uint4 res;
        __nv_bfloat162 *pr = reinterpret_cast<__nv_bfloat162 *>(&res);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 fa = __bfloat1622float2(pa[e]);
            const float2 fb = __bfloat1622float2(pb[e]);
            // an empty side (weight 0) contributes nothing, whatever it holds
            const float x = (ca != 0.f ? ca * fa.x : 0.f) + (cb != 0.f ? cb * fb.x : 0.f);
            const float y = (ca != 0.f ? ca * fa.y : 0.f) + (cb != 0.f ? cb * fb.y : 0.f);
            pr[e] = __floats2bfloat162_rn(x, y);
        }
        out[i] = res;
    }
    __syncwarp();
    if (lane == 0 && lse_out)
        lse_out[r] = l;
}

// N-way merge (the combine of a decode context-parallel step: every rank's
// partial over its shard of the keys).  Base-b log-sum-exp, b = e or 2 (the
// "AttentionBackend" page, "Limites y fallos": the combine must use the base
// the partials were made in).  One warp per row, 16-byte vectors along
// head_size; a part with lse = -inf holds no keys and adds nothing.
__global__ void __launch_bounds__(256)
    merge_partials_kernel(const uint4 *outs, const float *lses, int32_t num_parts,
                          uint4 *out, float *lse_out, int64_t rows, int32_t vecs_per_row,
                          int32_t base2)
{
    const int64_t r = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (r >= rows)
        return;
    // b^x as e^(x ln b): exact scaling of the exponent for b = 2
    const float ln_b = base2 ? 0.69314718055994530942f : 1.f;
    float m = -INFINITY;
    bool bad = false;
    for (int q = 0; q < num_parts; ++q) {
        const float l = lses[int64_t(q) * rows + r];
        bad = bad || !(l < INFINITY);  // +inf or NaN
        m = fmaxf(m, l);
    }
    if (lane == 0 && bad)
        flag_error(kErrBadPartial);
    float wsum = 0.f;
    if (m != -INFINITY)
        for (int q = 0; q < num_parts; ++q) {
            const float l = lses[int64_t(q) * rows + r];
            wsum += l == -INFINITY ? 0.f : expf((l - m) * ln_b);
        }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    for (int v = lane; v < vecs_per_row; v += 32) {
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (m != -INFINITY)
            for (int q = 0; q < num_parts; ++q) {
                const float l = lses[int64_t(q) * rows + r];
                if (l == -INFINITY)
                    continue;  // warp-uniform: the whole row shares l
                const float w = expf((l - m) * ln_b) * inv;
                const uint4 a = outs[(int64_t(q) * rows + r) * vecs_per_row + v];
                const __nv_bfloat162 *pa = reinterpret_cast<const __nv_bfloat162 *>(&a);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = __bfloat1622float2(pa[e]);
                    acc[2 * e] += w * f.x;
                    acc[2 * e + 1] += w * f.y;
                }
            }
        uint4 res;
        __nv_bfloat162 *pr = reinterpret_cast<__nv_bfloat162 *>(&res);
#pragma unroll
        for (int e = 0; e < 4; ++e)
            pr[e] = __floats2bfloat162_rn(acc[2 * e], acc[2 * e + 1]);
        out[r * vecs_per_row + v] = res;
    }
    if (lane == 0 && lse_out)
        lse_out[r] = wsum > 0.f ? m + logf(wsum) / ln_b : -INFINITY;
}

cudaError_t launch_merge_partials(const void *outs, const float *lses, int32_t num_parts,
                                  void *out, float *lse_out, int32_t num_tokens,
                                  int32_t num_heads, int32_t head_size, int32_t base2,
                                  cudaStream_t st)
{
    const int64_t rows = int64_t(num_tokens) * num_heads;
    if (rows == 0)
        return cudaSuccess;
    const unsigned grid = static_cast<unsigned>((rows * 32 + 255) / 256);
    count_launch();
    merge_partials_kernel<<<grid, 256, 0, st>>>(static_cast<const uint4 *>(outs), lses,
                                                num_parts, static_cast<uint4 *>(out), lse_out,
                                                rows, head_size * 2 / 16, base2);
    return cudaGetLastError();
}

cudaError_t launch_cascade_merge(const void *out_a, const float *lse_a, const void *out_b,
                                 const float *lse_b, void *out, float *lse_out,
                                 int32_t num_tokens, int32_t num_heads, int32_t head_size,
                                 cudaStream_t st)
{
    const int64_t rows = int64_t(num_tokens) * num_heads;
    if (rows == 0)
        return cudaSuccess;
    const unsigned grid = static_cast<unsigned>((rows * 32 + 255) / 256);
    count_launch();
    cascade_merge_kernel<<<grid, 256, 0, st>>>(
        static_cast<const uint4 *>(out_a), lse_a, static_cast<const uint4 *>(out_b), lse_b,
        static_cast<uint4 *>(out), lse_out, rows, head_size * 2 / 16);
    return cudaGetLastError();
}

uint32_t merge_take_error() { return take_device_error(); }

}  // namespace pka
