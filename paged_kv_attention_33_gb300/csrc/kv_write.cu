// kv_write.cu -- reshape_and_cache: scatter this step's K/V rows into the
// paged pool through slot_mapping.
//
// Pool layout [num_blocks, 2, block_size, num_kv_heads, head_size] (the
// "FlashAttention y FlashInfer" page, "Flujo de datos", get_kv_cache_shape):
// in NHD order the K row of slot (b, o) for all kv heads is one contiguous run
// of num_kv_heads*head_size bf16 at ((b*2 + 0)*block_size + o), the V row the
// same run at kv index 1; in HND order (the same page, "Resumen en una
// frase": the two layouts) head k's row is at ((b*2 + kv)*num_kv_heads + k) *
// block_size + o.  One warp moves one token: it loads the K and V rows with
// 16-byte non-coherent loads and stores them with 16-byte stores, one head's
// head_size*2 bytes at a time in HND.  The work is a pure copy (bit exact);
// HBM traffic is 2 x (read + write) of a row.
#include "common.cuh"
#include "internal.h"

namespace pka {

constexpr int kKvwThreads = 256;
constexpr int kKvwUnroll = 4;

__global__ void __launch_bounds__(kKvwThreads)
    reshape_and_cache_kernel(const uint4 *__restrict__ key, const uint4 *__restrict__ value,
                             uint4 *__restrict__ cache, const int64_t *__restrict__ slots,
                             int32_t num_tokens, int32_t row_vecs, int32_t head_vecs,
                             int32_t num_kv_heads, int32_t block_size, int64_t num_blocks,
                             int32_t hnd)
{
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * kKvwThreads + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (warp >= num_tokens)
        return;
    const int64_t slot = slots[warp];
    if (slot < 0)
        return;  // padding token
    if (slot >= num_blocks * block_size) {
        if (lane == 0)
            flag_error(kErrSlotOutOfPool);
        return;
    }
    const int64_t blk = slot / block_size;
    const int64_t off = slot - blk * block_size;
    // 16-byte chunk i of the token's row (head i / head_vecs) in the pool
    auto dst = [&](int kv, int i) -> uint4 * {
        if (!hnd)
            return cache + ((blk * 2 + kv) * block_size + off) * row_vecs + i;
        const int h = i / head_vecs;
        return cache + (((blk * 2 + kv) * num_kv_heads + h) * block_size + off) * head_vecs +
               (i - h * head_vecs);
    };
    const uint4 *ks = key + warp * row_vecs;
    const uint4 *vs = value + warp * row_vecs;
    for (int base = 0; base < row_vecs; base += 32 * kKvwUnroll) {
        uint4 kr[kKvwUnroll], vr[kKvwUnroll];
#pragma unroll
        for (int u = 0; u < kKvwUnroll; ++u) {
            const int i = base + u * 32 + lane;
            if (i < row_vecs) {
                kr[u] = __ldg(ks + i);
                vr[u] = __ldg(vs + i);
            }
        }
#pragma unroll
        for (int u = 0; u < kKvwUnroll; ++u) {
            const int i = base + u * 32 + lane;
            if (i < row_vecs) {
                *dst(0, i) = kr[u];
                *dst(1, i) = vr[u];
            }
        }
    }
}

// The same scatter into an fp8 e4m3 pool: every element is stored as
// e4m3(x / scale) (k_scale for K, v_scale for V; the quantisation of the
// "FlashAttention y FlashInfer" page's fp8 KV cache, per-tensor scale).  A
// lane moves one 16-element chunk: two 16-byte bf16 loads in, one 16-byte
// store of codes out.  HBM traffic is 2 x (2 + 1) bytes per element.
__global__ void __launch_bounds__(kKvwThreads)
    reshape_and_cache_fp8_kernel(const uint4 *__restrict__ key, const uint4 *__restrict__ value,
                                 uint4 *__restrict__ cache, const int64_t *__restrict__ slots,
                                 int32_t num_tokens, int32_t row_chunks, int32_t head_chunks,
                                 int32_t num_kv_heads, int32_t block_size, int64_t num_blocks,
                                 int32_t hnd, float k_scale, float v_scale)
{
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * kKvwThreads + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (warp >= num_tokens)
        return;
    const int64_t slot = slots[warp];
    if (slot < 0)
        return;
    if (slot >= num_blocks * block_size) {
        if (lane == 0)
            flag_error(kErrSlotOutOfPool);
        return;
    }
    const int64_t blk = slot / block_size;
    const int64_t off = slot - blk * block_size;
    auto dst = [&](int kv, int i) -> uint4 * {
        if (!hnd)
            return cache + ((blk * 2 + kv) * block_size + off) * row_chunks + i;
        const int h = i / head_chunks;
        return cache + (((blk * 2 + kv) * num_kv_heads + h) * block_size + off) * head_chunks +
               (i - h * head_chunks);
    };
    const uint4 *ks = key + warp * row_chunks * 2;
    const uint4 *vs = value + warp * row_chunks * 2;
    for (int i = lane; i < row_chunks; i += 32) {
        const uint4 k0 = __ldg(ks + 2 * i), k1 = __ldg(ks + 2 * i + 1);
        const uint4 v0 = __ldg(vs + 2 * i), v1 = __ldg(vs + 2 * i + 1);
        const uint2 kl = quantize8_e4m3(k0, k_scale), kh = quantize8_e4m3(k1, k_scale);
        const uint2 vl = quantize8_e4m3(v0, v_scale), vh = quantize8_e4m3(v1, v_scale);
        *dst(0, i) = make_uint4(kl.x, kl.y, kh.x, kh.y);
        *dst(1, i) = make_uint4(vl.x, vl.y, vh.x, vh.y);
    }
}

cudaError_t launch_reshape_and_cache_fp8(const void *key, const void *value, void *cache,
                                         const int64_t *slots, int32_t num_tokens,
                                         int32_t num_kv_heads, int32_t head_size,
                                         int32_t block_size, int64_t num_blocks, int32_t hnd,
                                         float k_scale, float v_scale, cudaStream_t st)
{
    if (num_tokens == 0)
        return cudaSuccess;
    const int32_t head_chunks = head_size / 16;
    const int32_t row_chunks = num_kv_heads * head_chunks;
    const int64_t threads = static_cast<int64_t>(num_tokens) * 32;
    const unsigned grid = static_cast<unsigned>((threads + kKvwThreads - 1) / kKvwThreads);
    count_launch();
    reshape_and_cache_fp8_kernel<<<grid, kKvwThreads, 0, st>>>(
        static_cast<const uint4 *>(key), static_cast<const uint4 *>(value),
        static_cast<uint4 *>(cache), slots, num_tokens, row_chunks, head_chunks, num_kv_heads,
        block_size, num_blocks, hnd, k_scale, v_scale);
    return cudaGetLastError();
}

cudaError_t launch_reshape_and_cache(const void *key, const void *value, void *cache,
                                     const int64_t *slots, int32_t num_tokens,
                                     int32_t num_kv_heads, int32_t head_size,
                                     int32_t block_size, int64_t num_blocks, int32_t hnd,
                                     cudaStream_t st)
{
    if (num_tokens == 0)
        return cudaSuccess;
    const int32_t head_vecs = head_size * 2 / 16;
    const int32_t row_vecs = num_kv_heads * head_vecs;
    const int64_t threads = static_cast<int64_t>(num_tokens) * 32;
    const unsigned grid = static_cast<unsigned>((threads + kKvwThreads - 1) / kKvwThreads);
    count_launch();
    reshape_and_cache_kernel<<<grid, kKvwThreads, 0, st>>>(
        static_cast<const uint4 *>(key), static_cast<const uint4 *>(value),
        static_cast<uint4 *>(cache), slots, num_tokens, row_vecs, head_vecs, num_kv_heads,
        block_size, num_blocks, hnd);
    return cudaGetLastError();
}

// CTAs per copied block (a shared prefix of a few large blocks is copied by
// more CTAs than it has blocks).
constexpr int kDequantSplit = 8;

// Blocks of an fp8 pool as bf16 code values (no scale: every e4m3 value is
// exact in bf16; the attention applies k_scale and v_scale) in a dense NHD
// scratch pool: the kDequantSplit CTAs (p, n*kDequantSplit + part) take block
// column n of block-table row s = first_row + p, copy (each a part of its
// chunks) pool block bt[s][n] to scratch block dst_base + p*row_blocks + n, and
// part 0 writes that id into the scratch table at [s][n] (row stride
// table_stride).  Columns at or past min(ceil(L_s / bs), col_limit) are
// left alone (the attention never reads them).  With `trigger` the launch after
// it (its programmatic dependent, which waits for this grid before it reads the
// copy) may start at once.
__global__ void __launch_bounds__(kKvwThreads)
    dequant_blocks_kernel(const uint4 *__restrict__ pool, uint4 *__restrict__ scratch,
                          int32_t *__restrict__ table, const int32_t *__restrict__ bt,
                          int32_t bt_stride, const int32_t *__restrict__ seq_lens,
                          int32_t first_row, int32_t row_blocks, int32_t col_limit,
                          int64_t dst_base, int32_t table_stride, int32_t block_size,
                          int32_t num_kv_heads, int32_t head_chunks, int64_t num_blocks,
                          int32_t hnd, int32_t trigger)
{
    if (trigger)
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // block n of row p, part `part` of its kDequantSplit slices of chunks
    const int32_t p = blockIdx.y, n = blockIdx.x / kDequantSplit, part = blockIdx.x % kDequantSplit;
    const int32_t s = first_row + p;
    const int32_t L = seq_lens[s];
    if (blockIdx.x == 0 && threadIdx.x == 0 && col_limit == row_blocks &&
        int64_t(L) > int64_t(row_blocks) * block_size)
        flag_error(kErrBadMetadata);  // longer than max_seq_len: its tail was not copied
    if (n >= col_limit || n * block_size >= L)
        return;
    const int64_t dst_blk = dst_base + int64_t(p) * row_blocks + n;
    if (part == 0 && threadIdx.x == 0)
        table[int64_t(s) * table_stride + n] = static_cast<int32_t>(dst_blk);
    const int32_t src_blk = bt[int64_t(s) * bt_stride + n];
    if (src_blk < 0 || src_blk >= num_blocks) {
        if (part == 0 && threadIdx.x == 0)
            flag_error(kErrBlockOutOfPool);
        return;
    }
    // 16-code chunk i of the block in NHD order: (kv, offset, head, chunk)
    const int32_t per_kv = block_size * num_kv_heads * head_chunks;
    for (int32_t i = part * kKvwThreads + threadIdx.x; i < 2 * per_kv;
         i += kDequantSplit * kKvwThreads) {
        const int32_t kv = i / per_kv, r = i % per_kv;
        const int32_t off = r / (num_kv_heads * head_chunks);
        const int32_t h = (r / head_chunks) % num_kv_heads, c = r % head_chunks;
        const int64_t src = hnd ? (((int64_t(src_blk) * 2 + kv) * num_kv_heads + h) * block_size +
                                   off) * head_chunks + c
                                : (int64_t(src_blk) * 2 * per_kv + i);
        const uint4 codes = pool[src];
        const uint32_t w[4] = {codes.x, codes.y, codes.z, codes.w};
        uint32_t o[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t lo, hi;  // f16 pairs of bytes (0, 1) and (2, 3)
            e4m3x4_to_f16x2x2(w[j], lo, hi);
            const __half2 a = *reinterpret_cast<const __half2 *>(&lo);
            const __half2 b = *reinterpret_cast<const __half2 *>(&hi);
            o[2 * j] = pack_bf16x2(__low2float(a), __high2float(a));
            o[2 * j + 1] = pack_bf16x2(__low2float(b), __high2float(b));
        }
        uint4 *d = scratch + (dst_blk * 2 * per_kv + i) * 2;
        d[0] = make_uint4(o[0], o[1], o[2], o[3]);
        d[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
}

cudaError_t launch_dequant_blocks(const Fwd &f, void *scratch, int32_t *table, int32_t first_row,
                                  int32_t num_rows, int32_t row_blocks, int32_t col_limit,
                                  int64_t dst_base, int32_t table_stride, bool dependent_follows)
{
    if (num_rows <= 0 || col_limit <= 0)
        return cudaSuccess;
    count_launch();
    dim3 grid(static_cast<unsigned>(col_limit * kDequantSplit), static_cast<unsigned>(num_rows));
    dequant_blocks_kernel<<<grid, kKvwThreads, 0, f.stream>>>(
        static_cast<const uint4 *>(f.kv_cache), static_cast<uint4 *>(scratch), table,
        f.block_table, f.bt_stride, f.seq_lens, first_row, row_blocks, col_limit, dst_base,
        table_stride, f.block_size, f.num_kv_heads, f.head_size / 16, f.num_blocks, f.kv_hnd,
        dependent_follows ? 1 : 0);
    return cudaGetLastError();
}

// Re-blocking of a bf16 pool with small pages for the tensor-core prefill.
// A prefill work item reads its K and V tiles (128 keys of one kv head) with
// one TMA box per page and 64-dim half; at 16-key pages that is 16 boxes of
// 2 KB per tile, and the tensor-core pass is then bound by how fast one SM
// issues boxes, not by its MMAs.  Copying the prefill sequences' keys into
// 128-key blocks first (2 x 140 MB of traffic for a 34K-token batch, against
// about a millisecond of MMAs) lets the pass read one box per tile half.
// One CTA per quarter (32 keys) of a 128-key destination block of one
// sequence: block-table row first_row + p, destination block dst_base +
// p * row_blocks + n (NHD, every kv head), its id stored at
// table[(first_row + p) * table_stride + n]; keys at and past L are not
// copied (the prefill pass never admits them).  With context_lo >= 0 (the
// pass reads every key tile that starts at or after the sequence's context
// ctx = L - q from the step's own rows) only the blocks that such a pass still
// reads here are copied: none when ctx <= context_lo (its first key), else
// those that start below ctx + 127.  A warp copies whole key rows (every
// head's K or V row of one key), lanes along the row.
constexpr int kReblockKeys = 128;
constexpr int kReblockSplit = 4;  // CTAs per destination block
constexpr int kReblockCtaKeys = kReblockKeys / kReblockSplit;

__global__ void __launch_bounds__(kKvwThreads)
    reblock_kernel(const uint4 *__restrict__ pool, uint4 *__restrict__ scratch,
                   int32_t *__restrict__ table, const int32_t *__restrict__ bt,
                   int32_t bt_stride, const int32_t *__restrict__ seq_lens,
                   const int32_t *__restrict__ qsl, int32_t context_lo, int32_t first_row,
                   int32_t row_blocks, int64_t dst_base, int32_t table_stride,
                   int32_t block_size, int32_t num_kv_heads, int32_t head_chunks,
                   int64_t num_blocks, int32_t hnd)
{
    __shared__ int32_t src_blk[kReblockCtaKeys];  // source block of each page (-1: none)
    const int32_t p = blockIdx.y;
    const int32_t n = blockIdx.x / kReblockSplit, quarter = blockIdx.x % kReblockSplit;
    const int32_t s = first_row + p;
    const int32_t L = seq_lens[s];
    if (blockIdx.x == 0 && threadIdx.x == 0 && int64_t(L) > int64_t(row_blocks) * kReblockKeys)
        flag_error(kErrBadMetadata);  // longer than max_seq_len: its tail was not copied
    const int32_t key0 = n * kReblockKeys + quarter * kReblockCtaKeys;  // first key copied
    if (n >= row_blocks || key0 >= L)
        return;
    if (context_lo >= 0) {
        const int32_t ctx = L - (qsl[s + 1] - qsl[s]);
        if (ctx <= context_lo || n * kReblockKeys >= ctx + kReblockKeys - 1)
            return;
    }
    const int32_t keys = min(kReblockCtaKeys, L - key0);
    const int64_t dst_blk = dst_base + int64_t(p) * row_blocks + n;
    if (quarter == 0 && threadIdx.x == 0)
        table[int64_t(s) * table_stride + n] = static_cast<int32_t>(dst_blk);
    const int32_t pages = (keys + block_size - 1) / block_size;  // block_size divides 32
    if (threadIdx.x < pages) {
        // (a column past the table is a length above max_seq_len: flagged too)
        const int32_t col = key0 / block_size + threadIdx.x;
        int32_t b = col < bt_stride ? bt[int64_t(s) * bt_stride + col] : -1;
        if (b < 0 || b >= num_blocks) {
            flag_error(kErrBlockOutOfPool);
            b = -1;
        }
        src_blk[threadIdx.x] = b;
    }
    __syncthreads();
    const int32_t row_chunks = num_kv_heads * head_chunks;  // 16-byte chunks of a key row
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int32_t r = warp; r < 2 * keys; r += kKvwThreads / 32) {
        const int32_t kv = r >= keys ? 1 : 0;
        const int32_t key = r - kv * keys;  // within this CTA's keys
        const int32_t b = src_blk[key / block_size];
        if (b < 0)
            continue;  // flagged above; the row is left as it was
        const int32_t off = (key0 + key) % block_size;
        uint4 *dst = scratch + ((dst_blk * 2 + kv) * kReblockKeys + quarter * kReblockCtaKeys +
                                key) * row_chunks;
        if (!hnd) {  // the row is contiguous in the pool too
            const uint4 *src = pool + ((int64_t(b) * 2 + kv) * block_size + off) * row_chunks;
#pragma unroll 4
            for (int32_t c = lane; c < row_chunks; c += 32)
                dst[c] = __ldcs(src + c);
        } else {  // one head's row at a time, block_size rows apart
            const uint4 *src = pool + (int64_t(b) * 2 + kv) * num_kv_heads * block_size * head_chunks +
                               int64_t(off) * head_chunks;
#pragma unroll 4
            for (int32_t c = lane; c < row_chunks; c += 32) {
                const int32_t h = c / head_chunks;
                dst[c] = __ldcs(src + (int64_t(h) * block_size * head_chunks + (c - h * head_chunks)));
            }
        }
    }
}

cudaError_t launch_reblock(const Fwd &f, void *scratch, int32_t *table, int32_t first_row,
                           int32_t num_rows, int32_t row_blocks, int64_t dst_base,
                           int32_t table_stride, int32_t context_lo)
{
    if (num_rows <= 0 || row_blocks <= 0)
        return cudaSuccess;
    if (kReblockCtaKeys % f.block_size != 0)
        return cudaErrorInvalidValue;
    count_launch();
    dim3 grid(static_cast<unsigned>(row_blocks * kReblockSplit), static_cast<unsigned>(num_rows));
    reblock_kernel<<<grid, kKvwThreads, 0, f.stream>>>(
        static_cast<const uint4 *>(f.kv_cache), static_cast<uint4 *>(scratch), table,
        f.block_table, f.bt_stride, f.seq_lens, f.qsl, context_lo, first_row, row_blocks, dst_base,
        table_stride, f.block_size, f.num_kv_heads, f.head_size * 2 / 16, f.num_blocks, f.kv_hnd);
    return cudaGetLastError();
}

uint32_t kv_write_take_error() { return take_device_error(); }

}  // namespace pka
