// noalloc.cu -- pka_paged_attn_forward_noalloc: the attention forward for
// callers that cannot allocate device memory.
//
// Some callers have no way to hand the library a workspace: a serving engine
// that reserved nearly all of HBM for its KV pool at start-up and keeps no
// allocator headroom, a plugin host that only passes input and output
// pointers, or a loop that must not call cudaMalloc because it can stall the
// whole device.  For them the split-KV partial results live in a buffer of
// fixed size that is part of the library's own device image
// (g_noalloc_scratch below): every GPU that loads the library holds it until
// the process exits, and no call here allocates or frees anything.
#include <mutex>

#include "internal.h"
#include "pka.h"

namespace pka {

// Capacity of the built-in scratch: split-KV and cascade partials (fp32).
constexpr size_t kNoallocScratchBytes = size_t(16) << 20;  // 16 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// The driver's cuCtxGetCurrent, found once through the runtime (the library
// does not link libcuda directly).
using CtxGetCurrentFn = CUresult (*)(CUcontext *);

static CtxGetCurrentFn ctx_get_current()
{
    static CtxGetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(p);
    });
    return fn;
}

// Device address of g_noalloc_scratch on the current device.  In host code
// the symbol's name stands for a host-side shadow, not for device memory, so
// the address is looked up once per device (with that device current) and
// cached together with the context it belongs to: when the device's context
// has been torn down and made again (cudaDeviceReset, a released and retained
// primary context), the context differs and the address is looked up anew.
static cudaError_t noalloc_scratch(void **out)
{
    static std::mutex mu;
    static void *ptrs[64] = {};
    static CUcontext ctxs[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= 64)
        return cudaErrorInvalidDevice;
    CtxGetCurrentFn get = ctx_get_current();
    auto current = [&]() -> CUcontext {
        CUcontext c = nullptr;
        return get && get(&c) == CUDA_SUCCESS ? c : nullptr;
    };
    std::lock_guard<std::mutex> lock(mu);
    const CUcontext ctx = current();
    if (!ptrs[dev] || !ctx || ctxs[dev] != ctx) {
        // (the lookup makes the runtime's context current if it was not yet;
        // a context that cannot be named is looked up on every call)
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess)
            return e;
        ptrs[dev] = p;
        ctxs[dev] = current();
    }
    *out = ptrs[dev];
    return cudaSuccess;
}

}  // namespace pka

extern "C" pka_status pka_paged_attn_forward_noalloc(
    const void *query, const void *kv_cache, const pka_meta *meta, void *out, float *lse,
    int32_t num_tokens, int32_t num_heads, int32_t num_kv_heads, int32_t head_size,
    int32_t block_size, int64_t num_blocks, float scale, int32_t causal, void *stream)
{
    // the smallest workspace the forward accepts (it leaves out optional
    // copies that do not fit)
    const size_t need = pka::workspace_size_min(meta, num_tokens, num_heads, num_kv_heads,
                                                head_size, block_size);
    if (need > pka::kNoallocScratchBytes) {
        pka::set_last_error("pka_paged_attn_forward_noalloc: this batch needs %zu bytes of "
                            "scratch, more than the %zu-byte built-in buffer; use "
                            "pka_paged_attn_forward with a workspace, or split the batch",
                            need, pka::kNoallocScratchBytes);
        return PKA_ERR_WORKSPACE;
    }
    void *scratch = nullptr;
    if (need > 0) {
        cudaError_t e = pka::noalloc_scratch(&scratch);
        if (e != cudaSuccess) {
            pka::set_last_error("pka_paged_attn_forward_noalloc: cudaGetSymbolAddress: %s",
                                cudaGetErrorString(e));
            return PKA_ERR_CUDA;
        }
    }
    // The forward zeroes the per-sequence counters it keeps in the scratch on
    // every call and writes the partial results in full before reading them,
    // so an earlier call's leftovers do no harm.
    return pka_paged_attn_forward(query, kv_cache, meta, out, lse, num_tokens, num_heads,
                                  num_kv_heads, head_size, block_size, num_blocks, scale, causal,
                                  scratch, need > 0 ? pka::kNoallocScratchBytes : 0, stream);
}
