// pkv_chunk_attn_bwd_noalloc: the chunk backward without any allocation.
//
// pkv_chunk_attn_bwd keeps its per-row statistics D = rowsum(dO * O) in a
// pool-owned scratch buffer that it grows with cudaMalloc when a larger chunk
// arrives. Some callers cannot let the library allocate at call time: code
// running under a strict memory budget or a caching allocator that owns all
// device memory, callers that must not synchronize the device (cudaMalloc
// and cudaFree can), and real-time loops that forbid allocation after
// start-up. This variant keeps the same scratch in a fixed file-scope
// __device__ array instead, so a call allocates nothing.
//
// Limits and sharing:
//   - the array holds kNoAllocMaxFloats floats (1 MiB); a call needs
//     n_q_heads * n_q of them, plus, with a page selection, a page list of at
//     most 1 + min(key pages, n_qp * n_kv_heads * kmax) entries, and is
//     rejected (PKV_ERR_INVALID) above that;
//   - every device that loads the library holds the array until exit;
//   - all calls share the one array: calls that overlap on the GPU (other
//     streams, other threads) race on it and must be serialised by the caller;
//   - each call rewrites the part it reads before reading it, so nothing has to
//     start at zero and leftovers from an earlier call do no harm.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "internal.h"

namespace pkv {
namespace {

constexpr size_t kNoAllocMaxFloats = size_t(1) << 18;   // 262144 floats = 1 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) float g_noalloc_scratch[kNoAllocMaxFloats];

// Device address of g_noalloc_scratch per device, taken once with that device
// current. In host code the symbol itself is only a host-side handle.
float* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

pkv_status scratch_for_current_device(float** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "pkv_chunk_attn_bwd_noalloc: cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices)
        return fail(PKV_ERR_INVALID, "pkv_chunk_attn_bwd_noalloc: device index out of range");
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess || !ptr)
            return cuda_fail(e != cudaSuccess ? e : cudaErrorInvalidSymbol,
                             "pkv_chunk_attn_bwd_noalloc: cudaGetSymbolAddress");
        g_scratch_addr[dev] = static_cast<float*>(ptr);
    }
    *out = g_scratch_addr[dev];
    return PKV_OK;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" pkv_status pkv_chunk_attn_bwd_noalloc(pkv_seq* s, const void* q, const void* o,
                                                 const void* dout, const float* lse,
                                                 int64_t q_start, int64_t n_q, void* dq,
                                                 const pkv_sel* sel, void* stream) {
    static const char* who = "pkv_chunk_attn_bwd_noalloc";
    // The same argument checks, pools, tables and dispatch as pkv_chunk_attn_bwd;
    // only the scratch differs.
    AttnArgs a;
    pkv_status st = attn_common(s, q, q_start, n_q, sel, &a, who);
    if (st != PKV_OK) return st;
    if (!o || !dout || !lse || !dq)
        return fail(PKV_ERR_INVALID, std::string(who) + ": o, dout, lse or dq is NULL");
    const size_t n_d = (size_t)a.Hq * (size_t)n_q;
    const size_t n_list = sel ? 1 + (size_t)bwd_pagelist_cap(a) : 0;
    const size_t n_mask = sel ? 1 + 2 * (size_t)bwd_selmask_words(a) : 0;
    const size_t need = n_d + n_list;
    if (need > kNoAllocMaxFloats)
        return fail(PKV_ERR_INVALID,
                    std::string(who) + ": n_q_heads * n_q" + (sel ? " + the page list" : "") +
                        " = " + std::to_string(need) + " exceeds the fixed scratch of " +
                        std::to_string(kNoAllocMaxFloats) +
                        " floats; use pkv_chunk_attn_bwd or a smaller chunk");
    float* scratch = nullptr;
    st = scratch_for_current_device(&scratch);
    if (st != PKV_OK) return st;
    a.o_in = o; a.dout = dout; a.lse_in = lse; a.dq = dq; a.Dbuf = scratch;
    a.pagelist = sel ? reinterpret_cast<int32_t*>(scratch + n_d) : nullptr;
    // The query-page masks when they fit too; otherwise the dK/dV kernel finds
    // each page's query pages by scanning the selection (the same lists).
    a.selmask = sel && need + n_mask <= kNoAllocMaxFloats
                    ? reinterpret_cast<uint64_t*>(
                          (reinterpret_cast<uintptr_t>(scratch + n_d + n_list) + 7) & ~uintptr_t(7))
                    : nullptr;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    // D = rowsum(dO * O): computed inside the tensor-core backward, by its own
    // kernel before the CUDA-core one.
    cudaError_t e;
    if (use_tc(s->pool, a)) {
        e = launch_attn_bwd_tc(a, cs);
    } else {
        e = launch_bwd_rowdot(a, cs);
        if (e == cudaSuccess) e = launch_attn_bwd_simt(a, cs);
    }
    // Staging on a side stream (pkv_prefetch, pkv_writeback_grads) orders itself
    // after this event: the slots this call reads and adds into stay untouched
    // until it has finished.
    if (e == cudaSuccess && s->used) e = cudaEventRecord(s->used, cs);
    if (e != cudaSuccess) return cuda_fail(e, "pkv_chunk_attn_bwd_noalloc: launch");
    return PKV_OK;
}
