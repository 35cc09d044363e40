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
//     n_q_heads * n_q of them and is rejected (PKV_ERR_INVALID) above that;
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
    if (!s || !q || !o || !dout || !lse || !dq)
        return fail(PKV_ERR_INVALID, std::string(who) + ": NULL argument");
    pkv_pool* p = s->pool;
    if (p->desc.residency == PKV_RES_META)
        return fail(PKV_ERR_INVALID, std::string(who) + ": META pool holds no data");
    const int64_t P = p->desc.page_size;
    if (n_q <= 0 || q_start < 0 || q_start % P != 0 || q_start + n_q > s->len)
        return fail(PKV_ERR_INVALID, std::string(who) +
                                         ": need q_start % P == 0 and q_start + n_q <= length");
    const size_t need = (size_t)p->desc.n_q_heads * (size_t)n_q;
    if (need > kNoAllocMaxFloats)
        return fail(PKV_ERR_INVALID,
                    std::string(who) + ": n_q_heads * n_q = " + std::to_string(need) +
                        " exceeds the fixed scratch of " + std::to_string(kNoAllocMaxFloats) +
                        " floats; use pkv_chunk_attn_bwd or a smaller chunk");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev != p->device)
        return fail(PKV_ERR_INVALID, std::string(who) + ": current device is not the pool's");
    float* scratch = nullptr;
    pkv_status st = scratch_for_current_device(&scratch);
    if (st != PKV_OK) return st;

    AttnArgs a{};
    a.P = (int)P; a.Hq = p->desc.n_q_heads; a.Hkv = p->desc.n_kv_heads;
    a.d = p->desc.head_dim; a.dtype = p->desc.dtype;
    a.q_start = q_start; a.n_q = n_q; a.q = q;
    if (p->desc.residency == PKV_RES_PINNED_HOST) {      // staged pages: read the slots
        a.kpool = p->kslot; a.vpool = p->vslot; a.dkpool = p->dkslot; a.dvpool = p->dvslot;
        a.bt = s->d_slot_of; a.num_phys = p->n_slots;
    } else {
        a.kpool = p->k; a.vpool = p->v; a.dkpool = p->dk; a.dvpool = p->dv;
        a.bt = s->d_bt; a.num_phys = p->desc.num_phys_pages;
    }
    a.err = p->d_err;
    a.tmap_k = p->tmaps_ready ? &p->tmap_k : nullptr;
    a.tmap_v = p->tmaps_ready ? &p->tmap_v : nullptr;
    if (sel) {
        if (!sel->pages || sel->kmax <= 0 || sel->n_qp != (n_q + P - 1) / P)
            return fail(PKV_ERR_INVALID, std::string(who) + ": selection does not match chunk");
        a.sel = sel->pages;
        a.kmax = sel->kmax;
    }
    a.o_in = o; a.dout = dout; a.lse_in = lse; a.dq = dq; a.Dbuf = scratch;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const bool tc = !(p->desc.flags & PKV_FLAG_SIMT_ONLY) && p->tmaps_ready && tc_supported(a);
    e = launch_bwd_rowdot(a, cs);
    if (e == cudaSuccess) e = tc ? launch_attn_bwd_tc(a, cs) : launch_attn_bwd_simt(a, cs);
    if (e != cudaSuccess) return cuda_fail(e, "pkv_chunk_attn_bwd_noalloc: launch");
    return PKV_OK;
}
