// Host-offload page streamer ("Out of the Memory Barrier", gist.science/de
// §2.C: the KV cache is moved asynchronously between GPU and CPU memory;
// gist.science/nl: pinned CPU memory and CUDA streams, the cache *and its
// gradients*; gist.science/ja §2.3).
//
// A PINNED_HOST pool keeps every K/V page and gradient page in mapped pinned
// host memory and owns n_slots page slots in HBM. Staging runs on a side
// stream, entirely in kernels (no per-page memcpy calls, no host sync):
//   plan      one CTA: dedupe the requested logical pages (flags), assign
//             slots in ascending page order (ordered compaction), fill the
//             logical-page -> slot table the attention kernels read;
//   copy      one CTA per (slot, KV head): copy the page's K and V (and, on
//             request, dK and dV) from host memory over NVLink-C2C / PCIe
//             into the slot with 16-byte loads;
//   writeback one CTA per (slot, KV head): copy the slot's dK and dV back
//             into the host gradient pages.
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"

namespace pkv {
namespace {

constexpr int kPlanThreads = 1024;
constexpr int kCopyThreads = 256;

// flags has n_pages entries; *count_out receives the number of staged slots.
__global__ void __launch_bounds__(kPlanThreads) stage_plan_kernel(const int32_t* pages, int64_t n,
        int64_t n_pages, int64_t n_slots, int32_t* flags, int32_t* slot_of, int32_t* slot_page,
        int32_t* count_out, int* err) {
    __shared__ int scan[kPlanThreads];
    const int tid = threadIdx.x;
    for (int64_t p = tid; p < n_pages; p += kPlanThreads) {
        flags[p] = pages ? 0 : 1;
        slot_of[p] = -1;
    }
    __syncthreads();
    if (pages) {
        for (int64_t i = tid; i < n; i += kPlanThreads) {
            const int32_t lp = pages[i];
            if (lp >= 0 && lp < n_pages) flags[lp] = 1;
        }
    }
    __syncthreads();
    const int64_t per = (n_pages + kPlanThreads - 1) / kPlanThreads;
    const int64_t p0 = (int64_t)tid * per, p1 = min64(n_pages, p0 + per);
    int cnt = 0;
    for (int64_t p = p0; p < p1; ++p) cnt += flags[p];
    scan[tid] = cnt;
    __syncthreads();
    for (int off = 1; off < kPlanThreads; off <<= 1) {
        const int v = tid >= off ? scan[tid - off] : 0;
        __syncthreads();
        scan[tid] += v;
        __syncthreads();
    }
    int rank = scan[tid] - cnt;
    for (int64_t p = p0; p < p1; ++p) {
        if (!flags[p]) continue;
        if (rank < n_slots) {
            slot_of[p] = rank;
            slot_page[rank] = (int32_t)p;
        } else {
            report_error(err, kErrSlots);
        }
        ++rank;
    }
    __syncthreads();
    if (tid == 0) *count_out = (int32_t)min64(scan[kPlanThreads - 1], n_slots);
}

__device__ __forceinline__ void copy16(void* dst, const void* src, size_t bytes) {
    const uint4* s = static_cast<const uint4*>(src);
    uint4* d = static_cast<uint4*>(dst);
    const size_t n = bytes / 16;
    for (size_t i = threadIdx.x; i < n; i += kCopyThreads) d[i] = s[i];
}

struct StageArgs {
    const int32_t* bt;           // logical -> physical (host pages)
    const int32_t* slot_page;    // slot -> logical
    const int32_t* count;        // number of staged slots (flags[n_pages])
    int64_t num_phys;
    int Hkv;
    size_t kv_bytes;             // one (page, head) tile of K or V
    size_t g_bytes;              // one (page, head) tile of dK or dV
    const uint8_t* k; const uint8_t* v; const uint8_t* dk; const uint8_t* dv;   // host pages
    uint8_t* ks; uint8_t* vs; uint8_t* dks; uint8_t* dvs;                       // slots
    int what;
    int* err;
};

__global__ void __launch_bounds__(kCopyThreads) stage_copy_kernel(StageArgs a) {
    const int s = blockIdx.x, h = blockIdx.y;
    if (s >= *a.count) return;
    const int32_t lp = a.slot_page[s];
    const int32_t pp = a.bt[lp];
    if (pp < 0 || pp >= a.num_phys) {
        if (threadIdx.x == 0) report_error(a.err, kErrBadPage);
        return;
    }
    const size_t src = (size_t)pp * a.Hkv + h, dst = (size_t)s * a.Hkv + h;
    if (a.what & PKV_STAGE_KV) {
        copy16(a.ks + dst * a.kv_bytes, a.k + src * a.kv_bytes, a.kv_bytes);
        copy16(a.vs + dst * a.kv_bytes, a.v + src * a.kv_bytes, a.kv_bytes);
    }
    if (a.what & PKV_STAGE_GRADS) {
        copy16(a.dks + dst * a.g_bytes, a.dk + src * a.g_bytes, a.g_bytes);
        copy16(a.dvs + dst * a.g_bytes, a.dv + src * a.g_bytes, a.g_bytes);
    }
}

__global__ void __launch_bounds__(kCopyThreads) stage_writeback_kernel(StageArgs a) {
    const int s = blockIdx.x, h = blockIdx.y;
    if (s >= *a.count) return;
    const int32_t lp = a.slot_page[s];
    const int32_t pp = a.bt[lp];
    if (pp < 0 || pp >= a.num_phys) {
        if (threadIdx.x == 0) report_error(a.err, kErrBadPage);
        return;
    }
    const size_t src = (size_t)s * a.Hkv + h, dst = (size_t)pp * a.Hkv + h;
    copy16(const_cast<uint8_t*>(a.dk) + dst * a.g_bytes, a.dks + src * a.g_bytes, a.g_bytes);
    copy16(const_cast<uint8_t*>(a.dv) + dst * a.g_bytes, a.dvs + src * a.g_bytes, a.g_bytes);
}

StageArgs stage_args(const pkv_seq* s, int what) {
    const pkv_pool* p = s->pool;
    StageArgs a{};
    a.bt = s->d_bt;
    a.slot_page = s->d_slot_page;
    a.count = s->d_flags + p->desc.num_phys_pages;
    a.num_phys = p->desc.num_phys_pages;
    a.Hkv = p->desc.n_kv_heads;
    a.kv_bytes = (size_t)p->desc.page_size * p->desc.head_dim * p->elem;
    a.g_bytes = (size_t)p->desc.page_size * p->desc.head_dim * sizeof(float);
    a.k = static_cast<const uint8_t*>(p->k); a.v = static_cast<const uint8_t*>(p->v);
    a.dk = reinterpret_cast<const uint8_t*>(p->dk); a.dv = reinterpret_cast<const uint8_t*>(p->dv);
    a.ks = static_cast<uint8_t*>(p->kslot); a.vs = static_cast<uint8_t*>(p->vslot);
    a.dks = reinterpret_cast<uint8_t*>(p->dkslot); a.dvs = reinterpret_cast<uint8_t*>(p->dvslot);
    a.what = what;
    a.err = p->d_err;
    return a;
}

}  // namespace

cudaError_t launch_stage_plan(const pkv_seq* s, const int32_t* pages, int64_t n, cudaStream_t st) {
    const pkv_pool* p = s->pool;
    // Planning covers the sequence's pages; the count goes to flags[num_phys_pages].
    const int64_t n_pages = (int64_t)s->bt.size();
    ProfScope ps("stage_plan_kernel", st);
    stage_plan_kernel<<<1, kPlanThreads, 0, st>>>(pages, n, n_pages, p->n_slots, s->d_flags,
                                                 s->d_slot_of, s->d_slot_page,
                                                 s->d_flags + p->desc.num_phys_pages, p->d_err);
    return cudaGetLastError();
}

cudaError_t launch_stage_copy(const pkv_seq* s, int what, cudaStream_t st) {
    const pkv_pool* p = s->pool;
    ProfScope ps("stage_copy_kernel", st);
    dim3 grid((unsigned)p->n_slots, p->desc.n_kv_heads);
    stage_copy_kernel<<<grid, kCopyThreads, 0, st>>>(stage_args(s, what));
    return cudaGetLastError();
}

cudaError_t launch_stage_writeback(const pkv_seq* s, cudaStream_t st) {
    const pkv_pool* p = s->pool;
    ProfScope ps("stage_writeback_kernel", st);
    dim3 grid((unsigned)p->n_slots, p->desc.n_kv_heads);
    stage_writeback_kernel<<<grid, kCopyThreads, 0, st>>>(stage_args(s, PKV_STAGE_GRADS));
    return cudaGetLastError();
}

}  // namespace pkv
