// Host-offload page streamer ("Out of the Memory Barrier", gist.science/de
// §2.C: the KV cache is moved asynchronously between GPU and CPU memory;
// gist.science/nl: pinned CPU memory and CUDA streams, the cache *and its
// gradients*; gist.science/ja §2.3).
//
// A PINNED_HOST pool keeps every K/V page and gradient page in mapped pinned
// host memory and owns n_slots page slots in HBM. A sequence's slots form a
// cache: a staged page keeps its slot across prefetches until another page
// needs the slot, so consecutive chunks, whose selections overlap heavily,
// move only the pages (and the contents) not already resident. Per slot the
// state word records what it holds:
//   KV     the page's keys and values;
//   G      the page's dK/dV (the slot is the authoritative copy while staged);
//   DIRTY  the gradients may differ from the host pages (set when gradients
//          are staged, since a backward call follows and adds into them);
//          written back on eviction, by pkv_writeback_grads and on release.
// Staging runs on a side stream, entirely in kernels (no per-page memcpy
// calls, no host sync):
//   plan      one CTA: dedupe the requested logical pages; resident pages keep
//             their slots and get only the missing contents; new pages take
//             empty slots first, then slots of pages not requested this time
//             (evicted); one copy job per slot that needs data;
//   copy      one CTA per (job, KV head): write an evicted dirty page's
//             gradients back, then copy the new page's K/V and/or dK/dV from
//             host memory over NVLink-C2C into the slot, 16-byte accesses;
//   writeback one CTA per (slot, KV head): copy a dirty slot's dK/dV back.
// Gradient pages known to be zero (after gradient zeroing, or fresh from an
// append) are only recorded as such per (page, KV head) in HBM: staging fills
// their slots with zeros instead of copying, and the record is dropped once a
// write-back has made the host page current.
#include <cuda_bf16.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace pkv {
namespace {

constexpr int kPlanThreads = 1024;
constexpr int kCopyThreads = 256;

// Block-wide exclusive scan of per-thread counts (kPlanThreads threads, warp
// shuffles then one pass over the warp totals); *total gets the sum.
__device__ int plan_scan(int v, int* sh, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int kWarps = kPlanThreads / 32;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sh[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int t = lane < kWarps ? sh[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        if (lane < kWarps) sh[lane] = t;                      // inclusive over warps
    }
    __syncthreads();
    const int base = warp > 0 ? sh[warp - 1] : 0;
    *total = sh[kWarps - 1];
    __syncthreads();                                          // sh reusable
    return base + x - v;
}

struct PlanArgs {
    const int32_t* pages;        // requested logical pages (entries < 0 ignored), or null = all
    int64_t n;
    int64_t n_pages;             // the sequence's logical pages
    int64_t n_slots;
    int want;                    // PKV_STAGE_KV | PKV_STAGE_GRADS
    int32_t* flags;              // [n_pages]: request flags
    int32_t* count_out;          // number of copy jobs
    int32_t* slot_of;            // [n_pages] logical -> slot or -1
    int32_t* slot_page;          // [n_slots] slot -> logical or -1
    int32_t* slot_state;         // [n_slots] kSlot* bits
    int32_t* avail;              // [n_slots] scratch
    int4* jobs;                  // [n_slots] (slot, page to write back or -1, new page, contents)
    unsigned long long* stats;   // [3] page-head counts: K/V in, grads in, grads out
    int Hkv;
    int* err;
};

__global__ void __launch_bounds__(kPlanThreads) stage_plan_kernel(PlanArgs a) {
    __shared__ int sh[kPlanThreads];
    __shared__ int n_jobs, n_kv, n_wb;
    const int tid = threadIdx.x;
    if (tid == 0) { n_jobs = 0; n_kv = 0; n_wb = 0; }
    for (int64_t p = tid; p < a.n_pages; p += kPlanThreads) a.flags[p] = a.pages ? 0 : 1;
    __syncthreads();
    if (a.pages) {
        for (int64_t i = tid; i < a.n; i += kPlanThreads) {
            const int32_t lp = a.pages[i];
            if (lp >= 0 && lp < a.n_pages) a.flags[lp] = 1;
        }
    }
    __syncthreads();
    // Resident requested pages keep their slots (mark them); count the new ones.
    const int64_t per = (a.n_pages + kPlanThreads - 1) / kPlanThreads;
    const int64_t p0 = (int64_t)tid * per, p1 = min64(a.n_pages, p0 + per);
    int n_new = 0;
    for (int64_t p = p0; p < p1; ++p) {
        if (!a.flags[p]) continue;
        const int32_t s = a.slot_of[p];
        if (s >= 0) a.slot_state[s] |= kSlotKeep;
        else ++n_new;
    }
    __syncthreads();
    int total_new;
    const int new_rank0 = plan_scan(n_new, sh, &total_new);
    // Slots a new page may take: empty ones first, then those of pages not
    // requested this time, each in ascending slot order.
    const int64_t sper = (a.n_slots + kPlanThreads - 1) / kPlanThreads;
    const int64_t s0 = (int64_t)tid * sper, s1 = min64(a.n_slots, s0 + sper);
    int n_empty = 0, n_evict = 0;
    for (int64_t s = s0; s < s1; ++s) {
        if (a.slot_page[s] < 0) ++n_empty;
        else if (!(a.slot_state[s] & kSlotKeep)) ++n_evict;
    }
    int tot_empty, tot_evict;
    const int e_rank0 = plan_scan(n_empty, sh, &tot_empty);
    const int v_rank0 = plan_scan(n_evict, sh, &tot_evict);
    {
        int er = e_rank0, vr = tot_empty + v_rank0;
        for (int64_t s = s0; s < s1; ++s) {
            if (a.slot_page[s] < 0) a.avail[er++] = (int32_t)s;
            else if (!(a.slot_state[s] & kSlotKeep)) a.avail[vr++] = (int32_t)s;
        }
    }
    __syncthreads();
    // Assign slots and emit copy jobs.
    const int64_t n_avail = (int64_t)tot_empty + tot_evict;
    int rank = new_rank0;
    for (int64_t p = p0; p < p1; ++p) {
        if (!a.flags[p]) continue;
        int32_t s = a.slot_of[p];
        int need, wb = -1;
        if (s >= 0) {
            need = a.want & ~a.slot_state[s] & (kSlotKV | kSlotG);
        } else {
            if (rank >= n_avail) {
                report_error(a.err, kErrSlots);
                ++rank;
                continue;
            }
            s = a.avail[rank++];
            const int32_t old = a.slot_page[s];
            if (old >= 0) {
                a.slot_of[old] = -1;
                if (a.slot_state[s] & kSlotDirty) wb = old;
            }
            a.slot_of[p] = s;
            a.slot_page[s] = (int32_t)p;
            a.slot_state[s] = 0;
            need = a.want & (kSlotKV | kSlotG);
        }
        if (need || wb >= 0) {
            const int j = atomicAdd(&n_jobs, 1);
            a.jobs[j] = make_int4(s, wb, (int)p, need);
            if (need & kSlotKV) atomicAdd(&n_kv, 1);
            if (wb >= 0) atomicAdd(&n_wb, 1);
        }
        // Staged gradients are about to be added into by a backward call.
        a.slot_state[s] = (a.slot_state[s] | need | ((a.want & kSlotG) ? kSlotDirty : 0)) & ~kSlotKeep;
    }
    __syncthreads();
    for (int64_t s = s0; s < s1; ++s) a.slot_state[s] &= ~kSlotKeep;
    if (tid == 0) {
        *a.count_out = n_jobs;
        atomicAdd(&a.stats[0], (unsigned long long)n_kv * a.Hkv);   // gradients in: by the copies
        atomicAdd(&a.stats[2], (unsigned long long)n_wb * a.Hkv);
    }
}

__device__ __forceinline__ void copy16(void* dst, const void* src, size_t bytes) {
    const uint4* s = static_cast<const uint4*>(src);
    uint4* d = static_cast<uint4*>(dst);
    const size_t n = bytes / 16;
    for (size_t i = threadIdx.x; i < n; i += kCopyThreads) d[i] = s[i];
}

__device__ __forceinline__ void zero16(void* dst, size_t bytes) {
    uint4* d = static_cast<uint4*>(dst);
    const size_t n = bytes / 16;
    for (size_t i = threadIdx.x; i < n; i += kCopyThreads) d[i] = make_uint4(0u, 0u, 0u, 0u);
}

struct StageArgs {
    const int32_t* bt;           // logical -> physical (host pages)
    const int4* jobs;
    const int32_t* count;        // number of jobs
    const int32_t* slot_page;    // slot -> logical
    int32_t* slot_state;
    int64_t num_phys;
    int64_t n_slots;
    int Hkv;
    size_t kv_bytes;             // one (page, head) tile of K or V
    size_t g_bytes;              // one (page, head) tile of dK or dV
    uint8_t* k; uint8_t* v; uint8_t* dk; uint8_t* dv;        // host pages
    uint8_t* ks; uint8_t* vs; uint8_t* dks; uint8_t* dvs;    // slots
    uint8_t* gzero;              // [num_phys * Hkv] gradient tiles recorded as zero
    unsigned long long* stats;
    int* err;
};

__device__ __forceinline__ bool page_ok(const StageArgs& a, int32_t lp, int64_t* pp) {
    *pp = lp >= 0 ? a.bt[lp] : -1;
    if (*pp < 0 || *pp >= a.num_phys) {
        if (threadIdx.x == 0) report_error(a.err, kErrBadPage);
        return false;
    }
    return true;
}

__device__ void stage_copy_job(const StageArgs& a, const int4 job, int h) {
    const size_t slot = (size_t)job.x * a.Hkv + h;
    int64_t pp;
    if (job.y >= 0 && page_ok(a, job.y, &pp)) {                 // evicted dirty gradients
        const size_t dst = (size_t)pp * a.Hkv + h;
        copy16(a.dk + dst * a.g_bytes, a.dks + slot * a.g_bytes, a.g_bytes);
        copy16(a.dv + dst * a.g_bytes, a.dvs + slot * a.g_bytes, a.g_bytes);
        if (threadIdx.x == 0) a.gzero[dst] = 0;                  // the host page is current
        __syncthreads();                                          // slot read before it is reused
    }
    if (!job.w || !page_ok(a, job.z, &pp)) return;
    const size_t src = (size_t)pp * a.Hkv + h;
    if (job.w & kSlotKV) {
        copy16(a.ks + slot * a.kv_bytes, a.k + src * a.kv_bytes, a.kv_bytes);
        copy16(a.vs + slot * a.kv_bytes, a.v + src * a.kv_bytes, a.kv_bytes);
    }
    if (job.w & kSlotG) {
        if (a.gzero[src]) {                                       // zero: nothing to copy
            zero16(a.dks + slot * a.g_bytes, a.g_bytes);
            zero16(a.dvs + slot * a.g_bytes, a.g_bytes);
        } else {
            copy16(a.dks + slot * a.g_bytes, a.dk + src * a.g_bytes, a.g_bytes);
            copy16(a.dvs + slot * a.g_bytes, a.dv + src * a.g_bytes, a.g_bytes);
            if (threadIdx.x == 0) atomicAdd(&a.stats[1], 1ull);
        }
    }
}

// One CTA per (job, KV head), the grid striding over the jobs of the plan
// (their number is known only on the device).
__global__ void __launch_bounds__(kCopyThreads) stage_copy_kernel(StageArgs a) {
    const int h = blockIdx.y;
    const int n_jobs = *a.count;
    for (int j = blockIdx.x; j < n_jobs; j += gridDim.x) stage_copy_job(a, a.jobs[j], h);
}

// Dirty gradient slots back to the host pages; with `release`, every slot's
// state is cleared afterwards by stage_release_kernel.
__global__ void __launch_bounds__(kCopyThreads) stage_writeback_kernel(StageArgs a) {
    const int s = blockIdx.x, h = blockIdx.y;
    if (!(a.slot_state[s] & kSlotDirty)) return;
    int64_t pp;
    if (!page_ok(a, a.slot_page[s], &pp)) return;
    const size_t src = (size_t)s * a.Hkv + h, dst = (size_t)pp * a.Hkv + h;
    copy16(a.dk + dst * a.g_bytes, a.dks + src * a.g_bytes, a.g_bytes);
    copy16(a.dv + dst * a.g_bytes, a.dvs + src * a.g_bytes, a.g_bytes);
    if (threadIdx.x == 0) {
        a.gzero[dst] = 0;                                         // the host page is current
        atomicAdd(&a.stats[2], 1ull);
    }
}

// After a write-back: clear DIRTY (release: empty every slot).
__global__ void stage_after_writeback_kernel(int32_t* slot_page, int32_t* slot_state,
                                             int32_t* slot_of, int64_t n_slots, int release) {
    for (int64_t s = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; s < n_slots;
         s += (int64_t)gridDim.x * blockDim.x) {
        if (release) {
            const int32_t p = slot_page[s];
            if (p >= 0) slot_of[p] = -1;
            slot_page[s] = -1;
            slot_state[s] = 0;
        } else {
            slot_state[s] &= ~kSlotDirty;
        }
    }
}

// Whole-sequence staging: slot i holds logical page i (the copy engines move
// runs of consecutive physical pages); every other slot is empty.
__global__ void stage_identity_kernel(int32_t* slot_page, int32_t* slot_state, int32_t* slot_of,
                                      int64_t n_pages, int64_t n_logical_cap, int64_t n_slots,
                                      int state) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n_logical_cap; i += stride) {
        if (i < n_slots) {
            slot_page[i] = i < n_pages ? (int32_t)i : -1;
            slot_state[i] = i < n_pages ? state : 0;
        }
        slot_of[i] = i < n_pages ? (int32_t)i : -1;
    }
}

StageArgs stage_args(const pkv_seq* s) {
    const pkv_pool* p = s->pool;
    StageArgs a{};
    a.bt = s->d_bt;
    a.jobs = s->d_jobs;
    a.count = s->d_flags + p->desc.num_phys_pages;
    a.slot_page = s->d_slot_page;
    a.slot_state = s->d_slot_state;
    a.num_phys = p->desc.num_phys_pages;
    a.n_slots = p->n_slots;
    a.Hkv = p->desc.n_kv_heads;
    a.kv_bytes = (size_t)p->desc.page_size * p->desc.head_dim * p->elem;
    a.g_bytes = (size_t)p->desc.page_size * p->desc.head_dim * sizeof(float);
    a.k = static_cast<uint8_t*>(p->k); a.v = static_cast<uint8_t*>(p->v);
    a.dk = reinterpret_cast<uint8_t*>(p->dk); a.dv = reinterpret_cast<uint8_t*>(p->dv);
    a.ks = static_cast<uint8_t*>(p->kslot); a.vs = static_cast<uint8_t*>(p->vslot);
    a.dks = reinterpret_cast<uint8_t*>(p->dkslot); a.dvs = reinterpret_cast<uint8_t*>(p->dvslot);
    a.gzero = p->gzero;
    a.stats = s->d_stats;
    a.err = p->d_err;
    return a;
}

}  // namespace

cudaError_t launch_stage_plan(const pkv_seq* s, const int32_t* pages, int64_t n, int want,
                              cudaStream_t st) {
    const pkv_pool* p = s->pool;
    PlanArgs a{};
    a.pages = pages; a.n = n;
    a.n_pages = (int64_t)s->bt.size();
    a.n_slots = p->n_slots;
    a.want = want;
    a.flags = s->d_flags; a.count_out = s->d_flags + p->desc.num_phys_pages;
    a.slot_of = s->d_slot_of; a.slot_page = s->d_slot_page;
    a.slot_state = s->d_slot_state; a.avail = s->d_avail; a.jobs = s->d_jobs;
    a.stats = s->d_stats; a.Hkv = p->desc.n_kv_heads; a.err = p->d_err;
    ProfScope ps("stage_plan_kernel", st);
    stage_plan_kernel<<<1, kPlanThreads, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_stage_copy(const pkv_seq* s, cudaStream_t st) {
    const pkv_pool* p = s->pool;
    ProfScope ps("stage_copy_kernel", st);
    dim3 grid((unsigned)std::min<int64_t>(p->n_slots, 512), p->desc.n_kv_heads);
    stage_copy_kernel<<<grid, kCopyThreads, 0, st>>>(stage_args(s));
    return cudaGetLastError();
}

cudaError_t launch_stage_writeback(const pkv_seq* s, bool release, cudaStream_t st) {
    const pkv_pool* p = s->pool;
    {
        ProfScope ps("stage_writeback_kernel", st);
        dim3 grid((unsigned)p->n_slots, p->desc.n_kv_heads);
        stage_writeback_kernel<<<grid, kCopyThreads, 0, st>>>(stage_args(s));
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return launch_stage_after_writeback(s, release, st);
}

cudaError_t launch_stage_after_writeback(const pkv_seq* s, bool release, cudaStream_t st) {
    const pkv_pool* p = s->pool;
    const unsigned blocks = (unsigned)std::min<int64_t>(1024, (p->n_slots + 255) / 256);
    stage_after_writeback_kernel<<<blocks, 256, 0, st>>>(s->d_slot_page, s->d_slot_state,
                                                         s->d_slot_of, p->n_slots, release ? 1 : 0);
    return cudaGetLastError();
}

cudaError_t launch_stage_identity(const pkv_seq* s, int64_t n_pages, int want, cudaStream_t st) {
    const pkv_pool* p = s->pool;
    const int state = (want & (kSlotKV | kSlotG)) | ((want & kSlotG) ? kSlotDirty : 0);
    const int64_t cap = p->desc.num_phys_pages;
    const unsigned blocks = (unsigned)std::min<int64_t>(1024, (cap + 255) / 256);
    stage_identity_kernel<<<blocks, 256, 0, st>>>(s->d_slot_page, s->d_slot_state, s->d_slot_of,
                                                  n_pages, cap, p->n_slots, state);
    return cudaGetLastError();
}

namespace {
__global__ void stage_invalidate_kv_kernel(const int32_t* slot_of, int32_t* slot_state, int64_t lp) {
    const int32_t s = slot_of[lp];
    if (s >= 0) slot_state[s] &= ~kSlotKV;
}
}  // namespace

cudaError_t launch_stage_invalidate_kv(const pkv_seq* s, int64_t lp, cudaStream_t st) {
    stage_invalidate_kv_kernel<<<1, 1, 0, st>>>(s->d_slot_of, s->d_slot_state, lp);
    return cudaGetLastError();
}

namespace {
// Sets (value 1) or clears (0) the zero record of (bt[i], h) for logical pages
// i < n and every KV head.
__global__ void gzero_set_kernel(const int32_t* bt, int64_t n, int64_t num_phys, int Hkv,
                                 uint8_t* gzero, uint8_t value, int* err) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n * Hkv; i += stride) {
        const int32_t pp = bt[i / Hkv];
        if (pp < 0 || pp >= num_phys) {
            report_error(err, kErrBadPage);
            continue;
        }
        gzero[(size_t)pp * Hkv + i % Hkv] = value;
    }
}

// Zeroes the gradients held by staged slots (state G), KV head blockIdx.y.
__global__ void __launch_bounds__(kCopyThreads) slot_grad_zero_kernel(StageArgs a) {
    const int h = blockIdx.y;
    for (int64_t s = blockIdx.x; s < a.n_slots; s += gridDim.x) {
        if (a.slot_page[s] < 0 || !(a.slot_state[s] & kSlotG)) continue;
        const size_t t = (size_t)s * a.Hkv + h;
        zero16(a.dks + t * a.g_bytes, a.g_bytes);
        zero16(a.dvs + t * a.g_bytes, a.g_bytes);
    }
}

// After the copy engines staged the gradients of logical pages [0, n) into
// slots 0..n-1: the slots of pages recorded as zero get zeros.
__global__ void __launch_bounds__(kCopyThreads) gzero_fill_slots_kernel(StageArgs a, int64_t n) {
    const int h = blockIdx.y;
    for (int64_t i = blockIdx.x; i < n; i += gridDim.x) {
        const int32_t pp = a.bt[i];
        if (pp < 0 || pp >= a.num_phys || !a.gzero[(size_t)pp * a.Hkv + h]) continue;
        const size_t t = (size_t)i * a.Hkv + h;
        zero16(a.dks + t * a.g_bytes, a.g_bytes);
        zero16(a.dvs + t * a.g_bytes, a.g_bytes);
    }
}

cudaError_t launch_gzero_set(const pkv_seq* s, int64_t n, uint8_t value, cudaStream_t st) {
    const pkv_pool* p = s->pool;
    if (n <= 0) return cudaSuccess;
    const int Hkv = p->desc.n_kv_heads;
    const unsigned blocks = (unsigned)std::min<int64_t>(1024, (n * Hkv + 255) / 256);
    ProfScope ps("gzero_set_kernel", st);
    gzero_set_kernel<<<blocks, 256, 0, st>>>(s->d_bt, n, p->desc.num_phys_pages, Hkv, p->gzero,
                                             value, p->d_err);
    return cudaGetLastError();
}
}  // namespace

cudaError_t launch_grad_zero_staged(const pkv_seq* s, cudaStream_t st) {
    const pkv_pool* p = s->pool;
    cudaError_t e = launch_gzero_set(s, (int64_t)s->bt.size(), 1, st);
    if (e != cudaSuccess) return e;
    ProfScope ps("slot_grad_zero_kernel", st);
    dim3 grid((unsigned)std::min<int64_t>(p->n_slots, 512), p->desc.n_kv_heads);
    slot_grad_zero_kernel<<<grid, kCopyThreads, 0, st>>>(stage_args(s));
    return cudaGetLastError();
}

cudaError_t launch_gzero_fill_slots(const pkv_seq* s, int64_t n, cudaStream_t st) {
    const pkv_pool* p = s->pool;
    if (n <= 0) return cudaSuccess;
    ProfScope ps("gzero_fill_slots_kernel", st);
    dim3 grid((unsigned)std::min<int64_t>(n, 512), p->desc.n_kv_heads);
    gzero_fill_slots_kernel<<<grid, kCopyThreads, 0, st>>>(stage_args(s), n);
    return cudaGetLastError();
}

cudaError_t launch_gzero_clear(const pkv_seq* s, int64_t n, cudaStream_t st) {
    return launch_gzero_set(s, n, 0, st);
}

}  // namespace pkv
