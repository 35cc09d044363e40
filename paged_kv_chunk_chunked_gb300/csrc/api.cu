// C-ABI layer of libpkv: argument validation, the page pool and block-table
// allocator, and dispatch to the kernels. See include/pkv.h for the contract.
//
// The paged memory manager follows "Out of the Memory Barrier" (gist.science/de
// §2.B; sciencestack.ai Fig. 3, Fig. 4): all page memory is allocated once, at
// pool creation; a sequence grows by taking pages off a free list and writing
// their indices into its block table, so appending never reallocates or copies
// the cache, and the gradient pages share the physical index of their K/V page.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <chrono>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <thread>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace pkv {

static thread_local std::string g_last_error;

pkv_status fail(pkv_status s, const std::string& msg) {
    g_last_error = msg;
    return s;
}

pkv_status cuda_fail(cudaError_t e, const char* what) {
    std::string m = std::string(what) + ": " + cudaGetErrorName(e) + " (" +
                    cudaGetErrorString(e) + ")";
    return fail(e == cudaErrorMemoryAllocation ? PKV_ERR_OOM : PKV_ERR_CUDA, m);
}

// ---------------------------------------------------------------- TMA descriptors

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn(std::string* why) {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    static std::string err;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                                         cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || p == nullptr) {
            err = "cuTensorMapEncodeTiled entry point not available";
        } else {
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        }
    });
    if (!fn && why) *why = err;
    return fn;
}

bool make_tmap_2d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, uint64_t inner,
                  uint64_t rows, uint64_t row_stride_bytes, uint32_t box_inner,
                  uint32_t box_rows, std::string* why) {
    auto fn = encode_fn(why);
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {row_stride_bytes};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t es[2] = {1, 1};
    CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        if (why) *why = "cuTensorMapEncodeTiled (2-D) failed with CUresult " + std::to_string(r);
        return false;
    }
    return true;
}

bool make_tmap_3d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, uint64_t d0,
                  uint64_t d1, uint64_t d2, uint64_t stride1_bytes, uint64_t stride2_bytes,
                  uint32_t b0, uint32_t b1, uint32_t b2, std::string* why) {
    auto fn = encode_fn(why);
    if (!fn) return false;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
    cuuint32_t box[3] = {b0, b1, b2};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        if (why) *why = "cuTensorMapEncodeTiled (3-D) failed with CUresult " + std::to_string(r);
        return false;
    }
    return true;
}

}  // namespace pkv

using namespace pkv;

// ---------------------------------------------------------------- helpers

static pkv_status validate_desc(const pkv_pool_desc* d) {
    if (!d) return fail(PKV_ERR_INVALID, "pkv_pool_create: desc is NULL");
    if (d->page_size <= 0 || d->page_size % 8)
        return fail(PKV_ERR_INVALID, "page_size must be a positive multiple of 8");
    if (d->n_kv_heads <= 0 || d->n_q_heads <= 0 || d->n_q_heads % d->n_kv_heads)
        return fail(PKV_ERR_INVALID, "n_q_heads must be a positive multiple of n_kv_heads");
    if (d->head_dim != 64 && d->head_dim != 128)
        return fail(PKV_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
    if (d->dtype != PKV_BF16 && d->dtype != PKV_F32)
        return fail(PKV_ERR_INVALID, "dtype must be PKV_BF16 or PKV_F32");
    if (d->residency < PKV_RES_DEVICE || d->residency > PKV_RES_META)
        return fail(PKV_ERR_INVALID, "unknown residency");
    if (d->num_phys_pages <= 0 || d->num_phys_pages > (int64_t(1) << 30))
        return fail(PKV_ERR_INVALID, "num_phys_pages out of range");
    if ((int64_t)d->num_phys_pages * d->n_kv_heads * d->page_size >= (int64_t(1) << 31))
        return fail(PKV_ERR_INVALID, "pool too large: pages*Hkv*P must be < 2^31 rows");
    return PKV_OK;
}

static bool is_device(const pkv_pool* p) { return p->desc.residency != PKV_RES_META; }

// Claims pages so that the sequence covers new_len tokens. Host-only; on
// failure nothing changes.
static pkv_status claim_pages(pkv_seq* s, int64_t new_len) {
    pkv_pool* p = s->pool;
    const int64_t P = p->desc.page_size;
    const int64_t need = (new_len + P - 1) / P;
    const int64_t have = (int64_t)s->bt.size();
    if (need <= have) return PKV_OK;
    const int64_t extra = need - have;
    if ((int64_t)p->free_list.size() < extra)
        return fail(PKV_ERR_OOM, "page pool exhausted: need " + std::to_string(extra) +
                                     " pages, " + std::to_string(p->free_list.size()) + " free");
    for (int64_t i = 0; i < extra; ++i) {
        int32_t pg = p->free_list.back();
        p->free_list.pop_back();
        p->in_use[pg] = 1;
        s->bt.push_back(pg);
        if (s->h_bt) s->h_bt[have + i] = pg;
    }
    return PKV_OK;
}

static void release_pages(pkv_seq* s) {
    pkv_pool* p = s->pool;
    // Later claims rewrite h_bt from entry 0: uploads still queued must have read it.
    if (s->bt_pending) {
        cudaEventSynchronize(s->bt_sent);
        s->bt_pending = false;
    }
    // Push back in reverse so a fresh sequence gets the same pages in the same order.
    for (auto it = s->bt.rbegin(); it != s->bt.rend(); ++it) {
        p->in_use[*it] = 0;
        p->free_list.push_back(*it);
    }
    s->bt.clear();
    s->len = 0;
    s->n_reserved_pages = 0;
    s->staged_all = 0;          // slots no longer mirror this sequence's pages
    if (s->d_slot_of) {
        // The slot cache holds the old pages: empty it (after every queued use).
        const size_t nb = (size_t)p->desc.num_phys_pages * sizeof(int32_t);
        cudaDeviceSynchronize();
        cudaMemset(s->d_slot_of, 0xff, nb);
        cudaMemset(s->d_slot_page, 0xff, p->n_slots * sizeof(int32_t));
        cudaMemset(s->d_slot_state, 0, p->n_slots * sizeof(int32_t));
        cudaDeviceSynchronize();
        s->dirty_possible = false;
    }
}

// Uploads block-table entries [from, bt.size()) to the device copy on stream.
// A kernel reads them from the mapped pinned mirror: a copy-engine transfer on
// the compute stream would queue behind bulk host-to-device copies issued on
// other streams (the inputs of later chunks) and hold the next kernel back.
static pkv_status upload_bt(pkv_seq* s, int64_t from, cudaStream_t st) {
    if (!is_device(s->pool)) return PKV_OK;
    const int64_t n = (int64_t)s->bt.size() - from;
    if (n <= 0) return PKV_OK;
    cudaError_t e = launch_bt_upload(s->h_bt_dev + from, s->d_bt + from, n, st);
    if (e == cudaSuccess) e = cudaEventRecord(s->bt_sent, st);
    if (e != cudaSuccess) return cuda_fail(e, "block-table upload");
    s->bt_pending = true;
    return PKV_OK;
}

static pkv_status check_stream_device(const pkv_pool* p) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev != p->device)
        return fail(PKV_ERR_INVALID, "the current CUDA device is not the pool's device");
    return PKV_OK;
}

// ---------------------------------------------------------------- C ABI

extern "C" {

const char* pkv_last_error(void) { return g_last_error.c_str(); }

pkv_status pkv_check(pkv_pool* pool) {
    if (!pool) return fail(PKV_ERR_INVALID, "pkv_check: pool is NULL");
    if (!is_device(pool)) return PKV_OK;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "pkv_check: cudaDeviceSynchronize");
    int h = 0;
    e = cudaMemcpy(&h, pool->d_err, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "pkv_check: read error word");
    if (h != 0) {
        int zero = 0;
        cudaMemcpy(pool->d_err, &zero, sizeof(int), cudaMemcpyHostToDevice);
        const char* what = h == pkv::kErrWaitTimeout ? "a bounded wait expired"
                         : h == pkv::kErrBadPage     ? "a page index was out of range"
                         : h == pkv::kErrTmemAlloc   ? "tensor-memory allocation failed"
                         : h == pkv::kErrSlots       ? "more pages staged than device slots"
                                                : "unknown device error";
        return fail(PKV_ERR_DEVICE_FAULT, std::string("device error ") + std::to_string(h) +
                                              ": " + what);
    }
    return PKV_OK;
}

pkv_status pkv_pool_create(const pkv_pool_desc* desc, pkv_pool** out) {
    if (!out) return fail(PKV_ERR_INVALID, "pkv_pool_create: out is NULL");
    *out = nullptr;
    pkv_status st = validate_desc(desc);
    if (st != PKV_OK) return st;
    pkv_pool* p = new pkv_pool();
    p->desc = *desc;
    p->elem = desc->dtype == PKV_BF16 ? 2 : 4;
    p->page_elems = (size_t)desc->n_kv_heads * desc->page_size * desc->head_dim;
    const int64_t np = desc->num_phys_pages;
    p->free_list.resize(np);
    for (int64_t i = 0; i < np; ++i) p->free_list[i] = (int32_t)(np - 1 - i);  // page 0 on top
    p->in_use.assign(np, 0);
    if (desc->residency == PKV_RES_META) {
        *out = p;
        return PKV_OK;
    }
    const bool host = desc->residency == PKV_RES_PINNED_HOST;
    if (host && (desc->n_device_slots <= 0 || desc->n_device_slots > np))
        { delete p; return fail(PKV_ERR_INVALID, "PINNED_HOST pools need 0 < n_device_slots <= num_phys_pages"); }
    cudaError_t e = cudaGetDevice(&p->device);
    if (e != cudaSuccess) { delete p; return cuda_fail(e, "cudaGetDevice"); }
    const size_t kv_bytes = p->page_elems * p->elem * np;
    const size_t g_bytes = p->page_elems * sizeof(float) * np;
    const size_t rep_bytes = (size_t)np * desc->n_kv_heads * desc->head_dim * sizeof(float);
    auto cleanup = [p, host]() {
        if (host) {
            cudaFreeHost(p->k); cudaFreeHost(p->v); cudaFreeHost(p->dk); cudaFreeHost(p->dv);
            cudaFree(p->kslot); cudaFree(p->vslot); cudaFree(p->dkslot); cudaFree(p->dvslot);
            cudaFree(p->gzero);
        } else {
            cudaFree(p->k); cudaFree(p->v); cudaFree(p->dk); cudaFree(p->dv);
        }
        cudaFree(p->rep); cudaFree(p->d_err); cudaFree(p->sel_state);
        delete p;
    };
    if (host) {
        // Pages in mapped pinned host memory (reachable by kernels over the
        // host link); slots and representatives in HBM.
        const unsigned fl = cudaHostAllocMapped | cudaHostAllocPortable;
        p->n_slots = desc->n_device_slots;
        const size_t skv = p->page_elems * p->elem * p->n_slots;
        const size_t sg = p->page_elems * sizeof(float) * p->n_slots;
        if ((e = cudaHostAlloc(&p->k, kv_bytes, fl)) != cudaSuccess ||
            (e = cudaHostAlloc(&p->v, kv_bytes, fl)) != cudaSuccess ||
            (e = cudaHostAlloc(reinterpret_cast<void**>(&p->dk), g_bytes, fl)) != cudaSuccess ||
            (e = cudaHostAlloc(reinterpret_cast<void**>(&p->dv), g_bytes, fl)) != cudaSuccess ||
            (e = cudaMalloc(&p->kslot, skv)) != cudaSuccess ||
            (e = cudaMalloc(&p->vslot, skv)) != cudaSuccess ||
            (e = cudaMalloc(reinterpret_cast<void**>(&p->dkslot), sg)) != cudaSuccess ||
            (e = cudaMalloc(reinterpret_cast<void**>(&p->dvslot), sg)) != cudaSuccess ||
            (e = cudaMalloc(reinterpret_cast<void**>(&p->gzero), (size_t)np * desc->n_kv_heads)) != cudaSuccess ||
            (e = cudaMemset(p->gzero, 0, (size_t)np * desc->n_kv_heads)) != cudaSuccess ||
            (e = cudaMalloc(reinterpret_cast<void**>(&p->rep), rep_bytes)) != cudaSuccess ||
            (e = cudaMalloc(reinterpret_cast<void**>(&p->d_err), sizeof(int))) != cudaSuccess) {
            cleanup();
            return cuda_fail(e, "pkv_pool_create: pinned pages / slots");
        }
        std::memset(p->k, 0, kv_bytes);
        std::memset(p->v, 0, kv_bytes);
    } else if ((e = cudaMalloc(&p->k, kv_bytes)) != cudaSuccess ||
               (e = cudaMalloc(&p->v, kv_bytes)) != cudaSuccess ||
               (e = cudaMalloc(reinterpret_cast<void**>(&p->dk), g_bytes)) != cudaSuccess ||
               (e = cudaMalloc(reinterpret_cast<void**>(&p->dv), g_bytes)) != cudaSuccess ||
               (e = cudaMalloc(reinterpret_cast<void**>(&p->rep), rep_bytes)) != cudaSuccess ||
               (e = cudaMalloc(reinterpret_cast<void**>(&p->d_err), sizeof(int))) != cudaSuccess) {
        cleanup();
        return cuda_fail(e, "pkv_pool_create: page memory");
    }
    const size_t state_bytes = (size_t)page_topk_state_ints(desc->n_kv_heads) * sizeof(int);
    if ((e = cudaMalloc(reinterpret_cast<void**>(&p->sel_state), state_bytes)) != cudaSuccess ||
        (e = cudaMemset(p->sel_state, 0, state_bytes)) != cudaSuccess) {
        cleanup();
        return cuda_fail(e, "pkv_pool_create: selection state");
    }
    if ((e = cudaMemset(p->d_err, 0, sizeof(int))) != cudaSuccess ||
        (!host && (e = cudaMemset(p->k, 0, kv_bytes)) != cudaSuccess) ||
        (!host && (e = cudaMemset(p->v, 0, kv_bytes)) != cudaSuccess) ||
        (e = cudaMemset(p->rep, 0, rep_bytes)) != cudaSuccess) {
        cleanup();
        return cuda_fail(e, "pkv_pool_create: memset");
    }
    if (desc->dtype == PKV_BF16 && (desc->head_dim == 128 || desc->head_dim == 64) &&
        desc->page_size == 128) {
        // The tensor-core kernels read K/V by TMA (boxes of 64 columns x 128
        // rows): the pool in HBM, or the slots.
        std::string why;
        void* kb = host ? p->kslot : p->k;
        void* vb = host ? p->vslot : p->v;
        const uint64_t rows = (uint64_t)(host ? p->n_slots : np) * desc->n_kv_heads * desc->page_size;
        const uint64_t dd = (uint64_t)desc->head_dim;
        // The dK/dV kernel adds its page's gradients into the fp32 pool (or
        // slots) by TMA reduce-add: boxes of 32 columns (128 bytes) x 128 rows.
        void* dkb = host ? p->dkslot : p->dk;
        void* dvb = host ? p->dvslot : p->dv;
        if (!make_tmap_2d(&p->tmap_k, kb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, dd, rows, dd * 2, 64,
                          128, &why) ||
            !make_tmap_2d(&p->tmap_v, vb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, dd, rows, dd * 2, 64,
                          128, &why) ||
            !make_tmap_2d(&p->tmap_dk, dkb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, dd, rows, dd * 4, 32,
                          128, &why) ||
            !make_tmap_2d(&p->tmap_dv, dvb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, dd, rows, dd * 4, 32,
                          128, &why)) {
            cleanup();
            return fail(PKV_ERR_CUDA, "pkv_pool_create: " + why);
        }
        p->tmaps_ready = true;
    }
    // Pool creation is synchronous: the memsets above are complete before any
    // stream, blocking or not, uses the pool.
    if ((e = cudaDeviceSynchronize()) != cudaSuccess) {
        cleanup();
        return cuda_fail(e, "pkv_pool_create: sync");
    }
    *out = p;
    return PKV_OK;
}

void pkv_pool_destroy(pkv_pool* p) {
    if (!p) return;
    std::vector<pkv_seq*> seqs = p->seqs;
    for (pkv_seq* s : seqs) pkv_seq_free(s);
    if (p->desc.residency == PKV_RES_PINNED_HOST) {
        cudaFreeHost(p->k); cudaFreeHost(p->v); cudaFreeHost(p->dk); cudaFreeHost(p->dv);
        cudaFree(p->kslot); cudaFree(p->vslot); cudaFree(p->dkslot); cudaFree(p->dvslot);
        cudaFree(p->gzero);
    } else if (is_device(p)) {
        cudaFree(p->k); cudaFree(p->v); cudaFree(p->dk); cudaFree(p->dv);
    }
    if (is_device(p)) {
        cudaFree(p->rep); cudaFree(p->d_err); cudaFree(p->scratch); cudaFree(p->sel_scratch);
        cudaFree(p->sel_state);
    }
    delete p;
}

pkv_status pkv_pool_free_pages(const pkv_pool* p, int64_t* n) {
    if (!p || !n) return fail(PKV_ERR_INVALID, "pkv_pool_free_pages: NULL argument");
    *n = (int64_t)p->free_list.size();
    return PKV_OK;
}

pkv_status pkv_pool_arrays(const pkv_pool* p, void** k, void** v, float** dk, float** dv,
                           float** rep) {
    if (!p) return fail(PKV_ERR_INVALID, "pkv_pool_arrays: pool is NULL");
    if (k) *k = p->k;
    if (v) *v = p->v;
    if (dk) *dk = p->dk;
    if (dv) *dv = p->dv;
    if (rep) *rep = p->rep;
    return PKV_OK;
}

pkv_status pkv_seq_create(pkv_pool* p, pkv_seq** out) {
    if (!p || !out) return fail(PKV_ERR_INVALID, "pkv_seq_create: NULL argument");
    *out = nullptr;
    pkv_seq* s = new pkv_seq();
    s->pool = p;
    if (is_device(p)) {
        const size_t bytes = (size_t)p->desc.num_phys_pages * sizeof(int32_t);
        cudaError_t e = cudaHostAlloc(reinterpret_cast<void**>(&s->h_bt), bytes,
                                      cudaHostAllocMapped | cudaHostAllocPortable);
        if (e == cudaSuccess)
            e = cudaHostGetDevicePointer(reinterpret_cast<void**>(&s->h_bt_dev), s->h_bt, 0);
        if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void**>(&s->d_bt), bytes);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s->bt_sent, cudaEventDisableTiming);
        if (e == cudaSuccess && p->desc.residency == PKV_RES_PINNED_HOST) {
            const size_t sb = p->n_slots * sizeof(int32_t);
            e = cudaMalloc(reinterpret_cast<void**>(&s->d_slot_of), bytes);
            if (e == cudaSuccess) e = cudaMemset(s->d_slot_of, 0xff, bytes);   // all -1
            if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void**>(&s->d_slot_page), sb);
            if (e == cudaSuccess) e = cudaMemset(s->d_slot_page, 0xff, sb);   // every slot empty
            if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void**>(&s->d_slot_state), sb);
            if (e == cudaSuccess) e = cudaMemset(s->d_slot_state, 0, sb);
            if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void**>(&s->d_avail), sb);
            if (e == cudaSuccess)
                e = cudaMalloc(reinterpret_cast<void**>(&s->d_jobs), p->n_slots * sizeof(int4));
            if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void**>(&s->d_stats), 4 * sizeof(unsigned long long));
            if (e == cudaSuccess) e = cudaMemset(s->d_stats, 0, 4 * sizeof(unsigned long long));
            if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void**>(&s->d_flags), bytes + sizeof(int32_t));
            if (e == cudaSuccess) e = cudaMemset(s->d_flags, 0, bytes + sizeof(int32_t));
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s->staged, cudaEventDisableTiming);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s->used, cudaEventDisableTiming);
        }
        // The initialisation above must be complete before any stream (including a
        // non-blocking side stream) touches the sequence.
        if (e == cudaSuccess) e = cudaDeviceSynchronize();
        if (e != cudaSuccess) {
            cudaFreeHost(s->h_bt);
            cudaFree(s->d_bt); cudaFree(s->d_slot_of); cudaFree(s->d_slot_page); cudaFree(s->d_flags);
            cudaFree(s->d_slot_state); cudaFree(s->d_avail); cudaFree(s->d_jobs); cudaFree(s->d_stats);
            if (s->staged) cudaEventDestroy(s->staged);
            if (s->used) cudaEventDestroy(s->used);
            if (s->bt_sent) cudaEventDestroy(s->bt_sent);
            delete s;
            return cuda_fail(e, "pkv_seq_create: block table");
        }
    }
    p->seqs.push_back(s);
    *out = s;
    return PKV_OK;
}

void pkv_seq_free(pkv_seq* s) {
    if (!s) return;
    release_pages(s);
    auto& v = s->pool->seqs;
    v.erase(std::remove(v.begin(), v.end(), s), v.end());
    if (is_device(s->pool)) {
        cudaFreeHost(s->h_bt);
        cudaFree(s->d_bt);
        cudaFree(s->d_slot_of); cudaFree(s->d_slot_page); cudaFree(s->d_flags);
        cudaFree(s->d_slot_state); cudaFree(s->d_avail); cudaFree(s->d_jobs); cudaFree(s->d_stats);
        if (s->staged) cudaEventDestroy(s->staged);
        if (s->used) cudaEventDestroy(s->used);
        if (s->bt_sent) cudaEventDestroy(s->bt_sent);
    }
    delete s;
}

pkv_status pkv_seq_reset(pkv_seq* s) {
    if (!s) return fail(PKV_ERR_INVALID, "pkv_seq_reset: seq is NULL");
    release_pages(s);
    return PKV_OK;
}

pkv_status pkv_seq_length(const pkv_seq* s, int64_t* len) {
    if (!s || !len) return fail(PKV_ERR_INVALID, "pkv_seq_length: NULL argument");
    *len = s->len;
    return PKV_OK;
}

pkv_status pkv_seq_reserve(pkv_seq* s, int64_t n_tok) {
    if (!s || n_tok < 0) return fail(PKV_ERR_INVALID, "pkv_seq_reserve: bad argument");
    return claim_pages(s, s->len + n_tok);
}

pkv_status pkv_get_block_table(const pkv_seq* s, int32_t* out, int64_t cap, int64_t* n) {
    if (!s || !n || (cap > 0 && !out))
        return fail(PKV_ERR_INVALID, "pkv_get_block_table: bad argument");
    *n = (int64_t)s->bt.size();
    const int64_t m = std::min<int64_t>(cap, *n);
    if (m > 0) std::memcpy(out, s->bt.data(), m * sizeof(int32_t));
    return PKV_OK;
}

pkv_status pkv_set_block_table(pkv_seq* s, const int32_t* bt, int64_t n) {
    if (!s || (n > 0 && !bt) || n < 0)
        return fail(PKV_ERR_INVALID, "pkv_set_block_table: bad argument");
    if (s->len != 0 || !s->bt.empty())
        return fail(PKV_ERR_INVALID, "pkv_set_block_table: the sequence must be empty");
    pkv_pool* p = s->pool;
    std::vector<uint8_t> seen(p->desc.num_phys_pages, 0);
    for (int64_t i = 0; i < n; ++i) {
        const int32_t pg = bt[i];
        if (pg < 0 || pg >= p->desc.num_phys_pages)
            return fail(PKV_ERR_INVALID, "pkv_set_block_table: entry " + std::to_string(i) +
                                             " = " + std::to_string(pg) + " out of range");
        if (p->in_use[pg] || seen[pg])
            return fail(PKV_ERR_INVALID, "pkv_set_block_table: page " + std::to_string(pg) +
                                             " is not free or appears twice");
        seen[pg] = 1;
    }
    // Remove the claimed pages from the free list, keeping its order otherwise.
    std::vector<int32_t> fl;
    fl.reserve(p->free_list.size());
    for (int32_t pg : p->free_list)
        if (!seen[pg]) fl.push_back(pg);
    p->free_list.swap(fl);
    s->bt.assign(bt, bt + n);
    for (int64_t i = 0; i < n; ++i) p->in_use[bt[i]] = 1;
    s->n_reserved_pages = n;
    if (is_device(p) && n > 0) {
        if (s->bt_pending) {                         // h_bt may still be a queued copy's source
            cudaEventSynchronize(s->bt_sent);
            s->bt_pending = false;
        }
        std::memcpy(s->h_bt, bt, n * sizeof(int32_t));
        cudaError_t e = cudaMemcpy(s->d_bt, s->h_bt, n * sizeof(int32_t), cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_fail(e, "pkv_set_block_table: upload");
    }
    return PKV_OK;
}

pkv_status pkv_append(pkv_seq* s, const void* k, const void* v, int64_t n_tok, void* stream) {
    if (!s || n_tok < 0) return fail(PKV_ERR_INVALID, "pkv_append: bad argument");
    if (n_tok == 0) return PKV_OK;
    if (!k || !v) return fail(PKV_ERR_INVALID, "pkv_append: k or v is NULL");
    pkv_pool* p = s->pool;
    if (!is_device(p)) return fail(PKV_ERR_INVALID, "pkv_append: META pool holds no data");
    pkv_status st = check_stream_device(p);
    if (st != PKV_OK) return st;
    const int64_t old_pages = (int64_t)s->bt.size();
    st = claim_pages(s, s->len + n_tok);
    if (st != PKV_OK) return st;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    st = upload_bt(s, old_pages, cs);
    if (st != PKV_OK) return st;
    if (s->d_slot_of && s->len % p->desc.page_size != 0) {
        // Extending a partial page that may be staged: its slot's K/V goes stale.
        cudaError_t e = cudaStreamWaitEvent(cs, s->staged, 0);
        if (e == cudaSuccess) e = launch_stage_invalidate_kv(s, s->len / p->desc.page_size, cs);
        if (e != cudaSuccess) return cuda_fail(e, "pkv_append: slot invalidation");
    }
    AppendArgs a{};
    a.P = p->desc.page_size; a.Hkv = p->desc.n_kv_heads; a.d = p->desc.head_dim;
    a.dtype = p->desc.dtype;
    a.k_in = k; a.v_in = v;
    a.kpool = p->k; a.vpool = p->v; a.dkpool = p->dk; a.dvpool = p->dv; a.rep = p->rep;
    a.bt = s->d_bt; a.num_phys = p->desc.num_phys_pages;
    a.old_len = s->len; a.n_tok = n_tok; a.gzero = p->gzero; a.err = p->d_err;
    if (p->gzero) s->gzero_possible = true;              // fresh pages are recorded as zero
    cudaError_t e = launch_append(a, cs);
    if (e == cudaSuccess && s->used) e = cudaEventRecord(s->used, cs);
    if (e != cudaSuccess) return cuda_fail(e, "pkv_append: launch");
    s->len += n_tok;
    return PKV_OK;
}

}  // extern "C"

pkv_status pkv::attn_common(pkv_seq* s, const void* q, int64_t q_start, int64_t n_q,
                            const pkv_sel* sel, AttnArgs* a, const char* who) {
    if (!s || !q) return fail(PKV_ERR_INVALID, std::string(who) + ": NULL argument");
    pkv_pool* p = s->pool;
    if (!is_device(p)) return fail(PKV_ERR_INVALID, std::string(who) + ": META pool");
    const int64_t P = p->desc.page_size;
    if (n_q <= 0 || q_start < 0 || q_start % P != 0 || q_start + n_q > s->len)
        return fail(PKV_ERR_INVALID,
                    std::string(who) + ": need q_start % P == 0 and q_start + n_q <= length (" +
                        std::to_string(q_start) + " + " + std::to_string(n_q) +
                        " vs " + std::to_string(s->len) + ")");
    pkv_status st = check_stream_device(p);
    if (st != PKV_OK) return st;
    *a = AttnArgs{};
    a->P = (int)P; a->Hq = p->desc.n_q_heads; a->Hkv = p->desc.n_kv_heads;
    a->d = p->desc.head_dim; a->dtype = p->desc.dtype;
    a->q_start = q_start; a->n_q = n_q; a->q = q;
    if (p->desc.residency == PKV_RES_PINNED_HOST) {
        // Attention reads the device slots through the logical-page -> slot table.
        a->kpool = p->kslot; a->vpool = p->vslot; a->dkpool = p->dkslot; a->dvpool = p->dvslot;
        a->bt = s->d_slot_of; a->num_phys = p->n_slots;
    } else {
        a->kpool = p->k; a->vpool = p->v; a->dkpool = p->dk; a->dvpool = p->dv;
        a->bt = s->d_bt; a->num_phys = p->desc.num_phys_pages;
    }
    a->err = p->d_err;
    a->tmap_k = p->tmaps_ready ? &p->tmap_k : nullptr;
    a->tmap_v = p->tmaps_ready ? &p->tmap_v : nullptr;
    a->tmap_dk = p->tmaps_ready ? &p->tmap_dk : nullptr;
    a->tmap_dv = p->tmaps_ready ? &p->tmap_dv : nullptr;
    if (sel) {
        const int64_t n_qp = (n_q + P - 1) / P;
        if (!sel->pages || sel->kmax <= 0 || sel->n_qp != n_qp)
            return fail(PKV_ERR_INVALID, std::string(who) + ": selection does not match chunk");
        a->sel = sel->pages;
        a->kmax = sel->kmax;
    }
    return PKV_OK;
}

bool pkv::use_tc(const pkv_pool* p, const AttnArgs& a) {
    return !(p->desc.flags & PKV_FLAG_SIMT_ONLY) && p->tmaps_ready && tc_supported(a);
}

extern "C" {

pkv_status pkv_chunk_attn_fwd(pkv_seq* s, const void* q, int64_t q_start, int64_t n_q, void* o,
                              float* lse, const pkv_sel* sel, void* stream) {
    AttnArgs a;
    pkv_status st = attn_common(s, q, q_start, n_q, sel, &a, "pkv_chunk_attn_fwd");
    if (st != PKV_OK) return st;
    if (!o || !lse) return fail(PKV_ERR_INVALID, "pkv_chunk_attn_fwd: o or lse is NULL");
    a.o = o; a.lse = lse;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaError_t e = use_tc(s->pool, a) ? launch_attn_fwd_tc(a, cs) : launch_attn_fwd_simt(a, cs);
    if (e == cudaSuccess && s->used) e = cudaEventRecord(s->used, cs);
    if (e != cudaSuccess) return cuda_fail(e, "pkv_chunk_attn_fwd: launch");
    return PKV_OK;
}

static pkv_status ensure_scratch(pkv_pool* p, size_t floats) {
    if (p->scratch_floats >= floats) return PKV_OK;
    // Called outside kernels in flight on the old buffer only after a device sync.
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "scratch grow: sync");
    cudaFree(p->scratch);
    p->scratch = nullptr;
    p->scratch_floats = 0;
    e = cudaMalloc(reinterpret_cast<void**>(&p->scratch), floats * sizeof(float));
    if (e != cudaSuccess) return cuda_fail(e, "scratch grow");
    p->scratch_floats = floats;
    return PKV_OK;
}

pkv_status pkv_chunk_attn_bwd(pkv_seq* s, const void* q, const void* o, const void* dout,
                              const float* lse, int64_t q_start, int64_t n_q, void* dq,
                              const pkv_sel* sel, void* stream) {
    AttnArgs a;
    pkv_status st = attn_common(s, q, q_start, n_q, sel, &a, "pkv_chunk_attn_bwd");
    if (st != PKV_OK) return st;
    if (!o || !dout || !lse || !dq)
        return fail(PKV_ERR_INVALID, "pkv_chunk_attn_bwd: o, dout, lse or dq is NULL");
    // Scratch: D [Hq * n_q] floats; with a selection, the union's page list
    // and (8-byte aligned) the per-(page, KV head) query-page masks.
    const size_t n_d = (size_t)a.Hq * n_q;
    const size_t n_list = sel ? 1 + (size_t)bwd_pagelist_cap(a) : 0;
    const size_t n_mask = sel ? 1 + 2 * (size_t)bwd_selmask_words(a) : 0;
    st = ensure_scratch(s->pool, n_d + n_list + n_mask);
    if (st != PKV_OK) return st;
    a.o_in = o; a.dout = dout; a.lse_in = lse; a.dq = dq; a.Dbuf = s->pool->scratch;
    a.pagelist = sel ? reinterpret_cast<int32_t*>(s->pool->scratch + n_d) : nullptr;
    a.selmask = sel ? reinterpret_cast<uint64_t*>(
                          (reinterpret_cast<uintptr_t>(s->pool->scratch + n_d + n_list) + 7) & ~uintptr_t(7))
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
    if (e == cudaSuccess && s->used) e = cudaEventRecord(s->used, cs);
    if (e != cudaSuccess) return cuda_fail(e, "pkv_chunk_attn_bwd: launch");
    return PKV_OK;
}

pkv_status pkv_grad_zero(pkv_seq* s, void* stream) {
    if (!s) return fail(PKV_ERR_INVALID, "pkv_grad_zero: seq is NULL");
    if (!is_device(s->pool)) return fail(PKV_ERR_INVALID, "pkv_grad_zero: META pool");
    if (s->bt.empty()) return PKV_OK;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (s->pool->desc.residency == PKV_RES_PINNED_HOST) {
        // Host pages are recorded as zero, not written; staged gradients are
        // zeroed in their slots once the last prefetch or write-back is done,
        // and later staging waits for this call.
        e = cudaStreamWaitEvent(cs, s->staged, 0);
        s->gzero_possible = true;
        if (e == cudaSuccess) e = launch_grad_zero_staged(s, cs);
        if (e == cudaSuccess) e = cudaEventRecord(s->used, cs);
    } else {
        e = launch_grad_zero(s->pool, s->d_bt, 0, (int64_t)s->bt.size(), cs);
    }
    if (e != cudaSuccess) return cuda_fail(e, "pkv_grad_zero: launch");
    return PKV_OK;
}

pkv_status pkv_grad_accumulate(pkv_seq* s, int64_t row0, int64_t n_rows, const float* dk,
                               const float* dv, void* stream) {
    if (!s) return fail(PKV_ERR_INVALID, "pkv_grad_accumulate: seq is NULL");
    if (!is_device(s->pool)) return fail(PKV_ERR_INVALID, "pkv_grad_accumulate: META pool");
    if (row0 < 0 || n_rows < 0 || row0 + n_rows > s->len)
        return fail(PKV_ERR_INVALID, "pkv_grad_accumulate: need 0 <= row0 and row0 + n_rows <= length");
    if ((reinterpret_cast<uintptr_t>(dk) | reinterpret_cast<uintptr_t>(dv)) & 15)
        return fail(PKV_ERR_INVALID, "pkv_grad_accumulate: dk and dv must be 16-byte aligned");
    if (n_rows == 0 || (!dk && !dv)) return PKV_OK;
    pkv_status st = check_stream_device(s->pool);
    if (st != PKV_OK) return st;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaError_t e = launch_grad_accumulate(s->pool, s->d_bt, row0, n_rows, dk, dv, cs);
    // A later gradient prefetch of a host pool copies these pages: order it after.
    if (e == cudaSuccess && s->used) e = cudaEventRecord(s->used, cs);
    if (e != cudaSuccess) return cuda_fail(e, "pkv_grad_accumulate: launch");
    return PKV_OK;
}

pkv_status pkv_gather(const pkv_seq* s, void* k, void* v, float* dk, float* dv, float* rep,
                      void* stream) {
    if (!s) return fail(PKV_ERR_INVALID, "pkv_gather: seq is NULL");
    if (!is_device(s->pool)) return fail(PKV_ERR_INVALID, "pkv_gather: META pool");
    if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) |
         reinterpret_cast<uintptr_t>(dk) | reinterpret_cast<uintptr_t>(dv)) & 15)
        return fail(PKV_ERR_INVALID, "pkv_gather: outputs must be 16-byte aligned");
    if (s->len == 0) return PKV_OK;
    cudaError_t e = launch_gather(s->pool, s->d_bt, 0, s->len, k, v, dk, dv, rep,
                                  static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "pkv_gather: launch");
    return PKV_OK;
}

pkv_status pkv_gather_rows(const pkv_seq* s, int64_t row0, int64_t n_rows, void* k, void* v,
                           float* dk, float* dv, void* stream) {
    if (!s) return fail(PKV_ERR_INVALID, "pkv_gather_rows: seq is NULL");
    if (!is_device(s->pool)) return fail(PKV_ERR_INVALID, "pkv_gather_rows: META pool");
    const int64_t P = s->pool->desc.page_size;
    if (row0 < 0 || n_rows < 0 || row0 % P != 0 || row0 + n_rows > s->len)
        return fail(PKV_ERR_INVALID, "pkv_gather_rows: need row0 % P == 0 and row0 + n_rows <= length");
    if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) |
         reinterpret_cast<uintptr_t>(dk) | reinterpret_cast<uintptr_t>(dv)) & 15)
        return fail(PKV_ERR_INVALID, "pkv_gather_rows: outputs must be 16-byte aligned");
    if (n_rows == 0) return PKV_OK;
    cudaError_t e = launch_gather(s->pool, s->d_bt, row0 / P, row0 + n_rows, k, v, dk, dv, nullptr,
                                  static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "pkv_gather_rows: launch");
    return PKV_OK;
}

pkv_status pkv_page_topk(pkv_seq* s, const void* q, int64_t q_start, int64_t n_q, int32_t k,
                         int32_t n_sink, int32_t n_local, int32_t* pages_out,
                         int32_t* counts_out, void* stream) {
    if (!s || !q || !pages_out) return fail(PKV_ERR_INVALID, "pkv_page_topk: NULL argument");
    pkv_pool* p = s->pool;
    if (!is_device(p)) return fail(PKV_ERR_INVALID, "pkv_page_topk: META pool");
    const int64_t P = p->desc.page_size;
    if (n_q <= 0 || q_start < 0 || q_start % P != 0 || q_start + n_q > s->len)
        return fail(PKV_ERR_INVALID, "pkv_page_topk: need q_start % P == 0 and q_start + n_q <= length");
    if (k < 0 || n_sink < 0 || n_local < 1)
        return fail(PKV_ERR_INVALID, "pkv_page_topk: need k >= 0, n_sink >= 0, n_local >= 1 "
                                     "(the query page itself is always visible)");
    const int64_t n_qp = (n_q + P - 1) / P;
    const int64_t last_qpg = q_start / P + n_qp - 1;
    if (last_qpg - n_local - n_sink + 1 > page_topk_max_candidates())
        return fail(PKV_ERR_UNSUPPORTED, "pkv_page_topk: more than " +
                                             std::to_string(page_topk_max_candidates()) +
                                             " candidate pages");
    pkv_status st = check_stream_device(p);
    if (st != PKV_OK) return st;
    const size_t need = page_topk_scratch_floats(q_start, n_q, (int)P, p->desc.n_kv_heads,
                                                 p->desc.head_dim, n_sink, n_local);
    if (p->sel_scratch_floats < need) {
        cudaError_t e = cudaDeviceSynchronize();
        if (e != cudaSuccess) return cuda_fail(e, "pkv_page_topk: sync");
        cudaFree(p->sel_scratch);
        p->sel_scratch = nullptr;
        p->sel_scratch_floats = 0;
        e = cudaMalloc(reinterpret_cast<void**>(&p->sel_scratch), need * sizeof(float));
        if (e != cudaSuccess) return cuda_fail(e, "pkv_page_topk: scratch");
        p->sel_scratch_floats = need;
    }
    cudaError_t e = launch_page_topk(p, s->d_bt, q, q_start, n_q, k, n_sink, n_local, pages_out,
                                     counts_out, p->sel_scratch, p->sel_state,
                                     static_cast<cudaStream_t>(stream));
    // A later pkv_prefetch of this selection must wait for it.
    if (e == cudaSuccess && s->used) e = cudaEventRecord(s->used, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "pkv_page_topk: launch");
    return PKV_OK;
}

pkv_status pkv_page_local(pkv_seq* s, int64_t q_start, int64_t n_q, int32_t n_sink,
                          int32_t n_local, int32_t* pages_out, int32_t* counts_out, void* stream) {
    if (!s || !pages_out) return fail(PKV_ERR_INVALID, "pkv_page_local: NULL argument");
    pkv_pool* p = s->pool;
    if (!is_device(p)) return fail(PKV_ERR_INVALID, "pkv_page_local: META pool");
    const int64_t P = p->desc.page_size;
    if (n_q <= 0 || q_start < 0 || q_start % P != 0 || q_start + n_q > s->len)
        return fail(PKV_ERR_INVALID, "pkv_page_local: need q_start % P == 0 and q_start + n_q <= length");
    if (n_sink < 0 || n_local < 1 || (int64_t)n_sink + n_local > (1 << 20))
        return fail(PKV_ERR_INVALID, "pkv_page_local: need n_sink >= 0 and 1 <= n_local "
                                     "(the query page itself is always visible)");
    pkv_status st = check_stream_device(p);
    if (st != PKV_OK) return st;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaError_t e = launch_page_local(q_start, n_q, (int)P, p->desc.n_kv_heads, n_sink, n_local,
                                      pages_out, counts_out, cs);
    // A later pkv_prefetch of this selection must wait for it.
    if (e == cudaSuccess && s->used) e = cudaEventRecord(s->used, cs);
    if (e != cudaSuccess) return cuda_fail(e, "pkv_page_local: launch");
    return PKV_OK;
}

static pkv_status host_pool_check(pkv_seq* s, const char* who) {
    if (!s) return fail(PKV_ERR_INVALID, std::string(who) + ": seq is NULL");
    if (s->pool->desc.residency != PKV_RES_PINNED_HOST)
        return fail(PKV_ERR_INVALID, std::string(who) + ": the pool is not PINNED_HOST");
    return check_stream_device(s->pool);
}

// Whole-sequence staging with the copy engines instead of copy kernels (no SM
// time taken from the attention kernels running meanwhile): logical page i goes
// to slot i, which is the plan kernel's assignment when every page is staged,
// in one cudaMemcpyAsync per run of consecutive physical pages per array.
static cudaError_t stage_all_dma(pkv_seq* s, int64_t n, int what, bool to_host, cudaStream_t cs) {
    const pkv_pool* p = s->pool;
    const size_t kv_page = p->page_elems * p->elem, g_page = p->page_elems * sizeof(float);
    for (int64_t i0 = 0; i0 < n;) {
        int64_t i1 = i0 + 1;
        while (i1 < n && s->bt[i1] == s->bt[i1 - 1] + 1) ++i1;
        const size_t pp = (size_t)s->bt[i0], len = (size_t)(i1 - i0), slot = (size_t)i0;
        auto cp = [&](void* slots, void* pages, size_t page_bytes) {
            uint8_t* d = static_cast<uint8_t*>(slots) + slot * page_bytes;
            uint8_t* h = static_cast<uint8_t*>(pages) + pp * page_bytes;
            return to_host ? cudaMemcpyAsync(h, d, len * page_bytes, cudaMemcpyDeviceToHost, cs)
                           : cudaMemcpyAsync(d, h, len * page_bytes, cudaMemcpyHostToDevice, cs);
        };
        cudaError_t e = cudaSuccess;
        if (what & PKV_STAGE_KV) {
            e = cp(p->kslot, p->k, kv_page);
            if (e == cudaSuccess) e = cp(p->vslot, p->v, kv_page);
        }
        if (e == cudaSuccess && (what & PKV_STAGE_GRADS)) {
            e = cp(p->dkslot, p->dk, g_page);
            if (e == cudaSuccess) e = cp(p->dvslot, p->dv, g_page);
        }
        if (e != cudaSuccess) return e;
        i0 = i1;
    }
    // Gradient pages recorded as zero: their copies were stale, so their slots
    // get zeros; once written back, the host pages are current.
    if (!(what & PKV_STAGE_GRADS) || !s->gzero_possible) return cudaSuccess;
    if (!to_host) return launch_gzero_fill_slots(s, n, cs);
    cudaError_t e = launch_gzero_clear(s, n, cs);
    if (n >= (int64_t)s->bt.size()) s->gzero_possible = false;   // every page written back
    return e;
}

pkv_status pkv_prefetch(pkv_seq* s, const int32_t* pages, int64_t n, int32_t what, void* side) {
    pkv_status st = host_pool_check(s, "pkv_prefetch");
    if (st != PKV_OK) return st;
    if (n < 0 || (n > 0 && !pages) || !(what & (PKV_STAGE_KV | PKV_STAGE_GRADS)) ||
        (what & ~(PKV_STAGE_KV | PKV_STAGE_GRADS)))
        return fail(PKV_ERR_INVALID, "pkv_prefetch: bad pages/n/what");
    if (s->bt.empty()) return PKV_OK;
    cudaStream_t cs = static_cast<cudaStream_t>(side);
    // Slots are rewritten: wait for the last append/attention call on this
    // sequence and for its last prefetch or writeback (which may have been
    // issued on another stream, e.g. write-backs on a device-to-host stream).
    cudaError_t e = cudaStreamWaitEvent(cs, s->used, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, s->staged, 0);
    const int64_t n_pages = (int64_t)s->bt.size();
    const bool all = n == 0 && n_pages <= s->pool->n_slots;
    if (all) {
        // Whole sequence: slot i <- page i, runs of consecutive physical pages
        // by the copy engines. Dirty gradient slots go back first.
        if (e == cudaSuccess && s->dirty_possible) {
            if (s->staged_all > 0) {
                const int64_t m = std::min<int64_t>(s->staged_all, n_pages);
                e = stage_all_dma(s, m, PKV_STAGE_GRADS, true, cs);
                s->h_stats[2] += m * s->pool->desc.n_kv_heads;
            } else {
                e = launch_stage_writeback(s, true, cs);
            }
        }
        if (e == cudaSuccess) e = launch_stage_identity(s, n_pages, what, cs);
        if (e == cudaSuccess) e = stage_all_dma(s, n_pages, what, false, cs);
        const int64_t ph = n_pages * s->pool->desc.n_kv_heads;
        if (what & PKV_STAGE_KV) s->h_stats[0] += ph;
        if (what & PKV_STAGE_GRADS) s->h_stats[1] += ph;
        s->staged_all = n_pages;
    } else {
        if (e == cudaSuccess && s->staged_all > 0) {
            // Leaving whole-sequence staging: its dirty gradients go back and
            // the cache starts empty.
            if (s->dirty_possible)
                e = stage_all_dma(s, std::min<int64_t>(s->staged_all, n_pages), PKV_STAGE_GRADS, true, cs);
            if (e == cudaSuccess) e = launch_stage_after_writeback(s, true, cs);
            if (s->dirty_possible) s->h_stats[2] += s->staged_all * s->pool->desc.n_kv_heads;
            s->dirty_possible = false;
        }
        s->staged_all = 0;
        if (e == cudaSuccess) e = launch_stage_plan(s, n > 0 ? pages : nullptr, n, what, cs);
        if (e == cudaSuccess) e = launch_stage_copy(s, cs);
    }
    if (what & PKV_STAGE_GRADS) s->dirty_possible = true;
    if (e == cudaSuccess) e = cudaEventRecord(s->staged, cs);
    if (e != cudaSuccess) return cuda_fail(e, "pkv_prefetch");
    return PKV_OK;
}

static pkv_status writeback(pkv_seq* s, void* side, bool release, const char* who) {
    pkv_status st = host_pool_check(s, who);
    if (st != PKV_OK) return st;
    cudaStream_t cs = static_cast<cudaStream_t>(side);
    cudaError_t e = cudaStreamWaitEvent(cs, s->used, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, s->staged, 0);
    if (s->staged_all > 0) {
        const int64_t n = std::min<int64_t>(s->staged_all, (int64_t)s->bt.size());
        if (e == cudaSuccess && s->dirty_possible) {
            e = stage_all_dma(s, n, PKV_STAGE_GRADS, true, cs);
            s->h_stats[2] += n * s->pool->desc.n_kv_heads;
        }
        if (e == cudaSuccess) e = launch_stage_after_writeback(s, release, cs);
        if (release) s->staged_all = 0;
    } else if (e == cudaSuccess) {
        e = launch_stage_writeback(s, release, cs);
    }
    s->dirty_possible = false;
    if (e == cudaSuccess) e = cudaEventRecord(s->staged, cs);
    if (e != cudaSuccess) return cuda_fail(e, who);
    return PKV_OK;
}

pkv_status pkv_writeback_grads(pkv_seq* s, void* side) {
    return writeback(s, side, false, "pkv_writeback_grads");
}

pkv_status pkv_release_slots(pkv_seq* s, void* side) {
    return writeback(s, side, true, "pkv_release_slots");
}

pkv_status pkv_stage_stats(pkv_seq* s, int64_t* kv_in, int64_t* grads_in, int64_t* grads_out) {
    pkv_status st = host_pool_check(s, "pkv_stage_stats");
    if (st != PKV_OK) return st;
    unsigned long long d[3] = {0, 0, 0};
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(d, s->d_stats, sizeof(d), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "pkv_stage_stats");
    if (kv_in) *kv_in = (int64_t)d[0] + s->h_stats[0];
    if (grads_in) *grads_in = (int64_t)d[1] + s->h_stats[1];
    if (grads_out) *grads_out = (int64_t)d[2] + s->h_stats[2];
    return PKV_OK;
}

pkv_status pkv_wait(pkv_seq* s, void* main, int64_t timeout_us) {
    pkv_status st = host_pool_check(s, "pkv_wait");
    if (st != PKV_OK) return st;
    if (timeout_us > 0) {
        // Bounded host poll: never blocks longer than timeout_us.
        const auto t0 = std::chrono::steady_clock::now();
        for (;;) {
            cudaError_t q = cudaEventQuery(s->staged);
            if (q == cudaSuccess) break;
            if (q != cudaErrorNotReady) return cuda_fail(q, "pkv_wait: event");
            const auto us = std::chrono::duration_cast<std::chrono::microseconds>(
                                std::chrono::steady_clock::now() - t0).count();
            if (us > timeout_us)
                return fail(PKV_ERR_TIMEOUT, "pkv_wait: staging not complete after " +
                                                 std::to_string(timeout_us) + " us");
            std::this_thread::sleep_for(std::chrono::microseconds(20));
        }
    }
    cudaError_t e = cudaStreamWaitEvent(static_cast<cudaStream_t>(main), s->staged, 0);
    if (e != cudaSuccess) return cuda_fail(e, "pkv_wait");
    return PKV_OK;
}

pkv_status pkv_selftest_umma(int32_t mode, const void* a, const void* b, float* d, int32_t lbo,
                             int32_t sbo) {
    if (mode < 0 || mode > 4 || !a || !b || !d)
        return fail(PKV_ERR_INVALID, "pkv_selftest_umma: bad argument");
    int* d_err = nullptr;
    cudaError_t e = cudaMalloc(reinterpret_cast<void**>(&d_err), sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "pkv_selftest_umma: alloc");
    cudaMemset(d_err, 0, sizeof(int));
    e = run_selftest_umma(mode, a, b, d, lbo, sbo, d_err);
    int h = 0;
    if (e == cudaSuccess) e = cudaMemcpy(&h, d_err, sizeof(int), cudaMemcpyDeviceToHost);
    cudaFree(d_err);
    if (e != cudaSuccess) return cuda_fail(e, "pkv_selftest_umma");
    if (h) return fail(PKV_ERR_DEVICE_FAULT, "pkv_selftest_umma: device error " + std::to_string(h));
    return PKV_OK;
}

}  // extern "C"
