// Host-side structures and kernel-launcher declarations shared by the C-ABI
// layer (api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>
#include <vector>

#include "../../include/pkv.h"

struct pkv_pool {
    pkv_pool_desc desc{};
    int device = 0;
    size_t elem = 2;                 // bytes per K/V element
    size_t page_elems = 0;           // Hkv * P * d: one physical page of K (or V)
    // Page memory (device for DEVICE pools, pinned host for PINNED_HOST pools).
    void* k = nullptr;
    void* v = nullptr;
    float* dk = nullptr;
    float* dv = nullptr;
    float* rep = nullptr;            // [num_phys, Hkv, d]
    int* d_err = nullptr;            // device error word
    std::vector<int32_t> free_list;  // stack of free physical pages (top = back)
    std::vector<uint8_t> in_use;     // per physical page
    std::vector<pkv_seq*> seqs;
    // Scratch (bwd row statistics D = rowsum(dO * O)), grown on demand.
    float* scratch = nullptr;
    size_t scratch_floats = 0;
    // Scratch of the page selection (partial page queries and scores), and
    // its work-queue counters (zeroed at creation; each call leaves them zero).
    float* sel_scratch = nullptr;
    size_t sel_scratch_floats = 0;
    int* sel_state = nullptr;
    // TMA descriptors over the K and V page pools (2-D: rows x d), with boxes
    // of 64 columns x 128 rows (whole pages). For a PINNED_HOST pool they
    // describe the device slots.
    CUtensorMap tmap_k{}, tmap_v{}, tmap_dk{}, tmap_dv{};
    bool tmaps_ready = false;
    // PINNED_HOST pools: k/v/dk/dv above are mapped pinned host pages; the
    // attention kernels read these device slots instead.
    int64_t n_slots = 0;
    void* kslot = nullptr;
    void* vslot = nullptr;
    float* dkslot = nullptr;
    float* dvslot = nullptr;
    // PINNED_HOST pools: per (physical page, KV head), 1 = the page's dK/dV
    // are zero and its host memory is stale (set by gradient zeroing and by
    // appends of fresh pages instead of writing zeros over the host link;
    // cleared by whatever writes the whole tile: write-backs, accumulation).
    uint8_t* gzero = nullptr;
};

struct pkv_seq {
    pkv_pool* pool = nullptr;
    std::vector<int32_t> bt;         // host block table
    int64_t n_reserved_pages = 0;    // pages pre-assigned by pkv_set_block_table not yet filled
    int32_t* h_bt = nullptr;         // pinned mirror the upload kernel reads (mapped)
    int32_t* h_bt_dev = nullptr;     // the mirror's device-side address (mapped)
    int32_t* d_bt = nullptr;         // device block table, capacity num_phys_pages
    // Recorded after every asynchronous upload from h_bt: entries already sent
    // are rewritten (after a reset) only once the last upload has executed.
    cudaEvent_t bt_sent = nullptr;
    bool bt_pending = false;
    int64_t len = 0;
    // PINNED_HOST pools: the slot cache (device), capacity num_phys_pages.
    int32_t* d_slot_of = nullptr;    // logical page -> device slot, or -1
    int32_t* d_slot_page = nullptr;  // device slot -> logical page or -1 [n_slots]
    int32_t* d_slot_state = nullptr; // kSlot* bits per slot [n_slots]
    int32_t* d_avail = nullptr;      // planning scratch [n_slots]
    int4* d_jobs = nullptr;          // copy jobs of the last plan [n_slots]
    int32_t* d_flags = nullptr;      // planning scratch [num_phys_pages + 1]; [num_phys_pages] = job count
    unsigned long long* d_stats = nullptr;   // page-heads moved by kernels: K/V in, grads in, grads out
    int64_t h_stats[3] = {0, 0, 0};  // the same, moved by the copy engines (whole-sequence staging)
    bool dirty_possible = false;     // a prefetch staged gradients since the last write-back
    bool gzero_possible = false;     // some page may be recorded as zero (pool gzero) since the
                                     // last whole-sequence write-back
    cudaEvent_t staged = nullptr;    // last event recorded on the side stream
    cudaEvent_t used = nullptr;      // last append/attention call on the sequence's slots
    int64_t staged_all = 0;          // > 0: the last prefetch staged pages [0, staged_all), slot i = page i
};

// Slot state bits (PINNED_HOST pools). KV and G match PKV_STAGE_KV and
// PKV_STAGE_GRADS.
enum : int { kSlotKV = 1, kSlotG = 2, kSlotDirty = 4, kSlotKeep = 8 };

namespace pkv {

// Brackets one kernel launch with CUDA events on its stream while profiling
// is enabled (pkv_profile_enable); a no-op otherwise.
struct ProfScope {
    ProfScope(const char* name, cudaStream_t s);
    ~ProfScope();
    ProfScope(const ProfScope&) = delete;
    ProfScope& operator=(const ProfScope&) = delete;
    const char* name;
    cudaStream_t s;
    cudaEvent_t a = nullptr, b = nullptr;
    bool active = false;
};

// Sets the thread's last-error message and returns the status.
pkv_status fail(pkv_status s, const std::string& msg);
pkv_status cuda_fail(cudaError_t e, const char* what);

struct AppendArgs {
    int P, Hkv, d, dtype;
    const void* k_in;
    const void* v_in;
    void* kpool;
    void* vpool;
    float* dkpool;
    float* dvpool;
    float* rep;
    const int32_t* bt;
    int64_t num_phys;
    int64_t old_len, n_tok;
    uint8_t* gzero;              // PINNED_HOST: record fresh gradient pages as zero
    int* err;
};
cudaError_t launch_append(const AppendArgs& a, cudaStream_t s);

// dst[i] = src[i], i < n, src in mapped pinned host memory (no copy engine).
cudaError_t launch_bt_upload(const int32_t* src, int32_t* dst, int64_t n, cudaStream_t s);
// Zero the gradient rows of the given logical pages range [p0, p1).
cudaError_t launch_grad_zero(const pkv_pool* pool, const int32_t* d_bt, int64_t p0, int64_t p1,
                             cudaStream_t s);
// Contiguous fp32 rows [row0, row0 + n_rows) x Hkv x d added into the gradient pages.
cudaError_t launch_grad_accumulate(const pkv_pool* pool, const int32_t* d_bt, int64_t row0,
                                   int64_t n_rows, const float* dk, const float* dv,
                                   cudaStream_t s);
// Logical pages [lp0, ceil(len / P)) -> outputs starting at row lp0 * P.
cudaError_t launch_gather(const pkv_pool* pool, const int32_t* d_bt, int64_t lp0, int64_t len,
                          void* k, void* v, float* dk, float* dv, float* rep, cudaStream_t s);

struct AttnArgs {
    int P, Hq, Hkv, d, dtype;
    int64_t q_start, n_q;            // keys 0 .. q_start + n_q - 1
    const void* q;
    const void* o_in;                // bwd: forward output
    const void* dout;                // bwd: dL/dO
    const float* lse_in;             // bwd: forward LSE
    void* o;                         // fwd out
    float* lse;                      // fwd out
    void* dq;                        // bwd out
    float* Dbuf;                     // bwd scratch [Hq, n_q]
    int32_t* pagelist;               // bwd scratch with a selection: [1 + bwd_pagelist_cap(a)]
    uint64_t* selmask;               // bwd scratch with a selection, or null: [bwd_selmask_words(a)]
    const void* kpool;
    const void* vpool;
    float* dkpool;
    float* dvpool;
    const int32_t* bt;
    int64_t num_phys;
    const int32_t* sel;              // sparse: [n_qp, Hkv, kmax] or null
    int kmax;
    int* err;
    const CUtensorMap* tmap_k;       // tensor-core path only: whole-page boxes
    const CUtensorMap* tmap_v;
    const CUtensorMap* tmap_dk;      // tensor-core path only: fp32 gradient rows,
    const CUtensorMap* tmap_dv;      // boxes of 32 columns x 128 rows (reduce-add)
};

// Validates the arguments shared by the attention entry points and fills a
// with the sequence's pools, block table (or slot table for PINNED_HOST pools),
// tensor maps and selection. Host-only; returns PKV_OK or an error with the
// last-error message set, naming `who`.
pkv_status attn_common(pkv_seq* s, const void* q, int64_t q_start, int64_t n_q,
                       const pkv_sel* sel, AttnArgs* a, const char* who);
// True when the tensor-core kernels take this call.
bool use_tc(const pkv_pool* p, const AttnArgs& a);

cudaError_t launch_attn_fwd_simt(const AttnArgs& a, cudaStream_t s);
cudaError_t launch_attn_bwd_simt(const AttnArgs& a, cudaStream_t s);
cudaError_t launch_bwd_rowdot(const AttnArgs& a, cudaStream_t s);

// Page selection of one chunk in one launch (topk_fused_kernel). scratch:
// page_topk_scratch_floats() floats; state: page_topk_state_ints(Hkv) ints,
// zero before the first call (each call leaves it zero again).
cudaError_t launch_page_topk(const pkv_pool* p, const int32_t* d_bt, const void* q,
                             int64_t q_start, int64_t n_q, int K, int n_sink, int n_local,
                             int32_t* out, int32_t* counts, float* scratch, int* state,
                             cudaStream_t s);
int64_t page_topk_max_candidates();
int page_topk_state_ints(int Hkv);
cudaError_t launch_page_local(int64_t q_start, int64_t n_q, int P, int Hkv, int n_sink,
                              int n_local, int32_t* out, int32_t* counts, cudaStream_t s);
// Floats of page-selection scratch: page queries [n_qp, Hkv, d], then scores
// [Hkv, n_qp, candidates rounded up to 4].
size_t page_topk_scratch_floats(int64_t q_start, int64_t n_q, int P, int Hkv, int D, int n_sink,
                                int n_local);

// Host offload (stream.cu): the slot cache of a PINNED_HOST sequence.
// Plan the staging of `pages` (null: every page) with contents `want`.
cudaError_t launch_stage_plan(const pkv_seq* s, const int32_t* pages, int64_t n, int want,
                              cudaStream_t st);
// Run the copy jobs of the last plan.
cudaError_t launch_stage_copy(const pkv_seq* s, cudaStream_t st);
// Dirty gradient slots back to the host pages (release: then empty the cache).
cudaError_t launch_stage_writeback(const pkv_seq* s, bool release, cudaStream_t st);
// The slot-state update that follows a write-back done by the copy engines.
cudaError_t launch_stage_after_writeback(const pkv_seq* s, bool release, cudaStream_t st);
// Whole-sequence staging: slot i <- logical page i for i < n_pages.
cudaError_t launch_stage_identity(const pkv_seq* s, int64_t n_pages, int want, cudaStream_t st);
// The partial page lp was extended by an append: its staged K/V is stale.
cudaError_t launch_stage_invalidate_kv(const pkv_seq* s, int64_t lp, cudaStream_t st);
// Gradient zeroing of a PINNED_HOST sequence: every (page, KV head) of its
// block table is recorded as zero, and gradients staged in its slots are zeroed.
cudaError_t launch_grad_zero_staged(const pkv_seq* s, cudaStream_t st);
// After the copy engines staged the gradients of logical pages [0, n) into
// slots 0..n-1: zero the slots of pages recorded as zero.
cudaError_t launch_gzero_fill_slots(const pkv_seq* s, int64_t n, cudaStream_t st);
// After the copy engines wrote the gradients of slots 0..n-1 back to logical
// pages [0, n): those host pages are current again.
cudaError_t launch_gzero_clear(const pkv_seq* s, int64_t n, cudaStream_t st);

bool tc_supported(const AttnArgs& a);
cudaError_t launch_attn_fwd_tc(const AttnArgs& a, cudaStream_t s);
// Entries of the backward's page-list scratch for a call with a selection:
// at most every key page, at most every listed entry (0 without a selection).
int64_t bwd_pagelist_cap(const AttnArgs& a);
// Words of the backward's per-(key page, KV head) masks of the query pages
// whose selection lists the page (ceil(n_qp / 64) words each); 0 without a
// selection. They replace a scan of the whole selection by every dK/dV CTA.
int64_t bwd_selmask_words(const AttnArgs& a);
cudaError_t launch_attn_bwd_tc(const AttnArgs& a, cudaStream_t s);

// TMA descriptor helpers (driver entry point fetched through the runtime).
bool make_tmap_2d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, uint64_t inner,
                  uint64_t rows, uint64_t row_stride_bytes, uint32_t box_inner,
                  uint32_t box_rows, std::string* why);
bool make_tmap_3d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, uint64_t d0,
                  uint64_t d1, uint64_t d2, uint64_t stride1_bytes, uint64_t stride2_bytes,
                  uint32_t b0, uint32_t b1, uint32_t b2, std::string* why);

cudaError_t run_selftest_umma(int mode, const void* a, const void* b, float* d, int lbo, int sbo,
                              int* d_err);

}  // namespace pkv
