/*
 * pkv.h -- C ABI of libpkv: paged chunk attention on one GB300 (sm_103a).
 *
 * The operations follow "Out of the Memory Barrier: A Highly Memory Efficient
 * Training System for LLMs with Million-Token Contexts" (OOMB), as described
 * on five web summaries of it:
 *   - chunk-recurrent training: a long sequence is cut into chunks processed
 *     one after another, every chunk attending to all earlier keys plus its
 *     own (gist.science/de §2.A; gist.science/ja §2.1; sciencestack.ai
 *     abstract, Fig. 1 caption);
 *   - a paged memory manager for the KV cache *and its gradients*: fixed-size
 *     pages reached through a block table, no reallocation on append, custom
 *     kernels running forward and backward directly on the cache and adding
 *     dK/dV in place (gist.science/de §2.B; gist.science/fr "Résumé
 *     technique" §2.B; sciencestack.ai Fig. 3 and Fig. 4 captions);
 *   - page-level sparse attention: top-K pages per query page picked by
 *     per-page representative vectors (gist.science/de §2.D; gist.science/nl
 *     "Pagina-niveau Sparse Attention"; sciencestack.ai Fig. 5 caption), and
 *     local attention layers for natively sparse models (gist.science/nl,
 *     same section);
 *   - asynchronous offload of the cache and its gradients to pinned host
 *     memory, overlapped with compute on CUDA streams (gist.science/de §2.C;
 *     gist.science/nl "Asynchrone CPU Offloading"; gist.science/ja §2.3).
 *
 * Conventions
 *   - Every function returns a pkv_status; no exception crosses the ABI.
 *     pkv_last_error() gives a message for the calling thread's last failure.
 *   - Argument errors are detected on the host before anything is launched
 *     (PKV_ERR_INVALID / PKV_ERR_UNSUPPORTED); nothing has been enqueued then.
 *   - Compute calls are asynchronous on the given stream (a cudaStream_t
 *     passed as void*; NULL = the legacy default stream). Device-side errors
 *     (a bounded wait that expired, an out-of-range page index) are recorded
 *     in the pool's device error word and reported by pkv_check().
 *   - "device pointer" = memory the current CUDA device can address
 *     (cudaMalloc, cudaMallocAsync, torch CUDA tensors); the caller owns it
 *     and keeps it alive until the work on the stream is complete.
 *   - Layouts are row-major, innermost dimension last:
 *       Q, O, dO, dQ   [n_q, Hq, d]        pool dtype
 *       K, V (append)  [n_tok, Hkv, d]     pool dtype
 *       LSE            [Hq, n_q]           float32, natural log
 *       K/V pages      [num_phys_pages, Hkv, P, d]  pool dtype (library-owned)
 *       dK/dV pages    [num_phys_pages, Hkv, P, d]  float32  (library-owned)
 *       representatives [num_phys_pages, Hkv, d]    float32  (library-owned)
 *   - Query head h reads KV head h / (Hq / Hkv) (consecutive grouping).
 *   - The softmax scale is 1/sqrt(d); LSE_i = ln sum_j exp(S_ij) of the
 *     scaled logits S_ij = q_i.k_j / sqrt(d).
 *   - A pool and its sequences are not thread-safe: calls on one pool come
 *     from one host thread at a time.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pkv_status {
    PKV_OK = 0,
    PKV_ERR_INVALID = 1,       /* bad argument or call order; nothing launched          */
    PKV_ERR_OOM = 2,           /* page pool (or device memory for the pool) exhausted    */
    PKV_ERR_CUDA = 3,          /* a CUDA runtime call failed (message has the CUDA error)*/
    PKV_ERR_TIMEOUT = 4,       /* a bounded host wait expired                            */
    PKV_ERR_DEVICE_FAULT = 5,  /* a kernel recorded an error in the device error word    */
    PKV_ERR_UNSUPPORTED = 6    /* no kernel for this dtype/shape combination             */
} pkv_status;

typedef enum pkv_dtype { PKV_BF16 = 0, PKV_F32 = 1 } pkv_dtype;

typedef enum pkv_residency {
    PKV_RES_DEVICE = 0,        /* pages in HBM                                           */
    PKV_RES_PINNED_HOST = 1,   /* pages in pinned host memory, streamed to device slots  */
    PKV_RES_META = 2           /* no page memory: block-table and free-list logic only   */
} pkv_residency;

/* Pool flags. */
#define PKV_FLAG_SIMT_ONLY 1u  /* use the CUDA-core kernels even where tensor-core ones exist */

typedef struct pkv_pool_desc {
    int32_t page_size;         /* P, tokens per page; multiple of 8                      */
    int32_t n_kv_heads;        /* Hkv                                                    */
    int32_t n_q_heads;         /* Hq, a multiple of Hkv                                  */
    int32_t head_dim;          /* d; 64 or 128 (tensor-core path: 128)                   */
    int32_t dtype;             /* pkv_dtype of K/V pages and of Q/O/dO/dQ                */
    int32_t residency;         /* pkv_residency                                          */
    int64_t num_phys_pages;    /* pages in the pool                                      */
    int64_t n_device_slots;    /* PINNED_HOST: device page slots for streamed pages      */
    uint32_t flags;            /* PKV_FLAG_*                                             */
    int32_t reserved;
} pkv_pool_desc;

typedef struct pkv_pool pkv_pool;
typedef struct pkv_seq pkv_seq;

/* A page selection for the sparse variant (written by pkv_page_topk or
 * pkv_page_local, or by the caller in the same format).
 * pages: device int32 [n_qp, Hkv, kmax]; entry (qp, h, :) lists the logical
 * pages visible to the chunk's query page qp through KV head h, ascending,
 * padded with -1. The last listed page of every row is the query page itself. */
typedef struct pkv_sel {
    const int32_t* pages;
    int32_t kmax;
    int32_t reserved;
    int64_t n_qp;
} pkv_sel;

/* ---------------------------------------------------------------- errors */

/* Message of the calling thread's last failed call ("" if none). Never NULL. */
const char* pkv_last_error(void);

/* Reads and clears the pool's device error word (synchronizes the device).
 * PKV_ERR_DEVICE_FAULT if a kernel recorded an error since the last check. */
pkv_status pkv_check(pkv_pool* pool);

/* ---------------------------------------------------------------- pool (a1)
 * Paged KV cache and paged KV-gradient pool (gist.science/de §2.B;
 * sciencestack.ai Fig. 3, Fig. 4). The library allocates all page memory at
 * creation, once: appends never allocate device memory. */

/* Creates a pool on the current CUDA device. Validates desc; PKV_ERR_OOM if
 * the page memory cannot be allocated. *out is NULL on failure. Synchronous
 * (synchronizes the device): the pool is fully initialised on return. */
pkv_status pkv_pool_create(const pkv_pool_desc* desc, pkv_pool** out);

/* Frees everything the pool owns, including its sequences. NULL-safe.
 * Work on the pool's memory must be complete. */
void pkv_pool_destroy(pkv_pool* pool);

/* Number of physical pages currently free. */
pkv_status pkv_pool_free_pages(const pkv_pool* pool, int64_t* n_free);

/* Device addresses of the pool's arrays (layouts above); any may be NULL.
 * For tests and for callers that read pages directly. For PINNED_HOST pools
 * these are host addresses of the pinned pages; there a gradient page that
 * was zeroed (pkv_grad_zero, or fresh from pkv_append) holds stale memory
 * until it is written back or accumulated into (pkv_gather reads it right). */
pkv_status pkv_pool_arrays(const pkv_pool* pool, void** k, void** v, float** dk,
                           float** dv, float** rep);

/* ---------------------------------------------------------------- sequences */

/* A sequence (one layer's KV of one sample) with an empty block table.
 * Synchronous (synchronizes the device). */
pkv_status pkv_seq_create(pkv_pool* pool, pkv_seq** out);

/* Returns the sequence's pages to the free list and frees it. NULL-safe.
 * Work on its pages must be complete (or ordered before later reuse on the
 * same stream). */
void pkv_seq_free(pkv_seq* seq);

/* Returns all pages to the free list; the sequence becomes empty. */
pkv_status pkv_seq_reset(pkv_seq* seq);

/* Current length in tokens. */
pkv_status pkv_seq_length(const pkv_seq* seq, int64_t* len);

/* Claims pages for n_tok more tokens (block-table growth only; no data is
 * written). PKV_ERR_OOM, with nothing claimed, if too few pages are free.
 * pkv_append calls this itself. */
pkv_status pkv_seq_reserve(pkv_seq* seq, int64_t n_tok);

/* Host copy of the block table: out[p] = physical page of logical page p.
 * *n = number of logical pages; at most cap entries are written. */
pkv_status pkv_get_block_table(const pkv_seq* seq, int32_t* out, int64_t cap, int64_t* n);

/* Pre-assigns physical pages bt[0..n) to logical pages 0..n-1 of an EMPTY
 * sequence (e.g. a seeded permutation). Every entry must be a free page of the
 * pool and appear once; otherwise PKV_ERR_INVALID and nothing changes. Later
 * appends fill these pages first. Synchronous. */
pkv_status pkv_set_block_table(pkv_seq* seq, const int32_t* bt, int64_t n);

/* ---------------------------------------------------------------- append (a2)
 * Writes n_tok new tokens' keys and values (device [n_tok, Hkv, d], pool
 * dtype) at positions len..len+n_tok-1 through the block table, claiming
 * pages as needed. In the same kernel it
 *   - recomputes the representative (fp32 mean of the stored keys, over the
 *     rows the page holds) of every page it touches (gist.science/de §2.D
 *     "repräsentative Vektoren");
 *   - zero-fills the rows of a partial last page beyond the new length;
 *   - zeroes the dK/dV gradient rows of every newly claimed page, so a page
 *     starts with zero gradient.
 * The current length must be a multiple of P unless it is the first append
 * after a partial page (then the partial page is completed first). */
pkv_status pkv_append(pkv_seq* seq, const void* k, const void* v, int64_t n_tok, void* stream);

/* ---------------------------------------------------------------- attention (a3, a4, a6)
 * One query chunk: queries at positions q_start..q_start+n_q-1, with
 * q_start % P == 0 and q_start + n_q <= the sequence length (the chunk's own
 * keys already appended; keys of later chunks may be in the pool too, as in
 * the backward sweep, and are never visible). Dense (sel == NULL): query i
 * sees keys 0..i.
 * Sparse (sel != NULL, from pkv_page_topk for this chunk): query i in the
 * chunk's query page qp sees the keys of the pages listed for (qp, h/g),
 * causally masked on its own page. */

/* O [n_q, Hq, d] (pool dtype) and LSE [Hq, n_q] float32. */
pkv_status pkv_chunk_attn_fwd(pkv_seq* seq, const void* q, int64_t q_start, int64_t n_q,
                              void* o, float* lse, const pkv_sel* sel, void* stream);

/* Recomputes P from LSE; writes dQ [n_q, Hq, d] (pool dtype) and ADDS this
 * chunk's dK/dV into the sequence's fp32 gradient pages (never zeroes them).
 * o and lse are the forward's outputs for the same chunk; dout is dL/dO.
 * Uses a pool-owned scratch buffer of Hq*n_q floats, plus, with a selection,
 * the list of the chunk's selected pages and, per (key page, KV head), a
 * bitmask of the query pages that list the page (grown on demand). */
pkv_status pkv_chunk_attn_bwd(pkv_seq* seq, const void* q, const void* o, const void* dout,
                              const float* lse, int64_t q_start, int64_t n_q, void* dq,
                              const pkv_sel* sel, void* stream);

/* pkv_chunk_attn_bwd without any allocation. Same arguments, outputs and
 * results as pkv_chunk_attn_bwd; the paper has no counterpart: it exists for
 * callers that cannot let the library allocate device memory at call time
 * (a fixed memory budget, an allocator that owns all device memory, code that
 * must not synchronize the device, loops that forbid allocation after
 * start-up). The per-row scratch lives in one fixed array of 262144 floats
 * (1 MiB) in the library's device image, held on every device that loads the
 * library until exit; a call needs n_q_heads * n_q floats (with a page
 * selection, plus 1 + min(key pages, n_qp * n_kv_heads * kmax) entries for
 * the list of selected pages) and is rejected
 * with PKV_ERR_INVALID above that. With a selection it also places, when they
 * fit, the query-page bitmasks (1 + 2 * key pages * n_kv_heads *
 * ceil(n_qp / 64) entries) there; when they do not, the dK/dV kernel finds
 * each page's query pages by scanning the selection (the same results). The first call on a device looks up the
 * array's device address (no allocation) and should come before any stream
 * capture. All calls share the array: calls that overlap on the GPU race and
 * must be serialised by the caller. Each call rewrites what it reads, so
 * nothing needs clearing between calls. Like pkv_chunk_attn_bwd it marks the
 * sequence as used on `stream`, so pkv_prefetch and pkv_writeback_grads on a
 * side stream wait for it before touching the staged slots. */
pkv_status pkv_chunk_attn_bwd_noalloc(pkv_seq* seq, const void* q, const void* o,
                                      const void* dout, const float* lse, int64_t q_start,
                                      int64_t n_q, void* dq, const pkv_sel* sel, void* stream);

/* Zeroes the gradient pages of the sequence's pages. For a PINNED_HOST pool
 * nothing is written over the host link: every (page, KV head) of the
 * sequence is recorded as zero in HBM (staging then fills slots with zeros
 * instead of copying, pkv_gather reads zeros, pkv_grad_accumulate writes the
 * whole page), and gradients already staged in the sequence's slots are
 * zeroed there, after its last prefetch or write-back; later staging waits
 * for this call. A write-back of the page makes its host memory current. */
pkv_status pkv_grad_zero(pkv_seq* seq, void* stream);

/* Adds contiguous float32 gradients into the sequence's gradient pages:
 * for rows r in [row0, row0 + n_rows) (any row0 >= 0, row0 + n_rows <= length)
 * and KV heads h, dK_pool[r, h, :] += dk[r - row0, h, :], and likewise dv;
 * dk/dv are caller-owned buffers [n_rows, Hkv, d], 16-byte aligned, either
 * may be NULL. One float32 addition per element, in stream order, no
 * atomics: the result is exact and deterministic. The gradient pages are the
 * paged, in-place accumulated dK/dV of "Out of the Memory Barrier"
 * (gist.science/de §2.B "Paged Memory Management"); this call lets gradients
 * of the cached keys computed elsewhere join them, and is the plain
 * read-modify-write stream of that pool (12 bytes of HBM per element).
 * For a PINNED_HOST pool it adds into the host gradient pages, so it must not
 * run while those pages are staged in device slots (the write-back would
 * overwrite the sum); a later gradient prefetch is ordered after it.
 * PKV_ERR_INVALID for a bad range or misaligned buffer. */
pkv_status pkv_grad_accumulate(pkv_seq* seq, int64_t row0, int64_t n_rows, const float* dk,
                               const float* dv, void* stream);

/* Copies the sequence's pages in logical order into contiguous device
 * buffers [len, Hkv, d] (k, v, dk, dv 16-byte aligned, else PKV_ERR_INVALID):
 * any of the outputs may be NULL. k/v in pool dtype,
 * dk/dv float32, rep [n_pages, Hkv, d] float32. For tests and for handing
 * dK/dV to the K/V projections. */
pkv_status pkv_gather(const pkv_seq* seq, void* k, void* v, float* dk, float* dv, float* rep,
                      void* stream);

/* The rows [row0, row0 + n_rows) of pkv_gather (row0 a multiple of the page
 * size, row0 + n_rows <= length) into buffers [n_rows, Hkv, d] whose row 0
 * is logical row row0; any output may be NULL. In a backward sweep over the
 * chunks in reverse, a chunk's dK/dV rows are final once its own backward has
 * run, so they can leave the GPU while earlier chunks are still computed.
 * PKV_ERR_INVALID for a bad range. */
pkv_status pkv_gather_rows(const pkv_seq* seq, int64_t row0, int64_t n_rows, void* k, void* v,
                           float* dk, float* dv, void* stream);

/* ---------------------------------------------------------------- page selection (a5)
 * For every query page qp of the chunk (P tokens, the last one possibly
 * partial) and KV head h:
 *   qbar  = mean of the chunk's queries over the page's tokens and the g
 *           query heads of the group (fp32);
 *   score = qbar . rep[page] for candidate pages n_sink .. qp_glob-n_local;
 *   keep the K highest scores (ties: lower page first), plus the sink pages
 *   [0, n_sink) and the local pages qp_glob-n_local+1 .. qp_glob.
 * Writes pages_out (device int32 [n_qp, Hkv, K+n_sink+n_local], ascending,
 * -1 padded) and, if counts_out is not NULL, counts_out (device int32
 * [n_qp, Hkv]). q_start and n_q as for attention. One kernel launch; it
 * works in a pool-owned scratch buffer (grown on demand, which synchronizes
 * the device) and the pool's selection counters, so selection calls on one
 * pool must not overlap on the GPU. At most 2^24 candidate pages per query
 * page, else PKV_ERR_UNSUPPORTED. */
pkv_status pkv_page_topk(pkv_seq* seq, const void* q, int64_t q_start, int64_t n_q, int32_t k,
                         int32_t n_sink, int32_t n_local, int32_t* pages_out,
                         int32_t* counts_out, void* stream);

/* Page lists of a local attention layer: natively sparse models use local
 * attention layers instead of a page scorer ("Out of the Memory Barrier",
 * gist.science/nl "Pagina-niveau Sparse Attention"). Page granular: query page
 * qp_glob of the chunk sees the sink pages [0, n_sink) and the local pages
 * qp_glob-n_local+1 .. qp_glob (causal inside its own page), the same list
 * for every KV head. Writes pages_out (device int32 [n_qp, Hkv,
 * n_sink+n_local], ascending, -1 padded) and, if not NULL, counts_out (device
 * int32 [n_qp, Hkv]) in the format pkv_page_topk writes, so the attention
 * calls and pkv_prefetch take it as a selection. Reads neither queries nor
 * representatives. q_start and n_q as for attention; n_sink >= 0,
 * n_local >= 1, else PKV_ERR_INVALID. */
pkv_status pkv_page_local(pkv_seq* seq, int64_t q_start, int64_t n_q, int32_t n_sink,
                          int32_t n_local, int32_t* pages_out, int32_t* counts_out, void* stream);

/* ---------------------------------------------------------------- host offload (a7)
 * For PINNED_HOST pools the K/V pages and their fp32 gradient pages live in
 * mapped pinned host memory (appends write them there; pkv_gather and
 * pkv_grad_accumulate work on them) and the pool owns n_device_slots page
 * slots in HBM; page representatives stay in HBM. Gradient pages known to be
 * zero (fresh from an append, or after pkv_grad_zero) are recorded as such in
 * HBM instead of being written: staging fills their slots with zeros, so they
 * cross the host link only when written back. Attention calls on such a pool read
 * the slots, so the pages a call needs must be staged first. One sequence
 * of the pool uses the slots at a time (one pool per layer to prefetch layer
 * l+1 while layer l computes).
 *
 * pkv_prefetch: on stream `side`, after the sequence's last append, page
 * selection or attention call (an internal event; a page list produced by
 * anything else must already be ordered before `side`), stages the logical
 * pages listed in
 * device int32 logical_pages[0..n) -- duplicates and -1 entries are ignored,
 * so a selection array from pkv_page_topk can be passed flattened -- or every
 * page of the sequence if logical_pages is NULL (n = 0). Pages get slots in
 * ascending page order; what = PKV_STAGE_KV copies K and V, PKV_STAGE_GRADS
 * copies dK and dV (or both). Kernels copy the pages over the host link;
 * nothing is allocated and the host does not wait.
 * The slots of a sequence are a cache: a listed page that is already staged
 * keeps its slot and gets only the contents it lacks, so consecutive chunks
 * whose selections overlap move only the difference. A page not staged takes
 * an empty slot, else the slot of a page this call does not list (evicted:
 * if its gradients were staged, they go back to the host first). More listed
 * pages than slots: the excess is not staged and records
 * PKV_ERR_DEVICE_FAULT for pkv_check. Staged gradients are the authoritative
 * copy until written back: host-side gradient calls (pkv_gather,
 * pkv_grad_accumulate) see them only after pkv_writeback_grads or
 * pkv_release_slots (pkv_grad_zero zeroes them in place). Whole-sequence staging (logical_pages NULL, when the
 * sequence fits the slots) puts page i in slot i and copies with the copy
 * engines; it first writes back gradients still staged.
 * pkv_writeback_grads: on `side`, after the sequence's last attention call,
 * copies the dK/dV of every slot whose gradients were staged since the last
 * write-back into the host gradient pages; the pages stay staged.
 * pkv_release_slots: the same write-back, then empties the sequence's slot
 * cache (the next prefetch stages every page it lists).
 * A prefetch also waits for the sequence's previous prefetch or writeback, so
 * write-backs may go on their own stream (both copy directions at once).
 * pkv_wait: makes stream `main` wait (on the GPU) for the sequence's last
 * prefetch or writeback; with timeout_us > 0 the host first polls for its
 * completion and returns PKV_ERR_TIMEOUT, enqueuing nothing, after
 * timeout_us microseconds. */
#define PKV_STAGE_KV 1
#define PKV_STAGE_GRADS 2
pkv_status pkv_prefetch(pkv_seq* seq, const int32_t* logical_pages, int64_t n, int32_t what,
                        void* side);
pkv_status pkv_writeback_grads(pkv_seq* seq, void* side);
pkv_status pkv_release_slots(pkv_seq* seq, void* side);
pkv_status pkv_wait(pkv_seq* seq, void* main, int64_t timeout_us);

/* Page-heads (one logical page of one KV head) the sequence's staging has
 * moved so far: K/V host-to-device, dK/dV host-to-device, dK/dV
 * device-to-host (write-backs and evictions). Gradient pages recorded as
 * zero that the slot cache fills with zeros in HBM are not counted as moved
 * (whole-sequence staging by the copy engines counts every page it copies).
 * Any output may be NULL.
 * Synchronizes the device. PINNED_HOST pools only (else PKV_ERR_INVALID). */
pkv_status pkv_stage_stats(pkv_seq* seq, int64_t* kv_in, int64_t* grads_in, int64_t* grads_out);

/* ---------------------------------------------------------------- profiling
 * Per-kernel device time, for benchmarks. pkv_profile_enable(1) clears old
 * records and makes every later kernel launch record a CUDA event pair on its
 * stream; pkv_profile_enable(0) stops recording. pkv_profile_collect waits for
 * the recorded events, writes up to max_kernels entries in order of first
 * launch -- names (64-byte NUL-terminated slots), summed milliseconds, launch
 * counts -- sets *n_kernels to the number of distinct kernels, and clears the
 * records. */
pkv_status pkv_profile_enable(int32_t on);
pkv_status pkv_profile_collect(int32_t max_kernels, char* names, double* total_ms,
                               int64_t* launches, int32_t* n_kernels);

/* ---------------------------------------------------------------- self-test
 * Runs one 128x128x64 bf16 tensor-core product (tcgen05, fp32 accumulator
 * in tensor memory) with the shared-memory operand layouts the attention
 * kernels use, synchronously on the current device, and writes
 * d [128,128] float32. Operands are device bf16 arrays:
 *   mode 0: a [128(M), 64(K)], b [128(N), 64(K)]  (both K-major): d = a . b^T
 *   mode 1: a [128(M), 64(K)], b [64(K), 128(N)]  (B MN-major):   d = a . b
 *   mode 2: a [64(K), 128(M)], b [64(K), 128(N)]  (both MN-major): d = a^T . b
 *   mode 3: a [128(M), 64(K)] placed in tensor memory, b [64(K), 128(N)]
 *           (B MN-major): d = a . b
 *   mode 4: issues no MMA, so the kernel's bounded wait for it expires (after
 *           about 4 s) and must return PKV_ERR_DEVICE_FAULT with the device
 *           in a usable state: the failure path of every kernel wait.
 * lbo/sbo override the MN-major descriptor byte offsets (0 = library
 * default). PKV_ERR_DEVICE_FAULT if a bounded wait expired. */
pkv_status pkv_selftest_umma(int32_t mode, const void* a, const void* b, float* d,
                             int32_t lbo, int32_t sbo);

#ifdef __cplusplus
}
#endif
#endif /* PKV_H */
