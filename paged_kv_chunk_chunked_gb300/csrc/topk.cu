// Page-level top-K selection for sparse attention ("Out of the Memory
// Barrier", gist.science/de §2.D: a Top-K procedure finds the most relevant KV
// pages from representative vectors; gist.science/nl: one representative
// vector per page; sciencestack.ai Fig. 5: retrieved key pages per query page).
//
// For every query page qp of the chunk and KV head h:
//   qbar  = mean of the chunk's queries over the page's tokens and the g query
//           heads reading KV head h (fp32);
//   score = qbar . rep[bt[p], h] for candidate pages p in [n_sink, qpg - n_local]
//           (qpg = the query page's index in the sequence);
//   keep the K best by (score descending, page ascending), plus the sink pages
//   [0, n_sink) and the local pages qpg-n_local+1 .. qpg; write them ascending,
//   padded with -1.
//
// One persistent launch per chunk (topk_fused_kernel). Its CTAs take work
// units from a queue in order, in three kinds, each kind per KV head:
//   A  the page query of one (query page, KV head): the mean of the page's
//      rows over the group's g heads, 16-byte loads, all of a thread's loads
//      in flight at once. Together the A units read the chunk's queries
//      once: this is the HBM stream of the chain.
//   B  scores of a tile of 32 candidate pages against every query page of the
//      chunk (the representatives transposed in shared memory), fp32 FMAs;
//      each representative leaves L2 once per chunk.
//   C  the selection of one (query page, KV head): a radix select of the K-th
//      best score over order-preserving 32-bit keys (digits of 11, 11 and 10
//      bits over the score row, staged in shared memory when it fits), then an
//      ordered compaction (ties at the threshold go to the lower pages).
// A B unit of head h waits until every A unit of h is done, a C unit until
// every B unit of h is; the queue holds every A unit, then every B unit, then
// every C unit. A CTA takes a unit only when it has finished the previous one,
// so a unit waits only on units earlier in the queue that running CTAs hold:
// any grid size is free of deadlock, and every wait is bounded. The last CTA
// to leave resets the queue and counters for the next call. Calls that share
// a pool's selection scratch must not overlap on the GPU.
#include <cuda_bf16.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace pkv {
namespace {

constexpr int kTkThreads = 256;
constexpr int kTile = 32;                 // candidate pages per scoring unit
constexpr int kQpBlk = 64;                // query pages per scoring pass
constexpr int kMaxSeg = 3;
constexpr int64_t kMaxCand = int64_t(1) << 24;
constexpr uint64_t kTkWaitNs = 4000000000ull;

enum : int { kUnitA = 0, kUnitB = 1, kUnitC = 2 };

struct Seg {
    int kind, kv0, nkv;       // units of this kind for KV heads kv0 .. kv0+nkv-1
};

struct TopkArgs {
    const void* q;            // [n_q, Hq, D] pool dtype
    const float* rep;         // [num_phys, Hkv, D]
    const int32_t* bt;
    int64_t num_phys;
    int Hq, Hkv, P;
    int64_t n_q;
    int n_qp;
    int64_t qp0;              // q_start / P
    int K, n_sink, n_local, kmax;
    int n_cand_max, n_tiles, stride;
    float* qbar;              // [n_qp, Hkv, D] page queries
    float* scores;            // [Hkv, n_qp, stride]
    int32_t* out;             // [n_qp, Hkv, kmax]
    int32_t* counts;          // [n_qp, Hkv] or null
    int* state;               // [0] queue, [1] CTAs done, [2, 2+Hkv) A done, [2+Hkv, 2+2Hkv) B done
    int* err;
    int total_units;
    int n_seg;
    Seg seg[kMaxSeg];
};

// Order-preserving map of a float to an unsigned int (ascending).
__device__ __forceinline__ uint32_t orderable(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ int ld_acquire(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint64_t gtimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Thread 0 waits (bounded) until *ctr >= target; the block then proceeds
// together. False (and the error recorded) if the wait gave up or another
// CTA recorded an error.
__device__ bool block_wait_count(const int* ctr, int target, int* err, int* s_ok) {
    if (threadIdx.x == 0) {
        int ok = 1;
        if (ld_acquire(ctr) < target) {
            const uint64_t t0 = gtimer();
            for (;;) {
                __nanosleep(128);
                if (ld_acquire(ctr) >= target) break;
                if (*reinterpret_cast<volatile int*>(err) != 0) { ok = 0; break; }
                if (gtimer() - t0 > kTkWaitNs) {
                    report_error(err, kErrWaitTimeout);
                    ok = 0;
                    break;
                }
            }
        }
        *s_ok = ok;
    }
    __syncthreads();
    return *s_ok != 0;
}

// Exclusive prefix sum over the block (kTkThreads threads); *total gets the sum.
__device__ int block_excl_scan(int v, int* warp_sums, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < kTkThreads / 32 ? warp_sums[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < kTkThreads / 32) warp_sums[lane] = w;    // inclusive over warps
    }
    __syncthreads();
    const int base = warp > 0 ? warp_sums[warp - 1] : 0;
    *total = warp_sums[kTkThreads / 32 - 1];
    __syncthreads();                                         // warp_sums reusable
    return base + x - v;
}

static_assert(kTkThreads == 256, "8 of the 2048 histogram bins per thread");

struct __align__(16) TopkSmem {
    int unit;
    int ok;
    uint32_t prefix;
    int krem;
    int warp_sums[kTkThreads / 32];
};

// ------------------------------------------------------------------ unit A
template <typename T, int D>
__device__ void unit_page_query(const TopkArgs& a, int kv, int qp, float* red) {
    constexpr int VPR = D * (int)sizeof(T) / 16, EPV = 16 / (int)sizeof(T);
    constexpr int RSTEP = kTkThreads / VPR;
    constexpr int U = 16;                 // 16-byte loads in flight per thread
    const int g = a.Hq / a.Hkv;
    const int64_t t0 = (int64_t)qp * a.P;
    const int n_tok = (int)min64(a.P, a.n_q - t0);
    const int rows = n_tok * g;                                   // (token, head of the group)
    const int vc = threadIdx.x % VPR, r0 = threadIdx.x / VPR;
    const T* q = static_cast<const T*>(a.q);
    float acc[EPV];
#pragma unroll
    for (int e = 0; e < EPV; ++e) acc[e] = 0.f;
    for (int rb = r0; rb < rows; rb += U * RSTEP) {
        uint4 u[U];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int r = rb + k * RSTEP;
            if (r < rows) {
                const int t = r / g, hh = r - t * g;
                u[k] = __ldg(reinterpret_cast<const uint4*>(q + ((t0 + t) * a.Hq + kv * g + hh) * D) + vc);
            } else {
                u[k] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
#pragma unroll
        for (int k = 0; k < U; ++k) {
            float f[EPV];
            widen16<T>(u[k], f);
#pragma unroll
            for (int e = 0; e < EPV; ++e) acc[e] += f[e];
        }
    }
#pragma unroll
    for (int e = 0; e < EPV; ++e) red[r0 * D + vc * EPV + e] = acc[e];
    __syncthreads();
    if (threadIdx.x < D) {
        float s = 0.f;
        for (int k = 0; k < RSTEP; ++k) s += red[k * D + threadIdx.x];
        a.qbar[((size_t)qp * a.Hkv + kv) * D + threadIdx.x] = s / (float)rows;
    }
}

// ------------------------------------------------------------------ unit B
// scores[kv][qp][c] = qbar[qp, kv, :] . rep[bt[n_sink + c], kv, :] for the
// tile's candidates c. The representatives sit transposed ([k][c]) so thread
// t, which scores candidate t % 32 against query pages t / 32, t / 32 + 8, ...,
// reads them without bank conflicts; a warp shares its query pages, whose rows
// are read as broadcasts.
// The tile's representatives, transposed into shared memory ([k][c]).
template <int D>
__device__ void load_rep_tile(const TopkArgs& a, int kv, int tile, float* smem) {
    float* rt = smem;                                   // [D][kTile]
    const int tid = threadIdx.x, c0 = tile * kTile;
    constexpr int NL = kTile * (D / 4) / kTkThreads;    // all of a thread's loads issued first
    float4 v[NL];
#pragma unroll
    for (int l = 0; l < NL; ++l) {
        const int i = tid + l * kTkThreads, c = i % kTile, k4 = i / kTile;
        v[l] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (c0 + c < a.n_cand_max) {
            const int32_t pp = a.bt[a.n_sink + c0 + c];
            if (pp >= 0 && pp < a.num_phys)
                v[l] = __ldg(reinterpret_cast<const float4*>(a.rep + ((size_t)pp * a.Hkv + kv) * D) + k4);
            else if (k4 == 0)
                report_error(a.err, kErrBadPage);
        }
    }
#pragma unroll
    for (int l = 0; l < NL; ++l) {
        const int i = tid + l * kTkThreads, c = i % kTile, k4 = i / kTile;
        rt[(4 * k4) * kTile + c] = v[l].x; rt[(4 * k4 + 1) * kTile + c] = v[l].y;
        rt[(4 * k4 + 2) * kTile + c] = v[l].z; rt[(4 * k4 + 3) * kTile + c] = v[l].w;
    }
}

// scores against every query page; the representatives are already in
// shared memory (load_rep_tile; the first barrier below publishes them).
template <int D>
__device__ void unit_scores(const TopkArgs& a, int kv, int tile, float* smem) {
    float* rt = smem;                                   // [D][kTile]
    float* qs = smem + D * kTile;                       // [kQpBlk][D]
    const int tid = threadIdx.x, c0 = tile * kTile;
    constexpr int G = kTkThreads / kTile;               // query-page groups
    constexpr int QPT = kQpBlk / G;                      // query pages per thread and pass
    const int c = tid % kTile, g0 = tid / kTile;
    for (int qb = 0; qb < a.n_qp; qb += kQpBlk) {
        const int nq = min(kQpBlk, a.n_qp - qb);
        __syncthreads();                                  // rt ready; qs free
        {
            constexpr int NQ = kQpBlk * (D / 4) / kTkThreads;
            float4 v[NQ];
#pragma unroll
            for (int l = 0; l < NQ; ++l) {
                const int i = tid + l * kTkThreads, r = i / (D / 4), k4 = i % (D / 4);
                v[l] = r < nq ? __ldcg(reinterpret_cast<const float4*>(
                                    a.qbar + ((size_t)(qb + r) * a.Hkv + kv) * D) + k4)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int l = 0; l < NQ; ++l) {
                const int i = tid + l * kTkThreads;
                reinterpret_cast<float4*>(qs)[i] = v[l];
            }
        }
        __syncthreads();
        float acc[QPT];
#pragma unroll
        for (int j = 0; j < QPT; ++j) acc[j] = 0.f;
#pragma unroll 4
        for (int k = 0; k < D; k += 4) {
            const float r0 = rt[k * kTile + c], r1 = rt[(k + 1) * kTile + c];
            const float r2 = rt[(k + 2) * kTile + c], r3 = rt[(k + 3) * kTile + c];
#pragma unroll
            for (int j = 0; j < QPT; ++j) {
                const float4 qv = *reinterpret_cast<const float4*>(qs + (g0 + j * G) * D + k);
                acc[j] = fmaf(qv.x, r0, acc[j]);
                acc[j] = fmaf(qv.y, r1, acc[j]);
                acc[j] = fmaf(qv.z, r2, acc[j]);
                acc[j] = fmaf(qv.w, r3, acc[j]);
            }
        }
        if (c0 + c < a.n_cand_max) {
#pragma unroll
            for (int j = 0; j < QPT; ++j) {
                const int r = g0 + j * G;
                if (r < nq) a.scores[((size_t)kv * a.n_qp + qb + r) * a.stride + c0 + c] = acc[j];
            }
        }
    }
}

// ------------------------------------------------------------------ unit C
// Padded position of score i in the staged row: one float of padding per 32,
// so the compaction's per-thread runs (stride = run length) hit distinct banks.
__device__ __forceinline__ int padded(int i) { return i + (i >> 5); }

// Keys of the score row: from the copy staged in shared memory (padded
// layout), or from L2. The source is a template argument, so every loop over
// the row has a single kind of load.
template <bool kStaged> struct RowKeys {
    const float* p;
    __device__ __forceinline__ uint32_t operator[](int i) const {
        return orderable(kStaged ? p[padded(i)] : __ldcg(p + i));
    }
};

// The row's n_top best candidates (of n; all when n_top == n), then the sink
// and local pages, into the selection row.
template <bool kStaged>
__device__ void select_row(const TopkArgs& a, int kv, int qp, TopkSmem& S, int* hist,
                           const RowKeys<kStaged> keys, int n, int n_top) {
    const int tid = threadIdx.x;
    const int64_t qpg = a.qp0 + qp;
    const int64_t c_lo = a.n_sink;
    const bool all = n_top == n;
    uint32_t thr = 0;                                             // the n_top-th best key
    int take_eq = 0;                                              // keys == thr to keep
    if (!all && n_top > 0) {
        // Radix select over digits of 11, 11 and 10 bits from the top: the first
        // digit reaches into the mantissa, so even scores of one sign and
        // magnitude spread over many of its 2048 bins.
        uint32_t prefix = 0, mask = 0;
        int krem = n_top;
        for (int pass = 0; pass < 3; ++pass) {
            const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
            const int width = pass == 2 ? 10 : 11;
            const uint32_t dmask = (1u << width) - 1u;
            for (int b = tid; b < 2048; b += kTkThreads) hist[b] = 0;
            __syncthreads();
            for (int i = tid; i < n; i += kTkThreads) {
                const uint32_t key = keys[i];
                if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & dmask], 1);
            }
            __syncthreads();
            // Thread t holds bins 2047-8t .. 2040-8t (best first); the block scan
            // finds the thread whose bins hold the krem-th best key.
            int c[8], sum = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) { c[j] = hist[2047 - 8 * tid - j]; sum += c[j]; }
            int total;
            const int excl = block_excl_scan(sum, S.warp_sums, &total);
            if (excl < krem && excl + sum >= krem) {
                int above = excl, b = 0;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (above + c[j] >= krem) { b = 2047 - 8 * tid - j; break; }
                    above += c[j];
                }
                S.krem = krem - above;
                S.prefix = prefix | ((uint32_t)b << shift);
            }
            __syncthreads();
            krem = S.krem;
            prefix = S.prefix;
            mask |= dmask << shift;
        }
        thr = prefix;
        take_eq = krem;
    }
    // Ordered compaction: thread t owns candidates [t * per, (t + 1) * per).
    const int per = (n + kTkThreads - 1) / kTkThreads;
    const int i0 = min(n, tid * per), i1 = min(n, i0 + per);
    int n_gt = 0, n_eq = 0;
    if (!all && n_top > 0) {
        for (int i = i0; i < i1; ++i) {
            const uint32_t key = keys[i];
            n_gt += key > thr;
            n_eq += key == thr;
        }
    }
    int total;
    const int eq_base = block_excl_scan(n_eq, S.warp_sums, &total);
    const int eq_keep = all || n_top == 0 ? 0 : max(0, min(n_eq, take_eq - eq_base));
    const int mine = all ? i1 - i0 : (n_top == 0 ? 0 : n_gt + eq_keep);
    const int pos0 = block_excl_scan(mine, S.warp_sums, &total);
    const int64_t s_end = min64(a.n_sink, qpg + 1);               // sink pages [0, s_end)
    const int64_t l_beg = max64(s_end, qpg - a.n_local + 1);      // local pages [l_beg, qpg]
    int32_t* out = a.out + ((size_t)qp * a.Hkv + kv) * a.kmax;
    if (mine > 0) {
        int pos = (int)s_end + pos0, eq_seen = 0;
        for (int i = i0; i < i1 && pos < a.kmax; ++i) {
            bool keep = all;
            if (!all) {
                const uint32_t key = keys[i];
                if (key > thr) keep = true;
                else if (key == thr) keep = eq_seen++ < eq_keep;
            }
            if (keep) out[pos++] = (int32_t)(c_lo + i);
        }
    }
    const int n_sel = (int)s_end + total + (int)(qpg - l_beg + 1);
    for (int i = tid; i < a.kmax; i += kTkThreads) {
        if (i < s_end) out[i] = i;
        else if (i >= (int)s_end + total && i < n_sel) out[i] = (int32_t)(l_beg + (i - s_end - total));
        else if (i >= n_sel) out[i] = -1;
    }
    if (a.counts && tid == 0) a.counts[(size_t)qp * a.Hkv + kv] = min(n_sel, a.kmax);
}

__device__ void unit_select(const TopkArgs& a, int kv, int qp, TopkSmem& S, int* hist2048,
                            float* rowbuf, int rowbuf_cap) {
    const int tid = threadIdx.x;
    const int64_t qpg = a.qp0 + qp;
    const int n = (int)max64(0, qpg - a.n_local - (int64_t)a.n_sink + 1);   // candidates of this row
    const int n_top = min(a.K, n);
    const float* row = a.scores + ((size_t)kv * a.n_qp + qp) * a.stride;
    if (n_top == n || n_top == 0 || padded(n) > rowbuf_cap) {
        select_row<false>(a, kv, qp, S, hist2048, RowKeys<false>{row}, n, n_top);
        return;
    }
    // Stage the row (16-byte aligned loads: the stride is a multiple of 4 floats).
    const int n4 = (n + 3) / 4;
    for (int i = tid; i < n4; i += 4 * kTkThreads) {
        float4 v[4];
#pragma unroll
        for (int l = 0; l < 4; ++l)
            if (i + l * kTkThreads < n4) v[l] = __ldcg(reinterpret_cast<const float4*>(row) + i + l * kTkThreads);
#pragma unroll
        for (int l = 0; l < 4; ++l) {
            const int b = 4 * (i + l * kTkThreads);
            if (b < 4 * n4) {
                rowbuf[padded(b)] = v[l].x; rowbuf[padded(b + 1)] = v[l].y;
                rowbuf[padded(b + 2)] = v[l].z; rowbuf[padded(b + 3)] = v[l].w;
            }
        }
    }
    __syncthreads();
    select_row<true>(a, kv, qp, S, hist2048, RowKeys<true>{rowbuf}, n, n_top);
}

template <typename T, int D>
__global__ void __launch_bounds__(kTkThreads) topk_fused_kernel(const __grid_constant__ TopkArgs a,
                                                                int rowbuf_cap) {
    extern __shared__ __align__(16) float dyn[];
    __shared__ TopkSmem S;
    __shared__ int s_hist[2048];
    int* const q_ctr = a.state;
    int* const cta_done = a.state + 1;
    int* const doneA = a.state + 2;
    int* const doneB = a.state + 2 + a.Hkv;
    for (;;) {
        if (threadIdx.x == 0)
            S.unit = *reinterpret_cast<volatile int*>(a.err) != 0 ? a.total_units : atomicAdd(q_ctr, 1);
        __syncthreads();
        int u = S.unit;
        if (u >= a.total_units) break;
        int kind = 0, kv = 0, loc = 0;
        for (int sgi = 0; sgi < a.n_seg; ++sgi) {
            const Seg sg = a.seg[sgi];
            const int per_kv = sg.kind == kUnitB ? a.n_tiles : a.n_qp;
            if (u < per_kv * sg.nkv) {
                kind = sg.kind;
                kv = sg.kv0 + u / per_kv;
                loc = u % per_kv;
                break;
            }
            u -= per_kv * sg.nkv;
        }
        if (kind == kUnitA) {
            unit_page_query<T, D>(a, kv, loc, dyn);
        } else if (kind == kUnitB) {
            load_rep_tile<D>(a, kv, loc, dyn);              // needs no A unit
            if (!block_wait_count(doneA + kv, a.n_qp, a.err, &S.ok)) break;
            unit_scores<D>(a, kv, loc, dyn);
        } else {
            if (!block_wait_count(doneB + kv, a.n_tiles, a.err, &S.ok)) break;
            unit_select(a, kv, loc, S, s_hist, dyn, rowbuf_cap);
        }
        __syncthreads();                                   // the unit's writes are issued
        if (threadIdx.x == 0 && kind != kUnitC) {
            __threadfence();
            atomicAdd(kind == kUnitA ? doneA + kv : doneB + kv, 1);
        }
    }
    // The last CTA out resets the queue and the counters for the next call.
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(cta_done, 1) == (int)gridDim.x - 1) {
            for (int i = 0; i < 2 + 2 * a.Hkv; ++i) a.state[i] = 0;
            __threadfence();
        }
    }
}

template <typename T, int D>
size_t topk_smem_bytes() {
    constexpr int VPR = D * (int)sizeof(T) / 16;
    const size_t a_bytes = (size_t)(kTkThreads / VPR) * D * sizeof(float);
    const size_t b_bytes = (size_t)(D * kTile + kQpBlk * D) * sizeof(float);
    return std::max(a_bytes, b_bytes);
}

template <typename T, int D>
cudaError_t launch_fused(const TopkArgs& a, cudaStream_t s) {
    static int per_sm = 0;
    static std::once_flag once;
    const size_t smem = topk_smem_bytes<T, D>();
    static cudaError_t init = cudaSuccess;
    std::call_once(once, [&] {
        init = cudaFuncSetAttribute(topk_fused_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)smem);
        if (init == cudaSuccess)
            init = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, topk_fused_kernel<T, D>,
                                                                 kTkThreads, smem);
    });
    if (init != cudaSuccess) return init;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int grid = std::max(1, std::min(a.total_units, std::max(1, per_sm) * std::max(1, sms)));
    ProfScope ps("topk_fused_kernel", s);
    topk_fused_kernel<T, D><<<grid, kTkThreads, smem, s>>>(a, (int)(smem / sizeof(float)));
    return cudaGetLastError();
}

// Local attention layers (gist.science/nl "Pagina-niveau Sparse Attention":
// natively sparse models use local attention instead of a scorer), page
// granular: query page qpg sees the sink pages [0, n_sink) and the local pages
// qpg-n_local+1 .. qpg, ascending, -1 padded; the same list for every KV head.
// One thread per output entry.
__global__ void local_kernel(int64_t qp0, int n_qp, int Hkv, int n_sink, int n_local,
                             int32_t* out, int32_t* counts) {
    const int kmax = n_sink + n_local;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)n_qp * Hkv * kmax) return;
    const int j = (int)(i % kmax);
    const int64_t row = i / kmax;                        // (query page, KV head)
    const int64_t qpg = qp0 + row / Hkv;
    const int64_t s_end = min64(n_sink, qpg + 1);        // sink pages [0, s_end)
    const int64_t l_beg = max64(s_end, qpg - n_local + 1);   // local pages [l_beg, qpg]
    const int64_t count = s_end + (qpg - l_beg + 1);
    int64_t page = -1;
    if (j < s_end) page = j;
    else if (j < count) page = l_beg + (j - s_end);
    out[i] = (int32_t)page;
    if (counts && j == 0) counts[row] = (int32_t)count;
}

}  // namespace

cudaError_t launch_page_local(int64_t q_start, int64_t n_q, int P, int Hkv, int n_sink,
                              int n_local, int32_t* out, int32_t* counts, cudaStream_t s) {
    const int64_t n_qp = (n_q + P - 1) / P;
    const int64_t total = n_qp * Hkv * (n_sink + n_local);
    ProfScope ps("local_kernel", s);
    local_kernel<<<(unsigned)((total + 255) / 256), 256, 0, s>>>(q_start / P, (int)n_qp, Hkv,
                                                                 n_sink, n_local, out, counts);
    return cudaGetLastError();
}

cudaError_t launch_page_topk(const pkv_pool* p, const int32_t* d_bt, const void* q, int64_t q_start,
                             int64_t n_q, int K, int n_sink, int n_local, int32_t* out,
                             int32_t* counts, float* scratch, int* state, cudaStream_t s) {
    const int P = p->desc.page_size, Hq = p->desc.n_q_heads, Hkv = p->desc.n_kv_heads;
    const int D = p->desc.head_dim;
    const int64_t n_qp = (n_q + P - 1) / P;
    TopkArgs a{};
    a.q = q; a.rep = p->rep; a.bt = d_bt; a.num_phys = p->desc.num_phys_pages;
    a.Hq = Hq; a.Hkv = Hkv; a.P = P; a.n_q = n_q; a.n_qp = (int)n_qp;
    a.qp0 = q_start / P; a.K = K; a.n_sink = n_sink; a.n_local = n_local;
    a.kmax = K + n_sink + n_local;
    // The chunk's last query page has the most candidates; rows of earlier
    // query pages use a prefix of the score row.
    const int64_t last_qpg = q_start / P + n_qp - 1;
    const int64_t n_cand = std::max<int64_t>(0, last_qpg - n_local - n_sink + 1);
    a.n_cand_max = (int)n_cand;
    a.n_tiles = (int)((n_cand + kTile - 1) / kTile);
    a.stride = (int)((n_cand + 3) / 4 * 4);
    a.qbar = scratch;
    a.scores = scratch + (size_t)n_qp * Hkv * D;
    a.out = out; a.counts = counts; a.state = state; a.err = p->d_err;
    // Queue order: every A unit, then every B unit, then every C unit. The A
    // units of all heads share the HBM stream and finish together; an order
    // interleaving the kinds over the heads was measured slower (the A units
    // spread out over twice the time).
    int ns = 0;
    auto add = [&](int kind, int kv0, int nkv) {
        if (kind == kUnitB && a.n_tiles == 0) return;
        a.seg[ns++] = Seg{kind, kv0, nkv};
    };
    add(kUnitA, 0, Hkv);
    add(kUnitB, 0, Hkv);
    add(kUnitC, 0, Hkv);
    a.n_seg = ns;
    int64_t total = 0;
    for (int i = 0; i < ns; ++i) {
        const Seg& sg = a.seg[i];
        const int64_t per = sg.kind == kUnitB ? a.n_tiles : n_qp;
        total += per * sg.nkv;
    }
    if (total >= (int64_t(1) << 30)) return cudaErrorInvalidValue;
    a.total_units = (int)total;
    if (p->desc.dtype == PKV_BF16)
        return D == 128 ? launch_fused<__nv_bfloat16, 128>(a, s) : launch_fused<__nv_bfloat16, 64>(a, s);
    return D == 128 ? launch_fused<float, 128>(a, s) : launch_fused<float, 64>(a, s);
}

int64_t page_topk_max_candidates() { return kMaxCand; }

int page_topk_state_ints(int Hkv) { return 2 + 2 * Hkv; }

size_t page_topk_scratch_floats(int64_t q_start, int64_t n_q, int P, int Hkv, int D, int n_sink,
                                int n_local) {
    const int64_t n_qp = (n_q + P - 1) / P;
    const int64_t n_cand = std::max<int64_t>(0, q_start / P + n_qp - 1 - n_local - n_sink + 1);
    return (size_t)n_qp * Hkv * D + (size_t)Hkv * n_qp * ((n_cand + 3) / 4 * 4);
}

}  // namespace pkv
