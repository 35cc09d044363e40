// Page-level top-K selection for sparse attention ("Out of the Memory
// Barrier", gist.science/de §2.D: a Top-K procedure finds the most relevant KV
// pages from representative vectors; gist.science/nl: one representative
// vector per page; sciencestack.ai Fig. 5: retrieved key pages per query page).
//
// For every query page qp of the chunk and KV head h:
//   qbar   = mean of the chunk's queries over the page's tokens and the g query
//            heads reading KV head h (fp32);
//   score  = qbar . rep[bt[p], h] for candidate pages p in [n_sink, qpg - n_local]
//            (qpg = the query page's index in the sequence);
//   keep the K best by (score descending, page ascending), plus the sink pages
//   [0, n_sink) and the local pages qpg-n_local+1 .. qpg; write them ascending,
//   padded with -1.
//
// Kernel 1 (qbar): one CTA per (query page, KV head); reads the page's
//   P x g query rows (g*d contiguous elements per token) with 16-byte loads and
//   reduces in fp32. This is the HBM-bound part: it reads the whole chunk's Q.
// Kernel 2 (select): one CTA per (query page, KV head); one warp per candidate
//   scores it with a coalesced 512-byte read of the representative, packs
//   (score, page) into one 64-bit key whose ascending order is the selection
//   order, sorts the keys in shared memory (bitonic), and compacts the chosen
//   pages in ascending order.
#include <cuda_bf16.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace pkv {
namespace {

constexpr int kQbarThreads = 512;
constexpr int kSelThreads = 1024;
constexpr int kMaxCand = 16384;           // sort buffer: 128 KB of 64-bit keys

template <typename T, int D>
__global__ void __launch_bounds__(kQbarThreads) qbar_kernel(const T* q, int64_t n_q, int Hq, int Hkv,
                                                             int P, float* qbar) {
    constexpr int VPR = D * (int)sizeof(T) / 16, EPV = 16 / (int)sizeof(T);
    constexpr int RSTEP = kQbarThreads / VPR;
    __shared__ float red[RSTEP][D];
    const int qp = blockIdx.x, h = blockIdx.y;
    const int g = Hq / Hkv;
    const int64_t t0 = (int64_t)qp * P;
    const int n_tok = (int)min64(P, n_q - t0);
    const int rows = n_tok * g;                     // (token, head-of-group) rows
    const int vc = threadIdx.x % VPR, r0 = threadIdx.x / VPR;
    float acc[EPV];
#pragma unroll
    for (int e = 0; e < EPV; ++e) acc[e] = 0.f;
    auto row_ptr = [&](int r) {
        const int t = r / g, hh = r % g;
        return reinterpret_cast<const uint4*>(q + ((t0 + t) * Hq + h * g + hh) * D) + vc;
    };
    // Eight independent 16-byte loads in flight per thread before any is used.
    constexpr int U = 8;
    int r = r0;
    for (; r + (U - 1) * RSTEP < rows; r += U * RSTEP) {
        uint4 u[U];
#pragma unroll
        for (int k = 0; k < U; ++k) u[k] = __ldg(row_ptr(r + k * RSTEP));
#pragma unroll
        for (int k = 0; k < U; ++k) {
            float f[EPV];
            widen16<T>(u[k], f);
#pragma unroll
            for (int e = 0; e < EPV; ++e) acc[e] += f[e];
        }
    }
    for (; r < rows; r += RSTEP) {
        float f[EPV];
        widen16<T>(__ldg(row_ptr(r)), f);
#pragma unroll
        for (int e = 0; e < EPV; ++e) acc[e] += f[e];
    }
#pragma unroll
    for (int e = 0; e < EPV; ++e) red[r0][vc * EPV + e] = acc[e];
    __syncthreads();
    if (threadIdx.x < D) {
        float s = 0.f;
        for (int k = 0; k < RSTEP; ++k) s += red[k][threadIdx.x];
        qbar[((size_t)qp * Hkv + h) * D + threadIdx.x] = s / (float)rows;
    }
}

// Order-preserving map of a float to an unsigned int (ascending).
__device__ __forceinline__ uint32_t orderable(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct SelArgs {
    const float* qbar;        // [n_qp, Hkv, D]
    const float* rep;         // [num_phys, Hkv, D]
    const int32_t* bt;
    int64_t num_phys;
    int Hkv, D;
    int64_t qp0;              // q_start / P
    int K, n_sink, n_local, kmax;
    int32_t* out;             // [n_qp, Hkv, kmax]
    int32_t* counts;          // [n_qp, Hkv] or null
    int* err;
};

__global__ void __launch_bounds__(kSelThreads) select_kernel(SelArgs a) {
    extern __shared__ uint64_t keys[];             // [n_pow2] sort keys; reused as flags
    __shared__ float qb[128];
    __shared__ int scan[kSelThreads];
    const int qp = blockIdx.x, h = blockIdx.y;
    const int64_t qpg = a.qp0 + qp;                // query page index in the sequence
    const int64_t c_lo = a.n_sink, c_hi = qpg - a.n_local;    // candidates [c_lo, c_hi]
    const int n_cand = (int)max64(0, c_hi - c_lo + 1);
    int n_pow2 = 1;
    while (n_pow2 < n_cand) n_pow2 <<= 1;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid < a.D) qb[tid] = a.qbar[((size_t)qp * a.Hkv + h) * a.D + tid];
    __syncthreads();

    // Scores: one warp per candidate, lane l reads floats 4l..4l+3 of the rep row.
    for (int c = warp; c < n_pow2; c += kSelThreads / 32) {
        uint64_t key = ~0ull;                      // padding sorts last
        if (c < n_cand) {
            const int64_t page = c_lo + c;
            const int32_t pp = a.bt[page];
            float s = 0.f;
            if (pp >= 0 && pp < a.num_phys) {
                const float* row = a.rep + ((size_t)pp * a.Hkv + h) * a.D;
                for (int k = lane * 4; k < a.D; k += 128) {
                    const float4 r = *reinterpret_cast<const float4*>(row + k);
                    s += r.x * qb[k] + r.y * qb[k + 1] + r.z * qb[k + 2] + r.w * qb[k + 3];
                }
            } else if (lane == 0) {
                report_error(a.err, kErrBadPage);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
            key = ((uint64_t)(~orderable(s)) << 32) | (uint32_t)page;
        }
        if (lane == 0) keys[c] = key;
    }
    __syncthreads();

    // Bitonic sort, ascending.
    for (int k = 2; k <= n_pow2; k <<= 1) {
        for (int jj = k >> 1; jj > 0; jj >>= 1) {
            for (int i = tid; i < n_pow2; i += kSelThreads) {
                const int ixj = i ^ jj;
                if (ixj > i) {
                    const uint64_t x = keys[i], y = keys[ixj];
                    const bool up = (i & k) == 0;
                    if ((x > y) == up) {
                        keys[i] = y;
                        keys[ixj] = x;
                    }
                }
            }
            __syncthreads();
        }
    }

    // Chosen pages: the first min(K, n_cand) sorted candidates, plus sink and local.
    const int n_top = min(a.K, n_cand);
    uint32_t top_page = 0xffffffffu;
    if (tid < n_top) top_page = (uint32_t)(keys[tid] & 0xffffffffu);
    __syncthreads();
    uint8_t* flag = reinterpret_cast<uint8_t*>(keys);      // [qpg + 1] page flags
    const int64_t n_pages = qpg + 1;
    for (int64_t p = tid; p < n_pages; p += kSelThreads)
        flag[p] = (p < a.n_sink || p > qpg - a.n_local) ? 1 : 0;
    __syncthreads();
    if (tid < n_top) flag[top_page] = 1;
    __syncthreads();

    // Ordered compaction: thread t owns a contiguous run of pages.
    const int64_t per = (n_pages + kSelThreads - 1) / kSelThreads;
    const int64_t p0 = (int64_t)tid * per, p1 = min64(n_pages, p0 + per);
    int cnt = 0;
    for (int64_t p = p0; p < p1; ++p) cnt += flag[p];
    scan[tid] = cnt;
    __syncthreads();
    for (int off = 1; off < kSelThreads; off <<= 1) {     // inclusive Hillis-Steele scan
        const int v = tid >= off ? scan[tid - off] : 0;
        __syncthreads();
        scan[tid] += v;
        __syncthreads();
    }
    int pos = scan[tid] - cnt;
    int32_t* out = a.out + ((size_t)qp * a.Hkv + h) * a.kmax;
    for (int64_t p = p0; p < p1; ++p)
        if (flag[p] && pos < a.kmax) out[pos++] = (int32_t)p;
    const int total = scan[kSelThreads - 1];
    for (int i = total + tid; i < a.kmax; i += kSelThreads) out[i] = -1;
    if (a.counts && tid == 0) a.counts[(size_t)qp * a.Hkv + h] = min(total, a.kmax);
}

}  // namespace

cudaError_t launch_page_topk(const pkv_pool* p, const int32_t* d_bt, const void* q, int64_t q_start,
                             int64_t n_q, int K, int n_sink, int n_local, int32_t* out,
                             int32_t* counts, float* qbar, cudaStream_t s) {
    const int P = p->desc.page_size, Hq = p->desc.n_q_heads, Hkv = p->desc.n_kv_heads;
    const int D = p->desc.head_dim;
    const int64_t n_qp = (n_q + P - 1) / P;
    dim3 grid((unsigned)n_qp, Hkv);
    {
        ProfScope ps("qbar_kernel", s);
        if (p->desc.dtype == PKV_BF16) {
            if (D == 128) qbar_kernel<__nv_bfloat16, 128><<<grid, kQbarThreads, 0, s>>>(static_cast<const __nv_bfloat16*>(q), n_q, Hq, Hkv, P, qbar);
            else qbar_kernel<__nv_bfloat16, 64><<<grid, kQbarThreads, 0, s>>>(static_cast<const __nv_bfloat16*>(q), n_q, Hq, Hkv, P, qbar);
        } else {
            if (D == 128) qbar_kernel<float, 128><<<grid, kQbarThreads, 0, s>>>(static_cast<const float*>(q), n_q, Hq, Hkv, P, qbar);
            else qbar_kernel<float, 64><<<grid, kQbarThreads, 0, s>>>(static_cast<const float*>(q), n_q, Hq, Hkv, P, qbar);
        }
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    SelArgs a{};
    a.qbar = qbar; a.rep = p->rep; a.bt = d_bt; a.num_phys = p->desc.num_phys_pages;
    a.Hkv = Hkv; a.D = D; a.qp0 = q_start / P; a.K = K; a.n_sink = n_sink; a.n_local = n_local;
    a.kmax = K + n_sink + n_local; a.out = out; a.counts = counts; a.err = p->d_err;
    // Largest candidate count of the chunk (its last query page) sizes the sort buffer.
    const int64_t last_qpg = q_start / P + n_qp - 1;
    const int64_t n_cand = std::max<int64_t>(0, last_qpg - n_local - n_sink + 1);
    int64_t n_pow2 = 1;
    while (n_pow2 < n_cand) n_pow2 <<= 1;
    const size_t smem = std::max<size_t>((size_t)n_pow2 * 8, (size_t)(last_qpg + 1));
    static size_t attr = 0;
    if (smem > 48 * 1024 && smem > attr) {
        cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
        attr = smem;
    }
    ProfScope ps("select_kernel", s);
    select_kernel<<<grid, kSelThreads, smem, s>>>(a);
    return cudaGetLastError();
}

int64_t page_topk_max_candidates() { return kMaxCand; }

}  // namespace pkv
