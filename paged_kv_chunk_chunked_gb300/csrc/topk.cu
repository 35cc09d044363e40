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
// Kernel 2 (score): one CTA per (tile of 64 candidate pages, KV head) reads
//   the tile's representatives once and scores them against every query page
//   of the chunk (a [n_qp x d] x [d x 64] product in fp32 on the CUDA cores:
//   64 query pages x 2048 pages x 128 is 17 MFLOP per head, too small for a
//   tensor-core pipeline to pay), so each representative leaves L2 once per
//   chunk instead of once per query page.
// Kernel 3 (select): one CTA per (query page, KV head) reads its score row,
//   packs (score, page) into one 64-bit key whose ascending order is the
//   selection order, sorts the keys in shared memory (bitonic), and compacts
//   the chosen pages in ascending order.
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

constexpr int kScoreThreads = 256;
constexpr int kScoreTile = 64;            // candidate pages per CTA
constexpr int kScoreQpMax = 16;           // query pages held in shared memory at once

// scores[h][qp][c] = qbar[qp, h, :] . rep[bt[n_sink + c], h, :] for the tile's
// candidates c. The tile's representatives are stored transposed ([k][c]), so
// thread t, which scores candidate t % 64 against query pages t / 64,
// t / 64 + 4, ..., reads them without bank conflicts; a warp shares its query
// pages, whose rows are read as broadcasts.
template <int D>
__global__ void __launch_bounds__(kScoreThreads) score_kernel(const float* qbar, const float* rep,
        const int32_t* bt, int64_t num_phys, int Hkv, int n_qp, int64_t c_lo, int n_cand,
        int stride, float* scores, int* err) {
    __shared__ float rt[D][kScoreTile];
    __shared__ __align__(16) float qs[kScoreQpMax][D];
    const int h = blockIdx.y, c0 = blockIdx.x * kScoreTile;
    const int tid = threadIdx.x;
    for (int i = tid; i < kScoreTile * (D / 4); i += kScoreThreads) {
        const int c = i % kScoreTile, k4 = i / kScoreTile;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (c0 + c < n_cand) {
            const int32_t pp = bt[c_lo + c0 + c];
            if (pp >= 0 && pp < num_phys)
                v = reinterpret_cast<const float4*>(rep + ((size_t)pp * Hkv + h) * D)[k4];
            else if (k4 == 0)
                report_error(err, kErrBadPage);
        }
        rt[4 * k4][c] = v.x; rt[4 * k4 + 1][c] = v.y; rt[4 * k4 + 2][c] = v.z; rt[4 * k4 + 3][c] = v.w;
    }
    constexpr int G = kScoreThreads / kScoreTile;            // query-page groups
    constexpr int QPT = kScoreQpMax / G;                      // query pages per thread and pass
    const int c = tid % kScoreTile, g0 = tid / kScoreTile;
    for (int qb = 0; qb < n_qp; qb += kScoreQpMax) {
        const int nq = min(kScoreQpMax, n_qp - qb);
        __syncthreads();                                      // rt ready; qs free
        for (int i = tid; i < kScoreQpMax * (D / 4); i += kScoreThreads) {
            const int r = i / (D / 4), k4 = i % (D / 4);
            reinterpret_cast<float4*>(qs[r])[k4] =
                r < nq ? reinterpret_cast<const float4*>(qbar + ((size_t)(qb + r) * Hkv + h) * D)[k4]
                       : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        __syncthreads();
        float acc[QPT];
#pragma unroll
        for (int j = 0; j < QPT; ++j) acc[j] = 0.f;
#pragma unroll 4
        for (int k = 0; k < D; k += 4) {
            const float r0 = rt[k][c], r1 = rt[k + 1][c], r2 = rt[k + 2][c], r3 = rt[k + 3][c];
#pragma unroll
            for (int j = 0; j < QPT; ++j) {
                const float4 qv = reinterpret_cast<const float4*>(qs[g0 + j * G])[k / 4];
                acc[j] = fmaf(qv.x, r0, acc[j]);
                acc[j] = fmaf(qv.y, r1, acc[j]);
                acc[j] = fmaf(qv.z, r2, acc[j]);
                acc[j] = fmaf(qv.w, r3, acc[j]);
            }
        }
        if (c0 + c < n_cand) {
#pragma unroll
            for (int j = 0; j < QPT; ++j) {
                const int r = g0 + j * G;
                if (r < nq) scores[((size_t)h * n_qp + qb + r) * stride + c0 + c] = acc[j];
            }
        }
    }
}

struct SelArgs {
    const float* scores;      // [Hkv, n_qp, stride]
    int stride, n_qp;
    int Hkv;
    int64_t qp0;              // q_start / P
    int K, n_sink, n_local, kmax;
    int32_t* out;             // [n_qp, Hkv, kmax]
    int32_t* counts;          // [n_qp, Hkv] or null
};

__global__ void __launch_bounds__(kSelThreads) select_kernel(SelArgs a) {
    extern __shared__ uint64_t keys[];             // [n_pow2] sort keys; reused as flags
    __shared__ int scan[kSelThreads];
    const int qp = blockIdx.x, h = blockIdx.y;
    const int64_t qpg = a.qp0 + qp;                // query page index in the sequence
    const int64_t c_lo = a.n_sink, c_hi = qpg - a.n_local;    // candidates [c_lo, c_hi]
    const int n_cand = (int)max64(0, c_hi - c_lo + 1);
    int n_pow2 = 1;
    while (n_pow2 < n_cand) n_pow2 <<= 1;
    const int tid = threadIdx.x;
    const float* srow = a.scores + ((size_t)h * a.n_qp + qp) * a.stride;
    for (int c = tid; c < n_pow2; c += kSelThreads) {
        uint64_t key = ~0ull;                      // padding sorts last
        if (c < n_cand) key = ((uint64_t)(~orderable(srow[c])) << 32) | (uint32_t)(c_lo + c);
        keys[c] = key;
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
    // Largest candidate count of the chunk (its last query page) sizes the
    // score rows and the sort buffer.
    const int64_t last_qpg = q_start / P + n_qp - 1;
    const int64_t n_cand = std::max<int64_t>(0, last_qpg - n_local - n_sink + 1);
    const int stride = (int)((n_cand + 3) / 4 * 4);
    float* scores = qbar + n_qp * Hkv * D;
    if (n_cand > 0) {
        dim3 sgrid((unsigned)((n_cand + kScoreTile - 1) / kScoreTile), Hkv);
        ProfScope ps("score_kernel", s);
        if (D == 128)
            score_kernel<128><<<sgrid, kScoreThreads, 0, s>>>(qbar, p->rep, d_bt, p->desc.num_phys_pages,
                    Hkv, (int)n_qp, n_sink, (int)n_cand, stride, scores, p->d_err);
        else
            score_kernel<64><<<sgrid, kScoreThreads, 0, s>>>(qbar, p->rep, d_bt, p->desc.num_phys_pages,
                    Hkv, (int)n_qp, n_sink, (int)n_cand, stride, scores, p->d_err);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    SelArgs a{};
    a.scores = scores; a.stride = stride; a.n_qp = (int)n_qp;
    a.Hkv = Hkv; a.qp0 = q_start / P; a.K = K; a.n_sink = n_sink; a.n_local = n_local;
    a.kmax = K + n_sink + n_local; a.out = out; a.counts = counts;
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

size_t page_topk_scratch_floats(int64_t q_start, int64_t n_q, int P, int Hkv, int D, int n_sink,
                                int n_local) {
    const int64_t n_qp = (n_q + P - 1) / P;
    const int64_t n_cand = std::max<int64_t>(0, q_start / P + n_qp - 1 - n_local - n_sink + 1);
    return (size_t)n_qp * Hkv * D + (size_t)Hkv * n_qp * ((n_cand + 3) / 4 * 4);
}

}  // namespace pkv
