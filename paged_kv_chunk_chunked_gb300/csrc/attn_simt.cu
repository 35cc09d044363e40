// CUDA-core (SIMT) paged chunk attention, forward and backward, fp32 math.
//
// This is the path for fp32 pools (exact to ~1e-6) and for shapes the
// tensor-core kernels do not cover (page sizes other than 128, d = 64). It
// computes the same thing as the tensor-core path: exact causal softmax
// attention of one query chunk over the keys reached through the block table
// (dense), or over the pages selected for each query page (sparse), with
// in-place accumulation of dK/dV into the paged gradient pool ("Out of the
// Memory Barrier", gist.science/de §2.B and §2.D; sciencestack.ai Fig. 3).
//
// Tiling: 16 query rows x 16 keys per step, 128 threads (8 per row). Key
// blocks of 16 never straddle a page (P % 16 == 0).
//   fwd      : CTA per (16 queries, q head), online softmax, writes O and LSE.
//   bwd dQ   : CTA per (16 queries, q head): P from LSE, dS, dQ.
//   bwd dK/dV: CTA per (16 keys, KV head), looping over the queries and the g
//              heads that see those keys; adds s*dK and dV into the gradient
//              pages (each row is owned by one CTA, so a plain add suffices).
#include <cuda_bf16.h>
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace pkv {
namespace {

constexpr int BM = 16, BN = 16, NT = 128;

template <typename T>
__device__ __forceinline__ float ld(const T* p) { return Elem<T>::load(p); }

// Loads a [16][D] tile of rows (token i, head h) of a [n, H, D] tensor; rows
// beyond n read as zero.
template <typename T, int D>
__device__ __forceinline__ void load_rows(float (*dst)[D + 1], const T* src, int64_t row0,
                                          int64_t n, int H, int h) {
    for (int i = threadIdx.x; i < 16 * D; i += NT) {
        const int r = i / D, c = i % D;
        const int64_t t = row0 + r;
        dst[r][c] = t < n ? ld(src + ((size_t)t * H + h) * D + c) : 0.f;
    }
}

// Loads 16 keys (and values) at positions kp0..kp0+15 (same page) of KV head kvh.
template <typename T, int D>
__device__ __forceinline__ bool load_keys(float (*Ks)[D + 1], float (*Vs)[D + 1],
                                          const AttnArgs& a, int64_t kp0, int kvh) {
    const int64_t lp = kp0 / a.P;
    const int32_t pp = a.bt[lp];
    if (pp < 0 || pp >= a.num_phys) {
        report_error(a.err, kErrBadPage);
        return false;
    }
    const int row0 = (int)(kp0 % a.P);
    const size_t base = (((size_t)pp * a.Hkv + kvh) * a.P + row0) * D;
    const T* kp = static_cast<const T*>(a.kpool) + base;
    const T* vp = static_cast<const T*>(a.vpool) + base;
    for (int i = threadIdx.x; i < 16 * D; i += NT) {
        const int r = i / D, c = i % D;
        Ks[r][c] = ld(kp + (size_t)r * D + c);
        if (Vs) Vs[r][c] = ld(vp + (size_t)r * D + c);
    }
    return true;
}

// Whether logical page lp is listed for (query page qp, KV head kvh).
__device__ __forceinline__ bool page_selected(const AttnArgs& a, int64_t qp, int kvh, int64_t lp) {
    const int32_t* row = a.sel + ((size_t)qp * a.Hkv + kvh) * a.kmax;
    for (int i = 0; i < a.kmax; ++i) {
        const int32_t x = row[i];
        if (x == lp) return true;
        if (x < 0 || x > lp) return false;   // ascending, -1 padded
    }
    return false;
}

// Iterates the key blocks visible to query rows [q0, q0+16) of the chunk: all
// blocks up to the last row's position (dense) or the blocks of the pages
// listed for the rows' query page (sparse). Calls f(kp0) for each.
template <typename F>
__device__ __forceinline__ void for_key_blocks(const AttnArgs& a, int64_t q0, int kvh, F&& f) {
    const int64_t last = a.q_start + min64(q0 + BM, a.n_q) - 1;  // max key position
    if (!a.sel) {
        for (int64_t kp0 = 0; kp0 <= last; kp0 += BN)
            if (!f(kp0)) return;
        return;
    }
    const int64_t qp = q0 / a.P;
    const int32_t* row = a.sel + ((size_t)qp * a.Hkv + kvh) * a.kmax;
    for (int i = 0; i < a.kmax; ++i) {
        const int32_t lp = row[i];
        if (lp < 0) break;
        for (int64_t kp0 = (int64_t)lp * a.P; kp0 < (int64_t)(lp + 1) * a.P && kp0 <= last;
             kp0 += BN)
            if (!f(kp0)) return;
    }
}

template <typename T, int D>
__global__ void __launch_bounds__(NT) fwd_simt(AttnArgs a) {
    constexpr int E = D / 8;                 // dims per thread: e*8 + sub
    __shared__ float Qs[BM][D + 1], Ks[BN][D + 1], Vs[BN][D + 1], Ps[BM][BN + 1];
    const int h = blockIdx.y, kvh = h / (a.Hq / a.Hkv);
    const int64_t q0 = (int64_t)blockIdx.x * BM;
    const int r = threadIdx.x / 8, sub = threadIdx.x % 8;
    const int64_t qpos = a.q_start + q0 + r;
    const float sl2 = rsqrtf((float)D) * kLog2e;
    load_rows<T, D>(Qs, static_cast<const T*>(a.q), q0, a.n_q, a.Hq, h);
    float m = -INFINITY, l = 0.f, o[E];
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] = 0.f;

    for_key_blocks(a, q0, kvh, [&](int64_t kp0) {
        __syncthreads();
        if (!load_keys<T, D>(Ks, Vs, a, kp0, kvh)) return false;
        __syncthreads();
        float x[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int c = sub + 8 * j;
            float acc = 0.f;
#pragma unroll 8
            for (int k = 0; k < D; ++k) acc += Qs[r][k] * Ks[c][k];
            x[j] = (kp0 + c <= qpos) ? acc * sl2 : -INFINITY;
        }
        float mx = fmaxf(x[0], x[1]);
#pragma unroll
        for (int off = 1; off < 8; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        const float m_new = fmaxf(m, mx);
        const float alpha = (m_new == -INFINITY) ? 1.f : exp2f(m - m_new);
        float p[2], ps = 0.f;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            p[j] = (x[j] == -INFINITY) ? 0.f : exp2f(x[j] - m_new);
            ps += p[j];
        }
#pragma unroll
        for (int off = 1; off < 8; off <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
        l = l * alpha + ps;
        m = m_new;
        Ps[r][sub] = p[0];
        Ps[r][sub + 8] = p[1];
        __syncwarp();
#pragma unroll
        for (int e = 0; e < E; ++e) o[e] *= alpha;
#pragma unroll 4
        for (int c = 0; c < BN; ++c) {
            const float pc = Ps[r][c];
#pragma unroll
            for (int e = 0; e < E; ++e) o[e] += pc * Vs[c][e * 8 + sub];
        }
        return true;
    });

    if (q0 + r < a.n_q) {
        const float inv = 1.f / l;
        T* orow = static_cast<T*>(a.o) + ((size_t)(q0 + r) * a.Hq + h) * D;
#pragma unroll
        for (int e = 0; e < E; ++e) Elem<T>::store(orow + e * 8 + sub, o[e] * inv);
        if (sub == 0) a.lse[(size_t)h * a.n_q + q0 + r] = (m + log2f(l)) * kLn2;
    }
}

template <typename T, int D>
__global__ void __launch_bounds__(NT) bwd_dq_simt(AttnArgs a) {
    constexpr int E = D / 8;
    __shared__ float Qs[BM][D + 1], dOs[BM][D + 1], Ks[BN][D + 1], Vs[BN][D + 1], Ps[BM][BN + 1];
    const int h = blockIdx.y, kvh = h / (a.Hq / a.Hkv);
    const int64_t q0 = (int64_t)blockIdx.x * BM;
    const int r = threadIdx.x / 8, sub = threadIdx.x % 8;
    const int64_t qpos = a.q_start + q0 + r;
    const float scale = rsqrtf((float)D);
    load_rows<T, D>(Qs, static_cast<const T*>(a.q), q0, a.n_q, a.Hq, h);
    load_rows<T, D>(dOs, static_cast<const T*>(a.dout), q0, a.n_q, a.Hq, h);
    const bool valid = q0 + r < a.n_q;
    const float lse = valid ? a.lse_in[(size_t)h * a.n_q + q0 + r] : 0.f;
    const float Dr = valid ? a.Dbuf[(size_t)h * a.n_q + q0 + r] : 0.f;
    float dq[E];
#pragma unroll
    for (int e = 0; e < E; ++e) dq[e] = 0.f;

    for_key_blocks(a, q0, kvh, [&](int64_t kp0) {
        __syncthreads();
        if (!load_keys<T, D>(Ks, Vs, a, kp0, kvh)) return false;
        __syncthreads();
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int c = sub + 8 * j;
            float s = 0.f, dp = 0.f;
#pragma unroll 8
            for (int k = 0; k < D; ++k) {
                s += Qs[r][k] * Ks[c][k];
                dp += dOs[r][k] * Vs[c][k];
            }
            const float p = (valid && kp0 + c <= qpos) ? expf(s * scale - lse) : 0.f;
            Ps[r][c] = p * (dp - Dr);
        }
        __syncwarp();
#pragma unroll 4
        for (int c = 0; c < BN; ++c) {
            const float ds = Ps[r][c];
#pragma unroll
            for (int e = 0; e < E; ++e) dq[e] += ds * Ks[c][e * 8 + sub];
        }
        return true;
    });
    if (valid) {
        T* row = static_cast<T*>(a.dq) + ((size_t)(q0 + r) * a.Hq + h) * D;
#pragma unroll
        for (int e = 0; e < E; ++e) Elem<T>::store(row + e * 8 + sub, dq[e] * scale);
    }
}

template <typename T, int D>
__global__ void __launch_bounds__(NT) bwd_dkdv_simt(AttnArgs a) {
    constexpr int E = D / 8;
    __shared__ float Ks[BN][D + 1], Vs[BN][D + 1], Qs[BM][D + 1], dOs[BM][D + 1];
    __shared__ float Ps[BN][BM + 1], DSs[BN][BM + 1], lse_s[BM], D_s[BM];
    const int kvh = blockIdx.y;
    const int g = a.Hq / a.Hkv;
    const int64_t kp0 = (int64_t)blockIdx.x * BN;       // first key of the block
    const int64_t lp = kp0 / a.P;
    const int r = threadIdx.x / 8, sub = threadIdx.x % 8;   // r = key row
    const float scale = rsqrtf((float)D);
    if (a.sel) {
        // Sparse: a page no query page of the chunk selected contributes nothing
        // (and, in a staged pool, need not be in a slot).
        bool used = false;
        for (int64_t qp = 0; qp * a.P < a.n_q && !used; ++qp) used = page_selected(a, qp, kvh, lp);
        if (!used) return;
    }
    if (!load_keys<T, D>(Ks, Vs, a, kp0, kvh)) return;
    float dk[E], dv[E];
#pragma unroll
    for (int e = 0; e < E; ++e) dk[e] = dv[e] = 0.f;
    const int64_t kpos = kp0 + r;

    // Query blocks of the chunk that can see this key block.
    const int64_t qb_first = max64(0, kp0 - a.q_start) / BM;
    const int64_t n_qb = (a.n_q + BM - 1) / BM;
    for (int64_t qb = qb_first; qb < n_qb; ++qb) {
        const int64_t q0 = qb * BM;
        if (a.sel && !page_selected(a, q0 / a.P, kvh, lp)) continue;
        for (int hh = 0; hh < g; ++hh) {
            const int h = kvh * g + hh;
            __syncthreads();
            load_rows<T, D>(Qs, static_cast<const T*>(a.q), q0, a.n_q, a.Hq, h);
            load_rows<T, D>(dOs, static_cast<const T*>(a.dout), q0, a.n_q, a.Hq, h);
            if (threadIdx.x < BM) {
                const int64_t i = q0 + threadIdx.x;
                lse_s[threadIdx.x] = i < a.n_q ? a.lse_in[(size_t)h * a.n_q + i] : 0.f;
                D_s[threadIdx.x] = i < a.n_q ? a.Dbuf[(size_t)h * a.n_q + i] : 0.f;
            }
            __syncthreads();
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int c = sub + 8 * j;                 // query column
                const int64_t i = q0 + c;
                float s = 0.f, dp = 0.f;
#pragma unroll 8
                for (int k = 0; k < D; ++k) {
                    s += Ks[r][k] * Qs[c][k];
                    dp += Vs[r][k] * dOs[c][k];
                }
                const bool vis = i < a.n_q && kpos <= a.q_start + i;
                const float p = vis ? expf(s * scale - lse_s[c]) : 0.f;
                Ps[r][c] = p;
                DSs[r][c] = p * (dp - D_s[c]);
            }
            __syncwarp();
#pragma unroll 4
            for (int c = 0; c < BM; ++c) {
                const float p = Ps[r][c], ds = DSs[r][c];
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    dv[e] += p * dOs[c][e * 8 + sub];
                    dk[e] += ds * Qs[c][e * 8 + sub];
                }
            }
        }
    }
    const int32_t pp = a.bt[lp];
    const size_t off = (((size_t)pp * a.Hkv + kvh) * a.P + (kpos % a.P)) * D;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        a.dkpool[off + e * 8 + sub] += dk[e] * scale;
        a.dvpool[off + e * 8 + sub] += dv[e];
    }
}

// D_i = sum_d dO_i * O_i per (query, head), stored [Hq, n_q] fp32.
template <typename T, int D>
__global__ void rowdot_kernel(AttnArgs a) {
    constexpr int VPR = D * (int)sizeof(T) / 16, EPV = 16 / (int)sizeof(T);
    const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / VPR;   // t*Hq + h
    const int vc = threadIdx.x % VPR;
    float acc = 0.f;
    if (row < a.n_q * a.Hq) {
        const uint4 x = __ldg(reinterpret_cast<const uint4*>(static_cast<const T*>(a.dout) + row * D) + vc);
        const uint4 y = __ldg(reinterpret_cast<const uint4*>(static_cast<const T*>(a.o_in) + row * D) + vc);
        float fx[EPV], fy[EPV];
        widen16<T>(x, fx);
        widen16<T>(y, fy);
#pragma unroll
        for (int e = 0; e < EPV; ++e) acc += fx[e] * fy[e];
    }
#pragma unroll
    for (int off = 1; off < VPR; off <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (vc == 0 && row < a.n_q * a.Hq) {
        const int64_t t = row / a.Hq;
        const int h = (int)(row % a.Hq);
        a.Dbuf[(size_t)h * a.n_q + t] = acc;
    }
}

template <typename T, int D>
cudaError_t fwd_launch(const AttnArgs& a, cudaStream_t s) {
    dim3 grid((unsigned)((a.n_q + BM - 1) / BM), a.Hq);
    ProfScope ps("fwd_simt", s);
    fwd_simt<T, D><<<grid, NT, 0, s>>>(a);
    return cudaGetLastError();
}

template <typename T, int D>
cudaError_t bwd_launch(const AttnArgs& a, cudaStream_t s) {
    dim3 g1((unsigned)((a.n_q + BM - 1) / BM), a.Hq);
    {
        ProfScope ps("bwd_dq_simt", s);
        bwd_dq_simt<T, D><<<g1, NT, 0, s>>>(a);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t n_keys = a.q_start + a.n_q;
    dim3 g2((unsigned)((n_keys + BN - 1) / BN), a.Hkv);
    ProfScope ps("bwd_dkdv_simt", s);
    bwd_dkdv_simt<T, D><<<g2, NT, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_fwd_simt(const AttnArgs& a, cudaStream_t s) {
    if (a.P % 16) return cudaErrorInvalidValue;
    if (a.dtype == PKV_BF16)
        return a.d == 128 ? fwd_launch<__nv_bfloat16, 128>(a, s) : fwd_launch<__nv_bfloat16, 64>(a, s);
    return a.d == 128 ? fwd_launch<float, 128>(a, s) : fwd_launch<float, 64>(a, s);
}

cudaError_t launch_attn_bwd_simt(const AttnArgs& a, cudaStream_t s) {
    if (a.P % 16) return cudaErrorInvalidValue;
    if (a.dtype == PKV_BF16)
        return a.d == 128 ? bwd_launch<__nv_bfloat16, 128>(a, s) : bwd_launch<__nv_bfloat16, 64>(a, s);
    return a.d == 128 ? bwd_launch<float, 128>(a, s) : bwd_launch<float, 64>(a, s);
}

cudaError_t launch_bwd_rowdot(const AttnArgs& a, cudaStream_t s) {
    const int64_t rows = a.n_q * a.Hq;
    const int vpr = a.d * (a.dtype == PKV_BF16 ? 2 : 4) / 16;
    const int threads = 256;
    const int64_t blocks = (rows * vpr + threads - 1) / threads;
    ProfScope ps("rowdot_kernel", s);
    if (a.dtype == PKV_BF16) {
        if (a.d == 128) rowdot_kernel<__nv_bfloat16, 128><<<(unsigned)blocks, threads, 0, s>>>(a);
        else rowdot_kernel<__nv_bfloat16, 64><<<(unsigned)blocks, threads, 0, s>>>(a);
    } else {
        if (a.d == 128) rowdot_kernel<float, 128><<<(unsigned)blocks, threads, 0, s>>>(a);
        else rowdot_kernel<float, 64><<<(unsigned)blocks, threads, 0, s>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace pkv
