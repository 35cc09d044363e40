// Page writes: append (scatter a chunk's K/V into its pages, page
// representatives, fresh-page gradient zeroing), gradient zeroing, gradient
// accumulation from contiguous rows, and the logical-order gather used by
// tests and by the K/V projections' backward.
//
// Representatives follow "Out of the Memory Barrier" (gist.science/de §2.D:
// relevant pages are found through per-page representative vectors): here the
// fp32 mean of the keys a page holds, per KV head.
//
// All four kernels are HBM-bound copies: one CTA per (logical page, KV head),
// 16-byte loads/stores, a row of d elements read by d*elem/16 consecutive
// threads so that every warp touches whole 32-byte sectors.
#include <cuda_bf16.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace pkv {
namespace {

constexpr int kThreads = 256;

// One CTA per (logical page, KV head, part): part 0 copies the page's new rows
// and writes its representative, part 1 zeroes the gradient rows of a fresh
// page, so the two streams run on different SMs. Part 0 issues up to kAppUnroll
// row loads per thread before the first store (a page's whole K and V in
// flight at P = d = 128, bf16).
constexpr int kAppThreads = 512;
constexpr int kAppUnroll = 4;

template <typename T, int D>
__global__ void __launch_bounds__(kAppThreads, 2) append_kernel(AppendArgs a) {
    constexpr int VPR = D * (int)sizeof(T) / 16;   // 16-byte vectors per row
    constexpr int EPV = 16 / (int)sizeof(T);       // elements per vector
    constexpr int RSTEP = kAppThreads / VPR;       // rows handled per pass
    __shared__ float red[RSTEP][D];

    const int P = a.P;
    const int64_t lp = a.old_len / P + blockIdx.x;  // logical page
    const int h = blockIdx.y;
    const int32_t pp = a.bt[lp];
    if (pp < 0 || pp >= a.num_phys) {
        report_error(a.err, kErrBadPage);
        return;
    }
    const int64_t new_len = a.old_len + a.n_tok;
    const int64_t page_start = lp * P;
    const int tid = threadIdx.x;
    const size_t page_off = ((size_t)pp * a.Hkv + h) * (size_t)P * D;

    if (blockIdx.z == 1) {
        // A page taken off the free list starts with zero gradient (for host
        // pages only recorded as such, nothing crosses the host link).
        if (page_start >= a.old_len && a.gzero) {
            if (tid == 0) a.gzero[(size_t)pp * a.Hkv + h] = 1;
        } else if (page_start >= a.old_len) {
            float4* g0 = reinterpret_cast<float4*>(a.dkpool + page_off);
            float4* g1 = reinterpret_cast<float4*>(a.dvpool + page_off);
            const int n4 = P * D / 4;
            const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int i = tid; i < n4; i += kAppThreads) {
                g0[i] = z;
                g1[i] = z;
            }
        }
        return;
    }

    const int vc = tid % VPR;
    const int r0 = tid / VPR;
    T* kpage = static_cast<T*>(a.kpool) + page_off;
    T* vpage = static_cast<T*>(a.vpool) + page_off;

    float acc[EPV];
#pragma unroll
    for (int e = 0; e < EPV; ++e) acc[e] = 0.f;

    for (int rb = r0; rb < P; rb += kAppUnroll * RSTEP) {
        uint4 kr[kAppUnroll], vr[kAppUnroll];
#pragma unroll
        for (int u = 0; u < kAppUnroll; ++u) {
            const int r = rb + u * RSTEP;
            const int64_t pos = page_start + r;
            kr[u] = vr[u] = make_uint4(0, 0, 0, 0);
            if (r < P && pos >= a.old_len && pos < new_len) {
                const size_t src = ((size_t)(pos - a.old_len) * a.Hkv + h) * D;
                kr[u] = __ldg(reinterpret_cast<const uint4*>(static_cast<const T*>(a.k_in) + src) + vc);
                vr[u] = __ldg(reinterpret_cast<const uint4*>(static_cast<const T*>(a.v_in) + src) + vc);
            } else if (r < P && pos < a.old_len) {
                kr[u] = reinterpret_cast<const uint4*>(kpage + (size_t)r * D)[vc];  // earlier append
            }
        }
#pragma unroll
        for (int u = 0; u < kAppUnroll; ++u) {
            const int r = rb + u * RSTEP;
            const int64_t pos = page_start + r;
            if (r >= P) continue;
            if (pos >= a.old_len) {           // new rows, and zero rows beyond the sequence
                reinterpret_cast<uint4*>(kpage + (size_t)r * D)[vc] = kr[u];
                reinterpret_cast<uint4*>(vpage + (size_t)r * D)[vc] = vr[u];
            }
            if (pos < new_len) {
                float f[EPV];
                widen16<T>(kr[u], f);
#pragma unroll
                for (int e = 0; e < EPV; ++e) acc[e] += f[e];
            }
        }
    }

#pragma unroll
    for (int e = 0; e < EPV; ++e) red[r0][vc * EPV + e] = acc[e];
    __syncthreads();
    if (tid < D) {
        float sum = 0.f;
#pragma unroll 4
        for (int g = 0; g < RSTEP; ++g) sum += red[g][tid];
        const int64_t valid = min64(P, new_len - page_start);
        a.rep[((size_t)pp * a.Hkv + h) * D + tid] = sum / (float)valid;
    }
}

__global__ void grad_zero_kernel(float* dk, float* dv, const int32_t* bt, int64_t p0, int64_t num_phys,
                                 int Hkv, int page_floats, int* err) {
    const int64_t lp = p0 + blockIdx.x;
    const int32_t pp = bt[lp];
    if (pp < 0 || pp >= num_phys) {
        report_error(err, kErrBadPage);
        return;
    }
    const size_t off = ((size_t)pp * Hkv + blockIdx.y) * page_floats;
    float4* a = reinterpret_cast<float4*>(dk + off);
    float4* b = reinterpret_cast<float4*>(dv + off);
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i = threadIdx.x; i < page_floats / 4; i += blockDim.x) {
        a[i] = z;
        b[i] = z;
    }
}

// Adds contiguous fp32 rows [row0, row1) x Hkv x D into the gradient pages of
// one (logical page, KV head): pool row += delta row, one fp32 addition per
// element, no atomics (each element has one owner in a launch). The gradient
// pool is paged like the K/V cache and accumulated in place (gist.science/de
// §2.B, in-place gradient accumulation). 12 bytes of HBM per element: read the
// delta, read and write the pool. Every thread keeps 4 + 4 loads of each
// tensor in flight. A host page recorded as zero (gzero) is written whole
// instead: the delta rows, zeros elsewhere; then the record is dropped.
template <int D>
__global__ void __launch_bounds__(kThreads) grad_accumulate_kernel(float* dkpool, float* dvpool,
        const float* dk, const float* dv, const int32_t* bt, int64_t num_phys, int P, int Hkv,
        int64_t row0, int64_t row1, uint8_t* gzero, int* err) {
    constexpr int V4 = D / 4;                        // float4 per row
    const int64_t lp = row0 / P + blockIdx.x;
    const int h = blockIdx.y;
    const int32_t pp = bt[lp];
    if (pp < 0 || pp >= num_phys) {
        report_error(err, kErrBadPage);
        return;
    }
    const int64_t r_lo = max64(row0, lp * P), r_hi = min64(row1, lp * P + P);
    const int n = (int)(r_hi - r_lo) * V4;           // float4 of this (page, head) per tensor
    const size_t page_off = ((size_t)pp * Hkv + h) * (size_t)P * D + (size_t)(r_lo - lp * P) * D;
    const size_t row_stride4 = (size_t)Hkv * V4;     // delta rows are [row, Hkv, D]
    const size_t src0 = (size_t)(r_lo - row0) * row_stride4 + (size_t)h * V4;
    const size_t tile = (size_t)pp * Hkv + h;
    if (gzero && gzero[tile]) {
        const int lo = (int)(r_lo - lp * P) * V4;    // the delta's float4 range in the tile
        const size_t tile_off = tile * (size_t)P * D;
        for (int t = 0; t < 2; ++t) {
            const float4* src = reinterpret_cast<const float4*>(t == 0 ? dk : dv);
            float4* dst = reinterpret_cast<float4*>((t == 0 ? dkpool : dvpool) + tile_off);
            for (int i = threadIdx.x; i < P * V4; i += kThreads) {
                float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
                const int j = i - lo;
                if (src && j >= 0 && j < n) x = __ldcs(src + src0 + (size_t)(j / V4) * row_stride4 + j % V4);
                dst[i] = x;
            }
        }
        if (threadIdx.x == 0) gzero[tile] = 0;
        return;
    }
    for (int t = 0; t < 2; ++t) {
        const float4* src = reinterpret_cast<const float4*>(t == 0 ? dk : dv);
        if (!src) continue;
        float4* dst = reinterpret_cast<float4*>((t == 0 ? dkpool : dvpool) + page_off);
        for (int base = 0; base < n; base += 4 * kThreads) {
            float4 g[4], x[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = base + u * kThreads + threadIdx.x;
                if (i < n) {
                    g[u] = __ldcs(src + src0 + (size_t)(i / V4) * row_stride4 + i % V4);
                    x[u] = dst[i];
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = base + u * kThreads + threadIdx.x;
                if (i < n)
                    dst[i] = make_float4(x[u].x + g[u].x, x[u].y + g[u].y, x[u].z + g[u].z,
                                         x[u].w + g[u].w);
            }
        }
    }
}

// Copies rows of one (logical page, KV head) into logical-order outputs, 16
// bytes per access (the page rows are contiguous; output rows are Hkv*D apart).
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) gather_kernel(const T* kpool, const T* vpool,
        const float* dkpool, const float* dvpool, const float* reppool, const int32_t* bt,
        int64_t num_phys, int P, int Hkv, int64_t lp0, int64_t len, T* k, T* v, float* dk,
        float* dv, float* rep, const uint8_t* gzero, int* err) {
    constexpr int VT = D * (int)sizeof(T) / 16;     // 16-byte vectors per K/V row
    constexpr int VF = D / 4;                       // 16-byte vectors per gradient row
    const int64_t lp = lp0 + blockIdx.x;            // logical page; outputs start at page lp0
    const int h = blockIdx.y;
    const int32_t pp = bt[lp];
    if (pp < 0 || pp >= num_phys) {
        report_error(err, kErrBadPage);
        return;
    }
    const size_t page_off = ((size_t)pp * Hkv + h) * (size_t)P * D;
    const int rows = (int)min64(P, len - lp * P);
    const size_t out_row0 = (size_t)(lp - lp0) * P;
    if (k || v) {
        const uint4* ks = reinterpret_cast<const uint4*>(kpool + page_off);
        const uint4* vs = reinterpret_cast<const uint4*>(vpool + page_off);
        for (int i = threadIdx.x; i < rows * VT; i += kThreads) {
            const int r = i / VT, c = i % VT;
            const size_t dst = ((out_row0 + r) * Hkv + h) * VT + c;
            if (k) reinterpret_cast<uint4*>(k)[dst] = ks[i];
            if (v) reinterpret_cast<uint4*>(v)[dst] = vs[i];
        }
    }
    if (dk || dv) {
        const float4* gk = reinterpret_cast<const float4*>(dkpool + page_off);
        const float4* gv = reinterpret_cast<const float4*>(dvpool + page_off);
        const bool zero = gzero && gzero[(size_t)pp * Hkv + h];   // recorded zero: memory stale
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int i = threadIdx.x; i < rows * VF; i += kThreads) {
            const int r = i / VF, c = i % VF;
            const size_t dst = ((out_row0 + r) * Hkv + h) * VF + c;
            if (dk) reinterpret_cast<float4*>(dk)[dst] = zero ? z : gk[i];
            if (dv) reinterpret_cast<float4*>(dv)[dst] = zero ? z : gv[i];
        }
    }
    if (rep && threadIdx.x < D)
        rep[((size_t)(lp - lp0) * Hkv + h) * D + threadIdx.x] =
            reppool[((size_t)pp * Hkv + h) * D + threadIdx.x];
}

template <typename T>
cudaError_t append_dispatch_d(const AppendArgs& a, cudaStream_t s, dim3 grid) {
    ProfScope ps("append_kernel", s);
    if (a.d == 128) append_kernel<T, 128><<<grid, kAppThreads, 0, s>>>(a);
    else append_kernel<T, 64><<<grid, kAppThreads, 0, s>>>(a);
    return cudaGetLastError();
}

template <typename T>
cudaError_t gather_dispatch(const pkv_pool* p, const int32_t* bt, int64_t lp0, int64_t len, void* k,
                            void* v, float* dk, float* dv, float* rep, cudaStream_t s) {
    const int P = p->desc.page_size, Hkv = p->desc.n_kv_heads;
    dim3 grid((unsigned)((len + P - 1) / P - lp0), Hkv);
#define PKV_GATHER_ARGS                                                                      \
    static_cast<const T*>(p->k), static_cast<const T*>(p->v), p->dk, p->dv, p->rep, bt,     \
        p->desc.num_phys_pages, P, Hkv, lp0, len, static_cast<T*>(k), static_cast<T*>(v), dk, \
        dv, rep, p->gzero, p->d_err
    ProfScope ps("gather_kernel", s);
    if (p->desc.head_dim == 128) gather_kernel<T, 128><<<grid, kThreads, 0, s>>>(PKV_GATHER_ARGS);
    else gather_kernel<T, 64><<<grid, kThreads, 0, s>>>(PKV_GATHER_ARGS);
#undef PKV_GATHER_ARGS
    return cudaGetLastError();
}

__global__ void bt_upload_kernel(const int32_t* src, int32_t* dst, int64_t n) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        dst[i] = src[i];
}

}  // namespace

cudaError_t launch_bt_upload(const int32_t* src, int32_t* dst, int64_t n, cudaStream_t s) {
    const int blocks = (int)std::min<int64_t>(64, (n + kThreads - 1) / kThreads);
    ProfScope ps("bt_upload_kernel", s);
    bt_upload_kernel<<<blocks, kThreads, 0, s>>>(src, dst, n);
    return cudaGetLastError();
}

cudaError_t launch_append(const AppendArgs& a, cudaStream_t s) {
    const int64_t first = a.old_len / a.P;
    const int64_t last = (a.old_len + a.n_tok - 1) / a.P;
    dim3 grid((unsigned)(last - first + 1), a.Hkv, 2);
    return a.dtype == PKV_BF16 ? append_dispatch_d<__nv_bfloat16>(a, s, grid)
                               : append_dispatch_d<float>(a, s, grid);
}

cudaError_t launch_grad_zero(const pkv_pool* p, const int32_t* d_bt, int64_t p0, int64_t p1,
                             cudaStream_t s) {
    if (p1 <= p0) return cudaSuccess;
    dim3 grid((unsigned)(p1 - p0), p->desc.n_kv_heads);
    ProfScope ps("grad_zero_kernel", s);
    grad_zero_kernel<<<grid, kThreads, 0, s>>>(p->dk, p->dv, d_bt, p0, p->desc.num_phys_pages,
                                               p->desc.n_kv_heads,
                                               p->desc.page_size * p->desc.head_dim, p->d_err);
    return cudaGetLastError();
}

cudaError_t launch_grad_accumulate(const pkv_pool* p, const int32_t* d_bt, int64_t row0,
                                   int64_t n_rows, const float* dk, const float* dv,
                                   cudaStream_t s) {
    if (n_rows <= 0 || (!dk && !dv)) return cudaSuccess;
    const int P = p->desc.page_size, Hkv = p->desc.n_kv_heads;
    const int64_t row1 = row0 + n_rows;
    dim3 grid((unsigned)((row1 - 1) / P - row0 / P + 1), Hkv);
#define PKV_ACC_ARGS \
    p->dk, p->dv, dk, dv, d_bt, p->desc.num_phys_pages, P, Hkv, row0, row1, p->gzero, p->d_err
    ProfScope ps("grad_accumulate_kernel", s);
    if (p->desc.head_dim == 128) grad_accumulate_kernel<128><<<grid, kThreads, 0, s>>>(PKV_ACC_ARGS);
    else grad_accumulate_kernel<64><<<grid, kThreads, 0, s>>>(PKV_ACC_ARGS);
#undef PKV_ACC_ARGS
    return cudaGetLastError();
}

cudaError_t launch_gather(const pkv_pool* p, const int32_t* d_bt, int64_t lp0, int64_t len, void* k,
                          void* v, float* dk, float* dv, float* rep, cudaStream_t s) {
    return p->desc.dtype == PKV_BF16
               ? gather_dispatch<__nv_bfloat16>(p, d_bt, lp0, len, k, v, dk, dv, rep, s)
               : gather_dispatch<float>(p, d_bt, lp0, len, k, v, dk, dv, rep, s);
}

}  // namespace pkv
