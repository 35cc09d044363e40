// Tensor-core (tcgen05) paged chunk attention forward, bf16 in / fp32 accumulate.
//
// Computes, for one query chunk, exact causal softmax attention over every
// key reached through the block table (dense) or over the pages selected for
// each query page (sparse), and saves the row log-sum-exp for the backward
// ("Out of the Memory Barrier": kernels that run forward and backward directly
// on the paged KV cache, gist.science/de §2.B, sciencestack.ai Fig. 3; page
// selection, gist.science/de §2.D).
//
// One CTA per (query tile of 128 rows = one query page, query head); key
// tiles are whole pages (P = 128), fetched by TMA with the physical page
// taken from the block table. Warp roles (224 threads):
//   warp 0      TMA producer: Q once, then K pages into a 3-stage ring.
//   warp 6      TMA producer: V pages into a 2-stage ring.
//   warp 1      MMA issuer (one thread): S_j = Q K_j^T into a double-buffered
//               TMEM tile, then O += P_{j-1} V_{j-1} (O lives in TMEM).
//   warps 2..5  softmax: one thread per query row; reads S_j from TMEM, keeps
//               the running max m and sum l, writes P_j (bf16) to shared
//               memory in the 128-byte-swizzled K-major layout, and rescales
//               O in TMEM only when m grows by more than 2^8 (P <= 256 then,
//               exactly representable range for bf16). Epilogue: O / l, LSE.
// TMEM columns: S0 [0,128), S1 [128,256), O [256,384) of a 512-column block.
#include <cuda_bf16.h>
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace pkv {
namespace {

constexpr int kTile = 128;                   // query rows = keys per tile = head dim
constexpr int kThreads = 224;
constexpr uint32_t kHalfBytes = 128 * 128;   // [128 rows][64 bf16] = 16 KB
constexpr uint32_t kTileBytes = 2 * kHalfBytes;
// Shared-memory tile offsets (bytes from a 1024-aligned base).
// K and V have separate rings: a K stage is free as soon as S_j completes, so
// K loads run kKStages - 1 tiles ahead; a V stage is free after PV_j.
constexpr int kKStages = 3, kVStages = 2;
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kTileBytes;
constexpr uint32_t kOffV = kOffK + kKStages * kTileBytes;
constexpr uint32_t kOffP = kOffV + kVStages * kTileBytes;
constexpr uint32_t kTilesBytes = kOffP + kTileBytes;    // 224 KB
constexpr uint32_t kSmemBytes = kTilesBytes + 1024;     // + alignment slack
constexpr float kRescaleThreshold = 8.0f;               // log2 units

struct FwdParams {
    int Hq, Hkv;
    int64_t q_start, n_q;
    void* o;
    float* lse;
    const int32_t* bt;
    int64_t num_phys;
    const int32_t* sel;
    int kmax;
    int* err;
};

struct __align__(8) FwdBarriers {
    uint64_t q_full;
    uint64_t k_full[kKStages], k_empty[kKStages], v_full[kVStages], v_empty[kVStages];
    uint64_t s_full[2];
    uint64_t p_full;
    uint64_t o_done;
    uint64_t drain;
    uint32_t tmem_base;
    int n_tiles;
};

// Number of key tiles and the logical page of tile j for this CTA.
__device__ __forceinline__ int tile_count(const FwdParams& p, int qt, int kvh) {
    if (!p.sel) return (int)(p.q_start / kTile) + qt + 1;
    const int32_t* row = p.sel + ((size_t)qt * p.Hkv + kvh) * p.kmax;
    int n = 0;
    while (n < p.kmax && row[n] >= 0) ++n;
    return n;
}
__device__ __forceinline__ int32_t tile_page(const FwdParams& p, int qt, int kvh, int j) {
    return p.sel ? p.sel[((size_t)qt * p.Hkv + kvh) * p.kmax + j] : j;
}

using tc::drain_wait;

// One producer warp: streams the K ring (and Q first) or the V ring. The whole
// warp walks the tiles (page indices come 32 at a time from a PageBatch);
// lane 0 issues the copies. A K load never waits behind a V stage in use.
__device__ __forceinline__ void produce_ring(const FwdParams& p, uint8_t* smem, FwdBarriers& B,
                                             const CUtensorMap& tmap_q, const CUtensorMap& tmap,
                                             bool is_k, int qt, int h, int kvh, int nt, int lane) {
    const int nst = is_k ? kKStages : kVStages;
    uint64_t* full = is_k ? B.k_full : B.v_full;
    uint64_t* empty = is_k ? B.k_empty : B.v_empty;
    uint8_t* base = smem + (is_k ? kOffK : kOffV);
    if (lane == 0) {
        tc::prefetch_tmap(&tmap);
        if (is_k) {
            tc::prefetch_tmap(&tmap_q);
            const int q_row0 = qt * kTile;
            tc::mbar_arrive_expect_tx(&B.q_full, kTileBytes);
            tc::tma_load_3d(smem + kOffQ, &tmap_q, &B.q_full, 0, h, q_row0);
            tc::tma_load_3d(smem + kOffQ + kHalfBytes, &tmap_q, &B.q_full, 64, h, q_row0);
        }
    }
    tc::PageBatch pages;
    pages.init(p.bt, p.sel ? p.sel + ((size_t)qt * p.Hkv + kvh) * p.kmax : nullptr, nt, lane);
    int issued = 0;
    for (int j = 0; j < nt; ++j) {
        const int st = j % nst;
        if (j >= nst &&
            !__all_sync(0xffffffffu, tc::mbar_wait(&empty[st], ((j / nst) - 1) & 1, p.err)))
            break;
        const int32_t pp = pages.get(j);
        if (pp < 0 || pp >= p.num_phys) {
            if (lane == 0) report_error(p.err, kErrBadPage);
            break;
        }
        if (lane == 0) {
            const int row = (int)(((int64_t)pp * p.Hkv + kvh) * kTile);
            uint8_t* dst = base + st * kTileBytes;
            tc::mbar_arrive_expect_tx(&full[st], kTileBytes);
            tc::tma_load_2d(dst, &tmap, &full[st], 0, row);
            tc::tma_load_2d(dst + kHalfBytes, &tmap, &full[st], 64, row);
        }
        issued = j + 1;
    }
    // Make sure none of this CTA's copies is still landing when it exits.
    if (lane == 0) {
        if (is_k) drain_wait(&B.q_full, 0);
        for (int j = max(0, issued - nst); j < issued; ++j) drain_wait(&full[j % nst], (j / nst) & 1);
    }
}

__global__ void __launch_bounds__(kThreads, 1)
fwd_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
              const __grid_constant__ CUtensorMap tmap_v, FwdParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ FwdBarriers B;

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int qt = (int)gridDim.x - 1 - (int)blockIdx.x;        // longest tiles first
    const int h = blockIdx.y;
    const int kvh = h / (p.Hq / p.Hkv);

    if (threadIdx.x == 0) {
        tc::mbar_init(&B.q_full, 1);
        for (int s = 0; s < kKStages; ++s) {
            tc::mbar_init(&B.k_full[s], 1);
            tc::mbar_init(&B.k_empty[s], 1);
        }
        for (int s = 0; s < kVStages; ++s) {
            tc::mbar_init(&B.v_full[s], 1);
            tc::mbar_init(&B.v_empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) tc::mbar_init(&B.s_full[s], 1);
        tc::mbar_init(&B.p_full, 128);
        tc::mbar_init(&B.o_done, 1);
        tc::mbar_init(&B.drain, 1);
        B.n_tiles = tile_count(p, qt, kvh);
        tc::fence_barrier_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(&B.tmem_base, 512);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = B.tmem_base;
    const int nt = B.n_tiles;

    if (warp == 0) {
        // ------------------------------------------------------------ Q + K producer
        produce_ring(p, smem, B, tmap_q, tmap_k, true, qt, h, kvh, nt, lane);
    } else if (warp == kThreads / 32 - 1) {
        // ------------------------------------------------------------ V producer
        produce_ring(p, smem, B, tmap_q, tmap_v, false, qt, h, kvh, nt, lane);
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs the loop (warp-uniform descriptors); one elected
        // lane issues the tcgen05 instructions and commits.
        const bool leader = tc::elect_one_sync();
        const uint32_t idesc = tc::idesc_bf16(128, 128, false, false);       // S = Q K^T
        const uint32_t idesc_pv = tc::idesc_bf16(128, 128, false, true);     // O += P V
        // Base descriptors; each MMA advances them by a compile-time offset.
        const uint64_t dq0 = tc::sdesc(tc::smem_u32(smem + kOffQ), 16, 1024);
        const uint64_t dp0 = tc::sdesc(tc::smem_u32(smem + kOffP), 16, 1024);
        const uint32_t tmem_o = tmem + 256;
        bool ok = tc::warp_wait(&B.q_full, 0, p.err);
        auto issue_pv = [&](int i) -> bool {
            if (!tc::warp_wait(&B.p_full, i & 1, p.err)) return false;
            if (!tc::warp_wait(&B.v_full[i % kVStages], (i / kVStages) & 1, p.err)) return false;
            tc::tc_fence_after();
            // A = P [128 q][128 keys] K-major; B = V [128 keys][128 d] MN-major:
            // 16 keys = 2 K-groups of 8 rows (1024 B apart); d spans the two
            // 64-column halves (16 KB apart).
            const uint64_t b0 = tc::sdesc(tc::smem_u32(smem + kOffV + (i % kVStages) * kTileBytes),
                                          kHalfBytes, 1024);
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    tc::mma_bf16(tmem_o, tc::sdesc_at(dp0, (kk >> 2) * kHalfBytes + (kk & 3) * 32),
                                 tc::sdesc_at(b0, kk * 2048), idesc_pv, (i > 0 || kk > 0) ? 1u : 0u);
                tc::mma_commit(&B.o_done);
                tc::mma_commit(&B.v_empty[i % kVStages]);
            }
            __syncwarp();
            return true;
        };
        for (int j = 0; ok && j < nt; ++j) {
            const int ks = j % kKStages;
            if (!tc::warp_wait(&B.k_full[ks], (j / kKStages) & 1, p.err)) { ok = false; break; }
            tc::tc_fence_after();
            const uint64_t dk0 = tc::sdesc(tc::smem_u32(smem + kOffK + ks * kTileBytes), 16, 1024);
            const uint32_t tmem_s = tmem + (j & 1) * 128;
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t koff = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
                    tc::mma_bf16(tmem_s, tc::sdesc_at(dq0, koff), tc::sdesc_at(dk0, koff), idesc,
                                 kk > 0 ? 1u : 0u);
                }
                tc::mma_commit(&B.s_full[j & 1]);
                tc::mma_commit(&B.k_empty[ks]);
            }
            __syncwarp();
            if (j > 0 && !issue_pv(j - 1)) { ok = false; break; }
        }
        if (ok && nt > 0) issue_pv(nt - 1);
        // Drain: nothing of ours may still run on the tensor core at exit.
        if (leader) {
            tc::mma_commit(&B.drain);
            drain_wait(&B.drain, 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax (128 threads)
        const int quad = warp & 3;                    // TMEM lane quadrant of this warp
        const int row = quad * 32 + lane;             // query row within the tile
        const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
        const float sl2 = rsqrtf(128.f) * kLog2e;
        const int64_t q_local = (int64_t)qt * kTile + row;
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        uint8_t* sP = smem + kOffP;
        for (int j = 0; j < nt; ++j) {
            const int st = j & 1;
            ok = tc::mbar_wait(&B.s_full[st], (j >> 1) & 1, p.err);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc::tc_fence_after();
            // Raw logits q.k; the scale is folded into the exp2 argument below.
            float x[128];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t r[32];
                tc::tmem_ld32(lane_base + st * 128 + c * 32, r);
                tc::tmem_wait_ld(r);
#pragma unroll
                for (int e = 0; e < 32; ++e) x[c * 32 + e] = __uint_as_float(r[e]);
            }
            if (j == nt - 1) {                        // own page: causal mask (key col > row)
#pragma unroll
                for (int c = 0; c < 128; ++c)
                    if (c > row) x[c] = -INFINITY;
            }
            // Row max with 8 independent chains (a single chain of 128 dependent
            // max operations would dominate the tile's latency).
            float mpart[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) mpart[k] = x[k];
#pragma unroll
            for (int c = 8; c < 128; ++c) mpart[c & 7] = fmaxf(mpart[c & 7], x[c]);
#pragma unroll
            for (int k = 4; k > 0; k >>= 1)
#pragma unroll
                for (int i = 0; i < k; ++i) mpart[i] = fmaxf(mpart[i], mpart[i + k]);
            const float mx = mpart[0] * sl2;          // scaled, log2 units
            float alpha = 1.f;
            bool rescale = false;
            if (mx > m + kRescaleThreshold) {
                alpha = (m == -INFINITY) ? 0.f : fast_exp2(m - mx);
                m = mx;
                rescale = true;
            }
            l *= alpha;
            uint32_t pk[64];
            float lpart[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) lpart[k] = 0.f;
            const float neg_m = -m;
#pragma unroll
            for (int c = 0; c < 64; ++c) {
                const float p0 = fast_exp2(fmaf(x[2 * c], sl2, neg_m));
                const float p1 = fast_exp2(fmaf(x[2 * c + 1], sl2, neg_m));
                pk[c] = pack_bf16x2(p0, p1);
                // Normalise by the sum of the bf16 weights the tensor core multiplies, so
                // O is a convex combination of values whatever the rounding of P.
                lpart[c & 7] += bf16lo(pk[c]) + bf16hi(pk[c]);
            }
#pragma unroll
            for (int k = 4; k > 0; k >>= 1)
#pragma unroll
                for (int i = 0; i < k; ++i) lpart[i] += lpart[i + k];
            l += lpart[0];
            if (j > 0) {                              // PV_{j-1} done: P buffer free, O stable
                ok = tc::mbar_wait(&B.o_done, (j - 1) & 1, p.err);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc::tc_fence_after();
                if (__any_sync(0xffffffffu, rescale)) {
                    const float f = rescale ? alpha : 1.f;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t r[32];
                        tc::tmem_ld32(lane_base + 256 + c * 32, r);
                        tc::tmem_wait_ld(r);
#pragma unroll
                        for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * f);
                        tc::tmem_st32(lane_base + 256 + c * 32, r);
                    }
                    tc::tmem_wait_st();
                }
            }
            // P row -> shared memory, 128-byte swizzle, keys 0..63 | 64..127 halves.
#pragma unroll
            for (int ch = 0; ch < 16; ++ch) {
                uint8_t* base = sP + (ch >> 3) * kHalfBytes;
                *reinterpret_cast<uint4*>(base + tc::sw128_offset(row, ch & 7)) =
                    make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
            }
            tc::fence_proxy_async_smem();
            tc::tc_fence_before();
            tc::mbar_arrive(&B.p_full);
        }
        if (ok && nt > 0) {
            ok = tc::mbar_wait(&B.o_done, (nt - 1) & 1, p.err);
            ok = __all_sync(0xffffffffu, ok);
        }
        if (ok && nt > 0) {
            tc::tc_fence_after();
            const float inv = 1.f / l;
            const bool valid = q_local < p.n_q;
            __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.o) + ((size_t)q_local * p.Hq + h) * kTile;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t r[32];
                tc::tmem_ld32(lane_base + 256 + c * 32, r);
                tc::tmem_wait_ld(r);
                if (valid) {
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(r[8 * v + 0]) * inv, __uint_as_float(r[8 * v + 1]) * inv);
                        w.y = pack_bf16x2(__uint_as_float(r[8 * v + 2]) * inv, __uint_as_float(r[8 * v + 3]) * inv);
                        w.z = pack_bf16x2(__uint_as_float(r[8 * v + 4]) * inv, __uint_as_float(r[8 * v + 5]) * inv);
                        w.w = pack_bf16x2(__uint_as_float(r[8 * v + 6]) * inv, __uint_as_float(r[8 * v + 7]) * inv);
                        *reinterpret_cast<uint4*>(orow + c * 32 + v * 8) = w;
                    }
                }
            }
            if (valid) p.lse[(size_t)h * p.n_q + q_local] = (m + log2f(l)) * kLn2;
        }
    }

    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, 512);
    }
}

}  // namespace

bool tc_supported(const AttnArgs& a) {
    return a.dtype == PKV_BF16 && a.d == 128 && a.P == 128 && a.tmap_k && a.tmap_v &&
           (reinterpret_cast<uintptr_t>(a.q) & 15) == 0;
}

cudaError_t launch_attn_fwd_tc(const AttnArgs& a, cudaStream_t s) {
    CUtensorMap tq;
    std::string why;
    if (!make_tmap_3d(&tq, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 128, a.Hq, a.n_q, 256,
                      (uint64_t)a.Hq * 256, 64, 1, 128, &why))
        return cudaErrorInvalidValue;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    FwdParams p{};
    p.Hq = a.Hq; p.Hkv = a.Hkv; p.q_start = a.q_start; p.n_q = a.n_q;
    p.o = a.o; p.lse = a.lse; p.bt = a.bt; p.num_phys = a.num_phys;
    p.sel = a.sel; p.kmax = a.kmax; p.err = a.err;
    dim3 grid((unsigned)((a.n_q + kTile - 1) / kTile), a.Hq);
    ProfScope ps("fwd_tc_kernel", s);
    fwd_tc_kernel<<<grid, kThreads, kSmemBytes, s>>>(tq, *a.tmap_k, *a.tmap_v, p);
    return cudaGetLastError();
}

}  // namespace pkv
