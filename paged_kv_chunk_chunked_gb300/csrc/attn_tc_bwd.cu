// Tensor-core (tcgen05) paged chunk attention backward, bf16 in / fp32 accumulate.
//
// Recomputes P from the saved LSE (activation recomputation, "Out of the
// Memory Barrier", gist.science/de §2.A) and computes, for one query chunk,
//   dQ_i  = s sum_j P_ij (dP_ij - D_i) k_j,       dP_ij = dO_i . v_j,
//   dK_j += s sum_{h,i} P_ij (dP_ij - D_i) q_i,   dV_j += sum_{h,i} P_ij dO_i,
// adding dK/dV in place into the paged fp32 gradient pool (gist.science/de
// §2.B: gradients accumulated in place; sciencestack.ai Fig. 3).
// D_i = rowsum(dO_i * O_i) comes from the row-dot kernel run before these.
//
// Two kernels, so that dQ needs no atomics and dK/dV one addition per element
// per CTA:
//   bwd_kv_tc_kernel  one CTA per (key page, KV head) -- or per share of its
//                     iterations when the grid is small. K of the page sits in
//                     tensor memory, V in shared memory; the CTA walks every
//                     64-query tile of the chunk that sees the page, for each
//                     of the g query heads of the group, and accumulates dK
//                     and dV in tensor memory. At the end it adds them into
//                     the page's gradient rows with vectorised
//                     red.global.add.v4.f32 (the red keeps earlier chunks'
//                     contributions and those of the page's other CTAs).
//   bwd_q_tc_kernel   one CTA per (128-query tile, query head); walks the
//                     visible keys a page (128 keys) at a time and accumulates
//                     dQ in tensor memory, written once as bf16.
// Warp roles in both: warp 0 TMA producer; warp 1 issues the S/dP (or
// S^T/dP^T) MMAs; warps 2..9 two softmax warpgroups, one thread per
// accumulator row, splitting each tile's columns; warp 10 issues the MMAs
// that consume the softmax output (dV/dK, or dQ). The S/dP buffer is released
// as soon as the softmax warps have read it, so the tensor core computes tile
// t+1 while they work on tile t. Wherever tensor memory has room, the MMAs
// take their A operand from it rather than from shared memory (an A operand in
// shared memory costs the tensor core ~33 extra cycles per instruction on this
// part): K, P^T and dS^T in the dK/dV kernel, Q and dS in the dQ kernel.
#include <cuda_bf16.h>
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace pkv {
namespace {

using tc::drain_wait;

// Warp 0 TMA; warp 1 issues the S/dP (or S^T/dP^T) MMAs; warps 2..9 two softmax
// warpgroups; warp 10 issues the MMAs that consume their output (dK/dV or dQ).
// An MMA issue blocks its thread for about the MMA's run time, so a single
// issuer would hold S(t+1) back behind the products of tile t.
constexpr int kThreads = 352;
constexpr int kWarpG = 10;
constexpr int kSoftmaxThreads = 256;
constexpr uint32_t KB = 1024;

struct BwdParams {
    int Hq, Hkv;
    int64_t q_start, n_q;
    const void* q;             // [n_q, Hq, d] bf16
    const void* kpool;         // [pages, Hkv, 128, d] bf16 (the tensor maps' base)
    const float* lse;          // [Hq, n_q]
    float* Dbuf;               // [Hq, n_q]: D = rowsum(dO * O), written by the dQ kernel
    void* dq;                  // [n_q, Hq, d] bf16
    float* dkpool;
    float* dvpool;
    const int32_t* bt;
    int64_t num_phys;
    const int32_t* sel;        // sparse: [n_qp, Hkv, kmax] selected pages, or null
    int kmax;
    int kv_splits;             // dK/dV kernel: CTAs per (page, KV head)
    const int32_t* pagelist;   // sparse: [count, pages...] the pages some query page lists
    const void* o;             // forward output (the dQ kernel computes D = rowsum(dO * O))
    const uint64_t* selmask;   // sparse, or null: [key page][KV head][words] query pages listing the page
    int* err;
};

// Query pages per chunk the sparse dK/dV kernel lists in shared memory (3
// bytes each): chunks of up to 262144 tokens at page 128. Longer chunks run
// on the CUDA-core kernel.
constexpr int kMaxSelQp = 2048;



// ============================================================================ dK / dV

// Shared-memory layout (offsets from a 1024-aligned base).
// Q/dO stage for tile t+1 is the one tile t-3 used: the load has two
// iterations of slack behind the gradient products of tile t-2.
// Every A operand except V lives in tensor memory: K (placed once by the
// softmax warps, the A of every S^T MMA), P^T and dS^T (written by the softmax
// warps, the A of the dV and dK MMAs). S^T/dP^T are single-buffered and
// released as soon as the softmax warps have read them (s_free), so S^T(t+1)
// overlaps their work on tile t; P^T/dS^T are rewritten once the gradient
// MMAs of the previous tile have read them (p_free).
constexpr int kv_STAGES = 4;
// Head dimension D = 128 or 64: a page (or a Q/dO tile) of one head is D / 64
// blocks of 64 columns.
template <int D> struct KVLayout {
    static_assert(D == 64 || D == 128, "head dim 64 or 128");
    static constexpr uint32_t kV = 0;                          // [128 keys][D]: D/64 16 KB blocks
    static constexpr uint32_t kQ = (D / 64) * 16 * KB;         // stages x [64 q][D]: D/64 8 KB blocks
    static constexpr uint32_t kQStage = (D / 64) * 8 * KB;
    static constexpr uint32_t kdO = kQ + kv_STAGES * kQStage;
    static constexpr uint32_t kSTAT = kdO + kv_STAGES * kQStage;   // stages x (64 lse*log2e + 64 D) floats
    static constexpr uint32_t kSMEM = kSTAT + kv_STAGES * 512 + 1024;
};
// Tensor-memory columns: S^T, dP^T (64 fp32 each), P^T, dS^T (64 bf16 = 32
// each), K (D bf16 = D/2), dK, dV accumulators (D fp32 each).
constexpr uint32_t kv_TS = 0, kv_TDP = 64, kv_TP = 128, kv_TDS = 160, kv_TK = 192, kv_TDK = 256,
                   kv_TDV = 384;

struct __align__(8) KVBar {
    uint64_t kv_full;
    uint64_t qdo_full[kv_STAGES], qdo_empty[kv_STAGES];
    uint64_t k_tmem;                 // K in TMEM (softmax threads)
    uint64_t s_full, s_free;
    uint64_t p_full, p_free;
    uint64_t acc_done;
    uint64_t drain[2];
    uint32_t tmem_base;
    int n_i;                         // 64-query tiles per head
    int epi_bad[2];                  // a warpgroup's epilogue lost a wait: its boxes are not added
    int16_t tiles[2 * kMaxSelQp];    // sparse: the tiles, ascending
    uint8_t sel_flag[kMaxSelQp];
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
bwd_kv_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_dk,
                 const __grid_constant__ CUtensorMap tm_dv, BwdParams p) {
    using L = KVLayout<D>;
    constexpr uint32_t kv_V = L::kV, kv_Q = L::kQ, kv_dO = L::kdO, kv_STAT = L::kSTAT;
    constexpr uint32_t kQS = L::kQStage;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ KVBar B;
    float* stat = reinterpret_cast<float*>(smem + kv_STAT);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    // Dense: grid (key page * splits + split, KV head); the CTAs that share a
    // page run side by side, so their gradient additions meet in L2 rather
    // than in DRAM. Sparse: grid (KV head, position in the chunk's selection
    // union) -- the union's CTAs are dispatched first, those past its end exit
    // at once.
    const int n_split = (int)p.kv_splits;
    int j, split, kvh;
    if (p.pagelist) {
        const int idx = (int)blockIdx.y;
        if (idx >= p.pagelist[0]) return;            // the whole CTA, before any barrier
        j = p.pagelist[1 + idx];
        split = 0;
        kvh = (int)blockIdx.x;
    } else {
        j = (int)blockIdx.x / n_split;               // logical key page
        split = (int)blockIdx.x % n_split;
        kvh = (int)blockIdx.y;
    }
    const int g = p.Hq / p.Hkv;
    const int64_t kfirst = (int64_t)j * 128;
    const int n_qt = (int)((p.n_q + 63) / 64);
    const int i0 = kfirst > p.q_start ? (int)((kfirst - p.q_start) / 64) : 0;
    const int32_t pp = p.bt[j];
    const bool page_ok = pp >= 0 && pp < p.num_phys;

    if (threadIdx.x == 0) {
        tc::mbar_init(&B.kv_full, 1);
        for (int s = 0; s < kv_STAGES; ++s) {
            tc::mbar_init(&B.qdo_full[s], 32);
            tc::mbar_init(&B.qdo_empty[s], 1);
        }
        tc::mbar_init(&B.k_tmem, kSoftmaxThreads);
        tc::mbar_init(&B.s_full, 1);
        tc::mbar_init(&B.s_free, kSoftmaxThreads);
        tc::mbar_init(&B.p_full, kSoftmaxThreads);
        tc::mbar_init(&B.p_free, 1);
        tc::mbar_init(&B.acc_done, 1);
        tc::mbar_init(&B.drain[0], 1);
        tc::mbar_init(&B.drain[1], 1);
        B.epi_bad[0] = B.epi_bad[1] = 0;
        tc::fence_barrier_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(&B.tmem_base, 512);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    // The page's V streams in while the query tiles are being listed.
    if (threadIdx.x == 0 && page_ok) {
        tc::prefetch_tmap(&tm_q);
        tc::prefetch_tmap(&tm_do);
        tc::mbar_arrive_expect_tx(&B.kv_full, (D / 64) * 16 * KB);
#pragma unroll
        for (int b = 0; b < D / 64; ++b)
            tc::tma_load_2d(smem + kv_V + b * 16 * KB, &tm_v, &B.kv_full, 64 * b,
                            (int)(((int64_t)pp * p.Hkv + kvh) * 128));
    }
    // Softmax threads: their K row (head dims [D/2 wg, D/2 wg + D/2)) is loaded
    // now and goes to tensor memory once the tiles are known.
    constexpr int NW = D / 4;
    uint32_t kw[NW];
    if (warp >= 2 && warp < 2 + kSoftmaxThreads / 32 && page_ok) {
        const int r = (warp & 3) * 32 + lane;
        const uint4* src = reinterpret_cast<const uint4*>(
            static_cast<const __nv_bfloat16*>(p.kpool) + (((size_t)pp * p.Hkv + kvh) * 128 + r) * D +
            ((warp - 2) >> 2) * (D / 2));
#pragma unroll
        for (int v = 0; v < NW / 4; ++v) {
            const uint4 u = __ldg(src + v);
            kw[4 * v] = u.x; kw[4 * v + 1] = u.y; kw[4 * v + 2] = u.z; kw[4 * v + 3] = u.w;
        }
    }

    // Query tiles that see this page: dense, every tile from i0 on; sparse, the
    // two 64-query halves of every query page whose selection lists page j --
    // read from the page's query-page mask when the union kernel wrote one,
    // else found by scanning the whole selection.
    if (p.sel && p.selmask) {
        if (warp == 0) {
            // Lane l holds mask word l (query pages 64 l ..); set bits in
            // ascending order, two tiles per query page.
            const int n_qp = (int)((p.n_q + 127) / 128);
            const int W = (n_qp + 63) / 64;                      // <= 32 (kMaxSelQp)
            const uint64_t m = lane < W ? p.selmask[((size_t)j * p.Hkv + kvh) * W + lane] : 0ull;
            const int c = __popcll(m);
            int incl = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            int pos = 2 * (incl - c);
            for (uint64_t mm = m; mm; mm &= mm - 1) {
                const int qp = lane * 64 + __ffsll((long long)mm) - 1;
                B.tiles[pos] = (int16_t)(2 * qp);
                if (2 * qp + 1 < n_qt) B.tiles[pos + 1] = (int16_t)(2 * qp + 1);
                pos += 2;
            }
            // Only the last query page can hold a single 64-query tile (odd n_qt).
            const int last = n_qp - 1;
            // (Both shuffles run on every lane, outside the lane-0 store.)
            const bool last_listed = (__shfl_sync(0xffffffffu, m, last / 64) >> (last % 64)) & 1ull;
            const int total = __shfl_sync(0xffffffffu, incl, 31);
            if (lane == 0) B.n_i = 2 * total - (((n_qt & 1) && last_listed) ? 1 : 0);
        }
    } else if (p.sel) {
        // Every thread checks a slice of all entries (coalesced, independent loads).
        const int n_qp = (int)((p.n_q + 127) / 128);
        for (int qp = threadIdx.x; qp < n_qp; qp += kThreads) B.sel_flag[qp] = 0;
        __syncthreads();
        const int n_ent = n_qp * p.kmax;
        for (int e = threadIdx.x; e < n_ent; e += kThreads) {
            const int qp = e / p.kmax, k = e - qp * p.kmax;
            if (p.sel[((size_t)qp * p.Hkv + kvh) * p.kmax + k] == j) B.sel_flag[qp] = 1;
        }
        __syncthreads();
        if (warp == 0) {
            // Compaction, 32 query pages per ballot; only the last query page
            // can hold a single 64-query tile (odd n_qt), and it lists last.
            int n = 0;
            for (int q0 = 0; q0 < n_qp; q0 += 32) {
                const int qp = q0 + lane;
                const bool f = qp < n_qp && B.sel_flag[qp];
                const unsigned m = __ballot_sync(0xffffffffu, f);
                if (f) {
                    const int pos = n + 2 * __popc(m & ((1u << lane) - 1u));
                    B.tiles[pos] = (int16_t)(2 * qp);
                    if (2 * qp + 1 < n_qt) B.tiles[pos + 1] = (int16_t)(2 * qp + 1);
                }
                n += 2 * __popc(m);
            }
            if (lane == 0) B.n_i = n - (((n_qt & 1) && B.sel_flag[n_qp - 1]) ? 1 : 0);
        }
    } else if (threadIdx.x == 0) {
        B.n_i = n_qt - i0;
    }
    __syncthreads();
    const uint32_t tmem = B.tmem_base;
    const int n_i = B.n_i;
    // A page no query tile uses needs no valid slot (sparse, staged pools).
    if (threadIdx.x == 0 && !page_ok && n_i > 0) report_error(p.err, kErrBadPage);
    // Iterations (head, 64-query tile), t = head * n_i + tile; split takes the
    // share [t_base, t_base + T) of them (the gradient epilogue adds, so any
    // partition of the iterations gives the same sums).
    const int t_all = n_i * g;
    const int t_base = (int)(((int64_t)t_all * split) / n_split);
    const int T = (int)(((int64_t)t_all * (split + 1)) / n_split) - t_base;
    auto tile_of = [&](int t) -> int {
        const int u = (t_base + t) % n_i;
        return p.sel ? (int)B.tiles[u] : i0 + u;
    };
    auto head_of = [&](int t) -> int { return kvh * g + (t_base + t) / n_i; };

    if (!page_ok || T == 0) {
        // No tile: only V's copy (issued for a valid page) is waited for.
        if (threadIdx.x == 0 && page_ok) drain_wait(&B.kv_full, 0);
    } else if (warp == 0) {
        // ---------------------------------------------------------------- producer
        // Per-query statistics of tile t (log2e * LSE, +inf past the chunk, and D),
        // two columns per lane; loaded one tile ahead so their latency overlaps
        // the wait for the next free stage.
        auto load_stats = [&](int t, float (&s)[4]) {
            if (t >= T) return;
            const int h = head_of(t);
            const int i = tile_of(t);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int64_t q = (int64_t)i * 64 + lane * 2 + e;
                const bool v = q < p.n_q;
                s[e] = v ? __ldg(p.lse + (size_t)h * p.n_q + q) * kLog2e : INFINITY;
                s[2 + e] = v ? __ldg(p.Dbuf + (size_t)h * p.n_q + q) : 0.f;
            }
        };
        int issued = 0;
        auto step = [&](int t, const float (&use)[4], float (&fill)[4]) -> bool {
            const int st = t % kv_STAGES;
            if (t >= kv_STAGES &&
                !__all_sync(0xffffffffu, tc::mbar_wait(&B.qdo_empty[st], ((t / kv_STAGES) - 1) & 1, p.err)))
                return false;
            if (lane == 0) {
                const int h = head_of(t);
                const int i = tile_of(t);
                uint8_t* q_dst = smem + kv_Q + st * kQS;
                uint8_t* do_dst = smem + kv_dO + st * kQS;
                tc::mbar_expect_tx(&B.qdo_full[st], 2 * kQS);
#pragma unroll
                for (int b = 0; b < D / 64; ++b) {
                    tc::tma_load_3d(q_dst + b * 8 * KB, &tm_q, &B.qdo_full[st], 64 * b, h, i * 64);
                    tc::tma_load_3d(do_dst + b * 8 * KB, &tm_do, &B.qdo_full[st], 64 * b, h, i * 64);
                }
            }
            load_stats(t + 1, fill);
            float* sst = stat + st * 128;
            sst[lane * 2] = use[0];
            sst[lane * 2 + 1] = use[1];
            sst[64 + lane * 2] = use[2];
            sst[64 + lane * 2 + 1] = use[3];
            tc::mbar_arrive(&B.qdo_full[st]);           // 32 arrivals + the tx bytes
            issued = t + 1;
            return true;
        };
        float sa[4], sb[4];
        load_stats(0, sa);
        for (int t = 0; t < T; t += 2) {
            if (!step(t, sa, sb)) break;
            if (t + 1 < T && !step(t + 1, sb, sa)) break;
        }
        if (lane == 0) {
            drain_wait(&B.kv_full, 0);
            for (int t = max(0, issued - kv_STAGES); t < issued; ++t)
                drain_wait(&B.qdo_full[t % kv_STAGES], (t / kv_STAGES) & 1);
        }
    } else if (warp == 1 || warp == kWarpG) {
        // ---------------------------------------------------------------- MMA issuers
        // Warp 1: S^T/dP^T(t); warp kWarpG: dV/dK(t). Each whole warp runs its
        // loop (warp-uniform descriptors); the elected lane issues.
        const bool leader = tc::elect_one_sync();
        const uint32_t id_s = tc::idesc_bf16(128, 64, false, false);    // S^T = K Q^T
        const uint32_t id_g = tc::idesc_bf16(128, D, false, true);      // dV += P^T dO
        const uint32_t t_dK = tmem + kv_TDK, t_dV = tmem + kv_TDV;
        const uint32_t t_S = tmem + kv_TS, t_dP = tmem + kv_TDP, t_K = tmem + kv_TK;
        bool ok = true;
        // Base descriptors; each MMA advances them by a compile-time offset.
        const uint64_t dV0 = tc::sdesc(tc::smem_u32(smem + kv_V), 16, 1024);
        const uint64_t dQk0 = tc::sdesc(tc::smem_u32(smem + kv_Q), 16, 1024);        // K-major
        const uint64_t ddOk0 = tc::sdesc(tc::smem_u32(smem + kv_dO), 16, 1024);
        const uint64_t dQm0 = tc::sdesc(tc::smem_u32(smem + kv_Q), 8 * KB, 1024);    // MN-major
        const uint64_t ddOm0 = tc::sdesc(tc::smem_u32(smem + kv_dO), 8 * KB, 1024);
        auto issue_s = [&](int t) -> bool {
            const int st = t % kv_STAGES;
            if (!tc::warp_wait(&B.qdo_full[st], (t / kv_STAGES) & 1, p.err)) return false;
            if (t > 0 && !tc::warp_wait(&B.s_free, (t - 1) & 1, p.err)) return false;
            tc::tc_fence_after();
            const uint32_t so = st * kQS;
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {   // K = d: 16 per MMA (8 columns of K)
                    const uint32_t ob = (kk >> 2) * 8 * KB + (kk & 3) * 32;
                    tc::mma_bf16_ts(t_S, t_K + kk * 8, tc::sdesc_at(dQk0, so + ob), id_s, kk > 0 ? 1u : 0u);
                }
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t oa = (kk >> 2) * 16 * KB + (kk & 3) * 32;
                    const uint32_t ob = (kk >> 2) * 8 * KB + (kk & 3) * 32;
                    tc::mma_bf16(t_dP, tc::sdesc_at(dV0, oa), tc::sdesc_at(ddOk0, so + ob), id_s,
                                 kk > 0 ? 1u : 0u);
                }
                tc::mma_commit(&B.s_full);
            }
            __syncwarp();
            return true;
        };
        auto issue_grad = [&](int t) -> bool {
            const int st = t % kv_STAGES;
            if (!tc::warp_wait(&B.p_full, t & 1, p.err)) return false;
            tc::tc_fence_after();
            const uint32_t so = st * kQS;
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)      // K = 64 queries, 16 per MMA (8 columns)
                    tc::mma_bf16_ts(t_dV, tmem + kv_TP + kk * 8, tc::sdesc_at(ddOm0, so + kk * 2048),
                                    id_g, (t > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc::mma_bf16_ts(t_dK, tmem + kv_TDS + kk * 8, tc::sdesc_at(dQm0, so + kk * 2048),
                                    id_g, (t > 0 || kk > 0) ? 1u : 0u);
                tc::mma_commit(&B.qdo_empty[st]);
                tc::mma_commit(&B.p_free);
            }
            __syncwarp();
            return true;
        };
        // The Q/dO stage of tile t is released by the gradient products of t,
        // which start only after the softmax has seen S^T(t) complete.
        const int role = warp == 1 ? 0 : 1;
        if (role == 0) {
            ok = tc::warp_wait(&B.kv_full, 0, p.err) && tc::warp_wait(&B.k_tmem, 0, p.err);
            for (int t = 0; ok && t < T; ++t) ok = issue_s(t);
        } else {
            for (int t = 0; ok && t < T; ++t) ok = issue_grad(t);
            if (ok && leader) tc::mma_commit(&B.acc_done);
        }
        if (leader) {
            tc::mma_commit(&B.drain[role]);
            drain_wait(&B.drain[role], 0);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- softmax-grad warps
        // Two warpgroups: warpgroup wg handles query columns [32 wg, 32 wg + 32)
        // of every key row (TMEM lane quadrant = warp % 4).
        const int wg = (warp - 2) >> 2;
        const int quad = warp & 3;
        const int r = quad * 32 + lane;                      // key row of the page
        const int64_t kpos = kfirst + r;
        const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
        const float sl2 = rsqrtf((float)D) * kLog2e;
        {
            // K row r, head dims [D/2 wg, D/2 wg + D/2) -> TMEM columns kv_TK + D/4 wg ..
            if constexpr (D == 128) tc::tmem_st32(lane_base + kv_TK + wg * 32, kw);
            else tc::tmem_st16(lane_base + kv_TK + wg * 16, kw);
            tc::tmem_wait_st();
            tc::tc_fence_before();
            tc::mbar_arrive(&B.k_tmem);
        }
        bool ok = true;
        for (int t = 0; t < T; ++t) {
            const int st = t % kv_STAGES;
            ok = tc::mbar_wait(&B.s_full, t & 1, p.err) &&
                 tc::mbar_wait(&B.qdo_full[st], (t / kv_STAGES) & 1, p.err);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc::tc_fence_after();
            const int i = tile_of(t);
            const int64_t q0 = p.q_start + (int64_t)i * 64 + wg * 32;   // position of my column 0
            const float* sst = stat + st * 128 + wg * 32;
            uint32_t sv[32], dv[32];
            tc::tmem_ld32(lane_base + kv_TS + wg * 32, sv);
            tc::tmem_ld32(lane_base + kv_TDP + wg * 32, dv);
            tc::tmem_wait_ld(sv);
            tc::tmem_wait_ld(dv);
            tc::tc_fence_before();
            tc::mbar_arrive(&B.s_free);                      // S^T/dP^T may be overwritten
            uint32_t pw[16], dw[16];
            // The columns' statistics, four at a time (one 16-byte broadcast load each).
            const float4* l4 = reinterpret_cast<const float4*>(sst);
            const float4* d4 = reinterpret_cast<const float4*>(sst + 64);
            auto grad4 = [&](int c, bool mask) {
                const float4 l = l4[c / 4], dd = d4[c / 4];
                const float lv[4] = {l.x, l.y, l.z, l.w}, dl[4] = {dd.x, dd.y, dd.z, dd.w};
                float pr[4], dr[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float pv = fast_exp2(fmaf(__uint_as_float(sv[c + e]), sl2, -lv[e]));
                    if (mask && kpos > q0 + c + e) pv = 0.f;
                    pr[e] = pv;
                    dr[e] = pv * (__uint_as_float(dv[c + e]) - dl[e]);
                }
                pw[c / 2] = pack_bf16x2(pr[0], pr[1]);
                pw[c / 2 + 1] = pack_bf16x2(pr[2], pr[3]);
                dw[c / 2] = pack_bf16x2(dr[0], dr[1]);
                dw[c / 2 + 1] = pack_bf16x2(dr[2], dr[3]);
            };
            if (kfirst + 127 > q0) {                         // crosses the diagonal: mask
#pragma unroll
                for (int c = 0; c < 32; c += 4) grad4(c, true);
            } else {
#pragma unroll
                for (int c = 0; c < 32; c += 4) grad4(c, false);
            }
            if (t > 0) {                                     // gradient MMAs of t-1 have read P^T/dS^T
                ok = __all_sync(0xffffffffu, tc::mbar_wait(&B.p_free, (t - 1) & 1, p.err));
                if (!ok) break;
            }
            tc::tmem_st16(lane_base + kv_TP + wg * 16, pw);
            tc::tmem_st16(lane_base + kv_TDS + wg * 16, dw);
            tc::tmem_wait_st();
            tc::tc_fence_before();
            tc::mbar_arrive(&B.p_full);
        }
        if (ok) ok = __all_sync(0xffffffffu, tc::mbar_wait(&B.acc_done, 0, p.err));
        // Warpgroup 0 adds dK (scaled), warpgroup 1 adds dV into the fp32 pool.
        // Each 32-column block of the page's 128 rows goes to shared memory (the
        // Q/dO stages, free once acc_done has completed) in the tensor map's
        // 128-byte swizzle (16-byte chunk v of row r at chunk v ^ (r % 8)), and
        // one thread adds the boxes by TMA reduce-add: whole-line reductions at
        // L2 instead of one 16-byte request per row and vector. Rows past the
        // sequence's end add zeros. Every softmax thread reaches the
        // warpgroup's barrier; a warp whose waits failed marks the warpgroup,
        // whose boxes are then not added (the error is already recorded).
        const float scale = wg == 0 ? rsqrtf((float)D) : 1.f;
        const uint32_t col = wg == 0 ? kv_TDK : kv_TDV;
        uint8_t* stage = smem + kv_Q + wg * (D / 32) * 16 * KB;   // D/32 boxes [128 rows][32 fp32]
        if (ok) {
            tc::tc_fence_after();
            const bool live = kpos < p.q_start + p.n_q;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t a[32];
                tc::tmem_ld32(lane_base + col + c * 32, a);
                tc::tmem_wait_ld(a);
                uint8_t* row_p = stage + c * 16 * KB + r * 128;
#pragma unroll
                for (int v = 0; v < 8; ++v) {
                    const float4 x = live ? make_float4(__uint_as_float(a[4 * v]) * scale,
                                                        __uint_as_float(a[4 * v + 1]) * scale,
                                                        __uint_as_float(a[4 * v + 2]) * scale,
                                                        __uint_as_float(a[4 * v + 3]) * scale)
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
                    *reinterpret_cast<float4*>(row_p + ((v ^ (r & 7)) << 4)) = x;
                }
            }
        } else if (lane == 0) {
            B.epi_bad[wg] = 1;
        }
        tc::fence_proxy_async_smem();
        if (wg == 0) asm volatile("bar.sync 1, 128;" ::: "memory");   // the warpgroup's rows are written
        else asm volatile("bar.sync 2, 128;" ::: "memory");
        if ((warp & 3) == 2 && lane == 0 && !B.epi_bad[wg]) {
            const CUtensorMap* tm = wg == 0 ? &tm_dk : &tm_dv;
            const int row0 = (int)(((int64_t)pp * p.Hkv + kvh) * 128);
#pragma unroll
            for (int c = 0; c < D / 32; ++c) tc::tma_reduce_add_2d(tm, stage + c * 16 * KB, 32 * c, row0);
            tc::bulk_commit();
            tc::bulk_wait_read();                          // the boxes are read before the CTA exits
        }
    }

    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, 512);
    }
}

// ============================================================================ dQ

// Whole-page key tiles (128 keys): S = Q K^T and dP = dO V^T are N = 128 MMAs
// into one buffer. The softmax warps release it as soon as they have read it
// (s_free), so S/dP of tile t+1 overlaps their work on tile t; dS (bf16) goes
// to tensor memory, read there as the A operand of dQ += dS K (ds_free: dQ of
// the previous tile has read it). Q, the A operand of every S MMA, is placed in
// tensor memory once. Tensor-core order: S/dP(t+1) ahead of dQ(t).
// K and V travel in separate rings: V is free once dP is computed, K only after dQ.
constexpr int q_KST = 4;
constexpr int q_VST = 2;
template <int D> struct QLayout {
    static constexpr uint32_t kTile = (D / 64) * 16 * KB;    // [128 rows][D]: D/64 16 KB blocks
    static constexpr uint32_t kdO = 0;
    static constexpr uint32_t kK = kTile;                     // stages x [128 keys][D]
    static constexpr uint32_t kV = kK + q_KST * kTile;
    static constexpr uint32_t kSMEM = kV + q_VST * kTile + 1024;
};
// Tensor-memory columns: S, dP (128 fp32 each), dQ (D fp32), dS (128 bf16 =
// 64), Q (D bf16 = D/2).
constexpr uint32_t q_TS = 0, q_TDP = 128, q_TDQ = 256, q_TDS = 384, q_TQ = 448;

struct __align__(8) QBar {
    uint64_t q_full;
    uint64_t k_full[q_KST], k_empty[q_KST];
    uint64_t v_full[q_VST], v_empty[q_VST];
    uint64_t q_tmem;                 // Q in TMEM (softmax threads)
    uint64_t s_full, s_free;
    uint64_t ds_full, ds_free;
    uint64_t acc_done;
    uint64_t drain[2];
    uint32_t tmem_base;
    float dpart[2][128];             // the two warpgroups' halves of each row's D
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
bwd_q_tc_kernel(const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, BwdParams p) {
    using L = QLayout<D>;
    constexpr uint32_t q_dO = L::kdO, q_K = L::kK, q_V = L::kV, kT = L::kTile;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ QBar B;

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int qt = (int)gridDim.x - 1 - (int)blockIdx.x;        // longest tiles first
    const int h = blockIdx.y;
    const int kvh = h / (p.Hq / p.Hkv);
    // Key tiles = visible pages (dense: pages 0..own; sparse: the listed pages).
    const int32_t* sel_row = p.sel ? p.sel + ((size_t)qt * p.Hkv + kvh) * p.kmax : nullptr;
    const int T = sel_row ? sel_count_warp(sel_row, p.kmax, lane) : (int)(p.q_start / 128) + qt + 1;

    if (threadIdx.x == 0) {
        tc::mbar_init(&B.q_full, 1);
        for (int s = 0; s < q_KST; ++s) {
            tc::mbar_init(&B.k_full[s], 1);
            tc::mbar_init(&B.k_empty[s], 1);
        }
        for (int s = 0; s < q_VST; ++s) {
            tc::mbar_init(&B.v_full[s], 1);
            tc::mbar_init(&B.v_empty[s], 1);
        }
        tc::mbar_init(&B.q_tmem, kSoftmaxThreads);
        tc::mbar_init(&B.s_full, 1);
        tc::mbar_init(&B.s_free, kSoftmaxThreads);
        tc::mbar_init(&B.ds_full, kSoftmaxThreads);
        tc::mbar_init(&B.ds_free, 1);
        tc::mbar_init(&B.acc_done, 1);
        tc::mbar_init(&B.drain[0], 1);
        tc::mbar_init(&B.drain[1], 1);
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

    if (warp == 0) {
        // Whole-warp producer: page indices arrive 32 at a time (PageBatch); lane 0 copies.
        if (lane == 0) {
            tc::prefetch_tmap(&tm_k);
            tc::prefetch_tmap(&tm_v);
            const int q_row0 = qt * 128;
            tc::mbar_arrive_expect_tx(&B.q_full, kT);
#pragma unroll
            for (int b = 0; b < D / 64; ++b)
                tc::tma_load_3d(smem + q_dO + b * 16 * KB, &tm_do, &B.q_full, 64 * b, h, q_row0);
        }
        tc::PageBatch pages;
        pages.init(p.bt, sel_row, T, lane);
        int k_issued = 0, v_issued = 0;
        for (int t = 0; t < T; ++t) {
            const int ks = t % q_KST, vs = t % q_VST;
            if (t >= q_KST &&
                !__all_sync(0xffffffffu, tc::mbar_wait(&B.k_empty[ks], ((t / q_KST) - 1) & 1, p.err)))
                break;
            const int32_t pp = pages.get(t);
            if (pp < 0 || pp >= p.num_phys) {
                if (lane == 0) report_error(p.err, kErrBadPage);
                break;
            }
            const int row = (int)(((int64_t)pp * p.Hkv + kvh) * 128);
            if (lane == 0) {
                uint8_t* kd = smem + q_K + ks * kT;
                tc::mbar_arrive_expect_tx(&B.k_full[ks], kT);
#pragma unroll
                for (int b = 0; b < D / 64; ++b)
                    tc::tma_load_2d(kd + b * 16 * KB, &tm_k, &B.k_full[ks], 64 * b, row);
            }
            k_issued = t + 1;
            if (t >= q_VST &&
                !__all_sync(0xffffffffu, tc::mbar_wait(&B.v_empty[vs], ((t / q_VST) - 1) & 1, p.err)))
                break;
            if (lane == 0) {
                uint8_t* vd = smem + q_V + vs * kT;
                tc::mbar_arrive_expect_tx(&B.v_full[vs], kT);
#pragma unroll
                for (int b = 0; b < D / 64; ++b)
                    tc::tma_load_2d(vd + b * 16 * KB, &tm_v, &B.v_full[vs], 64 * b, row);
            }
            v_issued = t + 1;
        }
        if (lane == 0) {
            drain_wait(&B.q_full, 0);
            for (int t = max(0, k_issued - q_KST); t < k_issued; ++t)
                drain_wait(&B.k_full[t % q_KST], (t / q_KST) & 1);
            for (int t = max(0, v_issued - q_VST); t < v_issued; ++t)
                drain_wait(&B.v_full[t % q_VST], (t / q_VST) & 1);
        }
    } else if (warp == 1 || warp == kWarpG) {
        // Warp 1: S/dP(t); warp kWarpG: dQ(t). Each whole warp runs its loop
        // (warp-uniform descriptors); the elected lane issues.
        const bool leader = tc::elect_one_sync();
        const uint32_t id_s = tc::idesc_bf16(128, 128, false, false);   // S = Q K^T
        const uint32_t id_q = tc::idesc_bf16(128, D, false, true);      // dQ += dS K
        const uint32_t t_S = tmem + q_TS, t_dP = tmem + q_TDP, t_dQ = tmem + q_TDQ, t_Q = tmem + q_TQ;
        bool ok = true;
        // Base descriptors; each MMA advances them by a compile-time offset.
        const uint64_t ddO0 = tc::sdesc(tc::smem_u32(smem + q_dO), 16, 1024);
        const uint64_t dKk0 = tc::sdesc(tc::smem_u32(smem + q_K), 16, 1024);       // K-major
        const uint64_t dVk0 = tc::sdesc(tc::smem_u32(smem + q_V), 16, 1024);
        const uint64_t dKm0 = tc::sdesc(tc::smem_u32(smem + q_K), 16 * KB, 1024);  // MN-major
        auto issue_s = [&](int t) -> bool {
            const int ks = t % q_KST, vs = t % q_VST;
            if (!tc::warp_wait(&B.k_full[ks], (t / q_KST) & 1, p.err)) return false;
            if (!tc::warp_wait(&B.v_full[vs], (t / q_VST) & 1, p.err)) return false;
            if (t > 0 && !tc::warp_wait(&B.s_free, (t - 1) & 1, p.err)) return false;
            tc::tc_fence_after();
            const uint32_t k_off = ks * kT, v_off = vs * kT;
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {   // K = d, 16 per MMA (8 columns of Q)
                    const uint32_t o = (kk >> 2) * 16 * KB + (kk & 3) * 32;
                    tc::mma_bf16_ts(t_S, t_Q + kk * 8, tc::sdesc_at(dKk0, k_off + o), id_s, kk > 0 ? 1u : 0u);
                }
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t o = (kk >> 2) * 16 * KB + (kk & 3) * 32;
                    tc::mma_bf16(t_dP, tc::sdesc_at(ddO0, o), tc::sdesc_at(dVk0, v_off + o), id_s,
                                 kk > 0 ? 1u : 0u);
                }
                tc::mma_commit(&B.s_full);
                tc::mma_commit(&B.v_empty[vs]);
            }
            __syncwarp();
            return true;
        };
        auto issue_dq = [&](int t) -> bool {
            const int ks = t % q_KST;
            if (!tc::warp_wait(&B.ds_full, t & 1, p.err)) return false;
            tc::tc_fence_after();
            const uint32_t t_dS = tmem + q_TDS, k_off = ks * kT;
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)      // K = 128 keys, 16 per MMA (8 columns)
                    tc::mma_bf16_ts(t_dQ, t_dS + kk * 8, tc::sdesc_at(dKm0, k_off + kk * 2048), id_q,
                                    (t > 0 || kk > 0) ? 1u : 0u);
                tc::mma_commit(&B.k_empty[ks]);
                tc::mma_commit(&B.ds_free);
            }
            __syncwarp();
            return true;
        };
        // K(t) is released by dQ(t), which starts only after the softmax has
        // seen S(t) complete, so S(t) has read K(t) by then too.
        const int role = warp == 1 ? 0 : 1;
        if (role == 0) {
            ok = tc::warp_wait(&B.q_full, 0, p.err) && tc::warp_wait(&B.q_tmem, 0, p.err);
            for (int t = 0; ok && t < T; ++t) ok = issue_s(t);
        } else {
            for (int t = 0; ok && t < T; ++t) ok = issue_dq(t);
            if (ok && T > 0 && leader) tc::mma_commit(&B.acc_done);
        }
        if (leader) {
            tc::mma_commit(&B.drain[role]);
            drain_wait(&B.drain[role], 0);
        }
        __syncwarp();
    } else {
        // Two warpgroups: warpgroup wg handles keys [64 wg, 64 wg + 64) of every
        // tile, and dQ columns [64 wg, 64 wg + 64) in the epilogue.
        const int wg = (warp - 2) >> 2;
        const int quad = warp & 3;
        const int r = quad * 32 + lane;                      // query row of the tile
        const int64_t q_local = (int64_t)qt * 128 + r;
        const int64_t qpos = p.q_start + q_local;
        const bool valid = q_local < p.n_q;
        const float lse2 = valid ? p.lse[(size_t)h * p.n_q + q_local] * kLog2e : INFINITY;
        const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
        const float sl2 = rsqrtf((float)D) * kLog2e;
        const int64_t first_diag = p.q_start + (int64_t)qt * 128;   // first key of the own page
        {
            // Q row, head dims [D/2 wg, D/2 wg + D/2) -> TMEM columns q_TQ + D/4 wg ..
            constexpr int NW = D / 4;
            uint32_t w[NW];
#pragma unroll
            for (int e = 0; e < NW; ++e) w[e] = 0u;          // rows past the chunk: Q = 0
            if (valid) {
                const uint4* src = reinterpret_cast<const uint4*>(
                    static_cast<const __nv_bfloat16*>(p.q) + ((size_t)q_local * p.Hq + h) * D + wg * (D / 2));
#pragma unroll
                for (int v = 0; v < NW / 4; ++v) {
                    const uint4 u = __ldg(src + v);
                    w[4 * v] = u.x; w[4 * v + 1] = u.y; w[4 * v + 2] = u.z; w[4 * v + 3] = u.w;
                }
            }
            if constexpr (D == 128) tc::tmem_st32(lane_base + q_TQ + wg * 32, w);
            else tc::tmem_st16(lane_base + q_TQ + wg * 16, w);
            tc::tmem_wait_st();
            tc::tc_fence_before();
            tc::mbar_arrive(&B.q_tmem);
        }
        // D = rowsum(dO * O) of this query row (the backward's D_i): this
        // warpgroup's half of the head dims, dO from the tile in shared memory
        // (once it has landed; 128-byte swizzle: 16-byte chunk j of row r at
        // j ^ (r % 8)) and O from global memory. The halves meet through shared
        // memory; warpgroup 0 writes D for the dK/dV kernel, which runs after
        // this one.
        bool ok = true;
        float Dr = 0.f;
        {
            constexpr int HC = D / 16;                      // 8-element chunks per half row
            uint4 ov[HC];
            if (valid) {
                const uint4* src = reinterpret_cast<const uint4*>(
                    static_cast<const __nv_bfloat16*>(p.o) + ((size_t)q_local * p.Hq + h) * D + wg * (D / 2));
#pragma unroll
                for (int c = 0; c < HC; ++c) ov[c] = __ldg(src + c);
            }
            ok = __all_sync(0xffffffffu, tc::mbar_wait(&B.q_full, 0, p.err));
            float part = 0.f;
            if (ok && valid) {
#pragma unroll
                for (int c = 0; c < HC; ++c) {
                    const int d0 = wg * (D / 2) + c * 8;
                    const int cb = (d0 % 64) / 8;
                    const uint4 dv4 = *reinterpret_cast<const uint4*>(
                        smem + q_dO + (d0 / 64) * 16 * KB + r * 128 + ((cb ^ (r & 7)) << 4));
                    float fo[8], fd[8];
                    widen16<__nv_bfloat16>(ov[c], fo);
                    widen16<__nv_bfloat16>(dv4, fd);
#pragma unroll
                    for (int e = 0; e < 8; ++e) part = fmaf(fd[e], fo[e], part);
                }
            }
            B.dpart[wg][r] = part;
            asm volatile("bar.sync %0, 64;" :: "r"(1 + quad) : "memory");   // the row's two warps
            Dr = part + B.dpart[wg ^ 1][r];
            if (wg == 0 && valid && ok) p.Dbuf[(size_t)h * p.n_q + q_local] = Dr;
        }
        for (int t = 0; ok && t < T; ++t) {
            ok = __all_sync(0xffffffffu, tc::mbar_wait(&B.s_full, t & 1, p.err));
            if (!ok) break;
            tc::tc_fence_after();
            const int64_t kbase = (int64_t)(sel_row ? sel_row[t] : t) * 128 + wg * 64;
            uint32_t s0[32], s1[32], d0[32], d1[32];
            tc::tmem_ld32(lane_base + q_TS + wg * 64, s0);
            tc::tmem_ld32(lane_base + q_TS + wg * 64 + 32, s1);
            tc::tmem_ld32(lane_base + q_TDP + wg * 64, d0);
            tc::tmem_ld32(lane_base + q_TDP + wg * 64 + 32, d1);
            tc::tmem_wait_ld(s0);
            tc::tmem_wait_ld(s1);
            tc::tmem_wait_ld(d0);
            tc::tmem_wait_ld(d1);
            tc::tc_fence_before();
            tc::mbar_arrive(&B.s_free);                      // S/dP buffer may be overwritten
            uint32_t dw[32];
            auto grad_half = [&](const uint32_t (&sv)[32], const uint32_t (&dv)[32], int c0, bool mask) {
#pragma unroll
                for (int c = 0; c < 32; c += 2) {
                    float dr[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        float pv = fast_exp2(fmaf(__uint_as_float(sv[c + e]), sl2, -lse2));
                        if (mask && kbase + c0 + c + e > qpos) pv = 0.f;
                        dr[e] = pv * (__uint_as_float(dv[c + e]) - Dr);
                    }
                    dw[(c0 + c) / 2] = pack_bf16x2(dr[0], dr[1]);
                }
            };
            if (kbase + 63 > first_diag) {                   // crosses the diagonal: mask
                grad_half(s0, d0, 0, true);
                grad_half(s1, d1, 32, true);
            } else {
                grad_half(s0, d0, 0, false);
                grad_half(s1, d1, 32, false);
            }
            if (t > 0) {                                     // dQ(t - 1) has read dS(t - 1)
                ok = __all_sync(0xffffffffu, tc::mbar_wait(&B.ds_free, (t - 1) & 1, p.err));
                if (!ok) break;
            }
            tc::tmem_st32(lane_base + q_TDS + wg * 32, dw);
            tc::tmem_wait_st();
            tc::tc_fence_before();
            tc::mbar_arrive(&B.ds_full);
        }
        if (ok && T > 0) ok = __all_sync(0xffffffffu, tc::mbar_wait(&B.acc_done, 0, p.err));
        if (ok && T > 0) {
            tc::tc_fence_after();
            const float scale = rsqrtf((float)D);
            __nv_bfloat16* row = static_cast<__nv_bfloat16*>(p.dq) + ((size_t)q_local * p.Hq + h) * D;
#pragma unroll
            for (int c = (D / 64) * wg; c < (D / 64) * (wg + 1); ++c) {
                uint32_t a[32];
                tc::tmem_ld32(lane_base + q_TDQ + c * 32, a);
                tc::tmem_wait_ld(a);
                if (valid) {
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(a[8 * v + 0]) * scale, __uint_as_float(a[8 * v + 1]) * scale);
                        w.y = pack_bf16x2(__uint_as_float(a[8 * v + 2]) * scale, __uint_as_float(a[8 * v + 3]) * scale);
                        w.z = pack_bf16x2(__uint_as_float(a[8 * v + 4]) * scale, __uint_as_float(a[8 * v + 5]) * scale);
                        w.w = pack_bf16x2(__uint_as_float(a[8 * v + 6]) * scale, __uint_as_float(a[8 * v + 7]) * scale);
                        *reinterpret_cast<uint4*>(row + c * 32 + v * 8) = w;
                    }
                }
            }
        }
    }

    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, 512);
    }
}

// The ascending union of the pages listed in a selection [n_ent entries],
// out = [count, pages...]. One CTA: flags in shared memory, then an ordered
// compaction (thread t owns a contiguous run of pages). With masks, also the
// query pages listing each (page, KV head), as W 64-bit words per pair.
constexpr int kUnionThreads = 1024;
__global__ void __launch_bounds__(kUnionThreads) sel_union_kernel(const int32_t* sel, int64_t n_ent,
                                                                  int n_pages, int32_t* out, int Hkv,
                                                                  int kmax, uint64_t* masks, int W,
                                                                  int masks_in_smem) {
    extern __shared__ __align__(16) uint8_t flag[];
    __shared__ int wsum[kUnionThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < n_pages; i += kUnionThreads) flag[i] = 0;
    // The masks are built with shared-memory atomics when they fit after the
    // flags (copied out at the end), else with global ones.
    const int64_t n_words = (int64_t)n_pages * Hkv * W;
    uint64_t* mk = masks && masks_in_smem ? reinterpret_cast<uint64_t*>(flag + ((n_pages + 15) & ~15)) : masks;
    if (mk)
        for (int64_t i = tid; i < n_words; i += kUnionThreads) mk[i] = 0ull;
    __syncthreads();
    // Eight entries are loaded before any is used, so their latencies overlap
    // (the atomics would otherwise order each load after the previous one).
    constexpr int kBatch = 8;
    for (int64_t e0 = tid; e0 < n_ent; e0 += (int64_t)kBatch * kUnionThreads) {
        int32_t pgs[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int64_t e = e0 + (int64_t)u * kUnionThreads;
            pgs[u] = e < n_ent ? __ldg(sel + e) : -1;
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int32_t pg = pgs[u];
            if (pg < 0 || pg >= n_pages) continue;
            flag[pg] = 1;
            if (mk) {
                // entry e = (query page, KV head, k): bit qp of the page's word qp / 64
                const int row = (int)((e0 + (int64_t)u * kUnionThreads) / kmax);
                const int qp = row / Hkv, kvh = row - qp * Hkv;
                atomicOr(reinterpret_cast<unsigned long long*>(mk + ((int64_t)pg * Hkv + kvh) * W + qp / 64),
                         1ull << (qp % 64));
            }
        }
    }
    __syncthreads();
    const int per = (n_pages + kUnionThreads - 1) / kUnionThreads;
    const int p0 = min(n_pages, tid * per), p1 = min(n_pages, p0 + per);
    int cnt = 0;
    for (int i = p0; i < p1; ++i) cnt += flag[i];
    int x = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int t = wsum[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        wsum[lane] = t;
    }
    __syncthreads();
    int pos = (warp > 0 ? wsum[warp - 1] : 0) + x - cnt;
    for (int i = p0; i < p1; ++i)
        if (flag[i]) out[1 + pos++] = i;
    if (tid == 0) out[0] = wsum[kUnionThreads / 32 - 1];
    if (masks && masks_in_smem)
        for (int64_t i = tid; i < n_words; i += kUnionThreads) masks[i] = mk[i];
}

template <int D>
static cudaError_t launch_bwd(const AttnArgs& a, cudaStream_t s) {
    CUtensorMap tq64, tdo64, tdo128;
    std::string why;
    const uint64_t s1 = (uint64_t)D * 2, s2 = (uint64_t)a.Hq * D * 2;
    if (!make_tmap_3d(&tq64, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, a.Hq, a.n_q, s1, s2, 64, 1, 64, &why) ||
        !make_tmap_3d(&tdo64, a.dout, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, a.Hq, a.n_q, s1, s2, 64, 1, 64, &why) ||
        !make_tmap_3d(&tdo128, a.dout, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, a.Hq, a.n_q, s1, s2, 64, 1, 128, &why))
        return cudaErrorInvalidValue;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(bwd_kv_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)KVLayout<D>::kSMEM);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(bwd_q_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)QLayout<D>::kSMEM);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    BwdParams p{};
    p.Hq = a.Hq; p.Hkv = a.Hkv; p.q_start = a.q_start; p.n_q = a.n_q; p.q = a.q; p.kpool = a.kpool;
    p.lse = a.lse_in; p.Dbuf = a.Dbuf; p.dq = a.dq; p.dkpool = a.dkpool; p.dvpool = a.dvpool;
    p.o = a.o_in;
    p.bt = a.bt; p.num_phys = a.num_phys; p.err = a.err;
    p.sel = a.sel; p.kmax = a.kmax;
    // The dQ kernel first: it computes D = rowsum(dO * O), which the dK/dV kernel reads.
    {
        dim3 g_q((unsigned)((a.n_q + 127) / 128), a.Hq);
        ProfScope ps("bwd_q_tc_kernel", s);
        bwd_q_tc_kernel<D><<<g_q, kThreads, QLayout<D>::kSMEM, s>>>(tdo128, *a.tmap_k, *a.tmap_v, p);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const int64_t n_keys = a.q_start + a.n_q;
    const int64_t n_key_pages = (n_keys + 127) / 128;
    // Key pages the dK/dV grid covers: every page (dense), or at most the
    // selection union's upper bound (its CTAs beyond the union's size exit).
    int64_t grid_pages = n_key_pages;
    // (The union's grid dimension is limited to 65535 pages; beyond that every
    // key page gets a CTA, as for dense calls.)
    const bool use_list = a.sel && bwd_pagelist_cap(a) <= 65535;
    if (use_list) {
        grid_pages = bwd_pagelist_cap(a);
        // Dynamic shared memory: the page flags, then (16-byte aligned) the
        // query-page masks when they fit.
        const int n_qp = (int)((a.n_q + 127) / 128);
        const int W = (n_qp + 63) / 64;
        const size_t mask_bytes = (size_t)n_key_pages * a.Hkv * W * sizeof(uint64_t);
        const size_t flags_bytes = ((size_t)n_key_pages + 15) & ~size_t(15);
        const int masks_in_smem = a.selmask && flags_bytes + mask_bytes <= 200 * 1024;
        const size_t fl = masks_in_smem ? flags_bytes + mask_bytes : (size_t)n_key_pages;
        static size_t attr_u = 0;
        if (fl > 48 * 1024 && fl > attr_u) {
            cudaError_t e = cudaFuncSetAttribute(sel_union_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)fl);
            if (e != cudaSuccess) return e;
            attr_u = fl;
        }
        ProfScope ps("sel_union_kernel", s);
        sel_union_kernel<<<1, kUnionThreads, fl, s>>>(a.sel, (int64_t)n_qp * a.Hkv * a.kmax,
                                                      (int)n_key_pages, a.pagelist, a.Hkv, a.kmax,
                                                      a.selmask, W, masks_in_smem);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        p.pagelist = a.pagelist;
        p.selmask = a.selmask;
    }
    // Small grids (early chunks) leave SMs idle behind a few long CTAs: split
    // each (page, KV head)'s iterations over up to 4 CTAs so that there are
    // >= ~8 waves. Every split adds the page's dK/dV rows into the pool once
    // more; measured on the dense 32K sweep, 8 waves was as fast as 16 (which
    // split the last chunk's pages 3 ways instead of 2) and faster than 4.
    int dev = 0, sm_count = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev);
    sm_count = std::max(sm_count, 1);
    // With a selection a page is seen by few query tiles (28 iterations per
    // page for a local layer with two pages per list): splitting would only
    // multiply the CTAs' start-up and gradient additions, so only dense calls split.
    const int64_t n_cta = grid_pages * a.Hkv;
    const int splits = a.sel ? 1
        : (int)std::min<int64_t>(4, std::max<int64_t>(1, (8 * (int64_t)sm_count + n_cta - 1) / n_cta));
    p.kv_splits = splits;
    const dim3 g_kv = use_list ? dim3(a.Hkv, (unsigned)grid_pages)
                               : dim3((unsigned)(grid_pages * splits), a.Hkv);
    {
        ProfScope ps("bwd_kv_tc_kernel", s);
        bwd_kv_tc_kernel<D><<<g_kv, kThreads, KVLayout<D>::kSMEM, s>>>(tq64, tdo64, *a.tmap_v, *a.tmap_dk,
                                                                       *a.tmap_dv, p);
    }
    return cudaGetLastError();
}

}  // namespace

int64_t bwd_pagelist_cap(const AttnArgs& a) {
    if (!a.sel) return 0;
    const int64_t n_key_pages = (a.q_start + a.n_q + a.P - 1) / a.P;
    const int64_t n_qp = (a.n_q + a.P - 1) / a.P;
    return std::min<int64_t>(n_key_pages, n_qp * a.Hkv * (int64_t)a.kmax);
}

int64_t bwd_selmask_words(const AttnArgs& a) {
    if (!a.sel) return 0;
    const int64_t n_key_pages = (a.q_start + a.n_q + a.P - 1) / a.P;
    const int64_t n_qp = (a.n_q + a.P - 1) / a.P;
    return n_key_pages * a.Hkv * ((n_qp + 63) / 64);
}

cudaError_t launch_attn_bwd_tc(const AttnArgs& a, cudaStream_t s) {
    // The sparse dK/dV kernel lists the selecting query pages in shared memory.
    if (a.sel && (a.n_q + 127) / 128 > kMaxSelQp) {
        const cudaError_t e = launch_bwd_rowdot(a, s);
        return e != cudaSuccess ? e : launch_attn_bwd_simt(a, s);
    }
    if ((reinterpret_cast<uintptr_t>(a.dout) & 15) || !a.tmap_k || (a.sel && !a.pagelist))
        return cudaErrorInvalidValue;
    return a.d == 64 ? launch_bwd<64>(a, s) : launch_bwd<128>(a, s);
}

}  // namespace pkv
