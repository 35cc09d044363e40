// Tensor-core (tcgen05) paged chunk attention forward, bf16 in / fp32 accumulate.
//
// Computes, for one query chunk, exact causal softmax attention over every
// key reached through the block table (dense) or over the pages selected for
// each query page (sparse), and saves the row log-sum-exp for the backward
// ("Out of the Memory Barrier": kernels that run forward and backward directly
// on the paged KV cache, gist.science/de §2.B, sciencestack.ai Fig. 3; page
// selection, gist.science/de §2.D).
//
// One CTA per (query tile of 128 rows = one query page, query head) -- or,
// for short page lists (local layers), per (query tile, KV group), looping
// over the group's query heads with its tensor memory, barriers and page
// list kept; key tiles are whole pages (P = 128), fetched by TMA with the
// physical page taken from the block table. Head dimension D = 128 or 64 (a template
// parameter; a page of one head is D / 64 blocks of 64 columns). Both MMAs take their A operand from tensor
// memory (an A operand in shared memory costs the tensor core a fixed ~33
// cycles per instruction on top of the math): Q is placed there once, and
// P overwrites the S columns it came from. Warp roles (352 threads):
//   warp 0       TMA producer: K pages into a 3-stage ring.
//   warp 10      TMA producer: V pages into a 2-stage ring. Each V stage
//                carries a constant extra 64-column block whose first column
//                is 1, so the PV MMA (N = D + 16) also accumulates the row sum
//                l = sum_j P_ij of exactly the bf16 weights it multiplies.
//   warp 1       MMA issuer (elected lane): S_j = Q K_j^T into a double-
//                buffered TMEM tile, then O += P_{j-1} V_{j-1} (O in TMEM).
//   warps 2..9   softmax, two warpgroups: thread (wg, row) owns keys
//                [64 wg, 64 wg + 64) of query row `row` in every tile. The two
//                partial row maxima meet through shared memory under a named
//                barrier shared by just the two warps that own those rows
//                (every iteration passes it exactly once, error or not, so it
//                cannot be left waiting). O (with l) is rescaled in TMEM only when m
//                grows by more than 2^8 (P <= 256 then, exactly representable
//                range for bf16), each warpgroup its own half of the columns.
//                Epilogue: O / l, LSE.
// TMEM columns: S0 [0,128), S1 [128,256), O [256, 256+D), l 256+D,
// Q [400, 400+D/2).
#include <cuda_bf16.h>
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace pkv {
namespace {

constexpr int kTile = 128;                   // query rows = keys per tile
constexpr int kThreads = 352;
constexpr int kSoftmaxThreads = 256;
constexpr uint32_t kHalfBytes = 128 * 128;   // [128 rows][64 bf16] = 16 KB
constexpr int kKStages = 3, kVStages = 2;
constexpr float kRescaleThreshold = 8.0f;                         // log2 units
constexpr int kShortList = 8;            // page lists up to this long: a CTA per (tile, KV group)

// Shared-memory tile offsets (bytes from a 1024-aligned base) and tensor-
// memory columns for head dimension D.
// K and V have separate rings: a K stage is free as soon as S_j completes, so
// K loads run kKStages - 1 tiles ahead; a V stage is free after PV_j.
template <int D> struct FwdLayout {
    static_assert(D == 64 || D == 128, "head dim 64 or 128");
    static constexpr int kBlocks = D / 64;                                 // 64-column blocks
    static constexpr uint32_t kTileBytes = kBlocks * kHalfBytes;
    static constexpr uint32_t kVStageBytes = kTileBytes + kHalfBytes;      // V + the ones block
    static constexpr uint32_t kOffK = 0;
    static constexpr uint32_t kOffV = kOffK + kKStages * kTileBytes;
    static constexpr uint32_t kTilesBytes = kOffV + kVStages * kVStageBytes;
    static constexpr uint32_t kSmemBytes = kTilesBytes + 1024;             // + alignment slack
    static constexpr uint32_t kColO = 256, kColL = kColO + D, kColQ = 400;
};

struct FwdParams {
    int Hq, Hkv;
    int heads_per_cta;               // consecutive query heads of one KV group per CTA
    int64_t q_start, n_q;
    const void* q;
    void* o;
    float* lse;
    const int32_t* bt;
    int64_t num_phys;
    const int32_t* sel;
    int kmax;
    int* err;
};

struct __align__(8) FwdBarriers {
    uint64_t q_full;                 // Q in TMEM (256 softmax arrivals)
    uint64_t q_empty;                // a head's S MMAs done: its Q may be replaced
    uint64_t o_free;                 // a head's O read by the epilogue (256 arrivals)
    uint64_t k_full[kKStages], k_empty[kKStages], v_full[kVStages], v_empty[kVStages];
    uint64_t s_full[2];
    uint64_t p_full;
    uint64_t o_done;
    uint64_t drain;
    uint32_t tmem_base;
    int n_tiles;
    float red[2][2][kTile];          // [parity][warpgroup][row]
};


// Tensor-memory column (within an S buffer) of P for keys [16 kk, 16 kk + 16):
// warpgroup wg packs its 64 keys into the first 32 of the 64 columns it read.
__device__ __forceinline__ uint32_t p_col(int kk) { return (kk >> 2) * 64 + (kk & 3) * 8; }

using tc::drain_wait;

// One producer warp: streams the K ring or the V ring. The whole warp walks
// the tiles (page indices come 32 at a time from a PageBatch); lane 0 issues
// the copies. A K load never waits behind a V stage in use.
template <int D>
__device__ __forceinline__ void produce_ring(const FwdParams& p, uint8_t* smem, FwdBarriers& B,
                                             const CUtensorMap& tmap, bool is_k, int qt, int kvh,
                                             int nt, int lane, tc::PageBatch& pages) {
    using L = FwdLayout<D>;
    const int nst = is_k ? kKStages : kVStages;
    uint64_t* full = is_k ? B.k_full : B.v_full;
    uint64_t* empty = is_k ? B.k_empty : B.v_empty;
    uint8_t* base = smem + (is_k ? L::kOffK : L::kOffV);
    if (lane == 0) tc::prefetch_tmap(&tmap);
    // The same pages for every head of the CTA: iteration it = head * nt + tile.
    // `pages` arrives initialised for the first head.
    int issued = 0;
    bool ok = true;
    for (int hi = 0; ok && hi < p.heads_per_cta; ++hi) {
        if (hi > 0) pages.init(p.bt, p.sel ? p.sel + ((size_t)qt * p.Hkv + kvh) * p.kmax : nullptr, nt, lane);
        for (int j = 0; j < nt; ++j) {
            const int it = hi * nt + j;
            const int st = it % nst;
            if (it >= nst &&
                !__all_sync(0xffffffffu, tc::mbar_wait(&empty[st], ((it / nst) - 1) & 1, p.err))) {
                ok = false;
                break;
            }
            const int32_t pp = pages.get(j);
            if (pp < 0 || pp >= p.num_phys) {
                if (lane == 0) report_error(p.err, kErrBadPage);
                ok = false;
                break;
            }
            if (lane == 0) {
                const int row = (int)(((int64_t)pp * p.Hkv + kvh) * kTile);
                uint8_t* dst = base + st * (is_k ? L::kTileBytes : L::kVStageBytes);
                tc::mbar_arrive_expect_tx(&full[st], L::kTileBytes);
#pragma unroll
                for (int b = 0; b < L::kBlocks; ++b)
                    tc::tma_load_2d(dst + b * kHalfBytes, &tmap, &full[st], 64 * b, row);
            }
            issued = it + 1;
        }
    }
    // Make sure none of this CTA's copies is still landing when it exits.
    if (lane == 0)
        for (int j = max(0, issued - nst); j < issued; ++j) drain_wait(&full[j % nst], (j / nst) & 1);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
fwd_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
              FwdParams p) {
    using L = FwdLayout<D>;
    constexpr uint32_t kTileBytes = L::kTileBytes, kVStageBytes = L::kVStageBytes;
    constexpr uint32_t kOffK = L::kOffK, kOffV = L::kOffV;
    constexpr uint32_t kColO = L::kColO, kColL = L::kColL, kColQ = L::kColQ;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ FwdBarriers B;

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int qt = (int)gridDim.x - 1 - (int)blockIdx.x;        // longest tiles first
    const int h0 = (int)blockIdx.y * p.heads_per_cta;           // this CTA's first query head
    const int kvh = h0 / (p.Hq / p.Hkv);
    const int nh = p.heads_per_cta;

    // The ones block of each V stage: row r holds 1 in column 0, zeros elsewhere
    // (128-byte swizzle: column 0 sits in 16-byte chunk r & 7 of the row).
    for (int i = threadIdx.x; i < kVStages * 128 * 8; i += kThreads) {
        const int st = i / 1024, r = (i / 8) % 128, ch = i % 8;
        uint8_t* blk = smem + kOffV + st * kVStageBytes + kTileBytes;
        *reinterpret_cast<uint4*>(blk + tc::sw128_offset(r, ch)) =
            make_uint4(ch == 0 ? 0x3f80u : 0u, 0u, 0u, 0u);
    }
    tc::fence_proxy_async_smem();
    // Before the set-up barrier: the producers' tile counts and page indices,
    // and the softmax threads' Q rows of the first head (their latency overlaps
    // barrier initialisation and the tensor-memory allocation).
    const int32_t* sel_row = p.sel ? p.sel + ((size_t)qt * p.Hkv + kvh) * p.kmax : nullptr;
    tc::PageBatch pages;
    int n_pre = 0;
    if (warp == 0 || warp == kThreads / 32 - 1) {
        n_pre = sel_row ? sel_count_warp(sel_row, p.kmax, lane) : (int)(p.q_start / kTile) + qt + 1;
        pages.init(p.bt, sel_row, n_pre, lane);
    }
    constexpr int NWQ = D / 4;                            // 32-bit words of Q per thread
    uint32_t qw[NWQ];
    const bool softmax_warp = warp >= 2 && warp < kThreads / 32 - 1;
    // Q row of head h, head dims [D/2 wg, D/2 wg + D/2) (rows past the chunk: 0).
    auto load_q = [&](int h) {
        const int64_t q_local = (int64_t)qt * kTile + (warp & 3) * 32 + lane;
#pragma unroll
        for (int e = 0; e < NWQ; ++e) qw[e] = 0u;
        if (q_local < p.n_q) {
            const uint4* src = reinterpret_cast<const uint4*>(
                static_cast<const __nv_bfloat16*>(p.q) + ((size_t)q_local * p.Hq + h) * D +
                ((warp - 2) >> 2) * (D / 2));
#pragma unroll
            for (int v = 0; v < NWQ / 4; ++v) {
                const uint4 u = __ldg(src + v);
                qw[4 * v] = u.x; qw[4 * v + 1] = u.y; qw[4 * v + 2] = u.z; qw[4 * v + 3] = u.w;
            }
        }
    };
    if (softmax_warp) load_q(h0);
    if (threadIdx.x == 0) {
        tc::mbar_init(&B.q_full, kSoftmaxThreads);
        tc::mbar_init(&B.q_empty, 1);
        tc::mbar_init(&B.o_free, kSoftmaxThreads);
        for (int s = 0; s < kKStages; ++s) {
            tc::mbar_init(&B.k_full[s], 1);
            tc::mbar_init(&B.k_empty[s], 1);
        }
        for (int s = 0; s < kVStages; ++s) {
            tc::mbar_init(&B.v_full[s], 1);
            tc::mbar_init(&B.v_empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) tc::mbar_init(&B.s_full[s], 1);
        tc::mbar_init(&B.p_full, kSoftmaxThreads);
        tc::mbar_init(&B.o_done, 1);
        tc::mbar_init(&B.drain, 1);
        tc::fence_barrier_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(&B.tmem_base, 512);
        tc::tmem_relinquish();
    } else if (warp == 0) {
        // Key tiles of this CTA: dense, pages 0..own; sparse, the listed pages.
        if (lane == 0) B.n_tiles = n_pre;
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = B.tmem_base;
    const int nt = B.n_tiles;

    if (warp == 0) {
        // ------------------------------------------------------------ K producer
        produce_ring<D>(p, smem, B, tmap_k, true, qt, kvh, nt, lane, pages);
    } else if (warp == kThreads / 32 - 1) {
        // ------------------------------------------------------------ V producer
        produce_ring<D>(p, smem, B, tmap_v, false, qt, kvh, nt, lane, pages);
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs the loop (warp-uniform descriptors); one elected
        // lane issues the tcgen05 instructions and commits.
        const bool leader = tc::elect_one_sync();
        const uint32_t idesc = tc::idesc_bf16(128, 128, false, false);       // S = Q K^T
        const uint32_t idesc_pv = tc::idesc_bf16(128, D + 16, false, true);  // [O l] += P [V 1]
        const uint32_t tmem_o = tmem + kColO, tmem_q = tmem + kColQ;
        const uint64_t dk0 = tc::sdesc(tc::smem_u32(smem + kOffK), 16, 1024);            // K-major
        const uint64_t dv0 = tc::sdesc(tc::smem_u32(smem + kOffV), kHalfBytes, 1024);    // MN-major
        bool ok = true;
        // P_i sits over S_i in TMEM; S_{i+2} reuses those columns but is issued
        // after PV_i, and the tensor core runs MMAs in issue order. Iteration
        // i = head * nt + tile; a head's first PV overwrites O (accumulate off)
        // once the epilogue has read the previous head's O (o_free).
        auto issue_pv = [&](int i) -> bool {
            const int vs = i % kVStages;
            const int hi = i / nt;
            const bool first = (i % nt) == 0;
            if (!tc::warp_wait(&B.p_full, i & 1, p.err)) return false;
            if (!tc::warp_wait(&B.v_full[vs], (i / kVStages) & 1, p.err)) return false;
            if (first && hi > 0 && !tc::warp_wait(&B.o_free, (hi - 1) & 1, p.err)) return false;
            tc::tc_fence_after();
            // B = [V 1] [128 keys][D + 16] MN-major: 16 keys = 2 K-groups of 8
            // rows (1024 B apart); columns span 64-column blocks 16 KB apart
            // (V's D / 64 blocks, then the ones block).
            const uint32_t tmem_p = tmem + (i & 1) * 128;
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    tc::mma_bf16_ts(tmem_o, tmem_p + p_col(kk), tc::sdesc_at(dv0, vs * kVStageBytes + kk * 2048),
                                    idesc_pv, (!first || kk > 0) ? 1u : 0u);
                tc::mma_commit(&B.o_done);
                tc::mma_commit(&B.v_empty[vs]);
            }
            __syncwarp();
            return true;
        };
        for (int hi = 0; ok && hi < nh; ++hi) {
            if (!tc::warp_wait(&B.q_full, hi & 1, p.err)) { ok = false; break; }
            for (int j = 0; ok && j < nt; ++j) {
                const int it = hi * nt + j;
                const int ks = it % kKStages;
                if (!tc::warp_wait(&B.k_full[ks], (it / kKStages) & 1, p.err)) { ok = false; break; }
                tc::tc_fence_after();
                const uint32_t tmem_s = tmem + (it & 1) * 128;
                if (leader) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {   // K = d: 16 per MMA, 8 TMEM columns of Q
                        const uint32_t koff = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
                        tc::mma_bf16_ts(tmem_s, tmem_q + kk * 8, tc::sdesc_at(dk0, ks * kTileBytes + koff),
                                        idesc, kk > 0 ? 1u : 0u);
                    }
                    tc::mma_commit(&B.s_full[it & 1]);
                    tc::mma_commit(&B.k_empty[ks]);
                }
                __syncwarp();
                if (j > 0 && !issue_pv(it - 1)) { ok = false; break; }
            }
            // Every S MMA of this head is issued: Q may be replaced once they finish.
            if (leader) tc::mma_commit(&B.q_empty);
            __syncwarp();
            if (ok && nt > 0 && !issue_pv(hi * nt + nt - 1)) ok = false;
        }
        // Drain: nothing of ours may still run on the tensor core at exit.
        if (leader) {
            tc::mma_commit(&B.drain);
            drain_wait(&B.drain, 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax (256 threads)
        const int wg = (warp - 2) >> 2;
        const int quad = warp & 3;                    // TMEM lane quadrant of this warp
        const int row = quad * 32 + lane;             // query row within the tile
        const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
        const float sl2 = rsqrtf((float)D) * kLog2e;
        const int64_t q_local = (int64_t)qt * kTile + row;
        const bool valid = q_local < p.n_q;
        bool ok = true;
        // Named barrier of the two warps (one per warpgroup) that own rows 32 quad ..
        const uint32_t pair_bar = 1 + quad;
        for (int hi = 0; hi < nh; ++hi) {
        const int h = h0 + hi;
        // The previous head's S MMAs must be done before its Q is replaced.
        if (hi > 0 && ok) ok = __all_sync(0xffffffffu, tc::mbar_wait(&B.q_empty, (hi - 1) & 1, p.err));
        if (ok) {
            // Q row of head h (loaded ahead) -> TMEM columns kColQ + D/4 wg ..
            if constexpr (D == 128) tc::tmem_st32(lane_base + kColQ + wg * 32, qw);
            else tc::tmem_st16(lane_base + kColQ + wg * 16, qw);
            tc::tmem_wait_st();
            tc::tc_fence_before();
        }
        tc::mbar_arrive(&B.q_full);
        float m = -INFINITY;
        for (int j = 0; j < nt; ++j) {
            const int it = hi * nt + j;
            const int st = it & 1;
            if (ok) ok = __all_sync(0xffffffffu, tc::mbar_wait(&B.s_full[st], (it >> 1) & 1, p.err));
            // Raw logits q.k of my 64 keys; the scale is folded into the exp2 argument.
            // (After a failed wait the loads just read stale columns: the loop goes
            // on only to keep meeting the partner warp, and writes nothing.)
            tc::tc_fence_after();
            float x[64];
            {
                uint32_t r0[32], r1[32];
                tc::tmem_ld32(lane_base + st * 128 + wg * 64, r0);
                tc::tmem_ld32(lane_base + st * 128 + wg * 64 + 32, r1);
                tc::tmem_wait_ld(r0);
                tc::tmem_wait_ld(r1);
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    x[e] = __uint_as_float(r0[e]);
                    x[32 + e] = __uint_as_float(r1[e]);
                }
            }
            if (j == nt - 1) {                        // own page: causal mask (key col > row)
#pragma unroll
                for (int c = 0; c < 64; ++c)
                    if (wg * 64 + c > row) x[c] = -INFINITY;
            }
            // Row max with 8 independent chains.
            float mpart[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) mpart[k] = x[k];
#pragma unroll
            for (int c = 8; c < 64; ++c) mpart[c & 7] = fmaxf(mpart[c & 7], x[c]);
#pragma unroll
            for (int k = 4; k > 0; k >>= 1)
#pragma unroll
                for (int i = 0; i < k; ++i) mpart[i] = fmaxf(mpart[i], mpart[i + k]);
            const float part = mpart[0];
            // The other warpgroup's half of the row (double-buffered by tile parity:
            // a slot is rewritten only after both warps have passed the next barrier).
            B.red[st][wg][row] = part;
            asm volatile("bar.sync %0, 64;" :: "r"(pair_bar) : "memory");
            if (!ok) continue;                        // keep meeting the partner warp
            const float mx = fmaxf(part, B.red[st][wg ^ 1][row]) * sl2;   // scaled, log2 units
            float alpha = 1.f;
            bool rescale = false;
            if (mx > m + kRescaleThreshold) {
                alpha = (m == -INFINITY) ? 0.f : fast_exp2(m - mx);
                m = mx;
                rescale = true;
            }
            uint32_t pk[32];
            const float neg_m = -m;
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const float p0 = fast_exp2(fmaf(x[2 * c], sl2, neg_m));
                const float p1 = fast_exp2(fmaf(x[2 * c + 1], sl2, neg_m));
                pk[c] = pack_bf16x2(p0, p1);
            }
            if (j > 0 && __any_sync(0xffffffffu, rescale)) {
                // PV_{j-1} must be done before O is touched (PV_j waits for this tile's P).
                ok = __all_sync(0xffffffffu, tc::mbar_wait(&B.o_done, (it - 1) & 1, p.err));
                if (!ok) continue;
                tc::tc_fence_after();
                const float f = rescale ? alpha : 1.f;
#pragma unroll
                for (int c = 0; c < D / 64; ++c) {        // this warpgroup's D / 2 columns of O
                    uint32_t r[32];
                    tc::tmem_ld32(lane_base + kColO + wg * (D / 2) + c * 32, r);
                    tc::tmem_wait_ld(r);
#pragma unroll
                    for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * f);
                    tc::tmem_st32(lane_base + kColO + wg * (D / 2) + c * 32, r);
                }
                if (wg == 1)                          // and the row sum l
                    tc::tmem_st1(lane_base + kColL,
                                 __float_as_uint(__uint_as_float(tc::tmem_ld1(lane_base + kColL)) * f));
            }
            // P over the first 32 of the 64 S columns this thread read.
            tc::tmem_st32(lane_base + st * 128 + wg * 64, pk);
            tc::tmem_wait_st();
            tc::tc_fence_before();
            tc::mbar_arrive(&B.p_full);
        }
        // The next head's Q rows load while this head's last PV and epilogue run.
        // (Loads issued before the tile loop, and left in flight during it, gave
        // nondeterministic O in a few tiles of multi-head CTAs, for a reason not
        // found; issued here, repeated calls are bit-identical.)
        if (hi + 1 < nh) load_q(h + 1);
        if (ok && nt > 0) ok = __all_sync(0xffffffffu, tc::mbar_wait(&B.o_done, (hi * nt + nt - 1) & 1, p.err));
        if (ok && nt > 0) {
            tc::tc_fence_after();
            // Normalise by the sum of the bf16 weights the tensor core multiplied, so
            // O is a convex combination of values whatever the rounding of P.
            const float l = __uint_as_float(tc::tmem_ld1(lane_base + kColL));
            const float inv = 1.f / l;
            __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.o) + ((size_t)q_local * p.Hq + h) * D;
#pragma unroll
            for (int c = (D / 64) * wg; c < (D / 64) * (wg + 1); ++c) {
                uint32_t r[32];
                tc::tmem_ld32(lane_base + kColO + c * 32, r);
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
            if (valid && wg == 0) p.lse[(size_t)h * p.n_q + q_local] = (m + log2f(l)) * kLn2;
        }
        // O and l of this head are read: the next head's first PV may overwrite them.
        tc::tc_fence_before();
        tc::mbar_arrive(&B.o_free);
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
    return a.dtype == PKV_BF16 && (a.d == 128 || a.d == 64) && a.P == 128 && a.tmap_k &&
           a.tmap_v && (reinterpret_cast<uintptr_t>(a.q) & 15) == 0;
}

template <int D>
static cudaError_t launch_fwd(const AttnArgs& a, cudaStream_t s) {
    constexpr uint32_t smem = FwdLayout<D>::kSmemBytes;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(fwd_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    FwdParams p{};
    p.Hq = a.Hq; p.Hkv = a.Hkv; p.q_start = a.q_start; p.n_q = a.n_q;
    p.q = a.q; p.o = a.o; p.lse = a.lse; p.bt = a.bt; p.num_phys = a.num_phys;
    p.sel = a.sel; p.kmax = a.kmax; p.err = a.err;
    // Short page lists (local layers): one CTA takes every query head of a KV
    // group, so its start-up (tensor memory, barriers, pipeline fill) is paid
    // once for the group's g heads instead of once per head.
    p.heads_per_cta = (a.sel && a.kmax <= kShortList) ? a.Hq / a.Hkv : 1;
    dim3 grid((unsigned)((a.n_q + kTile - 1) / kTile), a.Hq / p.heads_per_cta);
    ProfScope ps("fwd_tc_kernel", s);
    fwd_tc_kernel<D><<<grid, kThreads, smem, s>>>(*a.tmap_k, *a.tmap_v, p);
    return cudaGetLastError();
}

cudaError_t launch_attn_fwd_tc(const AttnArgs& a, cudaStream_t s) {
    return a.d == 64 ? launch_fwd<64>(a, s) : launch_fwd<128>(a, s);
}

}  // namespace pkv
