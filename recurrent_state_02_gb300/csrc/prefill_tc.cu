// prefill_tc.cu -- chunkwise prefill of normalised causal linear attention on
// the sm_103a tensor cores (tcgen05 MMAs, TMEM accumulators, TMA tiles).
//
// Method ("Linear attention：把历史写进状态", hs-black.github.io/posts/linear-attention):
// section "一个 chunk 的输出由两部分组成" splits the output of a chunk of C tokens into
// the read of the carried state and the in-chunk causal product,
//     num = Q~c Sprev + [(Q~c K~c^T) . M] Vc,   den = Q~c zprev + rowsum[(Q~c K~c^T) . M],
//     Snext = Sprev + K~c^T Vc,                 znext = zprev + sum of the rows of K~c,
// with Q~ = phi(Q), K~ = phi(K), phi(x) = ELU(x)+1 (section "关键改写：让求和先发生") and
// y = num / (den + eps) (section "ε 是数值保护").  With a per-token gate (section
// "加一个门：让旧记忆逐渐淡出") each term carries the product of the gates that act on
// it between its write and its read (section "门控递推为什么能做并行 scan？": the
// updates compose as affine maps).  Writing b_i for the in-chunk cumulative sum
// of log alpha up to row i:
//     Gamma_i = exp(b_i)              scales the carried state read by row i,
//     D_ij    = exp(b_i - b_j), j<=i  scales the in-chunk score of key j at row i,
//     w_j     = exp(b_last - b_j)     scales key j's write into Snext / znext,
// and a gate of exactly 0 cuts every product across it (tracked separately, so
// that alpha = 0 is exact rather than log(0)).
//
// One CTA owns one (b, h, 64-column slice of dv) and walks the chunks in order,
// carrying the FP32 state on chip: S lives in registers of the TMEM warps and
// z in shared memory.  Per chunk (C = 64, r = 128):
//   TMA      q, k (64 x 128) and the v slice (64 x 64) as BF16 tiles, 128-byte swizzle
//   phi      warps apply phi in place (FP32 math, BF16 result), compute
//            Q~ zprev and the new z in FP32, and the gate products
//   MMA      P   = Q~ K~^T           M=64  N=64  K=128  -> TMEM
//            dS  = K~^T (w . V)      M=128 N=64  K=64   -> TMEM
//            O   = Q~ Sprev          M=64  N=64  K=128  -> TMEM (Sprev as BF16 operand)
//            O  += A V               M=64  N=64  K=64   (A = masked, decayed P in BF16)
//   TMEM     warps: S <- Gamma_last S + dS (FP32), Sprev -> shared memory, P -> A
//            and its FP32 row sums, y = O / (den + eps) -> TMA store
// Every barrier wait is bounded; on expiry the kernel records a timeout in the
// device status word, drains its own copies and MMAs, frees TMEM and returns.

#include "kernels.h"
#include "sm103_ptx.cuh"

namespace la {
namespace {

constexpr int kC = 64;          // tokens per chunk
constexpr int kR = 128;         // feature width r
constexpr int kDVS = 64;        // value columns per CTA
constexpr int kStages = 3;      // TMA pipeline depth
constexpr int kThreads = 512;   // 16 warps
constexpr int kWarpTma = 0, kWarpMma = 1, kWarpTm0 = 4, kWarpPhi0 = 12;
constexpr int kTmWarps = 8, kPhiWarps = 4;

// TMEM columns (512 allocated).
constexpr uint32_t kColP = 0, kColDS = 128, kColO = 256, kColO2 = 384, kTmemCols = 512;

// Rows of an M = 64 accumulator sit in lanes 0..15 of each 32-lane quadrant:
// row i -> lane 32 * (i / 16) + i % 16.
constexpr int kM64RowsPerQuadrant = 16;

constexpr uint32_t kTileQ = kC * kR * 2;      // 16 KB: two 64-feature blocks of 64 x 128 B
constexpr uint32_t kTileV = kC * kDVS * 2;    // 8 KB
constexpr uint32_t kTileA = kC * kC * 2;      // 8 KB
constexpr uint32_t kTileSp = kR * kDVS * 2;   // 16 KB: 128 feature rows x 128 B
constexpr uint32_t kTileY = kC * kDVS * 2;    // 8 KB

struct alignas(16) Small {
    float gb[2][kC];            // cumulative log gate inside the chunk
    int gz[2][kC];              // last row <= i whose gate is 0 (-1: none)
    float gG[2][kC];            // Gamma_i
    float gw[2][kC];            // w_j
    float gC[2][4];             // Gamma of the whole chunk (element 0)
    float den_inter[2][kC];     // Q~_i . zprev
    float densum[2][2][kC];     // in-chunk row sums, two column halves
    float z[kR];                // carried z
    float zred[8][kR];          // z partial sums (8 row groups)
    float carry[4];
    uint64_t full[kStages], empty[kStages], phi_done[kStages];
    uint64_t P_full[2], P_empty[2], dS_full[2], dS_empty[2], Sp_full[2], Sp_empty[2];
    uint64_t A_full[2], A_empty[2], O_full[2], O_empty[2], aux_empty[2];
    uint64_t mma_done, tm_sync, phi_sync;
    uint32_t tmem_base;
    int abort_flag;
};

template <bool GATED>
struct Layout {
    static constexpr uint32_t kStageBytes = 2 * kTileQ + kTileV + (GATED ? kTileV : 0);
    static constexpr uint32_t kOffQ = 0;
    static constexpr uint32_t kOffK = kTileQ;
    static constexpr uint32_t kOffV = 2 * kTileQ;
    static constexpr uint32_t kOffVw = 2 * kTileQ + kTileV;
    static constexpr uint32_t kOffA = kStages * kStageBytes;
    static constexpr uint32_t kOffSp = kOffA + 2 * kTileA;
    static constexpr uint32_t kOffY = kOffSp + 2 * kTileSp;
    static constexpr uint32_t kOffSmall = kOffY + 2 * kTileY;
    static constexpr uint32_t kBytes = kOffSmall + sizeof(Small) + 1024;   // + alignment slack
    static_assert(kBytes <= 232448, "shared memory budget");
};

__device__ __forceinline__ float phi_elu1(float x) { return x > 0.f ? x + 1.f : __expf(x); }

struct Ctx {
    uint8_t *base;     // 1024-aligned shared memory base
    Small *sm;
    uint64_t limit;
    int *status;
};

// Records a timeout once and raises the CTA-wide abort flag.
__device__ __noinline__ void fail(Ctx &cx)
{
    if (!*reinterpret_cast<volatile int *>(&cx.sm->abort_flag)) {
        atomicExch(cx.status, kStatusTimeout);
        *reinterpret_cast<volatile int *>(&cx.sm->abort_flag) = 1;
    }
}

__device__ __forceinline__ bool aborted(const Ctx &cx)
{
    return *reinterpret_cast<volatile int *>(&cx.sm->abort_flag) != 0;
}

// Bounded wait by one thread.  Gives up when the time limit runs out (and then
// raises the abort flag) or as soon as another thread has raised it.
__device__ __forceinline__ bool wait(Ctx &cx, uint64_t *bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (aborted(cx)) return false;
            if (global_timer_ns() - t0 > cx.limit) {
                fail(cx);
                return false;
            }
        }
    }
}

// Every lane waits; the outcome is made uniform across the warp so that the
// warp stays converged for the .sync.aligned instructions that follow.
__device__ __forceinline__ bool warp_wait(Ctx &cx, uint64_t *bar, uint32_t parity)
{
    const bool ok = wait(cx, bar, parity);
    return __all_sync(0xffffffffu, ok);
}

// One arrival per warp, after every lane's preceding writes and fences.
__device__ __forceinline__ void warp_arrive(uint64_t *bar)
{
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// Bounded barrier among the warps that share `bar` (count = number of warps).
__device__ __forceinline__ bool group_sync(Ctx &cx, uint64_t *bar, uint32_t &phase)
{
    warp_arrive(bar);
    const bool ok = warp_wait(cx, bar, phase);
    phase ^= 1u;
    return ok;
}

template <bool GATED>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                  const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_y,
                  const PrefillTcArgs args)
{
    using L = Layout<GATED>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Small *sm = reinterpret_cast<Small *>(base + L::kOffSmall);
    Ctx cx{base, sm, args.wait_limit_ns, args.status};

    const int slice = blockIdx.x;
    const int h = blockIdx.y, b = blockIdx.z;
    const int bh = b * args.H + h;
    const int T = args.T;
    const int nch = (T + kC - 1) / kC;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    auto stage_ptr = [&](int s) { return base + s * L::kStageBytes; };

    // ------------------------------------------------------------ set-up
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm->full[s], 1);
            mbar_init(&sm->empty[s], 1);
            mbar_init(&sm->phi_done[s], kPhiWarps);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm->P_full[i], 1);
            mbar_init(&sm->P_empty[i], kTmWarps);
            mbar_init(&sm->dS_full[i], 1);
            mbar_init(&sm->dS_empty[i], kTmWarps);
            mbar_init(&sm->Sp_full[i], kTmWarps);
            mbar_init(&sm->Sp_empty[i], 1);
            mbar_init(&sm->A_full[i], kTmWarps);
            mbar_init(&sm->A_empty[i], 1);
            mbar_init(&sm->O_full[i], 1);
            mbar_init(&sm->O_empty[i], kTmWarps);
            mbar_init(&sm->aux_empty[i], kTmWarps);
        }
        mbar_init(&sm->mma_done, 1);
        mbar_init(&sm->tm_sync, kTmWarps);
        mbar_init(&sm->phi_sync, kPhiWarps);
        sm->abort_flag = 0;
        fence_mbarrier_init();
        tma_prefetch_desc(&map_q);
        tma_prefetch_desc(&map_k);
        tma_prefetch_desc(&map_v);
        tma_prefetch_desc(&map_y);
    }
    if (warp == kWarpMma) {
        tmem_alloc(&sm->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    if (warp >= kWarpPhi0) {
        const int p = threadIdx.x - kWarpPhi0 * 32;
        sm->z[p] = args.z0 ? args.z0[(size_t)bh * kR + p] : 0.f;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm->tmem_base;
    // The dv slices of one head form a cluster: no slice may write z_out (which
    // may alias z0) before every slice has read z0.
    if (gridDim.x > 1) {
        asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
        asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    }

    if (warp == kWarpTma) {
        // ------------------------------------------------------- producer
        if (lane == 0) {
            int issued = 0;
            for (int c = 0; c < nch; ++c) {
                const int s = c % kStages;
                if (c >= kStages && !wait(cx, &sm->empty[s], ((c / kStages) - 1) & 1)) break;
                if (aborted(cx)) break;
                uint8_t *st = stage_ptr(s);
                mbar_arrive_expect_tx(&sm->full[s], 2 * kTileQ + kTileV);
                const int t0 = c * kC;
                tma_load_3d(st + L::kOffQ, &map_q, &sm->full[s], 0, t0, bh);
                tma_load_3d(st + L::kOffQ + kTileQ / 2, &map_q, &sm->full[s], 64, t0, bh);
                tma_load_3d(st + L::kOffK, &map_k, &sm->full[s], 0, t0, bh);
                tma_load_3d(st + L::kOffK + kTileQ / 2, &map_k, &sm->full[s], 64, t0, bh);
                tma_load_3d(st + L::kOffV, &map_v, &sm->full[s], slice * kDVS, t0, bh);
                issued = c + 1;
            }
            if (aborted(cx)) {
                // Drain: every issued load must land before the CTA may exit.
                for (int c = (issued > kStages ? issued - kStages : 0); c < issued; ++c)
                    mbar_wait(&sm->full[c % kStages], (c / kStages) & 1, cx.limit);
            }
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------ MMA
        if (lane == 0) {
            constexpr uint32_t idP = idesc_bf16_f32(64, 64, false, false);
            constexpr uint32_t idDS = idesc_bf16_f32(128, 64, true, true);
            constexpr uint32_t idQS = idesc_bf16_f32(64, 64, false, true);
            constexpr uint32_t idAV = idesc_bf16_f32(64, 64, false, true);
            for (int c = 0; c < nch && !aborted(cx); ++c) {
                const int s = c % kStages, bb = c & 1, n = c >> 1;
                uint8_t *st = stage_ptr(s);
                const uint32_t aQ = smem_u32(st + L::kOffQ), aK = smem_u32(st + L::kOffK);
                const uint32_t aV = smem_u32(st + L::kOffV);
                const uint32_t aVw = GATED ? smem_u32(st + L::kOffVw) : aV;
                const uint32_t aA = smem_u32(base + L::kOffA + bb * kTileA);
                const uint32_t aSp = smem_u32(base + L::kOffSp + bb * kTileSp);
                if (!wait(cx, &sm->phi_done[s], (c / kStages) & 1)) break;
                // P = Q~ K~^T
                if (c >= 2 && !wait(cx, &sm->P_empty[bb], (n - 1) & 1)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = (kk >> 2) * (kTileQ / 2) + (kk & 3) * 32;
                    tc_mma_bf16(tmem + kColP + bb * 64, smem_desc_sw128(aQ + off, 16, 1024),
                                smem_desc_sw128(aK + off, 16, 1024), idP, kk > 0);
                }
                tc_commit(&sm->P_full[bb]);
                // dS = K~^T (w . V)
                if (c >= 2 && !wait(cx, &sm->dS_empty[bb], (n - 1) & 1)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc_mma_bf16(tmem + kColDS + bb * 64, smem_desc_sw128(aK + kk * 2048, kTileQ / 2, 1024),
                                smem_desc_sw128(aVw + kk * 2048, kTileV, 1024), idDS, kk > 0);
                tc_commit(&sm->dS_full[bb]);
                // O (inter) = Q~ Sprev
                if (c >= 2 && !wait(cx, &sm->O_empty[bb], (n - 1) & 1)) break;
                if (!wait(cx, &sm->Sp_full[bb], n & 1)) break;
                tc_fence_after();
                const uint32_t dInter = tmem + (GATED ? kColO2 : kColO) + bb * 64;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = (kk >> 2) * (kTileQ / 2) + (kk & 3) * 32;
                    tc_mma_bf16(dInter, smem_desc_sw128(aQ + off, 16, 1024),
                                smem_desc_sw128(aSp + kk * 2048, kTileSp, 1024), idQS, kk > 0);
                }
                tc_commit(&sm->Sp_empty[bb]);
                // O (intra) += A V
                if (!wait(cx, &sm->A_full[bb], n & 1)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc_mma_bf16(tmem + kColO + bb * 64, smem_desc_sw128(aA + kk * 32, 16, 1024),
                                smem_desc_sw128(aV + kk * 2048, kTileV, 1024), idAV, GATED ? kk > 0 : true);
                tc_commit(&sm->A_empty[bb]);
                tc_commit(&sm->O_full[bb]);
                tc_commit(&sm->empty[s]);
            }
            // Every MMA this thread issued completes before TMEM is released.
            tc_commit(&sm->mma_done);
            mbar_wait(&sm->mma_done, 0, cx.limit);
        }
    } else if (warp >= kWarpTm0 && warp < kWarpPhi0) {
        // ----------------------------------------------------- TMEM warps
        const int tw = warp - kWarpTm0;          // 0..7
        const int qd = warp & 3;                 // TMEM lane quadrant this warp may access
        const int hf = tw >> 2;                  // column half (0: columns 0..31, 1: 32..63)
        const uint32_t lane_base = static_cast<uint32_t>(qd * 32) << 16;
        const int srow = qd * 32 + lane;         // state row (feature index) of this thread
        const int prow = (lane < kM64RowsPerQuadrant) ? qd * kM64RowsPerQuadrant + lane : -1;
        const bool store_thread = (threadIdx.x == kWarpTm0 * 32);
        uint32_t sync_phase = 0;

        float S[32];
        {
            const float *src = args.S0 ? args.S0 + ((size_t)bh * kR + srow) * args.dv + slice * kDVS + hf * 32 : nullptr;
#pragma unroll
            for (int j = 0; j < 32; ++j) S[j] = src ? src[j] : 0.f;
        }
        float den_prev = 0.f, gam_prev = 1.f;

        // Outputs of chunk j: y = O / (den + eps) -> swizzled staging tile -> TMA store.
        auto epilogue = [&](int j, float den_j, float gam_j) -> bool {
            const int jb = j & 1;
            if (!warp_wait(cx, &sm->O_full[jb], (j >> 1) & 1)) return false;
            tc_fence_after();
            float o[32], o2[32];
            tc_ld_32x32b_x32(tmem + lane_base + kColO + jb * 64 + hf * 32, o);
            if (GATED) tc_ld_32x32b_x32(tmem + lane_base + kColO2 + jb * 64 + hf * 32, o2);
            tc_wait_ld();
            tc_fence_before();
            warp_arrive(&sm->O_empty[jb]);
            const float inv = 1.f / (den_j + args.eps);
            // the staging tile was last read by the store of chunk j-2
            if (store_thread) tma_store_wait_read<1>();
            if (!group_sync(cx, &sm->tm_sync, sync_phase)) return false;
            if (prow >= 0) {
                uint8_t *yt = base + L::kOffY + jb * kTileY;
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int c0 = q4 * 8 + e * 2;
                        const float a0 = GATED ? fmaf(gam_j, o2[c0], o[c0]) : o[c0];
                        const float a1 = GATED ? fmaf(gam_j, o2[c0 + 1], o[c0 + 1]) : o[c0 + 1];
                        w[e] = pack_bf16x2(a0 * inv, a1 * inv);
                    }
                    *reinterpret_cast<uint4 *>(yt + sw128_offset(prow, hf * 4 + q4)) = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
            fence_proxy_async_smem();
            if (!group_sync(cx, &sm->tm_sync, sync_phase)) return false;
            if (store_thread) {
                tma_store_3d(&map_y, base + L::kOffY + jb * kTileY, slice * kDVS, j * kC, bh);
                tma_store_commit();
            }
            warp_arrive(&sm->aux_empty[jb]);
            return true;
        };

        bool ok = true;
        for (int c = 0; c < nch; ++c) {
            const int bb = c & 1, n = c >> 1, s = c % kStages;
            // a(c): the state chunk c reads is the state after chunk c-1
            if (c >= 1) {
                const int pb = (c - 1) & 1;
                if (!warp_wait(cx, &sm->dS_full[pb], ((c - 1) >> 1) & 1)) { ok = false; break; }
                tc_fence_after();
                float d[32];
                tc_ld_32x32b_x32(tmem + lane_base + kColDS + pb * 64 + hf * 32, d);
                tc_wait_ld();
                tc_fence_before();
                warp_arrive(&sm->dS_empty[pb]);
                const float g = GATED ? sm->gC[pb][0] : 1.f;
#pragma unroll
                for (int j = 0; j < 32; ++j) S[j] = GATED ? fmaf(g, S[j], d[j]) : S[j] + d[j];
            }
            if (c >= 2 && !warp_wait(cx, &sm->Sp_empty[bb], (n - 1) & 1)) { ok = false; break; }
            {
                uint8_t *sp = base + L::kOffSp + bb * kTileSp;
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint4 w;
                    w.x = pack_bf16x2(S[q4 * 8 + 0], S[q4 * 8 + 1]);
                    w.y = pack_bf16x2(S[q4 * 8 + 2], S[q4 * 8 + 3]);
                    w.z = pack_bf16x2(S[q4 * 8 + 4], S[q4 * 8 + 5]);
                    w.w = pack_bf16x2(S[q4 * 8 + 6], S[q4 * 8 + 7]);
                    *reinterpret_cast<uint4 *>(sp + sw128_offset(srow, hf * 4 + q4)) = w;
                }
            }
            fence_proxy_async_smem();
            warp_arrive(&sm->Sp_full[bb]);

            // b(c): scores -> masked, decayed BF16 operand A and FP32 row sums
            if (!warp_wait(cx, &sm->phi_done[s], (c / kStages) & 1)) { ok = false; break; }
            if (!warp_wait(cx, &sm->P_full[bb], n & 1)) { ok = false; break; }
            tc_fence_after();
            float p[32];
            tc_ld_32x32b_x32(tmem + lane_base + kColP + bb * 64 + hf * 32, p);
            tc_wait_ld();
            tc_fence_before();
            warp_arrive(&sm->P_empty[bb]);
            float rowsum = 0.f;
            if (prow >= 0) {
                const float bi = GATED ? sm->gb[bb][prow] : 0.f;
                const int zi = GATED ? sm->gz[bb][prow] : -1;
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const int j = hf * 32 + jj;
                    float a = (j <= prow) ? p[jj] : 0.f;
                    if (GATED) a = (j <= prow && zi <= j) ? a * __expf(bi - sm->gb[bb][j]) : 0.f;
                    p[jj] = a;
                    rowsum += a;
                }
            }
            if (c >= 2 && !warp_wait(cx, &sm->A_empty[bb], (n - 1) & 1)) { ok = false; break; }
            if (prow >= 0) {
                uint8_t *at = base + L::kOffA + bb * kTileA;
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint4 w;
                    w.x = pack_bf16x2(p[q4 * 8 + 0], p[q4 * 8 + 1]);
                    w.y = pack_bf16x2(p[q4 * 8 + 2], p[q4 * 8 + 3]);
                    w.z = pack_bf16x2(p[q4 * 8 + 4], p[q4 * 8 + 5]);
                    w.w = pack_bf16x2(p[q4 * 8 + 6], p[q4 * 8 + 7]);
                    *reinterpret_cast<uint4 *>(at + sw128_offset(prow, hf * 4 + q4)) = w;
                }
                sm->densum[bb][hf][prow] = rowsum;
            }
            fence_proxy_async_smem();
            warp_arrive(&sm->A_full[bb]);
            if (!group_sync(cx, &sm->tm_sync, sync_phase)) { ok = false; break; }
            float den_cur = 0.f, gam_cur = 1.f;
            if (prow >= 0) {
                gam_cur = GATED ? sm->gG[bb][prow] : 1.f;
                den_cur = sm->densum[bb][0][prow] + sm->densum[bb][1][prow] + gam_cur * sm->den_inter[bb][prow];
            }
            // e(c-1): outputs of the previous chunk
            if (c >= 1 && !epilogue(c - 1, den_prev, gam_prev)) { ok = false; break; }
            den_prev = den_cur;
            gam_prev = gam_cur;
        }
        if (ok && nch >= 1) {
            // final state: fold in the last chunk's dS, then the last outputs
            const int lb = (nch - 1) & 1;
            if (warp_wait(cx, &sm->dS_full[lb], ((nch - 1) >> 1) & 1)) {
                tc_fence_after();
                float d[32];
                tc_ld_32x32b_x32(tmem + lane_base + kColDS + lb * 64 + hf * 32, d);
                tc_wait_ld();
                tc_fence_before();
                const float g = GATED ? sm->gC[lb][0] : 1.f;
                float *dst = args.S_out + ((size_t)bh * kR + srow) * args.dv + slice * kDVS + hf * 32;
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    float4 v4;
                    v4.x = GATED ? fmaf(g, S[j], d[j]) : S[j] + d[j];
                    v4.y = GATED ? fmaf(g, S[j + 1], d[j + 1]) : S[j + 1] + d[j + 1];
                    v4.z = GATED ? fmaf(g, S[j + 2], d[j + 2]) : S[j + 2] + d[j + 2];
                    v4.w = GATED ? fmaf(g, S[j + 3], d[j + 3]) : S[j + 3] + d[j + 3];
                    *reinterpret_cast<float4 *>(dst + j) = v4;
                }
                epilogue(nch - 1, den_prev, gam_prev);
            }
        }
        if (store_thread) tma_store_wait_all<0>();
    } else if (warp >= kWarpPhi0) {
        // ------------------------------------------------------ phi warps
        const int p = threadIdx.x - kWarpPhi0 * 32;   // 0..127
        const int cc = p & 15;                        // 8-feature column group
        const int rg = p >> 4;                        // 8-row group
        const int blk = cc >> 3, ch = cc & 7;
        uint32_t sync_phase = 0;
        bool ok = true;
        for (int c = 0; c < nch && ok; ++c) {
            const int s = c % kStages, bb = c & 1;
            const int nvalid = min(kC, T - c * kC);
            if (!warp_wait(cx, &sm->full[s], (c / kStages) & 1)) { ok = false; break; }
            if (c >= 2 && !warp_wait(cx, &sm->aux_empty[bb], ((c >> 1) - 1) & 1)) { ok = false; break; }
            uint8_t *st = stage_ptr(s);
            float gc = 1.f;
            if (GATED) {
                // in-chunk cumulative log gate and the last zero gate, rows 0..63
                float la = 0.f;
                int zl = -1;
                if (p < kC) {
                    const float a = (p < nvalid) ? args.alpha[(size_t)bh * T + (size_t)c * kC + p] : 1.f;
                    la = a > 0.f ? logf(a) : 0.f;
                    zl = a > 0.f ? -1 : p;
#pragma unroll
                    for (int off = 1; off < 32; off <<= 1) {
                        const float lo = __shfl_up_sync(0xffffffffu, la, off);
                        const int zo = __shfl_up_sync(0xffffffffu, zl, off);
                        if (lane >= off) { la += lo; zl = max(zl, zo); }
                    }
                    if (p == 31) { sm->carry[0] = la; sm->carry[1] = __int_as_float(zl); }
                }
                if (!group_sync(cx, &sm->phi_sync, sync_phase)) { ok = false; break; }
                if (p >= 32 && p < kC) {
                    la += sm->carry[0];
                    zl = max(zl, __float_as_int(sm->carry[1]));
                }
                if (p < kC) {
                    sm->gb[bb][p] = la;
                    sm->gz[bb][p] = zl;
                    sm->gG[bb][p] = zl < 0 ? expf(la) : 0.f;
                }
                if (!group_sync(cx, &sm->phi_sync, sync_phase)) { ok = false; break; }
                if (p < kC) {
                    const float blast = sm->gb[bb][kC - 1];
                    const int zlast = sm->gz[bb][kC - 1];
                    sm->gw[bb][p] = (zlast <= p) ? expf(blast - sm->gb[bb][p]) : 0.f;
                    if (p == 0) sm->gC[bb][0] = sm->gG[bb][kC - 1];
                }
                if (!group_sync(cx, &sm->phi_sync, sync_phase)) { ok = false; break; }
                gc = sm->gC[bb][0];
            }
            // phi(Q) in place, and Q~ . zprev per row (z is the state before this chunk)
            float zf[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) zf[e] = sm->z[cc * 8 + e];
#pragma unroll 2
            for (int rr = 0; rr < 8; ++rr) {
                const int row = rg * 8 + rr;
                uint4 *ptr = reinterpret_cast<uint4 *>(st + L::kOffQ + blk * (kTileQ / 2) + sw128_offset(row, ch));
                uint4 raw = *ptr;
                uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
                float part = 0.f;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float f0 = phi_elu1(bf16_lo(wv[e])), f1 = phi_elu1(bf16_hi(wv[e]));
                    wv[e] = pack_bf16x2(f0, f1);
                    part = fmaf(bf16_lo(wv[e]), zf[2 * e], part);
                    part = fmaf(bf16_hi(wv[e]), zf[2 * e + 1], part);
                }
                *ptr = make_uint4(wv[0], wv[1], wv[2], wv[3]);
#pragma unroll
                for (int off = 1; off < 16; off <<= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
                if (cc == 0) sm->den_inter[bb][row] = part;
            }
            // phi(K) in place (rows past the end of the sequence become 0), z partials
            float zacc[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) zacc[e] = 0.f;
#pragma unroll 2
            for (int rr = 0; rr < 8; ++rr) {
                const int row = rg * 8 + rr;
                uint4 *ptr = reinterpret_cast<uint4 *>(st + L::kOffK + blk * (kTileQ / 2) + sw128_offset(row, ch));
                uint4 raw = *ptr;
                uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
                const bool valid = row < nvalid;
                const float wr = GATED ? sm->gw[bb][row] : 1.f;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float f0 = valid ? phi_elu1(bf16_lo(wv[e])) : 0.f;
                    const float f1 = valid ? phi_elu1(bf16_hi(wv[e])) : 0.f;
                    wv[e] = pack_bf16x2(f0, f1);
                    zacc[2 * e] = fmaf(wr, bf16_lo(wv[e]), zacc[2 * e]);
                    zacc[2 * e + 1] = fmaf(wr, bf16_hi(wv[e]), zacc[2 * e + 1]);
                }
                *ptr = make_uint4(wv[0], wv[1], wv[2], wv[3]);
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) sm->zred[rg][cc * 8 + e] = zacc[e];
            if (GATED) {
                // w . V for the state update (same swizzled layout as V)
                const uint8_t *vsrc = st + L::kOffV;
                uint8_t *vdst = st + L::kOffVw;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t off = (uint32_t)(p * 4 + i) * 16u;
                    const int row = off >> 7;
                    const float wr = sm->gw[bb][row];
                    uint4 raw = *reinterpret_cast<const uint4 *>(vsrc + off);
                    uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) wv[e] = pack_bf16x2(wr * bf16_lo(wv[e]), wr * bf16_hi(wv[e]));
                    *reinterpret_cast<uint4 *>(vdst + off) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                }
            }
            fence_proxy_async_smem();
            warp_arrive(&sm->phi_done[s]);
            if (!group_sync(cx, &sm->phi_sync, sync_phase)) { ok = false; break; }
            {
                float acc = 0.f;
#pragma unroll
                for (int g = 0; g < 8; ++g) acc += sm->zred[g][p];
                sm->z[p] = fmaf(gc, sm->z[p], acc);
            }
            if (!group_sync(cx, &sm->phi_sync, sync_phase)) { ok = false; break; }
        }
        if (ok && slice == 0) args.z_out[(size_t)bh * kR + p] = sm->z[p];
    }

    // ---------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

cudaError_t launch_prefill_tc(const CUtensorMap &map_q, const CUtensorMap &map_k, const CUtensorMap &map_v,
                              const CUtensorMap &map_y, const PrefillTcArgs &a, int B, bool gated,
                              cudaStream_t stream)
{
    const dim3 grid(a.dv / kDVS, a.H, B);
    const uint32_t bytes = gated ? Layout<true>::kBytes : Layout<false>::kBytes;
    auto kern = gated ? prefill_tc_kernel<true> : prefill_tc_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = grid.x;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, map_q, map_k, map_v, map_y, a);
}

}  // namespace la
