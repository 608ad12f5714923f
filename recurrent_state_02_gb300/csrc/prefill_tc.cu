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
// carrying the FP32 state on chip (S and z in registers of the TMEM warps).
// Per chunk (C = 64, r = 128):
//   TMA    q, k (64 x 128) and the v slice (64 x 64) as BF16 tiles, 128-byte swizzle
//   phi    warps apply phi in place (FP32 math, BF16 result); with a gate they
//          also form the gate products, w . V and the row w
//   MMA    P   = Q~ K~^T            M=64  N=64  K=128  -> TMEM
//          dS  = K~^T (w . V)       M=128 N=64  K=64   -> TMEM
//          dz  = K~^T w             M=128 N=16  K=64   (column 0; w = 1 without a gate)
//          O   = Q~ Sprev           M=64  N=64  K=128  (Sprev as a BF16 operand)
//          dn  = Q~ [zhi, zlo]      M=64  N=16  K=128  (zprev split into two BF16 parts,
//                                                       so Q~ . zprev keeps ~16 bits)
//          O  += A V                M=64  N=64  K=64   (A = masked, decayed P in BF16)
//   TMEM   warps: S <- Gamma S + dS and z <- Gamma z + dz in FP32, Sprev and
//          [zhi, zlo] -> shared memory; P -> A and its FP32 row sums;
//          y = O / (Gamma dn + rowsum + eps) -> TMA store
// Every barrier wait is bounded; on expiry the kernel records a timeout in the
// device status word, drains its own copies and MMAs, frees TMEM and returns.

#include "kernels.h"
#include "sm103_ptx.cuh"

#include <cuda_bf16.h>

namespace la {
namespace {

constexpr int kC = 64;          // tokens per chunk
constexpr int kR = 128;         // feature width r
constexpr int kDVS = 64;        // value columns per CTA
constexpr int kThreads = 512;   // 16 warps
constexpr int kWarpTma = 0, kWarpMma = 1, kWarpTm0 = 4;
constexpr int kTmWarps = 8, kPhiWarps = 6, kPhiThreads = kPhiWarps * 32;

constexpr uint32_t kTileQ = kC * kR * 2;      // 16 KB: two 64-feature blocks of 64 rows x 128 B
constexpr uint32_t kTileV = kC * kDVS * 2;    // 8 KB
constexpr uint32_t kTileA = kC * kC * 2;      // 8 KB
constexpr uint32_t kTileSp = kR * kDVS * 2;   // 16 KB: 128 feature rows x 128 B
constexpr uint32_t kTileZ = 2 * 16 * 128;     // 4 KB: [zhi; zlo; 0..] 16 rows x 128 features, 2 blocks
constexpr uint32_t kTileW = 16 * 128;         // 2 KB: [w; 0..] 16 rows x 64 tokens
constexpr uint32_t kTileY = kC * kDVS * 2;    // 8 KB

__host__ __device__ constexpr bool is_phi_warp(int w) { return w == 2 || w == 3 || w >= 12; }

template <bool GATED>
struct Cfg {
    static constexpr int kStages = GATED ? 2 : 3;
    static constexpr int kNP = GATED ? 1 : 2;                  // P accumulator buffers
    // TMEM columns: P, then [dS | dz] and [O | dn] blocks of 80 (x2), then O_intra (gated, x2)
    static constexpr uint32_t kColP = 0;
    static constexpr uint32_t kColDS = kNP * 64;
    static constexpr uint32_t kColO = kColDS + 2 * 80;
    static constexpr uint32_t kColO2 = kColO + 2 * 80;
    static constexpr uint32_t kCols = kColO2 + (GATED ? 2 * 64 : 0);
    static_assert(kCols <= 512, "TMEM budget");
    // shared memory (offsets from a 1024-aligned base)
    static constexpr uint32_t kOffQ = 0, kOffK = kTileQ, kOffV = 2 * kTileQ;
    static constexpr uint32_t kOffVw = kOffV + kTileV;                      // gated
    static constexpr uint32_t kOffWg = kOffVw + (GATED ? kTileV : 0);       // gated: [w; 0] per stage
    static constexpr uint32_t kStageBytes = kOffWg + (GATED ? kTileW : 0);
    static constexpr uint32_t kOffA = kStages * kStageBytes;
    static constexpr uint32_t kOffSp = kOffA + 2 * kTileA;
    static constexpr uint32_t kOffZ = kOffSp + 2 * kTileSp;
    static constexpr uint32_t kOffY = kOffZ + 2 * kTileZ;
    static constexpr uint32_t kOffW1 = kOffY + 2 * kTileY;                  // ungated: [1; 0]
    static constexpr uint32_t kOffSmall = kOffW1 + kTileW;
};

struct alignas(16) Small {
    float gb[2][kC];            // cumulative log gate inside the chunk
    int gz[2][kC];              // last row <= i whose gate is 0 (-1: none)
    float gG[2][kC];            // Gamma_i
    float gw[2][kC];            // w_j
    float densum[2][2][kC];     // in-chunk row sums, two column halves
    float carry[4];
    uint64_t full[3], empty[3], phi_done[3];
    uint64_t P_full[2], P_empty[2], dS_full[2], dS_empty[2], Sp_full[2], Sp_empty[2];
    uint64_t A_full[2], A_empty[2], O_full[2], O_empty[2], aux_empty[2];
    uint64_t mma_done, tm_sync, phi_sync;
    uint32_t tmem_base;
    int abort_flag;
};

template <bool GATED>
constexpr uint32_t smem_bytes() { return Cfg<GATED>::kOffSmall + sizeof(Small) + 1024; }
static_assert(smem_bytes<false>() <= 232448, "shared memory budget");
static_assert(smem_bytes<true>() <= 232448, "shared memory budget");

// phi(x) = ELU(x) + 1: x + 1 for x > 0, e^x otherwise (NaN propagates).
__device__ __forceinline__ float phi_elu1(float x) { return x > 0.f ? x + 1.f : __expf(x); }

struct Ctx {
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

// Applies phi to the 8 BF16 values of one 16-byte chunk.
__device__ __forceinline__ uint4 phi8(uint4 raw)
{
    uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) w[e] = pack_bf16x2(phi_elu1(bf16_lo(w[e])), phi_elu1(bf16_hi(w[e])));
    return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ uint4 scale8(uint4 raw, float s)
{
    uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) w[e] = pack_bf16x2(s * bf16_lo(w[e]), s * bf16_hi(w[e]));
    return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ void store_bf16x16(uint8_t *tile, int row, int chunk0, const float (&v)[16])
{
    uint4 a, b;
    a.x = pack_bf16x2(v[0], v[1]);   a.y = pack_bf16x2(v[2], v[3]);
    a.z = pack_bf16x2(v[4], v[5]);   a.w = pack_bf16x2(v[6], v[7]);
    b.x = pack_bf16x2(v[8], v[9]);   b.y = pack_bf16x2(v[10], v[11]);
    b.z = pack_bf16x2(v[12], v[13]); b.w = pack_bf16x2(v[14], v[15]);
    *reinterpret_cast<uint4 *>(tile + sw128_offset(row, chunk0)) = a;
    *reinterpret_cast<uint4 *>(tile + sw128_offset(row, chunk0 + 1)) = b;
}

template <bool GATED>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                  const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_y,
                  const PrefillTcArgs args)
{
    using L = Cfg<GATED>;
    constexpr int NST = L::kStages, NP = L::kNP;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Small *sm = reinterpret_cast<Small *>(base + L::kOffSmall);
    Ctx cx{sm, args.wait_limit_ns, args.status};

    const int slice = blockIdx.x;
    const int h = blockIdx.y, b = blockIdx.z;
    const int bh = b * args.H + h;
    const int T = args.T;
    const int nch = (T + kC - 1) / kC;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    auto stage_ptr = [&](int s) { return base + s * L::kStageBytes; };

    // ------------------------------------------------------------ set-up
    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
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
    // Constant operand tiles: rows 1..15 of [w; 0] and rows 2..15 of [zhi; zlo; 0]
    // stay zero; the ungated [1; 0] tile is complete here.
    for (int i = threadIdx.x; i < 2 * (int)kTileZ / 16; i += kThreads)
        reinterpret_cast<uint4 *>(base + L::kOffZ)[i] = make_uint4(0, 0, 0, 0);
    if (GATED) {
        for (int s = 0; s < NST; ++s)
            for (int i = threadIdx.x; i < (int)kTileW / 16; i += kThreads)
                reinterpret_cast<uint4 *>(stage_ptr(s) + L::kOffWg)[i] = make_uint4(0, 0, 0, 0);
    } else {
        for (int i = threadIdx.x; i < (int)kTileW / 16; i += kThreads) {
            const int row = (i * 16) >> 7;
            const uint32_t one2 = 0x3F803F80u;   // two BF16 ones
            reinterpret_cast<uint4 *>(base + L::kOffW1)[i] =
                row == 0 ? make_uint4(one2, one2, one2, one2) : make_uint4(0, 0, 0, 0);
        }
    }
    fence_proxy_async_smem();
    if (warp == kWarpMma) {
        tmem_alloc(&sm->tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm->tmem_base;
    // The dv slices of one head form a cluster: no slice may write z_out (which
    // may alias z0) before every slice has read z0.  Every thread takes part.
    const bool clustered = gridDim.x > 1;
    float z_init = 0.f;
    if (warp >= kWarpTm0 && warp < kWarpTm0 + kTmWarps && args.z0)
        z_init = args.z0[(size_t)bh * kR + (warp & 3) * 32 + lane];
    if (clustered) {
        asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
        asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    }

    if (warp == kWarpTma) {
        // ------------------------------------------------------- producer
        if (lane == 0) {
            int issued = 0;
            for (int c = 0; c < nch; ++c) {
                const int s = c % NST;
                if (c >= NST && !wait(cx, &sm->empty[s], ((c / NST) - 1) & 1)) break;
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
                for (int c = (issued > NST ? issued - NST : 0); c < issued; ++c)
                    mbar_wait(&sm->full[c % NST], (c / NST) & 1, cx.limit);
            }
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------ MMA
        if (lane == 0) {
            constexpr uint32_t idP = idesc_bf16_f32(64, 64, false, false);
            constexpr uint32_t idDS = idesc_bf16_f32(128, 64, true, true);
            constexpr uint32_t idDZ = idesc_bf16_f32(128, 16, true, false);
            constexpr uint32_t idQS = idesc_bf16_f32(64, 64, false, true);
            constexpr uint32_t idDN = idesc_bf16_f32(64, 16, false, false);
            constexpr uint32_t idAV = idesc_bf16_f32(64, 64, false, true);
            const uint32_t aW1 = smem_u32(base + L::kOffW1);
            for (int c = 0; c < nch && !aborted(cx); ++c) {
                const int s = c % NST, bb = c & 1, n = c >> 1;
                const int pb = c % NP, pn = c / NP;
                uint8_t *st = stage_ptr(s);
                const uint32_t aQ = smem_u32(st + L::kOffQ), aK = smem_u32(st + L::kOffK);
                const uint32_t aV = smem_u32(st + L::kOffV);
                const uint32_t aVw = GATED ? smem_u32(st + L::kOffVw) : aV;
                const uint32_t aW = GATED ? smem_u32(st + L::kOffWg) : aW1;
                const uint32_t aA = smem_u32(base + L::kOffA + bb * kTileA);
                const uint32_t aSp = smem_u32(base + L::kOffSp + bb * kTileSp);
                const uint32_t aZ = smem_u32(base + L::kOffZ + bb * kTileZ);
                if (!wait(cx, &sm->phi_done[s], (c / NST) & 1)) break;
                // P = Q~ K~^T
                if (c >= NP && !wait(cx, &sm->P_empty[pb], (pn - 1) & 1)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = (kk >> 2) * (kTileQ / 2) + (kk & 3) * 32;
                    tc_mma_bf16(tmem + L::kColP + pb * 64, smem_desc_sw128(aQ + off, 16, 1024),
                                smem_desc_sw128(aK + off, 16, 1024), idP, kk > 0);
                }
                tc_commit(&sm->P_full[pb]);
                // dS = K~^T (w . V), dz = K~^T w
                if (c >= 2 && !wait(cx, &sm->dS_empty[bb], (n - 1) & 1)) break;
                tc_fence_after();
                const uint32_t dDS = tmem + L::kColDS + bb * 80;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t aKt = smem_desc_sw128(aK + kk * 2048, kTileQ / 2, 1024);
                    tc_mma_bf16(dDS, aKt, smem_desc_sw128(aVw + kk * 2048, kTileV, 1024), idDS, kk > 0);
                    tc_mma_bf16(dDS + 64, aKt, smem_desc_sw128(aW + kk * 32, 16, 1024), idDZ, kk > 0);
                }
                tc_commit(&sm->dS_full[bb]);
                // O (inter) = Q~ Sprev, dn = Q~ [zhi, zlo]
                if (c >= 2 && !wait(cx, &sm->O_empty[bb], (n - 1) & 1)) break;
                if (!wait(cx, &sm->Sp_full[bb], n & 1)) break;
                tc_fence_after();
                const uint32_t dO = tmem + L::kColO + bb * 80;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = (kk >> 2) * (kTileQ / 2) + (kk & 3) * 32;
                    const uint64_t aQd = smem_desc_sw128(aQ + off, 16, 1024);
                    tc_mma_bf16(dO, aQd, smem_desc_sw128(aSp + kk * 2048, kTileSp, 1024), idQS, kk > 0);
                    tc_mma_bf16(dO + 64, aQd, smem_desc_sw128(aZ + (kk >> 2) * (kTileZ / 2) + (kk & 3) * 32, 16, 1024),
                                idDN, kk > 0);
                }
                tc_commit(&sm->Sp_empty[bb]);
                // O (intra) (+)= A V
                if (!wait(cx, &sm->A_full[bb], n & 1)) break;
                tc_fence_after();
                const uint32_t dIn = GATED ? tmem + L::kColO2 + bb * 64 : dO;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc_mma_bf16(dIn, smem_desc_sw128(aA + kk * 32, 16, 1024),
                                smem_desc_sw128(aV + kk * 2048, kTileV, 1024), idAV, GATED ? kk > 0 : true);
                tc_commit(&sm->A_empty[bb]);
                tc_commit(&sm->O_full[bb]);
                tc_commit(&sm->empty[s]);
            }
            // Every MMA this thread issued completes before TMEM is released.
            tc_commit(&sm->mma_done);
            mbar_wait(&sm->mma_done, 0, cx.limit);
        }
    } else if (warp >= kWarpTm0 && warp < kWarpTm0 + kTmWarps) {
        // ----------------------------------------------------- TMEM warps
        const int tw = warp - kWarpTm0;          // 0..7
        const int qd = warp & 3;                 // TMEM lane quadrant this warp may access
        const int hf = tw >> 2;                  // column half (0: columns 0..31, 1: 32..63)
        const uint32_t lane_base = static_cast<uint32_t>(qd * 32) << 16;
        const int srow = qd * 32 + lane;         // state row (feature index) of this thread
        const int prow = qd * 16 + (lane & 15);  // row of the M = 64 tiles (16x32bx2 loads)
        const int pcol = hf * 32 + (lane >> 4) * 16;   // first of this thread's 16 columns
        const bool store_thread = (threadIdx.x == kWarpTm0 * 32);
        uint32_t sync_phase = 0;

        float S[32];
        float zr = z_init;
        {
            const float *src = args.S0 ? args.S0 + ((size_t)bh * kR + srow) * args.dv + slice * kDVS + hf * 32 : nullptr;
#pragma unroll
            for (int j = 0; j < 32; ++j) S[j] = src ? src[j] : 0.f;
        }
        float dintra_prev = 0.f, gam_prev = 1.f;

        // Outputs of chunk j: y = O / (den + eps) -> swizzled staging tile -> TMA store.
        auto epilogue = [&](int j, float dintra_j, float gam_j) -> bool {
            const int jb = j & 1;
            if (!warp_wait(cx, &sm->O_full[jb], (j >> 1) & 1)) return false;
            tc_fence_after();
            float o[16], o2[16], dn;
            tc_ld_16x32bx2_x16<16>(tmem + lane_base + L::kColO + jb * 80 + hf * 32, o);
            if (GATED) tc_ld_16x32bx2_x16<16>(tmem + lane_base + L::kColO2 + jb * 64 + hf * 32, o2);
            tc_ld_16x32bx2_x1<1>(tmem + lane_base + L::kColO + jb * 80 + 64, dn);
            tc_wait_ld();
            tc_fence_before();
            warp_arrive(&sm->O_empty[jb]);
            dn += __shfl_xor_sync(0xffffffffu, dn, 16);          // Q~ . zhi + Q~ . zlo
            const float inv = 1.f / (fmaf(gam_j, dn, dintra_j) + args.eps);
            float yv[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) yv[e] = (GATED ? fmaf(gam_j, o[e], o2[e]) : o[e]) * inv;
            store_bf16x16(base + L::kOffY + jb * kTileY, prow, pcol >> 3, yv);
            fence_proxy_async_smem();
            if (!group_sync(cx, &sm->tm_sync, sync_phase)) return false;
            if (store_thread) {
                tma_store_3d(&map_y, base + L::kOffY + jb * kTileY, slice * kDVS, j * kC, bh);
                tma_store_commit();
                // The next epilogue fills the other staging tile; before the one
                // after it refills this tile, this store must have read it.
                tma_store_wait_read<1>();
            }
            if (GATED) warp_arrive(&sm->aux_empty[jb]);
            return true;
        };

        bool ok = true;
        for (int c = 0; c < nch; ++c) {
            const int bb = c & 1, n = c >> 1, s = c % NST;
            const int pb = c % NP, pn = c / NP;
            // a(c): the state chunk c reads is the state after chunk c-1
            if (c >= 1) {
                const int ob = (c - 1) & 1;
                if (!warp_wait(cx, &sm->dS_full[ob], ((c - 1) >> 1) & 1)) { ok = false; break; }
                tc_fence_after();
                float d[32], dz;
                tc_ld_32x32b_x32(tmem + lane_base + L::kColDS + ob * 80 + hf * 32, d);
                tc_ld_32x32b_x1(tmem + lane_base + L::kColDS + ob * 80 + 64, dz);
                tc_wait_ld();
                tc_fence_before();
                warp_arrive(&sm->dS_empty[ob]);
                const float g = GATED ? sm->gG[ob][kC - 1] : 1.f;
#pragma unroll
                for (int j = 0; j < 32; ++j) S[j] = GATED ? fmaf(g, S[j], d[j]) : S[j] + d[j];
                zr = GATED ? fmaf(g, zr, dz) : zr + dz;
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
                if (hf == 0) {
                    // z as two BF16 parts, rows 0 and 1 of the K-major [zhi; zlo; 0] tile
                    const __nv_bfloat16 zhi = __float2bfloat16_rn(zr);
                    const __nv_bfloat16 zlo = __float2bfloat16_rn(zr - __bfloat162float(zhi));
                    uint8_t *zt = base + L::kOffZ + bb * kTileZ + (srow >> 6) * (kTileZ / 2);
                    const int f = srow & 63;
                    *reinterpret_cast<__nv_bfloat16 *>(zt + sw128_offset(0, f >> 3) + (f & 7) * 2) = zhi;
                    *reinterpret_cast<__nv_bfloat16 *>(zt + sw128_offset(1, f >> 3) + (f & 7) * 2) = zlo;
                }
            }
            fence_proxy_async_smem();
            warp_arrive(&sm->Sp_full[bb]);

            // b(c): scores -> masked, decayed BF16 operand A and FP32 row sums
            if (GATED && !warp_wait(cx, &sm->phi_done[s], (c / NST) & 1)) { ok = false; break; }
            if (!warp_wait(cx, &sm->P_full[pb], pn & 1)) { ok = false; break; }
            tc_fence_after();
            float p[16];
            tc_ld_16x32bx2_x16<16>(tmem + lane_base + L::kColP + pb * 64 + hf * 32, p);
            tc_wait_ld();
            tc_fence_before();
            warp_arrive(&sm->P_empty[pb]);
            float rowsum = 0.f;
            {
                const float bi = GATED ? sm->gb[bb][prow] : 0.f;
                const int zi = GATED ? sm->gz[bb][prow] : -1;
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int j = pcol + e;
                    float a = (j <= prow) ? p[e] : 0.f;
                    if (GATED) a = (j <= prow && zi <= j) ? a * __expf(bi - sm->gb[bb][j]) : 0.f;
                    p[e] = a;
                    rowsum += a;
                }
            }
            rowsum += __shfl_xor_sync(0xffffffffu, rowsum, 16);
            if (c >= 2 && !warp_wait(cx, &sm->A_empty[bb], (n - 1) & 1)) { ok = false; break; }
            store_bf16x16(base + L::kOffA + bb * kTileA, prow, pcol >> 3, p);
            if (lane < 16) sm->densum[bb][hf][prow] = rowsum;
            fence_proxy_async_smem();
            warp_arrive(&sm->A_full[bb]);
            if (!group_sync(cx, &sm->tm_sync, sync_phase)) { ok = false; break; }
            const float dintra_cur = sm->densum[bb][0][prow] + sm->densum[bb][1][prow];
            const float gam_cur = GATED ? sm->gG[bb][prow] : 1.f;
            // e(c-1): outputs of the previous chunk
            if (c >= 1 && !epilogue(c - 1, dintra_prev, gam_prev)) { ok = false; break; }
            dintra_prev = dintra_cur;
            gam_prev = gam_cur;
        }
        if (ok && nch >= 1) {
            // final state: fold in the last chunk's dS and dz, then the last outputs
            const int lb = (nch - 1) & 1;
            if (warp_wait(cx, &sm->dS_full[lb], ((nch - 1) >> 1) & 1)) {
                tc_fence_after();
                float d[32], dz;
                tc_ld_32x32b_x32(tmem + lane_base + L::kColDS + lb * 80 + hf * 32, d);
                tc_ld_32x32b_x1(tmem + lane_base + L::kColDS + lb * 80 + 64, dz);
                tc_wait_ld();
                tc_fence_before();
                const float g = GATED ? sm->gG[lb][kC - 1] : 1.f;
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
                if (slice == 0 && hf == 0) args.z_out[(size_t)bh * kR + srow] = GATED ? fmaf(g, zr, dz) : zr + dz;
                // publishes the store thread's last read-completion wait to every TMEM warp
                if (group_sync(cx, &sm->tm_sync, sync_phase)) epilogue(nch - 1, dintra_prev, gam_prev);
            }
        }
        if (store_thread) tma_store_wait_all<0>();
    } else if (is_phi_warp(warp)) {
        // ------------------------------------------------------ phi warps
        const int pp = (warp < 4 ? (warp - 2) * 32 : 64 + (warp - 12) * 32) + lane;   // 0..191
        uint32_t sync_phase = 0;
        bool ok = true;
        for (int c = 0; c < nch && ok; ++c) {
            const int s = c % NST, bb = c & 1;
            const int nvalid = min(kC, T - c * kC);
            if (!warp_wait(cx, &sm->full[s], (c / NST) & 1)) { ok = false; break; }
            uint8_t *st = stage_ptr(s);
            if (GATED) {
                if (c >= 2 && !warp_wait(cx, &sm->aux_empty[bb], ((c >> 1) - 1) & 1)) { ok = false; break; }
                // in-chunk cumulative log gate and the last zero gate, rows 0..63 (warps 2, 3)
                float la = 0.f;
                int zl = -1;
                if (pp < kC) {
                    const float a = (pp < nvalid) ? args.alpha[(size_t)bh * T + (size_t)c * kC + pp] : 1.f;
                    la = a > 0.f ? logf(a) : 0.f;
                    zl = a > 0.f ? -1 : pp;
#pragma unroll
                    for (int off = 1; off < 32; off <<= 1) {
                        const float lo = __shfl_up_sync(0xffffffffu, la, off);
                        const int zo = __shfl_up_sync(0xffffffffu, zl, off);
                        if (lane >= off) { la += lo; zl = max(zl, zo); }
                    }
                    if (pp == 31) { sm->carry[0] = la; sm->carry[1] = __int_as_float(zl); }
                }
                if (!group_sync(cx, &sm->phi_sync, sync_phase)) { ok = false; break; }
                if (pp >= 32 && pp < kC) {
                    la += sm->carry[0];
                    zl = max(zl, __float_as_int(sm->carry[1]));
                }
                if (pp < kC) {
                    sm->gb[bb][pp] = la;
                    sm->gz[bb][pp] = zl;
                    sm->gG[bb][pp] = zl < 0 ? expf(la) : 0.f;
                }
            }
            // phi(Q), phi(K) in place; key rows past the end of the sequence become 0
            for (int ci = pp; ci < 2048; ci += kPhiThreads) {
                const bool isk = ci >= 1024;
                const uint32_t off = (uint32_t)(ci & 1023) * 16u;
                uint4 *ptr = reinterpret_cast<uint4 *>(st + (isk ? L::kOffK : L::kOffQ) + off);
                const int row = (off & 8191u) >> 7;
                *ptr = (isk && row >= nvalid) ? make_uint4(0, 0, 0, 0) : phi8(*ptr);
            }
            if (GATED) {
                if (!group_sync(cx, &sm->phi_sync, sync_phase)) { ok = false; break; }
                if (pp < kC) {
                    const float blast = sm->gb[bb][kC - 1];
                    const int zlast = sm->gz[bb][kC - 1];
                    const float wj = (zlast <= pp) ? expf(blast - sm->gb[bb][pp]) : 0.f;
                    sm->gw[bb][pp] = wj;
                    // row 0 of the K-major [w; 0] operand
                    *reinterpret_cast<__nv_bfloat16 *>(st + L::kOffWg + sw128_offset(0, pp >> 3) + (pp & 7) * 2) =
                        __float2bfloat16_rn(wj);
                }
                if (!group_sync(cx, &sm->phi_sync, sync_phase)) { ok = false; break; }
                // w . V for the state update (same swizzled layout as V)
                for (int ci = pp; ci < (int)kTileV / 16; ci += kPhiThreads) {
                    const uint32_t off = (uint32_t)ci * 16u;
                    const uint4 raw = *reinterpret_cast<const uint4 *>(st + L::kOffV + off);
                    *reinterpret_cast<uint4 *>(st + L::kOffVw + off) = scale8(raw, sm->gw[bb][off >> 7]);
                }
            }
            fence_proxy_async_smem();
            warp_arrive(&sm->phi_done[s]);
        }
    }

    // ---------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

cudaError_t launch_prefill_tc(const CUtensorMap &map_q, const CUtensorMap &map_k, const CUtensorMap &map_v,
                              const CUtensorMap &map_y, const PrefillTcArgs &a, int B, bool gated,
                              cudaStream_t stream)
{
    const dim3 grid(a.dv / kDVS, a.H, B);
    const uint32_t bytes = gated ? smem_bytes<true>() : smem_bytes<false>();
    auto kern = gated ? prefill_tc_kernel<true> : prefill_tc_kernel<false>;
    // The attribute is set once per device (not during stream capture of later calls).
    static bool attr_set[2][64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[gated][dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return e;
        attr_set[gated][dev] = true;
    }
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
