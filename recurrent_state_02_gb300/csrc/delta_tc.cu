// delta_tc.cu -- the delta-rule memory chunk by chunk on the tensor cores (BF16
// operands, FP32 accumulators and state in TMEM).
//
// The rule ("Linear attention：把历史写进状态", hs-black.github.io/posts/linear-attention,
// section "Delta rule：先读旧答案，再写误差") writes, per token, beta_t k_t (v_t - S_{t-1}^T k_t)^T
// and reads y_t = S_t^T q_t after the write.  The pages give no block algorithm for
// it (section "训练时，状态更新也能按块并行"); this kernel uses one derived from the
// update.  For a chunk of C tokens with rows K, Q, V and the state S_prev before
// it, the written rows v'_s = beta_s (v_s - S_{s-1}^T k_s) satisfy, row by row,
//     (I + L) V' = diag(beta) X,   X = V - K S_prev,   L = diag(beta) strictly-lower(K K^T),
// so with T = (I + L)^{-1} diag(beta) (unit lower-triangular, solved per chunk)
//     V' = T X,   S_next = S_prev + K^T V',   O = Q S_prev + ((Q K^T) . M) V',
// M the causal mask with its diagonal (the read follows the write).
//
// T is solved in FP32 on CUDA cores in 2 x 2 blocks of 32 tokens: T00 and T11
// by forward substitution (one column per lane), T10 = -T11 (K1 K0^T) T00.
//
// One CTA of 256 threads per (b, h, 64-column slice of v).  Lane 0 of warp 0
// loads the chunk tiles by TMA (two stages, a chunk ahead); lane 0 of warp 1
// issues the MMAs; warps 0..3 solve for T; warps 4..7 move accumulators
// between TMEM and shared memory (warp w reads TMEM lanes of quadrant w % 4).
// The phases of a chunk follow each other behind CTA barriers:
//   1  G = K K^T, P = Q K^T, KS = K S_prev, O = Q S_prev   (MMA)
//   2  L (FP32), A = P . M, X = V - KS (BF16)             (TMEM warps)
//   3  T (BF16)                                          (solver warps, during 2's A and X)
//   4  V' = T X                                          (MMA)
//   5  V' (BF16)                                         (TMEM warps)
//   6  O += A V', S += K^T V'                            (MMA)
//   7  y = O (BF16), S_prev = S (BF16)                   (TMEM warps)
// Operand layouts follow the prefill kernel's: Q and K tiles of two 64-feature
// blocks and V-shaped tiles of 64 tokens x 64 values (128-byte swizzle), S_prev
// as four blocks of 16 columns (32-byte swizzle).

#include "delta_tc.h"
#include "tc_common.cuh"

namespace la {
namespace {

constexpr int kDThreads = 256;
constexpr int kDS = 64;                          // value columns per CTA
constexpr uint32_t kTQ = kC * kR * 2;            // 16 KB: Q or K tile
constexpr uint32_t kTV = kC * kDS * 2;           // 8 KB: V-shaped tile
constexpr uint32_t kStage = 2 * kTQ + kTV;       // 40 KB
constexpr int LD = 68;                           // FP32 row stride of Lt
constexpr int LDT = 36;                          // FP32 row stride of the 32 x 32 blocks
// shared memory (offsets from a 1024-aligned base)
constexpr uint32_t kOQ = 0, kOK = kTQ, kOV = 2 * kTQ;   // within a stage
constexpr uint32_t kOT = 2 * kStage;             // T (BF16, 64 x 64, A operand)
constexpr uint32_t kOA = kOT + kTV;              // A = P . M (BF16, 64 x 64)
constexpr uint32_t kOX = kOA + kTV;              // X (BF16, V-shaped)
constexpr uint32_t kOVp = kOX + kTV;             // V' (BF16, V-shaped)
constexpr uint32_t kOSp = kOVp + kTV;            // S_prev (BF16, 128 x 64: 4 blocks of 16 columns)
constexpr uint32_t kOL = kOSp + kR * kDS * 2;    // Lt (FP32, 64 x LD): Lt[u][i] for row i, column u
constexpr uint32_t kOT00 = kOL + kC * LD * 4;    // T00 (FP32, [u][j])
constexpr uint32_t kOT11t = kOT00 + 32 * LDT * 4;   // T11 transposed (FP32, [u][i])
constexpr uint32_t kOM = kOT11t + 32 * LDT * 4;  // M = (K1 K0^T) T00 (FP32, [u][j])
constexpr uint32_t kOBeta = kOM + 32 * LDT * 4;  // beta of the chunk, two buffers
constexpr uint32_t kOSmall = kOBeta + 2 * kC * 4;
static_assert(kOT % 1024 == 0 && kOA % 1024 == 0 && kOX % 1024 == 0 && kOVp % 1024 == 0 && kOSp % 1024 == 0,
              "swizzled tiles stay 1024-byte aligned");
static_assert(kOL % 16 == 0 && kOT00 % 16 == 0 && kOT11t % 16 == 0 && kOM % 16 == 0 && kOSmall % 16 == 0,
              "vector access alignment");
// TMEM columns (M = 64 accumulators use lanes 0..15 of each quadrant; S is M = 128)
constexpr uint32_t kCG = 0, kCP = 64, kCKS = 128, kCO = 192, kCVp = 256, kCS = 320;

struct alignas(16) DSmall {
    uint64_t full[2], mma;
    uint32_t tmem_base;
    int abort_flag;
};
constexpr uint32_t kDSmemBytes = kOSmall + sizeof(DSmall) + 1024;
static_assert(kDSmemBytes <= 232448, "shared memory budget");

__device__ __forceinline__ void named_barrier_arrive(int id, int nthreads)
{
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// 32 consecutive columns of one row of an M = 64 accumulator for this thread:
// threads 0..15 get columns [col, col + 32), threads 16..31 [col + 32, col + 64)
// of rows 16 q + (lane & 15).
__device__ __forceinline__ void ld64_row32(uint32_t taddr, float (&v)[32])
{
    float a[16], b[16];
    tc_ld_16x32bx2_x16<32>(taddr, a);
    tc_ld_16x32bx2_x16<32>(taddr + 16, b);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        v[i] = a[i];
        v[16 + i] = b[i];
    }
}

// 8 BF16 values as one 16-byte word.
__device__ __forceinline__ uint4 pack8(const float *f)
{
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                      pack_bf16x2(f[6], f[7]));
}

__device__ __forceinline__ void unpack8(uint4 w, float *f)
{
    const uint32_t x[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        f[2 * e] = bf16_lo(x[e]);
        f[2 * e + 1] = bf16_hi(x[e]);
    }
}

// Element (row, col) of a 64 x 64 BF16 tile with 128-byte rows and the 128-byte swizzle.
__device__ __forceinline__ uint32_t tile_off(int row, int col)
{
    return sw128_offset(row, col >> 3) + (uint32_t)(col & 7) * 2;
}

__device__ __forceinline__ uint16_t bf16_bits(float x) { return (uint16_t)(pack_bf16x2(x, 0.f) & 0xFFFFu); }

__global__ void __launch_bounds__(kDThreads, 1)
delta_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                const __grid_constant__ CUtensorMap map_v, const DeltaTcArgs args)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    DSmall *sm = reinterpret_cast<DSmall *>(base + kOSmall);
    float *Lt = reinterpret_cast<float *>(base + kOL);
    float *T00f = reinterpret_cast<float *>(base + kOT00);
    float *T11t = reinterpret_cast<float *>(base + kOT11t);
    float *Mf = reinterpret_cast<float *>(base + kOM);
    float *betas = reinterpret_cast<float *>(base + kOBeta);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nslice = args.dv / kDS;
    const int bh = blockIdx.x / nslice, slice = blockIdx.x % nslice;
    const int T = args.T, nch = (T + kC - 1) / kC;
    Ctx cx{&sm->abort_flag, args.wait_limit_ns, args.status};

    if (tid == 0) {
        mbar_init(&sm->full[0], 1);
        mbar_init(&sm->full[1], 1);
        mbar_init(&sm->mma, 1);
        sm->abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&sm->tmem_base, 512);
        tmem_relinquish();
    }
    // T's block above the diagonal stays zero
    for (int x = tid; x < (int)(kTV / 16); x += kDThreads)
        reinterpret_cast<uint4 *>(base + kOT)[x] = make_uint4(0, 0, 0, 0);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm->tmem_base;

    auto beta_of = [&](int t) -> float {
        return t < T ? (args.beta ? args.beta[(size_t)bh * T + t] : 1.f) : 0.f;
    };
    // lane 0 of warp 0: the TMA loads of chunk c into stage c % 2
    auto issue = [&](int c) {
        const int s = c & 1, t0 = c * kC;
        uint8_t *st = base + s * kStage;
        mbar_arrive_expect_tx(&sm->full[s], kStage);
        tma_load_3d(st + kOQ, &map_q, &sm->full[s], 0, t0, bh);
        tma_load_3d(st + kOQ + kTQ / 2, &map_q, &sm->full[s], 64, t0, bh);
        tma_load_3d(st + kOK, &map_k, &sm->full[s], 0, t0, bh);
        tma_load_3d(st + kOK + kTQ / 2, &map_k, &sm->full[s], 64, t0, bh);
        tma_load_3d(st + kOV, &map_v, &sm->full[s], slice * kDS, t0, bh);
    };
    int issued = 0;   // chunks whose loads were started (lane 0 of warp 0)
    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_desc(&map_q);
            tma_prefetch_desc(&map_k);
            tma_prefetch_desc(&map_v);
            for (; issued < 2 && issued < nch; ++issued) issue(issued);
        }
        betas[2 * lane] = beta_of(2 * lane);
        betas[2 * lane + 1] = beta_of(2 * lane + 1);
    }
    // the state: S in TMEM (FP32), S_prev in shared memory (BF16)
    const int q4 = warp & 3, ri = 16 * q4 + (lane & 15), hh = lane >> 4;   // TMEM warps: row, column half
    const uint32_t tq = tmem + ((uint32_t)(32 * q4) << 16);
    if (warp >= 4) {
        const int f = 32 * q4 + lane;
        float s0[32], s1[32];
        if (args.S0) {
            const float4 *src = reinterpret_cast<const float4 *>(args.S0 + ((size_t)bh * kR + f) * args.dv + slice * kDS);
#pragma unroll
            for (int m = 0; m < 16; ++m) {
                const float4 x = src[m];
                float *d = m < 8 ? &s0[4 * m] : &s1[4 * (m - 8)];
                d[0] = x.x; d[1] = x.y; d[2] = x.z; d[3] = x.w;
            }
        } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) s0[e] = s1[e] = 0.f;
        }
        tc_st_32x32b_x32(tq + kCS, s0);
        tc_st_32x32b_x32(tq + kCS + 32, s1);
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const float *src = b < 2 ? &s0[16 * b] : &s1[16 * (b - 2)];
            uint8_t *blk = base + kOSp + b * (kR * 32);
            *reinterpret_cast<uint4 *>(blk + sw32_offset(f, 0)) = pack8(src);
            *reinterpret_cast<uint4 *>(blk + sw32_offset(f, 8)) = pack8(src + 8);
        }
        tc_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
    }
    __syncthreads();

    constexpr uint32_t kHi128 = desc_hi(1024, 2), kHi32 = desc_hi(256, 6);
    constexpr uint32_t idKK = idesc_bf16_f32(64, 64, false, false);   // G, P
    constexpr uint32_t idKS = idesc_bf16_f32(64, 64, false, true);    // K S_prev, Q S_prev
    constexpr uint32_t idTV = idesc_bf16_f32(64, 64, false, true);    // T X, A V'
    constexpr uint32_t idDS = idesc_bf16_f32(128, 64, true, true);    // K^T V'
    const uint32_t aT = smem_u32(base + kOT), aA = smem_u32(base + kOA), aX = smem_u32(base + kOX);
    const uint32_t aVp = smem_u32(base + kOVp), aSp = smem_u32(base + kOSp);
    uint32_t mph = 0;       // completions of sm->mma consumed (every thread)
    int commits = 0;        // commits on sm->mma issued (lane 0 of warp 1)
    auto mma_wait = [&]() -> bool {
        const bool ok = warp_wait(cx, &sm->mma, mph & 1);
        ++mph;
        tc_fence_after();
        return ok;
    };

    int c = 0;
    for (; c < nch; ++c) {
        const int s = c & 1, t0 = c * kC;
        const uint32_t st = smem_u32(base + s * kStage);
        const float *bc = betas + s * kC;
        // warp 0: beta of the next chunk, stored in phase 7
        float bn0 = 0.f, bn1 = 0.f;
        if (warp == 0 && c + 1 < nch) {
            bn0 = beta_of(t0 + kC + 2 * lane);
            bn1 = beta_of(t0 + kC + 2 * lane + 1);
        }

        // ---- 1: G = K K^T, P = Q K^T, KS = K S_prev, O = Q S_prev
        if (warp == 1) {
            const bool ok = warp_wait(cx, &sm->full[s], (c >> 1) & 1);
            if (ok && lane == 0) {
                tc_fence_after();
                const uint32_t qlo = desc_lo(st + kOQ, 16), klo = desc_lo(st + kOK, 16), slo = desc_lo(aSp, kR * 32);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t o = ((kk >> 2) * (kTQ / 2) + (kk & 3) * 32) >> 4;
                    const uint32_t so = kk * (512 >> 4);
                    if (kk == 0) {
                        tc_mma_bf16_w<false>(tmem + kCG, klo, kHi128, klo, kHi128, idKK);
                        tc_mma_bf16_w<false>(tmem + kCP, qlo, kHi128, klo, kHi128, idKK);
                        tc_mma_bf16_w<false>(tmem + kCKS, klo, kHi128, slo, kHi32, idKS);
                        tc_mma_bf16_w<false>(tmem + kCO, qlo, kHi128, slo, kHi32, idKS);
                    } else {
                        tc_mma_bf16_w<true>(tmem + kCG, klo + o, kHi128, klo + o, kHi128, idKK);
                        tc_mma_bf16_w<true>(tmem + kCP, qlo + o, kHi128, klo + o, kHi128, idKK);
                        tc_mma_bf16_w<true>(tmem + kCKS, klo + o, kHi128, slo + so, kHi32, idKS);
                        tc_mma_bf16_w<true>(tmem + kCO, qlo + o, kHi128, slo + so, kHi32, idKS);
                    }
                }
                tc_commit(&sm->mma);
                ++commits;
            }
            __syncwarp();
        }
        if (__syncthreads_or(!mma_wait())) break;

        // ---- 2 and 3
        if (warp >= 4) {
            // L = diag(beta) strictly-lower(G) inside the two diagonal 32-blocks and
            // the raw block G10 = K1 K0^T, stored transposed: Lt[j][i] = L[i][j]
            {
                float g[32];
                ld64_row32(tq + kCG, g);
                tc_wait_ld();
                const bool raw = ri >= 32 && hh == 0, diag = (hh == 0) == (ri < 32);
                const float sc = raw ? 1.f : bc[ri];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int j = 32 * hh + e;
                    if (raw || (diag && j < ri)) Lt[j * LD + ri] = sc * g[e];
                }
            }
            named_barrier_arrive(1, kDThreads);   // Lt is ready for the solver warps
            float p[32], ks[32];
            ld64_row32(tq + kCP, p);
            ld64_row32(tq + kCKS, ks);
            tc_wait_ld();
            const uint8_t *vt = base + s * kStage + kOV;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const uint32_t off = sw128_offset(ri, 4 * hh + m);
                float a[8], vf[8];
                unpack8(*reinterpret_cast<const uint4 *>(vt + off), vf);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int j = 32 * hh + 8 * m + e;
                    a[e] = j <= ri ? p[8 * m + e] : 0.f;
                    vf[e] -= ks[8 * m + e];
                }
                *reinterpret_cast<uint4 *>(base + kOA + off) = pack8(a);
                *reinterpret_cast<uint4 *>(base + kOX + off) = pack8(vf);
            }
            fence_proxy_async_smem();
            tc_fence_before();
        } else {
            named_barrier_sync(1, kDThreads);
            // T00, T11 by forward substitution: lane j of warp 0 (1) owns column j
            // of the block; after step u, acc[u] is final and is subtracted from
            // the rows below it.
            if (warp < 2) {
                const int bb = 32 * warp;
                const float *Lb = Lt + bb * LD + bb;
                const float bl = bc[bb + lane];
                float acc[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) acc[i] = i == lane ? bl : 0.f;
#pragma unroll
                for (int u = 0; u < 31; ++u) {
                    const float t = acc[u];
#pragma unroll
                    for (int g4 = (u + 1) >> 2; g4 < 8; ++g4) {
                        const float4 l = *reinterpret_cast<const float4 *>(Lb + u * LD + 4 * g4);
                        const float lv[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (4 * g4 + e > u) acc[4 * g4 + e] = fmaf(-lv[e], t, acc[4 * g4 + e]);
                    }
                }
                if (warp == 0) {
#pragma unroll
                    for (int u = 0; u < 32; ++u) T00f[u * LDT + lane] = acc[u];
                } else {
#pragma unroll
                    for (int m = 0; m < 8; ++m)
                        *reinterpret_cast<float4 *>(T11t + lane * LDT + 4 * m) =
                            make_float4(acc[4 * m], acc[4 * m + 1], acc[4 * m + 2], acc[4 * m + 3]);
                }
#pragma unroll
                for (int u = 0; u < 32; ++u)
                    *reinterpret_cast<uint16_t *>(base + kOT + tile_off(bb + u, bb + lane)) = bf16_bits(acc[u]);
            }
            named_barrier_sync(2, 128);
            // M = G10 T00, rows 8 warp .. 8 warp + 7, column lane
            {
                float m8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
                for (int u = 0; u < 32; ++u) {
                    const float tj = T00f[u * LDT + lane];
                    const float4 g0 = *reinterpret_cast<const float4 *>(Lt + u * LD + 32 + 8 * warp);
                    const float4 g1 = *reinterpret_cast<const float4 *>(Lt + u * LD + 36 + 8 * warp);
                    m8[0] = fmaf(g0.x, tj, m8[0]); m8[1] = fmaf(g0.y, tj, m8[1]);
                    m8[2] = fmaf(g0.z, tj, m8[2]); m8[3] = fmaf(g0.w, tj, m8[3]);
                    m8[4] = fmaf(g1.x, tj, m8[4]); m8[5] = fmaf(g1.y, tj, m8[5]);
                    m8[6] = fmaf(g1.z, tj, m8[6]); m8[7] = fmaf(g1.w, tj, m8[7]);
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) Mf[(8 * warp + e) * LDT + lane] = m8[e];
            }
            named_barrier_sync(2, 128);
            // T10 = -T11 M
            {
                float o8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
                for (int u = 0; u < 32; ++u) {
                    const float mj = Mf[u * LDT + lane];
                    const float4 a0 = *reinterpret_cast<const float4 *>(T11t + u * LDT + 8 * warp);
                    const float4 a1 = *reinterpret_cast<const float4 *>(T11t + u * LDT + 4 + 8 * warp);
                    o8[0] = fmaf(a0.x, mj, o8[0]); o8[1] = fmaf(a0.y, mj, o8[1]);
                    o8[2] = fmaf(a0.z, mj, o8[2]); o8[3] = fmaf(a0.w, mj, o8[3]);
                    o8[4] = fmaf(a1.x, mj, o8[4]); o8[5] = fmaf(a1.y, mj, o8[5]);
                    o8[6] = fmaf(a1.z, mj, o8[6]); o8[7] = fmaf(a1.w, mj, o8[7]);
                }
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    *reinterpret_cast<uint16_t *>(base + kOT + tile_off(32 + 8 * warp + e, lane)) = bf16_bits(-o8[e]);
            }
            fence_proxy_async_smem();
        }
        __syncthreads();

        // ---- 4: V' = T X
        if (warp == 1) {
            if (lane == 0) {
                tc_fence_after();
                const uint32_t tlo = desc_lo(aT, 16), xlo = desc_lo(aX, kTV);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    if (kk == 0) tc_mma_bf16_w<false>(tmem + kCVp, tlo, kHi128, xlo, kHi128, idTV);
                    else tc_mma_bf16_w<true>(tmem + kCVp, tlo + kk * (32 >> 4), kHi128, xlo + kk * (2048 >> 4), kHi128, idTV);
                }
                tc_commit(&sm->mma);
                ++commits;
            }
            __syncwarp();
        }
        if (__syncthreads_or(!mma_wait())) break;

        // ---- 5: V' as BF16
        if (warp >= 4) {
            float vp[32];
            ld64_row32(tq + kCVp, vp);
            tc_wait_ld();
#pragma unroll
            for (int m = 0; m < 4; ++m)
                *reinterpret_cast<uint4 *>(base + kOVp + sw128_offset(ri, 4 * hh + m)) = pack8(&vp[8 * m]);
            fence_proxy_async_smem();
            tc_fence_before();
        }
        __syncthreads();

        // ---- 6: O += A V', S += K^T V'
        if (warp == 1) {
            if (lane == 0) {
                tc_fence_after();
                const uint32_t alo = desc_lo(aA, 16), vlo = desc_lo(aVp, kTV), klo = desc_lo(st + kOK, kTQ / 2);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc_mma_bf16_w<true>(tmem + kCO, alo + kk * (32 >> 4), kHi128, vlo + kk * (2048 >> 4), kHi128, idTV);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc_mma_bf16_w<true>(tmem + kCS, klo + kk * (2048 >> 4), kHi128, vlo + kk * (2048 >> 4), kHi128, idDS);
                tc_commit(&sm->mma);
                ++commits;
            }
            __syncwarp();
        }
        if (__syncthreads_or(!mma_wait())) break;
        // stage s has been read for the last time: load chunk c + 2 into it
        if (warp == 0 && lane == 0 && c + 2 < nch) {
            issue(c + 2);
            issued = c + 3;
        }

        // ---- 7: y = O, S_prev = S (BF16)
        if (warp >= 4) {
            const bool last = c + 1 == nch;
            float o[32];
            ld64_row32(tq + kCO, o);
            float s0[32], s1[32];
            if (!last) {
                tc_ld_32x32b_x32(tq + kCS, s0);
                tc_ld_32x32b_x32(tq + kCS + 32, s1);
            }
            tc_wait_ld();
            if (t0 + ri < T) {
                uint4 *dst = reinterpret_cast<uint4 *>(args.y + ((size_t)bh * T + t0 + ri) * args.dv + slice * kDS + 32 * hh);
#pragma unroll
                for (int m = 0; m < 4; ++m) dst[m] = pack8(&o[8 * m]);
            }
            if (!last) {
                const int f = 32 * q4 + lane;
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    const float *src = b < 2 ? &s0[16 * b] : &s1[16 * (b - 2)];
                    uint8_t *blk = base + kOSp + b * (kR * 32);
                    *reinterpret_cast<uint4 *>(blk + sw32_offset(f, 0)) = pack8(src);
                    *reinterpret_cast<uint4 *>(blk + sw32_offset(f, 8)) = pack8(src + 8);
                }
                fence_proxy_async_smem();
            }
            tc_fence_before();
        }
        if (warp == 0 && c + 1 < nch) {
            float *bnext = betas + ((c + 1) & 1) * kC;
            bnext[2 * lane] = bn0;
            bnext[2 * lane + 1] = bn1;
        }
        __syncthreads();
    }

    // ---------------------------------------------------------- teardown
    if (c == nch) {
        if (warp >= 4) {   // the final state, FP32
            float s0[32], s1[32];
            tc_ld_32x32b_x32(tq + kCS, s0);
            tc_ld_32x32b_x32(tq + kCS + 32, s1);
            tc_wait_ld();
            float4 *dst = reinterpret_cast<float4 *>(args.S_out + ((size_t)bh * kR + 32 * q4 + lane) * args.dv + slice * kDS);
#pragma unroll
            for (int m = 0; m < 8; ++m) dst[m] = make_float4(s0[4 * m], s0[4 * m + 1], s0[4 * m + 2], s0[4 * m + 3]);
#pragma unroll
            for (int m = 0; m < 8; ++m) dst[8 + m] = make_float4(s1[4 * m], s1[4 * m + 1], s1[4 * m + 2], s1[4 * m + 3]);
            tc_fence_before();
        }
    } else {
        // gave up waiting: the loads and MMAs already started complete before the CTA exits
        if (warp == 0 && lane == 0)
            for (int cc = (issued > 2 ? issued - 2 : 0); cc < issued; ++cc)
                mbar_wait(&sm->full[cc & 1], (cc >> 1) & 1, cx.limit);
        if (warp == 1 && lane == 0) {
            tc_commit(&sm->mma);
            mbar_wait(&sm->mma, commits & 1, cx.limit);
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

cudaError_t launch_delta_tc(const CUtensorMap &map_q, const CUtensorMap &map_k, const CUtensorMap &map_v,
                            const DeltaTcArgs &a, int B, cudaStream_t stream)
{
    const long long nblk = (long long)B * a.H * (a.dv / kDS);
    if (nblk < 1 || nblk > 0x7fffffffLL || a.T < 1) return cudaErrorInvalidValue;
    // The attribute is set once per device (not during stream capture of later calls).
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(delta_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    delta_tc_kernel<<<(unsigned)nblk, kDThreads, kDSmemBytes, stream>>>(map_q, map_k, map_v, a);
    return cudaGetLastError();
}

}  // namespace la
