// delta_tc.cu -- the delta-rule memory chunk by chunk on the tensor cores (BF16
// operands, FP32 accumulators and state in TMEM).
//
// The rule ("Linear attention：把历史写进状态", hs-black.github.io/posts/linear-attention,
// section "Delta rule：先读旧答案，再写误差") writes, per token, beta_t k_t (v_t - S_{t-1}^T k_t)^T
// and reads y_t = S_t^T q_t after the write.  The pages give no block algorithm for
// it (section "训练时，状态更新也能按块并行"); this one is derived from the update.
// For a chunk of C tokens with rows K, Q, V and the state S_prev before it, the
// written rows v'_s = beta_s (v_s - S_{s-1}^T k_s) satisfy, row by row,
//     (I + L) V' = diag(beta) X,   X = V - K S_prev,   L = diag(beta) strictly-lower(K K^T),
// so with T = (I + L)^{-1} diag(beta) (unit lower-triangular, one per chunk)
//     V' = T X,   S_next = S_prev + K^T V',   O = Q S_prev + ((Q K^T) . M) V',
// M the causal mask with its diagonal (the read follows the write).
//
// T and A = (Q K^T) . M depend on q, k and beta alone, so a first kernel
// (delta_t_kernel: one CTA per chunk) forms them for every chunk at once:
// [G; P] = [K; Q] K^T on the tensor cores, A from P, and T from G, solved in FP32
// on CUDA cores in 2 x 2 blocks of 32 tokens (T00 and T11 by forward
// substitution with one column per lane, T10 = -T11 (K1 K0^T) T00).  Both are
// stored as the BF16 shared-memory images of the chunk's operand tiles.
//
// The second kernel (delta_tc_kernel) carries the state.  With W = T K and
// U = T V (neither depends on the state) the written rows are V' = U - W S_prev,
// so a chunk needs two dependent rounds of products:
//   1  [V'; QS] = [U; 0] + [-W; Q] S_prev (M = 128)       (MMA)
//   2  V' (BF16)
//   3  [.; O] += [0; A] V', S += K^T V'                    (MMA)
//   4  S_prev = S (BF16)
// The per-chunk kernel also forms -W (once per head, where the chain would form
// it once per value slice) and stores it as the BF16 image of the operand rows,
// so the chain only loads it.  U of chunk n + 1 = [T; 0] V is formed right after
// round 3 of chunk n, off the chain, into the second of two accumulator buffers,
// where round 1 of chunk n + 1 accumulates onto it.  The warps of TMEM lanes
// 64..127, idle during rounds 1 to 3, store y of chunk n - 1 from the other
// buffer before U of chunk n + 1 overwrites it, so only S_prev stands between
// round 3 and the next round 1.  One CTA of 10 warps per (b, h, 64-column slice
// of v): warps 0..7 move accumulators between TMEM and shared memory (warp w:
// TMEM lane quadrant w % 4, column half w / 4), lane 0 of warp 8 issues every
// MMA and lane 0 of warp 9 loads (k, v, q by TMA; A, T and -W by bulk copies;
// two stages), so that neither waits on the other's work.
// Operand layouts follow the prefill kernel's: 64-feature blocks and V-shaped
// tiles of 64 rows x 128 bytes with the 128-byte swizzle, S_prev as four blocks
// of 16 columns with the 32-byte swizzle.

#include "delta_tc.h"
#include "tc_common.cuh"

namespace la {
namespace {

constexpr int kDS = 64;                          // value columns per CTA
constexpr uint32_t kTQ = kC * kR * 2;            // 16 KB: a Q or K tile (two 64-feature blocks)
constexpr uint32_t kTV = kC * kDS * 2;           // 8 KB: a 64 x 64 BF16 tile
constexpr int LD = 68;                           // FP32 row stride of Lt
constexpr int LDT = 36;                          // FP32 row stride of the 32 x 32 blocks
constexpr uint32_t kHi128 = desc_hi(1024, 2), kHi32 = desc_hi(256, 6);   // SBO and swizzle words

// ------------------------------------------------------------- T per chunk
constexpr int kPThreads = 128;
// K and Q interleaved by 64-feature block ([K; Q] is one 128-row operand per
// block); once [G; P] is complete the region holds L and the solve's FP32 blocks
constexpr uint32_t kPKQ = 0;
constexpr uint32_t kPL = 0;                      // Lt (FP32, 64 x LD): Lt[u][i] holds row i, column u
constexpr uint32_t kPT00 = kPL + kC * LD * 4;    // T00 (FP32, [u][j])
constexpr uint32_t kPT11t = kPT00 + 32 * LDT * 4;   // T11 transposed (FP32, [u][i])
constexpr uint32_t kPM = kPT11t + 32 * LDT * 4;  // M = (K1 K0^T) T00 (FP32, [u][j])
// T (BF16 image) in the rows of Lt that only the substitution of T11 reads: it is
// written once both substitutions are done (the products after them read Lt's
// first 32 rows, T00, T11 and M only)
constexpr uint32_t kPT = 9 * 1024;
// K again once T is complete, its two 64-feature blocks in space that is free by
// then: Lt's first rows, and T00 / T11
constexpr uint32_t kPK0 = 0, kPK1 = 18 * 1024;
constexpr uint32_t kPBeta = 2 * kTQ;             // beta of the chunk
constexpr uint32_t kPSmall = kPBeta + kC * 4;
static_assert(kPM + 32 * LDT * 4 <= 2 * kTQ, "L and the solve's blocks fit in the K, Q region");
static_assert(kPT >= (uint32_t)(kPL + 32 * LD * 4 + 32 * 4 + 32 * 4) && kPT + kTV <= kPT00,
              "T lies past what the products read of Lt and before T00");
static_assert(kPK0 + kTV <= kPT && kPK1 >= kPT + kTV && kPK1 + kTV <= kPM, "K lies clear of T and M");
// workspace per chunk: the A image, the T image, then -W = -T K as the images of
// its two 64-feature blocks
constexpr uint32_t kWsChunk = 4 * kTV;
static_assert(kPT % 1024 == 0 && kPL % 16 == 0 && kPT00 % 16 == 0 && kPT11t % 16 == 0 && kPM % 16 == 0 &&
                  kPSmall % 16 == 0,
              "alignment");

// --------------------------------------------------------- the state chain
constexpr int kMIssuer = 8, kMLoader = 9;        // warps 0..7 move accumulators, 8 issues MMAs, 9 loads
constexpr int kMThreads = 32 * (kMLoader + 1);
// a stage (two): K (two 64-feature blocks), T, a zero tile, A and V, so that
// [T; 0] and [0; A] are 128-row operands
constexpr uint32_t kSK = 0, kST = kTQ, kSZ = kST + kTV, kSA = kSZ + kTV, kSV = kSA + kTV;
constexpr uint32_t kStage = kSV + kTV;           // 48 KB
constexpr uint32_t kWQ = 2 * kTQ;                // [-W; Q] by 64-feature block: W_b at b kTQ, Q_b after it
constexpr uint32_t kMWQ = 2 * kStage;            // two [-W; Q] operands
constexpr uint32_t kMVp = kMWQ + 2 * kWQ;        // V' (BF16, V-shaped)
constexpr uint32_t kMSp = kMVp + kTV;            // S_prev (BF16, 128 x 64: 4 blocks of 16 columns)
constexpr uint32_t kMSmall = kMSp + kR * kDS * 2;
static_assert(kStage % 1024 == 0 && kMWQ % 1024 == 0 && kMVp % 1024 == 0 && kMSp % 1024 == 0,
              "swizzled tiles stay 1024-byte aligned");
// TMEM columns (M = 128 accumulators, row = lane): the two buffers [U / V'; QS / O]
// of even and odd chunks, then S
constexpr uint32_t kCD0 = 0, kCD1 = 64, kCS = 128, kMCols = 256;

struct alignas(16) DSmall {
    uint64_t full[2], mma, fin;
    uint32_t tmem_base;
    int abort_flag;
};
struct alignas(16) MSmall {
    uint64_t full_tv[2], full_ka[2], full_wq[2];   // the three load groups of a stage
    uint64_t mma1, mma3;      // rounds 1 and 3 of a chunk complete
    uint64_t fin;             // every MMA complete (teardown after a timeout)
    uint32_t tmem_base;
    int abort_flag;
};
constexpr uint32_t kPSmemBytes = kPSmall + sizeof(DSmall) + 1024;
constexpr uint32_t kMSmemBytes = kMSmall + sizeof(MSmall) + 1024;
static_assert(kMSmemBytes <= 232448 && kPSmemBytes <= 232448, "shared memory budget");

__device__ __forceinline__ uint8_t *align1024(uint8_t *p)
{
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// 8 BF16 values as one 16-byte word.
__device__ __forceinline__ uint4 pack8(const float *f)
{
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                      pack_bf16x2(f[6], f[7]));
}

__device__ __forceinline__ uint16_t bf16_bits(float x) { return (uint16_t)(pack_bf16x2(x, 0.f) & 0xFFFFu); }

// Element (row, col) of a 64 x 64 BF16 tile with 128-byte rows and the 128-byte swizzle.
__device__ __forceinline__ uint32_t tile_off(int row, int col)
{
    return sw128_offset(row, col >> 3) + (uint32_t)(col & 7) * 2;
}

// A = (Q K^T) . M, T = (I + L)^{-1} diag(beta) and -W = -T K of one chunk: one
// CTA of 128 threads per (b, h, chunk).  Writes the BF16 images of the A and T
// tiles (8 KB each) and of -W (two 64-feature blocks, 8 KB each) to ws.
__global__ void __launch_bounds__(kPThreads, 6)
delta_t_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
               const DeltaTcArgs args, int nch)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = align1024(smem_raw);
    DSmall *sm = reinterpret_cast<DSmall *>(base + kPSmall);
    float *Lt = reinterpret_cast<float *>(base + kPL);
    float *T00f = reinterpret_cast<float *>(base + kPT00);
    float *T11t = reinterpret_cast<float *>(base + kPT11t);
    float *Mf = reinterpret_cast<float *>(base + kPM);
    float *bc = reinterpret_cast<float *>(base + kPBeta);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.x / nch, c = blockIdx.x % nch, t0 = c * kC, T = args.T;
    Ctx cx{&sm->abort_flag, args.wait_limit_ns, args.status};

    if (tid == 0) {
        mbar_init(&sm->full[0], 1);
        mbar_init(&sm->full[1], 1);
        mbar_init(&sm->mma, 1);
        mbar_init(&sm->fin, 1);
        sm->abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&sm->tmem_base, 64);
        tmem_relinquish();
    }
    if (tid < kC) {
        const int t = t0 + tid;
        bc[tid] = t < T ? (args.beta ? args.beta[(size_t)bh * T + t] : 1.f) : 0.f;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm->tmem_base;
    if (tid == 0) {
        mbar_arrive_expect_tx(&sm->full[0], 2 * kTQ);
        tma_load_3d(base + kPKQ, &map_k, &sm->full[0], 0, t0, bh);
        tma_load_3d(base + kPKQ + kTQ / 2, &map_q, &sm->full[0], 0, t0, bh);
        tma_load_3d(base + kPKQ + kTQ, &map_k, &sm->full[0], 64, t0, bh);
        tma_load_3d(base + kPKQ + kTQ + kTQ / 2, &map_q, &sm->full[0], 64, t0, bh);
    }
    uint8_t *wsc = static_cast<uint8_t *>(args.ws) + ((size_t)bh * nch + c) * kWsChunk;

    // [G; P] = [K; Q] K^T (M = 128: G in TMEM lanes 0..63, P in lanes 64..127)
    bool issued = false, ok = true;
    if (warp == 1) {
        ok = warp_wait(cx, &sm->full[0], 0);
        if (ok && lane == 0) {
            tc_fence_after();
            constexpr uint32_t idGP = idesc_bf16_f32(128, 64, false, false);
            const uint32_t klo = desc_lo(smem_u32(base + kPKQ), 16);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t o = ((kk >> 2) * kTQ + (kk & 3) * 32) >> 4;
                if (kk == 0) tc_mma_bf16_w<false>(tmem, klo, kHi128, klo, kHi128, idGP);
                else tc_mma_bf16_w<true>(tmem, klo + o, kHi128, klo + o, kHi128, idGP);
            }
            tc_commit(&sm->mma);
            issued = true;
        }
        __syncwarp();
    }
    ok = warp_wait(cx, &sm->mma, 0) && ok;
    tc_fence_after();
    if (!__syncthreads_or(!ok)) {
        // Warps 0, 1 (TMEM lanes 0..63): L = diag(beta) strictly-lower(G) in the two
        // diagonal 32-blocks and the raw block G10 = K1 K0^T, stored transposed:
        // Lt[j][i] = L[i][j].  Warps 2, 3 (lanes 64..127): A = P . M, stored as the
        // BF16 image of its tile (row i: 128 bytes, 16-byte chunk x at x ^ (i % 8)).
        {
            const int ri = 32 * (warp & 1) + lane;   // token row of G (warps 0, 1) or P (2, 3)
            float v0[32], v1[32];
            const uint32_t tq = tmem + ((uint32_t)(32 * warp) << 16);
            tc_ld_32x32b_x32(tq, v0);
            tc_ld_32x32b_x32(tq + 32, v1);
            tc_wait_ld();
            if (warp < 2) {
                const float bi = bc[ri];
#pragma unroll
                for (int j = 0; j < 64; ++j) {
                    const float g = j < 32 ? v0[j] : v1[j - 32];
                    const bool raw = ri >= 32 && j < 32, diag = (j < 32) == (ri < 32);
                    if (raw || (diag && j < ri)) Lt[j * LD + ri] = (raw ? 1.f : bi) * g;
                }
            } else {
                uint8_t *arow = wsc + (size_t)ri * 128;
#pragma unroll
                for (int x = 0; x < 8; ++x) {
                    float a[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int j = 8 * x + e;
                        a[e] = j <= ri ? (j < 32 ? v0[j] : v1[j - 32]) : 0.f;
                    }
                    *reinterpret_cast<uint4 *>(arow + ((x ^ (ri & 7)) << 4)) = pack8(a);
                }
            }
        }
        __syncthreads();
        // T00, T11 by forward substitution: lane j of warp 0 (1) owns column j of
        // the block; after step u, acc[u] is final and is subtracted from the rows below.
        float acc[32];
        if (warp < 2) {
            const int bb = 32 * warp;
            const float *Lb = Lt + bb * LD + bb;
            const float bl = bc[bb + lane];
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
        }
        __syncthreads();
        // both substitutions are done: T00 and T11 into the T image (over Lt's last
        // rows), and zeros above the diagonal
        if (warp < 2) {
#pragma unroll
            for (int u = 0; u < 32; ++u)
                *reinterpret_cast<uint16_t *>(base + kPT + tile_off(32 * warp + u, 32 * warp + lane)) = bf16_bits(acc[u]);
        } else {
            const int i = tid - 64;   // 0..63: rows 0..31 of the image, two of its upper 16-byte chunks each
#pragma unroll
            for (int x = 0; x < 2; ++x)
                *reinterpret_cast<uint4 *>(base + kPT + sw128_offset(i >> 1, 4 + 2 * (i & 1) + x)) =
                    make_uint4(0, 0, 0, 0);
        }
        // M = G10 T00 and then T10 = -T11 M: thread (warp, lane) computes rows
        // 4 rg .. 4 rg + 3 and columns 2 cp, 2 cp + 1, rg = 2 warp + lane / 16 (the
        // two columns as one packed FP32 pair, each rounded as fmaf would)
        const int rg = 2 * warp + (lane >> 4), cp = lane & 15;
        {
            float2 m4[4] = {};
#pragma unroll 8
            for (int u = 0; u < 32; ++u) {
                const float2 tj = *reinterpret_cast<const float2 *>(T00f + u * LDT + 2 * cp);
                const float4 g = *reinterpret_cast<const float4 *>(Lt + u * LD + 32 + 4 * rg);
                const float gv[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) m4[e] = __ffma2_rn(make_float2(gv[e], gv[e]), tj, m4[e]);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) *reinterpret_cast<float2 *>(Mf + (4 * rg + e) * LDT + 2 * cp) = m4[e];
        }
        __syncthreads();
        {
            float2 o4[4] = {};
#pragma unroll 8
            for (int u = 0; u < 32; ++u) {
                const float2 mj = *reinterpret_cast<const float2 *>(Mf + u * LDT + 2 * cp);
                const float4 a = *reinterpret_cast<const float4 *>(T11t + u * LDT + 4 * rg);
                const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) o4[e] = __ffma2_rn(make_float2(av[e], av[e]), mj, o4[e]);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e)
                *reinterpret_cast<uint32_t *>(base + kPT + tile_off(32 + 4 * rg + e, 2 * cp)) =
                    pack_bf16x2(-o4[e].x, -o4[e].y);
        }
        // the T image (read by the MMAs below) and the solve's blocks (overwritten by
        // the reload of K) are done with in the generic proxy
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            mbar_arrive_expect_tx(&sm->full[1], kTQ);
            tma_load_3d(base + kPK0, &map_k, &sm->full[1], 0, t0, bh);
            tma_load_3d(base + kPK1, &map_k, &sm->full[1], 64, t0, bh);
        }
        uint4 *dst = reinterpret_cast<uint4 *>(wsc + kTV);
        const uint4 *src = reinterpret_cast<const uint4 *>(base + kPT);
        for (int x = tid; x < (int)(kTV / 16); x += kPThreads) dst[x] = src[x];

        // W = T K, one 64-feature block of K at a time (M = 64 into TMEM columns
        // 0..63: row 16 q + i in lane 32 q + i), stored negated as the BF16 image of
        // the rows the state chain multiplies by S_prev.  Thread (warp q, lane l):
        // row 16 q + l % 16, columns 16 (l / 16) + 32 c + [0, 16), c = 0, 1.
        constexpr uint32_t idW = idesc_bf16_f32(64, 64, false, true);
        bool wok = true;
        for (int b = 0; b < 2 && wok; ++b) {
            if (warp == 1) {
                if (b == 0) wok = warp_wait(cx, &sm->full[1], 0);
                if (wok && lane == 0) {
                    tc_fence_after();
                    const uint32_t tlo = desc_lo(smem_u32(base + kPT), 16);
                    const uint32_t klo = desc_lo(smem_u32(base + (b ? kPK1 : kPK0)), kTV);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        if (kk == 0) tc_mma_bf16_w<false>(tmem, tlo, kHi128, klo, kHi128, idW);
                        else tc_mma_bf16_w<true>(tmem, tlo + kk * (32 >> 4), kHi128, klo + kk * (2048 >> 4), kHi128, idW);
                    }
                    tc_commit(&sm->mma);
                }
                __syncwarp();
            }
            wok = warp_wait(cx, &sm->mma, (b + 1) & 1) && wok;
            if (wok) {
                tc_fence_after();
                const uint32_t tq = tmem + ((uint32_t)(32 * warp) << 16);
                const int row = 16 * warp + (lane & 15);
                float w0[16], w1[16];
                tc_ld_16x32bx2_x16<16>(tq, w0);
                tc_ld_16x32bx2_x16<16>(tq + 32, w1);
                tc_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    w0[e] = -w0[e];
                    w1[e] = -w1[e];
                }
                uint8_t *wrow = wsc + (2 + b) * kTV + (size_t)row * 128;
                const int x0 = 2 * (lane >> 4);   // first 16-byte chunk of the row for c = 0
                *reinterpret_cast<uint4 *>(wrow + ((x0 ^ (row & 7)) << 4)) = pack8(&w0[0]);
                *reinterpret_cast<uint4 *>(wrow + (((x0 + 1) ^ (row & 7)) << 4)) = pack8(&w0[8]);
                *reinterpret_cast<uint4 *>(wrow + (((x0 + 4) ^ (row & 7)) << 4)) = pack8(&w1[0]);
                *reinterpret_cast<uint4 *>(wrow + (((x0 + 5) ^ (row & 7)) << 4)) = pack8(&w1[8]);
            }
            tc_fence_before();
            wok = !__syncthreads_or(!wok);
        }
        if (!wok) {
            // gave up waiting: the reload and the MMAs already started complete before the CTA exits
            if (tid == 0) mbar_wait(&sm->full[1], 0, cx.limit);
            if (warp == 1 && lane == 0) {
                tc_commit(&sm->fin);
                mbar_wait(&sm->fin, 0, cx.limit);
            }
        }
    } else {
        // gave up waiting: the copy and the MMAs already started complete before the CTA exits
        if (tid == 0) mbar_wait(&sm->full[0], 0, cx.limit);
        if (warp == 1 && lane == 0 && issued) {
            tc_commit(&sm->mma);
            mbar_wait(&sm->mma, 1, cx.limit);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 64);
    }
}

// The state chain: one CTA of 10 warps per (b, h, 64-column slice of v).
__global__ void __launch_bounds__(kMThreads, 1)
delta_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                const __grid_constant__ CUtensorMap map_v, const DeltaTcArgs args, int nch)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = align1024(smem_raw);
    MSmall *sm = reinterpret_cast<MSmall *>(base + kMSmall);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nslice = args.dv / kDS;
    const int bh = blockIdx.x / nslice, slice = blockIdx.x % nslice;
    const int T = args.T;
    Ctx cx{&sm->abort_flag, args.wait_limit_ns, args.status};
    const uint8_t *tws = static_cast<const uint8_t *>(args.ws) + (size_t)bh * nch * kWsChunk;
    const bool issuer = warp == kMIssuer, loader = warp == kMLoader, tm = warp < kMIssuer;

    if (tid == 0) {
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            mbar_init(&sm->full_tv[s], 1);
            mbar_init(&sm->full_ka[s], 1);
            mbar_init(&sm->full_wq[s], 1);
        }
        mbar_init(&sm->mma1, 1);
        mbar_init(&sm->mma3, 1);
        mbar_init(&sm->fin, 1);
        sm->abort_flag = 0;
        fence_mbarrier_init();
    }
    if (issuer) {
        tmem_alloc(&sm->tmem_base, kMCols);
        tmem_relinquish();
    }
    for (int x = tid; x < 2 * (int)(kTV / 16); x += kMThreads)   // the zero tile of both stages
        reinterpret_cast<uint4 *>(base + (x / (int)(kTV / 16)) * kStage + kSZ)[x % (kTV / 16)] =
            make_uint4(0, 0, 0, 0);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm->tmem_base;

    // Loads of chunk n (lane 0 of the loading warp), in three groups by lifetime:
    // T and V (read by U of the chunk), K and A (read by round 3), and the
    // [-W; Q] operand (read by round 1; -W from the workspace, Q by TMA).
    auto load_tv = [&](int n) {
        uint8_t *st = base + (n & 1) * kStage;
        mbar_arrive_expect_tx(&sm->full_tv[n & 1], 2 * kTV);
        bulk_load(st + kST, tws + (size_t)n * kWsChunk + kTV, kTV, &sm->full_tv[n & 1]);
        tma_load_3d(st + kSV, &map_v, &sm->full_tv[n & 1], slice * kDS, n * kC, bh);
    };
    auto load_ka = [&](int n) {
        uint8_t *st = base + (n & 1) * kStage;
        mbar_arrive_expect_tx(&sm->full_ka[n & 1], kTQ + kTV);
        tma_load_3d(st + kSK, &map_k, &sm->full_ka[n & 1], 0, n * kC, bh);
        tma_load_3d(st + kSK + kTV, &map_k, &sm->full_ka[n & 1], 64, n * kC, bh);
        bulk_load(st + kSA, tws + (size_t)n * kWsChunk, kTV, &sm->full_ka[n & 1]);
    };
    auto load_wq = [&](int n) {
        uint8_t *wq = base + kMWQ + (n & 1) * kWQ;
        const uint8_t *w = tws + (size_t)n * kWsChunk + 2 * kTV;
        mbar_arrive_expect_tx(&sm->full_wq[n & 1], 2 * kTQ);
        bulk_load(wq, w, kTV, &sm->full_wq[n & 1]);
        bulk_load(wq + kTQ, w + kTV, kTV, &sm->full_wq[n & 1]);
        tma_load_3d(wq + kTV, &map_q, &sm->full_wq[n & 1], 0, n * kC, bh);
        tma_load_3d(wq + kTQ + kTV, &map_q, &sm->full_wq[n & 1], 64, n * kC, bh);
    };
    // chunks whose T, V and [-W; Q] loads / K, A loads were started (uniform in
    // the loading warp)
    int nld1 = 0, nld2 = 0;
    if (loader) {
        if (lane == 0) {
            tma_prefetch_desc(&map_q);
            tma_prefetch_desc(&map_k);
            tma_prefetch_desc(&map_v);
            for (int c = 0; c < 2 && c < nch; ++c) {
                load_tv(c);
                load_ka(c);
                load_wq(c);
            }
        }
        nld1 = nld2 = nch < 2 ? nch : 2;
    }
    // TMEM warps 0..7: lane quadrant q4, column half ch.  The state: S in TMEM
    // (FP32), S_prev in shared memory (BF16).
    const int q4 = warp & 3, ch = (warp >> 2) & 1;
    const uint32_t tq = tmem + ((uint32_t)(32 * q4) << 16);
    const int f = 32 * q4 + lane;          // accumulator row: state row, or token row of [V'; O]
    auto store_sp = [&](const float (&s)[32]) {
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            uint8_t *blk = base + kMSp + (2 * ch + b) * (kR * 32);
            *reinterpret_cast<uint4 *>(blk + sw32_offset(f, 0)) = pack8(&s[16 * b]);
            *reinterpret_cast<uint4 *>(blk + sw32_offset(f, 8)) = pack8(&s[16 * b + 8]);
        }
    };
    // warps of lanes 64..127: y of chunk n from the rows 64..127 of its buffer
    auto store_y = [&](int n) {
        float o[32];
        tc_ld_32x32b_x32(tq + ((n & 1) ? kCD1 : kCD0) + 32 * ch, o);
        tc_wait_ld();
        const int t = n * kC + f - 64;
        if (t < T) {
            uint4 *dst = reinterpret_cast<uint4 *>(args.y + ((size_t)bh * T + t) * args.dv + slice * kDS + 32 * ch);
#pragma unroll
            for (int m = 0; m < 4; ++m) dst[m] = pack8(&o[8 * m]);
        }
    };
    if (tm) {
        float s[32];
        if (args.S0) {
            const float4 *src = reinterpret_cast<const float4 *>(args.S0 + ((size_t)bh * kR + f) * args.dv +
                                                                 slice * kDS + 32 * ch);
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const float4 x = src[m];
                s[4 * m] = x.x; s[4 * m + 1] = x.y; s[4 * m + 2] = x.z; s[4 * m + 3] = x.w;
            }
        } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) s[e] = 0.f;
        }
        tc_st_32x32b_x32(tq + kCS + 32 * ch, s);
        store_sp(s);
        tc_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
    }
    __syncthreads();

    constexpr uint32_t idN64 = idesc_bf16_f32(128, 64, false, true);   // [-W; Q] S_prev, [T; 0] V, [0; A] V'
    constexpr uint32_t idS = idesc_bf16_f32(128, 64, true, true);      // K^T V'
    const uint32_t aVp = smem_u32(base + kMVp), aSp = smem_u32(base + kMSp);
    // issuing lane: U = [T; 0] V of chunk n into its accumulator buffer (rows
    // 64..127 start at zero)
    auto mma_u = [&](int n) {
        const uint32_t st = smem_u32(base + (n & 1) * kStage);
        const uint32_t tlo = desc_lo(st + kST, 16), vlo = desc_lo(st + kSV, kTV);
        const uint32_t d = tmem + ((n & 1) ? kCD1 : kCD0);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            if (kk == 0) tc_mma_bf16_w<false>(d, tlo, kHi128, vlo, kHi128, idN64);
            else tc_mma_bf16_w<true>(d, tlo + kk * (32 >> 4), kHi128, vlo + kk * (2048 >> 4), kHi128, idN64);
        }
    };

    bool ok = true;
    if (issuer) {   // U of chunk 0; its [-W; Q] operand
        ok = warp_wait(cx, &sm->full_tv[0], 0);
        if (ok && lane == 0) {
            tc_fence_after();
            mma_u(0);
        }
        __syncwarp();
        ok = ok && warp_wait(cx, &sm->full_wq[0], 0);
    }
    bool failed = __syncthreads_or(!ok);

    for (int n = 0; n < nch && !failed; ++n) {
        const int s = n & 1;
        const uint32_t st = smem_u32(base + s * kStage);
        const uint32_t dcol = s ? kCD1 : kCD0;
        const bool more = n + 1 < nch;

        if (issuer) {
            // ---- 1: [V'; QS] = [U; 0] + [-W; Q] S_prev ([-W; Q] was waited for
            // before the previous chunk's closing barrier)
            if (ok && lane == 0) {
                tc_fence_after();
                const uint32_t slo = desc_lo(aSp, kR * 32), wqlo = desc_lo(smem_u32(base + kMWQ + s * kWQ), 16);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    tc_mma_bf16_w<true>(tmem + dcol, wqlo + (((kk >> 2) * kTQ + (kk & 3) * 32) >> 4), kHi128,
                                        slo + kk * (512 >> 4), kHi32, idN64);
                tc_commit(&sm->mma1);
            }
            __syncwarp();
            // ---- 3 (once V' is stored): O += [0; A] V', S += K^T V'
            ok = ok && warp_wait(cx, &sm->full_ka[s], (n >> 1) & 1);
            named_barrier_sync(1, 160);
            if (ok && lane == 0) {
                tc_fence_after();
                const uint32_t zlo = desc_lo(st + kSZ, 16), vlo = desc_lo(aVp, kTV), klo = desc_lo(st + kSK, kTV);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc_mma_bf16_w<true>(tmem + dcol, zlo + kk * (32 >> 4), kHi128, vlo + kk * (2048 >> 4), kHi128, idN64);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc_mma_bf16_w<true>(tmem + kCS, klo + kk * (2048 >> 4), kHi128, vlo + kk * (2048 >> 4), kHi128, idS);
                tc_commit(&sm->mma3);
            }
            __syncwarp();
            // U of the next chunk, once y of the previous one (same buffer) has been read
            named_barrier_sync(2, 160);
            if (more) {
                ok = ok && warp_wait(cx, &sm->full_tv[s ^ 1], ((n + 1) >> 1) & 1);
                if (ok && lane == 0) {
                    tc_fence_after();
                    mma_u(n + 1);
                }
                __syncwarp();
                ok = ok && warp_wait(cx, &sm->full_wq[s ^ 1], ((n + 1) >> 1) & 1);
            }
        } else if (loader) {
            // stage s and [-W; Q] buffer s: chunk n + 2 once chunk n has been read
            if (n + 2 < nch) {
                ok = warp_wait(cx, &sm->mma1, n & 1);   // round 1 read [-W; Q]; U of the chunk read T, V before it
                if (ok) {
                    if (lane == 0) {
                        load_tv(n + 2);
                        load_wq(n + 2);
                    }
                    nld1 = n + 3;
                }
                ok = ok && warp_wait(cx, &sm->mma3, n & 1);   // round 3 read K, A
                if (ok) {
                    if (lane == 0) load_ka(n + 2);
                    nld2 = n + 3;
                }
                __syncwarp();
            }
        } else {
            if (q4 < 2) {
                // ---- 2: V' as BF16 (TMEM lanes 0..63)
                ok = warp_wait(cx, &sm->mma1, n & 1);
                if (ok) {
                    tc_fence_after();
                    float vp[32];
                    tc_ld_32x32b_x32(tq + dcol + 32 * ch, vp);
                    tc_wait_ld();
#pragma unroll
                    for (int m = 0; m < 4; ++m)
                        *reinterpret_cast<uint4 *>(base + kMVp + sw128_offset(f, 4 * ch + m)) = pack8(&vp[8 * m]);
                    fence_proxy_async_smem();
                    tc_fence_before();
                }
                named_barrier_sync(1, 160);
            } else {
                // y of the previous chunk, before U of the next chunk reuses its buffer
                if (n >= 1) {
                    tc_fence_after();
                    store_y(n - 1);
                    tc_fence_before();
                }
                named_barrier_sync(2, 160);
            }
            // ---- 4: S_prev = S (BF16)
            ok = ok && warp_wait(cx, &sm->mma3, n & 1);
            if (ok && more) {
                tc_fence_after();
                float sv[32];
                tc_ld_32x32b_x32(tq + kCS + 32 * ch, sv);
                tc_wait_ld();
                store_sp(sv);
                fence_proxy_async_smem();
            }
            tc_fence_before();
        }
        failed = __syncthreads_or(!ok);
    }

    // ---------------------------------------------------------- teardown
    if (!failed) {
        if (tm) {
            tc_fence_after();
            if (q4 >= 2) store_y(nch - 1);
            float sv[32];
            tc_ld_32x32b_x32(tq + kCS + 32 * ch, sv);
            tc_wait_ld();
            float4 *dst = reinterpret_cast<float4 *>(args.S_out + ((size_t)bh * kR + f) * args.dv + slice * kDS + 32 * ch);
#pragma unroll
            for (int m = 0; m < 8; ++m) dst[m] = make_float4(sv[4 * m], sv[4 * m + 1], sv[4 * m + 2], sv[4 * m + 3]);
            tc_fence_before();
        }
    } else if (loader && lane == 0) {
        // gave up waiting: the loads already started complete before the CTA exits
        for (int cc = (nld1 > 2 ? nld1 - 2 : 0); cc < nld1; ++cc) {
            mbar_wait(&sm->full_tv[cc & 1], (cc >> 1) & 1, cx.limit);
            mbar_wait(&sm->full_wq[cc & 1], (cc >> 1) & 1, cx.limit);
        }
        for (int cc = (nld2 > 2 ? nld2 - 2 : 0); cc < nld2; ++cc)
            mbar_wait(&sm->full_ka[cc & 1], (cc >> 1) & 1, cx.limit);
    } else if (issuer && lane == 0) {
        // and so do the MMAs
        tc_commit(&sm->fin);
        mbar_wait(&sm->fin, 0, cx.limit);
    }
    __syncthreads();
    if (issuer) {
        tc_fence_after();
        tmem_dealloc(tmem, kMCols);
    }
}

}  // namespace

size_t delta_tc_workspace_bytes(int B, int H, int T)
{
    if (B < 1 || H < 1 || T < 1) return 0;
    return (size_t)B * H * ((T + kC - 1) / kC) * kWsChunk;
}

cudaError_t launch_delta_tc(const CUtensorMap &map_q, const CUtensorMap &map_k, const CUtensorMap &map_v,
                            const DeltaTcArgs &a, int B, cudaStream_t stream)
{
    const int nch = (a.T + kC - 1) / kC;
    const long long nprep = (long long)B * a.H * nch, nmain = (long long)B * a.H * (a.dv / kDS);
    if (a.T < 1 || nprep > 0x7fffffffLL || nmain < 1 || nmain > 0x7fffffffLL) return cudaErrorInvalidValue;
    // The attributes are set once per device (not during stream capture of later calls).
    static OncePerDevice done_p, done_m;
    cudaError_t e = set_smem_once(delta_t_kernel, kPSmemBytes, done_p);
    if (e != cudaSuccess) return e;
    e = set_smem_once(delta_tc_kernel, kMSmemBytes, done_m);
    if (e != cudaSuccess) return e;
    delta_t_kernel<<<(unsigned)nprep, kPThreads, kPSmemBytes, stream>>>(map_q, map_k, a, nch);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    delta_tc_kernel<<<(unsigned)nmain, kMThreads, kMSmemBytes, stream>>>(map_q, map_k, map_v, a, nch);
    return cudaGetLastError();
}

}  // namespace la
