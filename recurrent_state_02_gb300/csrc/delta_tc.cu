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
// stored as the BF16 shared-memory images of the chunk's operand tiles.  The
// second kernel (delta_tc_kernel) then runs only the part that carries the state:
//   1  [KS; QS] = [K; Q] S_prev (M = 128)                  (MMA)
//   2  X = V - KS (BF16)
//   3  V' = T X                                            (MMA)
//   4  V' (BF16)
//   5  [.; O] = [KS; QS] + [0; A] V', S += K^T V'          (MMA)
//   6  y = O (BF16), S_prev = S (BF16)
// with one CTA of 256 threads per (b, h, 64-column slice of v); lane 0 of warp 0
// loads the tiles of a chunk (q, k, v by TMA, A and T by a bulk copy; two stages),
// lane 0 of warp 1 issues the MMAs, and all 8 warps move accumulators between
// TMEM and shared memory (warp w: TMEM lane quadrant w % 4, column half w / 4).
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
constexpr uint32_t kPT = 2 * kTQ;                // T (BF16 image)
constexpr uint32_t kPBeta = kPT + kTV;           // beta of the chunk
constexpr uint32_t kPSmall = kPBeta + kC * 4;
static_assert(kPM + 32 * LDT * 4 <= 2 * kTQ, "L and the solve's blocks fit in the K, Q region");
// workspace per chunk: the A image, then the T image
constexpr uint32_t kWsChunk = 2 * kTV;
static_assert(kPT % 1024 == 0 && kPL % 16 == 0 && kPT00 % 16 == 0 && kPT11t % 16 == 0 && kPM % 16 == 0 &&
                  kPSmall % 16 == 0,
              "alignment");

// --------------------------------------------------------- the state chain
constexpr int kMThreads = 256;
// a stage: K and Q interleaved by 64-feature block, so that [K; Q] is one
// 128-row operand per block, then V, a zero tile (rows 0..63 of the operand
// [0; A]), A and T (A and T arrive together from the workspace)
constexpr uint32_t kSK0 = 0, kSQ0 = kTQ / 2, kSK1 = kTQ, kSQ1 = kTQ + kTQ / 2, kSV = 2 * kTQ;
constexpr uint32_t kSZ = kSV + kTV, kSA = kSZ + kTV, kST = kSA + kTV;
constexpr uint32_t kStage = kST + kTV;           // 64 KB
constexpr uint32_t kMX = 2 * kStage;             // X (BF16, V-shaped)
constexpr uint32_t kMVp = kMX + kTV;             // V' (BF16, V-shaped)
constexpr uint32_t kMSp = kMVp + kTV;            // S_prev (BF16, 128 x 64: 4 blocks of 16 columns)
constexpr uint32_t kMSmall = kMSp + kR * kDS * 2;
static_assert(kStage % 1024 == 0 && kMX % 1024 == 0 && kMVp % 1024 == 0 && kMSp % 1024 == 0,
              "swizzled tiles stay 1024-byte aligned");
// TMEM columns: [KS; QS] then O (M = 128), V' (M = 64), S (M = 128)
constexpr uint32_t kCKQ = 0, kCV = 64, kCS = 128, kMCols = 256;

struct alignas(16) DSmall {
    uint64_t full[2], mma;
    uint32_t tmem_base;
    int abort_flag;
};
constexpr uint32_t kPSmemBytes = kPSmall + sizeof(DSmall) + 1024;
constexpr uint32_t kMSmemBytes = kMSmall + sizeof(DSmall) + 1024;
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

__device__ __forceinline__ void unpack8(uint4 w, float *f)
{
    const uint32_t x[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        f[2 * e] = bf16_lo(x[e]);
        f[2 * e + 1] = bf16_hi(x[e]);
    }
}

__device__ __forceinline__ uint16_t bf16_bits(float x) { return (uint16_t)(pack_bf16x2(x, 0.f) & 0xFFFFu); }

// Element (row, col) of a 64 x 64 BF16 tile with 128-byte rows and the 128-byte swizzle.
__device__ __forceinline__ uint32_t tile_off(int row, int col)
{
    return sw128_offset(row, col >> 3) + (uint32_t)(col & 7) * 2;
}

// A = (Q K^T) . M and T = (I + L)^{-1} diag(beta) of one chunk: one CTA of 128
// threads per (b, h, chunk).  Writes the 8 KB BF16 images of the A and T tiles
// to ws.
__global__ void __launch_bounds__(kPThreads)
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
        mbar_init(&sm->mma, 1);
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
    for (int x = tid; x < (int)(kTV / 16); x += kPThreads)   // the block above the diagonal stays zero
        reinterpret_cast<uint4 *>(base + kPT)[x] = make_uint4(0, 0, 0, 0);
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
                *reinterpret_cast<uint16_t *>(base + kPT + tile_off(bb + u, bb + lane)) = bf16_bits(acc[u]);
        }
        __syncthreads();
        // M = G10 T00 and then T10 = -T11 M: thread (warp, lane) computes rows
        // 4 rg .. 4 rg + 3 and columns 2 cp, 2 cp + 1, rg = 2 warp + lane / 16
        const int rg = 2 * warp + (lane >> 4), cp = lane & 15;
        {
            float2 m4[4] = {};
#pragma unroll 8
            for (int u = 0; u < 32; ++u) {
                const float2 tj = *reinterpret_cast<const float2 *>(T00f + u * LDT + 2 * cp);
                const float4 g = *reinterpret_cast<const float4 *>(Lt + u * LD + 32 + 4 * rg);
                const float gv[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    m4[e].x = fmaf(gv[e], tj.x, m4[e].x);
                    m4[e].y = fmaf(gv[e], tj.y, m4[e].y);
                }
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
                for (int e = 0; e < 4; ++e) {
                    o4[e].x = fmaf(av[e], mj.x, o4[e].x);
                    o4[e].y = fmaf(av[e], mj.y, o4[e].y);
                }
            }
#pragma unroll
            for (int e = 0; e < 4; ++e)
                *reinterpret_cast<uint32_t *>(base + kPT + tile_off(32 + 4 * rg + e, 2 * cp)) =
                    pack_bf16x2(-o4[e].x, -o4[e].y);
        }
        __syncthreads();
        uint4 *dst = reinterpret_cast<uint4 *>(wsc + kTV);
        const uint4 *src = reinterpret_cast<const uint4 *>(base + kPT);
        for (int x = tid; x < (int)(kTV / 16); x += kPThreads) dst[x] = src[x];
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

// The state chain: one CTA of 256 threads per (b, h, 64-column slice of v).
__global__ void __launch_bounds__(kMThreads, 1)
delta_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                const __grid_constant__ CUtensorMap map_v, const DeltaTcArgs args, int nch)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = align1024(smem_raw);
    DSmall *sm = reinterpret_cast<DSmall *>(base + kMSmall);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nslice = args.dv / kDS;
    const int bh = blockIdx.x / nslice, slice = blockIdx.x % nslice;
    const int T = args.T;
    Ctx cx{&sm->abort_flag, args.wait_limit_ns, args.status};
    const uint8_t *tws = static_cast<const uint8_t *>(args.ws) + (size_t)bh * nch * kWsChunk;

    if (tid == 0) {
        mbar_init(&sm->full[0], 1);
        mbar_init(&sm->full[1], 1);
        mbar_init(&sm->mma, 1);
        sm->abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&sm->tmem_base, kMCols);
        tmem_relinquish();
    }
    for (int x = tid; x < (int)(2 * kTV / 16); x += kMThreads)   // rows 0..63 of [0; A], both stages
        reinterpret_cast<uint4 *>(base + (x >= (int)(kTV / 16) ? kStage : 0) + kSZ)[x % (kTV / 16)] =
            make_uint4(0, 0, 0, 0);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm->tmem_base;

    // lane 0 of warp 0: the loads of chunk c into stage c % 2
    auto issue = [&](int c) {
        const int s = c & 1, t0 = c * kC;
        uint8_t *st = base + s * kStage;
        mbar_arrive_expect_tx(&sm->full[s], kStage - kTV);   // all but the zero tile
        tma_load_3d(st + kSK0, &map_k, &sm->full[s], 0, t0, bh);
        tma_load_3d(st + kSQ0, &map_q, &sm->full[s], 0, t0, bh);
        tma_load_3d(st + kSK1, &map_k, &sm->full[s], 64, t0, bh);
        tma_load_3d(st + kSQ1, &map_q, &sm->full[s], 64, t0, bh);
        tma_load_3d(st + kSV, &map_v, &sm->full[s], slice * kDS, t0, bh);
        bulk_load(st + kSA, tws + (size_t)c * kWsChunk, kWsChunk, &sm->full[s]);   // A, T
    };
    int issued = 0;   // chunks whose loads were started (lane 0 of warp 0)
    if (tid == 0) {
        tma_prefetch_desc(&map_q);
        tma_prefetch_desc(&map_k);
        tma_prefetch_desc(&map_v);
        for (; issued < 2 && issued < nch; ++issued) issue(issued);
    }
    // Warp w: TMEM lane quadrant q4, column half ch.  The state: S in TMEM (FP32),
    // S_prev in shared memory (BF16).
    const int q4 = warp & 3, ch = warp >> 2;
    const uint32_t tq = tmem + ((uint32_t)(32 * q4) << 16);
    const int f = 32 * q4 + lane;          // state row (M = 128 accumulators)
    const int rm = 16 * q4 + (lane & 15);  // token row of M = 64 accumulators
    const int cm = 32 * ch + 16 * (lane >> 4);   // their first column for this thread
    auto store_sp = [&](const float (&s)[32]) {
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            uint8_t *blk = base + kMSp + (2 * ch + b) * (kR * 32);
            *reinterpret_cast<uint4 *>(blk + sw32_offset(f, 0)) = pack8(&s[16 * b]);
            *reinterpret_cast<uint4 *>(blk + sw32_offset(f, 8)) = pack8(&s[16 * b + 8]);
        }
    };
    {
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

    constexpr uint32_t idKQ = idesc_bf16_f32(128, 64, false, true);   // [K; Q] S_prev, [0; A] V'
    constexpr uint32_t idTX = idesc_bf16_f32(64, 64, false, true);    // T X
    constexpr uint32_t idS = idesc_bf16_f32(128, 64, true, true);     // K^T V'
    const uint32_t aX = smem_u32(base + kMX);
    const uint32_t aVp = smem_u32(base + kMVp), aSp = smem_u32(base + kMSp);
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

        // ---- 1: [KS; QS] = [K; Q] S_prev
        if (warp == 1) {
            const bool ok = warp_wait(cx, &sm->full[s], (c >> 1) & 1);
            if (ok && lane == 0) {
                tc_fence_after();
                const uint32_t slo = desc_lo(aSp, kR * 32);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t kqlo = desc_lo(st + kSK0, 16) + (((kk >> 2) * kTQ + (kk & 3) * 32) >> 4);
                    if (kk == 0) tc_mma_bf16_w<false>(tmem + kCKQ, kqlo, kHi128, slo, kHi32, idKQ);
                    else tc_mma_bf16_w<true>(tmem + kCKQ, kqlo, kHi128, slo + kk * (512 >> 4), kHi32, idKQ);
                }
                tc_commit(&sm->mma);
                ++commits;
            }
            __syncwarp();
        }
        if (__syncthreads_or(!mma_wait())) break;

        // ---- 2: X = V - KS (token rows 0..63 are TMEM lanes 0..63)
        if (q4 < 2) {
            float ks[32];
            tc_ld_32x32b_x32(tq + kCKQ + 32 * ch, ks);
            tc_wait_ld();
            const uint8_t *vt = base + s * kStage + kSV;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const uint32_t off = sw128_offset(f, 4 * ch + m);
                float vf[8];
                unpack8(*reinterpret_cast<const uint4 *>(vt + off), vf);
#pragma unroll
                for (int e = 0; e < 8; ++e) vf[e] -= ks[8 * m + e];
                *reinterpret_cast<uint4 *>(base + kMX + off) = pack8(vf);
            }
            fence_proxy_async_smem();
            tc_fence_before();
        }
        __syncthreads();

        // ---- 3: V' = T X
        if (warp == 1) {
            if (lane == 0) {
                tc_fence_after();
                const uint32_t tlo = desc_lo(st + kST, 16), xlo = desc_lo(aX, kTV);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    if (kk == 0) tc_mma_bf16_w<false>(tmem + kCV, tlo, kHi128, xlo, kHi128, idTX);
                    else tc_mma_bf16_w<true>(tmem + kCV, tlo + kk * (32 >> 4), kHi128, xlo + kk * (2048 >> 4), kHi128, idTX);
                }
                tc_commit(&sm->mma);
                ++commits;
            }
            __syncwarp();
        }
        if (__syncthreads_or(!mma_wait())) break;

        // ---- 4: V' as BF16
        {
            float vp[16];
            tc_ld_16x32bx2_x16<16>(tq + kCV + 32 * ch, vp);
            tc_wait_ld();
#pragma unroll
            for (int m = 0; m < 2; ++m)
                *reinterpret_cast<uint4 *>(base + kMVp + sw128_offset(rm, (cm >> 3) + m)) = pack8(&vp[8 * m]);
            fence_proxy_async_smem();
            tc_fence_before();
        }
        __syncthreads();

        // ---- 5: O = QS + A V' (rows 64..127 of [KS; QS]), S += K^T V'
        if (warp == 1) {
            if (lane == 0) {
                tc_fence_after();
                const uint32_t zlo = desc_lo(st + kSZ, 16), vlo = desc_lo(aVp, kTV), klo = desc_lo(st + kSK0, kTQ);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc_mma_bf16_w<true>(tmem + kCKQ, zlo + kk * (32 >> 4), kHi128, vlo + kk * (2048 >> 4), kHi128, idKQ);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc_mma_bf16_w<true>(tmem + kCS, klo + kk * (2048 >> 4), kHi128, vlo + kk * (2048 >> 4), kHi128, idS);
                tc_commit(&sm->mma);
                ++commits;
            }
            __syncwarp();
        }
        if (__syncthreads_or(!mma_wait())) break;
        // stage s has been read for the last time: load chunk c + 2 into it
        if (tid == 0 && c + 2 < nch) {
            issue(c + 2);
            issued = c + 3;
        }

        // ---- 6: y = O, S_prev = S (BF16)
        {
            const bool last = c + 1 == nch;
            float sv[32], o[32];
            if (!last) tc_ld_32x32b_x32(tq + kCS + 32 * ch, sv);
            if (q4 >= 2) tc_ld_32x32b_x32(tq + kCKQ + 32 * ch, o);
            tc_wait_ld();
            const int r = f - 64;   // token row of O
            if (q4 >= 2 && t0 + r < T) {
                uint4 *dst = reinterpret_cast<uint4 *>(args.y + ((size_t)bh * T + t0 + r) * args.dv + slice * kDS + 32 * ch);
#pragma unroll
                for (int m = 0; m < 4; ++m) dst[m] = pack8(&o[8 * m]);
            }
            if (!last) {
                store_sp(sv);
                fence_proxy_async_smem();
            }
            tc_fence_before();
        }
        __syncthreads();
    }

    // ---------------------------------------------------------- teardown
    if (c == nch) {
        float sv[32];
        tc_ld_32x32b_x32(tq + kCS + 32 * ch, sv);
        tc_wait_ld();
        float4 *dst = reinterpret_cast<float4 *>(args.S_out + ((size_t)bh * kR + f) * args.dv + slice * kDS + 32 * ch);
#pragma unroll
        for (int m = 0; m < 8; ++m) dst[m] = make_float4(sv[4 * m], sv[4 * m + 1], sv[4 * m + 2], sv[4 * m + 3]);
        tc_fence_before();
    } else {
        // gave up waiting: the loads and MMAs already started complete before the CTA exits
        if (tid == 0)
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
