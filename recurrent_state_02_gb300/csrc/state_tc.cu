// state_tc.cu -- the state pass and the scan of the sequence-segmented prefill.
//
// Method ("Linear attention：把历史写进状态", hs-black.github.io/posts/linear-attention,
// section "门控递推为什么能做并行 scan？"): the per-token updates
//     S_t = alpha_t S_{t-1} + phi(k_t) v_t^T,   z_t = alpha_t z_{t-1} + phi(k_t)
// are affine maps of the state, and a run of them composes into one affine map
//     S -> A S + dS,   z -> A z + dz,
// with A the product of the run's gates and (dS, dz) the state the run would
// produce from a zero state.  state_tc_kernel computes (A, dS, dz) for each
// sub-segment (part) of a head's sequence as one accumulation over its chunks,
// dS = sum_j e_j phi(k_j) [v_j | 1]^T with e_j the product of the gates after
// token j within the part: each key row carries its whole decay, so the state in
// TMEM is never rescaled.  The chunks are walked from the part's end, and e_j =
// e^{offset} w_j with w_j the decay to the chunk's end and the offset summed
// over the chunks already walked (0 once a zero gate has been passed).
// seg_scan_kernel then applies the maps in sequence order to S0, z0 and writes
// the start state of every output segment, from which the prefill kernel
// processes the segments in parallel.
//
// The backward's key-side sweeps carry, in reversed time, the state
//     G_t = phi(q_t) dn_t^T + alpha_{t+1} G_{t+1},   g_t = dd_t phi(q_t) + alpha_{t+1} g_{t+1}
// (dn_t = dy_t / d_t, dd_t = -(dy_t . y_t) / d_t), which is affine in the same
// way.  The REV form of the state pass takes key phi(q), value dn and dd in
// place of the column of ones, each token weighted by its decay back to the
// part's start (Gamma_t within the chunk times the offset of the chunks before
// it, walked from the part's start); its map sends the state entering the
// sub-segment from the right to the state it hands to the left.
// The scan then applies the maps from the end of the sequence backwards,
// starting from dL/dS_T, dL/dz_T.

#include "tc_common.cuh"

namespace la {
namespace {

// Value columns per CTA (DVS): 64 or 128, as the chunk kernel.  A CTA owns one
// (b, h, DVS-column slice, part).
constexpr int kThreads = 384;       // 12 warps
constexpr int kWarpTma = 0, kWarpMma = 1, kWarpTm0 = 4, kTmWarps = 4;
// phi warps: 2, 3 and 8..11 (spread over the four schedulers)
__host__ __device__ constexpr bool is_phi_warp(int w) { return w == 2 || w == 3 || w >= 8; }
__host__ __device__ constexpr int phi_index(int w) { return w < 4 ? w - 2 : w - 6; }
constexpr int kPhiWarps = 6, kPhiThreads = kPhiWarps * 32;
constexpr uint32_t kTileK = kC * kR * 2;       // 16 KB: two 64-feature blocks of 64 rows x 128 B
constexpr uint32_t kBlkV = kC * 64 * 2;        // one 64-column block of V (8 KB)
constexpr uint32_t kTileOnes = kC * 128;       // 8 KB: the block of ones after V in [V | 1 0..]
constexpr int kMaxStages = 4;

// Two CTAs are resident per SM (each at most 113 KB of shared memory), so that
// the many short parts of a segment stream at the bandwidth of the SM.
// Per-chunk scalars: (reversed pass) 1 / d_t and dd_t (0 for rows past T);
// (gated) e^{offset}, the gate product between the chunk and the part's end
// (forward) or start (reversed) over the chunks walked before it, 0 past a zero gate.
struct alignas(16) RevRing {
    float invd[kAux][kC];
    float dd[kAux][kC];
    float eoff[kAux];
};

// REV: the reversed-time pass of the backward (DVS 128 only): the column block
// holds dd_t, so each stage carries its own after the value tile.
template <bool GATED, int DVS, bool REV = false>
struct SCfg {
    static_assert(DVS == 64 || DVS == 128, "value columns per CTA");
    static_assert(!REV || DVS == 128, "the reversed pass takes whole heads");
    static constexpr int kStages = REV ? 2 : DVS == 128 ? 3 : 4;
    static constexpr uint32_t kTileV = (DVS / 64) * kBlkV;
    static constexpr uint32_t kOffK = 0, kOffV = kTileK, kOffStageCol = kTileK + kTileV;
    static constexpr uint32_t kStageBytes = kTileK + kTileV + (REV ? kTileOnes : 0);
    static_assert(kStageBytes % 1024 == 0, "stage tiles stay 1024-byte aligned");
    static constexpr uint32_t kOffOnes = kStages * kStageBytes;
    static constexpr uint32_t kOffGate = kOffOnes + (REV ? 0 : kTileOnes);
    static constexpr uint32_t kOffRev = kOffGate + (GATED ? sizeof(GateRing) : 0);
    static constexpr uint32_t kOffSmall = kOffRev + ((REV || GATED) ? sizeof(RevRing) : 0);
    static constexpr uint32_t kTmemCols = DVS == 128 ? 256 : 128;   // [S | z]: DVS + 16 columns (z is column DVS)
};

struct alignas(16) SmallS {
    uint64_t full[kMaxStages], empty[kMaxStages], phi_done[kMaxStages];
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort_flag;
};

template <bool GATED, int DVS, bool REV = false>
__host__ __device__ constexpr uint32_t smem_bytes() { return SCfg<GATED, DVS, REV>::kOffSmall + sizeof(SmallS) + 1024; }
// two resident CTAs per SM: 2 x (bytes + 1 KB reserved) within the SM's 228 KB
static_assert(2 * (smem_bytes<true, 64>() + 1024) <= 233472, "shared memory budget");
static_assert(2 * (smem_bytes<false, 64>() + 1024) <= 233472, "shared memory budget");
static_assert(2 * (smem_bytes<true, 128>() + 1024) <= 233472, "shared memory budget");
static_assert(2 * (smem_bytes<false, 128>() + 1024) <= 233472, "shared memory budget");
static_assert(2 * (smem_bytes<true, 128, true>() + 1024) <= 233472, "shared memory budget");
static_assert(2 * (smem_bytes<false, 128, true>() + 1024) <= 233472, "shared memory budget");

template <bool GATED, int DVS, bool REV>
__global__ void __launch_bounds__(kThreads, 2)
state_tc_kernel(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                const StateTcArgs args)
{
    using L = SCfg<GATED, DVS, REV>;
    constexpr int NST = L::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    SmallS *sm = reinterpret_cast<SmallS *>(base + L::kOffSmall);
    GateRing *gr = reinterpret_cast<GateRing *>(base + L::kOffGate);   // gated only
    RevRing *rr = reinterpret_cast<RevRing *>(base + L::kOffRev);      // REV or gated
    Ctx cx{&sm->abort_flag, args.wait_limit_ns, args.status};

    // grid: (dv slice, h, b * nsub + m); sub-segment m is part j of output segment g.
    // Packed sequences: (dv slice, h, k * sub + j), part j of the segment that
    // ends at the varlen plan's boundary k (sub parts per boundary, from the plan).
    const int slice = blockIdx.x, h = blockIdx.y;
    const bool varlen = args.bds != nullptr;
    int b, g, j, seq0 = 0, T = args.T, seg_chunks = args.seg_chunks, sub_chunks = args.sub_chunks;
    size_t orow;   // row of this part's outputs in A and dS
    if (varlen) {
        const int sub = args.seg_len[2];
        const int2 e = args.bds[blockIdx.z / sub];
        if (e.x < 0) return;   // beyond the plan's boundaries: no work
        b = e.x;
        g = e.y;
        j = blockIdx.z % sub;
        seq0 = args.cu_seqlens[b];
        T = args.cu_seqlens[b + 1] - seq0;
        seg_chunks = args.seg_len[0];
        sub_chunks = args.seg_len[1];
        orow = (size_t)blockIdx.z * args.H + h;
    } else {
        b = blockIdx.z / args.nsub;
        const int m = blockIdx.z % args.nsub;
        g = m / args.sub_per_seg + args.seg_first;
        j = m % args.sub_per_seg;
        orow = (size_t)m * ((gridDim.z / args.nsub) * args.H) + b * args.H + h;
    }
    const int bh = b * args.H + h;
    // the last two TMA coordinates of a box starting at token t0, and the row of
    // token t's gate
    auto tma_c1 = [&](int t0) { return varlen ? h : t0; };
    auto tma_c2 = [&](int t0) { return varlen ? seq0 + t0 : bh; };
    auto gate_row = [&](int t) -> size_t { return varlen ? (size_t)(seq0 + t) * args.H + h : (size_t)bh * T + t; };
    const int cs = g * seg_chunks + j * sub_chunks;                           // first chunk
    const int nch = max(0, min(min(cs + sub_chunks, (g + 1) * seg_chunks), (T + kC - 1) / kC) - cs);
    const int tb = cs * kC;                                                   // first token
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // first token of the c-th chunk processed: from the part's end in forward time,
    // from its start in reversed time, so that the chunks walked before a chunk
    // are the ones its tokens decay through (their gate product is the offset)
    auto chunk_t0 = [&](int c) { return tb + (REV ? c : nch - 1 - c) * kC; };
    auto stage_ptr = [&](int s) { return base + s * L::kStageBytes; };

    // ------------------------------------------------------------ set-up
    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(&sm->full[s], (GATED || REV) ? 2 : 1);   // TMA bytes (+ gate data, scalars)
            mbar_init(&sm->empty[s], 1);
            mbar_init(&sm->phi_done[s], kPhiWarps);
        }
        mbar_init(&sm->mma_done, 1);
        sm->abort_flag = 0;
        fence_mbarrier_init();
        tma_prefetch_desc(&map_k);
        tma_prefetch_desc(&map_v);
    }
    if (REV) {
        // the column blocks of the stages: zero but for column 0, written per chunk
        for (int i = threadIdx.x; i < NST * (int)(kTileOnes / 16); i += kThreads)
            reinterpret_cast<uint4 *>(base + (i / (kTileOnes / 16)) * L::kStageBytes + L::kOffStageCol)[i % (kTileOnes / 16)] =
                make_uint4(0, 0, 0, 0);
        __syncthreads();
    } else {
        for (int i = threadIdx.x; i < (int)kTileOnes / 16; i += kThreads)
            reinterpret_cast<uint4 *>(base + L::kOffOnes)[i] = make_uint4(0, 0, 0, 0);
        __syncthreads();
        if (threadIdx.x < kC)   // element (column 0, token row k): 16-byte chunk 0 of row k after the swizzle
            *reinterpret_cast<uint16_t *>(base + L::kOffOnes + sw128_offset(threadIdx.x, 0)) = 0x3F80u;
    }
    fence_proxy_async_smem();
    if (warp == kWarpMma) {
        tmem_alloc(&sm->tmem_base, L::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm->tmem_base;
    // the state starts at zero, before any increment is issued
    if (warp >= kWarpTm0 && warp < kWarpTm0 + kTmWarps) {
        const uint32_t lb = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        float zero[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) zero[i] = 0.f;
#pragma unroll
        for (int pc = 0; pc < DVS / 32; ++pc) tc_st_32x32b_x32(lb + 32 * pc, zero);
        tc_st_32x32b_x1(lb + DVS, 0.f);
        tc_wait_st();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (warp == kWarpTma) {
        // ------------------------------------------------------- producer
        int issued = 0;
        float off = 0.f;   // gated: log of the gate product over the chunks walked so far
        bool cut = false;  // a zero gate has been walked
        for (int c = 0; c < nch; ++c) {
            const int s = c % NST;
            const int t0 = chunk_t0(c);
            float a0 = 1.f, a1 = 1.f;
            if (GATED) {
                if (t0 + 2 * lane < T) a0 = args.alpha[gate_row(t0 + 2 * lane)];
                if (t0 + 2 * lane + 1 < T) a1 = args.alpha[gate_row(t0 + 2 * lane + 1)];
            }
            float2 dv2 = make_float2(1.f, 1.f), dd2 = make_float2(0.f, 0.f);
            if (REV) {
                const float *dp = args.d + (size_t)bh * T, *ddp = args.dd + (size_t)bh * T;
                if (t0 + 2 * lane < T) { dv2.x = dp[t0 + 2 * lane]; dd2.x = ddp[t0 + 2 * lane]; }
                if (t0 + 2 * lane + 1 < T) { dv2.y = dp[t0 + 2 * lane + 1]; dd2.y = ddp[t0 + 2 * lane + 1]; }
            }
            // the ring entry of chunk c held chunk c - kAux's, which phi (its only
            // reader) finished before the MMA of chunk c - NST released the stage
            static_assert(kAux >= NST, "ring entries outlive their stage");
            if (c >= NST && !warp_wait(cx, &sm->empty[s], ((c / NST) - 1) & 1)) break;
            if (__shfl_sync(0xffffffffu, aborted(cx) ? 1 : 0, 0)) break;
            uint8_t *st = stage_ptr(s);
            if (lane == 0) {
                mbar_arrive_expect_tx(&sm->full[s], kTileK + L::kTileV);
                const int cy = tma_c1(t0), cz = tma_c2(t0);
                tma_load_3d(st + L::kOffK, &map_k, &sm->full[s], 0, cy, cz);
                tma_load_3d(st + L::kOffK + kTileK / 2, &map_k, &sm->full[s], 64, cy, cz);
#pragma unroll
                for (int vb = 0; vb < DVS / 64; ++vb)
                    tma_load_3d(st + L::kOffV + vb * kBlkV, &map_v, &sm->full[s], slice * DVS + vb * 64, cy, cz);
                if (c + NST < nch) {   // warm L2 for the load that reuses this stage
                    const int tp = chunk_t0(c + NST), yp = tma_c1(tp), zp = tma_c2(tp);
                    if (slice == 0) {
                        tma_prefetch_l2_3d(&map_k, 0, yp, zp);
                        tma_prefetch_l2_3d(&map_k, 64, yp, zp);
                    }
#pragma unroll
                    for (int vb = 0; vb < DVS / 64; ++vb) tma_prefetch_l2_3d(&map_v, slice * DVS + vb * 64, yp, zp);
                }
            }
            if (GATED) {
                gate_products(a0, a1, lane, c % kAux, gr);
                __syncwarp();
                if (lane == 0) rr->eoff[c % kAux] = cut ? 0.f : expf(off);
                const float blast = gr->gb[c % kAux][kC - 1];
                cut = cut || gr->gz[c % kAux][kC - 1] >= 0;
                off += blast;
            }
            if (REV) {
                *reinterpret_cast<float2 *>(&rr->invd[c % kAux][2 * lane]) = make_float2(1.f / dv2.x, 1.f / dv2.y);
                *reinterpret_cast<float2 *>(&rr->dd[c % kAux][2 * lane]) = dd2;
            }
            if (GATED || REV) warp_arrive(&sm->full[s]);
            issued = c + 1;
        }
        if (lane == 0 && aborted(cx)) {
            // Drain: every issued load must land before the CTA may exit.
            for (int c = (issued > NST ? issued - NST : 0); c < issued; ++c)
                mbar_wait(&sm->full[c % NST], (c / NST) & 1, cx.limit);
        }
        // the part's gate product (1 without a gate or chunks)
        if (lane == 0 && slice == 0 && !aborted(cx))
            args.A[orow] = (GATED && issued == nch) ? (cut ? 0.f : expf(off)) : 1.f;
        __syncwarp();
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------ MMA
        // [S | z] += K~'^T [V | 1] per chunk (K~' = diag(weight) K~ with a gate),
        // once phi of the chunk is done.  With 64 value columns one MMA
        // spans the V block and the first 16 columns of the ones block (at LBO);
        // with 128 the two V blocks and the ones block are two MMAs.
        if (lane == 0) {
            constexpr int NV = DVS == 64 ? 80 : DVS;
            constexpr uint32_t idDS = idesc_bf16_f32(128, NV, true, true);
            constexpr uint32_t idDS1 = idesc_bf16_f32(128, 16, true, true);
            constexpr uint32_t kHi128 = desc_hi(1024, 2);
            const uint32_t aOnes = smem_u32(base + L::kOffOnes);
            for (int c = 0; c < nch && !aborted(cx); ++c) {
                const int s = c % NST;
                const uint32_t st = smem_u32(stage_ptr(s));
                const uint32_t onesLo = desc_lo(REV ? st + L::kOffStageCol : aOnes, kBlkV);
                if (!wait(cx, &sm->phi_done[s], (c / NST) & 1)) break;
                tc_fence_after();
                const uint32_t klo = desc_lo(st + L::kOffK, kTileK / 2);   // K~^T: MN-major, two 64-feature blocks
                const uint32_t blo = desc_lo(st + L::kOffV, DVS == 64 ? aOnes - (st + L::kOffV) : kBlkV);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    tc_mma_bf16_w<true>(tmem, klo + kk * (2048 >> 4), kHi128, blo + kk * (2048 >> 4), kHi128, idDS);
                    if (DVS == 128)
                        tc_mma_bf16_w<true>(tmem + DVS, klo + kk * (2048 >> 4), kHi128, onesLo + kk * (2048 >> 4),
                                            kHi128, idDS1);
                }
                tc_commit(&sm->empty[s]);
            }
            tc_commit(&sm->mma_done);
            mbar_wait(&sm->mma_done, 0, cx.limit);
        }
        __syncwarp();
    } else if (warp >= kWarpTm0 && warp < kWarpTm0 + kTmWarps) {
        // ----------------------------------------------------- TMEM warps
        // Warp w holds feature rows 32 (w % 4) .. +31, all DVS columns and z,
        // 32 columns at a time (two resident CTAs per SM leave 85 registers a thread).
        const int qd = warp & 3;
        const uint32_t lane_base = static_cast<uint32_t>(qd * 32) << 16;
        const int srow = qd * 32 + lane;
        // the sub-segment's (dS, dz) once every increment has landed (the gates
        // are in the increments' row weights; the producer writes A)
        if (!aborted(cx)) {
            int ok = 1;
            if (lane == 0) ok = mbar_wait(&sm->mma_done, 0, cx.limit);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            __syncwarp();
            if (ok) {
                tc_fence_after();
                const size_t state_len = (size_t)kR * args.dv + kR;
                float *out = args.dS + orow * state_len;
                float *dst = out + (size_t)srow * args.dv + slice * DVS;
                float sh[32], zz;
                tc_ld_32x32b_x1(tmem + lane_base + DVS, zz);
#pragma unroll 1
                for (int pc = 0; pc < DVS / 32; ++pc) {
                    tc_ld_32x32b_x32(tmem + lane_base + 32 * pc, sh);
                    tc_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; i += 4)
                        *reinterpret_cast<float4 *>(dst + 32 * pc + i) = make_float4(sh[i], sh[i + 1], sh[i + 2], sh[i + 3]);
                }
                if (slice == 0) out[(size_t)kR * args.dv + srow] = zz;
            } else {
                fail(cx);
            }
        }
    } else if (is_phi_warp(warp)) {
        // ------------------------------------------------------ phi warps
        // phi(K) in place, with a gate times the row's decay to the part's end,
        // e^{offset} w_j (REV: to its start, e^{offset} Gamma_j); rows past the end
        // of the sequence become 0.  REV: the rows of V (dy) times 1 / d_t, and
        // dd_t in column 0 of the stage's column block.
        const int pp = phi_index(warp) * 32 + lane;
        for (int c = 0; c < nch; ++c) {
            const int s = c % NST;
            if (!warp_wait(cx, &sm->full[s], (c / NST) & 1)) break;
            const int nvalid = min(kC, T - chunk_t0(c));
            uint4 *kt = reinterpret_cast<uint4 *>(stage_ptr(s) + L::kOffK);
            const float *kw = REV ? gr->gG[c % kAux] : gr->gw[c % kAux];
            const float eoff = GATED ? rr->eoff[c % kAux] : 1.f;
            for (int ci = pp; ci < (int)kTileK / 16; ci += kPhiThreads) {
                const int row = (ci & 511) >> 3;   // 8 chunks per 128-byte row, 64 rows per block
                uint4 v = row < nvalid ? phi8(kt[ci]) : make_uint4(0, 0, 0, 0);
                if (GATED) v = scale8(v, eoff * kw[row]);
                kt[ci] = v;
            }
            if (REV) {
                uint4 *vt = reinterpret_cast<uint4 *>(stage_ptr(s) + L::kOffV);
                const float *invd = rr->invd[c % kAux];
                for (int ci = pp; ci < (int)L::kTileV / 16; ci += kPhiThreads) vt[ci] = scale8(vt[ci], invd[(ci & 511) >> 3]);
                if (pp < kC)
                    *reinterpret_cast<uint16_t *>(stage_ptr(s) + L::kOffStageCol + sw128_offset(pp, 0)) =
                        __bfloat16_as_ushort(__float2bfloat16_rn(rr->dd[c % kAux][pp]));
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
        tmem_dealloc(tmem, L::kTmemCols);
    }
}

// S_start[g] for every output segment g: the state before its first chunk
// (rev: the state entering it from the right).  One thread per 4 consecutive
// elements of a head's state (S then z); a thread issues the loads of up to 8
// parts before it runs their affine maps in order (rev: from the last part).
__global__ void seg_scan_kernel(const float *S0, const float *z0, const float *A, const float *dS, float *S_start,
                                int BH, int dv, int nsub, int sub_per_seg, int nseg, bool rev)
{
    const int bh = blockIdx.y;
    const int e = 4 * (blockIdx.x * blockDim.x + threadIdx.x);
    const int s_len = kR * dv;
    const int state_len = s_len + kR;
    if (e >= state_len) return;
    // S0 and z0 are 4-byte aligned; the workspace parts are 16-byte aligned
    float4 s;
    const float *src0 = e < s_len ? (S0 ? S0 + (size_t)bh * s_len + e : nullptr)
                                  : (z0 ? z0 + (size_t)bh * kR + (e - s_len) : nullptr);
    s = src0 ? make_float4(src0[0], src0[1], src0[2], src0[3]) : make_float4(0.f, 0.f, 0.f, 0.f);
    *reinterpret_cast<float4 *>(S_start + ((size_t)(rev ? nseg - 1 : 0) * BH + bh) * state_len + e) = s;
    for (int i0 = 0; i0 < nsub; i0 += 8) {
        float4 d[8];
        float a[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int m = rev ? nsub - 1 - (i0 + i) : i0 + i;
            d[i] = i0 + i < nsub ? *reinterpret_cast<const float4 *>(dS + ((size_t)m * BH + bh) * state_len + e)
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
            a[i] = i0 + i < nsub ? A[(size_t)m * BH + bh] : 1.f;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (i0 + i >= nsub) break;
            s.x = fmaf(a[i], s.x, d[i].x);
            s.y = fmaf(a[i], s.y, d[i].y);
            s.z = fmaf(a[i], s.z, d[i].z);
            s.w = fmaf(a[i], s.w, d[i].w);
            if (!rev) {
                // part m done: after the last part of segment m / sub_per_seg comes segment + 1
                const int m = i0 + i;
                if ((m + 1) % sub_per_seg == 0) {
                    const int g = (m + 1) / sub_per_seg;
                    if (g < nseg) *reinterpret_cast<float4 *>(S_start + ((size_t)g * BH + bh) * state_len + e) = s;
                }
            } else {
                // part m (of segment m / sub_per_seg + 1) done: at its segment's first part,
                // the state entering the segment before it from the right
                const int m = nsub - 1 - (i0 + i);
                if (m % sub_per_seg == 0) {
                    const int g = m / sub_per_seg;
                    *reinterpret_cast<float4 *>(S_start + ((size_t)g * BH + bh) * state_len + e) = s;
                }
            }
        }
    }
}

// Exclusive prefix sum over the 1024 threads of a block (v >= 0); total in *sum.
__device__ __forceinline__ int block_excl_scan(int v, int *warp_sums, int *sum)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        warp_sums[lane] = w;   // inclusive over warps
        if (lane == 31) *sum = w;
    }
    __syncthreads();
    const int before = (warp ? warp_sums[warp - 1] : 0) + x - v;
    __syncthreads();   // warp_sums and *sum are reused by the next call
    return before;
}

// Sum over a warp, then one shared atomic per warp (1024 threads adding to one
// word one by one would serialise).
__device__ __forceinline__ void block_add(unsigned long long v, unsigned long long *dst)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if ((threadIdx.x & 31) == 0 && v) atomicAdd(dst, v);
}

// Bucket of an item of c chunks in the longest-first order: c itself below 64,
// then 8 buckets per octave; larger items get smaller keys.
constexpr int kOrderBuckets = 64 + 8 * 26;
__device__ __forceinline__ int order_key(int c)
{
    int idx = c;
    if (c >= 64) {
        const int oct = 31 - __clz(c);   // >= 6
        idx = 64 + 8 * (oct - 6) + ((c >> (oct - 3)) & 7);
    }
    return kOrderBuckets - 1 - idx;
}

// Segments of a packed batch.  Sequence b (tokens cu[b] .. cu[b+1]-1, c_b chunks)
// takes ceil(c_b / L) segments of L chunks.  L is the larger of L_min and an SM's
// share of the batch's CTA-chunks (units CTAs per segment on sms SMs), so that
// only a sequence that would hold up the batch is split.  With L >= L_min the
// boundaries of valid disjoint sequences stay within floor(total_T / (64 L_min))
// = max_bds; if any sequence's bounds lie outside [0, total_T] (the chunk kernel
// records it) or the count exceeds max_bds regardless, no sequence is split.
// The boundaries and the start-state slots of the split sequences are numbered
// in sequence order; the items (every segment of every sequence) are written
// longest first, so that the chunk kernel's CTAs start in that order and the
// short ones fill in at the end (within a bucket of order_key, in no set order).
// The state pass has part_rows rows of CTAs: each boundary's segment is cut into
// sub parts (of at least about 4 chunks) so that the boundaries fill part_target
// of them (one wave of state CTAs), or one part each beyond that.
// seg_len receives L, the chunks per part and sub; split_seqs the split
// sequences (in no set order, then -1 up to max_bds).  A valid sequence of at most
// walk_max tokens (-1: none) is left to the token walk: no item, no segment.
constexpr int kPlanCache = 4096;   // chunk counts of the first sequences, in shared memory
__global__ void __launch_bounds__(1024, 1)
varlen_plan_kernel(const int *__restrict__ cu, int B, int total_T, int L_min, int units, int sms, int max_bds,
                   int part_rows, int part_target, int walk_max, int *__restrict__ seg_len, int4 *__restrict__ seq_info, int2 *__restrict__ items,
                   int2 *__restrict__ bds, int *__restrict__ split_seqs)
{
    __shared__ int warp_sums[32];
    __shared__ int tot[2];
    __shared__ unsigned long long acc[2];
    __shared__ int bucket[kOrderBuckets];
    __shared__ int cached[kPlanCache];
    __shared__ int n_split;
    // chunks of sequence b (-1 when its bounds are bad, -2 when the walk takes it)
    auto read_chunks = [&](int b) {
        const int s0 = cu[b], s1 = cu[b + 1];
        if (s0 < 0 || s1 < s0 || s1 > total_T) return -1;
        return s1 - s0 <= walk_max ? -2 : (s1 - s0 + kC - 1) / kC;
    };
    auto code = [&](int b) { return b < kPlanCache ? cached[b] : read_chunks(b); };
    auto chunks = [&](int b) { return max(0, code(b)); };
    if (threadIdx.x == 0) {
        acc[0] = acc[1] = 0;
        n_split = 0;
    }
    for (int i = threadIdx.x; i < kOrderBuckets; i += blockDim.x) bucket[i] = 0;
    __syncthreads();
    // pass 1: the batch's chunks, and whether every sequence is valid
    unsigned long long sum = 0;
    bool bad = false;
    for (int b = threadIdx.x; b < B; b += blockDim.x) {
        const int c = read_chunks(b);
        if (b < kPlanCache) cached[b] = c;
        bad = bad || c == -1;
        sum += max(c, 0);
    }
    block_add(sum, &acc[0]);
    const bool any_bad = __syncthreads_or(bad) != 0;
    const unsigned long long share = (acc[0] * (unsigned long long)units + sms - 1) / (unsigned long long)sms;
    const int L = (int)max((unsigned long long)L_min, min(share, (unsigned long long)0x3fffffff));
    // pass 2: the boundaries this L takes
    unsigned long long count = 0;
    for (int b = threadIdx.x; b < B; b += blockDim.x) {
        const int c = chunks(b);
        count += c > L ? (c + L - 1) / L - 1 : 0;
    }
    block_add(count, &acc[1]);
    __syncthreads();
    const bool split = !any_bad && acc[1] <= (unsigned long long)max_bds;
    const int n_bd = split ? (int)acc[1] : 0;
    // the segments of sequence b (x; 0: the walk's), and the chunks of the last one
    // (y; the others have L)
    auto segments = [&](int b) {
        if (code(b) == -2) return make_int2(0, 0);
        const int c = chunks(b);
        if (!split || c <= L) return make_int2(1, c);
        const int n = (c + L - 1) / L;
        return make_int2(n, c - (n - 1) * L);
    };
    // pass 3: how many items fall in each bucket of the order
    for (int b = threadIdx.x; b < B; b += blockDim.x) {
        const int2 sg = segments(b);
        if (sg.x > 1) atomicAdd(&bucket[order_key(L)], sg.x - 1);
        if (sg.x > 0) atomicAdd(&bucket[order_key(sg.y)], 1);
    }
    __syncthreads();
    // exclusive prefix over the buckets: their first rows in the item table
    {
        const int v = threadIdx.x < kOrderBuckets ? bucket[threadIdx.x] : 0;
        const int first = block_excl_scan(v, warp_sums, &tot[0]);
        if (threadIdx.x < kOrderBuckets) bucket[threadIdx.x] = first;
        __syncthreads();
    }
    const int n_items = tot[0];   // read before the scans below reuse tot
    // pass 4: prefix sums of boundaries and slots, tile by tile, and each item's row
    int carry_bd = 0, carry_slot = 0;
    for (int b0 = 0; b0 < B; b0 += blockDim.x) {
        const int b = b0 + threadIdx.x;
        const int2 sg = b < B ? segments(b) : make_int2(1, 0);
        const int nseg = sg.x, last = sg.y;
        const int nbd = max(0, nseg - 1), nslot = nseg > 1 ? nseg : 0;
        const int bd0 = carry_bd + block_excl_scan(nbd, warp_sums, &tot[0]);
        const int tile_bd = tot[0];
        const int slot0 = carry_slot + block_excl_scan(nslot, warp_sums, &tot[1]);
        const int tile_slot = tot[1];
        if (b < B) {
            seq_info[b] = make_int4(nseg, nseg > 1 ? slot0 : -1, bd0, 0);
            for (int g = 0; g < nseg; ++g)
                items[atomicAdd(&bucket[order_key(g + 1 < nseg ? L : last)], 1)] = make_int2(b, g);
            for (int g = 0; g + 1 < nseg; ++g) bds[bd0 + g] = make_int2(b, g);
            if (nseg > 1) split_seqs[atomicAdd(&n_split, 1)] = b;
        }
        carry_bd += tile_bd;
        carry_slot += tile_slot;
        __syncthreads();   // tot is rewritten by the next tile
    }
    // the parts of a boundary's segment: as many as the rows allow, of >= ~4 chunks
    if (threadIdx.x == 0) {
        int sub = n_bd ? min(part_rows, part_target) / n_bd : 1;
        sub = max(1, min(sub, (L + 3) / 4));
        const int sub_chunks = (L + sub - 1) / sub;
        seg_len[0] = L;
        seg_len[1] = sub_chunks;
        seg_len[2] = (L + sub_chunks - 1) / sub_chunks;
    }
    // pass 5: the rows past the plan's items, boundaries and split sequences do nothing
    for (int i = n_items + threadIdx.x; i < B + max_bds; i += blockDim.x) items[i] = make_int2(-1, 0);
    for (int k = carry_bd + threadIdx.x; k < part_rows; k += blockDim.x) bds[k] = make_int2(-1, 0);
    for (int i = n_split + threadIdx.x; i < max_bds; i += blockDim.x) split_seqs[i] = -1;
}

// The start state of every segment of every split sequence: slot 0 holds S0, z0;
// slot g the state after the maps of the parts that end at boundary first + g - 1
// (S -> A S + dS, in order; sub parts per boundary).  A block takes one head of
// one split sequence and 512 consecutive float4 of its state; each thread holds
// 2 of them and has the loads of 8 parts in flight at a time.
constexpr int kScanVec = 2, kScanParts = 8;
__global__ void __launch_bounds__(256)
varlen_scan_kernel(const float *S0, const float *z0, const float *__restrict__ A, const float *__restrict__ dS,
                   float *__restrict__ S_start,
                   const int4 *__restrict__ seq_info, const int *__restrict__ split_seqs,
                   const int *__restrict__ seg_len, int H, int dv)
{
    const int b = split_seqs[blockIdx.x / H], h = blockIdx.x % H;
    if (b < 0) return;
    const int4 si = seq_info[b];
    const int sub = seg_len[2];
    const int bh = b * H + h;
    const int s_len = kR * dv;
    const int state_len = s_len + kR;
    int e[kScanVec];
    float4 s[kScanVec];
#pragma unroll
    for (int q = 0; q < kScanVec; ++q) {
        e[q] = 4 * ((blockIdx.y * kScanVec + q) * blockDim.x + threadIdx.x);
        s[q] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (e[q] < state_len) {
            // S0 and z0 are 4-byte aligned; the workspace parts are 16-byte aligned
            const float *src0 = e[q] < s_len ? (S0 ? S0 + (size_t)bh * s_len + e[q] : nullptr)
                                             : (z0 ? z0 + (size_t)bh * kR + (e[q] - s_len) : nullptr);
            if (src0) s[q] = make_float4(src0[0], src0[1], src0[2], src0[3]);
            *reinterpret_cast<float4 *>(S_start + ((size_t)si.y * H + h) * state_len + e[q]) = s[q];
        }
    }
    const int nparts = (si.x - 1) * sub;
    const size_t part0 = (size_t)si.z * sub;
    for (int p0 = 0; p0 < nparts; p0 += kScanParts) {
        float4 d[kScanParts][kScanVec];
        float a[kScanParts];
#pragma unroll
        for (int i = 0; i < kScanParts; ++i) {
            const size_t row = (part0 + p0 + i) * H + h;
            const bool ok = p0 + i < nparts;
            a[i] = ok ? A[row] : 1.f;
#pragma unroll
            for (int q = 0; q < kScanVec; ++q)
                d[i][q] = (ok && e[q] < state_len) ? *reinterpret_cast<const float4 *>(dS + row * state_len + e[q])
                                                   : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int i = 0; i < kScanParts; ++i) {
            if (p0 + i >= nparts) break;
#pragma unroll
            for (int q = 0; q < kScanVec; ++q) {
                s[q].x = fmaf(a[i], s[q].x, d[i][q].x);
                s[q].y = fmaf(a[i], s[q].y, d[i][q].y);
                s[q].z = fmaf(a[i], s[q].z, d[i][q].z);
                s[q].w = fmaf(a[i], s[q].w, d[i][q].w);
            }
            if ((p0 + i + 1) % sub == 0) {
                const int g = (p0 + i + 1) / sub;
#pragma unroll
                for (int q = 0; q < kScanVec; ++q)
                    if (e[q] < state_len)
                        *reinterpret_cast<float4 *>(S_start + ((size_t)(si.y + g) * H + h) * state_len + e[q]) = s[q];
            }
        }
    }
}

}  // namespace

cudaError_t launch_varlen_plan(const int *cu_seqlens, int B, int total_T, int min_seg_chunks, int units, int sms,
                               int max_bds, int part_rows, int part_target, int walk_max, int *seg_len,
                               int4 *seq_info, int2 *items, int2 *bds, int *split_seqs, cudaStream_t stream)
{
    if (B < 1 || min_seg_chunks < 1 || units < 1 || sms < 1 || max_bds < 0 || total_T < 0 || part_rows < max_bds ||
        (max_bds > 0 && part_target < 1) || walk_max < -1)
        return cudaErrorInvalidValue;
    varlen_plan_kernel<<<1, 1024, 0, stream>>>(cu_seqlens, B, total_T, min_seg_chunks, units, sms, max_bds,
                                                part_rows, part_target, walk_max, seg_len, seq_info, items, bds,
                                                split_seqs);
    return cudaGetLastError();
}

cudaError_t launch_varlen_scan(const float *S0, const float *z0, const float *A, const float *dS, float *S_start,
                               const int4 *seq_info, const int *split_seqs, const int *seg_len, int max_bds, int H,
                               int dv, cudaStream_t stream)
{
    if (max_bds < 1 || H < 1 || (long long)max_bds * H > 0x7fffffffLL) return cudaErrorInvalidValue;
    const int n4 = (kR * dv + kR) / 4;
    const dim3 grid(max_bds * H, (n4 + 256 * kScanVec - 1) / (256 * kScanVec));
    varlen_scan_kernel<<<grid, 256, 0, stream>>>(S0, z0, A, dS, S_start, seq_info, split_seqs, seg_len, H, dv);
    return cudaGetLastError();
}

cudaError_t launch_state_tc(const CUtensorMap &map_k, const CUtensorMap &map_v, const StateTcArgs &a, int B,
                            bool gated, int dvs, cudaStream_t stream, bool rev, int grid_z)
{
    if ((dvs != 64 && dvs != 128) || (rev && (dvs != 128 || !a.d || !a.dd))) return cudaErrorInvalidValue;
    if (a.bds && (rev || grid_z < 1 || !a.cu_seqlens || !a.seg_len)) return cudaErrorInvalidValue;
    const dim3 grid(a.dv / dvs, a.H, a.bds ? grid_z : B * a.nsub);
    using KernFn = void (*)(const CUtensorMap, const CUtensorMap, const StateTcArgs);
    const int v = rev ? 4 + (gated ? 1 : 0) : (gated ? 1 : 0) + (dvs == 128 ? 2 : 0);
    static const KernFn kerns[6] = {state_tc_kernel<false, 64, false>,  state_tc_kernel<true, 64, false>,
                                    state_tc_kernel<false, 128, false>, state_tc_kernel<true, 128, false>,
                                    state_tc_kernel<false, 128, true>,  state_tc_kernel<true, 128, true>};
    static const uint32_t bytes[6] = {smem_bytes<false, 64>(),        smem_bytes<true, 64>(),
                                      smem_bytes<false, 128>(),       smem_bytes<true, 128>(),
                                      smem_bytes<false, 128, true>(), smem_bytes<true, 128, true>()};
    static OncePerDevice attr_set[6];
    const cudaError_t e = set_smem_once(kerns[v], bytes[v], attr_set[v]);
    if (e != cudaSuccess) return e;
    kerns[v]<<<grid, kThreads, bytes[v], stream>>>(map_k, map_v, a);
    return cudaGetLastError();
}

cudaError_t launch_seg_scan(const float *S0, const float *z0, const float *A, const float *dS, float *S_start,
                            int BH, int dv, int nsub, int sub_per_seg, int nseg, cudaStream_t stream, bool rev)
{
    const int state_len = kR * dv + kR;
    const dim3 grid((state_len / 4 + 255) / 256, BH);
    seg_scan_kernel<<<grid, 256, 0, stream>>>(S0, z0, A, dS, S_start, BH, dv, nsub, sub_per_seg, nseg, rev);
    return cudaGetLastError();
}

}  // namespace la
