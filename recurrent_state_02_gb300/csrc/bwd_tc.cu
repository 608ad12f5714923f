// bwd_tc.cu -- the three gradient sweeps of the gated linear-attention recurrence
// on the sm_103a tensor cores (BF16 operands, FP32 accumulators and state in TMEM).
//
// The pages give no backward; the gradients follow from the recurrence of
// "Linear attention：把历史写进状态" (hs-black.github.io/posts/linear-attention),
// sections "公式里的每个维度" and "加一个门：让旧记忆逐渐淡出", by the chain rule.  With
// q~ = phi(q), k~ = phi(k), d_t = q~_t . z_t + eps, dn_t = dy_t / d_t,
// dd_t = -(dy_t . y_t) / d_t and the decay D(s, t) = alpha_{s+1} ... alpha_t:
//     dq~_t = sum_{s<=t} D(s,t) k~_s (v_s . dn_t + dd_t) + D0(t) (S0 dn_t + dd_t z0)
//     dk~_s = sum_{t>=s} D(s,t) q~_t (v_s . dn_t + dd_t) + D(s,T) (dS_T v_s + dz_T)
//     dv_s  = sum_{t>=s} D(s,t) dn_t (k~_s . q~_t)        + D(s,T) dS_T^T k~_s
// Each is an unnormalised causal linear attention with the operands' roles
// permuted, the last two in reversed time, so each runs as the chunk form of the
// prefill (section "一个 chunk 的输出由两部分组成"): per chunk of 64 tokens the read
// of the carried state plus the masked in-chunk product, then the state hand-off.
//
//   mode  time     query  key   value  state (TMEM, FP32)         read operand
//   dq    forward  dn     v     k~     [S | z] = sum k~ [v | 1]^T  [S_prev] as K-major B
//   dk    reverse  v      dn    q~     [G | g] = sum q~ [dn | dd]^T [G_prev] as K-major B
//   dv    reverse  k~     q~    dn     G = sum q~ dn^T             [G_prev] as MN-major B
//
// The columns of 1 and dd enter as rank-1 terms, so every product keeps K = 128:
// the TMEM warps add dd_t to the scores (per row for dq, per column for dk); the
// read of the state's z (dq) or g (dk) column is a fifth K step of the in-chunk
// product, [c_t] [z_hi; z_lo] with c_t = dd_t Gamma_t (dq) or w_s (dk); and the
// state product adds a block whose column 0 holds 1 (dq) or dd_t (dk).
//
// Gates (the explicit form: products scaled per row after the scores).  b_i is
// the in-chunk cumulative log gate, Gamma_i = e^{b_i}, w_i = e^{b_last - b_i}.  In
// forward time row i reads the carried state with weight Gamma_i and key j enters
// the next state with weight w_j; in reversed time row s reads it with weight w_s
// (the decay from s to the chunk's end) and token t enters with Gamma_t (the
// decay back to the chunk's start, including its own gate).  In both directions
// the state is first decayed by Gamma_last, and the in-chunk score of a later
// token t and an earlier token s carries e^{b_t - b_s}; a gate of exactly 0 cuts
// every product across it.
//
// Outputs: dq = phi'(q) dq~ and dk = phi'(k) dk~ (q, k read again in the
// epilogue), dv; the per-token terms q~ . dq~ (+) and k~ . dk~ (-) of dlog alpha;
// <dS_T, S_T> + <dz_T, z_T> (dq's final state) and dS0, dz0 (dk's final state).
// Every barrier wait is bounded; on expiry the kernel records a timeout in the
// device status word, drains its own copies and MMAs, frees TMEM and returns.

#include "tc_common.cuh"

namespace la {
namespace {

constexpr int kModeDq = 0, kModeDk = 1, kModeDv = 2;

constexpr int kThreads = 768;   // 24 warps, the roles of the prefill kernel
constexpr int kWarpTma = 0, kWarpMma = 1, kWarpMmaP = 22, kWarpMmaS = 23, kWarpTm0 = 4, kTmWarps = 16;
constexpr uint32_t kPrepMask = 0x30000Cu;   // warps 2, 3, 20, 21: one per scheduler
constexpr int kPrepWarps = 4, kPrepThreads = kPrepWarps * 32;
__host__ __device__ constexpr bool is_prep_warp(int w) { return (kPrepMask >> w) & 1u; }
__host__ __device__ constexpr int prep_index(int w) { return __builtin_popcount(kPrepMask & ((1u << w) - 1u)); }

constexpr int kStages = 3;
constexpr uint32_t kTile = kC * 128 * 2;       // 16 KB: 64 token rows x 128 columns, two 64-column blocks
constexpr uint32_t kBlk = kTile / 2;           // 8 KB block (128-byte rows, 128-byte swizzle)
constexpr uint32_t kTileA = kC * kC * 2;       // 8 KB
constexpr uint32_t kBlkSp = kR * 32;           // 4 KB: 16 columns of the 128-row state operand (32-byte swizzle)
constexpr uint32_t kTileSp = 8 * kBlkSp;       // 32 KB
constexpr uint32_t kBlkW = kC * 32;            // 2 KB: 64 token rows x 16 columns, 32-byte swizzle
constexpr uint32_t kBlkZ = 16 * 128 * 2;       // 4 KB: 16 rows x 128 columns (two 64-column halves), 128-byte swizzle

// Per-chunk scalars beside the gate products.
struct alignas(16) BwdRing {
    GateRing g;                 // gated only
    float invd[kAux][kC];       // 1 / d_t (1 for rows past T)
    float dd[kAux][kC];         // dd_t (0 for rows past T)
};

template <int MODE>
struct BCfg {
    static constexpr bool kRev = MODE != kModeDq;
    static constexpr bool kWblk = MODE != kModeDv;      // the block of 1 / dd_t after the key tile
    static constexpr bool kSpK = MODE != kModeDv;       // the read operand is K-major
    static constexpr int kHW = kWblk ? 144 : 128;       // state columns (z or g in column 128)
    // stage: query, key and value tiles, then the column block of the state product
    static constexpr uint32_t kOffQry = 0, kOffKey = kTile, kOffVal = 2 * kTile, kOffWblk = 3 * kTile;
    static constexpr uint32_t kStageBytes = 3 * kTile + (kWblk ? kBlkW : 0);
    static_assert(kStageBytes % 1024 == 0, "stage tiles stay 1024-byte aligned");
    // per A buffer (x2): the 64 x 64 A tile, and (dq, dk) the fifth K step of the
    // in-chunk product: Z = [z_hi; z_lo; 0..] (16 x 128) and W5 = [c_t, c_t, 0..] (64 x 16)
    static constexpr uint32_t kOffA = kStages * kStageBytes;
    static constexpr uint32_t kOffZ = kOffA + 2 * kTileA;
    static constexpr uint32_t kOffW5 = kOffZ + (kWblk ? 2 * kBlkZ : 0);
    static constexpr uint32_t kOffSp = kOffW5 + (kWblk ? 2 * kBlkW : 0);
    static constexpr uint32_t kOffRing = kOffSp + kTileSp;
    static constexpr uint32_t kOffSmall = kOffRing + sizeof(BwdRing);
    // TMEM: P (64), the state (kHW), [O] x 2 (128 each)
    static constexpr uint32_t kColP = 0, kColH = 64, kColO = kColH + kHW;
    static_assert(kColO + 2 * 128 <= 512, "TMEM budget");
};

struct alignas(16) BSmall {
    uint64_t full[kStages], empty[kStages], prep_done[kStages], sc_done[kStages];
    uint64_t P_full, H_full, tm_read[2], ops_full[2], Sp_empty, A_empty[2], O_full[2], O_empty[2], aux_empty[kAux];
    uint64_t mma_done[3];
    uint32_t tmem_base;
    int abort_flag;
    float red[2];
};

template <int MODE>
constexpr uint32_t smem_bytes() { return BCfg<MODE>::kOffSmall + sizeof(BSmall) + 1024; }
static_assert(smem_bytes<kModeDq>() <= 232448 && smem_bytes<kModeDk>() <= 232448 && smem_bytes<kModeDv>() <= 232448,
              "shared memory budget");

// One sweep (MODE) of one head (blockIdx.y, blockIdx.z), or of segment blockIdx.x of it.
template <int MODE, bool GATED>
__device__ __forceinline__ void
bwd_sweep(const CUtensorMap &map_q, const CUtensorMap &map_k, const CUtensorMap &map_v, const CUtensorMap &map_dy,
          const BwdTcArgs &args)
{
    using L = BCfg<MODE>;
    constexpr bool REV = L::kRev;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    BSmall *sm = reinterpret_cast<BSmall *>(base + L::kOffSmall);
    BwdRing *ring = reinterpret_cast<BwdRing *>(base + L::kOffRing);
    GateRing *gr = &ring->g;
    Ctx cx{&sm->abort_flag, args.limit_ns, args.status};

    const int h = blockIdx.y, b = blockIdx.z;
    const int bh = b * args.H + h;
    const int T = args.T;
    // this CTA's chunks: segment blockIdx.x of the head's sequence (all of it when nseg == 1)
    const int seg = blockIdx.x, nseg = gridDim.x;
    const int nch_all = (T + kC - 1) / kC;
    const int c_begin = nseg > 1 ? seg * args.seg_chunks : 0;
    const int c_end = nseg > 1 ? min(nch_all, c_begin + args.seg_chunks) : nch_all;
    const int nch = max(0, c_end - c_begin);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // chunk of iteration c (reversed time walks the chunks from the end)
    auto chunk_of = [&](int c) { return REV ? c_end - 1 - c : c_begin + c; };
    auto stage_ptr = [&](int s) { return base + s * L::kStageBytes; };
    // the tensor maps of the query, key and value tiles
    const CUtensorMap *mq = MODE == kModeDq ? &map_dy : MODE == kModeDk ? &map_v : &map_k;
    const CUtensorMap *mk = MODE == kModeDq ? &map_v : MODE == kModeDk ? &map_dy : &map_q;
    const CUtensorMap *mv = MODE == kModeDq ? &map_k : MODE == kModeDk ? &map_q : &map_dy;

    // ------------------------------------------------------------ set-up
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm->full[s], 2);               // TMA bytes + the producer's scalars
            mbar_init(&sm->empty[s], 3);              // one commit from each MMA issuer
            mbar_init(&sm->prep_done[s], kPrepWarps);
            mbar_init(&sm->sc_done[s], kPrepWarps);
        }
        mbar_init(&sm->P_full, 1);
        mbar_init(&sm->H_full, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm->tm_read[i], kTmWarps);
            mbar_init(&sm->ops_full[i], kTmWarps);
            mbar_init(&sm->A_empty[i], 1);
            mbar_init(&sm->O_full[i], 1);
            mbar_init(&sm->O_empty[i], kTmWarps);
        }
        mbar_init(&sm->Sp_empty, 1);
        for (int i = 0; i < kAux; ++i) mbar_init(&sm->aux_empty[i], kTmWarps);
        for (int i = 0; i < 3; ++i) mbar_init(&sm->mma_done[i], 1);
        sm->abort_flag = 0;
        sm->red[0] = sm->red[1] = 0.f;
        fence_mbarrier_init();
        tma_prefetch_desc(mq);
        tma_prefetch_desc(mk);
        tma_prefetch_desc(mv);
    }
    // A: the blocks above (dq) or below (dk, dv) the diagonal stay 0; the column
    // blocks: zero, column 0 = 1 (dq; gated chunks overwrite it with w_j)
    for (int i = threadIdx.x; i < (int)(2 * kTileA / 16); i += kThreads)
        reinterpret_cast<uint4 *>(base + L::kOffA)[i] = make_uint4(0, 0, 0, 0);
    if (L::kWblk) {
        for (int i = threadIdx.x; i < kStages * (int)(kBlkW / 16); i += kThreads)
            reinterpret_cast<uint4 *>(stage_ptr(i / (kBlkW / 16)) + L::kOffWblk)[i % (kBlkW / 16)] = make_uint4(0, 0, 0, 0);
        for (int i = threadIdx.x; i < (int)((2 * kBlkZ + 2 * kBlkW) / 16); i += kThreads)
            reinterpret_cast<uint4 *>(base + L::kOffZ)[i] = make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
    if (MODE == kModeDq && threadIdx.x < kStages * kC)
        *reinterpret_cast<uint16_t *>(stage_ptr(threadIdx.x / kC) + L::kOffWblk + sw32_offset(threadIdx.x % kC, 0)) =
            0x3F80u;
    fence_proxy_async_smem();
    if (warp == kWarpMma) {
        tmem_alloc(&sm->tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm->tmem_base;

    if (warp == kWarpTma) {
        // ------------------------------------------------------- producer
        // Lane 0 loads the three tiles of a stage; the warp then forms the chunk's
        // gate products and scalars (1 / d_t, dd_t) and makes the stage's second
        // arrival.
        int issued = 0;
        for (int c = 0; c < nch; ++c) {
            const int s = c % kStages;
            const int t0 = chunk_of(c) * kC;
            float a0 = 1.f, a1 = 1.f, d0 = 1.f, d1 = 1.f, e0 = 0.f, e1 = 0.f;
            const int ta = t0 + 2 * lane, tb = ta + 1;
            if (ta < T) {
                if (GATED) a0 = args.alpha[(size_t)bh * T + ta];
                d0 = args.d[(size_t)bh * T + ta];
                e0 = args.dd[(size_t)bh * T + ta];
            }
            if (tb < T) {
                if (GATED) a1 = args.alpha[(size_t)bh * T + tb];
                d1 = args.d[(size_t)bh * T + tb];
                e1 = args.dd[(size_t)bh * T + tb];
            }
            if (c >= kStages && !warp_wait(cx, &sm->empty[s], ((c / kStages) - 1) & 1)) break;
            if (c >= kAux && !warp_wait(cx, &sm->aux_empty[c % kAux], ((c / kAux) - 1) & 1)) break;
            if (__shfl_sync(0xffffffffu, aborted(cx) ? 1 : 0, 0)) break;
            uint8_t *st = stage_ptr(s);
            if (lane == 0) {
                mbar_arrive_expect_tx(&sm->full[s], 3 * kTile);
                const uint32_t offs[3] = {L::kOffQry, L::kOffKey, L::kOffVal};
                const CUtensorMap *maps[3] = {mq, mk, mv};
#pragma unroll
                for (int m = 0; m < 3; ++m) {
                    tma_load_3d(st + offs[m], maps[m], &sm->full[s], 0, t0, bh);
                    tma_load_3d(st + offs[m] + kBlk, maps[m], &sm->full[s], 64, t0, bh);
                }
            }
            const int gq = c % kAux;
            *reinterpret_cast<float2 *>(&ring->invd[gq][2 * lane]) = make_float2(1.f / d0, 1.f / d1);
            *reinterpret_cast<float2 *>(&ring->dd[gq][2 * lane]) = make_float2(e0, e1);
            if (GATED) gate_products(a0, a1, lane, gq, gr);
            warp_arrive(&sm->full[s]);
            issued = c + 1;
        }
        if (lane == 0 && aborted(cx)) {
            for (int c = (issued > kStages ? issued - kStages : 0); c < issued; ++c)
                mbar_wait(&sm->full[c % kStages], (c / kStages) & 1, cx.limit);
        }
        __syncwarp();
    } else if (warp == kWarpMma || warp == kWarpMmaS || warp == kWarpMmaP) {
        // ------------------------------------------------------------ MMA
        if (lane == 0) {
            constexpr uint32_t idP = idesc_bf16_f32(64, 64, false, false);
            constexpr uint32_t idH = idesc_bf16_f32(128, 128, true, true);
            constexpr uint32_t idH1 = idesc_bf16_f32(128, 16, true, true);
            constexpr uint32_t idRd = idesc_bf16_f32(64, 128, false, !L::kSpK);
            constexpr uint32_t idAV = idesc_bf16_f32(64, 128, false, true);
            constexpr uint32_t kHi128 = desc_hi(1024, 2), kHi32 = desc_hi(256, 6);
            constexpr uint32_t kHi128Z = desc_hi(1024, 2);   // Z: 8-row atoms 1 KB apart along K
            // K-major 64-row tile, K step kk of 16 columns: block kk / 4, 32 bytes a step inside it
            auto kstep = [](int kk) -> uint32_t { return (((kk >> 2) * kBlk) + (kk & 3) * 32) >> 4; };
            bool ok = true;
            if (warp == kWarpMmaP) {
                // P = Q K^T for chunk c, once the prep warps are done with chunk c and
                // the TMEM warps have read P of chunk c - 1
                for (int c = 0; c < nch && ok && !aborted(cx); ++c) {
                    const int s = c % kStages;
                    const uint32_t st = smem_u32(stage_ptr(s));
                    if (!wait(cx, &sm->prep_done[s], (c / kStages) & 1)) { ok = false; break; }
                    if (c >= 1 && !wait(cx, &sm->tm_read[(c - 1) & 1], ((c - 1) >> 1) & 1)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t qlo = desc_lo(st + L::kOffQry, 16), klo = desc_lo(st + L::kOffKey, 16);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        if (kk == 0) tc_mma_bf16_w<false>(tmem + L::kColP, qlo, kHi128, klo, kHi128, idP);
                        else tc_mma_bf16_w<true>(tmem + L::kColP, qlo + kstep(kk), kHi128, klo + kstep(kk), kHi128, idP);
                    }
                    tc_commit(&sm->P_full);
                    tc_commit(&sm->empty[s]);
                }
            } else if (warp == kWarpMmaS) {
                // state += SA^T SB for chunk c, once its operands are scaled and the
                // TMEM warps have read (and decayed) the state
                for (int c = 0; c < nch && ok && !aborted(cx); ++c) {
                    const int s = c % kStages;
                    const uint32_t st = smem_u32(stage_ptr(s));
                    if (!wait(cx, GATED ? &sm->sc_done[s] : &sm->prep_done[s], (c / kStages) & 1)) { ok = false; break; }
                    if (!wait(cx, &sm->tm_read[c & 1], (c >> 1) & 1)) { ok = false; break; }
                    tc_fence_after();
                    // dq, dk: SA = value tile, SB = [key | column block]; dv: SA = key, SB = value
                    const uint32_t aSA = st + (MODE == kModeDv ? L::kOffKey : L::kOffVal);
                    const uint32_t aSB = st + (MODE == kModeDv ? L::kOffVal : L::kOffKey);
                    const uint32_t alo = desc_lo(aSA, kBlk), blo = desc_lo(aSB, kBlk);
                    const uint32_t wlo = desc_lo(st + L::kOffWblk, kBlkW);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        tc_mma_bf16_w<true>(tmem + L::kColH, alo + kk * (2048 >> 4), kHi128, blo + kk * (2048 >> 4), kHi128,
                                            idH);
                        // the column block: 16 token rows of 32 bytes a K step
                        if (L::kWblk)
                            tc_mma_bf16_w<true>(tmem + L::kColH + 128, alo + kk * (2048 >> 4), kHi128,
                                                wlo + kk * (512 >> 4), kHi32, idH1);
                    }
                    tc_commit(&sm->H_full);
                    tc_commit(&sm->empty[s]);
                }
            } else {
                // [O] = Q' S_prev + A V for chunk c, into the buffer of chunk c - 2
                for (int c = 0; c < nch && ok && !aborted(cx); ++c) {
                    const int s = c % kStages, bb = c & 1, n = c >> 1;
                    const uint32_t st = smem_u32(stage_ptr(s));
                    if (GATED && !wait(cx, &sm->sc_done[s], (c / kStages) & 1)) break;
                    if (!wait(cx, &sm->ops_full[bb], n & 1)) break;
                    if (c >= 2 && !wait(cx, &sm->O_empty[bb], ((c >> 1) - 1) & 1)) break;
                    tc_fence_after();
                    const uint32_t dO = tmem + L::kColO + bb * 128;
                    const uint32_t qlo = desc_lo(st + L::kOffQry, 16);
                    const uint32_t sp = smem_u32(base + L::kOffSp);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        // K-major read operand: block kk holds columns 16 kk .. +15 of all
                        // 128 rows; MN-major: rows 16 kk .. +15 of every block (LBO apart)
                        const uint32_t blo = L::kSpK ? desc_lo(sp + kk * kBlkSp, kBlkSp) : desc_lo(sp + kk * 512, kBlkSp);
                        if (kk == 0) tc_mma_bf16_w<false>(dO, qlo, kHi128, blo, kHi32, idRd);
                        else tc_mma_bf16_w<true>(dO, qlo + kstep(kk), kHi128, blo, kHi32, idRd);
                    }
                    tc_commit(&sm->Sp_empty);
                    const uint32_t alo = desc_lo(smem_u32(base + L::kOffA + bb * kTileA), 16);
                    const uint32_t vlo = desc_lo(st + L::kOffVal, kBlk);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc_mma_bf16_w<true>(dO, alo + kk * (32 >> 4), kHi128, vlo + kk * (2048 >> 4), kHi128, idAV);
                    if (L::kWblk) {
                        // the read of the state's z (dq) or g (dk) column: [c_t c_t 0..] [z_hi; z_lo; 0..]
                        const uint32_t w5 = desc_lo(smem_u32(base + L::kOffW5 + bb * kBlkW), kBlkW);
                        const uint32_t z5 = desc_lo(smem_u32(base + L::kOffZ + bb * kBlkZ), kBlkZ / 2);
                        tc_mma_bf16_w<true>(dO, w5, kHi32, z5, kHi128Z, idAV);
                    }
                    tc_commit(&sm->A_empty[bb]);
                    tc_commit(&sm->O_full[bb]);
                    tc_commit(&sm->empty[s]);
                }
            }
            uint64_t *done = &sm->mma_done[warp == kWarpMma ? 0 : warp == kWarpMmaP ? 1 : 2];
            tc_commit(done);
            mbar_wait(done, 0, cx.limit);
        }
        __syncwarp();
    } else if (warp >= kWarpTm0 && warp < kWarpTm0 + kTmWarps) {
        // ----------------------------------------------------- TMEM warps
        // Iteration c reads the state after chunk c-1 (the read operand of chunk c;
        // with a gate it is then decayed in place by Gamma_last of chunk c), turns
        // the scores of chunk c into A, and finishes the outputs of chunk c-1.
        const int tw = warp - kWarpTm0;
        const int qd = warp & 3, qq = tw >> 2;
        const uint32_t lane_base = static_cast<uint32_t>(qd * 32) << 16;
        const int srow = qd * 32 + lane;                        // state row (feature)
        const int prow = qd * 16 + (lane & 15);                 // row of the M = 64 tiles
        const int pcol = qq * 16 + (lane >> 4) * 8;             // first of 8 columns of P and A
        const int ocol = qq * 32 + (lane >> 4) * 16;            // first of 16 columns of O
        // pieces of A that are always zero: above the diagonal (forward) or below it (reversed)
        const bool a_zero = REV ? qq < qd : qq > qd;
        const uint32_t tH = tmem + lane_base + L::kColH + qq * 32;
        const uint32_t tz = tmem + lane_base + L::kColH + 128;    // z or g (dq, dk)
        {
            // initial state: [S0 | z0] (dq), [dS_T | dz_T] (dk), dS_T (dv), or zero; with
            // segments, the state entering the segment (from the left for dq, from the
            // right for dk and dv), which the state passes wrote [S (128 x 128) | z]
            const float *S_init = MODE == kModeDq ? args.S0 : args.dS_T;
            const float *z_init = MODE == kModeDq ? args.z0 : args.dz_T;
            if (S_init) S_init += (size_t)bh * kR * 128;
            if (z_init) z_init += (size_t)bh * kR;
            if (nseg > 1) {
                const size_t state_len = (size_t)kR * 128 + kR;
                const int BH = gridDim.z * args.H;
                S_init = (MODE == kModeDq ? args.seg_state_f : args.seg_state_r) + ((size_t)seg * BH + bh) * state_len;
                z_init = S_init + (size_t)kR * 128;
            }
            float S[32];
            const float *src = S_init ? S_init + (size_t)srow * 128 + qq * 32 : nullptr;
#pragma unroll
            for (int j = 0; j < 32; ++j) S[j] = src ? src[j] : 0.f;
            tc_st_32x32b_x32(tH, S);
            if (L::kWblk && qq == 0) tc_st_32x32b_x1(tz, z_init ? z_init[srow] : 0.f);
            tc_wait_st();
        }
        float fin_acc = 0.f;
        for (int c = 0; c < nch + 1; ++c) {
            const bool has_b = c < nch;
            const bool has_p = has_b && !a_zero;
            const bool has_e = c >= 1;
            const int bb = c & 1, gq = c % kAux;
            if (c >= 1 && !warp_wait(cx, &sm->H_full, (c - 1) & 1)) break;
            if (has_b && !warp_wait(cx, &sm->prep_done[c % kStages], (c / kStages) & 1)) break;   // scalars of chunk c
            if (has_p && !warp_wait(cx, &sm->P_full, c & 1)) break;
            tc_fence_after();
            float S[32], zr = 0.f, p[8];
            tc_ld_32x32b_x32(tH, S);
            if (L::kWblk && qq == 0) tc_ld_32x32b_x1(tz, zr);
            if (has_p) tc_ld_16x32bx2_x8<8>(tmem + lane_base + L::kColP + qq * 16, p);
            tc_wait_ld();
            uint32_t spk[16];
            if (has_b) {
#pragma unroll
                for (int j = 0; j < 16; ++j) spk[j] = pack_bf16x2(S[2 * j], S[2 * j + 1]);
            }
            if (GATED && has_b) {
                const float g = gr->gG[gq][kC - 1];
#pragma unroll
                for (int j = 0; j < 32; ++j) S[j] *= g;
                tc_st_32x32b_x32(tH, S);
                if (L::kWblk && qq == 0) tc_st_32x32b_x1(tz, g * zr);
                tc_wait_st();
            }
            tc_fence_before();
            if (has_b) warp_arrive(&sm->tm_read[bb]);

            if (has_b) {
                // A: the causal mask (dq: j <= i; dk, dv: t >= s), the rank-1 dd term
                // (dq: + dd_i of the row; dk: + dd_t of the column) and, with a gate,
                // the in-chunk decay e^{b_later - b_earlier} cut at zero gates
                if (has_p) {
                    const float ddr = MODE == kModeDq ? ring->dd[gq][prow] : 0.f;
                    const int zr_i = GATED ? gr->gz[gq][prow] : -1;
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int j = pcol + e;
                        const bool in = REV ? j >= prow : j <= prow;
                        float a = p[e] + (MODE == kModeDq ? ddr : MODE == kModeDk ? ring->dd[gq][j] : 0.f);
                        if (GATED) {
                            // later token L, earlier token E
                            const int Lt = REV ? j : prow, Et = REV ? prow : j;
                            const bool cut = (REV ? gr->gz[gq][j] : zr_i) > Et;
                            a = (in && !cut) ? a * __expf(gr->gb[gq][Lt] - gr->gb[gq][Et]) : 0.f;
                        } else {
                            a = in ? a : 0.f;
                        }
                        p[e] = a;
                    }
                }
                if (c >= 2 && !warp_wait(cx, &sm->A_empty[bb], ((c >> 1) - 1) & 1)) break;
                if (has_p)
                    *reinterpret_cast<uint4 *>(base + L::kOffA + bb * kTileA + sw128_offset(prow, pcol >> 3)) =
                        make_uint4(pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3]), pack_bf16x2(p[4], p[5]),
                                   pack_bf16x2(p[6], p[7]));
                if (L::kWblk && qq == 0) {
                    // the fifth K step of the in-chunk product: row i of W5 = [c_i, c_i, 0..]
                    // (dq: c = dd Gamma, dk: c = w) and Z = [z_hi; z_lo] of the state read
                    if (lane < 16) {
                        const float cw = MODE == kModeDq ? ring->dd[gq][prow] * (GATED ? gr->gG[gq][prow] : 1.f)
                                                         : (GATED ? gr->gw[gq][prow] : 1.f);
                        *reinterpret_cast<uint32_t *>(base + L::kOffW5 + bb * kBlkW + sw32_offset(prow, 0)) =
                            pack_bf16x2(cw, cw);
                    }
                    const float zhi = __bfloat162float(__float2bfloat16_rn(zr));
                    // element (row k, column f) of Z: half f / 64, 8-row atom k / 8, 128-byte row k % 8
                    uint8_t *zb = base + L::kOffZ + bb * kBlkZ + (srow >> 6) * (kBlkZ / 2);
                    const int fc = srow & 63;
                    *reinterpret_cast<uint16_t *>(zb + 0 * 128 + ((((fc >> 3) ^ 0) << 4) | ((fc & 7) * 2))) =
                        __bfloat16_as_ushort(__float2bfloat16_rn(zhi));
                    *reinterpret_cast<uint16_t *>(zb + 1 * 128 + ((((fc >> 3) ^ 1) << 4) | ((fc & 7) * 2))) =
                        __bfloat16_as_ushort(__float2bfloat16_rn(zr - zhi));
                }
                // the read operand is free once chunk c-1's read is done
                if (c >= 1 && !warp_wait(cx, &sm->Sp_empty, (c - 1) & 1)) break;
                uint8_t *sp = base + L::kOffSp;
#pragma unroll
                for (int hb = 0; hb < 2; ++hb) {
                    uint8_t *blk = sp + (2 * qq + hb) * kBlkSp;
                    *reinterpret_cast<uint4 *>(blk + sw32_offset(srow, 0)) =
                        make_uint4(spk[8 * hb], spk[8 * hb + 1], spk[8 * hb + 2], spk[8 * hb + 3]);
                    *reinterpret_cast<uint4 *>(blk + sw32_offset(srow, 8)) =
                        make_uint4(spk[8 * hb + 4], spk[8 * hb + 5], spk[8 * hb + 6], spk[8 * hb + 7]);
                }
                fence_proxy_async_smem();
                __syncwarp();
                warp_arrive(&sm->ops_full[bb]);
            } else {
                // c == nch: the final state (of the whole sequence only in the first
                // segment for dk, in the last for dq)
                if (MODE == kModeDk && seg == 0) {
                    // dS0 = alpha_1 G_1, dz0 = alpha_1 g_1: the state carried past the first chunk
                    float *dst = args.dS0 + ((size_t)bh * kR + srow) * 128 + qq * 32;
#pragma unroll
                    for (int j = 0; j < 32; j += 4) *reinterpret_cast<float4 *>(dst + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
                    if (qq == 0) args.dz0[(size_t)bh * kR + srow] = zr;
                } else if (MODE == kModeDq && GATED && seg == nseg - 1 && (args.dS_T || args.dz_T)) {
                    // <dS_T, S_T> + <dz_T, z_T> over this thread's entries
                    if (args.dS_T) {
                        const float *g = args.dS_T + ((size_t)bh * kR + srow) * 128 + qq * 32;
#pragma unroll
                        for (int j = 0; j < 32; ++j) fin_acc += S[j] * g[j];
                    }
                    if (args.dz_T && qq == 0) fin_acc += zr * args.dz_T[(size_t)bh * kR + srow];
                }
            }

            if (has_e) {
                // outputs of chunk ce = c - 1
                const int ce = c - 1, ob = ce & 1, gqe = ce % kAux;
                if (!warp_wait(cx, &sm->O_full[ob], (ce >> 1) & 1)) break;
                tc_fence_after();
                float o[16];
                tc_ld_16x32bx2_x16<16>(tmem + lane_base + L::kColO + ob * 128 + qq * 32, o);
                tc_wait_ld();
                tc_fence_before();
                warp_arrive(&sm->O_empty[ob]);
                warp_arrive(&sm->aux_empty[gqe]);   // scalars of chunk ce are done
                const int t = chunk_of(ce) * kC + prow;
                if (t < T) {
                    const size_t row = (size_t)bh * T + t;
                    uint16_t *out = (MODE == kModeDq ? args.dq : MODE == kModeDk ? args.dk : args.dv) + row * 128 + ocol;
                    float dot = 0.f;
                    if (MODE != kModeDv) {
                        // phi' and the dlog alpha term phi(x) . dx~ with x = q (dq) or k (dk)
                        const uint16_t *xs = (MODE == kModeDq ? args.q : args.k) + row * 128 + ocol;
                        const uint4 x0 = *reinterpret_cast<const uint4 *>(xs), x1 = *reinterpret_cast<const uint4 *>(xs + 8);
                        const uint32_t xw[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const float xa = bf16_lo(xw[j]), xb = bf16_hi(xw[j]);
                            // phi(x) = x + 1 and phi'(x) = 1 for x > 0, both e^x otherwise:
                            // one exponential serves both
                            const float ea = __expf(fminf(xa, 0.f)), eb = __expf(fminf(xb, 0.f));
                            const float pa = xa > 0.f ? xa + 1.f : ea, pb = xb > 0.f ? xb + 1.f : eb;
                            const float da = xa > 0.f ? 1.f : ea, db = xb > 0.f ? 1.f : eb;
                            dot += pa * o[2 * j] + pb * o[2 * j + 1];
                            o[2 * j] *= da;
                            o[2 * j + 1] *= db;
                        }
                    }
                    uint4 y0, y1;
                    y0.x = pack_bf16x2(o[0], o[1]); y0.y = pack_bf16x2(o[2], o[3]);
                    y0.z = pack_bf16x2(o[4], o[5]); y0.w = pack_bf16x2(o[6], o[7]);
                    y1.x = pack_bf16x2(o[8], o[9]); y1.y = pack_bf16x2(o[10], o[11]);
                    y1.z = pack_bf16x2(o[12], o[13]); y1.w = pack_bf16x2(o[14], o[15]);
                    reinterpret_cast<uint4 *>(out)[0] = y0;
                    reinterpret_cast<uint4 *>(out)[1] = y1;
                    // this thread's 16 columns of the row's dlog alpha term
                    if (MODE != kModeDv && args.tok_sum) atomicAdd(&args.tok_sum[row], MODE == kModeDq ? dot : -dot);
                }
            }
        }
        if (MODE == kModeDq && GATED) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) fin_acc += __shfl_xor_sync(0xffffffffu, fin_acc, o);
            if (lane == 0 && fin_acc != 0.f) atomicAdd(&args.fin[bh], fin_acc);
        }
    } else if (is_prep_warp(warp)) {
        // ------------------------------------------------------ prep warps
        // In place on the stage: phi of the q and k tiles (rows past T of a key or
        // value of phi become 0), dy times 1 / d_t (dn), the column block of dk
        // (dd_t); with a gate, once P of the chunk is complete, the query rows
        // times their read weight and the state operand's rows (and column block)
        // times their write weight.
        const int pp = prep_index(warp) * 32 + lane;   // 0..127
        // 16-byte chunk ci of a 64 x 128 tile: token row (ci & 511) >> 3
        auto each = [&](uint8_t *tile, auto fn) {
            uint4 *t4 = reinterpret_cast<uint4 *>(tile);
#pragma unroll 4
            for (int ci = pp; ci < (int)(kTile / 16); ci += kPrepThreads) t4[ci] = fn(t4[ci], (ci & 511) >> 3);
        };
        auto scale_rows = [&](uint8_t *tile, const float *wt) { each(tile, [&](uint4 v, int row) { return scale8(v, wt[row]); }); };
        auto scale_pending = [&](int x, bool waited) -> bool {
            // chunk x: once its P has read the unscaled tiles (waited: this warp has
            // already waited for that P, and must not wait again: see below)
            const int sx = x % kStages, gx = x % kAux;
            if (!waited && !warp_wait(cx, &sm->P_full, x & 1)) return false;
            uint8_t *st = stage_ptr(sx);
            const float *rw = MODE == kModeDq ? gr->gG[gx] : gr->gw[gx];   // read weights of the query rows
            const float *ww = MODE == kModeDq ? gr->gw[gx] : gr->gG[gx];   // write weights of the state operand rows
            scale_rows(st + L::kOffQry, rw);
            scale_rows(st + L::kOffKey, ww);
            if (L::kWblk && pp < kC) {
                const float cv = (MODE == kModeDq ? 1.f : ring->dd[gx][pp]) * ww[pp];
                *reinterpret_cast<uint16_t *>(st + L::kOffWblk + sw32_offset(pp, 0)) =
                    __bfloat16_as_ushort(__float2bfloat16_rn(cv));
            }
            fence_proxy_async_smem();
            warp_arrive(&sm->sc_done[sx]);
            return true;
        };
        bool ok = true;
        for (int c = 0; c < nch && ok; ++c) {
            const int s = c % kStages, gq = c % kAux;
            if (!warp_wait(cx, &sm->full[s], (c / kStages) & 1)) { ok = false; break; }
            uint8_t *st = stage_ptr(s);
            const int nvalid = min(kC, T - chunk_of(c) * kC);
            const float *invd = ring->invd[gq];
            auto phi_tile = [&](uint8_t *tile, bool zero_pad) {
                each(tile, [&](uint4 v, int row) { return (zero_pad && row >= nvalid) ? make_uint4(0, 0, 0, 0) : phi8(v); });
            };
            if (MODE == kModeDq) {
                scale_rows(st + L::kOffQry, invd);   // dn
                phi_tile(st + L::kOffVal, true);     // k~ (value; its rows past T would add to the state)
            } else if (MODE == kModeDk) {
                scale_rows(st + L::kOffKey, invd);   // dn
                phi_tile(st + L::kOffVal, true);     // q~
                if (!GATED && pp < kC)
                    *reinterpret_cast<uint16_t *>(st + L::kOffWblk + sw32_offset(pp, 0)) =
                        __bfloat16_as_ushort(__float2bfloat16_rn(ring->dd[gq][pp]));
            } else {
                phi_tile(st + L::kOffQry, false);    // k~ (query: rows past T are never stored)
                phi_tile(st + L::kOffKey, true);     // q~ (key)
                scale_rows(st + L::kOffVal, invd);   // dn
            }
            fence_proxy_async_smem();
            // One score buffer: P of chunk c (issued once this chunk is announced)
            // completes the barrier phase after chunk c-1's, of the other parity; a
            // wait for chunk c-1's parity begun after P of chunk c had completed
            // would wait for chunk c+1's P, which needs this warp.  So chunk c-1's
            // P is waited for here, before chunk c is announced, and not again.
            if (GATED && c >= 1 && !warp_wait(cx, &sm->P_full, (c - 1) & 1)) { ok = false; break; }
            warp_arrive(&sm->prep_done[s]);
            if (GATED && c >= 1 && !scale_pending(c - 1, true)) ok = false;
        }
        // the last chunk's P is the last phase: nothing can complete after it
        if (GATED && ok && nch >= 1) scale_pending(nch - 1, false);
    }

    // ---------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// One sweep per launch.  (The three side by side in one launch, 3 x B x H CTAs,
// ran slower: SMs running different sweeps thrash the shared instruction cache.)
template <int MODE, bool GATED>
__global__ void __launch_bounds__(kThreads, 1)
bwd_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
              const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_dy,
              const BwdTcArgs args)
{
    bwd_sweep<MODE, GATED>(map_q, map_k, map_v, map_dy, args);
}

}  // namespace

cudaError_t launch_bwd_tc(const CUtensorMap *maps, const BwdTcArgs &a, int B, bool gated, cudaStream_t stream,
                          int first_mode, int end_mode)
{
    using KernFn = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap, const BwdTcArgs);
    static const KernFn kerns[2][3] = {{bwd_tc_kernel<kModeDq, false>, bwd_tc_kernel<kModeDk, false>,
                                        bwd_tc_kernel<kModeDv, false>},
                                       {bwd_tc_kernel<kModeDq, true>, bwd_tc_kernel<kModeDk, true>,
                                        bwd_tc_kernel<kModeDv, true>}};
    static const uint32_t bytes[3] = {smem_bytes<kModeDq>(), smem_bytes<kModeDk>(), smem_bytes<kModeDv>()};
    static OncePerDevice attr_set[2][3];
    if (first_mode < 0 || end_mode > 3 || first_mode >= end_mode) return cudaErrorInvalidValue;
    for (int m = first_mode; m < end_mode; ++m) {
        cudaError_t e = set_smem_once(kerns[gated][m], bytes[m], attr_set[gated][m]);
        if (e != cudaSuccess) return e;
        kerns[gated][m]<<<dim3(a.nseg, a.H, B), kThreads, bytes[m], stream>>>(maps[0], maps[1], maps[2], maps[3], a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace la
