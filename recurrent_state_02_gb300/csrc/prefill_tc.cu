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
// carrying the FP32 state on chip (S and z in TMEM, where the state-increment
// MMA accumulates them).
// Per chunk (C = 64, r = 128):
//   TMA    q, k (64 x 128) and the v slice (64 x 64) as BF16 tiles, 128-byte swizzle
//   gate   (with a gate) the producer warp forms the chunk's gate products and
//          the row w while the tiles are in flight
//   phi    warps apply phi in place in packed BF16 arithmetic (phi_bf16x2); with a gate they
//          scale, once P is done, the rows of Q~ by Gamma_i and those of K~ by w_j
//   MMA    P   = Q~ K~^T            M=64  N=64  K=128  -> TMEM
//          dS  = K~'^T V            M=128 N=64  K=64   -> TMEM (K~' = diag(w) K~, or K~
//          dz  = K~'^T 1            M=128 N=16  K=64    without a gate; [V | 1] operand)
//          O   = Q~' Sprev          M=64  N=64  K=128  (Sprev as a BF16 operand;
//                                                       Q~' = Gamma Q~, or Q~ without a gate)
//          dn  = Q~' [zhi, zlo]     M=64  N=16  K=128  (zprev split into two BF16 parts,
//                                                       so Q~' . zprev keeps ~16 bits)
//          O  += A [V | 1]          M=64  N=80  K=64   (A = masked, decayed P in BF16;
//                                                       column 64 gains the row sums of A)
//   TMEM   warps: decay the TMEM state by Gamma_last (with a gate) before dS and
//          dz land on it, Sprev and [zhi, zlo] -> shared memory; P -> A;
//          y = O / (dn + eps) -> global memory (16-byte streaming stores)
// Every barrier wait is bounded; on expiry the kernel records a timeout in the
// device status word, drains its own copies and MMAs, frees TMEM and returns.

#include "tc_common.cuh"

namespace la {
namespace {

// Value columns per CTA (DVS): 64 (a head's dv is split over a cluster of CTAs)
// or 128 (one CTA owns a whole head: phi(Q), phi(K) and the scores are formed
// once per head; sequence segments then fill the GPU).
// 24 warps.  Warp w runs on scheduler w % 4 and may access TMEM lane quadrant
// w % 4.  Warps 4..19 are the TMEM warps (four per quadrant); the producer, the
// three MMA issuers and the phi warps are spread so that every scheduler hosts
// four TMEM warps, one phi warp and one light warp.
constexpr int kThreads = 768;
#ifndef LA_PHI_WARPS
#define LA_PHI_WARPS 0x30000Cu   // warps 2, 3, 20, 21: one per scheduler
#endif
// MMA issuers: warp 1 for O (chunk c's Q~ Sprev + A V), kWarpMmaP for the
// scores, kWarpMmaS for the state increments
#ifndef LA_MMAP_WARP
#define LA_MMAP_WARP 22
#endif
#ifndef LA_MMAS_WARP
#define LA_MMAS_WARP 23
#endif
constexpr int kWarpTma = 0, kWarpMma = 1, kWarpMmaS = LA_MMAS_WARP, kWarpMmaP = LA_MMAP_WARP, kWarpTm0 = 4;
constexpr uint32_t kPhiMask = LA_PHI_WARPS;
constexpr int kTmWarps = 16, kPhiWarps = __builtin_popcount(kPhiMask), kPhiThreads = kPhiWarps * 32;
constexpr int kIssuers = 3;
constexpr uint32_t kFixedRoles = 0x3u | (((1u << kTmWarps) - 1u) << kWarpTm0);   // producer, O issuer, TMEM warps
static_assert((kPhiMask & (kFixedRoles | (1u << kWarpMmaS) | (1u << kWarpMmaP))) == 0 && kWarpMmaS != kWarpMmaP &&
                  kWarpMmaS >= kWarpTm0 + kTmWarps && kWarpMmaP >= kWarpTm0 + kTmWarps && kWarpMmaS < kThreads / 32 &&
                  kWarpMmaP < kThreads / 32 && (kPhiMask >> (kThreads / 32)) == 0,
              "warp roles overlap");
// TMEM warp (quadrant qd, column quarter qq) owns rows 16 qd .. +15 and columns
// 16 qq .. +15 of the 64 x 64 tiles P, A and O, and state columns 16 qq .. +15
// of feature rows 32 qd .. +31.  Its piece of A lies strictly above the
// diagonal (always zero) when qq > qd: 6 of the 16 warps never read P.
constexpr uint32_t kTileQ = kC * kR * 2;      // 16 KB: two 64-feature blocks of 64 rows x 128 B
constexpr uint32_t kTileA = kC * kC * 2;      // 8 KB
constexpr uint32_t kBlkV = kC * 64 * 2;       // one 64-column block of V (8 KB)
constexpr uint32_t kBlkSpZ = kR * 32;         // one 16-column block of [Sprev | z] (4 KB)
// the block of ones that follows V in the [V | 1 0..] operand (128-byte swizzle,
// column 0 = 1)
constexpr uint32_t kTileOnes = kC * 128;      // 8 KB

__host__ __device__ constexpr bool is_phi_warp(int w) { return (kPhiMask >> w) & 1u; }
__host__ __device__ constexpr int phi_index(int w) { return __builtin_popcount(kPhiMask & ((1u << w) - 1u)); }

#ifndef LA_STAGES
#define LA_STAGES 4
#endif
// The gated kernel spends about twice as long per chunk, so three stages cover its
// load latency; the shared memory of the fourth holds its gate ring and a second
// [Sprev | z] tile, which lets the TMEM warps write chunk c+1's operand while the
// O MMA of chunk c still reads the other one.
#ifndef LA_STAGES_GATED
#define LA_STAGES_GATED 3
#endif
#ifndef LA_SP_BUFS
#define LA_SP_BUFS 2
#endif

#ifndef LA_STAGES_HEAD
#define LA_STAGES_HEAD 3
#endif
#ifndef LA_SP_BUFS_HEAD
#define LA_SP_BUFS_HEAD 1
#endif

template <bool GATED, int DVS>
struct Cfg {
    static_assert(DVS == 64 || DVS == 128, "value columns per CTA");
    static constexpr bool kHead = DVS == 128;
    // The whole-head CTA needs 48 KB per stage and a 36 KB [Sprev | z] tile, so it
    // keeps three stages and one such tile.
    static constexpr int kStages = kHead ? LA_STAGES_HEAD : (GATED ? LA_STAGES_GATED : LA_STAGES);
    static constexpr int kSpBufs = kHead ? LA_SP_BUFS_HEAD : LA_SP_BUFS;   // [Sprev | z] tiles
    static constexpr int kNP = kHead ? 1 : 2;                  // P accumulator buffers
    static constexpr int kNO = kHead ? 2 : 3;                  // [O | dn] accumulator buffers
    static constexpr int kLag = kNO - 1;                       // outputs of chunk c - kLag finish in iteration c
    static constexpr int kW = DVS + 16;                        // [S | z] and [O | dn] columns
    static constexpr int kSC = DVS / 4;                        // state and output columns per TMEM warp
    // TMEM columns: P (x kNP), the state [S | z] (z is column DVS) and [O | dn]
    // blocks (x kNO; dn is columns DVS and DVS + 1)
    static constexpr uint32_t kColP = 0;
    static constexpr uint32_t kColS = kNP * 64;
    static constexpr uint32_t kColO = kColS + kW;
    static constexpr uint32_t kCols = kColO + kNO * kW;
    static_assert(kCols <= 512, "TMEM budget");
    // V tile and [Sprev | zhi zlo 0..] tile: 128 feature rows x kW columns in
    // 32-byte-swizzled blocks of 16 columns; block DVS/16 holds zhi (column 0) and zlo (1)
    static constexpr uint32_t kTileV = (DVS / 64) * kBlkV;
    static constexpr uint32_t kTileSpZ = (kW / 16) * kBlkSpZ;
    // shared memory (offsets from a 1024-aligned base).  A stage holds Q, K and V;
    // with 128 value columns it also holds its own block of ones right after the
    // two V blocks, so that [V | 1] is three blocks one LBO apart and its
    // products are one MMA per K step (the ones blocks are written once).
    static constexpr uint32_t kOffQ = 0, kOffK = kTileQ, kOffV = 2 * kTileQ;
    static constexpr uint32_t kOffStageOnes = kOffV + kTileV;
    static constexpr uint32_t kStageBytes = kOffV + kTileV + (kHead ? kTileOnes : 0);
    static_assert(kStageBytes % 1024 == 0, "stage tiles stay 1024-byte aligned");
    // A is double-buffered
    static constexpr uint32_t kOffA = kStages * kStageBytes;
    static constexpr uint32_t kOffSpZ = kOffA + 2 * kTileA;
    static constexpr uint32_t kOffOnes = kOffSpZ + kSpBufs * kTileSpZ;   // (64 value columns)
    static constexpr uint32_t kOffGate = kOffOnes + (kHead ? 0 : kTileOnes);
    static constexpr uint32_t kOffSmall = kOffGate + (GATED ? sizeof(GateRing) : 0);
};

struct alignas(16) Small {
    uint64_t full[4], empty[4], phi_done[4], sc_done[4];
    // tm_read[c % 2]: the TMEM warps have read the state and P of chunk c's
    // iteration; ops_full[c % 2]: they have written its Sprev and A; O_empty[c % kNO]:
    // they have read O of chunk c
    uint64_t P_full[2], dS_full, tm_read[2], ops_full[2], Sp_empty;
    uint64_t A_empty[2], O_full[3], O_empty[3], aux_empty[kAux];
    uint64_t mma_done[kIssuers];
    uint32_t tmem_base;
    int abort_flag;
};

template <bool GATED, int DVS>
constexpr uint32_t smem_bytes() { return Cfg<GATED, DVS>::kOffSmall + sizeof(Small) + 1024; }
static_assert(smem_bytes<false, 64>() <= 232448, "shared memory budget");
static_assert(smem_bytes<true, 64>() <= 232448, "shared memory budget");
static_assert(smem_bytes<false, 128>() <= 232448, "shared memory budget");
static_assert(smem_bytes<true, 128>() <= 232448, "shared memory budget");

// This CTA's sequence b and segment g of it, the sequence's segment count, the
// chunks per segment, and the S_start slot its start state is read from (-1: S0
// itself).  Segments come
// from the varlen plan's item table, or grid.z enumerates (b, segment) of the
// [B, H, T, d] layout with args.nseg segments per sequence.
struct CtaUnit {
    int b, seg, nseg, len, slot;
};
template <bool ITEMS>
__device__ __forceinline__ CtaUnit cta_unit(const PrefillTcArgs &args)
{
    if (ITEMS) {
        const int2 it = args.items[blockIdx.z];
        const int4 si = args.seq_info[it.x];
        return CtaUnit{it.x, it.y, si.x, args.seg_len[0], si.x > 1 ? si.y + it.y : -1};
    }
    const int B = gridDim.z / args.nseg, b = blockIdx.z / args.nseg, seg = blockIdx.z % args.nseg;
    return CtaUnit{b, seg, args.nseg, args.seg_chunks, args.S_start ? seg * B + b : -1};
}

// The kernel body for one CTA.  FAST (gated whole-head CTAs only): every chunk
// of this CTA carries its gates as row weights (see cta_all_fast), so the body is
// built without the explicit path.  PLAIN: [B, H, T, d] inputs and one segment
// per head (no packed sequences, no scanned start states).  SAVE: the stores a
// training forward asks for (d_t, and the states entering the backward's
// segments) are compiled in; the other bodies carry none of their code.  ITEMS:
// the CTA's sequence and segment come from the varlen plan's item table.
template <bool GATED, int DVS, bool FAST, bool PLAIN, bool SAVE, bool ITEMS>
__device__ __forceinline__ void
prefill_body(const CUtensorMap &map_q, const CUtensorMap &map_k, const CUtensorMap &map_v, const PrefillTcArgs &args)
{
    using L = Cfg<GATED, DVS>;
    static_assert(!FAST || (GATED && L::kHead), "the row-weight body is for gated whole-head CTAs");
    constexpr int NST = L::kStages, NP = L::kNP, SC = L::kSC;
    static_assert(NP == 1 || NP == 2, "score buffers");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Small *sm = reinterpret_cast<Small *>(base + L::kOffSmall);
    GateRing *gr = reinterpret_cast<GateRing *>(base + L::kOffGate);   // gated only
    Ctx cx{&sm->abort_flag, args.wait_limit_ns, args.status};

    const int slice = blockIdx.x;
    const int h = blockIdx.y;
    const CtaUnit u = PLAIN ? CtaUnit{(int)blockIdx.z, 0, 1, 0, -1} : cta_unit<ITEMS>(args);
    const int b = u.b, seg = u.seg;
    const int bh = b * args.H + h;
    // Packed sequences of different lengths (cu_seqlens; no segments) or the
    // [B, H, T, d] layout.  A sequence whose bounds are inconsistent with the
    // total is recorded as a shape error and processes no tokens.
    const bool varlen = !PLAIN && args.cu_seqlens != nullptr;
    int seq0 = 0, T = args.T;
    if (varlen) {
        seq0 = args.cu_seqlens[b];
        const int seq1 = args.cu_seqlens[b + 1];
        if (seq0 < 0 || seq1 < seq0 || seq1 > args.T) {
            if (threadIdx.x == 0) atomicExch(args.status, kStatusShape);
            seq0 = 0;
            T = 0;
        } else {
            T = seq1 - seq0;
        }
    }
    // row of token t (of this sequence) in q, k, v, y (rows of d values) and alpha
    auto tok_row = [&](int t) -> size_t { return varlen ? (size_t)(seq0 + t) * args.H + h : (size_t)bh * T + t; };
    // the last two TMA coordinates of a box starting at token t0
    auto tma_c1 = [&](int t0) { return varlen ? h : t0; };
    auto tma_c2 = [&](int t0) { return varlen ? seq0 + t0 : bh; };
    const int nch_all = (T + kC - 1) / kC;
    const int c0 = seg * u.len;                                               // first chunk of the segment
    const int nch = (!PLAIN && u.nseg > 1) ? min(u.len, nch_all - c0) : nch_all;   // its chunk count
    const int tb = c0 * kC;                                                   // its first token
    const bool last_seg = PLAIN || seg == u.nseg - 1;
    // start state of this head: S0/z0, or the scanned state of the segment
    const size_t state_len = (size_t)kR * args.dv + kR;
    const bool scanned = u.slot >= 0;
    const float *S_init = scanned ? args.S_start + ((size_t)u.slot * args.H + h) * state_len
                                  : (args.S0 ? args.S0 + (size_t)bh * kR * args.dv : nullptr);
    const float *z_init_src = scanned ? S_init + (size_t)kR * args.dv : (args.z0 ? args.z0 + (size_t)bh * kR : nullptr);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    auto stage_ptr = [&](int s) { return base + s * L::kStageBytes; };

    // ------------------------------------------------------------ set-up
    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(&sm->full[s], GATED ? 2 : 1);   // TMA bytes (+ gate data)
            mbar_init(&sm->empty[s], kIssuers);   // one commit from each MMA issuer
            mbar_init(&sm->phi_done[s], kPhiWarps);
            mbar_init(&sm->sc_done[s], kPhiWarps);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm->P_full[i], 1);
            mbar_init(&sm->tm_read[i], kTmWarps);
            mbar_init(&sm->ops_full[i], kTmWarps);
            mbar_init(&sm->A_empty[i], 1);
        }
        for (int i = 0; i < 3; ++i) {
            mbar_init(&sm->O_full[i], 1);
            mbar_init(&sm->O_empty[i], kTmWarps);
        }
        mbar_init(&sm->Sp_empty, 1);
        for (int i = 0; i < kAux; ++i) mbar_init(&sm->aux_empty[i], kTmWarps);
        mbar_init(&sm->dS_full, 1);
        for (int i = 0; i < kIssuers; ++i) mbar_init(&sm->mma_done[i], 1);
        sm->abort_flag = 0;
        fence_mbarrier_init();
        tma_prefetch_desc(&map_q);
        tma_prefetch_desc(&map_k);
        tma_prefetch_desc(&map_v);
    }
    // Constant operand parts: the z block (columns 64..79) of the [Sprev | z]
    // tile starts at zero (only columns 64 and 65 are written later); the ones
    // block is complete here (column 0 = 1 in every token row).
    for (int i = threadIdx.x; i < (int)(2 * kTileA / 16); i += kThreads)   // A: the blocks above the diagonal stay 0
        reinterpret_cast<uint4 *>(base + L::kOffA)[i] = make_uint4(0, 0, 0, 0);
    for (int i = threadIdx.x; i < L::kSpBufs * (kBlkSpZ / 16); i += kThreads) {
        const int buf = i / (kBlkSpZ / 16), j = i % (kBlkSpZ / 16);
        reinterpret_cast<uint4 *>(base + L::kOffSpZ + buf * L::kTileSpZ + (DVS / 16) * kBlkSpZ)[j] =
            make_uint4(0, 0, 0, 0);
    }
    // the ones block(s): one after the stages (64 value columns) or one per stage
    constexpr int kNOnes = L::kHead ? NST : 1;
    auto ones_ptr = [&](int i) {
        return base + (L::kHead ? i * L::kStageBytes + L::kOffStageOnes : L::kOffOnes);
    };
    for (int i = threadIdx.x; i < kNOnes * (int)(kTileOnes / 16); i += kThreads)
        reinterpret_cast<uint4 *>(ones_ptr(i / (kTileOnes / 16)))[i % (kTileOnes / 16)] = make_uint4(0, 0, 0, 0);
    __syncthreads();
    if (threadIdx.x < kNOnes * kC)   // element (column 0, token row k): 16-byte chunk 0 of row k after the swizzle
        *reinterpret_cast<uint16_t *>(ones_ptr(threadIdx.x / kC) + sw128_offset(threadIdx.x % kC, 0)) = 0x3F80u;
    fence_proxy_async_smem();
    if (warp == kWarpMma) {
        tmem_alloc(&sm->tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm->tmem_base;
    // The dv slices of one head (and segment) form a cluster: no slice may write
    // z_out (which may alias z0) before every slice has read z0.  Every thread
    // takes part.  (Segmented runs read their start state from the workspace.)
    const bool clustered = gridDim.x > 1;
    float z_init = 0.f;
    if (warp >= kWarpTm0 && warp < kWarpTm0 + kTmWarps && z_init_src)
        z_init = z_init_src[(warp & 3) * 32 + lane];
    if (clustered) {
        asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
        asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    }

    if (warp == kWarpTma) {
        // ------------------------------------------------------- producer
        // Lane 0 issues the tile loads of a stage.  With a gate the whole warp
        // then forms the chunk's gate products and makes the stage's second
        // arrival; the gates are read before the wait for the free stage, so
        // their latency hides behind it.
        int issued = 0;
        for (int c = 0; c < nch; ++c) {
            const int s = c % NST;
            const int t0 = tb + c * kC;
            float a0 = 1.f, a1 = 1.f;
            if (GATED) {
                if (t0 + 2 * lane < T) a0 = args.alpha[tok_row(t0 + 2 * lane)];
                if (t0 + 2 * lane + 1 < T) a1 = args.alpha[tok_row(t0 + 2 * lane + 1)];
            }
            if (c >= NST && !warp_wait(cx, &sm->empty[s], ((c / NST) - 1) & 1)) break;
            if (GATED && c >= kAux && !warp_wait(cx, &sm->aux_empty[c % kAux], ((c / kAux) - 1) & 1)) break;
            if (__shfl_sync(0xffffffffu, aborted(cx) ? 1 : 0, 0)) break;
            uint8_t *st = stage_ptr(s);
            if (lane == 0) {
                mbar_arrive_expect_tx(&sm->full[s], 2 * kTileQ + L::kTileV);
                const int cy = tma_c1(t0), cz = tma_c2(t0);
                tma_load_3d(st + L::kOffQ, &map_q, &sm->full[s], 0, cy, cz);
                tma_load_3d(st + L::kOffQ + kTileQ / 2, &map_q, &sm->full[s], 64, cy, cz);
                tma_load_3d(st + L::kOffK, &map_k, &sm->full[s], 0, cy, cz);
                tma_load_3d(st + L::kOffK + kTileQ / 2, &map_k, &sm->full[s], 64, cy, cz);
#pragma unroll
                for (int vb = 0; vb < DVS / 64; ++vb)
                    tma_load_3d(st + L::kOffV + vb * kBlkV, &map_v, &sm->full[s], slice * DVS + vb * 64, cy, cz);
                // The load of chunk c + NST waits for this stage to come free, which
                // takes about as long as a load from HBM: warm L2 for it now.
                if (c + NST < nch) {
                    const int tp = t0 + NST * kC, yp = tma_c1(tp), zp = tma_c2(tp);
                    if (slice == 0) {   // the other slices of the head read the same q, k
                        tma_prefetch_l2_3d(&map_q, 0, yp, zp);
                        tma_prefetch_l2_3d(&map_q, 64, yp, zp);
                        tma_prefetch_l2_3d(&map_k, 0, yp, zp);
                        tma_prefetch_l2_3d(&map_k, 64, yp, zp);
                    }
#pragma unroll
                    for (int vb = 0; vb < DVS / 64; ++vb) tma_prefetch_l2_3d(&map_v, slice * DVS + vb * 64, yp, zp);
                }
            }
            if (GATED) {
                gate_products(a0, a1, lane, c % kAux, gr);
                warp_arrive(&sm->full[s]);
            }
            issued = c + 1;
        }
        if (lane == 0 && aborted(cx)) {
            // Drain: every issued load must land before the CTA may exit.
            for (int c = (issued > NST ? issued - NST : 0); c < issued; ++c)
                mbar_wait(&sm->full[c % NST], (c / NST) & 1, cx.limit);
        }
        __syncwarp();
    } else if (warp == kWarpMma || warp == kWarpMmaS || warp == kWarpMmaP) {
        // ------------------------------------------------------------ MMA
        // Three issuers, each lane 0 of its warp (tcgen05.mma and tcgen05.commit
        // are issued by one thread; the other lanes wait at the teardown
        // barrier), share the tensor pipe: warp kWarpMma issues chunk c's
        // O = Q~ Sprev + A V, warp kWarpMmaP the scores P = Q~ K~^T up to NP
        // chunks ahead, warp kWarpMmaS the state increments as soon as the
        // TMEM warps have read the state.  Each commits its own arrival on a
        // stage's empty barrier after its last read of it.
        if (lane == 0) {
            constexpr uint32_t idP = idesc_bf16_f32(64, 64, false, false);
            // [S | z] increment and [O | dn] += A [V | 1] (column DVS gains the row
            // sums of A): one MMA per K step spans the V block(s) and the first 16
            // columns of the ones block, LBO apart (64 value columns: the shared
            // ones block after the stages; 128: the stage's own, one block after V).
            constexpr uint32_t idDS = idesc_bf16_f32(128, L::kW, true, true);
            constexpr uint32_t idQS = idesc_bf16_f32(64, L::kW, false, true);   // [O | dn] = Q~ [Sprev | z]
            constexpr uint32_t idAV = idesc_bf16_f32(64, L::kW, false, true);
            const uint32_t aOnes = smem_u32(base + L::kOffOnes);
            constexpr uint32_t kHi128 = desc_hi(1024, 2), kHi32 = desc_hi(256, 6);   // SBO and swizzle words
            // P = Q~ K~^T for chunk c
            auto issue_p = [&](int c) -> bool {
                const int s = c % NST, pb = c % NP;
                const uint32_t st = smem_u32(stage_ptr(s));
                const uint32_t aQ = st + L::kOffQ, aK = st + L::kOffK;
                if (!wait(cx, &sm->phi_done[s], (c / NST) & 1)) return false;
                // the P buffer of chunk c - NP has been read
                if (c >= NP && !wait(cx, &sm->tm_read[(c - NP) & 1], ((c - NP) >> 1) & 1)) return false;
                tc_fence_after();
                const uint32_t qlo = desc_lo(aQ, 16), klo = desc_lo(aK, 16), dP = tmem + L::kColP + pb * 64;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t o = ((kk >> 2) * (kTileQ / 2) + (kk & 3) * 32) >> 4;
                    if (kk == 0) tc_mma_bf16_w<false>(dP, qlo + o, kHi128, klo + o, kHi128, idP);
                    else tc_mma_bf16_w<true>(dP, qlo + o, kHi128, klo + o, kHi128, idP);
                }
                tc_commit(&sm->P_full[pb]);
                tc_commit(&sm->empty[s]);   // this issuer's last read of stage s
                return true;
            };
            // [S | z] += K~'^T [V | 1] for chunk c, K~' = diag(w) K~ with a gate,
            // once phi of chunk c is done (with a gate: its rows scaled, after P
            // of chunk c) and the TMEM warps have read (and, with a gate,
            // decayed) the state after chunk c-1
            auto issue_ds = [&](int c) -> bool {
                const int s = c % NST;
                const uint32_t st = smem_u32(stage_ptr(s));
                const uint32_t aK = st + L::kOffK;
                // B = [V | 1]: the V tile, then (64 value columns) the ones block at LBO
                const uint32_t blo = desc_lo(st + L::kOffV, L::kHead ? kBlkV : aOnes - (st + L::kOffV));
                if (!GATED && !wait(cx, &sm->phi_done[s], (c / NST) & 1)) return false;
                if (GATED && !wait(cx, &sm->sc_done[s], (c / NST) & 1)) return false;
                if (!wait(cx, &sm->tm_read[c & 1], (c >> 1) & 1)) return false;   // state read (and decayed)
                tc_fence_after();
                const uint32_t dS = tmem + L::kColS;
                const uint32_t klo = desc_lo(aK, kTileQ / 2);   // K~^T: MN-major, two 64-feature blocks
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc_mma_bf16_w<true>(dS, klo + kk * (2048 >> 4), kHi128, blo + kk * (2048 >> 4), kHi128, idDS);
                tc_commit(&sm->dS_full);
                tc_commit(&sm->empty[s]);   // this issuer's last read of stage s
                return true;
            };
            bool ok = true;
            if (warp == kWarpMmaP) {
                for (int c = 0; c < nch && ok && !aborted(cx); ++c) ok = issue_p(c);
            } else if (warp == kWarpMmaS) {
                for (int c = 0; c < nch && ok && !aborted(cx); ++c) ok = issue_ds(c);
            }
            for (int c = 0; warp == kWarpMma && c < nch && ok && !aborted(cx); ++c) {
                const int s = c % NST, bb = c & 1, n = c >> 1;
                const uint32_t st = smem_u32(stage_ptr(s));
                const uint32_t aQ = st + L::kOffQ, aV = st + L::kOffV;
                const uint32_t aA = smem_u32(base + L::kOffA + bb * kTileA);
                const int sb = c % L::kSpBufs;
                const uint32_t aSpZ = smem_u32(base + L::kOffSpZ + sb * L::kTileSpZ);
                // [O | dn] = Q~ [Sprev | zhi zlo] (gated: Q~ rows already scaled by Gamma_i),
                // then [O | dn] += A [V | 1], into the buffer that held O of chunk c - kNO
                const int ob = c % L::kNO;
                if (GATED && !wait(cx, &sm->sc_done[s], (c / NST) & 1)) break;
                if (!wait(cx, &sm->ops_full[bb], n & 1)) break;
                if (c >= L::kNO && !wait(cx, &sm->O_empty[ob], ((c / L::kNO) - 1) & 1)) break;
                tc_fence_after();
                const uint32_t dO = tmem + L::kColO + ob * L::kW;
                const uint32_t qlo = desc_lo(aQ, 16), slo = desc_lo(aSpZ, kBlkSpZ);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t o = ((kk >> 2) * (kTileQ / 2) + (kk & 3) * 32) >> 4;
                    if (kk == 0) tc_mma_bf16_w<false>(dO, qlo, kHi128, slo, kHi32, idQS);
                    else tc_mma_bf16_w<true>(dO, qlo + o, kHi128, slo + kk * (512 >> 4), kHi32, idQS);
                }
                if (L::kSpBufs == 1) tc_commit(&sm->Sp_empty);
                const uint32_t alo = desc_lo(aA, 16);
                const uint32_t vlo = desc_lo(aV, L::kHead ? kBlkV : aOnes - aV);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc_mma_bf16_w<true>(dO, alo + kk * (32 >> 4), kHi128, vlo + kk * (2048 >> 4), kHi128, idAV);
                tc_commit(&sm->A_empty[bb]);
                tc_commit(&sm->O_full[ob]);
                tc_commit(&sm->empty[s]);
            }
            // Every MMA issued above completes before TMEM is released.
            uint64_t *done = &sm->mma_done[warp == kWarpMma ? 0 : warp == kWarpMmaP ? 1 : 2];
            tc_commit(done);
            mbar_wait(done, 0, cx.limit);
        }
        __syncwarp();
    } else if (warp >= kWarpTm0 && warp < kWarpTm0 + kTmWarps) {
        // ----------------------------------------------------- TMEM warps
        // The FP32 state [S | z] lives in TMEM, where the MMAs accumulate the
        // state increments.  Iteration c reads the state after chunk c-1 (it
        // becomes Sprev of chunk c; with a gate it is then decayed by Gamma_last
        // of chunk c in place, ahead of chunk c's increment), turns the scores of
        // chunk c into A, and finishes the outputs of chunk c - kLag.  Each warp
        // stores its own 16-row x SC-column piece of y.
        constexpr int LAG = L::kLag;
        const int tw = warp - kWarpTm0;          // 0..15
        const int qd = warp & 3;                 // TMEM lane quadrant this warp may access
        const int qq = tw >> 2;                  // column quarter
        const uint32_t lane_base = static_cast<uint32_t>(qd * 32) << 16;
        const int srow = qd * 32 + lane;         // state row (feature index) of this thread
        const int prow = qd * 16 + (lane & 15);  // row of the M = 64 tiles (16x32bx2 loads)
        const int pcol = qq * 16 + (lane >> 4) * 8;   // first of this thread's 8 columns of P and A
        const int ocol = qq * SC + (lane >> 4) * (SC / 2);   // first of its SC/2 columns of O and y
        const bool a_zero = qq > qd;             // this warp's piece of A is above the diagonal
        const uint32_t tS = tmem + lane_base + L::kColS + qq * SC;   // this thread's SC state columns
        const uint32_t tz = tmem + lane_base + L::kColS + DVS;       // z (column DVS; qq == 0 warps)
        auto ld_state = [&](float (&v)[SC]) {
            if constexpr (SC == 16) tc_ld_32x32b_x16(tS, v);
            else tc_ld_32x32b_x32(tS, v);
        };
        auto st_state = [&](const float (&v)[SC]) {
            if constexpr (SC == 16) tc_st_32x32b_x16(tS, v);
            else tc_st_32x32b_x32(tS, v);
        };
        {
            // initial state: 16-byte loads when the start state is 16-byte aligned
            // (the scanned segment states always are; a caller's S0 may be 4-byte aligned)
            float S[SC];
            const float *src = S_init ? S_init + (size_t)srow * args.dv + slice * DVS + qq * SC : nullptr;
            if (src && (reinterpret_cast<uintptr_t>(S_init) & 15) == 0) {
#pragma unroll
                for (int j = 0; j < SC; j += 4) {
                    const float4 v4 = *reinterpret_cast<const float4 *>(src + j);
                    S[j] = v4.x; S[j + 1] = v4.y; S[j + 2] = v4.z; S[j + 3] = v4.w;
                }
            } else {
#pragma unroll
                for (int j = 0; j < SC; ++j) S[j] = src ? src[j] : 0.f;
            }
            st_state(S);
            if (qq == 0) tc_st_32x32b_x1(tz, z_init);
            tc_wait_st();
        }

        for (int c = 0; c < nch + LAG; ++c) {
            const bool has_s = c <= nch;              // the state after chunk c-1
            const bool has_b = c < nch;               // Sprev and scores of chunk c
            const bool has_p = has_b && !a_zero;
            const bool has_e = c >= LAG;              // outputs of chunk c - LAG
            const int bb = c & 1, pb = c % NP, pn = c / NP;
            if (has_s && c >= 1 && !warp_wait(cx, &sm->dS_full, (c - 1) & 1)) break;
            if (has_b && GATED && !warp_wait(cx, &sm->phi_done[c % NST], (c / NST) & 1)) break;
            if (has_p && !warp_wait(cx, &sm->P_full[pb], pn & 1)) break;
            tc_fence_after();
            float S[SC], zr = 0.f, p[8];
            if (has_s) {
                ld_state(S);
                if (qq == 0) tc_ld_32x32b_x1(tz, zr);
            }
            if (has_p) tc_ld_16x32bx2_x8<8>(tmem + lane_base + L::kColP + pb * 64 + qq * 16, p);
            tc_wait_ld();
            // on request, the state entering chunk c where a segment of the backward starts
            if (SAVE && has_s && args.bwd_states && ((c0 + c) % args.bwd_seg_chunks) == 0 &&
                (c0 + c) / args.bwd_seg_chunks < args.bwd_nseg) {
                float *dst = args.bwd_states + ((size_t)((c0 + c) / args.bwd_seg_chunks) * args.bwd_heads + bh) *
                                                   (kR * 128 + kR);
#pragma unroll
                for (int j = 0; j < SC; j += 4)
                    *reinterpret_cast<float4 *>(dst + (size_t)srow * 128 + slice * DVS + qq * SC + j) =
                        make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
                if (slice == 0 && qq == 0) dst[kR * 128 + srow] = zr;
            }
            // Sprev of chunk c (BF16) and z split into two BF16 parts.  With a gate
            // the state is decayed by the chunk's gate product Gamma_last before its
            // increment lands; a fast chunk (whole head) reads the decayed state:
            // its outputs are O' = w_i O (see the epilogue).
            const bool fast = GATED && L::kHead && has_b && (FAST || gr->gf[c % kAux] != 0);
            uint32_t spk[SC / 2];
            float zhi = 0.f, zsp = zr;
            if (GATED && has_b) {
                const float g = gr->gG[c % kAux][kC - 1];
                if (!fast) {
#pragma unroll
                    for (int j = 0; j < SC / 2; ++j) spk[j] = pack_bf16x2(S[2 * j], S[2 * j + 1]);
                }
#pragma unroll
                for (int j = 0; j < SC; ++j) S[j] *= g;
                st_state(S);
                if (qq == 0) tc_st_32x32b_x1(tz, g * zr);
                if (fast) {
#pragma unroll
                    for (int j = 0; j < SC / 2; ++j) spk[j] = pack_bf16x2(S[2 * j], S[2 * j + 1]);
                    zsp = g * zr;
                }
                tc_wait_st();
            } else if (has_b) {
#pragma unroll
                for (int j = 0; j < SC / 2; ++j) spk[j] = pack_bf16x2(S[2 * j], S[2 * j + 1]);
            }
            if (has_b) zhi = __bfloat162float(__float2bfloat16_rn(zsp));
            tc_fence_before();
            if (has_b) warp_arrive(&sm->tm_read[bb]);

            // A = the causal mask (and, with a gate, the in-chunk decay) applied to P;
            // without a gate, or for a fast chunk, a piece strictly below the
            // diagonal is P itself
            if (has_p && ((GATED && !fast) || qq == qd)) {
                const int gq = c % kAux;
                const float bi = GATED ? gr->gb[gq][prow] : 0.f;
                const int zi = GATED ? gr->gz[gq][prow] : -1;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int j = pcol + e;
                    float a = (j <= prow) ? p[e] : 0.f;
                    if (GATED && !fast) a = (j <= prow && zi <= j) ? a * __expf(bi - gr->gb[gq][j]) : 0.f;
                    p[e] = a;
                }
            }

            // shared-memory operands (ahead of the outputs: the O issuer waits for them)
            if (has_b) {
                const int sb = c % L::kSpBufs;
                // A first: its buffer held chunk c-2's, free once that chunk's O MMAs
                // are done (which, with two Sprev buffers, also frees this Sprev buffer)
                if (c >= 2 && !warp_wait(cx, &sm->A_empty[bb], ((c >> 1) - 1) & 1)) break;
                if (!a_zero)
                    *reinterpret_cast<uint4 *>(base + L::kOffA + bb * kTileA + sw128_offset(prow, pcol >> 3)) =
                        make_uint4(pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3]), pack_bf16x2(p[4], p[5]),
                                   pack_bf16x2(p[6], p[7]));
                // with one Sprev buffer, it is free once chunk c-1's Q~ Sprev is done
                if (L::kSpBufs == 1 && c >= 1 && !warp_wait(cx, &sm->Sp_empty, (c - 1) & 1)) break;
                // Sprev columns SC qq .. +SC-1 of row srow: 16-column blocks SC/16 qq ..
                uint8_t *spz = base + L::kOffSpZ + sb * L::kTileSpZ;
#pragma unroll
                for (int hb = 0; hb < SC / 16; ++hb) {
                    uint8_t *blk = spz + (qq * (SC / 16) + hb) * kBlkSpZ;
                    *reinterpret_cast<uint4 *>(blk + sw32_offset(srow, 0)) =
                        make_uint4(spk[8 * hb], spk[8 * hb + 1], spk[8 * hb + 2], spk[8 * hb + 3]);
                    *reinterpret_cast<uint4 *>(blk + sw32_offset(srow, 8)) =
                        make_uint4(spk[8 * hb + 4], spk[8 * hb + 5], spk[8 * hb + 6], spk[8 * hb + 7]);
                }
                // z as two BF16 parts in columns DVS (zhi) and DVS + 1 (zlo)
                if (qq == 0)
                    *reinterpret_cast<uint32_t *>(spz + (DVS / 16) * kBlkSpZ + sw32_offset(srow, 0)) =
                        pack_bf16x2(zhi, zsp - zhi);
                fence_proxy_async_smem();
                warp_arrive(&sm->ops_full[bb]);
            } else if (has_s && last_seg) {
                // c == nch: the state after the last chunk
                float *dst = args.S_out + ((size_t)bh * kR + srow) * args.dv + slice * DVS + qq * SC;
#pragma unroll
                for (int j = 0; j < SC; j += 4)
                    *reinterpret_cast<float4 *>(dst + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
                if (slice == 0 && qq == 0) args.z_out[(size_t)bh * kR + srow] = zr;
            }

            // outputs of chunk c - LAG: columns DVS and DVS + 1 of [O | dn] hold
            // Q~' . zprev in two parts plus the row sums of A
            if (has_e) {
                const int ce = c - LAG;
                const int ob = ce % L::kNO;
                if (!warp_wait(cx, &sm->O_full[ob], (ce / L::kNO) & 1)) break;
                tc_fence_after();
                float o[SC / 2], dn;
                if constexpr (SC == 16) tc_ld_16x32bx2_x8<8>(tmem + lane_base + L::kColO + ob * L::kW + qq * SC, o);
                else tc_ld_16x32bx2_x16<16>(tmem + lane_base + L::kColO + ob * L::kW + qq * SC, o);
                tc_ld_16x32bx2_x1<1>(tmem + lane_base + L::kColO + ob * L::kW + DVS, dn);
                tc_wait_ld();
                tc_fence_before();
                warp_arrive(&sm->O_empty[ob]);
                dn += __shfl_xor_sync(0xffffffffu, dn, 16);
                // a fast chunk's row i holds O' = w_i O and dn' = w_i dn: y = O' / (dn' + eps w_i)
                float epsw = args.eps, wrow = 1.f;
                if (GATED && L::kHead && (FAST || gr->gf[ce % kAux] != 0)) {
                    wrow = gr->gw[ce % kAux][prow];
                    epsw *= wrow;
                }
                if (GATED) warp_arrive(&sm->aux_empty[ce % kAux]);   // gate data of chunk ce is done
                float inv;   // approximate reciprocal: y is rounded to BF16 below
                asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(inv) : "f"(dn + epsw));
                // SC/2 columns (16 or 32 bytes) of token row prow, straight to global
                // memory (streaming stores: y is not read again here)
                const int t = tb + ce * kC + prow;
                // d_t on request (one lane per row): the denominator of y, divided
                // by the row weight where the chunk carries one
                if (SAVE && args.d_out && slice == 0 && qq == 0 && lane < 16 && t < T)
                    args.d_out[tok_row(t)] = (GATED && L::kHead) ? (dn + epsw) / wrow : dn + epsw;
                if (t < T) {
                    uint4 *dst = reinterpret_cast<uint4 *>(args.y + tok_row(t) * args.dv + slice * DVS + ocol);
#pragma unroll
                    for (int v8 = 0; v8 < SC / 16; ++v8) {
                        uint4 yp;
                        yp.x = pack_bf16x2(o[8 * v8 + 0] * inv, o[8 * v8 + 1] * inv);
                        yp.y = pack_bf16x2(o[8 * v8 + 2] * inv, o[8 * v8 + 3] * inv);
                        yp.z = pack_bf16x2(o[8 * v8 + 4] * inv, o[8 * v8 + 5] * inv);
                        yp.w = pack_bf16x2(o[8 * v8 + 6] * inv, o[8 * v8 + 7] * inv);
                        __stcs(dst + v8, yp);
                    }
                }
            }
        }
    } else if (is_phi_warp(warp)) {
        // ------------------------------------------------------ phi warps
        const int pp = phi_index(warp) * 32 + lane;   // 0..159
        // gated: once P of chunk x is complete (it read the unscaled tiles), the
        // rows of Q~ are scaled in place by Gamma_i (O = (Gamma Q~) Sprev) and
        // the rows of K~ by w_j (dS = (w K~)^T V, dz = (w K~)^T 1).  waited: this
        // warp has already waited for that P (and must not wait again: see below)
        auto scale_qk = [&](int x, bool waited) -> bool {
            const int sx = x % NST;
            if (!waited && !warp_wait(cx, &sm->P_full[x % NP], (x / NP) & 1)) return false;
            uint4 *qk = reinterpret_cast<uint4 *>(stage_ptr(sx) + L::kOffQ);
            const float *gam = gr->gG[x % kAux];
            const float *w = gr->gw[x % kAux];
            constexpr int kFull = 2048 / kPhiThreads, kRest = 2048 - kFull * kPhiThreads;
#pragma unroll
            for (int it = 0; it <= kFull; ++it) {
                const int ci = pp + it * kPhiThreads;   // 16-byte chunk; token row (ci & 511) >> 3
                if (it < kFull || pp < kRest) qk[ci] = scale8(qk[ci], (ci < 1024 ? gam : w)[(ci & 511) >> 3]);
            }
            fence_proxy_async_smem();
            warp_arrive(&sm->sc_done[sx]);
            return true;
        };
        // Gated, whole head: a chunk flagged fast (gate_products) carries its gates
        // as row weights w_j on K~ instead, applied with phi: then P' = Q~ K~'^T =
        // P diag(w), so A' [V | 1] = sum_j A_ij w_j [v_j | 1] and K~'^T [V | 1] is
        // the state increment, and neither tile waits for a scaling after P.
        constexpr bool kFastOk = GATED && L::kHead;
        auto is_fast = [&](int x) { return FAST || (kFastOk && gr->gf[x % kAux] != 0); };
        bool ok = true, f_last = false;
        for (int c = 0; c < nch && ok; ++c) {
            const int s = c % NST;
            const int nvalid = min(kC, T - tb - c * kC);
            if (!warp_wait(cx, &sm->full[s], (c / NST) & 1)) { ok = false; break; }
            uint8_t *st = stage_ptr(s);
            // the flags of chunks c and c-1 (the ring entry of c-1 cannot be reused
            // before P of chunk c, which waits for this iteration's phi_done)
            const bool f_cur = is_fast(c), f_prev = c >= 1 && is_fast(c - 1);
            f_last = f_cur;
            // phi(Q), phi(K) in place (the two tiles are contiguous: 2048 chunks of
            // 16 bytes, K from chunk 1024); key rows past the end of the sequence
            // become 0; a fast chunk's key rows times w_j
            static_assert(L::kOffK == L::kOffQ + kTileQ, "Q and K tiles are contiguous");
            uint4 *qk = reinterpret_cast<uint4 *>(st + L::kOffQ);
            constexpr int kFull = 2048 / kPhiThreads, kRest = 2048 - kFull * kPhiThreads;
            if (nvalid == kC && !f_cur) {
#pragma unroll
                for (int it = 0; it < kFull; ++it) qk[pp + it * kPhiThreads] = phi8(qk[pp + it * kPhiThreads]);
                if (pp < kRest) qk[pp + kFull * kPhiThreads] = phi8(qk[pp + kFull * kPhiThreads]);
            } else if (nvalid == kC) {
                const float *w = gr->gw[c % kAux];
#pragma unroll
                for (int it = 0; it <= kFull; ++it) {
                    const int ci = pp + it * kPhiThreads;
                    if (it < kFull || pp < kRest) {
                        const uint4 v = phi8(qk[ci]);
                        qk[ci] = ci >= 1024 ? scale8(v, w[(ci & 511) >> 3]) : v;
                    }
                }
            } else {
                const float *w = gr->gw[c % kAux];
                for (int ci = pp; ci < 2048; ci += kPhiThreads) {
                    const int row = (ci & 511) >> 3;   // 8 chunks per 128-byte row, 64 rows per block
                    uint4 v = (ci >= 1024 && row >= nvalid) ? make_uint4(0, 0, 0, 0) : phi8(qk[ci]);
                    if (f_cur && ci >= 1024) v = scale8(v, w[row]);
                    qk[ci] = v;
                }
            }
            fence_proxy_async_smem();
            // With one score buffer, whose barrier completes a phase per chunk, a
            // wait for chunk x's parity is only sound while the barrier is in chunk
            // x's phase or the one after it: begun later, it would wait for chunk
            // x+2's P (which needs this warp); begun earlier, before chunk x-1's P
            // had completed, it would return at once.  So chunk c-1's P is waited
            // for here, for every chunk (fast or slow), before phi of chunk c is
            // announced, and not again.
            const bool waited = GATED && NP == 1 && c >= 1;
            if (waited && !warp_wait(cx, &sm->P_full[0], (c - 1) & 1)) {
                ok = false;
                break;
            }
            warp_arrive(&sm->phi_done[s]);
            if (GATED && f_cur) warp_arrive(&sm->sc_done[s]);   // nothing to scale after P
            // P of chunk c-1 was issued once phi of chunk c-1 was done and has
            // normally completed while phi of chunk c ran
            if (GATED && c >= 1 && !f_prev && !scale_qk(c - 1, waited)) ok = false;
        }
        // the last chunk's P is the last phase: nothing can complete after it
        if (GATED && ok && nch >= 1 && !f_last) scale_qk(nch - 1, false);
    }

    // ---------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// Whether every chunk of this CTA's sequence (segment) carries its gates as row
// weights: no gate is exactly 0, and within every chunk the decay w_0 =
// e^{b_last - b_0} (the product of the chunk's gates after its first) stays
// above e^{kFastGateLog + 4}, a margin over the producer's own test (gate_products),
// whose sums run in another order.  All threads take part; the result is the
// same for every thread.
template <bool PLAIN, bool ITEMS>
__device__ __forceinline__ bool cta_all_fast(const PrefillTcArgs &args)
{
    const CtaUnit u = PLAIN ? CtaUnit{(int)blockIdx.z, 0, 1, 0, -1} : cta_unit<ITEMS>(args);
    const int h = blockIdx.y, b = u.b, seg = u.seg;
    const int bh = b * args.H + h;
    const bool varlen = args.cu_seqlens != nullptr;
    int seq0 = 0, T = args.T;
    bool ok = args.alpha != nullptr;
    if (varlen) {
        seq0 = args.cu_seqlens[b];
        const int seq1 = args.cu_seqlens[b + 1];
        if (seq0 < 0 || seq1 < seq0 || seq1 > args.T) ok = false;   // the general body records the error
        T = seq1 - seq0;
    }
    const int nch_all = ok ? (T + kC - 1) / kC : 0;
    const int c0 = seg * u.len;
    const int nch = u.nseg > 1 ? min(u.len, nch_all - c0) : nch_all;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int c = warp; ok && c < nch; c += kThreads / 32) {
        const int t0 = (c0 + c) * kC + 2 * lane;
        float a0 = 1.f, a1 = 1.f;
        if (t0 < T) a0 = args.alpha[varlen ? (size_t)(seq0 + t0) * args.H + h : (size_t)bh * T + t0];
        if (t0 + 1 < T) a1 = args.alpha[varlen ? (size_t)(seq0 + t0 + 1) * args.H + h : (size_t)bh * T + t0 + 1];
        const bool zero = !(a0 > 0.f) || !(a1 > 0.f);
        float lsum = (lane == 0 ? 0.f : logf(fmaxf(a0, 1e-30f))) + logf(fmaxf(a1, 1e-30f));   // rows 1..63
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
        ok = !__any_sync(0xffffffffu, zero) && lsum >= kFastGateLog + 4.f;
    }
    return __syncthreads_and(ok) != 0;
}

template <bool GATED, int DVS, bool PLAIN, bool SAVE = false, bool ITEMS = false>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                  const __grid_constant__ CUtensorMap map_v, const PrefillTcArgs args)
{
    // a row of the varlen plan's item table beyond its items: no work (every CTA
    // of a cluster has the same row)
    if (ITEMS && args.items[blockIdx.z].x < 0) return;
    if constexpr (GATED && Cfg<GATED, DVS>::kHead) {
        if (cta_all_fast<PLAIN, ITEMS>(args)) {
            prefill_body<GATED, DVS, true, PLAIN, SAVE, ITEMS>(map_q, map_k, map_v, args);
            return;
        }
    }
    prefill_body<GATED, DVS, false, PLAIN, SAVE, ITEMS>(map_q, map_k, map_v, args);
}

}  // namespace

cudaError_t launch_prefill_tc(const CUtensorMap &map_q, const CUtensorMap &map_k, const CUtensorMap &map_v,
                              const PrefillTcArgs &a, int B, bool gated, int dvs, cudaStream_t stream,
                              int grid_z)
{
    if (dvs != 64 && dvs != 128) return cudaErrorInvalidValue;
    if (a.items && (grid_z < 1 || !a.seq_info || !a.seg_len || !a.cu_seqlens || !a.S_start))
        return cudaErrorInvalidValue;
    const dim3 grid(a.dv / dvs, a.H, a.items ? grid_z : B * a.nseg);
    using KernFn = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const PrefillTcArgs);
    // plain: [B, H, T, d] inputs and one segment per head; save: the general body
    // with the training stores
    const bool save = a.d_out != nullptr || a.bwd_states != nullptr;
    const bool plain = !save && a.cu_seqlens == nullptr && a.nseg == 1 && a.S_start == nullptr && !a.items;
    // items: the varlen plan's segments (never with the training stores)
    if (a.items && save) return cudaErrorInvalidValue;
    const int v = (gated ? 1 : 0) + (dvs == 128 ? 2 : 0) + (save ? 8 : a.items ? 12 : plain ? 4 : 0);
    static const KernFn kerns[16] = {
        prefill_tc_kernel<false, 64, false>,       prefill_tc_kernel<true, 64, false>,
        prefill_tc_kernel<false, 128, false>,      prefill_tc_kernel<true, 128, false>,
        prefill_tc_kernel<false, 64, true>,        prefill_tc_kernel<true, 64, true>,
        prefill_tc_kernel<false, 128, true>,       prefill_tc_kernel<true, 128, true>,
        prefill_tc_kernel<false, 64, false, true>, prefill_tc_kernel<true, 64, false, true>,
        prefill_tc_kernel<false, 128, false, true>, prefill_tc_kernel<true, 128, false, true>,
        prefill_tc_kernel<false, 64, false, false, true>, prefill_tc_kernel<true, 64, false, false, true>,
        prefill_tc_kernel<false, 128, false, false, true>, prefill_tc_kernel<true, 128, false, false, true>};
    static const uint32_t bytes[4] = {smem_bytes<false, 64>(), smem_bytes<true, 64>(), smem_bytes<false, 128>(),
                                      smem_bytes<true, 128>()};
    // The attribute is set once per device (not during stream capture of later calls).
    static OncePerDevice attr_set[16];
    const cudaError_t e = set_smem_once(kerns[v], bytes[v & 3], attr_set[v]);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = bytes[v & 3];
    cfg.stream = stream;
    // the dv slices of a head (and segment) form a cluster
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = grid.x;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kerns[v], map_q, map_k, map_v, a);
}

}  // namespace la
