// backward.cu -- gradients of the gated linear-attention recurrence, in FP32 on
// CUDA cores.
//
// The pages give no backward formula; these kernels apply the chain rule to the
// recurrence of "Linear attention：把历史写进状态" (hs-black.github.io/posts/linear-attention),
// sections "公式里的每个维度" and "加一个门：让旧记忆逐渐淡出".  With q~ = phi(q),
// k~ = phi(k), y_t = n_t / d_t, n_t = S_t^T q~_t, d_t = q~_t . z_t + eps:
//   dn_t = dy_t / d_t,   dd_t = -(dy_t . y_t) / d_t
//   G_t = q~_t dn_t^T + alpha_{t+1} G_{t+1},   g_t = dd_t q~_t + alpha_{t+1} g_{t+1}
//   dq~_t = S_t dn_t + dd_t z_t,   dk~_t = G_t v_t + g_t,   dv_t = G_t^T k~_t
//   dS0 = alpha_1 G_1,   dz0 = alpha_1 g_1
// and, for the gates, with A_t the running sum of log alpha (the state terms
// depend on alpha only through e^{A_t} on the read side and e^{-A_s} on the
// write side):
//   dL/d log alpha_u = sum_{t >= u} (q~_t . dq~_t - k~_t . dk~_t) + <dS_T, S_T> + <dz_T, z_T>.
//
// d_t comes from a pass over (head, 32 features) warps that runs z's recurrence,
// dd_t from a bandwidth-bound pass over tokens.
// Each of dq, dk and dv is a gated rank-1 recurrence with a read that does not
// feed back into the state, so the three are one kernel in three modes:
//   kFwdDq: forward in time, one column per feature i, state S[i, :] and z_i;
//   kRevDk: reverse in time, one column per feature i, state G[i, :] and g_i;
//   kRevDv: reverse in time, one column per value j, state G[:, j].
// A CTA holds 32 columns; a lane holds L/8 state rows of two columns, the row
// groups interleaved in blocks of 4 as in the delta-rule kernel.  A lane keeps
// its partial reads of 8 tokens (2 columns each) and reduce-scatters them over
// the 8 row groups at once (14 shuffles per 8 tokens), after which row-group
// lane g holds both column totals of the group's token g.  Tokens come 32 at a
// time: the TMA unit copies a block's two vector rows (contiguous) and its two
// column slices into a double-buffered raw stage two blocks ahead, and the CTA
// converts a landed block once to FP32, already transformed (phi, dy / d_t).
// Finally a pass of one CTA per head turns the per-token terms into dalpha.

#include "side_lane.h"
#include "tc_common.cuh"

#include <cuda_bf16.h>

namespace la {
namespace {

constexpr int kBT = 32;          // tokens per staged block
constexpr int kBWarps = 4;
constexpr int kBThreads = 32 * kBWarps;
constexpr int kBCols = 32;       // columns per CTA

enum Mode { kFwdDq = 0, kRevDk = 1, kRevDv = 2 };

// phi and its derivative with the hardware exponential: for the arguments
// x <= 0 where it is used, the relative error is about 2.4e-7 + 6e-8 |x| (the
// rounding of x log2 e and of the base-2 exponential), far inside the
// backward's tolerance
__device__ __forceinline__ float phi_f(float x) { return x > 0.f ? x + 1.f : __expf(x); }
__device__ __forceinline__ float dphi_f(float x) { return x > 0.f ? 1.f : __expf(x); }

__device__ __forceinline__ float2 lo2(float4 a) { return make_float2(a.x, a.y); }
__device__ __forceinline__ float2 hi2(float4 a) { return make_float2(a.z, a.w); }

// ------------------------------------------------------------ d_t and dd_t

// z_t and the feature sum of d_t, in three fully parallel steps over segments of
// kZLen tokens (one warp per (b, h, segment); lane l holds features 4l .. 4l+3, so
// that a warp reads whole 256-byte token rows; at r < 128 the upper lanes hold
// none).  z_t = alpha_t z_{t-1} + phi(k_t) is affine in z: bwd_zmap_kernel runs
// each segment from z = 0, which gives its map z -> P z + zs; bwd_zscan_kernel
// applies the maps in order to z0 and writes the state entering every segment;
// bwd_zdot_kernel runs each segment again from there.  Tokens go in batches of
// ZB(Tin) whose loads are all issued before the recurrence uses them; the
// products q~_{t,i} z_{t,i} of a batch are summed over the warp's features by a
// reduce-scatter across the lanes (lane l ends with token l mod ZB) and written
// to d_acc[t].
constexpr int kZLen = 128;       // tokens per segment
constexpr int kZWarps = 8;       // warps (segments) per CTA

template <typename Tin> struct ZBatch { static constexpr int n = 16; };
template <> struct ZBatch<float> { static constexpr int n = 8; };

// Four adjacent features of one token row, raw.
__device__ __forceinline__ uint2 load_quad(const __nv_bfloat16 *p) { return *reinterpret_cast<const uint2 *>(p); }
__device__ __forceinline__ float4 load_quad(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ float4 unpack_quad(uint2 raw)
{
    return make_float4(bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y));
}
__device__ __forceinline__ float4 unpack_quad(float4 raw) { return raw; }

// Sums v[0..NB) over the 32 lanes: afterwards v[0] of lane l holds the total of
// index l mod NB.  Each halving step swaps the half of the values that a lane
// gives away with its partner lane and adds the half it keeps.
template <int NB>
__device__ __forceinline__ float lane_reduce_scatter(float (&v)[NB], int lane)
{
#pragma unroll
    for (int s = NB / 2; s >= 1; s >>= 1) {
        const bool up = (lane & s) != 0;
#pragma unroll
        for (int i = 0; i < s; ++i) {
            const float give = up ? v[i] : v[i + s];
            const float keep = up ? v[i + s] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, give, s);
        }
    }
#pragma unroll
    for (int s = NB; s < 32; s <<= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], s);
    return v[0];
}

// The warp's place: segment, head, first feature, whether its lane holds features.
struct ZWarp {
    int seg, bh, i0, ta, te;
    bool live, valid;
};

__device__ __forceinline__ ZWarp z_warp(int r, int T, int nzs)
{
    ZWarp w;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    w.seg = blockIdx.y * kZWarps + warp;
    w.bh = blockIdx.x;
    w.i0 = 4 * lane;
    w.live = w.i0 < r;
    w.valid = w.seg < nzs;
    w.ta = min(T, w.seg * kZLen);
    w.te = min(T, w.ta + kZLen);
    return w;
}

// z <- a z + phi(k) for four features.
__device__ __forceinline__ void z_step(float4 &z, float a, float4 k)
{
    z.x = a * z.x + phi_f(k.x);
    z.y = a * z.y + phi_f(k.y);
    z.z = a * z.z + phi_f(k.z);
    z.w = a * z.w + phi_f(k.w);
}

// 1: the map (P, zs) of every segment; zs [B*H][nzs][r], P [B*H][nzs].
template <typename Tin>
__global__ void __launch_bounds__(32 * kZWarps)
bwd_zmap_kernel(const Tin *__restrict__ k, const float *__restrict__ alpha, int T, int r, int nzs,
                float *__restrict__ zs_out, float *__restrict__ P_out)
{
    constexpr int NB = ZBatch<Tin>::n;
    using Raw = decltype(load_quad(static_cast<const Tin *>(nullptr)));
    const ZWarp w = z_warp(r, T, nzs);
    if (!w.valid) return;   // whole warps only
    const int lane = threadIdx.x & 31;
    const Tin *kp = k + (size_t)w.bh * T * r + w.i0;
    const float *ap = alpha ? alpha + (size_t)w.bh * T : nullptr;
    float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    float P = 1.f;
    for (int t0 = w.ta; t0 < w.te; t0 += NB) {
        const int nt = min(NB, w.te - t0);
        Raw kr[NB];
#pragma unroll
        for (int t = 0; t < NB; ++t) kr[t] = (t < nt && w.live) ? load_quad(kp + (size_t)(t0 + t) * r) : Raw{};
        const float al = (ap && lane < nt) ? ap[t0 + lane] : 1.f;
#pragma unroll
        for (int t = 0; t < NB; ++t) {
            const float a = __shfl_sync(0xffffffffu, al, t);
            if (t < nt) {
                z_step(z, a, unpack_quad(kr[t]));
                P *= a;
            }
        }
    }
    const size_t sidx = (size_t)w.bh * nzs + w.seg;
    if (w.live) *reinterpret_cast<float4 *>(zs_out + sidx * r + w.i0) = z;
    if (lane == 0) P_out[sidx] = P;
}

// 2: the state entering every segment, z_start [B*H][nzs][r]: one warp per (b, h)
// applies the maps in order to z0, loading 8 of them at a time.
__global__ void __launch_bounds__(32)
bwd_zscan_kernel(const float *__restrict__ z0, const float *__restrict__ zs, const float *__restrict__ P, int r,
                 int nzs, float *__restrict__ z_start)
{
    const int lane = threadIdx.x, bh = blockIdx.x, i0 = 4 * lane;
    const bool live = i0 < r;
    float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    if (z0 && live) {   // z0 is only 4-byte aligned
        const float *zp = z0 + (size_t)bh * r + i0;
        z = make_float4(zp[0], zp[1], zp[2], zp[3]);
    }
    for (int s0 = 0; s0 < nzs; s0 += 8) {
        float4 m[8];
        float p[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const size_t sidx = (size_t)bh * nzs + s0 + i;
            const bool in = s0 + i < nzs;
            m[i] = (in && live) ? *reinterpret_cast<const float4 *>(zs + sidx * r + i0) : make_float4(0.f, 0.f, 0.f, 0.f);
            p[i] = in ? P[sidx] : 1.f;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (s0 + i >= nzs) break;
            if (live) *reinterpret_cast<float4 *>(z_start + ((size_t)bh * nzs + s0 + i) * r + i0) = z;
            z.x = p[i] * z.x + m[i].x;
            z.y = p[i] * z.y + m[i].y;
            z.z = p[i] * z.z + m[i].z;
            z.w = p[i] * z.w + m[i].w;
        }
    }
}

// 3: every segment again from its entering state, with the products summed into
// d_acc (one warp holds all of a token's features: a plain store).
template <typename Tin>
__global__ void __launch_bounds__(32 * kZWarps)
bwd_zdot_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k, const float *__restrict__ alpha, int T, int r,
                int nzs, const float *__restrict__ z_start, float *__restrict__ d_acc)
{
    constexpr int NB = ZBatch<Tin>::n;
    using Raw = decltype(load_quad(static_cast<const Tin *>(nullptr)));
    const ZWarp w = z_warp(r, T, nzs);
    if (!w.valid) return;   // whole warps only
    const int lane = threadIdx.x & 31;
    const Tin *kp = k + (size_t)w.bh * T * r + w.i0, *qp = q + (size_t)w.bh * T * r + w.i0;
    const float *ap = alpha ? alpha + (size_t)w.bh * T : nullptr;
    float4 z = w.live ? *reinterpret_cast<const float4 *>(z_start + ((size_t)w.bh * nzs + w.seg) * r + w.i0)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
    for (int t0 = w.ta; t0 < w.te; t0 += NB) {
        const int nt = min(NB, w.te - t0);
        Raw kr[NB], qr[NB];
#pragma unroll
        for (int t = 0; t < NB; ++t) {
            kr[t] = (t < nt && w.live) ? load_quad(kp + (size_t)(t0 + t) * r) : Raw{};
            qr[t] = (t < nt && w.live) ? load_quad(qp + (size_t)(t0 + t) * r) : Raw{};
        }
        const float al = (ap && lane < nt) ? ap[t0 + lane] : 1.f;
        float prod[NB];
#pragma unroll
        for (int t = 0; t < NB; ++t) {
            const float a = __shfl_sync(0xffffffffu, al, t);
            prod[t] = 0.f;
            if (t < nt) {
                z_step(z, a, unpack_quad(kr[t]));
                const float4 qv = unpack_quad(qr[t]);
                if (w.live) prod[t] = phi_f(qv.x) * z.x + phi_f(qv.y) * z.y + phi_f(qv.z) * z.z + phi_f(qv.w) * z.w;
            }
        }
        const float sum = lane_reduce_scatter<NB>(prod, lane);
        if (lane < nt) d_acc[(size_t)w.bh * T + t0 + lane] = sum;
    }
}

// d_t = d_src[t] + eps and dd_t = -(dy_t . y_t) / d_t: two tokens per warp step,
// 16 lanes per token, 16-byte loads.  d_src is d itself (the z pass's feature
// sums) or the forward's d_t (then eps = 0).
template <typename Tin>
__global__ void __launch_bounds__(256)
bwd_dd_kernel(const Tin *__restrict__ y, const Tin *__restrict__ dy, int dv, long long n, float eps,
              const float *d_src, float *d, float *__restrict__ dd)
{
    constexpr int kV = 16 / (int)sizeof(Tin);
    const int nch = dv / kV;
    const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
    const int lane = threadIdx.x & 31, hl = lane & 15;
    for (long long tok0 = warp * 2; tok0 < n; tok0 += nwarps * 2) {
        const long long tok = tok0 + (lane >> 4);
        float s = 0.f;
        if (tok < n) {
            for (int c = hl; c < nch; c += 16) {
                const size_t off = (size_t)tok * dv + (size_t)c * kV;
                const uint4 a = *reinterpret_cast<const uint4 *>(dy + off), b = *reinterpret_cast<const uint4 *>(y + off);
                if constexpr (sizeof(Tin) == 2) {
                    const uint32_t ua[4] = {a.x, a.y, a.z, a.w}, ub[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) s += bf16_lo(ua[e]) * bf16_lo(ub[e]) + bf16_hi(ua[e]) * bf16_hi(ub[e]);
                } else {
                    s += __uint_as_float(a.x) * __uint_as_float(b.x) + __uint_as_float(a.y) * __uint_as_float(b.y) +
                         __uint_as_float(a.z) * __uint_as_float(b.z) + __uint_as_float(a.w) * __uint_as_float(b.w);
                }
            }
        }
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (tok < n && hl == 0) {
            const float den = d_src[tok] + eps;
            d[tok] = den;
            dd[tok] = -s / den;
        }
    }
}

// ------------------------------------------------------- the three sweeps

template <typename Tin, int L>
struct RecSmem {
    // raw stages, written by the TMA unit: the block's rows of the two vector
    // sources, and its slices of the two column sources
    Tin rb[2][kBT][L];
    Tin rw[2][kBT][L];
    Tin ra[2][kBT][kBCols];
    Tin rx[2][kBT][kBCols];
    // the converted block
    float b[kBT][L];        // the rank-1 write's vector (b_t)
    float w[kBT][L];        // the read's vector (w_t)
    float a[kBT][kBCols];   // the write's per-column coefficient
    float x[kBT][kBCols];   // the column's own q or k (dq, dk: for phi and phi')
    float o[kBT][kBCols];   // outputs of the block
    float gam[kBT];         // gate applied to the state before this token's write
    float dd[kBT];          // dd_t
    float invd[kBT];        // 1 / d_t
    float sum[kBT];         // per-token sum over this CTA's columns (dalpha terms)
    uint64_t full[2];
    int flag;
};

struct RecArgs {
    const void *q, *k, *v, *dy;
    const float *alpha, *S0, *z0, *dS_T, *dz_T, *d, *dd;
    void *out;              // dq, dk or dv
    float *tok_sum;         // [B*H*T] dalpha terms (atomic adds), kFwdDq and kRevDk
    float *fin;             // [B*H] <dS_T, S_T> + <dz_T, z_T>, kFwdDq
    float *dS0, *dz0;       // kRevDk
    int *status;
    unsigned long long limit_ns;
    int H, T, r, dv;
};

enum Op { kPlain = 0, kPhi = 1, kScale = 2 };

// nrows rows of W elements (row stride W in both) from a raw block to FP32,
// transformed by op (kScale: times invd[row]); 8 (BF16) or 4 (FP32) per step.
template <typename Tin, int W, int op>
__device__ __forceinline__ void convert(const Tin *src, float *dst, int nrows, const float *invd)
{
    constexpr int kV = 16 / (int)sizeof(Tin), nch = W / kV;
    for (int c = threadIdx.x; c < nrows * nch; c += kBThreads) {
        const int t = c / nch;
        const uint4 u = reinterpret_cast<const uint4 *>(src)[c];
        float f[kV];
        if constexpr (sizeof(Tin) == 2) {
            const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                f[2 * e] = bf16_lo(w4[e]);
                f[2 * e + 1] = bf16_hi(w4[e]);
            }
        } else {
            f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
            f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
        }
        const float s = op == kScale ? invd[t] : 1.f;
#pragma unroll
        for (int e = 0; e < kV; ++e) f[e] = op == kPhi ? phi_f(f[e]) : (op == kScale ? f[e] * s : f[e]);
#pragma unroll
        for (int e = 0; e < kV; e += 4)
            *reinterpret_cast<float4 *>(dst + (size_t)c * kV + e) = make_float4(f[e], f[e + 1], f[e + 2], f[e + 3]);
    }
}

__device__ __forceinline__ void store8(__nv_bfloat16 *p, const float *f)
{
    *reinterpret_cast<uint4 *>(p) = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                                               pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
}
__device__ __forceinline__ void store8(float *p, const float *f)
{
    reinterpret_cast<float4 *>(p)[0] = make_float4(f[0], f[1], f[2], f[3]);
    reinterpret_cast<float4 *>(p)[1] = make_float4(f[4], f[5], f[6], f[7]);
}

template <typename Tin, int Mode, int L>
__global__ void __launch_bounds__(kBThreads)
rec_kernel(RecArgs p)
{
    constexpr int F = L / 32;                   // float4 row blocks per lane
    constexpr int kEl = (int)sizeof(Tin);
    extern __shared__ __align__(16) unsigned char smem_raw[];
    RecSmem<Tin, L> &sm = *reinterpret_cast<RecSmem<Tin, L> *>(smem_raw);
    const int T = p.T, r = p.r, dv = p.dv;
    const int ncol_total = Mode == kRevDv ? dv : r;
    const int nslice = ncol_total / kBCols;
    const int bh = blockIdx.x / nslice, c0 = (blockIdx.x % nslice) * kBCols;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, jj = lane & 3;
    const int jl = warp * 8 + 2 * jj;           // first of the lane's two columns (local)
    const Tin *qi = static_cast<const Tin *>(p.q), *ki = static_cast<const Tin *>(p.k);
    const Tin *vi = static_cast<const Tin *>(p.v), *dyi = static_cast<const Tin *>(p.dy);
    Tin *out = static_cast<Tin *>(p.out);
    // the sources of the staged arrays
    const Tin *srcB = Mode == kFwdDq ? vi : (Mode == kRevDk ? dyi : qi);   // rows of length L
    const Tin *srcW = Mode == kFwdDq ? dyi : (Mode == kRevDk ? vi : ki);
    const Tin *srcA = Mode == kFwdDq ? ki : (Mode == kRevDk ? qi : dyi);   // rows of length ncol_total
    const Tin *srcX = Mode == kFwdDq ? qi : ki;
    const int nblk = (T + kBT - 1) / kBT;
    auto block_of = [&](int bi) { return Mode == kFwdDq ? bi : nblk - 1 - bi; };
    Ctx cx{&sm.flag, p.limit_ns, p.status};

    if (tid == 0) {
        mbar_init(&sm.full[0], 1);
        mbar_init(&sm.full[1], 1);
        sm.flag = 0;
        fence_mbarrier_init();
    }
    __syncthreads();

    // Warp 0 starts the copies of the bi-th block in processing order into stage bi & 1.
    auto issue = [&](int bi) {
        const int st = bi & 1, t0 = block_of(bi) * kBT, nt = min(kBT, T - t0);
        const size_t tok0 = (size_t)bh * T + t0;
        const uint32_t rowbytes = (uint32_t)(nt * L * kEl), colbytes = (uint32_t)(kBCols * kEl);
        const uint32_t ncolsrc = Mode == kRevDv ? 1u : 2u;
        if (lane == 0) mbar_arrive_expect_tx(&sm.full[st], 2 * rowbytes + ncolsrc * nt * colbytes);
        __syncwarp();
        if (lane == 0) bulk_load(&sm.rb[st][0][0], srcB + tok0 * L, rowbytes, &sm.full[st]);
        if (lane == 1) bulk_load(&sm.rw[st][0][0], srcW + tok0 * L, rowbytes, &sm.full[st]);
        if (lane < nt) {
            const size_t off = (tok0 + lane) * (size_t)ncol_total + c0;
            bulk_load(&sm.ra[st][lane][0], srcA + off, colbytes, &sm.full[st]);
            if (Mode != kRevDv) bulk_load(&sm.rx[st][lane][0], srcX + off, colbytes, &sm.full[st]);
        }
    };
    if (warp == 0) {
        if (nblk > 0) issue(0);
        if (nblk > 1) issue(1);
    }
    // per-token scalars of the bi-th block, one token per thread of warp 0
    struct Scalars { float gam, dd, invd; };
    auto fetch = [&](int bi) -> Scalars {
        const int t0 = block_of(bi) * kBT, nt = min(kBT, T - t0);
        Scalars sc{1.f, 0.f, 1.f};
        if (tid < nt) {
            const size_t tok = (size_t)bh * T + t0 + tid;
            // forward: alpha_t acts before token t's write; reverse: alpha_{t+1} (1 after the last token)
            const int ta = Mode == kFwdDq ? t0 + tid : t0 + tid + 1;
            sc.gam = (p.alpha && ta < T) ? p.alpha[(size_t)bh * T + ta] : 1.f;
            sc.dd = Mode == kRevDv ? 0.f : p.dd[tok];
            sc.invd = 1.f / p.d[tok];
        }
        return sc;
    };
    Scalars sc = fetch(0);

    // state: X[m][c][h] holds rows 4 (8 m + g) + 2h, + 1 of column c0 + jl + c
    float2 X[F][2][2];
    float e[2] = {0.f, 0.f};                    // z_i (kFwdDq) or g_i (kRevDk) of the two columns
#pragma unroll
    for (int m = 0; m < F; ++m)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int row = 4 * (8 * m + g) + 2 * h;
            float2 u = make_float2(0.f, 0.f), w2 = u;   // (row, columns 0/1), (row + 1, ...)
            const float *s0 = Mode == kFwdDq ? p.S0 : p.dS_T;
            if (s0 && Mode != kRevDv) {
                // state of column (feature) c = row c of S0 or dS_T, length dv
                const float *s = s0 + (size_t)bh * r * dv;
                u = make_float2(s[(size_t)(c0 + jl) * dv + row], s[(size_t)(c0 + jl + 1) * dv + row]);
                w2 = make_float2(s[(size_t)(c0 + jl) * dv + row + 1], s[(size_t)(c0 + jl + 1) * dv + row + 1]);
            } else if (s0) {
                // state of column (value) c = column c of dS_T, length r
                const float *s = s0 + (size_t)bh * r * dv;
                u = *reinterpret_cast<const float2 *>(s + (size_t)row * dv + c0 + jl);
                w2 = *reinterpret_cast<const float2 *>(s + (size_t)(row + 1) * dv + c0 + jl);
            }
            X[m][0][h] = make_float2(u.x, w2.x);
            X[m][1][h] = make_float2(u.y, w2.y);
        }
    {
        const float *e0 = Mode == kFwdDq ? p.z0 : (Mode == kRevDk ? p.dz_T : nullptr);
        if (e0) {
            e[0] = e0[(size_t)bh * r + c0 + jl];
            e[1] = e0[(size_t)bh * r + c0 + jl + 1];
        }
    }

    // the outputs of a processed block: 8 columns per step, and the dalpha terms
    auto flush = [&](int bi) {
        const int t0 = block_of(bi) * kBT, nt = min(kBT, T - t0);
        for (int c = tid; c < nt * (kBCols / 8); c += kBThreads) {
            const int t = c / (kBCols / 8), ch = (c % (kBCols / 8)) * 8;
            store8(out + ((size_t)bh * T + t0 + t) * ncol_total + c0 + ch, &sm.o[t][ch]);
        }
        if (Mode != kRevDv && tid < nt) {
            const float v = sm.sum[tid];
            atomicAdd(&p.tok_sum[(size_t)bh * T + t0 + tid], Mode == kFwdDq ? v : -v);
        }
    };

    int bi = 0;
    for (; bi < nblk; ++bi) {
        const int st = bi & 1, nt = min(kBT, T - block_of(bi) * kBT);
        const bool ok = wait(cx, &sm.full[st], (bi >> 1) & 1);
        if (__syncthreads_or(!ok)) break;   // also: the previous block's compute has finished
        if (bi > 0) flush(bi - 1);
        if (tid < kBT) {
            sm.gam[tid] = sc.gam;
            sm.dd[tid] = sc.dd;
            sm.invd[tid] = sc.invd;
            sm.sum[tid] = 0.f;
        }
        __syncthreads();
        convert<Tin, L, Mode == kRevDv ? kPhi : (Mode == kRevDk ? kScale : kPlain)>(&sm.rb[st][0][0], &sm.b[0][0], nt,
                                                                                     sm.invd);
        convert<Tin, L, Mode == kRevDv ? kPhi : (Mode == kFwdDq ? kScale : kPlain)>(&sm.rw[st][0][0], &sm.w[0][0], nt,
                                                                                     sm.invd);
        convert<Tin, kBCols, Mode == kRevDv ? kScale : kPhi>(&sm.ra[st][0][0], &sm.a[0][0], nt, sm.invd);
        if (Mode != kRevDv) convert<Tin, kBCols, kPlain>(&sm.rx[st][0][0], &sm.x[0][0], nt, sm.invd);
        __syncthreads();                    // FP32 block ready; the raw stage is free again
        if (warp == 0 && bi + 2 < nblk) issue(bi + 2);
        if (bi + 1 < nblk) sc = fetch(bi + 1);

        // Tokens in groups of 8 (in processing order).  Each lane keeps its partial
        // reads of the group (8 tokens x 2 columns) and the scalar recurrence after
        // each token; one reduce-scatter over the 8 row groups then leaves row-group
        // lane g with both column totals of the group's token g.
        for (int s0 = 0; s0 < nt; s0 += 8) {
            float part[8][2], eh[8][2];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                part[u][0] = part[u][1] = 0.f;
                eh[u][0] = eh[u][1] = 0.f;
                if (s0 + u < nt) {   // warp-uniform
                    const int t = Mode == kFwdDq ? s0 + u : nt - 1 - (s0 + u);
                    const float gm = sm.gam[t];
                    const float2 a0 = make_float2(sm.a[t][jl], sm.a[t][jl]);
                    const float2 a1 = make_float2(sm.a[t][jl + 1], sm.a[t][jl + 1]);
                    const float4 *br = reinterpret_cast<const float4 *>(&sm.b[t][0]) + g;
                    const float4 *wr = reinterpret_cast<const float4 *>(&sm.w[t][0]) + g;
                    float2 r0a = make_float2(0.f, 0.f), r0b = r0a, r1a = r0a, r1b = r0a;
                    const float2 g2 = make_float2(gm, gm);
#pragma unroll
                    for (int m = 0; m < F; ++m) {
                        const float4 bb = br[8 * m], ww = wr[8 * m];
                        if (p.alpha) {
                            X[m][0][0] = __fmul2_rn(X[m][0][0], g2);
                            X[m][0][1] = __fmul2_rn(X[m][0][1], g2);
                            X[m][1][0] = __fmul2_rn(X[m][1][0], g2);
                            X[m][1][1] = __fmul2_rn(X[m][1][1], g2);
                        }
                        X[m][0][0] = __ffma2_rn(lo2(bb), a0, X[m][0][0]);
                        X[m][0][1] = __ffma2_rn(hi2(bb), a0, X[m][0][1]);
                        X[m][1][0] = __ffma2_rn(lo2(bb), a1, X[m][1][0]);
                        X[m][1][1] = __ffma2_rn(hi2(bb), a1, X[m][1][1]);
                        r0a = __ffma2_rn(X[m][0][0], lo2(ww), r0a);
                        r0b = __ffma2_rn(X[m][0][1], hi2(ww), r0b);
                        r1a = __ffma2_rn(X[m][1][0], lo2(ww), r1a);
                        r1b = __ffma2_rn(X[m][1][1], hi2(ww), r1b);
                    }
                    // the scalar recurrences: z_i += k~ (forward), g_i += dd q~ (reverse dk)
                    if (Mode == kFwdDq) {
                        e[0] = fmaf(gm, e[0], a0.x);
                        e[1] = fmaf(gm, e[1], a1.x);
                    } else if (Mode == kRevDk) {
                        const float ddt = sm.dd[t];
                        e[0] = fmaf(gm, e[0], ddt * a0.x);
                        e[1] = fmaf(gm, e[1], ddt * a1.x);
                    }
                    const float2 s0v = __fadd2_rn(r0a, r0b), s1v = __fadd2_rn(r1a, r1b);
                    part[u][0] = s0v.x + s0v.y;
                    part[u][1] = s1v.x + s1v.y;
                    eh[u][0] = e[0];
                    eh[u][1] = e[1];
                }
            }
            // reduce-scatter over lane bits 4, 3, 2 (row-group bits 2, 1, 0): each step
            // keeps the half of the tokens whose index bit matches the lane's bit
            const bool lb4 = lane & 16, lb3 = lane & 8, lb2 = lane & 4;
            float h4[4][2], h4e[4][2];
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const float keep = lb4 ? part[4 + u][c] : part[u][c], send = lb4 ? part[u][c] : part[4 + u][c];
                    h4[u][c] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
                    h4e[u][c] = lb4 ? eh[4 + u][c] : eh[u][c];
                }
            float h2[2][2], h2e[2][2];
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const float keep = lb3 ? h4[2 + u][c] : h4[u][c], send = lb3 ? h4[u][c] : h4[2 + u][c];
                    h2[u][c] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
                    h2e[u][c] = lb3 ? h4e[2 + u][c] : h4e[u][c];
                }
            float tot[2], ev[2];
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const float keep = lb2 ? h2[1][c] : h2[0][c], send = lb2 ? h2[0][c] : h2[1][c];
                tot[c] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
                ev[c] = lb2 ? h2e[1][c] : h2e[0][c];
            }
            // this lane's token of the group: u = g
            const bool have = s0 + g < nt;
            const int t = Mode == kFwdDq ? s0 + g : nt - 1 - (s0 + g);
            if (Mode == kRevDv) {                   // dv = G_t^T k~_t
                if (have) {
                    sm.o[t][jl] = tot[0];
                    sm.o[t][jl + 1] = tot[1];
                }
            } else {
                // dq~ = S_t dn_t + dd_t z_t, or dk~ = G_t v_t + g_t; then phi' and the dalpha term
                float ts = 0.f;
                if (have) {
                    const float ddt = Mode == kFwdDq ? sm.dd[t] : 1.f;
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const float dt = tot[c] + ddt * ev[c];
                        const float xv = sm.x[t][jl + c];
                        sm.o[t][jl + c] = dt * dphi_f(xv);
                        ts += phi_f(xv) * dt;
                    }
                }
                // the warp's 8 columns of this token: lanes jj = 0..3 of row group g
                ts += __shfl_xor_sync(0xffffffffu, ts, 1);
                ts += __shfl_xor_sync(0xffffffffu, ts, 2);
                if (have && jj == 0) atomicAdd(&sm.sum[t], ts);
            }
        }
    }

    if (bi < nblk) {
        // gave up waiting: let the copies already started land before the CTA exits
        if (tid == 0)
            for (int bb = bi; bb < nblk && bb < bi + 2; ++bb) mbar_wait(&sm.full[bb & 1], (bb >> 1) & 1, p.limit_ns);
        __syncthreads();
        return;
    }
    __syncthreads();
    if (nblk > 0) flush(nblk - 1);

    // final state terms
    if (Mode == kFwdDq && (p.dS_T || p.dz_T)) {
        // <dS_T, S_T> + <dz_T, z_T> over this CTA's rows of S
        float acc = 0.f;
        if (p.dS_T) {
            const float *s = p.dS_T + (size_t)bh * r * dv;
#pragma unroll
            for (int m = 0; m < F; ++m)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int row = 4 * (8 * m + g) + 2 * h;
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        acc += X[m][c][h].x * s[(size_t)(c0 + jl + c) * dv + row];
                        acc += X[m][c][h].y * s[(size_t)(c0 + jl + c) * dv + row + 1];
                    }
                }
        }
        if (p.dz_T && g == 0)   // one lane per column pair adds z
            acc += e[0] * p.dz_T[(size_t)bh * r + c0 + jl] + e[1] * p.dz_T[(size_t)bh * r + c0 + jl + 1];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) atomicAdd(&p.fin[bh], acc);
    }
    if (Mode == kRevDk) {
        // dS0 = alpha_1 G_1, dz0 = alpha_1 g_1 (alpha_1: the first token's gate)
        const float a1 = p.alpha ? p.alpha[(size_t)bh * T] : 1.f;
        float *s = p.dS0 + (size_t)bh * r * dv;
#pragma unroll
        for (int m = 0; m < F; ++m)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int row = 4 * (8 * m + g) + 2 * h;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    s[(size_t)(c0 + jl + c) * dv + row] = a1 * X[m][c][h].x;
                    s[(size_t)(c0 + jl + c) * dv + row + 1] = a1 * X[m][c][h].y;
                }
            }
        if (g == 0) {
            p.dz0[(size_t)bh * r + c0 + jl] = a1 * e[0];
            p.dz0[(size_t)bh * r + c0 + jl + 1] = a1 * e[1];
        }
    }
}

// ------------------------------------------------------------------ dalpha

// dalpha_u = (fin + sum_{t >= u} tok_sum[t]) / alpha_u for every token of one
// (b, h), one CTA per (b, h), in tiles of kDaTile tokens from the end of the
// sequence: a tile is staged in shared memory (coalesced loads, padded so that
// the runs below hit distinct banks), each thread sums a run of kDaRun
// consecutive tokens, a suffix scan over the runs (warp shuffles, then across
// warps) gives every run the sum of what follows it, the run is walked
// backwards, and the tile leaves by coalesced stores.
constexpr int kDaThreads = 256, kDaTile = 4096, kDaRun = kDaTile / kDaThreads;
__device__ __forceinline__ int da_pad(int x) { return x + (x >> 5); }

__global__ void __launch_bounds__(kDaThreads)
bwd_dalpha_kernel(const float *__restrict__ tok_sum, const float *__restrict__ fin, const float *__restrict__ alpha,
                  int T, float *__restrict__ dalpha)
{
    __shared__ float buf[kDaTile + kDaTile / 32];
    __shared__ float wsum[kDaThreads / 32];
    const int bh = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float *ts = tok_sum + (size_t)bh * T, *al = alpha + (size_t)bh * T;
    float *out = dalpha + (size_t)bh * T;
    float carry = fin[bh];   // the final-state term plus every later tile
    for (int tile = (T + kDaTile - 1) / kDaTile - 1; tile >= 0; --tile) {
        const int t0 = tile * kDaTile, n = min(kDaTile, T - t0);
        for (int x = tid; x < kDaTile; x += kDaThreads) buf[da_pad(x)] = x < n ? ts[t0 + x] : 0.f;
        __syncthreads();
        float run = 0.f;
#pragma unroll
        for (int j = 0; j < kDaRun; ++j) run += buf[da_pad(tid * kDaRun + j)];
        float suf = run;   // runs tid .. the warp's last
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float v = __shfl_down_sync(0xffffffffu, suf, o);
            if (lane + o < 32) suf += v;
        }
        if (lane == 0) wsum[warp] = suf;
        __syncthreads();
        float c = carry + (suf - run);
        for (int w = warp + 1; w < kDaThreads / 32; ++w) c += wsum[w];
#pragma unroll
        for (int j = kDaRun - 1; j >= 0; --j) {
            const int x = da_pad(tid * kDaRun + j);
            c += buf[x];
            buf[x] = c;
        }
        __syncthreads();
        for (int x = tid; x < n; x += kDaThreads) out[t0 + x] = buf[da_pad(x)] / al[t0 + x];
#pragma unroll
        for (int w = 0; w < kDaThreads / 32; ++w) carry += wsum[w];
        __syncthreads();   // before the next tile reuses buf and wsum
    }
}

template <typename Tin, int Mode>
cudaError_t launch_rec(const RecArgs &a, int B, int L, cudaStream_t stream)
{
    const int ncol = Mode == kRevDv ? a.dv : a.r;
    const unsigned grid = (unsigned)((long long)B * a.H * (ncol / kBCols));
    auto go = [&](auto kern, size_t bytes) -> cudaError_t {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
        if (e != cudaSuccess) return e;
        kern<<<grid, kBThreads, bytes, stream>>>(a);
        return cudaGetLastError();
    };
    switch (L) {
    case 32: return go(rec_kernel<Tin, Mode, 32>, sizeof(RecSmem<Tin, 32>));
    case 64: return go(rec_kernel<Tin, Mode, 64>, sizeof(RecSmem<Tin, 64>));
    case 128: return go(rec_kernel<Tin, Mode, 128>, sizeof(RecSmem<Tin, 128>));
    default: return cudaErrorInvalidValue;
    }
}

template <typename Tin>
cudaError_t launch_bwd_t(const BackwardArgs &a, int B, cudaStream_t stream)
{
    const int BH = B * a.H;
    const size_t n = (size_t)BH * a.T;
    float *d = a.ws, *dd = d + n, *tok_sum = dd + n, *fin = tok_sum + n;
    cudaError_t e;
    // With the tensor-core sweeps over sequence segments, the state passes and
    // their scans go on a side stream: the forward pass (k, v only) beside the z
    // pass and d_t; the reversed pass (which needs d_t) beside the dq sweep.
    const bool segmented = sizeof(Tin) == 2 && a.maps && a.nseg > 1;
    SideLane *side = segmented ? side_lane() : nullptr;
    const cudaStream_t ss = side ? side->stream : stream;
    if (side) {   // the side work comes after everything the caller enqueued before
        if ((e = cudaEventRecord(side->ev[0], stream)) != cudaSuccess) return e;
        if ((e = cudaStreamWaitEvent(ss, side->ev[0], 0)) != cudaSuccess) return e;
    }
    const size_t state = (size_t)128 * 128 + 128;
    const size_t a_floats = ((size_t)a.nsub * BH * 4 + 255) / 256 * 64;
    const size_t pass_floats = a_floats + (size_t)a.nsub * BH * state + (size_t)a.nseg * BH * state;
    StateTcArgs sa;
    const float *Sf = a.states_in;
    if (segmented) {
        // the states entering each segment: the prefill's state pass and scan in
        // forward time (for dq), and (below) their reversed form over (phi(q), dn,
        // dd) from dS_T, dz_T (for dk and dv); each pass's workspace is A
        // [nsub][BH] (256-byte aligned), the parts' maps [nsub][BH][state], the
        // segment states [nseg][BH][state]
        sa.alpha = a.alpha; sa.H = a.H; sa.T = a.T; sa.dv = 128;
        sa.nsub = a.nsub; sa.sub_per_seg = a.sub_per_seg; sa.sub_chunks = a.sub_chunks;
        sa.seg_chunks = a.seg_chunks; sa.status = a.status; sa.wait_limit_ns = a.limit_ns;
        // forward: segments 0 .. nseg-2 over (phi(k), v), unless the forward kept them
        if (!Sf) {
            float *pf = a.seg_ws;
            sa.A = pf; sa.dS = pf + a_floats; sa.seg_first = 0;
            if ((e = launch_state_tc(a.maps[1], a.maps[2], sa, B, a.alpha != nullptr, 128, ss)) != cudaSuccess) return e;
            float *sf = pf + a_floats + (size_t)a.nsub * BH * state;
            if ((e = launch_seg_scan(a.S0, a.z0, sa.A, sa.dS, sf, BH, 128, a.nsub, a.sub_per_seg, a.nseg, ss)) !=
                cudaSuccess)
                return e;
            Sf = sf;
            if (side && (e = cudaEventRecord(side->ev[3], ss)) != cudaSuccess) return e;
        }
    }
    // d accumulates the feature sums; tok_sum and fin accumulate dalpha terms
    if ((e = cudaMemsetAsync(a.ws, 0, sizeof(float) * (3 * n + BH), stream)) != cudaSuccess) return e;
    if (!a.d_in) {
        // z_t per segment of kZLen tokens: maps, scan, products
        const int nzs = (a.T + kZLen - 1) / kZLen;
        // zs and z_start are read as float4: they start on a 16-byte boundary (r is a multiple of 4)
        float *zP = fin + BH;
        float *zs = a.ws + (3 * n + BH + (size_t)BH * nzs + 3) / 4 * 4, *zst = zs + (size_t)BH * nzs * a.r;
        const dim3 grid((unsigned)BH, (nzs + kZWarps - 1) / kZWarps, 1);
        bwd_zmap_kernel<Tin><<<grid, 32 * kZWarps, 0, stream>>>(static_cast<const Tin *>(a.k), a.alpha, a.T, a.r, nzs, zs, zP);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        bwd_zscan_kernel<<<dim3((unsigned)BH, 1), 32, 0, stream>>>(a.z0, zs, zP, a.r, nzs, zst);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        bwd_zdot_kernel<Tin><<<grid, 32 * kZWarps, 0, stream>>>(static_cast<const Tin *>(a.q), static_cast<const Tin *>(a.k),
                                                                a.alpha, a.T, a.r, nzs, zst, d);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    // d_t = the feature sums + eps, or the forward's d_t as it stands
    bwd_dd_kernel<Tin><<<152 * 8, 256, 0, stream>>>(static_cast<const Tin *>(a.y), static_cast<const Tin *>(a.dy),
                                                      a.dv, (long long)n, a.d_in ? 0.f : a.eps,
                                                      a.d_in ? a.d_in : d, d, dd);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if constexpr (sizeof(Tin) == 2) {
        if (a.maps) {
            // the three sweeps on the tensor cores
            BwdTcArgs t;
            t.alpha = a.alpha; t.S0 = a.S0; t.z0 = a.z0; t.dS_T = a.dS_T; t.dz_T = a.dz_T;
            t.d = d; t.dd = dd;
            t.q = static_cast<const uint16_t *>(a.q); t.k = static_cast<const uint16_t *>(a.k);
            t.dq = static_cast<uint16_t *>(a.dq); t.dk = static_cast<uint16_t *>(a.dk);
            t.dv = static_cast<uint16_t *>(a.dv_out);
            t.tok_sum = a.alpha ? tok_sum : nullptr; t.fin = a.alpha ? fin : nullptr;
            t.dS0 = a.dS0; t.dz0 = a.dz0;
            t.H = a.H; t.T = a.T; t.status = a.status; t.limit_ns = a.limit_ns;
            if (segmented) {
                // reversed: segments 1 .. nseg-1 over (phi(q), dy / d, dd), once d_t is done
                if (side) {
                    if ((e = cudaEventRecord(side->ev[1], stream)) != cudaSuccess) return e;
                    if ((e = cudaStreamWaitEvent(ss, side->ev[1], 0)) != cudaSuccess) return e;
                }
                float *pr = a.seg_ws + pass_floats;
                sa.A = pr; sa.dS = pr + a_floats; sa.seg_first = 1; sa.d = d; sa.dd = dd;
                if ((e = launch_state_tc(a.maps[0], a.maps[3], sa, B, a.alpha != nullptr, 128, ss, true)) != cudaSuccess)
                    return e;
                float *Sr = pr + a_floats + (size_t)a.nsub * BH * state;
                if ((e = launch_seg_scan(a.dS_T, a.dz_T, sa.A, sa.dS, Sr, BH, 128, a.nsub, a.sub_per_seg, a.nseg, ss,
                                         true)) != cudaSuccess)
                    return e;
                if (side && (e = cudaEventRecord(side->ev[2], ss)) != cudaSuccess) return e;
                t.nseg = a.nseg; t.seg_chunks = a.seg_chunks; t.seg_state_f = Sf; t.seg_state_r = Sr;
                // dq once the forward states are there; dk and dv once the reversed ones are
                if (side && !a.states_in && (e = cudaStreamWaitEvent(stream, side->ev[3], 0)) != cudaSuccess) return e;
                if ((e = launch_bwd_tc(a.maps, t, B, a.alpha != nullptr, stream, 0, 1)) != cudaSuccess) return e;
                if (side && (e = cudaStreamWaitEvent(stream, side->ev[2], 0)) != cudaSuccess) return e;
                if ((e = launch_bwd_tc(a.maps, t, B, a.alpha != nullptr, stream, 1, 3)) != cudaSuccess) return e;
            } else if ((e = launch_bwd_tc(a.maps, t, B, a.alpha != nullptr, stream)) != cudaSuccess) {
                return e;
            }
            if (a.alpha && a.dalpha) {
                bwd_dalpha_kernel<<<BH, kDaThreads, 0, stream>>>(tok_sum, fin, a.alpha, a.T, a.dalpha);
                if ((e = cudaGetLastError()) != cudaSuccess) return e;
            }
            return cudaSuccess;
        }
    }
    RecArgs p;
    p.q = a.q; p.k = a.k; p.v = a.v; p.dy = a.dy;
    p.alpha = a.alpha; p.S0 = a.S0; p.z0 = a.z0; p.dS_T = a.dS_T; p.dz_T = a.dz_T; p.d = d; p.dd = dd;
    p.tok_sum = tok_sum; p.fin = fin; p.dS0 = a.dS0; p.dz0 = a.dz0;
    p.status = a.status; p.limit_ns = a.limit_ns;
    p.H = a.H; p.T = a.T; p.r = a.r; p.dv = a.dv;
    p.out = a.dq;
    if ((e = launch_rec<Tin, kFwdDq>(p, B, a.dv, stream)) != cudaSuccess) return e;
    p.out = a.dk;
    if ((e = launch_rec<Tin, kRevDk>(p, B, a.dv, stream)) != cudaSuccess) return e;
    p.out = a.dv_out;
    if ((e = launch_rec<Tin, kRevDv>(p, B, a.r, stream)) != cudaSuccess) return e;
    if (a.alpha && a.dalpha) {
        bwd_dalpha_kernel<<<BH, kDaThreads, 0, stream>>>(tok_sum, fin, a.alpha, a.T, a.dalpha);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

// d, dd, tok_sum [B*H*T], fin [B*H], then the z pass's segment maps: P [B*H][nzs],
// zs and z_start [B*H][nzs][r] (r <= 128)
size_t backward_workspace_floats(int B, int H, int T)
{
    const size_t BH = (size_t)B * H, nzs = ((size_t)T + kZLen - 1) / kZLen;
    return BH * ((size_t)3 * T + 1) + BH * nzs * (1 + 2 * 128) + 4;
}

cudaError_t launch_backward(const BackwardArgs &a, int B, bool bf16, cudaStream_t stream)
{
    return bf16 ? launch_bwd_t<__nv_bfloat16>(a, B, stream) : launch_bwd_t<float>(a, B, stream);
}

}  // namespace la
