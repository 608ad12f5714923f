// delta.cu -- the delta-rule memory on CUDA cores, token by token.
//
// Method ("Linear attention：把历史写进状态", hs-black.github.io/posts/linear-attention,
// section "Delta rule：先读旧答案，再写误差"): a fast-weight memory without the
// normaliser.  Each token reads the memory's current answer for its key, writes
// back beta times the error, and the query reads the updated memory:
//     p_t = S_{t-1}^T k_t,   S_t = S_{t-1} + beta_t k_t (v_t - p_t)^T,   y_t = S_t^T q_t.
// The pages give the update and say that a block form needs its own algorithm
// (section "训练时，状态更新也能按块并行"); this kernel runs the recurrence as
// written, in FP32 with the state in registers.
//
// Every column j of S is an independent recurrence: p_j, the error and the
// update of column j involve column j alone.  So the value columns are split
// over CTAs and warps with no exchange between them; only the sums over the r
// rows (S^T k and S^T q) are reduced, inside a warp.
//
// The limit of this token loop is shared-memory bandwidth: every lane needs the
// token's k and q values for each of its rows, and a warp-wide 16-byte shared
// load costs at least two cycles even when it broadcasts.  So a lane holds a
// few rows of two columns (the loaded k, q values serve both), and a warp splits
// the rows into 8 groups: lane (g, jj), g = lane / 4, owns the r/8 rows
// {4 (8 m + g) + e : m < r/32, e < 4} of columns 2 jj and 2 jj + 1 of its
// warp's 8.  A quarter-warp then reads two adjacent 16-byte words per load.
// A CTA has 4 warps and 32 columns.
//
// The output is read after the write, y_t = S_t^T q_t.  Since S_t = S_{t-1} +
// k_t c_t^T with c_t = beta_t (v_t - p_t), it equals S_{t-1}^T q_t + c_t (k_t . q_t):
// both reads use S_{t-1}, and the next token's reads wait only for the write.
// The four partial sums of a lane (p and S^T q for its two columns) are
// reduced over the 8 row groups by a reduce-scatter (each step sends half of
// what a lane holds), after which each lane holds one total; three shuffles
// hand c back to every lane of the column pair.  Per token a lane does
// 3 r/4 packed FP32 FMAs (f32x2) and 8 shuffles; k . q comes once per token
// from the staged rows.
//
// Tokens arrive in blocks of kTB: the TMA unit copies the block's q and k
// (contiguous) and the CTA's slice of each v row into a double-buffered raw
// stage, two blocks ahead; the CTA converts a landed block to FP32 once, and y
// leaves through shared memory, one coalesced block at a time.

#include "tc_common.cuh"

#include <cuda_bf16.h>

namespace la {
namespace {

constexpr int kTB = 32;                  // tokens per staged block
constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int NC = 32;                   // value columns per CTA (8 per warp, 2 per lane)

template <typename Tin, int r>
struct DeltaCfg {
    static constexpr int F = r / 32;               // float4 row blocks per lane (r/8 rows)
    static constexpr int kEl = (int)sizeof(Tin);
    static constexpr int RS = r + 4;               // FP32 row stride of q, k (16-byte pad)
    // byte offsets in dynamic shared memory
    static constexpr int kRawQ = kTB * r * kEl;    // one raw q (or k) block
    static constexpr int kRawV = kTB * NC * kEl;   // one raw v block (row stride NC)
    static constexpr int kRawStage = 2 * kRawQ + kRawV;
    static constexpr int kOffQ = 2 * kRawStage;    // FP32 q [kTB][RS]
    static constexpr int kOffK = kOffQ + kTB * RS * 4;
    static constexpr int kOffV = kOffK + kTB * RS * 4;    // FP32 v [kTB][NC]
    static constexpr int kOffY = kOffV + kTB * NC * 4;    // FP32 y [kTB][NC]
    static constexpr int kOffB = kOffY + kTB * NC * 4;    // beta [kTB]
    static constexpr int kOffBar = kOffB + kTB * 4;       // full[2]
    static constexpr int kOffFlag = kOffBar + 16;
    static constexpr int kBytes = kOffFlag + 16;
    static_assert(kRawQ % 16 == 0 && kRawV % 16 == 0, "16-byte staging");
};

__device__ __forceinline__ void bf16x8_to_f32(uint4 w, float *dst)
{
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
    float f[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        f[2 * e] = __uint_as_float(u[e] << 16);
        f[2 * e + 1] = __uint_as_float(u[e] & 0xffff0000u);
    }
    reinterpret_cast<float4 *>(dst)[0] = make_float4(f[0], f[1], f[2], f[3]);
    reinterpret_cast<float4 *>(dst)[1] = make_float4(f[4], f[5], f[6], f[7]);
}

// nrows rows of w elements (w a multiple of 8) from a raw block (rows packed) to
// FP32 rows of stride ds floats.
template <typename Tin, int w, int ds>
__device__ __forceinline__ void to_f32(const unsigned char *src, float *dst, int nrows)
{
    if constexpr (sizeof(Tin) == 2) {
        constexpr int n8 = w / 8;
        for (int i = threadIdx.x; i < nrows * n8; i += kThreads)
            bf16x8_to_f32(reinterpret_cast<const uint4 *>(src)[i], dst + (i / n8) * ds + (i % n8) * 8);
    } else {
        constexpr int n4 = w / 4;
        for (int i = threadIdx.x; i < nrows * n4; i += kThreads)
            *reinterpret_cast<float4 *>(dst + (i / n4) * ds + (i % n4) * 4) = reinterpret_cast<const float4 *>(src)[i];
    }
}

// 8 FP32 values as one 16-byte (FP32: two) global store of the output type.
__device__ __forceinline__ void store8(__nv_bfloat16 *p, const float *f)
{
    uint4 w;
    w.x = pack_bf16x2(f[0], f[1]);
    w.y = pack_bf16x2(f[2], f[3]);
    w.z = pack_bf16x2(f[4], f[5]);
    w.w = pack_bf16x2(f[6], f[7]);
    *reinterpret_cast<uint4 *>(p) = w;
}
__device__ __forceinline__ void store8(float *p, const float *f)
{
    reinterpret_cast<float4 *>(p)[0] = make_float4(f[0], f[1], f[2], f[3]);
    reinterpret_cast<float4 *>(p)[1] = make_float4(f[4], f[5], f[6], f[7]);
}

__device__ __forceinline__ float2 lo2(float4 a) { return make_float2(a.x, a.y); }
__device__ __forceinline__ float2 hi2(float4 a) { return make_float2(a.z, a.w); }

// k_t . q_t of token `lane` of the block (lanes >= nt return 0), in FP32 from the
// staged rows, always in the same order.  The padded row stride RS puts the
// rows of the 8 lanes of a quarter-warp in 8 different bank groups.
template <int r, int RS>
__device__ __forceinline__ float kq_of_lane(const float *fk, const float *fq, int lane, int nt)
{
    constexpr int n4 = r / 4;
    if (lane >= nt) return 0.f;
    const float4 *a = reinterpret_cast<const float4 *>(fk + lane * RS);
    const float4 *b = reinterpret_cast<const float4 *>(fq + lane * RS);
    float2 s0 = make_float2(0.f, 0.f), s1 = s0;
#pragma unroll 8
    for (int f = 0; f < n4; ++f) {
        const float4 x = a[f], y = b[f];
        s0 = __ffma2_rn(lo2(x), lo2(y), s0);
        s1 = __ffma2_rn(hi2(x), hi2(y), s1);
    }
    const float2 s = __fadd2_rn(s0, s1);
    return s.x + s.y;
}

// Per-lane view of one token: its rows of k and q, and where the token's v, beta
// and output live in the staged block.
struct TokenIo {
    const float *fk, *fq;   // staged rows (stride RS), offset to this lane's first row block
    const float *fv;        // v of the token, column 0 of the CTA
    const float *fb;        // beta of the token
    float *fy;              // output row of the token
};

// One token for one lane.  S2[m][c][h] holds rows 4 (8 m + g) + 2h, + 1 of the
// lane's column c (of 2); kk, qq hold the same rows of k_t and q_t.
//  - partial sums over the lane's rows: p_c = S_{t-1}^T k, u_c = S_{t-1}^T q;
//  - reduce-scatter over the 8 row groups (lane bits 4, 3, 2): after it, lane
//    bit 4 says whether the lane holds a p (0) or a u (1), bit 3 which column;
//  - the p lanes form c = beta (v_j - p_j); the u lanes take it from their
//    partner and write y_j = u_j + c (k . q); every lane fetches c of both its
//    columns and writes S += k c.
// The next token's k and q are loaded into kn, qn meanwhile (token offset tn).
template <int F, int RS>
__device__ __forceinline__ void token_step(float2 (&S2)[F][2][2], const float4 (&kk)[F], const float4 (&qq)[F],
                                           float4 (&kn)[F], float4 (&qn)[F], const TokenIo &io, int tn, float kq,
                                           int lane, int col)
{
    float2 pa[2][2], ua[2][2];
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int h = 0; h < 2; ++h) pa[c][h] = ua[c][h] = make_float2(0.f, 0.f);
#pragma unroll
    for (int m = 0; m < F; ++m)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            pa[c][0] = __ffma2_rn(S2[m][c][0], lo2(kk[m]), pa[c][0]);
            pa[c][1] = __ffma2_rn(S2[m][c][1], hi2(kk[m]), pa[c][1]);
            ua[c][0] = __ffma2_rn(S2[m][c][0], lo2(qq[m]), ua[c][0]);
            ua[c][1] = __ffma2_rn(S2[m][c][1], hi2(qq[m]), ua[c][1]);
        }
    {
        const float4 *kr = reinterpret_cast<const float4 *>(io.fk + tn * RS);
        const float4 *qr = reinterpret_cast<const float4 *>(io.fq + tn * RS);
#pragma unroll
        for (int m = 0; m < F; ++m) {
            kn[m] = kr[8 * m];
            qn[m] = qr[8 * m];
        }
    }
    float val[4];   // p_0, p_1, u_0, u_1 over this lane's rows
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        const float2 ps = __fadd2_rn(pa[c][0], pa[c][1]), us = __fadd2_rn(ua[c][0], ua[c][1]);
        val[c] = ps.x + ps.y;
        val[2 + c] = us.x + us.y;
    }
    // reduce-scatter: bit 4 keeps p (0) or u (1), bit 3 keeps column 0 or 1
    const bool b4 = lane & 16, b3 = lane & 8;
    float k0 = b4 ? val[2] : val[0], k1 = b4 ? val[3] : val[1];
    const float s0 = b4 ? val[0] : val[2], s1 = b4 ? val[1] : val[3];
    k0 += __shfl_xor_sync(0xffffffffu, s0, 16);
    k1 += __shfl_xor_sync(0xffffffffu, s1, 16);
    float tot = b3 ? k1 : k0;
    tot += __shfl_xor_sync(0xffffffffu, b3 ? k0 : k1, 8);
    tot += __shfl_xor_sync(0xffffffffu, tot, 4);
    // p lanes: c = beta (v_j - p_j); u lanes take c from their partner (lane ^ 16)
    const float cp = b4 ? 0.f : *io.fb * (io.fv[col] - tot);
    const float cu = __shfl_xor_sync(0xffffffffu, cp, 16);
    if (b4 && !(lane & 4)) io.fy[col] = fmaf(cu, kq, tot);
    // c of columns 0 and 1 of this lane's pair: the p lanes jj and jj + 8
    const int jj = lane & 3;
    const float c0 = __shfl_sync(0xffffffffu, cp, jj), c1 = __shfl_sync(0xffffffffu, cp, jj + 8);
    const float2 cc[2] = {make_float2(c0, c0), make_float2(c1, c1)};
#pragma unroll
    for (int m = 0; m < F; ++m)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            S2[m][c][0] = __ffma2_rn(lo2(kk[m]), cc[c], S2[m][c][0]);
            S2[m][c][1] = __ffma2_rn(hi2(kk[m]), cc[c], S2[m][c][1]);
        }
}

template <typename Tin, int r>
__global__ void __launch_bounds__(kThreads)
delta_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k, const Tin *__restrict__ v,
             const float *__restrict__ beta, const float *S0, int T, int dv, int nslice, Tin *__restrict__ y,
             float *S_out, int *status, unsigned long long limit_ns)
{
    using Cfg = DeltaCfg<Tin, r>;
    constexpr int F = Cfg::F, RS = Cfg::RS;
    extern __shared__ __align__(128) unsigned char smem[];
    float *fq = reinterpret_cast<float *>(smem + Cfg::kOffQ);
    float *fk = reinterpret_cast<float *>(smem + Cfg::kOffK);
    float *fv = reinterpret_cast<float *>(smem + Cfg::kOffV);
    float *fy = reinterpret_cast<float *>(smem + Cfg::kOffY);
    float *fb = reinterpret_cast<float *>(smem + Cfg::kOffB);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Cfg::kOffBar);
    int *flag = reinterpret_cast<int *>(smem + Cfg::kOffFlag);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, jj = lane & 3;
    const int bh = blockIdx.x / nslice;
    const int c0 = (blockIdx.x % nslice) * NC;     // first value column of this CTA
    const int jl = warp * 8 + 2 * jj;              // local column of the lane's pair
    const int col = jl + ((lane >> 3) & 1);        // local column of this lane's reduced total
    const int nblk = (T + kTB - 1) / kTB;
    Ctx cx{flag, limit_ns, status};

    if (tid == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        *flag = 0;
        fence_mbarrier_init();
    }
    __syncthreads();

    const Tin *qh = q + (size_t)bh * T * r, *kh = k + (size_t)bh * T * r;
    const Tin *vh = v + (size_t)bh * T * dv + c0;
    // Warp 0 starts the copies of block b into stage b & 1.
    auto issue = [&](int b) {
        const int st = b & 1, t0 = b * kTB, nt = min(kTB, T - t0);
        unsigned char *raw = smem + st * Cfg::kRawStage;
        const uint32_t qbytes = (uint32_t)(nt * r * Cfg::kEl), vrow = (uint32_t)(NC * Cfg::kEl);
        if (lane == 0) mbar_arrive_expect_tx(&full[st], 2 * qbytes + nt * vrow);
        __syncwarp();
        if (lane == 0) bulk_load(raw, qh + (size_t)t0 * r, qbytes, &full[st]);
        if (lane == 1) bulk_load(raw + Cfg::kRawQ, kh + (size_t)t0 * r, qbytes, &full[st]);
        if (lane < nt) bulk_load(raw + 2 * Cfg::kRawQ + lane * vrow, vh + (size_t)(t0 + lane) * dv, vrow, &full[st]);
    };
    if (warp == 0) {
        if (nblk > 0) issue(0);
        if (nblk > 1) issue(1);
    }

    // S2[m][c][h]: rows 4 (8 m + g) + 2h and + 1 of column c0 + jl + c
    float2 S2[F][2][2];
#pragma unroll
    for (int m = 0; m < F; ++m)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int row = 4 * (8 * m + g) + 2 * h;
            float2 a = make_float2(0.f, 0.f), b = a;
            if (S0) {
                const float *src = S0 + ((size_t)bh * r + row) * dv + c0 + jl;
                a = *reinterpret_cast<const float2 *>(src);        // row, columns jl, jl + 1
                b = *reinterpret_cast<const float2 *>(src + dv);   // row + 1
            }
            S2[m][0][h] = make_float2(a.x, b.x);
            S2[m][1][h] = make_float2(a.y, b.y);
        }
    float b_next = 1.f;
    if (beta && tid < kTB && tid < T) b_next = beta[(size_t)bh * T + tid];

    Tin *yh = y + (size_t)bh * T * dv + c0;
    auto store_y = [&](int b) {   // NC columns of nt rows, 8 per thread per pass
        const int t0 = b * kTB, nt = min(kTB, T - t0);
        for (int e = tid; e < nt * (NC / 8); e += kThreads) {
            const int t = e / (NC / 8), c = (e % (NC / 8)) * 8;
            store8(yh + (size_t)(t0 + t) * dv + c, fy + t * NC + c);
        }
    };

    int b = 0;
    for (; b < nblk; ++b) {
        const int st = b & 1, t0 = b * kTB, nt = min(kTB, T - t0);
        const bool ok = wait(cx, &full[st], (b >> 1) & 1);
        if (__syncthreads_or(!ok)) break;   // also: block b - 1's compute has finished
        if (b > 0) store_y(b - 1);
        const unsigned char *raw = smem + st * Cfg::kRawStage;
        to_f32<Tin, r, RS>(raw, fq, nt);
        to_f32<Tin, r, RS>(raw + Cfg::kRawQ, fk, nt);
        to_f32<Tin, NC, NC>(raw + 2 * Cfg::kRawQ, fv, nt);
        if (tid < kTB) fb[tid] = b_next;
        __syncthreads();                    // FP32 block ready; the raw stage is free again
        if (warp == 0 && b + 2 < nblk) issue(b + 2);
        if (beta && tid < kTB && t0 + kTB + tid < T) b_next = beta[(size_t)bh * T + t0 + kTB + tid];
        const float kq_reg = kq_of_lane<r, RS>(fk, fq, lane, nt);   // lane l: token l of the block
        float4 kA[F], qA[F], kB[F], qB[F];
        {
            const float4 *kr = reinterpret_cast<const float4 *>(fk) + g;
            const float4 *qr = reinterpret_cast<const float4 *>(fq) + g;
#pragma unroll
            for (int m = 0; m < F; ++m) {
                kA[m] = kr[8 * m];
                qA[m] = qr[8 * m];
            }
        }
        TokenIo io{fk + 4 * g, fq + 4 * g, fv, fb, fy};
        // tokens in pairs, the operand registers alternating between A and B
#pragma unroll 1
        for (int t = 0; t < nt; t += 2) {
            TokenIo it = io;
            it.fv += t * NC; it.fb += t; it.fy += t * NC;
            token_step<F, RS>(S2, kA, qA, kB, qB, it, min(t + 1, nt - 1), __shfl_sync(0xffffffffu, kq_reg, t), lane,
                              col);
            if (t + 1 < nt) {
                it.fv += NC; it.fb += 1; it.fy += NC;
                token_step<F, RS>(S2, kB, qB, kA, qA, it, min(t + 2, nt - 1), __shfl_sync(0xffffffffu, kq_reg, t + 1),
                                  lane, col);
            }
        }
    }

    if (b < nblk) {
        // gave up waiting: let the copies already started land before the CTA exits
        if (tid == 0)
            for (int bb = b; bb < nblk && bb < b + 2; ++bb) mbar_wait(&full[bb & 1], (bb >> 1) & 1, limit_ns);
        __syncthreads();
        return;
    }
    __syncthreads();
    if (nblk > 0) store_y(nblk - 1);
#pragma unroll
    for (int m = 0; m < F; ++m)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int row = 4 * (8 * m + g) + 2 * h;
            float *dst = S_out + ((size_t)bh * r + row) * dv + c0 + jl;
            *reinterpret_cast<float2 *>(dst) = make_float2(S2[m][0][h].x, S2[m][1][h].x);
            *reinterpret_cast<float2 *>(dst + dv) = make_float2(S2[m][0][h].y, S2[m][1][h].y);
        }
}

template <typename Tin, int r>
cudaError_t launch_r(const void *q, const void *k, const void *v, const float *beta, const float *S0, int B, int H,
                     int T, int dv, void *y, float *S_out, int *status, unsigned long long limit_ns,
                     cudaStream_t stream)
{
    using Cfg = DeltaCfg<Tin, r>;
    auto kern = delta_kernel<Tin, r>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kBytes);
    if (e != cudaSuccess) return e;
    const int nslice = dv / NC;
    kern<<<(unsigned)((long long)B * H * nslice), kThreads, Cfg::kBytes, stream>>>(
        static_cast<const Tin *>(q), static_cast<const Tin *>(k), static_cast<const Tin *>(v), beta, S0, T, dv,
        nslice, static_cast<Tin *>(y), S_out, status, limit_ns);
    return cudaGetLastError();
}

template <typename Tin>
cudaError_t launch_t(const void *q, const void *k, const void *v, const float *beta, const float *S0, int B, int H,
                     int T, int r, int dv, void *y, float *S_out, int *status, unsigned long long limit_ns,
                     cudaStream_t stream)
{
    switch (r) {
    case 32: return launch_r<Tin, 32>(q, k, v, beta, S0, B, H, T, dv, y, S_out, status, limit_ns, stream);
    case 64: return launch_r<Tin, 64>(q, k, v, beta, S0, B, H, T, dv, y, S_out, status, limit_ns, stream);
    case 128: return launch_r<Tin, 128>(q, k, v, beta, S0, B, H, T, dv, y, S_out, status, limit_ns, stream);
    case 256: return launch_r<Tin, 256>(q, k, v, beta, S0, B, H, T, dv, y, S_out, status, limit_ns, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_delta(const void *q, const void *k, const void *v, bool bf16, const float *beta, const float *S0,
                         int B, int H, int T, int r, int dv, void *y, float *S_out, int *status,
                         unsigned long long limit_ns, cudaStream_t stream)
{
    if (bf16)
        return launch_t<__nv_bfloat16>(q, k, v, beta, S0, B, H, T, r, dv, y, S_out, status, limit_ns, stream);
    return launch_t<float>(q, k, v, beta, S0, B, H, T, r, dv, y, S_out, status, limit_ns, stream);
}

}  // namespace la
