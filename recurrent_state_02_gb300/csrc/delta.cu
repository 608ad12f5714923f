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
// Every column j of S is an independent recurrence: p_j, the error e_j and the
// update of column j involve column j alone.  So the value columns are split
// over CTAs and warps with no exchange between them; only the sums over the r
// rows (S^T k and S^T q) are reduced, inside a warp.
//
// A CTA has 4 warps and covers NC = 4 * (32 / G) columns of one (b, h), with
// G = r / 32 row groups: lane (g, jj) of warp w owns column w * 32/G + jj and
// the 32 rows {4 (G m + g) + e : m < 8, e < 4}.  Interleaving the row groups in
// blocks of 4 makes the 16-byte shared loads of k and q conflict-free: the G
// groups of a warp read G adjacent 16-byte words.
//
// The output is read after the write, y_t = S_t^T q_t.  Since S_t = S_{t-1} +
// k_t c_t^T with c_t = beta_t (v_t - p_t), it equals S_{t-1}^T q_t + c_t (k_t . q_t):
// both reads then use S_{t-1}, share one shuffle tree, and the next token's read
// of S_t waits only for the write.  Per token a lane does 48 packed FP32 FMAs
// (f32x2: S^T k, S^T q, the rank-1 write) and one log2(G)-step reduction of two
// values; k . q comes once per token from the staged rows.
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

template <typename Tin, int G>
struct DeltaCfg {
    static constexpr int r = 32 * G;               // key width
    static constexpr int kCols = 32 / G;           // value columns per warp
    static constexpr int NC = kWarps * kCols;      // value columns per CTA
    static constexpr int kEl = (int)sizeof(Tin);
    // byte offsets in dynamic shared memory
    static constexpr int kRawQ = kTB * r * kEl;    // one raw q (or k) block
    static constexpr int kRawV = kTB * NC * kEl;   // one raw v block (row stride NC)
    static constexpr int kRawStage = 2 * kRawQ + kRawV;
    static constexpr int RS = r + 4;               // FP32 row stride of q, k (16-byte pad)
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

__device__ __forceinline__ void store_out(float *p, size_t i, float x) { p[i] = x; }
__device__ __forceinline__ void store_out(__nv_bfloat16 *p, size_t i, float x) { p[i] = __float2bfloat16_rn(x); }

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

// One token for one lane, from S_{t-1} (S2) and the token's k, q (kk, qq):
//  - over the lane's rows, p = S_{t-1}^T k and u = S_{t-1}^T q, then both summed
//    over the warp's row groups in one shuffle tree;
//  - c = beta (v_j - p), the write S += k c, and the output
//    y_j = u + c (k . q), which equals S_t^T q since S_t = S_{t-1} + k c^T.
// So the read of the query does not wait for the write.  The next token's k and
// q are loaded into kn, qn meanwhile (token tn of the staged block).
template <int G, int kCols, int RS>
__device__ __forceinline__ void token_step(float2 (&S2)[16], const float4 (&kk)[8], const float4 (&qq)[8],
                                           float4 (&kn)[8], float4 (&qn)[8], const float *fk, const float *fq,
                                           float vj, float bt, float kq, int tn, int g, float *yout)
{
    float2 p0 = make_float2(0.f, 0.f), p1 = p0, p2 = p0, p3 = p0, u0 = p0, u1 = p0, u2 = p0, u3 = p0;
#pragma unroll
    for (int m = 0; m < 8; m += 2) {
        p0 = __ffma2_rn(S2[2 * m], lo2(kk[m]), p0);
        p1 = __ffma2_rn(S2[2 * m + 1], hi2(kk[m]), p1);
        p2 = __ffma2_rn(S2[2 * m + 2], lo2(kk[m + 1]), p2);
        p3 = __ffma2_rn(S2[2 * m + 3], hi2(kk[m + 1]), p3);
        u0 = __ffma2_rn(S2[2 * m], lo2(qq[m]), u0);
        u1 = __ffma2_rn(S2[2 * m + 1], hi2(qq[m]), u1);
        u2 = __ffma2_rn(S2[2 * m + 2], lo2(qq[m + 1]), u2);
        u3 = __ffma2_rn(S2[2 * m + 3], hi2(qq[m + 1]), u3);
    }
    const float4 *kr = reinterpret_cast<const float4 *>(fk + tn * RS) + g;
    const float4 *qr = reinterpret_cast<const float4 *>(fq + tn * RS) + g;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        kn[m] = kr[G * m];
        qn[m] = qr[G * m];
    }
    const float2 ps = __fadd2_rn(__fadd2_rn(p0, p1), __fadd2_rn(p2, p3));
    const float2 us = __fadd2_rn(__fadd2_rn(u0, u1), __fadd2_rn(u2, u3));
    float2 s = make_float2(ps.x + ps.y, us.x + us.y);
#pragma unroll
    for (int o = kCols; o < 32; o <<= 1)
        s = __fadd2_rn(s, make_float2(__shfl_xor_sync(0xffffffffu, s.x, o), __shfl_xor_sync(0xffffffffu, s.y, o)));
    const float c = bt * (vj - s.x);
    if (g == 0) *yout = fmaf(c, kq, s.y);
    const float2 c2 = make_float2(c, c);
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        S2[2 * m] = __ffma2_rn(lo2(kk[m]), c2, S2[2 * m]);
        S2[2 * m + 1] = __ffma2_rn(hi2(kk[m]), c2, S2[2 * m + 1]);
    }
}

template <typename Tin, int G>
__global__ void __launch_bounds__(kThreads)
delta_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k, const Tin *__restrict__ v,
             const float *__restrict__ beta, const float *S0, int T, int dv, int nslice, Tin *__restrict__ y,
             float *S_out, int *status, unsigned long long limit_ns)
{
    using Cfg = DeltaCfg<Tin, G>;
    constexpr int r = Cfg::r, kCols = Cfg::kCols, NC = Cfg::NC, RS = Cfg::RS;
    extern __shared__ __align__(128) unsigned char smem[];
    float *fq = reinterpret_cast<float *>(smem + Cfg::kOffQ);
    float *fk = reinterpret_cast<float *>(smem + Cfg::kOffK);
    float *fv = reinterpret_cast<float *>(smem + Cfg::kOffV);
    float *fy = reinterpret_cast<float *>(smem + Cfg::kOffY);
    float *fb = reinterpret_cast<float *>(smem + Cfg::kOffB);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Cfg::kOffBar);
    int *flag = reinterpret_cast<int *>(smem + Cfg::kOffFlag);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int jj = lane % kCols, g = lane / kCols;
    const int bh = blockIdx.x / nslice;
    const int c0 = (blockIdx.x % nslice) * NC;     // first value column of this CTA
    const int ncv = min(NC, dv - c0);              // its columns (a multiple of kCols)
    const int jl = warp * kCols + jj;              // local column of this lane
    const bool active = warp * kCols < ncv;        // warp-uniform
    const int j = c0 + jl;
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
        const uint32_t qbytes = (uint32_t)(nt * r * Cfg::kEl), vrow = (uint32_t)(ncv * Cfg::kEl);
        if (lane == 0) mbar_arrive_expect_tx(&full[st], 2 * qbytes + nt * vrow);
        __syncwarp();
        if (lane == 0) bulk_load(raw, qh + (size_t)t0 * r, qbytes, &full[st]);
        if (lane == 1) bulk_load(raw + Cfg::kRawQ, kh + (size_t)t0 * r, qbytes, &full[st]);
        if (lane < nt) bulk_load(raw + 2 * Cfg::kRawQ + lane * NC * Cfg::kEl, vh + (size_t)(t0 + lane) * dv, vrow,
                                 &full[st]);
    };
    if (warp == 0) {
        if (nblk > 0) issue(0);
        if (nblk > 1) issue(1);
    }

    // S2[2m + h] holds rows 4 (G m + g) + 2h and + 1 of column j.
    float2 S2[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) S2[i] = make_float2(0.f, 0.f);
    if (S0 && active) {
        const float *src = S0 + (size_t)bh * r * dv + j;
#pragma unroll
        for (int m = 0; m < 8; ++m)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int row = 4 * (G * m + g) + 2 * h;
                S2[2 * m + h] = make_float2(src[(size_t)row * dv], src[(size_t)(row + 1) * dv]);
            }
    }
    float b_next = 1.f;
    if (beta && tid < kTB && tid < T) b_next = beta[(size_t)bh * T + tid];

    Tin *yh = y + (size_t)bh * T * dv + c0;
    auto store_y = [&](int b) {
        const int t0 = b * kTB, nt = min(kTB, T - t0);
        for (int e = tid; e < nt * ncv; e += kThreads) {
            const int t = e / ncv, c = e - t * ncv;
            store_out(yh, (size_t)(t0 + t) * dv + c, fy[t * NC + c]);
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
        if (!active) continue;
        const float kq_reg = kq_of_lane<r, RS>(fk, fq, lane, nt);   // lane l: token l of the block
        float4 kA[8], qA[8], kB[8], qB[8];
        {
            const float4 *kr = reinterpret_cast<const float4 *>(fk) + g;
            const float4 *qr = reinterpret_cast<const float4 *>(fq) + g;
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                kA[m] = kr[G * m];
                qA[m] = qr[G * m];
            }
        }
        // tokens in pairs, the operand registers alternating between A and B
#pragma unroll 1
        for (int t = 0; t < nt; t += 2) {
            token_step<G, kCols, RS>(S2, kA, qA, kB, qB, fk, fq, fv[t * NC + jl], fb[t],
                                        __shfl_sync(0xffffffffu, kq_reg, t), min(t + 1, nt - 1), g,
                                        fy + t * NC + jl);
            if (t + 1 < nt)
                token_step<G, kCols, RS>(S2, kB, qB, kA, qA, fk, fq, fv[(t + 1) * NC + jl], fb[t + 1],
                                            __shfl_sync(0xffffffffu, kq_reg, t + 1), min(t + 2, nt - 1), g,
                                            fy + (t + 1) * NC + jl);
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
    if (active) {
        float *dst = S_out + (size_t)bh * r * dv + j;
#pragma unroll
        for (int m = 0; m < 8; ++m)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int row = 4 * (G * m + g) + 2 * h;
                dst[(size_t)row * dv] = S2[2 * m + h].x;
                dst[(size_t)(row + 1) * dv] = S2[2 * m + h].y;
            }
    }
}

template <typename Tin, int G>
cudaError_t launch_g(const void *q, const void *k, const void *v, const float *beta, const float *S0, int B, int H,
                     int T, int dv, void *y, float *S_out, int *status, unsigned long long limit_ns,
                     cudaStream_t stream)
{
    using Cfg = DeltaCfg<Tin, G>;
    auto kern = delta_kernel<Tin, G>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kBytes);
    if (e != cudaSuccess) return e;
    const int nslice = (dv + Cfg::NC - 1) / Cfg::NC;
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
    case 32: return launch_g<Tin, 1>(q, k, v, beta, S0, B, H, T, dv, y, S_out, status, limit_ns, stream);
    case 64: return launch_g<Tin, 2>(q, k, v, beta, S0, B, H, T, dv, y, S_out, status, limit_ns, stream);
    case 128: return launch_g<Tin, 4>(q, k, v, beta, S0, B, H, T, dv, y, S_out, status, limit_ns, stream);
    case 256: return launch_g<Tin, 8>(q, k, v, beta, S0, B, H, T, dv, y, S_out, status, limit_ns, stream);
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
