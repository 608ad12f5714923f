// decode.cu -- single-token decode on the fixed-size S/z state, state init,
// and the diagnostic bounded-wait probe.
//
// Decode ("Linear attention：把历史写进状态", sections "公式里的每个维度" and
// "查询时，分子和分母一起读"; gate from "加一个门：让旧记忆逐渐淡出"):
//     S <- alpha S + phi(k) v^T,   z <- alpha z + phi(k),
//     y  = phi(q)^T S / (phi(q)^T z + eps)           (update before read)
// The step reads and rewrites r*dv + r FP32 state words per head and does two
// FMAs per state word, so it is bound by HBM bandwidth ("它省掉了什么，又把难题放在哪？":
// each step reads O(d_phi * dv) of state).  The r = dv = 128 kernel streams S
// with 16-byte accesses, one warp per 16 rows, 4 columns per lane, with all
// 16 row loads of a thread in flight before any arithmetic, and reduces the
// numerator across warps in shared memory and the denominator with warp
// shuffles.

#include "kernels.h"
#include "sm103_ptx.cuh"

#include <cuda_bf16.h>

namespace la {
namespace {

__device__ __forceinline__ float phi_exact(float x) { return x > 0.f ? x + 1.f : expf(x); }

template <bool BF16>
__device__ __forceinline__ float load_elem(const void *p, size_t i)
{
    if (BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p)[i]);
    return reinterpret_cast<const float *>(p)[i];
}

template <bool BF16>
__device__ __forceinline__ void store_elem(void *p, size_t i, float x)
{
    if (BF16) reinterpret_cast<__nv_bfloat16 *>(p)[i] = __float2bfloat16_rn(x);
    else reinterpret_cast<float *>(p)[i] = x;
}

// Four consecutive elements (8-byte aligned for BF16, 16-byte for FP32): a raw load,
// widened to floats when used.
template <bool BF16> struct Quad;
template <> struct Quad<true> {
    using raw = uint2;
    static __device__ __forceinline__ uint2 load(const void *p, size_t i)
    {
        return *reinterpret_cast<const uint2 *>(reinterpret_cast<const __nv_bfloat16 *>(p) + i);
    }
    static __device__ __forceinline__ float4 widen(uint2 w)
    {
        return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u), __uint_as_float(w.y << 16),
                           __uint_as_float(w.y & 0xFFFF0000u));
    }
};
template <> struct Quad<false> {
    using raw = float4;
    static __device__ __forceinline__ float4 load(const void *p, size_t i)
    {
        return *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(p) + i);
    }
    static __device__ __forceinline__ float4 widen(float4 w) { return w; }
};

__device__ __forceinline__ float4 ld_stream(const float4 *p)
{
    float4 v;
    asm volatile("ld.global.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ void st_stream(float4 *p, float4 v)
{
    asm volatile("st.global.cs.v4.f32 [%0], {%1,%2,%3,%4};" ::"l"(p), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
                 : "memory");
}

// r = dv = 128: one CTA of 256 threads per (b, h).
template <bool BF16>
__global__ void __launch_bounds__(256)
decode128_kernel(const void *__restrict__ q, const void *__restrict__ k, const void *__restrict__ v,
                 const float *__restrict__ alpha, float *__restrict__ S, float *__restrict__ z, float eps,
                 void *__restrict__ y)
{
    constexpr int R = 128, DV = 128;
    __shared__ float qf[R], kf[R];
    __shared__ float4 num_part[8][32];
    __shared__ float den_part[4];
    const int bh = blockIdx.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const float a = alpha ? alpha[bh] : 1.f;

    // 16 rows of S per warp, 4 columns per lane: issue every load first.
    float4 *Srow = reinterpret_cast<float4 *>(S + (size_t)bh * R * DV) + (size_t)warp * 16 * (DV / 4) + lane;
    float4 s[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) s[i] = ld_stream(Srow + i * (DV / 4));

    if (tid < R) {
        qf[tid] = phi_exact(load_elem<BF16>(q, (size_t)bh * R + tid));
        kf[tid] = phi_exact(load_elem<BF16>(k, (size_t)bh * R + tid));
    }
    float4 vv;
    vv.x = load_elem<BF16>(v, (size_t)bh * DV + lane * 4 + 0);
    vv.y = load_elem<BF16>(v, (size_t)bh * DV + lane * 4 + 1);
    vv.z = load_elem<BF16>(v, (size_t)bh * DV + lane * 4 + 2);
    vv.w = load_elem<BF16>(v, (size_t)bh * DV + lane * 4 + 3);
    __syncthreads();

    // z and the denominator: warps 0..3 own features 0..127
    if (tid < R) {
        const float zn = fmaf(a, z[(size_t)bh * R + tid], kf[tid]);
        z[(size_t)bh * R + tid] = zn;
        float part = qf[tid] * zn;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
        if (lane == 0) den_part[warp] = part;
    }

    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int row = warp * 16 + i;
        const float kr = kf[row], qr = qf[row];
        float4 t;
        t.x = fmaf(a, s[i].x, kr * vv.x);
        t.y = fmaf(a, s[i].y, kr * vv.y);
        t.z = fmaf(a, s[i].z, kr * vv.z);
        t.w = fmaf(a, s[i].w, kr * vv.w);
        st_stream(Srow + i * (DV / 4), t);
        acc.x = fmaf(qr, t.x, acc.x);
        acc.y = fmaf(qr, t.y, acc.y);
        acc.z = fmaf(qr, t.z, acc.z);
        acc.w = fmaf(qr, t.w, acc.w);
    }
    num_part[warp][lane] = acc;
    __syncthreads();
    if (tid < DV) {
        const float *np = reinterpret_cast<const float *>(num_part);
        float n = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) n += np[w * DV + tid];
        const float den = den_part[0] + den_part[1] + den_part[2] + den_part[3];
        store_elem<BF16>(y, (size_t)bh * DV + tid, n / (den + eps));
    }
}

// A short continuation, T <= kMultiMaxT tokens per (b, h) from a carried state,
// r = dv = 128: the layout of decode128_kernel, with the state kept in registers
// from the first token to the last, so that it is read and written once for all
// T.  Every token's phi(q), phi(k), v and gate are read into shared memory up
// front, in flight together with the state; each token then costs one block
// barrier (the numerator's per-warp parts are double-buffered).  S0 and z0 are
// read whole before anything is written, so they may alias S_out and z_out.
// d_out (or nullptr) receives the denominators.
// The tokens' phi(q), phi(k) (FP32) and v live in 48 KB of dynamic shared memory
// laid out for 32 tokens whatever T (fixed offsets; registers already hold the
// kernel to 2 CTAs per SM); they are loaded in halves of 16 tokens, so that the raw
// loads held in registers stay those of 16.
constexpr int kMultiMaxT = 32, kMultiHalf = 16;
constexpr uint32_t kMultiTokenBytes = 128 * 4 * 3;
// PACKED: sequences packed token-major ([total_T, H, d], alpha [total_T, H]);
// CTA (b, h) walks sequence b if its bounds are valid and it has at most
// kMultiMaxT tokens (T is then ignored), and otherwise leaves it to the chunk
// kernel.
template <bool BF16, int HALVES, bool PACKED = false>
__global__ void __launch_bounds__(256, 2)
decode128_multi_kernel(const void *__restrict__ q, const void *__restrict__ k, const void *__restrict__ v,
                       const float *__restrict__ alpha, const float *S0, const float *z0, float *S_out,
                       float *z_out, int T, float eps, void *__restrict__ y, float *__restrict__ d_out,
                       const int *__restrict__ cu_seqlens = nullptr, int H = 1)
{
    constexpr int R = 128, DV = 128;
    extern __shared__ float4 multi_smem[];
    float(*qf)[R] = reinterpret_cast<float(*)[R]>(multi_smem);
    float(*kf)[R] = reinterpret_cast<float(*)[R]>(multi_smem + kMultiMaxT * (R / 4));
    float4(*vs)[DV / 4] = reinterpret_cast<float4(*)[DV / 4]>(multi_smem + 2 * kMultiMaxT * (R / 4));
    __shared__ float al[kMultiMaxT];
    __shared__ float4 num_part[2][8][32];
    __shared__ float den_part[2][4];
    const int bh = blockIdx.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const size_t row0 = (size_t)warp * 16 * (DV / 4) + lane;   // this thread's first float4 of S
    int seq0 = 0;
    if (PACKED) {
        const int b = bh / H;
        seq0 = cu_seqlens[b];
        const int seq1 = cu_seqlens[b + 1];
        if (seq0 < 0 || seq1 < seq0 || seq1 > T || seq1 - seq0 > kMultiMaxT) return;   // not this kernel's
        T = seq1 - seq0;
    }
    // row of token t of this head in q, k, v, y (rows of 128) and alpha
    const size_t tok0 = (size_t)bh * T;
    auto row = [&](int t) -> size_t { return PACKED ? (size_t)(seq0 + t) * H + bh % H : tok0 + t; };

    float4 s[16];
    if (S0) {
        const float4 *src = reinterpret_cast<const float4 *>(S0 + (size_t)bh * R * DV) + row0;
#pragma unroll
        for (int i = 0; i < 16; ++i) s[i] = ld_stream(src + i * (DV / 4));
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) s[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float zr = (tid < R && z0) ? z0[(size_t)bh * R + tid] : 0.f;
    // 4 elements per load (32 loads a token row), all of a thread's loads of a
    // half issued before any is used
    constexpr int kLoads = kMultiHalf * R / 4 / 256;   // per thread, tensor and half
    using Raw = typename Quad<BF16>::raw;   // the loads stay raw until they are stored
    const float a_t = (tid < T && alpha) ? alpha[row(tid)] : 1.f;
#pragma unroll
    for (int hv = 0; hv < HALVES; ++hv) {
        const int h0 = hv * kMultiHalf;
        const int nvec = min(kMultiHalf, T - h0) * R / 4, v0 = h0 * R / 4;
        Raw rq[kLoads], rk[kLoads], rv[kLoads];
#pragma unroll
        for (int it = 0; it < kLoads; ++it) {
            const int e = tid + it * 256;
            if (e < nvec) {
                const size_t off = row((v0 + e) / (R / 4)) * R + 4 * (size_t)((v0 + e) % (R / 4));
                rq[it] = Quad<BF16>::load(q, off);
                rk[it] = Quad<BF16>::load(k, off);
                rv[it] = Quad<BF16>::load(v, off);   // DV == R
            }
        }
#pragma unroll
        for (int it = 0; it < kLoads; ++it) {
            const int e = tid + it * 256;
            if (e < nvec) {
                const float4 fq = Quad<BF16>::widen(rq[it]), fk = Quad<BF16>::widen(rk[it]);
                reinterpret_cast<float4 *>(&qf[0][0])[v0 + e] =
                    make_float4(phi_exact(fq.x), phi_exact(fq.y), phi_exact(fq.z), phi_exact(fq.w));
                reinterpret_cast<float4 *>(&kf[0][0])[v0 + e] =
                    make_float4(phi_exact(fk.x), phi_exact(fk.y), phi_exact(fk.z), phi_exact(fk.w));
                reinterpret_cast<float4 *>(&vs[0][0])[v0 + e] = Quad<BF16>::widen(rv[it]);
            }
        }
    }
    if (tid < T) al[tid] = a_t;
    __syncthreads();

    const bool gated = alpha != nullptr;
    for (int t = 0; t < T; ++t) {
        const int pb = t & 1;
        const float a = al[t];
        const float4 vv = vs[t][lane];
        if (tid < R) {
            zr = fmaf(a, zr, kf[t][tid]);
            float part = qf[t][tid] * zr;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
            if (lane == 0) den_part[pb][warp] = part;
        }
        // two columns per instruction (packed FP32 pairs, each lane rounded as
        // its scalar fmaf / multiply would be)
        const float2 v01 = make_float2(vv.x, vv.y), v23 = make_float2(vv.z, vv.w), a2 = make_float2(a, a);
        float2 acc01 = make_float2(0.f, 0.f), acc23 = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int row = warp * 16 + i;
            const float2 kr = make_float2(kf[t][row], kf[t][row]), qr = make_float2(qf[t][row], qf[t][row]);
            float2 s01 = make_float2(s[i].x, s[i].y), s23 = make_float2(s[i].z, s[i].w);
            if (gated) {
                s01 = __ffma2_rn(a2, s01, __fmul2_rn(kr, v01));
                s23 = __ffma2_rn(a2, s23, __fmul2_rn(kr, v23));
            } else {
                s01 = __ffma2_rn(kr, v01, s01);
                s23 = __ffma2_rn(kr, v23, s23);
            }
            acc01 = __ffma2_rn(qr, s01, acc01);
            acc23 = __ffma2_rn(qr, s23, acc23);
            s[i] = make_float4(s01.x, s01.y, s23.x, s23.y);
        }
        num_part[pb][warp][lane] = make_float4(acc01.x, acc01.y, acc23.x, acc23.y);
        // one barrier per token: the parts of token t - 1 (the other buffer) were
        // read before any thread passed this barrier's previous phase
        __syncthreads();
        if (tid < DV) {
            const float *np = reinterpret_cast<const float *>(num_part[pb]);
            float n = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) n += np[w * DV + tid];
            const float den = den_part[pb][0] + den_part[pb][1] + den_part[pb][2] + den_part[pb][3] + eps;
            store_elem<BF16>(y, row(t) * DV + tid, n / den);
            if (d_out && tid == 0) d_out[row(t)] = den;
        }
    }
    float4 *dst = reinterpret_cast<float4 *>(S_out + (size_t)bh * R * DV) + row0;
#pragma unroll
    for (int i = 0; i < 16; ++i) st_stream(dst + i * (DV / 4), s[i]);
    if (tid < R) z_out[(size_t)bh * R + tid] = zr;
}

// Any r, dv <= 256: thread j owns column j (and feature j for z), rows in order.
template <bool BF16>
__global__ void __launch_bounds__(256)
decode_generic_kernel(const void *__restrict__ q, const void *__restrict__ k, const void *__restrict__ v,
                      const float *__restrict__ alpha, float *__restrict__ S, float *__restrict__ z, int r,
                      int dv, float eps, void *__restrict__ y)
{
    __shared__ float qf[256], kf[256], red[8];
    const int bh = blockIdx.x, tid = threadIdx.x;
    const float a = alpha ? alpha[bh] : 1.f;
    float part = 0.f;
    if (tid < r) {
        qf[tid] = phi_exact(load_elem<BF16>(q, (size_t)bh * r + tid));
        kf[tid] = phi_exact(load_elem<BF16>(k, (size_t)bh * r + tid));
        const float zn = fmaf(a, z[(size_t)bh * r + tid], kf[tid]);
        z[(size_t)bh * r + tid] = zn;
        part = qf[tid] * zn;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
    if ((tid & 31) == 0) red[tid >> 5] = part;
    __syncthreads();
    if (tid < dv) {
        float den = 0.f;
        for (int w = 0; w < 8; ++w) den += red[w];
        const float vj = load_elem<BF16>(v, (size_t)bh * dv + tid);
        float *Sc = S + (size_t)bh * r * dv + tid;
        float n = 0.f;
        for (int i = 0; i < r; ++i) {
            const float t = fmaf(a, Sc[(size_t)i * dv], kf[i] * vj);
            Sc[(size_t)i * dv] = t;
            n = fmaf(qf[i], t, n);
        }
        store_elem<BF16>(y, (size_t)bh * dv + tid, n / (den + eps));
    }
}

__global__ void state_init_kernel(float *__restrict__ S, float *__restrict__ z, long long nS, long long nz)
{
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < nS; i += stride) S[i] = 0.f;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < nz; i += stride) z[i] = 0.f;
}

// Waits on a barrier that nothing completes, for at most limit_ns, then records
// a timeout in the status word -- the same path every kernel takes when a wait
// runs out.
__global__ void wait_probe_kernel(int *status, unsigned long long limit_ns)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbarrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait(&bar, 0, limit_ns)) atomicExch(status, kStatusTimeout);
}

}  // namespace

cudaError_t launch_decode(const void *q, const void *k, const void *v, bool bf16, const float *alpha, float *S,
                          float *z, int B, int H, int r, int dv, float eps, void *y, bool fast128,
                          cudaStream_t stream)
{
    const long long nbh = (long long)B * H;   // the caller bounds it by INT_MAX
    if (nbh < 1 || nbh > 0x7fffffffLL) return cudaErrorInvalidValue;
    if (fast128) {
        if (bf16) decode128_kernel<true><<<(unsigned)nbh, 256, 0, stream>>>(q, k, v, alpha, S, z, eps, y);
        else decode128_kernel<false><<<(unsigned)nbh, 256, 0, stream>>>(q, k, v, alpha, S, z, eps, y);
    } else {
        if (bf16) decode_generic_kernel<true><<<(unsigned)nbh, 256, 0, stream>>>(q, k, v, alpha, S, z, r, dv, eps, y);
        else decode_generic_kernel<false><<<(unsigned)nbh, 256, 0, stream>>>(q, k, v, alpha, S, z, r, dv, eps, y);
    }
    return cudaGetLastError();
}

cudaError_t launch_decode_multi(const void *q, const void *k, const void *v, bool bf16, const float *alpha,
                                const float *S0, const float *z0, float *S_out, float *z_out, int B, int H, int T,
                                float eps, void *y, float *d_out, cudaStream_t stream)
{
    const long long nbh = (long long)B * H;
    if (nbh < 1 || nbh > 0x7fffffffLL || T < 1 || T > kMultiMaxT) return cudaErrorInvalidValue;
    // the limit is raised once (the first call on a device must not be inside a
    // stream capture)
    // one half of 16 tokens or two
    using Kern = void (*)(const void *, const void *, const void *, const float *, const float *, const float *,
                          float *, float *, int, float, void *, float *, const int *, int);
    static const Kern kerns[4] = {decode128_multi_kernel<false, 1>, decode128_multi_kernel<false, 2>,
                                  decode128_multi_kernel<true, 1>, decode128_multi_kernel<true, 2>};
    static OncePerDevice attr_set[4];
    const int ki = (bf16 ? 2 : 0) + (T > kMultiHalf ? 1 : 0);
    const uint32_t bytes = kMultiMaxT * kMultiTokenBytes;
    const cudaError_t e = set_smem_once(kerns[ki], bytes, attr_set[ki]);
    if (e != cudaSuccess) return e;
    kerns[ki]<<<(unsigned)nbh, 256, bytes, stream>>>(q, k, v, alpha, S0, z0, S_out, z_out, T, eps, y, d_out, nullptr,
                                                      1);
    return cudaGetLastError();
}

cudaError_t launch_decode_multi_packed(const void *q, const void *k, const void *v, bool bf16, const float *alpha,
                                       const float *S0, const float *z0, float *S_out, float *z_out,
                                       const int *cu_seqlens, int B, int H, int total_T, float eps, void *y,
                                       cudaStream_t stream)
{
    const long long nbh = (long long)B * H;
    if (nbh < 1 || nbh > 0x7fffffffLL || total_T < 0 || !cu_seqlens) return cudaErrorInvalidValue;
    using Kern = void (*)(const void *, const void *, const void *, const float *, const float *, const float *,
                          float *, float *, int, float, void *, float *, const int *, int);
    static const Kern kerns[2] = {decode128_multi_kernel<false, 2, true>, decode128_multi_kernel<true, 2, true>};
    static OncePerDevice attr_set[2];
    const int ki = bf16 ? 1 : 0;
    const uint32_t bytes = kMultiMaxT * kMultiTokenBytes;
    const cudaError_t e = set_smem_once(kerns[ki], bytes, attr_set[ki]);
    if (e != cudaSuccess) return e;
    kerns[ki]<<<(unsigned)nbh, 256, bytes, stream>>>(q, k, v, alpha, S0, z0, S_out, z_out, total_T, eps, y, nullptr,
                                                      cu_seqlens, H);
    return cudaGetLastError();
}

cudaError_t launch_state_init(float *S, float *z, long long n_S, long long n_z, cudaStream_t stream)
{
    long long n = n_S > n_z ? n_S : n_z;
    long long blocks = (n + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;
    if (blocks < 1) blocks = 1;
    state_init_kernel<<<(unsigned)blocks, 256, 0, stream>>>(S, z, n_S, n_z);
    return cudaGetLastError();
}

cudaError_t launch_wait_probe(int *status, unsigned long long limit_ns, cudaStream_t stream)
{
    wait_probe_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
    return cudaGetLastError();
}

}  // namespace la
