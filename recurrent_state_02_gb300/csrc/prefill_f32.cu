// prefill_f32.cu -- exact FP32 prefill on CUDA cores, for FP32 inputs.
//
// The chunk formula is an exact reorganisation of the token recurrence
// ("Linear attention：把历史写进状态", sections "一个 chunk 的输出由两部分组成" and
// "动手实验": chunk boundaries do not change the result), so for FP32 inputs, where
// BF16 tensor-core operands would not meet a 1e-5 tolerance, this kernel runs
// the recurrence itself in FP32 (section "最小递推里，每一行都有张量意义"):
//     S <- alpha_t S + phi(k_t) v_t^T,  z <- alpha_t z + phi(k_t),
//     y_t = phi(q_t)^T S / (phi(q_t)^T z + eps).
// One CTA of 256 threads per (b, h, slice of up to 128 value columns): the slice
// of S [r x 128] lives in shared memory, thread j owns column j of the slice;
// thread i < r owns feature i of z (z and the denominator are recomputed by the
// CTAs of every slice, which need them alike).  The slices of a head run as one
// thread-block cluster.

#include "kernels.h"

namespace la {
namespace {

constexpr int kMaxR = 256;       // features (threads)
constexpr int kSlice = 128;      // value columns per CTA

__device__ __forceinline__ float phi_exact(float x) { return x > 0.f ? x + 1.f : expf(x); }

__global__ void __launch_bounds__(kMaxR)
prefill_f32_kernel(const float *__restrict__ q, const float *__restrict__ k, const float *__restrict__ v,
                   const float *__restrict__ alpha, const float *__restrict__ S0, const float *__restrict__ z0,
                   int H, int T, int r, int dv, float eps, float *__restrict__ y, float *S_out, float *z_out,
                   float *__restrict__ d_out)
{
    extern __shared__ float S[];   // [r][ds]
    __shared__ float qf[kMaxR], kf[kMaxR], red[kMaxR / 32];
    const int bh = blockIdx.y * H + blockIdx.x;
    const int c0 = blockIdx.z * kSlice, ds = min(kSlice, dv - c0);   // this CTA's value columns
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    for (int e = tid; e < r * ds; e += blockDim.x) {
        const int i = e / ds, j = e - i * ds;
        S[e] = S0 ? S0[((size_t)bh * r + i) * dv + c0 + j] : 0.f;
    }
    float zi = (tid < r && z0) ? z0[(size_t)bh * r + tid] : 0.f;
    // The slices of one head form a cluster: no slice may write z_out (which may
    // alias z0) before every slice has read z0.
    if (gridDim.z > 1) {
        asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
        asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    }
    __syncthreads();

    const float *qh = q + (size_t)bh * T * r, *kh = k + (size_t)bh * T * r, *vh = v + (size_t)bh * T * dv + c0;
    float *yh = y + (size_t)bh * T * dv + c0;
    for (int t = 0; t < T; ++t) {
        const float a = alpha ? alpha[(size_t)bh * T + t] : 1.f;
        float part = 0.f;
        if (tid < r) {
            const float qv = phi_exact(qh[(size_t)t * r + tid]);
            const float kv = phi_exact(kh[(size_t)t * r + tid]);
            qf[tid] = qv;
            kf[tid] = kv;
            zi = fmaf(a, zi, kv);
            part = qv * zi;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
        if (lane == 0) red[warp] = part;
        __syncthreads();
        if (tid < ds) {
            float den = 0.f;
#pragma unroll
            for (int w = 0; w < kMaxR / 32; ++w) den += red[w];
            const float vj = vh[(size_t)t * dv + tid];
            float n = 0.f;
            for (int i = 0; i < r; ++i) {
                const float s = fmaf(a, S[i * ds + tid], kf[i] * vj);
                S[i * ds + tid] = s;
                n = fmaf(qf[i], s, n);
            }
            yh[(size_t)t * dv + tid] = n / (den + eps);
            if (d_out && tid == 0 && blockIdx.z == 0) d_out[(size_t)bh * T + t] = den + eps;
        }
        __syncthreads();
    }
    for (int e = tid; e < r * ds; e += blockDim.x) {
        const int i = e / ds, j = e - i * ds;
        S_out[((size_t)bh * r + i) * dv + c0 + j] = S[e];
    }
    if (tid < r && blockIdx.z == 0) z_out[(size_t)bh * r + tid] = zi;
}

}  // namespace

cudaError_t launch_prefill_f32(const float *q, const float *k, const float *v, const float *alpha, const float *S0,
                               const float *z0, int B, int H, int T, int r, int dv, float eps, float *y,
                               float *S_out, float *z_out, cudaStream_t stream, float *d_out)
{
    const int ds = dv < kSlice ? dv : kSlice;
    const size_t smem = sizeof(float) * (size_t)r * ds;
    // The attribute is set once per device to the largest size this kernel accepts.
    static OncePerDevice attr_set;
    const cudaError_t e = set_smem_once(prefill_f32_kernel, (uint32_t)(sizeof(float) * kMaxR * kSlice), attr_set);
    if (e != cudaSuccess) return e;
    const int nslice = (dv + kSlice - 1) / kSlice;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(H, B, nslice);
    cfg.blockDim = dim3(kMaxR, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = nslice;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, prefill_f32_kernel, q, k, v, alpha, S0, z0, H, T, r, dv, eps, y, S_out, z_out,
                              d_out);
}

}  // namespace la
