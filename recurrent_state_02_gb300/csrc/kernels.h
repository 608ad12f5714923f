// kernels.h -- launchers behind the C ABI (internal; not part of the public header).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace la {

// Device status word values (same numbering as la_status).
constexpr int kStatusTimeout = 7;

// Default limit for every on-chip barrier wait inside a kernel.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

struct PrefillTcArgs {
    const float *alpha;   // [B,H,T] or nullptr
    const float *S0;      // [B,H,128,dv] or nullptr
    const float *z0;      // [B,H,128] or nullptr
    float *S_out;         // [B,H,128,dv]
    float *z_out;         // [B,H,128]
    uint16_t *y;          // [B,H,T,dv] BF16 bits
    int H, T, dv;
    float eps;
    int *status;          // device status word
    unsigned long long wait_limit_ns;
};

// BF16 tensor-core prefill; r == 128, dv a multiple of 64, chunk 64.
// Tensor maps: q, k over [B*H, T, 128]; v over [B*H, T, dv] (BF16, 128-byte
// swizzle, boxes of 64 x 64).
cudaError_t launch_prefill_tc(const CUtensorMap &map_q, const CUtensorMap &map_k,
                              const CUtensorMap &map_v, const PrefillTcArgs &a, int B, bool gated,
                              cudaStream_t stream);

// Exact FP32 token recurrence (CUDA cores), r, dv <= 128.
cudaError_t launch_prefill_f32(const float *q, const float *k, const float *v, const float *alpha,
                               const float *S0, const float *z0, int B, int H, int T, int r, int dv,
                               float eps, float *y, float *S_out, float *z_out, cudaStream_t stream);

// Decode step; bf16 selects the q/k/v/y element type (else FP32).
cudaError_t launch_decode(const void *q, const void *k, const void *v, bool bf16, const float *alpha,
                          float *S, float *z, int B, int H, int r, int dv, float eps, void *y,
                          bool fast128, cudaStream_t stream);

cudaError_t launch_state_init(float *S, float *z, long long n_S, long long n_z, cudaStream_t stream);

cudaError_t launch_wait_probe(int *status, unsigned long long limit_ns, cudaStream_t stream);

}  // namespace la
