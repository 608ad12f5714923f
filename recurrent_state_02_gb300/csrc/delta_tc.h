// delta_tc.h -- launcher of the chunked tensor-core delta-rule kernel (internal).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace la {

struct DeltaTcArgs {
    const float *beta;    // [B,H,T] or nullptr (beta == 1)
    const float *S0;      // [B,H,128,dv] or nullptr (zero); 16-byte aligned
    float *S_out;         // [B,H,128,dv]; may equal S0; 16-byte aligned
    uint16_t *y;          // [B,H,T,dv] BF16 bits
    void *ws;             // [B*H][ceil(T/64)][16 KB]: A = (Q K^T) . M and T of every chunk
                          // (BF16 shared-memory images, 8 KB each)
    int H, T, dv;         // T >= 1, dv a multiple of 64
    int *status;          // device status word
    unsigned long long wait_limit_ns;
};

// Bytes of the workspace launch_delta_tc needs (16-byte aligned).
size_t delta_tc_workspace_bytes(int B, int H, int T);

// BF16 delta rule in chunks of 64 tokens on the tensor cores; r == 128.  Two
// kernels: A and T of every chunk into a.ws, then the state chain, one CTA per
// (b, h, 64-column slice of v).  Tensor maps: q, k over [B*H, T, 128]; v over
// [B*H, T, dv] (BF16, 128-byte swizzle, boxes of 64 x 64).
cudaError_t launch_delta_tc(const CUtensorMap &map_q, const CUtensorMap &map_k, const CUtensorMap &map_v,
                            const DeltaTcArgs &a, int B, cudaStream_t stream);

}  // namespace la
