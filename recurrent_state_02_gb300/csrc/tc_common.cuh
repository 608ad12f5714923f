// tc_common.cuh -- device helpers shared by the tensor-core linear-attention
// kernels: bounded mbarrier waits with a CTA-wide abort flag, warp-level
// arrive/wait, the packed-BF16 feature map phi(x) = ELU(x) + 1, row scaling
// and the per-chunk gate products.
#pragma once

#include "kernels.h"
#include "sm103_ptx.cuh"

#include <cuda_bf16.h>

namespace la {
namespace {

constexpr int kC = 64;          // tokens per chunk
constexpr int kR = 128;         // feature width r

#ifndef LA_WAIT_HINT_NS
#define LA_WAIT_HINT_NS 20000
#endif
constexpr uint32_t kWaitHintNs = LA_WAIT_HINT_NS;


// Gate data ring depth: the producer writes chunk c's entry at most a stage ring
// (of at most kAux stages) ahead of its consumers: once it may refill the stage
// of chunk c - stages, every consumer has released the entry of that chunk.
constexpr int kAux = 4;

// Gate products of the chunks in flight (gated kernel only; chunk c in entry c % kAux).
struct alignas(16) GateRing {
    float gb[kAux][kC];         // cumulative log gate inside the chunk
    int gz[kAux][kC];           // last row <= i whose gate is 0 (-1: none)
    float gG[kAux][kC];         // Gamma_i
    float gw[kAux][kC];         // w_j
    int gf[kAux];               // 1: no zero gate and w_0 >= 2^-64 (see kFastGateLog)
};

// A chunk whose smallest write weight w_0 = e^{b_last - b_0} is at least
// e^{kFastGateLog} (and which has no zero gate) may carry its gates as row
// weights w_j on V (the rows of the scaled accumulators then stay far from
// FP32 underflow); others take the exact path of explicit gate products.
constexpr float kFastGateLog = -44.0f;   // e^-44 ~ 2^-63.5

// phi(x) = ELU(x) + 1 on a pair of BF16 values, in packed BF16 arithmetic:
// phi(x) = max(min(e^x, 1), x + 1).  For x <= 0, e^x >= 1 + x picks e^x; for
// x > 0, min(e^x, 1) = 1 <= x + 1 picks x + 1 (NaN propagates through the .NaN
// forms).  e^x = 2^(x log2 e) with log2 e split into two BF16 parts, so that
// the product is rounded once; the base-2 exponential is the hardware
// approximation with flush-to-zero (phi = 0 below x = -87.3).
__device__ __forceinline__ uint32_t phi_bf16x2(uint32_t x)
{
    constexpr uint32_t kLog2eHi = 0x3FB93FB9u;   // 1.4453125
    constexpr uint32_t kLog2eLo = 0xBB2CBB2Cu;   // -0.00262451171875
    constexpr uint32_t kOne = 0x3F803F80u;
    constexpr uint32_t kZero = 0x80008000u;      // -0
    uint32_t t, e, p, r;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(t) : "r"(x), "r"(kLog2eLo), "r"(kZero));
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(t) : "r"(x), "r"(kLog2eHi), "r"(t));
    asm("ex2.approx.ftz.bf16x2 %0, %1;" : "=r"(e) : "r"(t));
    asm("min.NaN.bf16x2 %0, %1, %2;" : "=r"(e) : "r"(e), "r"(kOne));
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(p) : "r"(x), "r"(kOne), "r"(kOne));
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(e), "r"(p));
    return r;
}

struct Ctx {
    int *abort_flag;   // CTA-wide flag in shared memory
    uint64_t limit;    // wait limit in ns
    int *status;       // device status word
};

// Records a timeout once and raises the CTA-wide abort flag.
__device__ __noinline__ void fail(Ctx &cx)
{
    if (!*reinterpret_cast<volatile int *>(cx.abort_flag)) {
        atomicExch(cx.status, kStatusTimeout);
        *reinterpret_cast<volatile int *>(cx.abort_flag) = 1;
    }
}

__device__ __forceinline__ bool aborted(const Ctx &cx)
{
    return *reinterpret_cast<volatile int *>(cx.abort_flag) != 0;
}

// Bounded wait by one thread.  Gives up when the time limit runs out (and then
// raises the abort flag) or as soon as another thread has raised it.  HINT_NS:
// how long the thread may be suspended in hardware per try while the phase is
// incomplete (0: it polls).
template <uint32_t HINT_NS = kWaitHintNs>
__device__ __forceinline__ bool wait(Ctx &cx, uint64_t *bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (HINT_NS ? mbar_try_wait_hint(bar, parity, HINT_NS) : mbar_try_wait(bar, parity)) return true;
        if (aborted(cx)) return false;
        if (global_timer_ns() - t0 > cx.limit) {
            fail(cx);
            return false;
        }
    }
}

// Warp-wide wait.  Fast path: every lane tests the phase (each lane acquires
// for itself) and the vote keeps the branch uniform.  Otherwise lane 0 waits
// (bounded) while the other lanes are parked at the warp barrier; the outcome
// is broadcast so that the warp stays converged for the .sync.aligned
// instructions that follow, and the warp barrier orders the other lanes'
// later accesses after lane 0's acquire.
__device__ __forceinline__ bool warp_wait(Ctx &cx, uint64_t *bar, uint32_t parity)
{
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    int ok = 1;
    if ((threadIdx.x & 31) == 0) ok = wait(cx, bar, parity);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    return ok != 0;
}

// One arrival per warp, after every lane's preceding writes and fences (the
// warp barrier orders them before lane 0's release).
__device__ __forceinline__ void warp_arrive(uint64_t *bar)
{
    __syncwarp();
    mbar_arrive_if(bar, (threadIdx.x & 31) == 0);
}

// Applies phi to the 8 BF16 values of one 16-byte chunk.
__device__ __forceinline__ uint4 phi8(uint4 raw)
{
    return make_uint4(phi_bf16x2(raw.x), phi_bf16x2(raw.y), phi_bf16x2(raw.z), phi_bf16x2(raw.w));
}

// Multiplies the 8 BF16 values of one 16-byte chunk by s, rounded to BF16: one
// packed multiply per pair (the product is rounded to BF16 again).
__device__ __forceinline__ uint4 scale8(uint4 raw, float s)
{
    const uint32_t s2 = pack_bf16x2(s, s);
    uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(w[e]) : "r"(w[e]), "r"(s2));
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Gate products of one chunk, by one warp; lane l holds tokens 2l and 2l + 1
// (gates past the end of the sequence are 1).  b_i is the in-chunk inclusive
// sum of log alpha, zl_i the last row <= i whose gate is exactly 0 (-1: none);
// Gamma_i = e^{b_i} (0 once a zero gate has been passed) and w_j =
// e^{b_last - b_j} (0 for keys before the chunk's last zero gate).
__device__ __forceinline__ void gate_products(float a0, float a1, int lane, int gq, GateRing *gr)
{
    const int j0 = 2 * lane;
    const float l0 = a0 > 0.f ? logf(a0) : 0.f;
    const float l1 = a1 > 0.f ? logf(a1) : 0.f;
    const int zp0 = a0 > 0.f ? -1 : j0;
    const int zp1 = a1 > 0.f ? zp0 : j0 + 1;
    // inclusive warp scan of the pair totals (sum) and the pair's last zero gate (max)
    float inc = l0 + l1;
    int zinc = zp1;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float lo = __shfl_up_sync(0xffffffffu, inc, off);
        const int zo = __shfl_up_sync(0xffffffffu, zinc, off);
        if (lane >= off) { inc += lo; zinc = max(zinc, zo); }
    }
    float ex = __shfl_up_sync(0xffffffffu, inc, 1);
    int zex = __shfl_up_sync(0xffffffffu, zinc, 1);
    if (lane == 0) { ex = 0.f; zex = -1; }
    const float b0 = ex + l0, b1 = b0 + l1;
    const int z0 = max(zex, zp0), z1 = max(zex, zp1);
    const float blast = __shfl_sync(0xffffffffu, b1, 31);
    const int zlast = __shfl_sync(0xffffffffu, z1, 31);
    const float w0 = zlast <= j0 ? expf(blast - b0) : 0.f;
    const float w1 = zlast <= j0 + 1 ? expf(blast - b1) : 0.f;
    *reinterpret_cast<float2 *>(&gr->gb[gq][j0]) = make_float2(b0, b1);
    *reinterpret_cast<int2 *>(&gr->gz[gq][j0]) = make_int2(z0, z1);
    *reinterpret_cast<float2 *>(&gr->gG[gq][j0]) = make_float2(z0 < 0 ? expf(b0) : 0.f, z1 < 0 ? expf(b1) : 0.f);
    *reinterpret_cast<float2 *>(&gr->gw[gq][j0]) = make_float2(w0, w1);
    const float bfirst = __shfl_sync(0xffffffffu, b0, 0);
    if (lane == 0) gr->gf[gq] = (zlast < 0 && blast - bfirst >= kFastGateLog) ? 1 : 0;
}

}  // namespace
}  // namespace la
