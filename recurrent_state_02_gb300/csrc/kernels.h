// kernels.h -- launchers behind the C ABI (internal; not part of the public header).
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace la {

// Per-device one-time set-up (kernel attributes, cached look-ups) for devices
// 0 .. kMaxDevices-1.  The flags and cached values are atomics: host threads
// that make their first call on a device at the same time may each do the
// (idempotent) set-up, and none reads a half-written value.
constexpr int kMaxDevices = 64;
struct OncePerDevice {
    std::atomic<bool> done[kMaxDevices];
};

// The current device, or -1 when it cannot be read or lies beyond kMaxDevices.
inline int current_device_index()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

// Raises kern's dynamic shared-memory limit to `bytes`, once per device (the
// first call on a device must not be inside a stream capture).
template <typename K>
cudaError_t set_smem_once(K kern, uint32_t bytes, OncePerDevice &once)
{
    const int dev = current_device_index();
    if (dev < 0) return cudaErrorInvalidDevice;
    if (!once.done[dev].load(std::memory_order_acquire)) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
        if (e != cudaSuccess) return e;
        once.done[dev].store(true, std::memory_order_release);
    }
    return cudaSuccess;
}

// Device status word values (same numbering as la_status).
constexpr int kStatusShape = 2;
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
    float *d_out = nullptr;   // alpha's layout, or nullptr: d_t = phi(q_t) . z_t + eps of every token
    // or nullptr: the state [S | z] entering every bwd_seg_chunks-th chunk, for the
    // backward's segments ([bwd_nseg][bwd_heads][128 * dv + 128], dv == 128)
    float *bwd_states = nullptr;
    int bwd_seg_chunks = 0, bwd_nseg = 0, bwd_heads = 0;
    int H, T, dv;
    int nseg;             // sequence segments per head (1: the whole sequence in one CTA)
    int seg_chunks;       // chunks per segment (nseg > 1)
    const float *S_start; // nseg > 1: [nseg][B*H][128*dv + 128] start state of each segment (S then z)
    // Packed sequences of different lengths: sequence b is tokens cu_seqlens[b] ..
    // cu_seqlens[b+1]-1 of q, k [T, H, 128], v, y [T, H, dv], alpha [T, H] (T the
    // total); the tensor maps are token-major views.  nullptr: [B, H, T, d] layout.
    const int *cu_seqlens;
    // Packed sequences split into segments (the varlen plan's tables; else nullptr):
    // items[blockIdx.z] = (b, g), segment g of sequence b (b < 0: no work; the
    // plan writes the longest segments first), and seq_info[b] = (segments, first
    // S_start slot, first boundary, 0).  A
    // sequence of more than one segment starts every segment from S_start[slot + g]
    // ([slot][H][128*dv + 128]); one of a single segment reads S0 itself.
    const int2 *items = nullptr;
    const int4 *seq_info = nullptr;
    const int *seg_len = nullptr;   // with items: chunks per segment (in place of seg_chunks)
    float eps;
    int *status;          // device status word
    unsigned long long wait_limit_ns;
};

// BF16 tensor-core prefill; r == 128, dv a multiple of dvs, chunk 64.  dvs: value
// columns per CTA, 64 (the slices of a head form a cluster) or 128 (one CTA per
// head and segment).  Tensor maps: q, k over [B*H, T, 128]; v over [B*H, T, dv]
// (BF16, 128-byte swizzle, boxes of 64 x 64).
// grid_z (0: B * nseg) rows of CTAs; the varlen plan's item count when a.items is set.
cudaError_t launch_prefill_tc(const CUtensorMap &map_q, const CUtensorMap &map_k,
                              const CUtensorMap &map_v, const PrefillTcArgs &a, int B, bool gated, int dvs,
                              cudaStream_t stream, int grid_z = 0);

// State pass of the sequence-segmented BF16 prefill (r == 128, dv a multiple of
// dvs, chunk 64): for every sub-segment of a head's sequence, the state it would
// produce from a zero state and the product of its gates.
struct StateTcArgs {
    const float *alpha;   // [B,H,T] or nullptr
    float *dS;            // [nsub][B*H][128*dv + 128]: S then z of each sub-segment
    float *A;             // [nsub][B*H]: product of each sub-segment's gates (1 without a gate)
    int H, T, dv;
    int nsub;             // sub-segments per head: the first nseg - 1 output segments,
    int sub_per_seg;      //   each split into sub_per_seg parts
    int sub_chunks;       // chunks per part (the last part of a segment may be shorter)
    int seg_chunks;       // chunks per output segment
    int seg_first = 0;    // segment of the first part (the reversed pass covers segments 1 .. nseg-1)
    const float *d = nullptr;    // reversed pass: d_t and dd_t [B*H*T] of the backward
    const float *dd = nullptr;
    // Packed sequences (token-major maps, alpha [T, H]): bds[k] = (b, g) for the
    // varlen plan's boundary k, the full segment g of sequence b that ends there
    // (b < 0: none); part j of it is CTA row k * sub + j (sub = seg_len[2]), and
    // its outputs are row (k * sub + j) * H + h of A and dS.
    const int *cu_seqlens = nullptr;
    const int2 *bds = nullptr;
    const int *seg_len = nullptr;   // with bds: chunks per segment, per part, parts per segment
    int *status;          // device status word
    unsigned long long wait_limit_ns;
};

// grid (dv/dvs, H, B*nsub) with dvs (64 or 128) value columns per CTA; tensor maps
// k over [B*H, T, 128] and v over [B*H, T, dv] as for launch_prefill_tc.
// rev: the backward's reversed pass (dvs 128, seg_first 1): k is the map of q,
// v the map of dy, and d, dd are given; the part maps carry [G | g].
// grid_z (0: B * nsub) rows of CTAs; boundaries * sub_per_seg when a.bds is set.
cudaError_t launch_state_tc(const CUtensorMap &map_k, const CUtensorMap &map_v, const StateTcArgs &a, int B,
                            bool gated, int dvs, cudaStream_t stream, bool rev = false, int grid_z = 0);

// The varlen plan: from cu_seqlens [B + 1] (device), the segment length L >=
// min_seg_chunks (from the batch's chunks, units CTAs per segment, sms SMs), and
// sequence b of c_b chunks takes max(1, ceil(c_b / L)) segments; with bounds
// outside [0, total_T] anywhere, or more than max_bds boundaries, one segment
// each; a valid sequence of at most walk_max tokens (-1: none) takes no segment
// (the token walk handles it).  Writes seg_len [3] (L, chunks per part, parts per
// boundary's segment, so that the boundaries fill about part_target of the
// part_rows >= max_bds rows), seq_info [B], items [B + max_bds] (longest segments
// first), bds [part_rows] and split_seqs [max_bds] (see PrefillTcArgs and
// StateTcArgs; unused entries -1).  One CTA.
cudaError_t launch_varlen_plan(const int *cu_seqlens, int B, int total_T, int min_seg_chunks, int units, int sms,
                               int max_bds, int part_rows, int part_target, int walk_max, int *seg_len,
                               int4 *seq_info, int2 *items, int2 *bds, int *split_seqs, cudaStream_t stream);

// The varlen scan: for every split sequence (split_seqs, max_bds entries) and head
// h, S_start[slot + 0] = S0[b], z0[b] (zero if null), then S_start[slot + g] the
// state after the maps of boundary (first + g - 1)'s parts, in order.
cudaError_t launch_varlen_scan(const float *S0, const float *z0, const float *A, const float *dS, float *S_start,
                               const int4 *seq_info, const int *split_seqs, const int *seg_len, int max_bds, int H,
                               int dv, cudaStream_t stream);

// S_start[g][bh] (S then z) for g < nseg: S0/z0 (zero if null) carried through the
// sub-segment maps S -> A S + dS in order.  rev: the maps of the reversed pass,
// applied from the last part backwards to S0/z0 (dL/dS_T, dL/dz_T), give the
// state entering segment g from the right in S_start[g].
cudaError_t launch_seg_scan(const float *S0, const float *z0, const float *A, const float *dS, float *S_start,
                            int BH, int dv, int nsub, int sub_per_seg, int nseg, cudaStream_t stream,
                            bool rev = false);

// Exact FP32 token recurrence (CUDA cores), r, dv <= 256.
cudaError_t launch_prefill_f32(const float *q, const float *k, const float *v, const float *alpha,
                               const float *S0, const float *z0, int B, int H, int T, int r, int dv,
                               float eps, float *y, float *S_out, float *z_out, cudaStream_t stream,
                               float *d_out = nullptr);

// Decode step; bf16 selects the q/k/v/y element type (else FP32).
cudaError_t launch_decode(const void *q, const void *k, const void *v, bool bf16, const float *alpha,
                          float *S, float *z, int B, int H, int r, int dv, float eps, void *y,
                          bool fast128, cudaStream_t stream);
// T tokens per (b, h) (r = dv = 128) from S0, z0 (nullptr: zero) into S_out, z_out
// (may alias), y [B,H,T,dv]; d_out (or nullptr) [B,H,T].
// The same walk over packed sequences (token-major, cu_seqlens [B + 1]): sequence
// b's H heads are walked when its bounds lie in [0, total_T] and it has at most
// 32 tokens (none of them: S0, z0 copied); the others are left untouched.
cudaError_t launch_decode_multi_packed(const void *q, const void *k, const void *v, bool bf16, const float *alpha,
                                       const float *S0, const float *z0, float *S_out, float *z_out,
                                       const int *cu_seqlens, int B, int H, int total_T, float eps, void *y,
                                       cudaStream_t stream);
cudaError_t launch_decode_multi(const void *q, const void *k, const void *v, bool bf16, const float *alpha,
                                const float *S0, const float *z0, float *S_out, float *z_out, int B, int H, int T,
                                float eps, void *y, float *d_out, cudaStream_t stream);

// Delta-rule memory, token recurrence in FP32 (CUDA cores): r in {32, 64, 128, 256},
// dv a multiple of 32; q, k, v, y 16-byte aligned; bf16 selects the q/k/v/y type.
cudaError_t launch_delta(const void *q, const void *k, const void *v, bool bf16, const float *beta, const float *S0,
                         int B, int H, int T, int r, int dv, void *y, float *S_out, int *status,
                         unsigned long long limit_ns, cudaStream_t stream);

// Gradients of the gated recurrence (FP32 on CUDA cores): r, dv in {32, 64, 128};
// q, k, v, y, dy, dq, dk, dv_out 16-byte aligned.
struct BackwardArgs {
    const void *q, *k, *v, *y, *dy;             // [B,H,T,r] / [B,H,T,dv], element type per bf16 flag
    const float *alpha, *S0, *z0, *dS_T, *dz_T; // optional (nullptr)
    void *dq, *dk, *dv_out;                     // [B,H,T,r], [B,H,T,r], [B,H,T,dv]
    float *dalpha;                              // [B,H,T] (with alpha)
    float *dS0, *dz0;                           // [B,H,r,dv], [B,H,r]
    float *ws;                                  // backward_workspace_floats(B, H, T) floats
    const float *d_in = nullptr;                // [B,H,T] d_t from the forward, or nullptr (the z pass forms it)
    const float *states_in = nullptr;           // the forward's states at the segment starts, or nullptr
    int H, T, r, dv;
    float eps;
    int *status;                                // device status word
    unsigned long long limit_ns;
    // BF16 with r == dv == 128: tensor maps of q, k, v, dy over [B*H, T, 128] (boxes
    // of 64 x 64, 128-byte swizzle); the three sweeps then run on the tensor cores.
    // nullptr: the sweeps run on CUDA cores.
    const CUtensorMap *maps;
    // Tensor-core sweeps over sequence segments (nseg > 1): each CTA takes
    // seg_chunks chunks of one head; the entering states come from the state
    // passes (forward for dq, reversed for dk and dv), each split into nsub parts
    // (sub_per_seg per segment, sub_chunks chunks each), in seg_ws.
    int nseg = 1, seg_chunks = 0, sub_per_seg = 1, sub_chunks = 0, nsub = 0;
    float *seg_ws = nullptr;
};
size_t backward_workspace_floats(int B, int H, int T);

// The three gradient sweeps on the tensor cores (BF16, r == dv == 128), given
// d_t (with eps) and dd_t: dq, dk, dv, the dlog alpha terms (tok_sum, fin; may be
// nullptr without a gate) and dS0, dz0.
struct BwdTcArgs {
    const float *alpha, *S0, *z0, *dS_T, *dz_T;  // optional (nullptr)
    const float *d, *dd;                         // [B*H*T]
    const uint16_t *q, *k;                       // BF16 [B,H,T,128] (phi and phi' in the epilogues)
    uint16_t *dq, *dk, *dv;                      // BF16 [B,H,T,128]
    float *tok_sum, *fin;                        // [B*H*T], [B*H] (accumulated), or nullptr
    float *dS0, *dz0;                            // [B,H,128,128], [B,H,128]
    int H, T;
    // nseg > 1: CTA (g, h, b) takes chunks g * seg_chunks .. of its head and starts
    // from seg_state_f (dq) or seg_state_r (dk, dv) [nseg][B*H][128*128 + 128]
    int nseg = 1, seg_chunks = 0;
    const float *seg_state_f = nullptr, *seg_state_r = nullptr;
    int *status;
    unsigned long long limit_ns;
};
// Sweeps first_mode .. end_mode - 1 (0 dq, 1 dk, 2 dv), in that order.
cudaError_t launch_bwd_tc(const CUtensorMap *maps, const BwdTcArgs &a, int B, bool gated, cudaStream_t stream,
                          int first_mode = 0, int end_mode = 3);
cudaError_t launch_backward(const BackwardArgs &a, int B, bool bf16, cudaStream_t stream);

cudaError_t launch_state_init(float *S, float *z, long long n_S, long long n_z, cudaStream_t stream);

cudaError_t launch_wait_probe(int *status, unsigned long long limit_ns, cudaStream_t stream);

}  // namespace la
