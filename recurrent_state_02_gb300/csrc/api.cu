// api.cu -- the C ABI declared in include/linattn.h: argument validation,
// kernel selection, TMA descriptor set-up and the device status word.
#include "../../include/linattn.h"
#include "delta_tc.h"
#include "kernels.h"
#include "side_lane.h"

#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace {

// Device status word: 0, or the la_status of the last failure a kernel recorded.
__device__ int g_status = 0;

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    // looked up once; concurrent first calls may each look it up (same value)
    static std::atomic<EncodeTiledFn> cached{nullptr};
    EncodeTiledFn fn = cached.load(std::memory_order_acquire);
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess) {
            fn = reinterpret_cast<EncodeTiledFn>(p);
            cached.store(fn, std::memory_order_release);
        }
    }
    return fn;
}

// Sequence segmentation of the BF16 prefill.  The chunk kernel runs one CTA per
// (b, h, dvs-column slice): 64-column slices when they fill one wave of the GPU
// without segments, a whole head (dv == 128) otherwise -- it forms phi(Q),
// phi(K) and the scores once per head, about half the instructions of two
// slices per chunk, but a chunk takes longer; when that leaves at least half of
// the SMs idle and
// the sequence is long enough, every head's chunks are split into nseg segments
// that run in parallel from scanned start states.  The state pass over the first
// nseg - 1 segments runs one CTA per (b, h, dvs-column slice, part), two resident
// per SM; each segment is cut into sub_per_seg parts, the count that minimises
// (waves of state CTAs) x (chunks per part + a per-CTA set-up cost).
// LA_HEAD_CTA: 0 = always slices, 1 = the rule above, 2 = whole heads whenever dv == 128
#ifndef LA_HEAD_CTA
#define LA_HEAD_CTA 1
#endif
// Continuations of at most this many tokens take the decode-shaped token walk.
#ifndef LA_DECODE_MAX_T
#define LA_DECODE_MAX_T 32
#endif
constexpr int kMinSegChunks = 16;    // at least 1024 tokens per segment
constexpr int kStateCtasPerSm = 2;   // resident state-pass CTAs per SM
constexpr int kStateCtaSetup = 2;    // set-up and pipeline fill of a state CTA, in chunks
// Largest workspace a plan may ask for.  With one part per segment every plan of
// a device with up to about 240 SMs stays below it (the plan keeps
// (parts + segments) * heads below about 2 * SMs states of 66 KB); finer parts
// are used only while they fit.
constexpr size_t kMaxPlanWorkspace = size_t(32) << 20;
constexpr size_t kMaxBwdPlanWorkspace = size_t(1) << 30;   // the backward's two state passes

struct SegPlan {
    int dvs = 64;   // value columns per chunk-kernel CTA
    int nseg = 1, seg_chunks = 0, sub_per_seg = 1, sub_chunks = 0, nsub = 0;
};

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace (FP32): A [nsub][B*H], dS [nsub][B*H][state], S_start [nseg][B*H][state],
// state = 128*dv + 128 (S then z); every part starts on a 256-byte boundary.
size_t seg_workspace_bytes(int nsub, int nseg, int B, int H, int dv)
{
    if (nseg <= 1) return 0;
    const size_t BH = (size_t)B * H, state = 128 * (size_t)dv + 128;
    return round_up((size_t)nsub * BH * 4, 256) + (size_t)nsub * BH * state * 4 + (size_t)nseg * BH * state * 4;
}

int sm_count()
{
    static std::atomic<int> count[la::kMaxDevices];
    const int dev = la::current_device_index();
    if (dev < 0) return 0;
    int n = count[dev].load(std::memory_order_relaxed);
    if (!n) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        count[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

// Value columns per chunk-kernel CTA for B*H heads of dv columns on `sms` SMs.
int head_width(long long B, long long H, int dv, long long sms)
{
    if (dv != 128 || LA_HEAD_CTA == 0) return 64;
    if (LA_HEAD_CTA == 2) return 128;
    const long long slices = B * H * (dv / 64);
    return (5 * slices >= 4 * sms && slices <= sms) ? 64 : 128;
}

// Segments of nch chunks for `units` chunk-kernel CTAs per segment (one resident
// per SM), and the parts of the state pass over nseg - 1 of them (one CTA per
// (unit of the state pass, part), kStateCtasPerSm resident per SM), within
// max_ws bytes of workspace (ws_of(nsub, nseg)).
template <typename WsFn>
SegPlan plan_segments(SegPlan p, long long units, long long state_units, int nch, long long max_ws, WsFn ws_of)
{
    const long long sms = sm_count();
    long long g = units > 0 ? sms / units : 0;
    g = g < nch / kMinSegChunks ? g : nch / kMinSegChunks;
    if (g < 2) return p;
    const int L = (int)((nch + g - 1) / g);
    const int G = (nch + L - 1) / L;
    if (G < 2) return p;
    const long long sunits = state_units * (G - 1);
    const long long slots = kStateCtasPerSm * sms;
    long long best_cost = -1;
    int best_n = 1;
    for (int n = 1; n <= L; ++n) {
        const int Ln = (L + n - 1) / n, parts = (L + Ln - 1) / Ln;
        if (n > 1 && (long long)ws_of((G - 1) * parts, G) > max_ws) break;
        const long long waves = (sunits * n + slots - 1) / slots;
        const long long cost = waves * ((L + n - 1) / n + kStateCtaSetup);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best_n = n;
        }
    }
    const int L1 = (L + best_n - 1) / best_n;
    p.nseg = G;
    p.seg_chunks = L;
    p.sub_chunks = L1;
    p.sub_per_seg = (L + L1 - 1) / L1;
    p.nsub = (G - 1) * p.sub_per_seg;
    return p;
}

SegPlan seg_plan(int B, int H, int T, int dv)
{
    SegPlan p;
    p.dvs = head_width(B, H, dv, sm_count());
    const long long units = (long long)B * H * (dv / p.dvs);   // chunk-kernel CTAs per segment
    return plan_segments(p, units, units, (T + 63) / 64, (long long)kMaxPlanWorkspace,
                         [&](int nsub, int nseg) { return seg_workspace_bytes(nsub, nseg, B, H, dv); });
}

// The backward's tensor-core sweeps (one whole-head CTA per segment) over the
// same kind of segments; their two state passes (forward for dq, reversed for
// dk and dv) take whole heads too, and each has a workspace of the forward's layout.
SegPlan bwd_seg_plan(int B, int H, int T)
{
    SegPlan p;
    p.dvs = 128;
    const long long units = (long long)B * H;
    return plan_segments(p, units, units, (T + 63) / 64, (long long)kMaxBwdPlanWorkspace,
                         [&](int nsub, int nseg) { return 2 * seg_workspace_bytes(nsub, nseg, B, H, 128); });
}

size_t seg_workspace_bytes(const SegPlan &p, int B, int H, int dv)
{
    return seg_workspace_bytes(p.nsub, p.nseg, B, H, dv);
}

// Segments of a packed batch (la_prefill_varlen).  The host knows B, H and the
// total only; the device plan splits each sequence into segments of L >= min_seg
// chunks once it has read the lengths, so min_seg bounds the boundaries by
// total_T / (64 min_seg).  min_seg is a quarter of an SM's share of the largest
// possible batch of CTA-chunks, which keeps (boundaries x CTAs per segment) below
// 4 SMs' worth, and so the workspace, whatever the total.  The state pass gets
// part_rows >= max_bds rows of CTAs; the plan shares about one wave of them
// (part_target) among the boundaries it makes (more parts would shorten the
// pass but lengthen the scan, which composes them one after another).  With the
// token walk for short sequences the plan is made even when no sequence can be
// split (max_bds 0: its tables only).  Workspace (256-byte aligned parts):
// seg_len int[3], seq_info int4[B], items int2[B + max_bds], bds int2[part_rows],
// split_seqs int[max_bds], A and dS of part_rows parts, and 2 max_bds start-state
// slots (a split sequence has at most twice as many segments as boundaries).
struct VarlenPlan {
    int dvs = 64, units = 0, min_seg = 0, max_bds = 0, part_rows = 0, part_target = 0;
    size_t off_info = 0, off_items = 0, off_bds = 0, off_split = 0, off_A = 0, off_dS = 0, off_S = 0, bytes = 0;
};

// walk: short sequences go to the token walk, which needs the plan's tables even
// when no sequence can be split.
VarlenPlan varlen_plan(int B, int H, int total_T, int dv, bool walk)
{
    VarlenPlan p;
    const long long sms = sm_count();
    p.dvs = head_width(B, H, dv, sms);
    p.units = H * (dv / p.dvs);
    if (sms <= 0 || total_T < 0 || B < 1 || B > 65535) return p;
    const long long work = ((long long)(total_T + 63) / 64 + B) * p.units;   // CTA-chunks at most
    long long L = (work + 4 * sms - 1) / (4 * sms);
    if (L < kMinSegChunks) L = kMinSegChunks;
    long long nb = (long long)total_T / (64 * L);
    if (B + nb > 65535) nb = 0;   // grid rows of the chunk kernel
    if (nb < 1 && !walk) return p;
    const long long wave = (kStateCtasPerSm * sms + p.units - 1) / p.units;
    long long rows = nb < 1 ? 0 : wave < nb ? nb : wave;
    if (rows > 65535) rows = 65535;
    p.min_seg = (int)L;
    p.max_bds = (int)nb;
    p.part_rows = (int)rows;
    p.part_target = (int)(wave < rows ? wave : rows);
    const size_t state = 128 * (size_t)dv + 128;
    p.off_info = 256;   // after seg_len
    p.off_items = p.off_info + round_up(16 * (size_t)B, 256);
    p.off_bds = p.off_items + round_up(8 * ((size_t)B + nb), 256);
    p.off_split = p.off_bds + round_up(8 * (size_t)rows, 256);
    p.off_A = p.off_split + round_up(4 * (size_t)nb, 256);
    p.off_dS = p.off_A + round_up(4 * (size_t)rows * H, 256);
    p.off_S = p.off_dS + round_up(4 * (size_t)rows * H * state, 256);
    p.bytes = p.off_S + 4 * 2 * (size_t)nb * H * state;
    return p;
}

// Scratch of la_prefill_chunked_noalloc: a fixed buffer in the library's device
// image, for callers that cannot pass device memory of their own.  It holds the
// largest workspace a plan asks for (kMaxPlanWorkspace).
constexpr size_t kNoAllocScratchBytes = kMaxPlanWorkspace;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch on the current device, looked up once per device
// (the first call there does it, with that device current); nullptr on failure.
// Host threads whose first calls on a device meet may each look it up: the
// cache is an atomic, and every look-up yields the same address.
void *noalloc_scratch()
{
    static std::atomic<void *> addr[la::kMaxDevices];
    const int dev = la::current_device_index();
    if (dev < 0) return nullptr;
    void *p = addr[dev].load(std::memory_order_acquire);
    if (!p) {
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
        addr[dev].store(p, std::memory_order_release);
    }
    return p;
}

// 3-D BF16 view [planes, rows, cols] (cols innermost) with boxes of box_cols x
// box_rows; rows past the end of a plane read as zero and are never written.
bool make_map_bf16(CUtensorMap *map, const void *ptr, long long planes, long long rows, long long cols,
                   unsigned box_cols, unsigned box_rows, CUtensorMapSwizzle swizzle)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)planes};
    const cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)cols * rows * 2};
    const cuuint32_t box[3] = {box_cols, box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Token-major packed view [tokens, heads, cols] (cols innermost): boxes of
// box_cols x 1 head x box_rows tokens, so a box lands in shared memory exactly
// like a box_rows x box_cols tile of the [planes, rows, cols] view.
bool make_map_bf16_tok(CUtensorMap *map, const void *ptr, long long tokens, long long heads, long long cols,
                       unsigned box_cols, unsigned box_rows, CUtensorMapSwizzle swizzle)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)heads, (cuuint64_t)(tokens > 0 ? tokens : 1)};
    const cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)cols * heads * 2};
    const cuuint32_t box[3] = {box_cols, 1, box_rows};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int *status_word()
{
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return nullptr;
    return static_cast<int *>(p);
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

la_status from_cuda(cudaError_t e) { return e == cudaSuccess ? LA_OK : LA_ERR_CUDA; }

}  // namespace

extern "C" {

const char *la_status_string(la_status s)
{
    switch (s) {
    case LA_OK: return "LA_OK";
    case LA_ERR_NULL: return "LA_ERR_NULL: a required pointer is NULL";
    case LA_ERR_SHAPE: return "LA_ERR_SHAPE: a size is out of range or sizes disagree";
    case LA_ERR_DTYPE: return "LA_ERR_DTYPE: unknown element type";
    case LA_ERR_ALIGN: return "LA_ERR_ALIGN: a pointer is not aligned as the kernel requires";
    case LA_ERR_UNSUPPORTED: return "LA_ERR_UNSUPPORTED: request not implemented by this build";
    case LA_ERR_CUDA: return "LA_ERR_CUDA: a CUDA runtime call or launch failed";
    case LA_ERR_TIMEOUT: return "LA_ERR_TIMEOUT: a kernel gave up waiting on an on-chip barrier";
    case LA_ERR_WORKSPACE: return "LA_ERR_WORKSPACE: workspace too small";
    }
    return "unknown la_status";
}

la_status la_state_init(float *S, float *z, int B, int H, int r, int dv, la_stream_t stream)
{
    if (!S || !z) return LA_ERR_NULL;
    if (B < 1 || H < 1 || r < 1 || dv < 1) return LA_ERR_SHAPE;
    if (!aligned(S, 4) || !aligned(z, 4)) return LA_ERR_ALIGN;
    const long long nz = (long long)B * H * r, nS = nz * dv;
    return from_cuda(la::launch_state_init(S, z, nS, nz, reinterpret_cast<cudaStream_t>(stream)));
}

size_t la_prefill_workspace_bytes(int B, int H, int T, int r, int dv, int chunk)
{
    if (B < 1 || H < 1 || T < 1 || r != 128 || (dv != 64 && dv != 128) || chunk < 1) return 0;
    return seg_workspace_bytes(seg_plan(B, H, T, dv), B, H, dv);
}

// la_prefill_chunked and la_prefill_chunked_save; d_out may be nullptr.
static la_status prefill_chunked_impl(const void *q, const void *k, const void *v, la_dtype dtype,
                                      const float *alpha, const float *S0, const float *z0, int B, int H, int T,
                                      int r, int dv, int chunk, float eps, void *y, float *S_out, float *z_out,
                                      float *d_out, float *states_out, void *workspace, size_t workspace_bytes,
                                      la_stream_t stream)
{
    if (!q || !k || !v || !y || !S_out || !z_out) return LA_ERR_NULL;
    if (B < 1 || H < 1 || T < 1 || r < 1 || dv < 1 || chunk < 1) return LA_ERR_SHAPE;
    if (dtype != LA_DTYPE_BF16 && dtype != LA_DTYPE_FP32) return LA_ERR_DTYPE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

    if (states_out && !aligned(states_out, 16)) return LA_ERR_ALIGN;
    if (dtype == LA_DTYPE_FP32) {
        if (r > 256 || dv > 256) return LA_ERR_UNSUPPORTED;
        const void *ptrs[] = {q, k, v, y, S_out, z_out, alpha, S0, z0, d_out};
        for (const void *p : ptrs)
            if (p && !aligned(p, 4)) return LA_ERR_ALIGN;
        return from_cuda(la::launch_prefill_f32(static_cast<const float *>(q), static_cast<const float *>(k),
                                                static_cast<const float *>(v), alpha, S0, z0, B, H, T, r, dv, eps,
                                                static_cast<float *>(y), S_out, z_out, st, d_out));
    }

    // BF16: tensor-core kernel.  It computes in chunks of 64 tokens whatever chunk
    // length is asked for: the result does not depend on the chunk length beyond
    // rounding ("Linear attention：把历史写进状态", section "动手实验").
    if (r != 128 || (dv != 64 && dv != 128)) return LA_ERR_UNSUPPORTED;
    if ((long long)B * H > 0x7fffffffLL) return LA_ERR_SHAPE;
    {
        const void *ptrs16[] = {q, k, v, y, S_out};
        for (const void *p : ptrs16)
            if (!aligned(p, 16)) return LA_ERR_ALIGN;
        const void *ptrs4[] = {alpha, S0, z0, z_out, d_out};
        for (const void *p : ptrs4)
            if (p && !aligned(p, 4)) return LA_ERR_ALIGN;
    }
    // A short continuation (a few tokens per request from a carried state) is a
    // decode-shaped job: the state-resident token walk reads and writes the state
    // once, where the chunk kernel's set-up for a single partial chunk would
    // dominate.  It computes the same recurrence in FP32 (phi in FP32 from the
    // inputs; no BF16 operands).
    if (T <= LA_DECODE_MAX_T && T <= 32 && dv == 128 && (!S0 || aligned(S0, 16)))
        return from_cuda(la::launch_decode_multi(q, k, v, true, alpha, S0, z0, S_out, z_out, B, H, T, eps, y, d_out,
                                                 st));
    const SegPlan plan = seg_plan(B, H, T, dv);
    const size_t need = seg_workspace_bytes(plan, B, H, dv);
    if (need) {
        if (!workspace || workspace_bytes < need) return LA_ERR_WORKSPACE;
        if (!aligned(workspace, 256)) return LA_ERR_ALIGN;
    }
    int *status = status_word();
    if (!status) return LA_ERR_CUDA;
    CUtensorMap mq, mk, mv;
    const long long planes = (long long)B * H;
    // q, k, v: 64 x 64 load boxes, 128-byte swizzle
    const CUtensorMapSwizzle sw128 = CU_TENSOR_MAP_SWIZZLE_128B;
    if (!make_map_bf16(&mq, q, planes, T, r, 64, 64, sw128) || !make_map_bf16(&mk, k, planes, T, r, 64, 64, sw128) ||
        !make_map_bf16(&mv, v, planes, T, dv, 64, 64, sw128))
        return LA_ERR_CUDA;
    la::PrefillTcArgs a;
    a.alpha = alpha;
    a.S0 = S0;
    a.z0 = z0;
    a.S_out = S_out;
    a.z_out = z_out;
    a.y = static_cast<uint16_t *>(y);
    a.d_out = d_out;
    if (states_out && r == 128 && dv == 128) {
        const SegPlan bp = bwd_seg_plan(B, H, T);
        if (bp.nseg > 1) {
            a.bwd_states = states_out;
            a.bwd_seg_chunks = bp.seg_chunks;
            a.bwd_nseg = bp.nseg;
            a.bwd_heads = B * H;
        }
    }
    a.H = H;
    a.T = T;
    a.dv = dv;
    a.eps = eps;
    a.status = status;
    a.wait_limit_ns = la::kWaitLimitNs;
    a.nseg = 1;
    a.seg_chunks = 0;
    a.S_start = nullptr;
    a.cu_seqlens = nullptr;
    if (need) {
        // state pass over the first nseg - 1 segments, scan, then every segment in parallel
        const size_t BH = (size_t)B * H, state = 128 * (size_t)dv + 128;
        float *ws = static_cast<float *>(workspace);
        float *A = ws;
        float *dS = ws + round_up((size_t)plan.nsub * BH * 4, 256) / 4;
        float *S_start = dS + (size_t)plan.nsub * BH * state;
        la::StateTcArgs sa;
        sa.alpha = alpha;
        sa.dS = dS;
        sa.A = A;
        sa.H = H;
        sa.T = T;
        sa.dv = dv;
        sa.nsub = plan.nsub;
        sa.sub_per_seg = plan.sub_per_seg;
        sa.sub_chunks = plan.sub_chunks;
        sa.seg_chunks = plan.seg_chunks;
        sa.status = status;
        sa.wait_limit_ns = la::kWaitLimitNs;
        cudaError_t e = la::launch_state_tc(mk, mv, sa, B, alpha != nullptr, plan.dvs, st);
        if (e == cudaSuccess)
            e = la::launch_seg_scan(S0, z0, A, dS, S_start, (int)BH, dv, plan.nsub, plan.sub_per_seg, plan.nseg, st);
        if (e != cudaSuccess) return from_cuda(e);
        a.nseg = plan.nseg;
        a.seg_chunks = plan.seg_chunks;
        a.S_start = S_start;
    }
    return from_cuda(la::launch_prefill_tc(mq, mk, mv, a, B, alpha != nullptr, plan.dvs, st));
}

la_status la_prefill_chunked(const void *q, const void *k, const void *v, la_dtype dtype, const float *alpha,
                             const float *S0, const float *z0, int B, int H, int T, int r, int dv, int chunk,
                             float eps, void *y, float *S_out, float *z_out, void *workspace,
                             size_t workspace_bytes, la_stream_t stream)
{
    return prefill_chunked_impl(q, k, v, dtype, alpha, S0, z0, B, H, T, r, dv, chunk, eps, y, S_out, z_out, nullptr,
                                nullptr, workspace, workspace_bytes, stream);
}

la_status la_prefill_chunked_save(const void *q, const void *k, const void *v, la_dtype dtype, const float *alpha,
                                  const float *S0, const float *z0, int B, int H, int T, int r, int dv, int chunk,
                                  float eps, void *y, float *S_out, float *z_out, float *d_out, float *states_out,
                                  void *workspace, size_t workspace_bytes, la_stream_t stream)
{
    if (!d_out) return LA_ERR_NULL;
    return prefill_chunked_impl(q, k, v, dtype, alpha, S0, z0, B, H, T, r, dv, chunk, eps, y, S_out, z_out, d_out,
                                states_out, workspace, workspace_bytes, stream);
}

size_t la_backward_states_bytes(int B, int H, int T)
{
    if (B < 1 || H < 1 || T < 1) return 0;
    const SegPlan p = bwd_seg_plan(B, H, T);
    return p.nseg > 1 ? sizeof(float) * (size_t)p.nseg * B * H * (128 * 128 + 128) : 0;
}

// The most tokens of a packed sequence the token walk takes (-1: none).
int varlen_walk_max() { return LA_DECODE_MAX_T < 1 ? -1 : LA_DECODE_MAX_T < 32 ? LA_DECODE_MAX_T : 32; }

size_t la_prefill_varlen_workspace_bytes(int B, int H, int total_T, int r, int dv)
{
    if (B < 1 || H < 1 || total_T < 0 || r != 128 || (dv != 64 && dv != 128)) return 0;
    if ((long long)B * H > 0x7fffffffLL || (long long)total_T * H > 0x7fffffffLL) return 0;
    // sized for the walk (which runs even when there are no tokens at all: the
    // states are handed on) (the call takes it when S0 allows)
    return varlen_plan(B, H, total_T, dv, dv == 128 && varlen_walk_max() >= 0).bytes;
}

la_status la_prefill_varlen(const void *q, const void *k, const void *v, la_dtype dtype, const float *alpha,
                            const float *S0, const float *z0, const int *cu_seqlens, int B, int H, int total_T,
                            int r, int dv, int chunk, float eps, void *y, float *S_out, float *z_out,
                            void *workspace, size_t workspace_bytes, la_stream_t stream)
{
    if (!cu_seqlens || !S_out || !z_out) return LA_ERR_NULL;
    if (total_T > 0 && (!q || !k || !v || !y)) return LA_ERR_NULL;
    if (B < 1 || H < 1 || total_T < 0 || r < 1 || dv < 1 || chunk < 1) return LA_ERR_SHAPE;
    if (dtype != LA_DTYPE_BF16 && dtype != LA_DTYPE_FP32) return LA_ERR_DTYPE;
    if (dtype != LA_DTYPE_BF16 || r != 128 || (dv != 64 && dv != 128)) return LA_ERR_UNSUPPORTED;
    if ((long long)B * H > 0x7fffffffLL || (long long)total_T * H > 0x7fffffffLL) return LA_ERR_SHAPE;
    {
        const void *ptrs16[] = {q, k, v, y, S_out};
        for (const void *p : ptrs16)
            if (p && !aligned(p, 16)) return LA_ERR_ALIGN;
        const void *ptrs4[] = {alpha, S0, z0, z_out, cu_seqlens};
        for (const void *p : ptrs4)
            if (p && !aligned(p, 4)) return LA_ERR_ALIGN;
    }
    // sequences of at most 32 tokens (a short continuation each) take the token walk,
    // which reads S0 as float4
    const int walk_max = (dv == 128 && (!S0 || aligned(S0, 16))) ? varlen_walk_max() : -1;
    const VarlenPlan plan = varlen_plan(B, H, total_T, dv, walk_max >= 0);
    if (plan.bytes) {
        if (!workspace || workspace_bytes < plan.bytes) return LA_ERR_WORKSPACE;
        if (!aligned(workspace, 256)) return LA_ERR_ALIGN;
    }
    int *status = status_word();
    if (!status) return LA_ERR_CUDA;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // token-major views [total_T, H, d]; with no tokens at all no tile is ever
    // loaded, and any aligned address serves as the maps' base
    const void *qb = total_T ? q : S_out, *kb = total_T ? k : S_out, *vb = total_T ? v : S_out;
    CUtensorMap mq, mk, mv;
    const CUtensorMapSwizzle sw128 = CU_TENSOR_MAP_SWIZZLE_128B;
    if (!make_map_bf16_tok(&mq, qb, total_T, H, r, 64, 64, sw128) || !make_map_bf16_tok(&mk, kb, total_T, H, r, 64, 64, sw128) ||
        !make_map_bf16_tok(&mv, vb, total_T, H, dv, 64, 64, sw128))
        return LA_ERR_CUDA;
    la::PrefillTcArgs a;
    a.alpha = alpha;
    a.S0 = S0;
    a.z0 = z0;
    a.S_out = S_out;
    a.z_out = z_out;
    a.y = static_cast<uint16_t *>(y);
    a.H = H;
    a.T = total_T;
    a.dv = dv;
    a.eps = eps;
    a.status = status;
    a.wait_limit_ns = la::kWaitLimitNs;
    a.nseg = 1;
    a.seg_chunks = 0;
    a.S_start = nullptr;
    a.cu_seqlens = cu_seqlens;
    if (!plan.bytes)
        return from_cuda(la::launch_prefill_tc(mq, mk, mv, a, B, alpha != nullptr, plan.dvs, st));
    // the walk over the short sequences, the plan (segment length and tables) on the
    // device, the state pass over the segments that end at a boundary, the scan of
    // each split sequence, then every other segment in parallel
    // The walk touches only the short sequences and the chain below only the others,
    // so the walk runs on a side stream beside the chain (ordered by events: after
    // what the caller enqueued before, and before what it enqueues after).
    la::SideLane *side = walk_max >= 0 ? la::side_lane() : nullptr;
    if (walk_max >= 0) {
        const cudaStream_t ws_ = side ? side->stream : st;
        cudaError_t ew = cudaSuccess;
        if (side && (ew = cudaEventRecord(side->ev[0], st)) == cudaSuccess) ew = cudaStreamWaitEvent(ws_, side->ev[0], 0);
        if (ew == cudaSuccess)
            ew = la::launch_decode_multi_packed(q, k, v, true, alpha, S0, z0, S_out, z_out, cu_seqlens, B, H, total_T,
                                                eps, y, ws_);
        if (ew == cudaSuccess && side) ew = cudaEventRecord(side->ev[1], ws_);
        if (ew != cudaSuccess) return from_cuda(ew);
    }
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    int *seg_len = reinterpret_cast<int *>(ws);
    int4 *seq_info = reinterpret_cast<int4 *>(ws + plan.off_info);
    int2 *items = reinterpret_cast<int2 *>(ws + plan.off_items);
    int2 *bds = reinterpret_cast<int2 *>(ws + plan.off_bds);
    int *split_seqs = reinterpret_cast<int *>(ws + plan.off_split);
    float *A = reinterpret_cast<float *>(ws + plan.off_A);
    float *dS = reinterpret_cast<float *>(ws + plan.off_dS);
    float *S_start = reinterpret_cast<float *>(ws + plan.off_S);
    cudaError_t e = la::launch_varlen_plan(cu_seqlens, B, total_T, plan.min_seg, plan.units, sm_count(),
                                           plan.max_bds, plan.part_rows, plan.part_target, walk_max, seg_len,
                                           seq_info, items, bds, split_seqs, st);
    la::StateTcArgs sa;
    sa.alpha = alpha;
    sa.dS = dS;
    sa.A = A;
    sa.H = H;
    sa.T = total_T;
    sa.dv = dv;
    sa.nsub = 0;
    sa.sub_per_seg = 1;   // the plan's parts per segment are in seg_len
    sa.sub_chunks = 0;
    sa.seg_chunks = 0;
    sa.cu_seqlens = cu_seqlens;
    sa.bds = bds;
    sa.seg_len = seg_len;
    sa.status = status;
    sa.wait_limit_ns = la::kWaitLimitNs;
    if (e == cudaSuccess && plan.max_bds > 0)
        e = la::launch_state_tc(mk, mv, sa, B, alpha != nullptr, plan.dvs, st, false, plan.part_rows);
    if (e == cudaSuccess && plan.max_bds > 0)
        e = la::launch_varlen_scan(S0, z0, A, dS, S_start, seq_info, split_seqs, seg_len, plan.max_bds, H, dv, st);
    if (e != cudaSuccess) return from_cuda(e);
    a.items = items;
    a.seq_info = seq_info;
    a.seg_len = seg_len;
    a.S_start = S_start;   // read only for split sequences (none when max_bds is 0)
    e = la::launch_prefill_tc(mq, mk, mv, a, B, alpha != nullptr, plan.dvs, st, B + plan.max_bds);
    if (e == cudaSuccess && side) e = cudaStreamWaitEvent(st, side->ev[1], 0);   // join the walk
    return from_cuda(e);
}

la_status la_prefill_chunked_noalloc(const void *q, const void *k, const void *v, la_dtype dtype,
                                     const float *alpha, const float *S0, const float *z0, int B, int H, int T,
                                     int r, int dv, int chunk, float eps, void *y, float *S_out, float *z_out,
                                     la_stream_t stream)
{
    const size_t need = dtype == LA_DTYPE_BF16 ? la_prefill_workspace_bytes(B, H, T, r, dv, chunk) : 0;
    if (need > kNoAllocScratchBytes) return LA_ERR_WORKSPACE;
    void *scratch = nullptr;
    if (need) {
        scratch = noalloc_scratch();
        if (!scratch) return LA_ERR_CUDA;
    }
    return la_prefill_chunked(q, k, v, dtype, alpha, S0, z0, B, H, T, r, dv, chunk, eps, y, S_out, z_out, scratch,
                              need, stream);
}

la_status la_decode_step(const void *q, const void *k, const void *v, la_dtype dtype, const float *alpha, float *S,
                         float *z, int B, int H, int r, int dv, float eps, void *y, la_stream_t stream)
{
    if (!q || !k || !v || !S || !z || !y) return LA_ERR_NULL;
    if (B < 1 || H < 1 || r < 1 || dv < 1) return LA_ERR_SHAPE;
    if (dtype != LA_DTYPE_BF16 && dtype != LA_DTYPE_FP32) return LA_ERR_DTYPE;
    if (r > 256 || dv > 256) return LA_ERR_UNSUPPORTED;
    if ((long long)B * H > 0x7fffffffLL) return LA_ERR_SHAPE;   // one CTA per (b, h)
    const uintptr_t el = dtype == LA_DTYPE_BF16 ? 2 : 4;
    if (!aligned(q, el) || !aligned(k, el) || !aligned(v, el) || !aligned(y, el)) return LA_ERR_ALIGN;
    if (!aligned(S, 4) || !aligned(z, 4) || (alpha && !aligned(alpha, 4))) return LA_ERR_ALIGN;
    const bool fast = r == 128 && dv == 128 && aligned(S, 16);
    return from_cuda(la::launch_decode(q, k, v, dtype == LA_DTYPE_BF16, alpha, S, z, B, H, r, dv, eps, y, fast,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

// Backward workspace: the per-token FP32 terms, then (when the tensor-core sweeps
// run over segments) the forward and the reversed state passes' parts and
// segment states, each in the prefill's layout.
size_t bwd_base_bytes(int B, int H, int T) { return round_up(sizeof(float) * la::backward_workspace_floats(B, H, T), 256); }

size_t la_backward_workspace_bytes(int B, int H, int T)
{
    if (B < 1 || H < 1 || T < 1) return 0;
    const SegPlan p = bwd_seg_plan(B, H, T);
    return bwd_base_bytes(B, H, T) + 2 * seg_workspace_bytes(p.nsub, p.nseg, B, H, 128);
}

// la_prefill_backward and la_prefill_backward_saved; d (the forward's d_t) may be nullptr.
static la_status prefill_backward_impl(const void *q, const void *k, const void *v, la_dtype dtype,
                                       const float *alpha, const float *S0, const float *z0, int B, int H, int T,
                                       int r, int dv, float eps, const void *y, const void *dy, const float *d,
                                       const float *states, const float *dS_T, const float *dz_T, void *dq, void *dk,
                                       void *dv_out,
                                       float *dalpha, float *dS0, float *dz0, void *workspace,
                                       size_t workspace_bytes, la_stream_t stream)
{
    if (!q || !k || !v || !y || !dy || !dq || !dk || !dv_out || !dS0 || !dz0) return LA_ERR_NULL;
    if (B < 1 || H < 1 || T < 1 || r < 1 || dv < 1) return LA_ERR_SHAPE;
    if (dtype != LA_DTYPE_BF16 && dtype != LA_DTYPE_FP32) return LA_ERR_DTYPE;
    if ((r != 32 && r != 64 && r != 128) || (dv != 32 && dv != 64 && dv != 128)) return LA_ERR_UNSUPPORTED;
    if ((long long)B * H * 4 > 0x7fffffffLL) return LA_ERR_UNSUPPORTED;
    // token arrays are staged by TMA bulk copies and written 16 bytes at a time
    for (const void *p : {q, k, v, y, dy, (const void *)dq, (const void *)dk, (const void *)dv_out})
        if (!aligned(p, 16)) return LA_ERR_ALIGN;
    for (const void *p : {(const void *)alpha, (const void *)S0, (const void *)z0, (const void *)dz_T,
                          (const void *)dalpha, (const void *)dS0, (const void *)dz0, (const void *)d})
        if (p && !aligned(p, 4)) return LA_ERR_ALIGN;
    if (dS_T && !aligned(dS_T, 8)) return LA_ERR_ALIGN;
    if (!workspace || workspace_bytes < la_backward_workspace_bytes(B, H, T)) return LA_ERR_WORKSPACE;
    if (!aligned(workspace, 16)) return LA_ERR_ALIGN;
    la::BackwardArgs a;
    a.q = q; a.k = k; a.v = v; a.y = y; a.dy = dy;
    a.alpha = alpha; a.S0 = S0; a.z0 = z0; a.dS_T = dS_T; a.dz_T = dz_T;
    a.dq = dq; a.dk = dk; a.dv_out = dv_out; a.dalpha = dalpha; a.dS0 = dS0; a.dz0 = dz0;
    a.ws = static_cast<float *>(workspace);
    a.d_in = d;
    if (states && !aligned(states, 16)) return LA_ERR_ALIGN;
    a.H = H; a.T = T; a.r = r; a.dv = dv; a.eps = eps;
    a.status = status_word();
    a.limit_ns = la::kWaitLimitNs;
    if (!a.status) return LA_ERR_CUDA;
    // BF16 at r == dv == 128: the sweeps run on the tensor cores, which read q, k,
    // v and dy through TMA descriptors
    CUtensorMap maps[4];
    a.maps = nullptr;
    if (dtype == LA_DTYPE_BF16 && r == 128 && dv == 128) {
        const long long planes = (long long)B * H;
        const CUtensorMapSwizzle sw128 = CU_TENSOR_MAP_SWIZZLE_128B;
        if (!make_map_bf16(&maps[0], q, planes, T, 128, 64, 64, sw128) ||
            !make_map_bf16(&maps[1], k, planes, T, 128, 64, 64, sw128) ||
            !make_map_bf16(&maps[2], v, planes, T, 128, 64, 64, sw128) ||
            !make_map_bf16(&maps[3], dy, planes, T, 128, 64, 64, sw128))
            return LA_ERR_CUDA;
        a.maps = maps;
        const SegPlan p = bwd_seg_plan(B, H, T);
        if (p.nseg > 1) {
            a.nseg = p.nseg;
            a.seg_chunks = p.seg_chunks;
            a.sub_per_seg = p.sub_per_seg;
            a.sub_chunks = p.sub_chunks;
            a.nsub = p.nsub;
            a.seg_ws = reinterpret_cast<float *>(static_cast<char *>(workspace) + bwd_base_bytes(B, H, T));
            a.states_in = states;
        }
    }
    return from_cuda(la::launch_backward(a, B, dtype == LA_DTYPE_BF16, reinterpret_cast<cudaStream_t>(stream)));
}

la_status la_prefill_backward(const void *q, const void *k, const void *v, la_dtype dtype, const float *alpha,
                              const float *S0, const float *z0, int B, int H, int T, int r, int dv, float eps,
                              const void *y, const void *dy, const float *dS_T, const float *dz_T, void *dq,
                              void *dk, void *dv_out, float *dalpha, float *dS0, float *dz0, void *workspace,
                              size_t workspace_bytes, la_stream_t stream)
{
    return prefill_backward_impl(q, k, v, dtype, alpha, S0, z0, B, H, T, r, dv, eps, y, dy, nullptr, nullptr, dS_T,
                                 dz_T, dq, dk, dv_out, dalpha, dS0, dz0, workspace, workspace_bytes, stream);
}

la_status la_prefill_backward_saved(const void *q, const void *k, const void *v, la_dtype dtype, const float *alpha,
                                    const float *S0, const float *z0, int B, int H, int T, int r, int dv,
                                    const void *y, const void *dy, const float *d, const float *states,
                                    const float *dS_T, const float *dz_T, void *dq, void *dk, void *dv_out,
                                    float *dalpha, float *dS0, float *dz0, void *workspace, size_t workspace_bytes,
                                    la_stream_t stream)
{
    if (!d) return LA_ERR_NULL;
    return prefill_backward_impl(q, k, v, dtype, alpha, S0, z0, B, H, T, r, dv, 0.f, y, dy, d, states, dS_T, dz_T, dq,
                                 dk, dv_out, dalpha, dS0, dz0, workspace, workspace_bytes, stream);
}

la_status la_delta_rule(const void *q, const void *k, const void *v, la_dtype dtype, const float *beta,
                        const float *S0, int B, int H, int T, int r, int dv, void *y, float *S_out,
                        la_stream_t stream)
{
    if (!S_out || (T > 0 && (!q || !k || !v || !y))) return LA_ERR_NULL;
    if (B < 1 || H < 1 || T < 0 || r < 1 || dv < 1) return LA_ERR_SHAPE;
    if (dtype != LA_DTYPE_BF16 && dtype != LA_DTYPE_FP32) return LA_ERR_DTYPE;
    if ((r != 32 && r != 64 && r != 128 && r != 256) || dv % 32 != 0) return LA_ERR_UNSUPPORTED;
    // one CTA per (b, h, 32-column slice)
    if ((long long)B * H * (dv / 32) > 0x7fffffffLL) return LA_ERR_UNSUPPORTED;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(y, 16)) return LA_ERR_ALIGN;
    if (!aligned(S_out, 8) || (S0 && !aligned(S0, 8)) || (beta && !aligned(beta, 4))) return LA_ERR_ALIGN;
    int *status = status_word();
    if (!status) return LA_ERR_CUDA;
    return from_cuda(la::launch_delta(q, k, v, dtype == LA_DTYPE_BF16, beta, S0, B, H, T, r, dv, y, S_out, status,
                                      la::kWaitLimitNs, reinterpret_cast<cudaStream_t>(stream)));
}

size_t la_delta_chunked_workspace_bytes(int B, int H, int T)
{
    return la::delta_tc_workspace_bytes(B, H, T);
}

la_status la_delta_rule_chunked(const void *q, const void *k, const void *v, la_dtype dtype, const float *beta,
                                const float *S0, int B, int H, int T, int r, int dv, void *y, float *S_out,
                                void *workspace, size_t workspace_bytes, la_stream_t stream)
{
    if (!S_out || (T > 0 && (!q || !k || !v || !y))) return LA_ERR_NULL;
    if (B < 1 || H < 1 || T < 0 || r < 1 || dv < 1) return LA_ERR_SHAPE;
    if (dtype != LA_DTYPE_BF16) return LA_ERR_DTYPE;
    if (r != 128 || dv % 64 != 0) return LA_ERR_UNSUPPORTED;
    // one CTA per (b, h, 64-column slice)
    if ((long long)B * H * (dv / 64) > 0x7fffffffLL) return LA_ERR_UNSUPPORTED;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(y, 16)) return LA_ERR_ALIGN;
    if (!aligned(S_out, 16) || (S0 && !aligned(S0, 16)) || (beta && !aligned(beta, 4))) return LA_ERR_ALIGN;
    if (T > 0) {
        if (!workspace || workspace_bytes < la::delta_tc_workspace_bytes(B, H, T)) return LA_ERR_WORKSPACE;
        if (!aligned(workspace, 16)) return LA_ERR_ALIGN;
    }
    int *status = status_word();
    if (!status) return LA_ERR_CUDA;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // no tokens: S_out = S0, as the token kernel does it
    if (T == 0)
        return from_cuda(la::launch_delta(q, k, v, true, beta, S0, B, H, T, r, dv, y, S_out, status,
                                          la::kWaitLimitNs, st));
    CUtensorMap mq, mk, mv;
    const long long planes = (long long)B * H;
    const CUtensorMapSwizzle sw128 = CU_TENSOR_MAP_SWIZZLE_128B;
    if (!make_map_bf16(&mq, q, planes, T, r, 64, 64, sw128) || !make_map_bf16(&mk, k, planes, T, r, 64, 64, sw128) ||
        !make_map_bf16(&mv, v, planes, T, dv, 64, 64, sw128))
        return LA_ERR_CUDA;
    la::DeltaTcArgs a;
    a.beta = beta;
    a.S0 = S0;
    a.S_out = S_out;
    a.y = static_cast<uint16_t *>(y);
    a.ws = workspace;
    a.H = H;
    a.T = T;
    a.dv = dv;
    a.status = status;
    a.wait_limit_ns = la::kWaitLimitNs;
    return from_cuda(la::launch_delta_tc(mq, mk, mv, a, B, st));
}

la_status la_last_device_status(la_stream_t stream)
{
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return LA_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_status, sizeof(int)) != cudaSuccess) return LA_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_status, &zero, sizeof(int)) != cudaSuccess) return LA_ERR_CUDA;
    }
    return static_cast<la_status>(v);
}

la_status la_debug_wait_probe(unsigned long long limit_ns, la_stream_t stream)
{
    if (limit_ns > 1000000000ull) return LA_ERR_SHAPE;
    int *status = status_word();
    if (!status) return LA_ERR_CUDA;
    return from_cuda(la::launch_wait_probe(status, limit_ns, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
