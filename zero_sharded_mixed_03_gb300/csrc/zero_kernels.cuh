// zero_kernels.cuh -- the device code of the sharded mixed-precision AdamW step for GB300
// (sm_103a): the fused reduce + AdamW + cast kernel (128-bit register loads, or a variant
// whose tiles are staged into shared memory by cp.async.bulk copies), the gradient-norm
// pre-pass, the offload reduction, the device-side commit/skip, the skip re-cast and the
// stage-3 gathers, with the launch-parameter blocks and constants the host side shares.
// Included by zero_step.cu alone (whose host code launches these kernels).
//
// Page: "Zero Redundancy Optimizer (ZeRO) and Fully Sharded Data Parallelism
// (FSDP): Mathematical Foundations ..." (llms.blog):
//   "Execution Flow for ZeRO-1" steps 2-4 (reduce-scatter of the averaged
//   gradient, shard update, all-gather of the 16-bit shards), "ZeRO-Stage 2"
//   (gradients reduced as produced, here per bucket), "ZeRO-3 / FSDP Layer
//   Execution Lifecycle" (per-unit all-gather and reduce-scatter).
//
// The path is elementwise plus a reduction over N_d ranks: about 15 flops per
// parameter against 2*N_d + 26 bytes, far below any tensor-core ridge, so it
// is written for HBM bandwidth: 128-bit loads/stores, one pass, fp32 state
// double-buffered so the global skip decision needs no second pass.  The
// decision itself stays on the GPU: the current half of every ping-pong pair,
// the applied-step count t and the loss scale live in the caller's workspace,
// so consecutive steps are enqueued back to back with no host round trip.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "zero_internal.h"

namespace zero {
namespace {

constexpr int kThreads = 128;     // 128-thread blocks: 72 registers, 7 blocks resident per SM
constexpr int kMaxSegs = 32;      // work items per launch (more are split across launches)
constexpr int kWideSegs = 256;    // capacity of the wide parameter block (calls with many items)
constexpr int kScalarSlots = 16;  // per segment: up to 7 head + 7 tail elements
// Contribution slices loaded (128-bit each) per batch before they are summed; from
// kWideRankBatchFrom ranks on (kWideNormBatchFrom for the reductions without an update),
// kWideRankBatch.
constexpr int kRankBatch = 4;
constexpr int kWideRankBatch = 16;
constexpr int kWideRankBatchFrom = 41;
constexpr int kWideNormBatchFrom = 32;
// The gradient-norm pre-pass reads nothing else, so it keeps more slices in flight.
constexpr int kNormRankBatch = 8;

// ------------------------------------------------------------------ device-resident step state

// First 96 bytes of the workspace.  Written by the commit (the last re-cast block or
// commit_kernel), by the host before the first step, and by the kernels' atomics (flag,
// error, norm tickets); read by the step and re-cast kernels of the following step.
struct DevState {
    uint32_t flag;          // OR of the non-finite flags of the open step
    uint32_t cur;           // current half of every ping-pong pair
    uint32_t last_skipped;  // 1 if the last finished step was skipped
    uint32_t blocks_done;   // blocks of the running norm launch that have stored their partial
    int64_t t;              // applied steps
    int64_t skipped;        // skipped steps, total
    int64_t good;           // applied steps since the last change of the loss scale
    int64_t finished;       // finished steps (applied + skipped)
    double scale;           // loss scale of the next step
    double norm2;           // open step: sum of fp32(g*g) so far
    double last_norm2;      // last finished step's sum
    uint32_t norm_valid;    // open step computed a norm
    uint32_t last_norm_valid;
    uint32_t error;         // bit 0: a barrier wait of the staged step ran out; bit 1: a drain
                            // ran out; bit 2: a barrier wait of the staged gather ran out
                            // (sticky until read; every step finished meanwhile is discarded)
    uint32_t pad32;
    int64_t pad;
};
static_assert(sizeof(DevState) == 96, "DevState layout");

static_assert(sizeof(DevState) <= kStateBytes, "DevState fits its workspace slot");

// ------------------------------------------------------------------ launch parameters

struct KSeg {
    float* p[2];       // master, both halves, at the segment start
    float* m[2];
    float* v[2];
    uint16_t* out16;
    int64_t c_off;     // element offset into every contribution buffer
    int64_t n;         // elements
    int64_t nvec;      // aligned vectors in the body
    int64_t vbeg;      // index of the first body vector in the launch
    int32_t head;      // scalar elements before the body
    int32_t tail;      // scalar elements after the body
};

struct CommitParams {
    DevState* st;
    double growth, backoff, min_scale;
    int64_t interval;
    int32_t dynamic;           // 0: fixed loss scale (no back-off, no growth)
};

template <int MS>
struct StepParamsT {
    const uint16_t* c[ZERO_MAX_RANKS];
    KSeg seg[MS];
    float k[9];        // b1, 1-b1, b2, 1-b2, eps, lr*wd, lr/bc1, sqrt(bc2), inv
    double lr;         // device mode: lr/bc1 is formed on the GPU from the table
    double beta1, beta2;
    const double* bias;        // device mode: bias-correction table (pairs)
    int64_t bias_len;          // entries 1..bias_len are valid
    int32_t bias_saturates;    // entries beyond bias_len equal entry bias_len
    int32_t n_d;
    int32_t n_seg;
    int32_t pad;
    int64_t total_vec;
    uint32_t* flag;
    DevState* st;              // nullptr: host mode (constants in k, current half 0)
    double max_norm;           // clip mode: the bound on the global gradient norm
    double* partials;          // norm modes: one slot per block
    CommitParams commit;       // re-cast launch that also closes the step
    int32_t do_commit;
    // bulk-staged kernel: tile geometry and the bound on each barrier wait
    int32_t tile;              // body elements per tile (a multiple of 8)
    int32_t stages;            // ring depth
    int64_t n_tiles;           // tiles over all segments of the launch
    uint64_t wait_ns;
};
// The usual parameter block (4 KB), and a wide one (26 KB, under the 32 KB kernel-parameter
// limit) for calls with many work items, e.g. per-parameter plans (one item per tensor chunk).
using StepParams = StepParamsT<kMaxSegs>;
using StepParamsWide = StepParamsT<kWideSegs>;

// One copy of a stage-3 all-gather streamed inside a step launch ("Overlapping Computation
// and Communication Streams": the next unit's all-gather runs while this unit is reduced and
// updated).  Compact, so that the wide block stays under the 32 KB kernel-parameter limit:
// the destination is g_dst + dst_off; source and destination share one 16-byte phase, and
// the unaligned head and tail are derived from the destination's address.
struct GCopy {
    const uint16_t* src;
    uint32_t dst_off;   // element offset of the copy in the gather destination
    uint32_t n;         // elements
    uint32_t cbeg;      // first chunk of this copy among the launch's gather chunks
    uint32_t pad;
};

template <int MS, int MG>
struct StepGatherParamsT : StepParamsT<MS> {
    GCopy gc[MG];
    uint16_t* g_dst;    // the gathered unit's full buffer
    int32_t g_n;        // copies
    int32_t g_chunk;    // elements per chunk (a multiple of 8, at most one ring buffer)
    int64_t g_chunks;   // chunks over the vector bodies of all copies
};
using StepGatherParams = StepGatherParamsT<kMaxSegs, kMaxSegs>;
using StepGatherParamsWide = StepGatherParamsT<kWideSegs, kWideSegs>;
static_assert(sizeof(StepGatherParamsWide) <= 32764, "kernel parameter limit");

template <typename PT>
struct HasGather : std::false_type {};
template <int MS, int MG>
struct HasGather<StepGatherParamsT<MS, MG>> : std::true_type {};

// Elements before the first 16-byte boundary of a 16-bit stream starting at p (at most n).
__device__ __forceinline__ int64_t head_elems(const void* p, int64_t n)
{
    const int64_t h = (int64_t)(((16u - ((uint32_t)(uintptr_t)p & 15u)) & 15u) >> 1);
    return h < n ? h : n;
}

struct CopySeg {
    const uint16_t* src;
    uint16_t* dst;
    int64_t n, nvec, vbeg;
    int64_t cbeg;           // bulk-staged gather: first chunk of this copy
    int32_t head, tail;
};

template <int MS>
struct CopyParamsT {
    CopySeg seg[MS];
    int n_seg;
    int64_t total_vec;
    // bulk-staged gather only
    uint32_t* err;          // the plan's error word
    uint64_t wait_ns;       // bound on each barrier wait
    int32_t chunk;          // elements per bulk copy (a multiple of 8)
    int32_t stages;         // ring entries
    int64_t n_chunks;       // chunks of all copies of the launch
};
// 32 copies (1.8 KB), or 256 (14 KB) for gathers of many chunks (per-parameter plans)
using CopyParams = CopyParamsT<kMaxSegs>;
using CopyParamsWide = CopyParamsT<kWideSegs>;

// ------------------------------------------------------------------ element helpers

// 16-bit -> fp32 widening (exact).  bf16 is the upper half of an IEEE binary32.
template <int DT>
__device__ __forceinline__ float widen1(uint16_t h)
{
    if constexpr (DT == ZERO_BF16) return __uint_as_float((uint32_t)h << 16);
    else return __half2float(__ushort_as_half(h));
}

template <int DT>
__device__ __forceinline__ void widen2(uint32_t w, float& lo, float& hi)
{
    if constexpr (DT == ZERO_BF16) {
        lo = __uint_as_float(w << 16);
        hi = __uint_as_float(w & 0xFFFF0000u);
    } else {
        __half2 h = *reinterpret_cast<const __half2*>(&w);
        float2 f = __half22float2(h);
        lo = f.x;
        hi = f.y;
    }
}

// fp32 -> 16-bit, round to nearest even.
template <int DT>
__device__ __forceinline__ uint16_t narrow1(float f)
{
    if constexpr (DT == ZERO_BF16) return __bfloat16_as_ushort(__float2bfloat16_rn(f));
    else return __half_as_ushort(__float2half_rn(f));
}

template <int DT>
__device__ __forceinline__ uint32_t narrow2(float lo, float hi)
{
    if constexpr (DT == ZERO_BF16) {
        __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&b);
    } else {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
}

__device__ __forceinline__ bool nonfinite(float g)
{
    return (__float_as_uint(g) & 0x7F800000u) == 0x7F800000u;
}

// The constants that depend on t, the loss scale and the gradient norm, formed per block.
struct StepK {
    float step;   // lr / (1 - beta1^t)
    float bc2s;   // sqrt(1 - beta2^t)
    float inv;    // 1 / (N_d * loss_scale)
    float coef;   // clip mode: min(1, max_norm / (norm + 1e-6)); else 1
};

// What the fused kernel does with the gradient norm.
enum { kPlain = 0, kNormAcc = 1, kClip = 2 };

// Per-thread sum of the fp32 squares as an unevaluated pair hi + lo of floats, extended by an
// error-free TwoSum (Knuth) per term: ~48 significant bits from fp32 operations only (GB300's
// fp64 rate is far below its fp32 rate).  Converted to double once, at the end of the thread.
struct NormAcc {
    float hi = 0.0f, lo = 0.0f;
    __device__ __forceinline__ void add(float p)
    {
        const float s = __fadd_rn(hi, p);
        const float bp = __fsub_rn(s, hi);
        const float ap = __fsub_rn(s, bp);
        const float e = __fadd_rn(__fsub_rn(hi, ap), __fsub_rn(p, bp));
        hi = s;
        lo = __fadd_rn(lo, e);
    }
    __device__ __forceinline__ double value() const { return (double)hi + (double)lo; }
};

// AdamW on one element with separately rounded IEEE operations (no contraction):
//   m = b1 m + (1-b1) g ; v = b2 v + (1-b2) g^2 ; d = sqrt(v)/sqrt(bc2) + eps
//   p = p - (lr wd) p   ; p = p - (lr/bc1) (m / d)
// k[0..5] (b1, 1-b1, b2, 1-b2, eps, lr*wd) stay in the kernel parameters.
__device__ __forceinline__ void adamw1(float g, float& p, float& m, float& v, const float* k,
                                       const StepK& sk)
{
    m = __fadd_rn(__fmul_rn(k[0], m), __fmul_rn(k[1], g));
    v = __fadd_rn(__fmul_rn(k[2], v), __fmul_rn(k[3], __fmul_rn(g, g)));
    const float d = __fadd_rn(__fdiv_rn(__fsqrt_rn(v), sk.bc2s), k[4]);
    p = __fsub_rn(p, __fmul_rn(k[5], p));
    p = __fsub_rn(p, __fmul_rn(sk.step, __fdiv_rn(m, d)));
}

__device__ __forceinline__ uint4 ld_stream(const void* p)
{
    return __ldcs(reinterpret_cast<const uint4*>(p));
}

__device__ __forceinline__ uint2 ld_stream8(const void* p)
{
    return __ldcs(reinterpret_cast<const uint2*>(p));
}

// The step's fp32 constants and the current half, formed once per block by thread 0.
// Device mode: t and the loss scale come from the workspace; the fp32 roundings of
// lr/bc1, sqrt(bc2) and 1/(N_d*scale) are the same IEEE double operations the host uses.
template <typename PT>
__device__ __forceinline__ void block_constants(const PT& P, float* sk, int* scur)
{
    if (threadIdx.x == 0) {
        sk[0] = P.k[6];
        sk[1] = P.k[7];
        sk[2] = P.k[8];
        sk[3] = 1.0f;
        int cur = 0;
        if (P.st) {
            const volatile DevState* st = P.st;
            const int64_t t = st->t + 1;   // the step being applied
            double bc1, bc2s;
            if (t <= P.bias_len || P.bias_saturates) {
                const int64_t i = t <= P.bias_len ? t : P.bias_len;
                bc1 = P.bias[2 * i];
                bc2s = P.bias[2 * i + 1];
            } else {
                bc1 = __dsub_rn(1.0, pow(P.beta1, (double)t));
                bc2s = __dsqrt_rn(__dsub_rn(1.0, pow(P.beta2, (double)t)));
            }
            sk[0] = __double2float_rn(__ddiv_rn(P.lr, bc1));
            sk[1] = __double2float_rn(bc2s);
            sk[2] = __double2float_rn(__ddiv_rn(1.0, __dmul_rn((double)P.n_d, st->scale)));
            if (P.max_norm > 0.0) {
                double c = __ddiv_rn(P.max_norm, __dadd_rn(__dsqrt_rn(st->norm2), 1e-6));
                if (c > 1.0) c = 1.0;
                sk[3] = __double2float_rn(c);
            }
            cur = (int)st->cur;
        }
        *scur = cur;
    }
    __syncthreads();
}

// ------------------------------------------------------------------ fused step kernel

template <int DT, int MODE, typename PT>
__device__ __forceinline__ bool step_scalar(const PT& P, const KSeg& S, int64_t e,
                                            const StepK& sk, int cur, NormAcc& norm2)
{
    float sum = 0.0f;
    for (int r = 0; r < P.n_d; ++r) sum = __fadd_rn(sum, widen1<DT>(P.c[r][S.c_off + e]));
    const float g = __fmul_rn(sum, sk.inv);
    if constexpr (MODE == kNormAcc) norm2.add(__fmul_rn(g, g));
    const float gu = MODE == kClip ? __fmul_rn(g, sk.coef) : g;
    float p = S.p[cur][e], m = S.m[cur][e], v = S.v[cur][e];
    adamw1(gu, p, m, v, P.k, sk);
    S.p[cur ^ 1][e] = p;
    S.m[cur ^ 1][e] = m;
    S.v[cur ^ 1][e] = v;
    S.out16[e] = narrow1<DT>(p);
    return nonfinite(g);
}

// Eight consecutive elements starting at e: 128-bit loads of the N_d contribution slices
// (batches of NB ranks in flight), 2 x 128-bit per fp32 state array, 128-bit 16-bit store.
template <int DT, int NB, int MODE, typename PT>
__device__ __forceinline__ bool step_vec8(const PT& P, const KSeg& S, int64_t e,
                                          const StepK& sk, int cur, NormAcc& norm2)
{
    const float* pin = S.p[cur] + e;
    const float* min_ = S.m[cur] + e;
    const float* vin = S.v[cur] + e;
    const float4 p0 = __ldcs(reinterpret_cast<const float4*>(pin));
    const float4 p1 = __ldcs(reinterpret_cast<const float4*>(pin) + 1);
    const float4 m0 = __ldcs(reinterpret_cast<const float4*>(min_));
    const float4 m1 = __ldcs(reinterpret_cast<const float4*>(min_) + 1);
    const float4 v0 = __ldcs(reinterpret_cast<const float4*>(vin));
    const float4 v1 = __ldcs(reinterpret_cast<const float4*>(vin) + 1);

    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
    for (int r0 = 0; r0 < P.n_d; r0 += NB) {
        uint4 c[NB];
#pragma unroll
        for (int q = 0; q < NB; ++q)
            if (r0 + q < P.n_d) c[q] = ld_stream(P.c[r0 + q] + S.c_off + e);
#pragma unroll
        for (int q = 0; q < NB; ++q) {
            if (r0 + q < P.n_d) {
                const uint32_t w[4] = {c[q].x, c[q].y, c[q].z, c[q].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float lo, hi;
                    widen2<DT>(w[j], lo, hi);
                    acc[2 * j] = __fadd_rn(acc[2 * j], lo);
                    acc[2 * j + 1] = __fadd_rn(acc[2 * j + 1], hi);
                }
            }
        }
    }

    float p[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
    float m[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
    float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    bool bad = false;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float g = __fmul_rn(acc[j], sk.inv);
        bad |= nonfinite(g);
        if constexpr (MODE == kNormAcc) norm2.add(__fmul_rn(g, g));
        const float gu = MODE == kClip ? __fmul_rn(g, sk.coef) : g;
        adamw1(gu, p[j], m[j], v[j], P.k, sk);
    }
    float4* pout = reinterpret_cast<float4*>(S.p[cur ^ 1] + e);
    float4* mout = reinterpret_cast<float4*>(S.m[cur ^ 1] + e);
    float4* vout = reinterpret_cast<float4*>(S.v[cur ^ 1] + e);
    __stcs(pout, make_float4(p[0], p[1], p[2], p[3]));
    __stcs(pout + 1, make_float4(p[4], p[5], p[6], p[7]));
    __stcs(mout, make_float4(m[0], m[1], m[2], m[3]));
    __stcs(mout + 1, make_float4(m[4], m[5], m[6], m[7]));
    __stcs(vout, make_float4(v[0], v[1], v[2], v[3]));
    __stcs(vout + 1, make_float4(v[4], v[5], v[6], v[7]));
    uint4 o;
    o.x = narrow2<DT>(p[0], p[1]);
    o.y = narrow2<DT>(p[2], p[3]);
    o.z = narrow2<DT>(p[4], p[5]);
    o.w = narrow2<DT>(p[6], p[7]);
    __stcs(reinterpret_cast<uint4*>(S.out16 + e), o);
    return bad;
}

// Sum of one double over a block of NT threads in a fixed pattern (shuffle tree per warp,
// warps in order); the result is valid in thread 0.
template <int NT>
__device__ __forceinline__ double block_sum_fixed(double x, double* warp_sum)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_down_sync(0xFFFFFFFFu, x, o);
    if ((threadIdx.x & 31) == 0) warp_sum[threadIdx.x >> 5] = x;
    __syncthreads();
    double b = 0.0;
    if (threadIdx.x == 0)
        for (int w = 0; w < NT / 32; ++w) b += warp_sum[w];
    __syncthreads();
    return b;
}

// Block sum of the per-thread norm partials, stored in this block's slot; the last block of
// the launch to store (an atomic ticket, nothing waits) adds all slots to the step's norm in a
// fixed order (thread t takes slots t, t + 128, ...; then the fixed block pattern), so the sum
// does not depend on which blocks finish first.
template <int NT, typename PT>
__device__ __forceinline__ void block_norm_commit(const PT& P, double part)
{
    __shared__ double warp_sum[NT / 32];
    __shared__ bool last;
    const double b = block_sum_fixed<NT>(part, warp_sum);
    if (threadIdx.x == 0) {
        P.partials[blockIdx.x] = b;
        __threadfence();
        const unsigned ticket = atomicAdd(&P.st->blocks_done, 1u);
        last = ticket == gridDim.x - 1;
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    const volatile double* slots = P.partials;
    double x = 0.0;
    for (unsigned i = threadIdx.x; i < gridDim.x; i += NT) x += slots[i];
    const double sum = block_sum_fixed<NT>(x, warp_sum);
    if (threadIdx.x == 0) {
        volatile DevState* st = P.st;
        st->norm2 = st->norm2 + sum;
        st->norm_valid = 1;
        st->blocks_done = 0;
        __threadfence();
    }
}

// Persistent grid-stride kernel over the concatenated body vectors of all segments, plus
// kScalarSlots scalar slots per segment for the unaligned head and tail.  VEC = 8: 128-bit
// body; VEC = 1: every element is a body vector of one (streams of different phases).
// Reads the current half of each pair and writes the other.
template <int DT, int NB, int VEC, int MODE, typename PT>
__global__ void __launch_bounds__(kThreads) fused_step_kernel(const __grid_constant__ PT P)
{
    __shared__ float sk4[4];
    __shared__ int scur;
    block_constants(P, sk4, &scur);
    const StepK sk = {sk4[0], sk4[1], sk4[2], sk4[3]};
    const int cur = scur;
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    bool bad = false;
    NormAcc norm2;

    if constexpr (VEC == 8) {
        for (int64_t q = tid; q < (int64_t)P.n_seg * kScalarSlots; q += stride) {
            const KSeg& S = P.seg[q / kScalarSlots];
            const int k = (int)(q % kScalarSlots);
            int64_t e = -1;
            if (k < S.head) e = k;
            else if (k - S.head < S.tail) e = S.head + 8 * S.nvec + (k - S.head);
            if (e >= 0) bad |= step_scalar<DT, MODE>(P, S, e, sk, cur, norm2);
        }
    }

    int s = 0;
    for (int64_t vi = tid; vi < P.total_vec; vi += stride) {
        while (vi >= P.seg[s].vbeg + P.seg[s].nvec) ++s;
        const KSeg& S = P.seg[s];
        if constexpr (VEC == 8)
            bad |= step_vec8<DT, NB, MODE>(P, S, S.head + 8 * (vi - S.vbeg), sk, cur, norm2);
        else
            bad |= step_scalar<DT, MODE>(P, S, vi - S.vbeg, sk, cur, norm2);
    }

    // Global non-finite flag: one OR across the block, one atomic per block that saw one.
    if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(P.flag, 1u);
    if constexpr (MODE == kNormAcc) block_norm_commit<kThreads>(P, norm2.value());
}

// ------------------------------------------------------------------ bulk-staged step kernel

// The same step with its HBM reads staged through shared memory by the TMA engine.  Warp
// kBulkConsumers (one lane) is the producer: per tile it issues 1-D cp.async.bulk copies of
// the N_d contribution slices and of the master/m/v slices into the next buffer of a ring,
// all completing on that buffer's "full" mbarrier.  The consumer warps wait on it, reduce and
// update from shared memory (quads of 4 elements: 64-bit and 128-bit shared loads without
// bank conflicts), store the new state and the 16-bit cast straight to HBM, and release the
// buffer on its "empty" mbarrier.  Every wait is bounded (P.wait_ns of %globaltimer and an
// iteration cap); one that runs out sets DevState::error and ends that warp's loop, and the
// producer waits (bounded again) for every copy it issued before the block returns.
constexpr int kBulkConsumers = 4;                        // consumer warps
constexpr int kBulkThreads = 32 * (kBulkConsumers + 1);  // + the producer warp
constexpr int kBulkBarrierBytes = 256;                   // full[16] + empty[16] mbarriers
constexpr int kBulkMaxStages = 16;
constexpr int kBulkMaxTile = 8192;
constexpr uint64_t kDrainNs = 2000000000ull;             // bound on the final drain
// Tiles of at most this many bulk copies (N_d + 3) are issued by lane 0 alone, in order; larger
// ones by all 32 lanes of the producer warp.  Measured on GB300 (ragged ZeRO-2 step, fraction
// of the copy bandwidth, one lane / 32 lanes): N_d = 7: 1.012 / 1.004, 8: 0.974 / 0.968,
// 16: 1.036 / 1.030, 24: 1.024 / 1.017; 32: 0.939 / 0.965, 40: 0.944 / 0.983, 47: 0.942 /
// 1.003, 48 (512-element tiles): 0.956 / 1.006.  From N_d = 32 on, one lane's sequential issue
// of the tile's copies no longer keeps up.
constexpr int kOneIssuerMaxCopies = 30;
constexpr uint32_t kWaitIterCap = 1u << 26;              // polls per wait, whatever the clock

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking probe of the same condition.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait until the phase of parity `parity` of barrier `bar` has completed.  False when
// limit_ns of %globaltimer (or kWaitIterCap polls) pass first; limit 0 gives up as soon as
// the first, non-blocking probe fails.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_test(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 0; i < kWaitIterCap; ++i) {
        if (global_ns() - t0 >= limit_ns) return false;
        if (mbar_try(bar, parity)) return true;
    }
    return false;
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ uint64_t evict_first_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 1-D bulk copy global -> shared of `bytes` (both addresses 16-byte aligned, bytes a multiple
// of 16), completing on barrier `bar`; every byte is read once, so L2 evicts it first.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                          uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// 1-D bulk copy shared -> global of `bytes` (16-byte aligned addresses, a multiple of 16
// bytes), tracked as part of this thread's current bulk group.
__device__ __forceinline__ void bulk_store(void* dst, uint32_t src, uint32_t bytes, uint64_t policy)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;"
                 ::"l"(dst), "r"(src), "r"(bytes), "l"(policy)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until at most N bulk groups of this thread still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until every bulk group of this thread has completed (its writes performed).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Launch tile `tile` (tiles increase along a thread's loop): segment s, first body element
// e0 and length (a multiple of 8).  s and base (first tile of segment s) carry the walk.
struct TileRef {
    int64_t e0;
    int32_t len;
};

template <typename PT>
__device__ __forceinline__ TileRef locate_tile(const PT& P, int64_t tile, int& s, int64_t& base)
{
    for (;;) {
        const int64_t nt = (8 * P.seg[s].nvec + P.tile - 1) / P.tile;
        if (tile < base + nt) break;
        base += nt;
        ++s;
    }
    const KSeg& S = P.seg[s];
    const int64_t off = (tile - base) * P.tile;
    TileRef r;
    r.e0 = S.head + off;
    r.len = (int32_t)min((int64_t)P.tile, 8 * S.nvec - off);
    return r;
}

// Walk over the gather chunks of a step launch in increasing order (chunk ids c, c + grid,
// ...): the copy holding the current chunk and its chunk range (from the host's first-chunk
// table) are carried along.  Returns the chunk's first body element and length; *src / *dst
// are the copy's streams.
template <typename PT>
struct GChunkWalk {
    int s = -1;
    int64_t first = 0, end = 0;

    __device__ __forceinline__ TileRef at(const PT& P, int64_t c, const uint16_t** src, uint16_t** dst)
    {
        while (c >= end) {
            ++s;
            first = end;
            end = s + 1 < P.g_n ? (int64_t)P.gc[s + 1].cbeg : P.g_chunks;
        }
        const GCopy& C = P.gc[s];
        uint16_t* d = P.g_dst + C.dst_off;
        const int64_t head = head_elems(d, C.n);
        const int64_t body = ((int64_t)C.n - head) / 8 * 8;
        const int64_t off = (c - first) * P.g_chunk;
        TileRef r;
        r.e0 = head + off;
        r.len = (int32_t)min((int64_t)P.g_chunk, body - off);
        *src = C.src;
        *dst = d;
        return r;
    }
};

// Four consecutive elements e .. e+3 (quad q of the tile in buffer `buf`).
template <int DT, int MODE, typename PT>
__device__ __forceinline__ bool step_quad_staged(const PT& P, const KSeg& S, const unsigned char* buf,
                                                 int64_t e, int q, const StepK& sk, int cur,
                                                 NormAcc& norm2)
{
    const int tile = P.tile;
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    const unsigned char* c = buf + 8 * q;
#pragma unroll 4
    for (int r = 0; r < P.n_d; ++r) {
        const uint2 w = *reinterpret_cast<const uint2*>(c + (size_t)r * tile * 2);
        float a, b, d, f;
        widen2<DT>(w.x, a, b);
        widen2<DT>(w.y, d, f);
        acc[0] = __fadd_rn(acc[0], a);
        acc[1] = __fadd_rn(acc[1], b);
        acc[2] = __fadd_rn(acc[2], d);
        acc[3] = __fadd_rn(acc[3], f);
    }
    const unsigned char* sb = buf + (size_t)P.n_d * tile * 2 + 16 * q;
    const float4 p4 = *reinterpret_cast<const float4*>(sb);
    const float4 m4 = *reinterpret_cast<const float4*>(sb + (size_t)tile * 4);
    const float4 v4 = *reinterpret_cast<const float4*>(sb + (size_t)tile * 8);
    float p[4] = {p4.x, p4.y, p4.z, p4.w};
    float m[4] = {m4.x, m4.y, m4.z, m4.w};
    float v[4] = {v4.x, v4.y, v4.z, v4.w};
    bool bad = false;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float g = __fmul_rn(acc[j], sk.inv);
        bad |= nonfinite(g);
        if constexpr (MODE == kNormAcc) norm2.add(__fmul_rn(g, g));
        const float gu = MODE == kClip ? __fmul_rn(g, sk.coef) : g;
        adamw1(gu, p[j], m[j], v[j], P.k, sk);
    }
    __stcs(reinterpret_cast<float4*>(S.p[cur ^ 1] + e), make_float4(p[0], p[1], p[2], p[3]));
    __stcs(reinterpret_cast<float4*>(S.m[cur ^ 1] + e), make_float4(m[0], m[1], m[2], m[3]));
    __stcs(reinterpret_cast<float4*>(S.v[cur ^ 1] + e), make_float4(v[0], v[1], v[2], v[3]));
    __stcs(reinterpret_cast<uint2*>(S.out16 + e), make_uint2(narrow2<DT>(p[0], p[1]), narrow2<DT>(p[2], p[3])));
    return bad;
}

// Persistent: block b takes tiles b, b + grid, ...; its k-th tile uses buffer k % stages.
// Dynamic shared memory (from a 128-byte boundary): kBulkBarrierBytes of mbarriers, then
// `stages` buffers of tile * (2 N_d + 12) bytes: N_d contribution slices (tile * 2 bytes
// each), master, m, v.
// With a gather in the parameters (StepGatherParamsT: the next unit's all-gather), the
// producer lane continues after its last tile: block b takes gather chunks grid-1-b,
// 2 grid-1-b, ... (the blocks with one tile fewer start first), loads each through the next
// ring buffer once the consumers have released it (or, for a buffer that held a gather chunk,
// once that chunk's bulk store has read it), one load ahead of the stores, and writes it
// back with a bulk store; the consumer warps copy the copies' unaligned heads and tails.  A
// wait that runs out sets bit 2 of the error word (as the standalone gather does).
template <int DT, int MODE, typename PT>
__global__ void __launch_bounds__(kBulkThreads) bulk_step_kernel(const __grid_constant__ PT P)
{
    static_assert(MODE != kNormAcc, "norm-report steps run fused_step_kernel");
    extern __shared__ __align__(128) unsigned char bulk_raw[];
    __shared__ float sk4[4];
    __shared__ int scur;
    // 128-byte aligned start whatever the static shared memory before it (launches add 128 B)
    const uint32_t raw = (uint32_t)__cvta_generic_to_shared(bulk_raw);
    const uint32_t full0 = (raw + 127u) & ~127u;
    const unsigned char* bulk_smem = bulk_raw + (full0 - raw);
    const uint32_t empty0 = full0 + 8u * kBulkMaxStages;
    const uint32_t stage_bytes = (uint32_t)P.tile * (2u * (uint32_t)P.n_d + 12u);
    if (threadIdx.x == 0) {
        for (int i = 0; i < P.stages; ++i) {
            mbar_init(full0 + 8u * i, 1);
            mbar_init(empty0 + 8u * i, kBulkConsumers);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    block_constants(P, sk4, &scur);   // ends with __syncthreads: the barriers are ready
    const StepK sk = {sk4[0], sk4[1], sk4[2], sk4[3]};
    const int cur = scur;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    bool bad = false;
    uint32_t err = 0;
    NormAcc norm2;

    if (warp < kBulkConsumers) {
        const int ct = threadIdx.x;
        constexpr int kCT = 32 * kBulkConsumers;
        int s = 0;
        int64_t base = 0;
        uint32_t k = 0;
        for (int64_t tile = blockIdx.x; tile < P.n_tiles; tile += gridDim.x, ++k) {
            const TileRef T = locate_tile(P, tile, s, base);
            const uint32_t st = k % (uint32_t)P.stages;
            const bool ok = mbar_wait(full0 + 8u * st, (k / (uint32_t)P.stages) & 1u, P.wait_ns);
            if (__any_sync(0xFFFFFFFFu, !ok)) {
                err |= 1u;
                break;
            }
            const KSeg& S = P.seg[s];
            const unsigned char* buf = bulk_smem + kBulkBarrierBytes + (size_t)st * stage_bytes;
            for (int q = ct; q < T.len / 4; q += kCT)
                bad |= step_quad_staged<DT, MODE>(P, S, buf, T.e0 + 4 * q, q, sk, cur, norm2);
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8u * st);
        }
        // Unaligned heads and tails (plain loads) after the tiles, from the last blocks first:
        // round-robin gives the first blocks the extra tile of a partial last round.
        const int64_t rb = (int64_t)gridDim.x - 1 - blockIdx.x;
        for (int64_t q = rb * kCT + ct; q < (int64_t)P.n_seg * kScalarSlots; q += (int64_t)gridDim.x * kCT) {
            const KSeg& S = P.seg[q / kScalarSlots];
            const int k = (int)(q % kScalarSlots);
            int64_t e = -1;
            if (k < S.head) e = k;
            else if (k - S.head < S.tail) e = S.head + 8 * S.nvec + (k - S.head);
            if (e >= 0) bad |= step_scalar<DT, MODE>(P, S, e, sk, cur, norm2);
        }
        if constexpr (HasGather<PT>::value) {
            // the gather copies' unaligned heads and tails (plain copies)
            for (int64_t q = (int64_t)blockIdx.x * kCT + ct; q < (int64_t)P.g_n * kScalarSlots;
                 q += (int64_t)gridDim.x * kCT) {
                const GCopy& C = P.gc[q / kScalarSlots];
                const int j = (int)(q % kScalarSlots);
                uint16_t* d = P.g_dst + C.dst_off;
                const int64_t head = head_elems(d, C.n);
                const int64_t body = ((int64_t)C.n - head) / 8 * 8;
                const int64_t tail = (int64_t)C.n - head - body;
                int64_t e = -1;
                if (j < head) e = j;
                else if (j - head < tail) e = head + body + (j - head);
                if (e >= 0) d[e] = C.src[e];
            }
        }
    } else if (P.n_d + 3 > kOneIssuerMaxCopies || lane == 0) {
        // The producer: lane 0 waits for a free buffer and arms its barrier with the tile's byte
        // count; the tile's N_d + 3 bulk copies are issued by lane 0 alone or, for tiles of
        // many copies, by the 32 lanes of the warp between them.  Lane 0 alone then streams a
        // gather (if any) and drains.
        const uint64_t policy = evict_first_policy();
        const uint32_t ring0 = full0 + kBulkBarrierBytes;
        const uint32_t cbytes = (uint32_t)P.tile * 2u, sbytes = (uint32_t)P.tile * 4u;
        int s = 0;
        int64_t base = 0;
        uint32_t k = 0;   // tiles issued
        if (P.n_d + 3 <= kOneIssuerMaxCopies) {
            for (int64_t tile = blockIdx.x; tile < P.n_tiles; tile += gridDim.x, ++k) {
                const TileRef T = locate_tile(P, tile, s, base);
                const uint32_t st = k % (uint32_t)P.stages;
                if (k >= (uint32_t)P.stages &&
                    !mbar_wait(empty0 + 8u * st, ((k / (uint32_t)P.stages) - 1u) & 1u, P.wait_ns)) {
                    err |= 1u;
                    break;
                }
                const KSeg& S = P.seg[s];
                const uint32_t full = full0 + 8u * st;
                const uint32_t dst = ring0 + st * stage_bytes;
                const uint32_t len = (uint32_t)T.len;
                mbar_arrive_expect_tx(full, len * (2u * (uint32_t)P.n_d + 12u));
                for (int r = 0; r < P.n_d; ++r)
                    bulk_load(dst + (uint32_t)r * cbytes, P.c[r] + S.c_off + T.e0, 2u * len, full, policy);
                const uint32_t sdst = dst + (uint32_t)P.n_d * cbytes;
                bulk_load(sdst, S.p[cur] + T.e0, 4u * len, full, policy);
                bulk_load(sdst + sbytes, S.m[cur] + T.e0, 4u * len, full, policy);
                bulk_load(sdst + 2u * sbytes, S.v[cur] + T.e0, 4u * len, full, policy);
            }
        } else {
            for (int64_t tile = blockIdx.x; tile < P.n_tiles; tile += gridDim.x, ++k) {
                const TileRef T = locate_tile(P, tile, s, base);
                const uint32_t st = k % (uint32_t)P.stages;
                bool ok = true;
                if (lane == 0 && k >= (uint32_t)P.stages)
                    ok = mbar_wait(empty0 + 8u * st, ((k / (uint32_t)P.stages) - 1u) & 1u, P.wait_ns);
                if (!__shfl_sync(0xFFFFFFFFu, (int)ok, 0)) {
                    if (lane == 0) err |= 1u;
                    break;
                }
                const KSeg& S = P.seg[s];
                const uint32_t full = full0 + 8u * st;
                const uint32_t dst = ring0 + st * stage_bytes;
                const uint32_t len = (uint32_t)T.len;
                if (lane == 0) mbar_arrive_expect_tx(full, len * (2u * (uint32_t)P.n_d + 12u));
                __syncwarp();
                const uint32_t sdst = dst + (uint32_t)P.n_d * cbytes;
                for (int c = lane; c < P.n_d + 3; c += 32) {
                    if (c < P.n_d) {
                        bulk_load(dst + (uint32_t)c * cbytes, P.c[c] + S.c_off + T.e0, 2u * len, full, policy);
                    } else {
                        const int j = c - P.n_d;
                        const float* src = j == 0 ? S.p[cur] : (j == 1 ? S.m[cur] : S.v[cur]);
                        bulk_load(sdst + (uint32_t)j * sbytes, src + T.e0, 4u * len, full, policy);
                    }
                }
            }
        }
        if (lane == 0) {
            const uint32_t ns = (uint32_t)P.stages;
            uint32_t used = k;   // ring buffers filled so far (tiles, then gather chunks)
            if constexpr (HasGather<PT>::value) {
                const int64_t grid = gridDim.x;
                const int64_t rb = grid - 1 - blockIdx.x;
                const int64_t mine = (!err && P.g_chunks > rb) ? (P.g_chunks - 1 - rb) / grid + 1 : 0;
                GChunkWalk<PT> lw, sw;
                int64_t lc = rb, sc = rb, issued = 0;
                // load of gather chunk `issued` into ring use k + issued: its buffer held a tile
                // (wait until the consumers release it) or the gather chunk ns uses before (whose
                // store has read it: the caller waited for all but the newest store group)
                auto issue = [&]() -> bool {
                    const uint32_t u = k + (uint32_t)issued, st = u % ns;
                    if (u >= ns && u - ns < k && !mbar_wait(empty0 + 8u * st, ((u / ns) - 1u) & 1u, P.wait_ns))
                        return false;
                    const uint16_t* src;
                    uint16_t* dst;
                    const TileRef T = lw.at(P, lc, &src, &dst);
                    const uint32_t full = full0 + 8u * st;
                    mbar_arrive_expect_tx(full, 2u * (uint32_t)T.len);
                    bulk_load(ring0 + st * stage_bytes, src + T.e0, 2u * (uint32_t)T.len, full, policy);
                    lc += grid;
                    ++issued;
                    return true;
                };
                if (mine > 0 && !issue()) err |= 4u;
                for (int64_t j = 0; j < mine && !err; ++j) {
                    const uint32_t u = k + (uint32_t)j, st = u % ns;
                    if (!mbar_wait(full0 + 8u * st, (u / ns) & 1u, P.wait_ns)) {
                        err |= 4u;
                        break;
                    }
                    const uint16_t* src;
                    uint16_t* dst;
                    const TileRef T = sw.at(P, sc, &src, &dst);
                    bulk_store(dst + T.e0, ring0 + st * stage_bytes, 2u * (uint32_t)T.len, policy);
                    bulk_commit();
                    sc += grid;
                    if (issued < mine) {
                        bulk_wait_read<1>();   // the store of chunk j - 1 has read its buffer
                        if (!issue()) {
                            err |= 4u;
                            break;
                        }
                    }
                }
                used = k + (uint32_t)issued;
            }
            // Drain: the last phase issued on each buffer completes before the block returns, and
            // so does every bulk store.
            for (uint32_t j = used > ns ? used - ns : 0u; j < used; ++j)
                if (!mbar_wait(full0 + 8u * (j % ns), (j / ns) & 1u, kDrainNs)) err |= 2u;
            if constexpr (HasGather<PT>::value) bulk_wait_all();
        }
    }
    if (err) atomicOr(&P.st->error, err);

    // Global non-finite flag: one OR across the block, one atomic per block that saw one.
    if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(P.flag, 1u);
}

// Gradient-norm pre-pass: the reduction of the fused kernel without the update; reads only
// the contributions.
template <int DT, int NB, int VEC, typename PT>
__global__ void __launch_bounds__(kThreads) grad_norm_kernel(const __grid_constant__ PT P)
{
    __shared__ float sk4[4];
    __shared__ int scur;
    block_constants(P, sk4, &scur);
    const float inv = sk4[2];
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    NormAcc norm2;
    auto one = [&](const KSeg& S, int64_t e) {
        float sum = 0.0f;
        for (int r = 0; r < P.n_d; ++r) sum = __fadd_rn(sum, widen1<DT>(P.c[r][S.c_off + e]));
        const float g = __fmul_rn(sum, inv);
        norm2.add(__fmul_rn(g, g));
    };
    if constexpr (VEC == 8) {
        for (int64_t q = tid; q < (int64_t)P.n_seg * kScalarSlots; q += stride) {
            const KSeg& S = P.seg[q / kScalarSlots];
            const int k = (int)(q % kScalarSlots);
            int64_t e = -1;
            if (k < S.head) e = k;
            else if (k - S.head < S.tail) e = S.head + 8 * S.nvec + (k - S.head);
            if (e >= 0) one(S, e);
        }
    }
    int s = 0;
    for (int64_t vi = tid; vi < P.total_vec; vi += stride) {
        while (vi >= P.seg[s].vbeg + P.seg[s].nvec) ++s;
        const KSeg& S = P.seg[s];
        if constexpr (VEC == 8) {
            const int64_t e = S.head + 8 * (vi - S.vbeg);
            float acc[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
            for (int r0 = 0; r0 < P.n_d; r0 += NB) {
                uint4 c[NB];
#pragma unroll
                for (int q = 0; q < NB; ++q)
                    if (r0 + q < P.n_d) c[q] = ld_stream(P.c[r0 + q] + S.c_off + e);
#pragma unroll
                for (int q = 0; q < NB; ++q) {
                    if (r0 + q < P.n_d) {
                        const uint32_t w[4] = {c[q].x, c[q].y, c[q].z, c[q].w};
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            float lo, hi;
                            widen2<DT>(w[j], lo, hi);
                            acc[2 * j] = __fadd_rn(acc[2 * j], lo);
                            acc[2 * j + 1] = __fadd_rn(acc[2 * j + 1], hi);
                        }
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float g = __fmul_rn(acc[j], inv);
                norm2.add(__fmul_rn(g, g));
            }
        } else {
            one(S, vi - S.vbeg);
        }
    }
    block_norm_commit<kThreads>(P, norm2.value());
}

// ZeRO-Offload: the reduction of the fused kernel, its averaged gradient written into the
// rank's pinned host buffer (S.p[0]) over NVLink-C2C instead of feeding an on-GPU update.
// STORE = false: the same reduction writing nothing, for the step's non-finite flag alone (a
// pass over HBM that lets the host know the skip decision before the gradients have landed).
template <int DT, int NB, int VEC, typename PT, bool STORE>
__global__ void __launch_bounds__(kThreads) reduce_to_host_kernel(const __grid_constant__ PT P)
{
    __shared__ float sk4[4];
    __shared__ int scur;
    block_constants(P, sk4, &scur);
    const float inv = sk4[2];
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    bool bad = false;
    auto one = [&](const KSeg& S, int64_t e) {
        float sum = 0.0f;
        for (int r = 0; r < P.n_d; ++r) sum = __fadd_rn(sum, widen1<DT>(P.c[r][S.c_off + e]));
        const float g = __fmul_rn(sum, inv);
        bad |= nonfinite(g);
        if constexpr (STORE) S.p[0][e] = g;
    };
    if constexpr (VEC == 8) {
        for (int64_t q = tid; q < (int64_t)P.n_seg * kScalarSlots; q += stride) {
            const KSeg& S = P.seg[q / kScalarSlots];
            const int k = (int)(q % kScalarSlots);
            int64_t e = -1;
            if (k < S.head) e = k;
            else if (k - S.head < S.tail) e = S.head + 8 * S.nvec + (k - S.head);
            if (e >= 0) one(S, e);
        }
    }
    // Vector path in halves of the 8-element vectors: each thread reduces 4 elements (one
    // 8-byte load per rank) and writes them with one 16-byte store, so a warp's store covers
    // whole 128-byte lines of host memory.  (With 8 elements per thread, each of its two
    // 16-byte stores covered half of every line, and the writes over NVLink-C2C ran at
    // 85 GB/s against the link's ~190 GB/s.)
    int s = 0;
    const int64_t units = VEC == 8 ? 2 * P.total_vec : P.total_vec;
    for (int64_t u = tid; u < units; u += stride) {
        const int64_t vi = VEC == 8 ? u >> 1 : u;
        while (vi >= P.seg[s].vbeg + P.seg[s].nvec) ++s;
        const KSeg& S = P.seg[s];
        if constexpr (VEC == 8) {
            const int64_t e = S.head + 8 * (vi - S.vbeg) + 4 * (u & 1);
            float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            for (int r0 = 0; r0 < P.n_d; r0 += NB) {
                uint2 c[NB];
#pragma unroll
                for (int q = 0; q < NB; ++q)
                    if (r0 + q < P.n_d) c[q] = ld_stream8(P.c[r0 + q] + S.c_off + e);
#pragma unroll
                for (int q = 0; q < NB; ++q) {
                    if (r0 + q < P.n_d) {
                        float a, b, d, f;
                        widen2<DT>(c[q].x, a, b);
                        widen2<DT>(c[q].y, d, f);
                        acc[0] = __fadd_rn(acc[0], a);
                        acc[1] = __fadd_rn(acc[1], b);
                        acc[2] = __fadd_rn(acc[2], d);
                        acc[3] = __fadd_rn(acc[3], f);
                    }
                }
            }
            float g[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                g[j] = __fmul_rn(acc[j], inv);
                bad |= nonfinite(g[j]);
            }
            if constexpr (STORE) *reinterpret_cast<float4*>(S.p[0] + e) = make_float4(g[0], g[1], g[2], g[3]);
        } else {
            one(S, vi - S.vbeg);
        }
    }
    if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(P.flag, 1u);
}

// ------------------------------------------------------------------ skip: re-cast + commit

// On a flagged (or discarded) step the fused kernels have already written 16-bit values of
// the rejected update; rewrite them from the unchanged current master.  Every block returns at once when
// the flag is clear (the usual case), so the launch costs a few microseconds.
template <int DT, int VEC, typename PT>
__global__ void __launch_bounds__(kThreads) recast_kernel(const __grid_constant__ PT P)
{
    __shared__ int go, scur;
    if (threadIdx.x == 0) {
        const volatile DevState* st = P.st;
        go = (st->flag | st->error) != 0;
        scur = (int)st->cur;
    }
    __syncthreads();
    const int cur = scur;
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    if (go && VEC == 8) {
        for (int64_t q = tid; q < (int64_t)P.n_seg * kScalarSlots; q += stride) {
            const KSeg& S = P.seg[q / kScalarSlots];
            const int k = (int)(q % kScalarSlots);
            int64_t e = -1;
            if (k < S.head) e = k;
            else if (k - S.head < S.tail) e = S.head + 8 * S.nvec + (k - S.head);
            if (e >= 0) S.out16[e] = narrow1<DT>(S.p[cur][e]);
        }
    }
    int s = 0;
    if constexpr (VEC == 8) {
        // four vectors per thread and iteration, loads before stores: the launch has one block
        // per SM, so each thread keeps several loads in flight
        constexpr int kU = 4;
        for (int64_t v0 = go ? tid : P.total_vec; v0 < P.total_vec; v0 += kU * stride) {
            float4 a[kU], b[kU];
            uint16_t* dst[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int64_t vi = v0 + u * stride;
                dst[u] = nullptr;
                if (vi < P.total_vec) {
                    while (vi >= P.seg[s].vbeg + P.seg[s].nvec) ++s;
                    const KSeg& S = P.seg[s];
                    const int64_t e = S.head + 8 * (vi - S.vbeg);
                    a[u] = __ldcs(reinterpret_cast<const float4*>(S.p[cur] + e));
                    b[u] = __ldcs(reinterpret_cast<const float4*>(S.p[cur] + e) + 1);
                    dst[u] = S.out16 + e;
                }
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                if (dst[u]) {
                    uint4 o;
                    o.x = narrow2<DT>(a[u].x, a[u].y);
                    o.y = narrow2<DT>(a[u].z, a[u].w);
                    o.z = narrow2<DT>(b[u].x, b[u].y);
                    o.w = narrow2<DT>(b[u].z, b[u].w);
                    __stcs(reinterpret_cast<uint4*>(dst[u]), o);
                }
            }
        }
    } else {
        for (int64_t vi = go ? tid : P.total_vec; vi < P.total_vec; vi += stride) {
            while (vi >= P.seg[s].vbeg + P.seg[s].nvec) ++s;
            const KSeg& S = P.seg[s];
            const int64_t e = vi - S.vbeg;
            S.out16[e] = narrow1<DT>(S.p[cur][e]);
        }
    }
    // The last launch of the re-cast also closes the step.  Clean step (the usual case):
    // nothing was re-cast and the commit leaves the flag clear, so block 0 commits at once; a
    // block that reads the state after that still sees a clear flag and does nothing.
    // Flagged or discarded step: the last block to finish (atomic ticket; every block read
    // the flag and the current half before taking its ticket) commits.
    if (P.do_commit && !go) {
        if (blockIdx.x == 0 && threadIdx.x == 0) {
            commit_state(P.commit);
            __threadfence();
        }
        return;
    }
    if (P.do_commit) {
        __shared__ bool last;
        __syncthreads();
        if (threadIdx.x == 0) {
            __threadfence();
            last = atomicAdd(&P.st->blocks_done, 1u) == gridDim.x - 1;
        }
        __syncthreads();
        if (last && threadIdx.x == 0) {
            __threadfence();
            reinterpret_cast<volatile DevState*>(P.st)->blocks_done = 0;
            commit_state(P.commit);
            __threadfence();
        }
    }
}

// Close the step on the device: flag clear -> flip the current half, t += 1, count a clean
// step and grow the scale after `interval` of them; flag set -> keep the state, back the
// scale off (not below min_scale).  Then clear the flag for the next step.  While the error
// word is set (a bounded wait ran out) the step is discarded: nothing but the flag moves.
__device__ __forceinline__ void commit_state(const CommitParams& C)
{
    volatile DevState* st = C.st;
    // All fields are loaded first (independent loads: one round trip to L2), then the new
    // values are formed and stored.
    const uint32_t error = st->error, flag = st->flag, cur = st->cur, norm_valid = st->norm_valid;
    const int64_t t = st->t, skipped = st->skipped, good = st->good, finished = st->finished;
    const double scale = st->scale, norm2 = st->norm2;
    uint32_t n_cur = cur, n_last = 1;
    int64_t n_t = t, n_skipped = skipped, n_good = good;
    double n_scale = scale;
    if (error) {
        // discarded: nothing else moves
    } else if (flag) {
        n_skipped = skipped + 1;
        if (C.dynamic) {
            const double sc = scale * C.backoff;
            n_scale = sc < C.min_scale ? C.min_scale : sc;
        }
        n_good = 0;
    } else {
        n_last = 0;
        n_cur = cur ^ 1u;
        n_t = t + 1;
        n_good = good + 1;
        if (C.dynamic && C.interval > 0 && n_good >= C.interval) {
            n_scale = scale * C.growth;
            n_good = 0;
        }
    }
    st->last_skipped = n_last;
    st->cur = n_cur;
    st->t = n_t;
    st->skipped = n_skipped;
    st->good = n_good;
    st->scale = n_scale;
    st->finished = error ? finished : finished + 1;
    st->flag = 0;
    st->last_norm2 = norm2;
    st->last_norm_valid = norm_valid;
    st->norm2 = 0.0;
    st->norm_valid = 0;
}

__global__ void commit_kernel(const CommitParams C)
{
    if (blockIdx.x != 0 || threadIdx.x != 0) return;
    commit_state(C);
}

// ------------------------------------------------------------------ gather kernel (stage 3)

template <int VEC, typename CP>
__global__ void __launch_bounds__(kThreads) gather_kernel(const __grid_constant__ CP P)
{
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    if constexpr (VEC == 8) {
        for (int64_t q = tid; q < (int64_t)P.n_seg * kScalarSlots; q += stride) {
            const CopySeg& S = P.seg[q / kScalarSlots];
            const int k = (int)(q % kScalarSlots);
            int64_t e = -1;
            if (k < S.head) e = k;
            else if (k - S.head < S.tail) e = S.head + 8 * S.nvec + (k - S.head);
            if (e >= 0) S.dst[e] = S.src[e];
        }
    }
    // Body: block b copies one contiguous range of vectors, its threads striding by the block
    // size, so that a thread's walk over the copy list (up to 256 items) starts with a binary
    // search and then advances at most a few items.
    const int64_t per = ((P.total_vec + gridDim.x - 1) / gridDim.x + blockDim.x - 1) / blockDim.x *
                        blockDim.x;
    const int64_t v0 = (int64_t)blockIdx.x * per + threadIdx.x;
    const int64_t v_end = min(P.total_vec, ((int64_t)blockIdx.x + 1) * per);
    if (v0 >= v_end) return;
    int lo = 0, hi = P.n_seg - 1;   // last item whose first vector is at or before v0
    while (lo < hi) {
        const int mid = (lo + hi + 1) / 2;
        if (P.seg[mid].vbeg <= v0) lo = mid;
        else hi = mid - 1;
    }
    int s = lo;
    for (int64_t vi = v0; vi < v_end; vi += blockDim.x) {
        while (vi >= P.seg[s].vbeg + P.seg[s].nvec) ++s;
        const CopySeg& S = P.seg[s];
        if constexpr (VEC == 8) {
            const int64_t e = S.head + 8 * (vi - S.vbeg);
            __stcs(reinterpret_cast<uint4*>(S.dst + e), __ldcs(reinterpret_cast<const uint4*>(S.src + e)));
        } else {
            const int64_t e = vi - S.vbeg;
            S.dst[e] = S.src[e];
        }
    }
}

// ------------------------------------------------------------------ bulk-staged gather (stage 3)

// The register-load gather above keeps one 16-byte load per thread in flight (~30 KB per SM),
// which leaves copies of a ~100 MB unit latency-bound.  Here one lane per block moves the
// bytes with 1-D bulk copies through a ring of `stages` shared-memory chunks: global ->
// shared loads complete on the chunk's mbarrier (bounded waits), shared -> global bulk stores
// are tracked as bulk groups, and the loads run stages - kGatherStoresPending chunks ahead of
// the stores, so each block keeps ~(stages - 2) chunks of loads in flight.  The other lanes
// copy the unaligned heads and tails with plain loads.  Block b takes chunks b, b + grid, ...
// (a chunk never crosses the end of a copy).  A wait that runs out sets bit 2 of the error
// word; the lane then waits (bounded) for the loads it issued and for its stores, and returns.
constexpr int kGatherThreads = 32;
constexpr int kGatherStoresPending = 2;      // bulk stores left in flight when a chunk is reused
constexpr int kGatherMaxStages = 32;
constexpr int kGatherBarrierBytes = 8 * kGatherMaxStages;
constexpr int kGatherMaxChunk = 32768;
// Default geometry, measured on GB300: 32 KB copies, four entries (two loads ahead), a 128 KB
// ring and so one block per SM.  Against register loads: 1.3B units (100 MB) 5.55 -> 5.74
// TB/s, Llama rank-view units (405 MB) 6.17 -> 6.54 TB/s, per-parameter gathers even (1.3B)
// and +6 % (Llama).  Smaller copies with more blocks per SM gathered the 1.3B units faster
// (6.1 TB/s with 24 KB x 4) but slowed the Llama step kernel that follows each gather from
// 0.95 to 0.92 of the copy bandwidth.
constexpr int kGatherDefaultChunk = 16384;
constexpr int kGatherDefaultStages = 4;

// Walk over the chunks of a launch in increasing order (chunk ids b, b + grid, ...): the
// copy holding the current chunk and its chunk range (from the host's first-chunk table) are
// carried along, so a step costs compares and adds, also across runs of one-chunk copies.
template <typename CP>
struct ChunkWalk {
    int s = -1;
    int64_t first = 0, end = 0;   // chunk ids of copy s: [first, end)

    __device__ __forceinline__ TileRef at(const CP& P, int64_t c)
    {
        while (c >= end) {
            ++s;
            first = end;
            end = s + 1 < P.n_seg ? P.seg[s + 1].cbeg : P.n_chunks;
        }
        const CopySeg& S = P.seg[s];
        const int64_t off = (c - first) * P.chunk;
        TileRef r;
        r.e0 = S.head + off;
        r.len = (int32_t)min((int64_t)P.chunk, 8 * S.nvec - off);
        return r;
    }
};

template <typename CP>
__global__ void __launch_bounds__(kGatherThreads) bulk_gather_kernel(const __grid_constant__ CP P)
{
    extern __shared__ __align__(128) unsigned char gather_raw[];
    const uint32_t raw = (uint32_t)__cvta_generic_to_shared(gather_raw);
    const uint32_t full0 = (raw + 127u) & ~127u;
    const uint32_t ring0 = full0 + kGatherBarrierBytes;
    const uint32_t ns = (uint32_t)P.stages, cbytes = (uint32_t)P.chunk * 2u;
    const int lane = threadIdx.x;
    if (lane == 0) {
        for (uint32_t i = 0; i < ns; ++i) mbar_init(full0 + 8u * i, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncwarp();
    if (lane != 0) {
        // unaligned heads and tails: plain copies by the other lanes, while lane 0 streams
        constexpr int kLanes = kGatherThreads - 1;
        for (int64_t q = (int64_t)blockIdx.x * kLanes + (lane - 1); q < (int64_t)P.n_seg * kScalarSlots;
             q += (int64_t)gridDim.x * kLanes) {
            const CopySeg& S = P.seg[q / kScalarSlots];
            const int k = (int)(q % kScalarSlots);
            int64_t e = -1;
            if (k < S.head) e = k;
            else if (k - S.head < S.tail) e = S.head + 8 * S.nvec + (k - S.head);
            if (e >= 0) S.dst[e] = S.src[e];
        }
        return;
    }
    const uint64_t policy = evict_first_policy();
    const int64_t grid = gridDim.x;
    const int64_t mine = P.n_chunks > blockIdx.x ? (P.n_chunks - 1 - blockIdx.x) / grid + 1 : 0;
    const int64_t ahead = (int64_t)ns - kGatherStoresPending;
    ChunkWalk<CP> lw, sw;             // load / store walkers
    uint32_t err = 0;
    // loads: chunk id, ring entry and count issued; stores: the same, with the entry's phase
    int64_t lc = blockIdx.x, issued = 0;
    uint32_t lst = 0;
    auto issue_load = [&]() {
        const TileRef T = lw.at(P, lc);
        const uint32_t full = full0 + 8u * lst;
        mbar_arrive_expect_tx(full, 2u * (uint32_t)T.len);
        bulk_load(ring0 + lst * cbytes, P.seg[lw.s].src + T.e0, 2u * (uint32_t)T.len, full, policy);
        lc += grid;
        ++issued;
        if (++lst == ns) lst = 0;
    };
    while (issued < mine && issued < ahead) issue_load();
    int64_t sc = blockIdx.x, j = 0;
    uint32_t sst = 0, phase = 0;
    for (; j < mine; ++j) {
        if (!mbar_wait(full0 + 8u * sst, phase, P.wait_ns)) {
            err |= 4u;
            break;
        }
        const TileRef T = sw.at(P, sc);
        bulk_store(P.seg[sw.s].dst + T.e0, ring0 + sst * cbytes, 2u * (uint32_t)T.len, policy);
        bulk_commit();
        sc += grid;
        if (++sst == ns) {
            sst = 0;
            phase ^= 1u;
        }
        if (issued < mine) {
            // the next load reuses the entry of the chunk stored kGatherStoresPending groups
            // before the newest
            bulk_wait_read<kGatherStoresPending>();
            issue_load();
        }
    }
    // Drain: every load issued and not yet waited for lands, and every store completes,
    // before the block's shared memory goes away.
    for (; j < issued; ++j) {
        if (!mbar_wait(full0 + 8u * sst, phase, kDrainNs)) err |= 2u;
        if (++sst == ns) {
            sst = 0;
            phase ^= 1u;
        }
    }
    bulk_wait_all();
    if (err && P.err) atomicOr(P.err, err);
}

}  // namespace
}  // namespace zero
