// zero_offload.cpp -- the host side of ZeRO-Offload on a Grace-Blackwell node: the fp32 AdamW
// update of host-resident master/m/v, run by CPU threads.
//
// Page: "Zero Redundancy Optimizer (ZeRO) and Fully Sharded Data Parallelism (FSDP):
// Mathematical Foundations ..." (llms.blog), "ZeRO-Offload Mechanics": the forward and
// backward passes stay on the GPU, the AdamW step (O(1) operations per parameter) runs on the
// host CPU over fp32 state in host memory, gradients travel to the host and updated
// parameters back.  Here the GPU writes the averaged fp32 gradient straight into pinned host
// memory over NVLink-C2C; this file updates the state and produces the 16-bit parameters.
//
// Built with -O3 -ffp-contract=off: every fp32 operation is separately rounded in the order
// the GPU kernel uses, so offloaded and on-GPU updates agree bit for bit.  With
// -fno-math-errno the loops vectorise (IEEE division and square root have exact vector forms
// on Arm and x86; errno would only be set for a negative square-root argument, and v >= 0).
#include <algorithm>
#include <cmath>
#include <cstring>
#include <thread>
#include <vector>

#include "zero_internal.h"

namespace zero {
namespace {

inline uint32_t bits_of(float f)
{
    uint32_t u;
    std::memcpy(&u, &f, sizeof(u));
    return u;
}

// fp32 -> bfloat16, round to nearest even (bf16 is the upper half of a binary32).
inline uint16_t to_bf16(float f)
{
    uint32_t u = bits_of(f);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x0040u);   // quiet NaN
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

inline float float_of(uint32_t u)
{
    float f;
    std::memcpy(&f, &u, sizeof(f));
    return f;
}

// fp32 -> IEEE binary16, round to nearest even, subnormals and overflow to infinity included,
// without branches (so that loops over it vectorise):
//  - normal halves: rebias the exponent (subtract 112 << 23) and round the 13 dropped
//    mantissa bits to nearest even -- a carry into the exponent is the correct result;
//  - subnormal halves (|f| < 2^-14): |f| + 0.5 puts the half's ulp, 2^-24, at the last place
//    of the float, so the fp32 addition itself rounds to nearest even; what it added to 0.5
//    is the half's bit pattern (1024 = the smallest normal);
//  - |f| rounding past 65504 -> infinity; NaN -> quiet NaN with the sign kept.
inline uint16_t to_fp16(float f)
{
    const uint32_t u = bits_of(f);
    const uint32_t sign = (u >> 16) & 0x8000u;
    const uint32_t a = u & 0x7FFFFFFFu;
    const uint32_t nrm = (a - 0x38000000u + 0x0FFFu + ((a >> 13) & 1u)) >> 13;
    const uint32_t sub = bits_of(float_of(a) + 0.5f) - 0x3F000000u;
    uint32_t h = a >= 0x38800000u ? nrm : sub;
    h = a >= 0x477FF000u ? 0x7C00u : h;
    h = a > 0x7F800000u ? 0x7E00u : h;
    return (uint16_t)(sign | h);
}

template <bool FP16>
void adamw_span(const CpuSpan& s, const float* k)
{
    const float b1 = k[0], omb1 = k[1], b2 = k[2], omb2 = k[3], eps = k[4], lrwd = k[5];
    const float step = k[6], bc2s = k[7];
    float* __restrict p = s.master;
    float* __restrict m = s.m;
    float* __restrict v = s.v;
    const float* __restrict g = s.grad;
    uint16_t* __restrict out = s.out16;
    for (int64_t i = 0; i < s.n; ++i) {
        const float gi = g[i];
        const float mi = b1 * m[i] + omb1 * gi;
        const float vi = b2 * v[i] + omb2 * (gi * gi);
        const float d = std::sqrt(vi) / bc2s + eps;
        float pi = p[i] - lrwd * p[i];
        pi = pi - step * (mi / d);
        m[i] = mi;
        v[i] = vi;
        p[i] = pi;
        out[i] = FP16 ? to_fp16(pi) : to_bf16(pi);
    }
}

template <bool FP16>
void recast_span(const CpuSpan& s)
{
    for (int64_t i = 0; i < s.n; ++i) s.out16[i] = FP16 ? to_fp16(s.master[i]) : to_bf16(s.master[i]);
}

}  // namespace

void cpu_adamw(const std::vector<CpuSpan>& spans, const float k[9], int dtype16, bool skipped,
               int threads)
{
    // Cut the spans into pieces of ~64K elements and deal them to the threads in turn.
    constexpr int64_t kPiece = 1 << 16;
    std::vector<CpuSpan> pieces;
    for (const CpuSpan& s : spans)
        for (int64_t o = 0; o < s.n; o += kPiece) {
            CpuSpan q = s;
            q.n = std::min(kPiece, s.n - o);
            q.master += o;
            q.m += o;
            q.v += o;
            q.grad += o;
            q.out16 += o;
            pieces.push_back(q);
        }
    const int nt = std::max(1, std::min<int>(threads, (int)pieces.size()));
    auto work = [&](int tid) {
        for (size_t i = (size_t)tid; i < pieces.size(); i += (size_t)nt) {
            const CpuSpan& q = pieces[i];
            if (skipped) {
                if (dtype16 == ZERO_FP16) recast_span<true>(q);
                else recast_span<false>(q);
            } else if (dtype16 == ZERO_FP16) {
                adamw_span<true>(q, k);
            } else {
                adamw_span<false>(q, k);
            }
        }
    };
    if (nt == 1) {
        work(0);
        return;
    }
    std::vector<std::thread> pool;
    for (int t = 1; t < nt; ++t) pool.emplace_back(work, t);
    work(0);
    for (auto& th : pool) th.join();
}

}  // namespace zero
