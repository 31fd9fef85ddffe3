// zero_oracle.cpp -- CPU ORACLE of the sharded mixed-precision AdamW step.
//
// TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, single-threaded
// definition that the GPU path is checked against.  Only the tests, the smoke
// check and the benchmark's CPU-baseline leg may load it.  It shares no code,
// header, table or helper with the GPU library (the only common module is the
// seeded input generator, which holds none of the step's arithmetic).
//
// Sources (web pages; cited by title and section):
//   [ZF]  "Zero Redundancy Optimizer (ZeRO) and Fully Sharded Data Parallelism
//          (FSDP): Mathematical Foundations of Memory Partitioning, Communication
//          Complexity, and Overlapped Execution" (llms.blog)
//   [ZP]  "ZeRO: Memory Optimizations Toward Training Trillion Parameter
//          Models" summary card (fanout.sh)
//
// Readings where the pages are silent (the pages never write out AdamW,
// loss scaling, overflow handling or buckets):
//   R1 AdamW = decoupled weight decay (Loshchilov & Hutter) with Adam's bias
//      correction (Kingma & Ba); eps outside the square root; decay applied to
//      the pre-update weight; t counts applied steps, 1-based.
//   R2 The reduced gradient is sum_r c_r (fp32, r ascending) times
//      inv = fp32(1 / (N_d * loss_scale)), one multiply after the sum.
//   R3 Reduction precision is fp32 (not a 16-bit ring).
//   R4 Padding: only the tail of each flat buffer, up to a multiple of N_d.
//   R5 A step with any non-finite reduced gradient element is skipped as a
//      whole: master/m/v and t unchanged, 16-bit params re-cast from master.
//   R6 16-bit casts round to nearest, ties to even.
//   R7 All fp32 arithmetic uses separately rounded operations in the order
//      written below (built with -ffp-contract=off, no fast-math).
//   R8 Optional global gradient norm and clipping: norm^2 = sum over the
//      updated elements of fp32(g*g), summed in double, g the averaged,
//      unscaled, unclipped gradient; clipping multiplies g by
//      fp32(min(1, max_norm / (sqrt(norm^2) + 1e-6))) before AdamW (the rule
//      of torch.nn.utils.clip_grad_norm_).  The skip flag is taken on g.
//
// Parity pins (tests/test_oracle_pins.py): closed-form memory and
// communication figures of [ZF]; brute-force tables on tiny inputs; DDP
// equivalence ([ZF] "Mathematical Formulation of ZeRO Partitioning Stages":
// sharding keeps the exact semantics of data parallelism); torch.optim.AdamW
// and numpy/torch 16-bit conversions as library cross-checks; closed forms of
// the first AdamW step.  What the pins fix up to rounding rather than bit for
// bit is the choice among equally valid fp32 operation orders of the update
// (R1/R7) and of the reduction (R2/R3): a reading, shared with the GPU path.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

// ---------------------------------------------------------------------------
// 16-bit encodings ([ZF] "Static Memory Allocation": parameters and gradients
// are stored in FP16 or BF16).  Written from the IEEE-754 / bfloat16 format
// definitions: value = (-1)^s * 2^(E - bias) * (1 + M / 2^mbits), subnormals
// at E = 0.
// ---------------------------------------------------------------------------

float widen_bf16(uint16_t h)
{
    const int s = (h >> 15) & 1;
    const int E = (h >> 7) & 0xFF;
    const int M = h & 0x7F;
    double mag;
    if (E == 0) mag = std::ldexp((double)M, -133);
    else if (E == 0xFF) mag = (M == 0) ? INFINITY : NAN;
    else mag = std::ldexp((double)(128 + M), E - 134);
    return (float)(s ? -mag : mag);
}

float widen_fp16(uint16_t h)
{
    const int s = (h >> 15) & 1;
    const int E = (h >> 10) & 0x1F;
    const int M = h & 0x3FF;
    double mag;
    if (E == 0) mag = std::ldexp((double)M, -24);
    else if (E == 0x1F) mag = (M == 0) ? INFINITY : NAN;
    else mag = std::ldexp((double)(1024 + M), E - 25);
    return (float)(s ? -mag : mag);
}

// Round |x| (exact, in double) to a binary format with `mbits` mantissa bits,
// exponent range [emin, emax]; returns the magnitude encoding.  rint() rounds
// to nearest, ties to even, in the default rounding mode.
uint16_t round_mag(double x, int mbits, int emin, int emax, int bias, uint16_t inf_bits)
{
    if (x == 0.0) return 0;
    if (std::isinf(x)) return inf_bits;
    const double min_normal = std::ldexp(1.0, emin);
    if (x < min_normal) {
        // subnormal: units of 2^(emin - mbits); q == 2^mbits encodes the min normal
        double q = std::rint(std::ldexp(x, mbits - emin));
        return (uint16_t)q;
    }
    int ex = 0;
    (void)std::frexp(x, &ex);  // x = fr * 2^ex, fr in [0.5, 1)
    int e = ex - 1;            // 2^e <= x < 2^(e+1)
    double q = std::rint(std::ldexp(x, mbits - e));  // in [2^mbits, 2^(mbits+1)]
    if (q == std::ldexp(1.0, mbits + 1)) {
        q = std::ldexp(1.0, mbits);
        e += 1;
    }
    if (e > emax) return inf_bits;
    const uint32_t mant = (uint32_t)q - (1u << mbits);
    return (uint16_t)(((uint32_t)(e + bias) << mbits) | mant);
}

uint16_t round_bf16(float f)
{
    if (std::isnan(f)) return 0x7FC0;
    const uint16_t sign = std::signbit(f) ? 0x8000 : 0;
    return (uint16_t)(sign | round_mag(std::fabs((double)f), 7, -126, 127, 127, 0x7F80));
}

uint16_t round_fp16(float f)
{
    if (std::isnan(f)) return 0x7E00;
    const uint16_t sign = std::signbit(f) ? 0x8000 : 0;
    return (uint16_t)(sign | round_mag(std::fabs((double)f), 10, -14, 15, 15, 0x7C00));
}

inline float widen16(uint16_t h, int is_fp16) { return is_fp16 ? widen_fp16(h) : widen_bf16(h); }
inline uint16_t round16(float f, int is_fp16) { return is_fp16 ? round_fp16(f) : round_bf16(f); }

// ---------------------------------------------------------------------------
// Step constants (R1, R2): computed in double on the host, rounded once to fp32.
// ---------------------------------------------------------------------------
struct Consts {
    float b1, omb1, b2, omb2, eps, lrwd, step, bc2s, inv;
};

Consts make_consts(double lr, double beta1, double beta2, double eps, double wd, int64_t t,
                   double loss_scale, int n_d)
{
    Consts k;
    const double bc1 = 1.0 - std::pow(beta1, (double)t);
    const double bc2 = 1.0 - std::pow(beta2, (double)t);
    k.b1 = (float)beta1;
    k.omb1 = (float)(1.0 - beta1);
    k.b2 = (float)beta2;
    k.omb2 = (float)(1.0 - beta2);
    k.eps = (float)eps;
    k.lrwd = (float)(lr * wd);
    k.step = (float)(lr / bc1);
    k.bc2s = (float)std::sqrt(bc2);
    k.inv = (float)(1.0 / ((double)n_d * loss_scale));
    return k;
}

Consts unpack(const float* k9)
{
    Consts k;
    k.b1 = k9[0]; k.omb1 = k9[1]; k.b2 = k9[2]; k.omb2 = k9[3]; k.eps = k9[4];
    k.lrwd = k9[5]; k.step = k9[6]; k.bc2s = k9[7]; k.inv = k9[8];
    return k;
}

// ---------------------------------------------------------------------------
// Reduce-scatter's reduction for one element ([ZF] "Execution Flow for
// ZeRO-1", step 2: each rank receives the averaged gradient of its
// partition), unscaled by the loss scale (R2), and the non-finite test (R5).
// ---------------------------------------------------------------------------
inline float reduce_one(int n_d, const uint16_t* const* c, int64_t idx, int is_fp16, float inv)
{
    float sum = 0.0f;
    for (int r = 0; r < n_d; ++r) sum = sum + widen16(c[r][idx], is_fp16);
    return sum * inv;
}

inline int nonfinite(float g) { return std::isfinite(g) ? 0 : 1; }

// Clip coefficient of R8 (NaN stays NaN; only a skipped step can see one).
float clip_coef(double norm2, double max_norm)
{
    double c = max_norm / (std::sqrt(norm2) + 1e-6);
    if (c > 1.0) c = 1.0;
    return (float)c;
}

// AdamW on one element, fp32, in this order (R1, R7).
inline void adamw_one(float g, float& p, float& m, float& v, const Consts& k)
{
    m = k.b1 * m + k.omb1 * g;
    v = k.b2 * v + k.omb2 * (g * g);
    const float denom = std::sqrt(v) / k.bc2s + k.eps;
    p = p - k.lrwd * p;
    p = p - k.step * (m / denom);
}

// ---------------------------------------------------------------------------
// Flat-buffer partition ([ZF] "FSDP-1: FlatParameter and Module-Level
// Wrapping": a unit's tensors are flattened into one 1-D buffer, padded to be
// divisible by N_d and sliced into N_d equal chunks).  Stages 1/2 use one unit
// covering every tensor; stage 3 one flat buffer per unit.
// ---------------------------------------------------------------------------
struct Unit {
    int64_t first, count, numel, numel_pad, shard, base, shard_base;
};

struct Layout {
    std::vector<Unit> units;
    std::vector<int64_t> tensor_offset;  // global flat offset of each tensor
    int64_t total_pad = 0;               // sum of numel_pad
    int64_t shard_total = 0;             // sum of shard sizes (elements per rank)
};

bool make_layout(const int64_t* sizes, int64_t n_tensors, const int64_t* unit_first,
                 int64_t n_units, int n_d, Layout& L)
{
    if (n_d < 1 || n_tensors < 0) return false;
    std::vector<int64_t> firsts;
    if (unit_first == nullptr || n_units <= 0) firsts.push_back(0);
    else firsts.assign(unit_first, unit_first + n_units);
    if (firsts[0] != 0) return false;
    for (size_t u = 1; u < firsts.size(); ++u)
        if (firsts[u] <= firsts[u - 1] || firsts[u] > n_tensors) return false;
    L.units.clear();
    L.tensor_offset.assign((size_t)n_tensors, 0);
    int64_t base = 0, shard_base = 0;
    for (size_t u = 0; u < firsts.size(); ++u) {
        Unit U;
        U.first = firsts[u];
        U.count = ((u + 1 < firsts.size()) ? firsts[u + 1] : n_tensors) - U.first;
        U.numel = 0;
        for (int64_t t = U.first; t < U.first + U.count; ++t) {
            if (sizes[t] < 0) return false;
            L.tensor_offset[(size_t)t] = base + U.numel;
            U.numel += sizes[t];
        }
        // smallest multiple of n_d that is >= numel
        U.numel_pad = U.numel;
        while (U.numel_pad % n_d != 0) U.numel_pad += 1;
        U.shard = U.numel_pad / n_d;
        U.base = base;
        U.shard_base = shard_base;
        base += U.numel_pad;
        shard_base += U.shard;
        L.units.push_back(U);
    }
    L.total_pad = base;
    L.shard_total = shard_base;
    return true;
}

}  // namespace

extern "C" {

// ---- 16-bit conversions (exported for the pins) ----
float orc_widen16(uint16_t h, int is_fp16) { return widen16(h, is_fp16); }
uint16_t orc_round16(float f, int is_fp16) { return round16(f, is_fp16); }

void orc_widen16_array(const uint16_t* h, int64_t n, int is_fp16, float* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = widen16(h[i], is_fp16);
}

void orc_round16_array(const float* f, int64_t n, int is_fp16, uint16_t* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = round16(f[i], is_fp16);
}

// ---- constants: out[9] = b1, 1-b1, b2, 1-b2, eps, lr*wd, lr/bc1, sqrt(bc2), 1/(N*scale) ----
void orc_consts(double lr, double beta1, double beta2, double eps, double wd, int64_t t,
                double loss_scale, int n_d, float* out)
{
    Consts k = make_consts(lr, beta1, beta2, eps, wd, t, loss_scale, n_d);
    const float v[9] = {k.b1, k.omb1, k.b2, k.omb2, k.eps, k.lrwd, k.step, k.bc2s, k.inv};
    std::memcpy(out, v, sizeof(v));
}

// ---- A3/A4: g[i] = inv * sum_r c_r[i]; returns 1 if any g[i] is non-finite ----
int orc_reduce(int64_t n, int n_d, const uint16_t* const* contrib, int is_fp16, float inv,
               float* g)
{
    int flag = 0;
    for (int64_t i = 0; i < n; ++i) {
        g[i] = reduce_one(n_d, contrib, i, is_fp16, inv);
        flag |= nonfinite(g[i]);
    }
    return flag;
}

// ---- A5/A6: AdamW on n elements, then the 16-bit cast ----
void orc_adamw(int64_t n, const float* g, float* p, float* m, float* v, const float* k9,
               int is_fp16, uint16_t* out16)
{
    const Consts k = unpack(k9);
    for (int64_t i = 0; i < n; ++i) {
        adamw_one(g[i], p[i], m[i], v[i], k);
        if (out16) out16[i] = round16(p[i], is_fp16);
    }
}

// ---- skipped step: 16-bit params re-cast from the unchanged master (R5) ----
void orc_recast(int64_t n, const float* p, int is_fp16, uint16_t* out16)
{
    for (int64_t i = 0; i < n; ++i) out16[i] = round16(p[i], is_fp16);
}

// ---- A1 tables ----
// unit_rows: n_units rows of 7 int64 = first, count, numel, numel_pad, shard, base, shard_base.
// Returns the number of units, or -1 on invalid input.
int64_t orc_layout(const int64_t* sizes, int64_t n_tensors, const int64_t* unit_first,
                   int64_t n_units, int n_d, int64_t* tensor_offset, int64_t* unit_rows,
                   int64_t cap_units)
{
    Layout L;
    if (!make_layout(sizes, n_tensors, unit_first, n_units, n_d, L)) return -1;
    if ((int64_t)L.units.size() > cap_units) return -1;
    for (int64_t t = 0; t < n_tensors; ++t) tensor_offset[t] = L.tensor_offset[(size_t)t];
    for (size_t u = 0; u < L.units.size(); ++u) {
        const Unit& U = L.units[u];
        const int64_t row[7] = {U.first, U.count, U.numel, U.numel_pad, U.shard, U.base,
                                U.shard_base};
        std::memcpy(unit_rows + 7 * u, row, sizeof(row));
    }
    return (int64_t)L.units.size();
}

// Shard segments: rows of 6 int64 = (rank, unit, tensor or -1 for padding,
// offset inside the tensor (or inside the padding), rank-local shard offset,
// length).  Order: rank, then unit, then ascending flat position.  Each row is
// the intersection of the shard interval [base + r*S, base + (r+1)*S) with one
// tensor's interval (tensors in flattening order), then with the unit's tail
// padding.  Returns the row count (rows beyond `cap` are counted, not written).
int64_t orc_shard_segments(const int64_t* sizes, int64_t n_tensors, const int64_t* unit_first,
                           int64_t n_units, int n_d, int64_t* rows, int64_t cap)
{
    Layout L;
    if (!make_layout(sizes, n_tensors, unit_first, n_units, n_d, L)) return -1;
    int64_t count = 0;
    auto emit = [&](int64_t r, int64_t u, int64_t t, int64_t in_off, int64_t sh_off, int64_t len) {
        if (count < cap) {
            const int64_t row[6] = {r, u, t, in_off, sh_off, len};
            std::memcpy(rows + 6 * count, row, sizeof(row));
        }
        ++count;
    };
    for (int r = 0; r < n_d; ++r) {
        for (size_t u = 0; u < L.units.size(); ++u) {
            const Unit& U = L.units[u];
            const int64_t lo = U.base + (int64_t)r * U.shard, hi = lo + U.shard;
            for (int64_t t = U.first; t < U.first + U.count; ++t) {
                const int64_t t_lo = L.tensor_offset[(size_t)t], t_hi = t_lo + sizes[t];
                const int64_t a = (t_lo > lo) ? t_lo : lo;
                const int64_t e = (t_hi < hi) ? t_hi : hi;
                if (a < e) emit(r, (int64_t)u, t, a - t_lo, U.shard_base + (a - lo), e - a);
            }
            const int64_t p_lo = U.base + U.numel, p_hi = U.base + U.numel_pad;
            const int64_t a = (p_lo > lo) ? p_lo : lo;
            const int64_t e = (p_hi < hi) ? p_hi : hi;
            if (a < e) emit(r, (int64_t)u, -1, a - p_lo, U.shard_base + (a - lo), e - a);
        }
    }
    return count;
}

// Bucket segments (stages 1/2, one unit): bucket b = [b*B, min((b+1)*B, phi_pad))
// intersected with shard r = [r*S, (r+1)*S).  Rows of 5 int64 =
// (bucket, rank, flat start, rank-local shard offset, length), bucket-major.
// bucket_elems == 0 means one bucket over the whole buffer.
int64_t orc_bucket_segments(int64_t phi_pad, int n_d, int64_t bucket_elems, int64_t* rows,
                            int64_t cap)
{
    if (n_d < 1 || phi_pad < 0 || bucket_elems < 0 || phi_pad % n_d != 0) return -1;
    const int64_t S = phi_pad / n_d;
    const int64_t B = (bucket_elems == 0) ? phi_pad : bucket_elems;
    int64_t count = 0;
    int64_t b = 0;
    for (int64_t lo = 0; lo < phi_pad; lo += B, ++b) {
        const int64_t hi = (lo + B < phi_pad) ? lo + B : phi_pad;
        for (int r = 0; r < n_d; ++r) {
            const int64_t s_lo = (int64_t)r * S, s_hi = s_lo + S;
            const int64_t a = (lo > s_lo) ? lo : s_lo;
            const int64_t e = (hi < s_hi) ? hi : s_hi;
            if (a < e) {
                if (count < cap) {
                    const int64_t row[5] = {b, r, a, a - s_lo, e - a};
                    std::memcpy(rows + 5 * count, row, sizeof(row));
                }
                ++count;
            }
        }
    }
    return count;
}

// ---- A10 accounting ([ZF] "Static Memory Allocation", eq. M_static and the
// 18-Phi variant; "ZeRO-Stage 1/2/3" eqs. M(ZeRO-1), M(ZeRO-2), M(ZeRO-3/FSDP)).
// Per-rank bytes at the padded size phi_pad with shard = phi_pad / N.
// out[15] = for stage s in (DDP, Z1, Z2, Z3): params, grads, optimizer state
// (12 values), then DDP total with fp32 gradient buffers, then 0, 0.
void orc_memory(int64_t phi_pad, int n_d, int64_t* out)
{
    const int64_t S = phi_pad / n_d;
    const int64_t rows[4][3] = {
        {2 * phi_pad, 2 * phi_pad, 12 * phi_pad},  // DDP: every state replicated
        {2 * phi_pad, 2 * phi_pad, 12 * S},        // P_os
        {2 * phi_pad, 2 * S, 12 * S},              // P_os+g
        {2 * S, 2 * S, 12 * S},                    // P_os+g+p
    };
    for (int s = 0; s < 4; ++s)
        for (int j = 0; j < 3; ++j) out[3 * s + j] = rows[s][j];
    out[12] = 2 * phi_pad + 4 * phi_pad + 12 * phi_pad;  // fp32 gradient buffers
    out[13] = 0;
    out[14] = 0;
}

// ---- A10 communication ([ZF] "Standard Ring-AllReduce Communication
// Analysis", "ZeRO-1 and ZeRO-2 Communication Volume", "ZeRO-3 and FSDP
// Communication Volume").  Elements sent (= received) per rank per step.
// One ring collective over phi_pad elements moves (N-1)/N * phi_pad = (N-1)*S.
// out[4] = DDP (scatter-reduce + all-gather), ZeRO-1, ZeRO-2, ZeRO-3
// (forward all-gather + backward all-gather + reduce-scatter).
void orc_comm(int64_t phi_pad, int n_d, int64_t* out)
{
    const int64_t S = phi_pad / n_d;
    const int64_t one = (int64_t)(n_d - 1) * S;
    out[0] = one + one;        // V_scatter + V_gather
    out[1] = one + one;        // reduce-scatter + all-gather
    out[2] = one + one;
    out[3] = one + one + one;  // forward AG + backward AG + backward RS
}

// ---- Whole sharded step over a plan (stages 1/2/3) ----
// contrib[r]: rank r's 16-bit gradient over the global flat index space
//             (sum of padded unit sizes), padding entries zero.
// bound[r]:   1 if rank r's shard is updated in this process.
// p/m/v[r]:   rank r's fp32 state, logical layout (sum of unit shards).
// shard16[r]: stage 3: rank r's 16-bit parameter shard (logical layout).
// full16:     stages 1/2: the flat 16-bit parameter buffer (phi_pad).
// k9:         orc_consts(...) for this step.
// Returns the global non-finite flag (1 = step skipped, state untouched).
// Same as orc_sharded_step, with the optional global gradient norm and clipping (R8):
// max_norm > 0 clips; *norm2_out (if not NULL) receives norm^2.
int orc_sharded_step_ex(const int64_t* sizes, int64_t n_tensors, const int64_t* unit_first,
                        int64_t n_units, int n_d, int stage, int64_t bucket_elems, int is_fp16,
                        const uint16_t* const* contrib, const int32_t* bound, float* const* p,
                        float* const* m, float* const* v, uint16_t* const* shard16,
                        uint16_t* full16, const float* k9, double max_norm, double* norm2_out)
{
    Layout L;
    if (!make_layout(sizes, n_tensors, unit_first, n_units, n_d, L)) return -1;
    if (stage != 3 && L.units.size() != 1) return -1;
    const Consts k = unpack(k9);

    // Phase 1: reduce-scatter into each bound rank's gradient shard, bucket by
    // bucket (stages 1/2) or unit by unit (stage 3); OR the non-finite flags.
    std::vector<std::vector<float>> g((size_t)n_d);
    for (int r = 0; r < n_d; ++r)
        if (bound[r]) g[(size_t)r].assign((size_t)L.shard_total, 0.0f);
    int flag = 0;
    double norm2 = 0.0;
    if (stage != 3) {
        const Unit& U = L.units[0];
        const int64_t nrows = orc_bucket_segments(U.numel_pad, n_d, bucket_elems, nullptr, 0);
        std::vector<int64_t> rows((size_t)(5 * (nrows > 0 ? nrows : 1)));
        orc_bucket_segments(U.numel_pad, n_d, bucket_elems, rows.data(), nrows);
        for (int64_t j = 0; j < nrows; ++j) {
            const int64_t r = rows[5 * j + 1], a = rows[5 * j + 2], off = rows[5 * j + 3],
                          len = rows[5 * j + 4];
            if (!bound[r]) continue;
            for (int64_t i = 0; i < len; ++i) {
                const float gi = reduce_one(n_d, contrib, a + i, is_fp16, k.inv);
                g[(size_t)r][(size_t)(off + i)] = gi;
                flag |= nonfinite(gi);
                norm2 += (double)(gi * gi);
            }
        }
    } else {
        for (const Unit& U : L.units)
            for (int r = 0; r < n_d; ++r) {
                if (!bound[r]) continue;
                for (int64_t i = 0; i < U.shard; ++i) {
                    const float gi = reduce_one(n_d, contrib, U.base + r * U.shard + i, is_fp16,
                                                k.inv);
                    g[(size_t)r][(size_t)(U.shard_base + i)] = gi;
                    flag |= nonfinite(gi);
                    norm2 += (double)(gi * gi);
                }
            }
    }

    if (norm2_out) *norm2_out = norm2;
    const float coef = max_norm > 0.0 ? clip_coef(norm2, max_norm) : 1.0f;

    // Phase 2: update each bound rank's shard and cast it into the all-gather
    // destination, or, on a skipped step, re-cast the unchanged master.
    for (int r = 0; r < n_d; ++r) {
        if (!bound[r]) continue;
        for (const Unit& U : L.units)
            for (int64_t i = 0; i < U.shard; ++i) {
                const size_t j = (size_t)(U.shard_base + i);
                const float gj = max_norm > 0.0 ? g[(size_t)r][j] * coef : g[(size_t)r][j];
                if (!flag) adamw_one(gj, p[r][j], m[r][j], v[r][j], k);
                const uint16_t h = round16(p[r][j], is_fp16);
                if (stage != 3) full16[U.base + r * U.shard + i] = h;
                else shard16[r][j] = h;
            }
    }
    return flag;
}

int orc_sharded_step(const int64_t* sizes, int64_t n_tensors, const int64_t* unit_first,
                     int64_t n_units, int n_d, int stage, int64_t bucket_elems, int is_fp16,
                     const uint16_t* const* contrib, const int32_t* bound, float* const* p,
                     float* const* m, float* const* v, uint16_t* const* shard16,
                     uint16_t* full16, const float* k9)
{
    return orc_sharded_step_ex(sizes, n_tensors, unit_first, n_units, n_d, stage, bucket_elems,
                               is_fp16, contrib, bound, p, m, v, shard16, full16, k9, 0.0,
                               nullptr);
}

float orc_clip_coef(double norm2, double max_norm) { return clip_coef(norm2, max_norm); }

// ---- FSDP-2 per-parameter sharding ([ZF] "FSDP-2: Per-Parameter Sharding via DTensor
// (fully_shard)": tensors are sharded individually along their leading dimension, Shard(0),
// without flattening).  Reading: tensor t with d0_t rows of cols_t = size_t / d0_t elements;
// chunk c_t = ceil(d0_t / N_d) rows; rank r owns rows [r c_t, min((r+1) c_t, d0_t)); every
// rank's local shard is c_t * cols_t elements (rows beyond d0_t are padding).  A unit's
// gradient buffer is its tensors concatenated without padding; rank r's local shards follow
// each other in (unit, tensor) order. ----

namespace {
struct PChunk {
    int64_t rank, unit, tensor, row0, rows, cols, c_rows, contrib_off, state_off;
};

bool pp_chunks(const int64_t* sizes, const int64_t* dim0, int64_t n_tensors, const int64_t* unit_first,
               int64_t n_units, int n_d, std::vector<PChunk>& out, std::vector<int64_t>& unit_base,
               int64_t& per_rank)
{
    std::vector<int64_t> firsts;
    if (unit_first == nullptr || n_units <= 0) firsts.push_back(0);
    else firsts.assign(unit_first, unit_first + n_units);
    if (n_d < 1 || firsts[0] != 0) return false;
    for (size_t u = 1; u < firsts.size(); ++u)
        if (firsts[u] <= firsts[u - 1] || firsts[u] > n_tensors) return false;
    for (int64_t t = 0; t < n_tensors; ++t)
        if (sizes[t] < 0 || dim0[t] < 0 || (dim0[t] == 0 && sizes[t] != 0) ||
            (dim0[t] > 0 && sizes[t] % dim0[t] != 0))
            return false;
    out.clear();
    unit_base.assign(firsts.size() + 1, 0);
    for (size_t u = 0; u < firsts.size(); ++u) {
        const int64_t end = (u + 1 < firsts.size()) ? firsts[u + 1] : n_tensors;
        int64_t numel = 0;
        for (int64_t t = firsts[u]; t < end; ++t) numel += sizes[t];
        unit_base[u + 1] = unit_base[u] + numel;
    }
    per_rank = 0;
    for (int r = 0; r < n_d; ++r) {
        int64_t state = 0;
        for (size_t u = 0; u < firsts.size(); ++u) {
            const int64_t end = (u + 1 < firsts.size()) ? firsts[u + 1] : n_tensors;
            int64_t off = 0;  // tensor offset inside the unit's gradient buffer
            for (int64_t t = firsts[u]; t < end; ++t) {
                PChunk c;
                c.rank = r;
                c.unit = (int64_t)u;
                c.tensor = t;
                c.cols = dim0[t] > 0 ? sizes[t] / dim0[t] : 0;
                c.c_rows = (dim0[t] + n_d - 1) / n_d;
                c.row0 = r * c.c_rows;
                int64_t last = c.row0 + c.c_rows;
                if (last > dim0[t]) last = dim0[t];
                c.rows = last > c.row0 ? last - c.row0 : 0;
                c.contrib_off = off + c.row0 * c.cols;
                c.state_off = state;
                out.push_back(c);
                state += c.c_rows * c.cols;
                off += sizes[t];
            }
        }
        per_rank = state;   // the same for every rank
    }
    return true;
}
}  // namespace

// Rows of 9 int64: rank, unit, tensor, first row, owned rows, cols, chunk rows, offset of the
// owned rows in the unit's gradient buffer, offset of the local shard in the rank's state.
// Order: rank, unit, tensor.  Returns the row count (-1 on invalid input).
int64_t orc_pp_chunks(const int64_t* sizes, const int64_t* dim0, int64_t n_tensors,
                      const int64_t* unit_first, int64_t n_units, int n_d, int64_t* rows, int64_t cap,
                      int64_t* per_rank_out)
{
    std::vector<PChunk> ch;
    std::vector<int64_t> ub;
    int64_t per_rank = 0;
    if (!pp_chunks(sizes, dim0, n_tensors, unit_first, n_units, n_d, ch, ub, per_rank)) return -1;
    if (per_rank_out) *per_rank_out = per_rank;
    for (size_t i = 0; i < ch.size() && (int64_t)i < cap; ++i) {
        const PChunk& c = ch[i];
        const int64_t row[9] = {c.rank, c.unit, c.tensor, c.row0, c.rows, c.cols, c.c_rows,
                                c.contrib_off, c.state_off};
        std::memcpy(rows + 9 * i, row, sizeof(row));
    }
    return (int64_t)ch.size();
}

// Whole per-parameter-sharded step.  contrib[r]: rank r's gradient over every unit's buffer
// (units concatenated, unpadded); p/m/v/shard16[r]: rank r's local shards (padded layout).
// Returns the global non-finite flag.
// The per-parameter step with the optional global gradient norm and clipping (R8, as in
// orc_sharded_step_ex): norm^2 sums fp32(g*g) in double over the bound ranks' chunks in chunk
// order; max_norm > 0 multiplies each g by clip_coef before AdamW; *norm2_out (if not NULL)
// receives norm^2.
int orc_pp_step_ex(const int64_t* sizes, const int64_t* dim0, int64_t n_tensors,
                   const int64_t* unit_first, int64_t n_units, int n_d, int is_fp16,
                   const uint16_t* const* contrib, const int32_t* bound, float* const* p,
                   float* const* m, float* const* v, uint16_t* const* shard16, const float* k9,
                   double max_norm, double* norm2_out)
{
    std::vector<PChunk> ch;
    std::vector<int64_t> ub;
    int64_t per_rank = 0;
    if (!pp_chunks(sizes, dim0, n_tensors, unit_first, n_units, n_d, ch, ub, per_rank)) return -1;
    const Consts k = unpack(k9);
    std::vector<std::vector<float>> g((size_t)n_d);
    for (int r = 0; r < n_d; ++r)
        if (bound[r]) g[(size_t)r].assign((size_t)per_rank, 0.0f);
    int flag = 0;
    double norm2 = 0.0;
    for (const PChunk& c : ch) {
        if (!bound[c.rank]) continue;
        for (int64_t i = 0; i < c.rows * c.cols; ++i) {
            const float gi = reduce_one(n_d, contrib, ub[(size_t)c.unit] + c.contrib_off + i, is_fp16,
                                        k.inv);
            g[(size_t)c.rank][(size_t)(c.state_off + i)] = gi;
            flag |= nonfinite(gi);
            norm2 += (double)(gi * gi);
        }
    }
    if (norm2_out) *norm2_out = norm2;
    const float coef = max_norm > 0.0 ? clip_coef(norm2, max_norm) : 1.0f;
    for (const PChunk& c : ch) {
        if (!bound[c.rank]) continue;
        const int r = (int)c.rank;
        for (int64_t i = 0; i < c.rows * c.cols; ++i) {
            const size_t j = (size_t)(c.state_off + i);
            const float gj = max_norm > 0.0 ? g[(size_t)r][j] * coef : g[(size_t)r][j];
            if (!flag) adamw_one(gj, p[r][j], m[r][j], v[r][j], k);
            shard16[r][j] = round16(p[r][j], is_fp16);
        }
    }
    return flag;
}

int orc_pp_step(const int64_t* sizes, const int64_t* dim0, int64_t n_tensors,
                const int64_t* unit_first, int64_t n_units, int n_d, int is_fp16,
                const uint16_t* const* contrib, const int32_t* bound, float* const* p,
                float* const* m, float* const* v, uint16_t* const* shard16, const float* k9)
{
    return orc_pp_step_ex(sizes, dim0, n_tensors, unit_first, n_units, n_d, is_fp16, contrib, bound, p, m,
                          v, shard16, k9, 0.0, nullptr);
}

// All-gather of unit `unit` into its unpadded buffer: every rank's owned rows of every tensor.
int orc_pp_gather(const int64_t* sizes, const int64_t* dim0, int64_t n_tensors,
                  const int64_t* unit_first, int64_t n_units, int n_d, int64_t unit,
                  const uint16_t* const* shard16, uint16_t* full_unit)
{
    std::vector<PChunk> ch;
    std::vector<int64_t> ub;
    int64_t per_rank = 0;
    if (!pp_chunks(sizes, dim0, n_tensors, unit_first, n_units, n_d, ch, ub, per_rank)) return -1;
    for (const PChunk& c : ch)
        if (c.unit == unit)
            for (int64_t i = 0; i < c.rows * c.cols; ++i)
                full_unit[c.contrib_off + i] = shard16[c.rank][c.state_off + i];
    return 0;
}

// ---- A8 commit/skip of the dynamic loss scale (R5): on a flagged step the
// scale backs off (not below min_scale) and the clean-step counter restarts;
// after `interval` consecutive applied steps the scale grows.  Returns the
// number of applied steps after this one (t unchanged on a skip). ----
int64_t orc_scaler_update(int flag, int64_t t, double* scale, int64_t* good, double growth,
                          double backoff, int64_t interval, double min_scale)
{
    if (flag) {
        double s = *scale * backoff;
        *scale = (s < min_scale) ? min_scale : s;
        *good = 0;
        return t;
    }
    *good += 1;
    if (interval > 0 && *good >= interval) {
        *scale = *scale * growth;
        *good = 0;
    }
    return t + 1;
}

// ---- Unsharded data parallelism, brute force: all-reduce (sum over ranks,
// r ascending, times inv) of the full buffers, then one AdamW over all n
// elements.  Returns the non-finite flag. ----
int orc_ddp_step(int64_t n, int n_d, const uint16_t* const* contrib, int is_fp16, float* p,
                 float* m, float* v, uint16_t* out16, const float* k9)
{
    const Consts k = unpack(k9);
    std::vector<float> g((size_t)n);
    int flag = 0;
    for (int64_t i = 0; i < n; ++i) {
        g[(size_t)i] = reduce_one(n_d, contrib, i, is_fp16, k.inv);
        flag |= nonfinite(g[(size_t)i]);
    }
    for (int64_t i = 0; i < n; ++i) {
        if (!flag) adamw_one(g[(size_t)i], p[i], m[i], v[i], k);
        out16[i] = round16(p[i], is_fp16);
    }
    return flag;
}

// ---- Stage 3 all-gather of one unit ([ZF] "ZeRO-3 / FSDP Layer Execution
// Lifecycle"): full[r*S_u + i] = shard16[r][shard_base_u + i], padding kept. ----
int orc_gather_unit(const int64_t* sizes, int64_t n_tensors, const int64_t* unit_first,
                    int64_t n_units, int n_d, int64_t unit, const uint16_t* const* shard16,
                    uint16_t* full_unit)
{
    Layout L;
    if (!make_layout(sizes, n_tensors, unit_first, n_units, n_d, L)) return -1;
    if (unit < 0 || unit >= (int64_t)L.units.size()) return -1;
    const Unit& U = L.units[(size_t)unit];
    for (int r = 0; r < n_d; ++r)
        for (int64_t i = 0; i < U.shard; ++i)
            full_unit[r * U.shard + i] = shard16[r][U.shard_base + i];
    return 0;
}

}  // extern "C"
