/*
 * synth_core.h -- seeded, counter-based synthetic input generator.
 *
 * This module produces the INPUTS of the sharded mixed-precision AdamW step
 * (initial 16-bit parameters and the per-rank 16-bit gradient contributions).
 * It holds none of the step's arithmetic: no reduction, no optimizer update,
 * no cast of updated weights.  Both the CPU oracle and the GPU harness include
 * this one header, so a value generated on the host and on the device is the
 * same bit pattern by construction (integer hashing plus one IEEE fp32
 * multiply, no contraction possible).
 *
 * Definition of element i of a stream with key K (all integer ops mod 2^64):
 *   x      = splitmix64(K + i)
 *   n      = lane0(x) + lane1(x) + lane2(x) + lane3(x) - 131070   (16-bit lanes)
 *   value  = fp32(n) * c,   c = fp32(sigma / sqrt((65536^2 - 1) / 3))
 *            (sum of four discrete uniforms: an Irwin-Hall approximation of
 *             N(0, sigma), truncated at about 3.46 sigma)
 *   if outliers are on and splitmix64(K_out + i) % 100 == 0: value *= 100.0f
 *   bits   = round-to-nearest-even of value to bf16 or fp16
 *   if i == inject_index: bits = inject_bits (a planted inf/nan)
 *
 * splitmix64 is the published mixing function of Steele, Lea and Flood,
 * "Fast splittable pseudorandom number generators" (OOPSLA 2014), with the
 * finaliser constants of Vigna's public-domain reference.
 */
#ifndef SYNTH_CORE_H
#define SYNTH_CORE_H

#include <stdint.h>
#include <math.h>

#if defined(__CUDACC__)
#define SYN_HD __host__ __device__ __forceinline__
#else
#define SYN_HD static inline
#endif

enum { SYN_BF16 = 0, SYN_FP16 = 1 };

/* stream kinds */
enum { SYN_KIND_PARAM = 1, SYN_KIND_GRAD = 2, SYN_KIND_SIZES = 3 };

SYN_HD uint64_t syn_splitmix64(uint64_t x)
{
    uint64_t z = x + 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

/* Key of one stream: (seed, workload id, kind, step, rank). */
SYN_HD uint64_t syn_key(uint64_t seed, uint64_t workload, uint64_t kind,
                        uint64_t step, uint64_t rank)
{
    uint64_t h = syn_splitmix64(seed);
    h = syn_splitmix64(h ^ (workload + 0x100ull));
    h = syn_splitmix64(h ^ (kind + 0x200ull));
    h = syn_splitmix64(h ^ (step + 0x300ull));
    h = syn_splitmix64(h ^ (rank + 0x400ull));
    return h;
}

/* Second key, for the outlier decision of the same stream. */
SYN_HD uint64_t syn_outlier_key(uint64_t key)
{
    return syn_splitmix64(key ^ 0x6F75746C69657273ull);
}

SYN_HD int32_t syn_irwin_hall(uint64_t x)
{
    int32_t s = (int32_t)(x & 0xFFFFu) + (int32_t)((x >> 16) & 0xFFFFu) +
                (int32_t)((x >> 32) & 0xFFFFu) + (int32_t)((x >> 48) & 0xFFFFu);
    return s - 131070;
}

SYN_HD uint32_t syn_f32_bits(float f)
{
    union { float f; uint32_t u; } c;
    c.f = f;
    return c.u;
}

/* Generator-side rounding of an fp32 draw to bf16 (nearest, ties to even). */
SYN_HD uint16_t syn_to_bf16(float f)
{
    uint32_t u = syn_f32_bits(f);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u)
        return (uint16_t)((u >> 16) | 0x0040u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* Generator-side rounding of an fp32 draw to IEEE binary16 (nearest, ties to even). */
SYN_HD uint16_t syn_to_fp16(float f)
{
    uint32_t u = syn_f32_bits(f);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    uint32_t a = u & 0x7FFFFFFFu;
    if (a > 0x7F800000u) return (uint16_t)(sign | 0x7E00u);          /* nan */
    if (a >= 0x477FF000u) return (uint16_t)(sign | 0x7C00u);         /* >= 65520 -> inf */
    if (a >= 0x38800000u) {                                           /* normal half */
        uint32_t r = a - (112u << 23);
        r += 0x0FFFu + ((r >> 13) & 1u);
        return (uint16_t)(sign | (r >> 13));
    }
    /* subnormal half (or zero): units of 2^-24 */
    uint32_t e = a >> 23;
    if (e < 101u) return sign;                                        /* < 2^-25 -> 0 */
    uint32_t m = (a & 0x7FFFFFu) | 0x800000u;
    uint32_t sh = 126u - e;                                           /* 14 .. 25 */
    uint32_t q = m >> sh;
    uint32_t rem = m & ((1u << sh) - 1u);
    uint32_t half = 1u << (sh - 1u);
    if (rem > half || (rem == half && (q & 1u))) q += 1u;
    return (uint16_t)(sign | q);
}

/* fp32 scale of the Irwin-Hall integer, computed in double on the host.
 * sqrt is an IEEE-754 basic operation (correctly rounded on every platform). */
static inline float syn_scale_for_sigma(double sigma)
{
    /* std of the sum of four uniforms on {0..65535} is sqrt((65536^2-1)/3) */
    return (float)(sigma / sqrt((65536.0 * 65536.0 - 1.0) / 3.0));
}

typedef struct {
    uint64_t key;           /* syn_key(...) of the stream */
    uint64_t out_key;       /* syn_outlier_key(key) */
    int64_t inject_index;   /* -1: none */
    float scale;            /* syn_scale_for_sigma(sigma) */
    int32_t dtype;          /* SYN_BF16 or SYN_FP16 */
    int32_t outliers;       /* 1: 1 % of entries x100 */
    uint32_t inject_bits;   /* 16-bit pattern planted at inject_index */
} syn_stream_t;

static inline syn_stream_t syn_make_stream(uint64_t seed, uint64_t workload, uint64_t kind,
                                           uint64_t step, uint64_t rank, double sigma,
                                           int dtype, int outliers, int64_t inject_index,
                                           uint32_t inject_bits)
{
    syn_stream_t s;
    s.key = syn_key(seed, workload, kind, step, rank);
    s.out_key = syn_outlier_key(s.key);
    s.inject_index = inject_index;
    s.scale = syn_scale_for_sigma(sigma);
    s.dtype = dtype;
    s.outliers = outliers;
    s.inject_bits = inject_bits;
    return s;
}

/* Element i (absolute stream index) of a stream. */
SYN_HD uint16_t syn_value(const syn_stream_t* s, uint64_t i)
{
    if ((int64_t)i == s->inject_index) return (uint16_t)s->inject_bits;
    float v = (float)syn_irwin_hall(syn_splitmix64(s->key + i)) * s->scale;
    if (s->outliers && (syn_splitmix64(s->out_key + i) % 100ull) == 0ull) v = v * 100.0f;
    return s->dtype == SYN_FP16 ? syn_to_fp16(v) : syn_to_bf16(v);
}

#endif /* SYNTH_CORE_H */
