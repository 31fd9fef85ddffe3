// Host-side check of the offloaded update's pipeline (zero_offload.cpp), no GPU involved:
// cpu_adamw_overlapped with groups released one by one (with random delays) must give the
// bits of cpu_adamw, hand back every 16-bit element exactly once in span order, and stop
// cleanly when a wait gives up; with a clipping coefficient, the update must equal the plain
// update of gradients scaled by that coefficient beforehand (one fp32 multiply each).  Built
// and run by tests/test_offload_host.py.
#include <chrono>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <random>
#include <thread>
#include <vector>

#include "zero_internal.h"

using zero::CpuSpan;

namespace {

struct Buffers {
    std::vector<float> p, m, v, g;
    std::vector<uint16_t> out;
};

Buffers make(int64_t n, uint32_t seed)
{
    std::mt19937 rng(seed);
    std::normal_distribution<float> nd(0.0f, 0.02f);
    Buffers b;
    b.p.resize(n);
    b.m.resize(n);
    b.v.resize(n);
    b.g.resize(n);
    b.out.assign(n, 0xFFFF);
    for (int64_t i = 0; i < n; ++i) {
        b.p[i] = nd(rng);
        b.m[i] = nd(rng) * 0.1f;
        b.v[i] = std::fabs(nd(rng)) * 0.01f;
        b.g[i] = nd(rng) * 0.5f;
    }
    return b;
}

std::vector<CpuSpan> spans_of(Buffers& b, const std::vector<int64_t>& sizes)
{
    std::vector<CpuSpan> s;
    int64_t off = 0;
    for (int64_t n : sizes) {
        s.push_back(CpuSpan{b.p.data() + off, b.m.data() + off, b.v.data() + off, b.g.data() + off,
                            b.out.data() + off, n});
        off += n;
    }
    return s;
}

int check(zero::WorkerPool* pool, const std::vector<int64_t>& sizes, const std::vector<int>& groups,
          int dtype16, int threads, int fail_at, uint32_t seed, float coef = 1.0f)
{
    int64_t n = 0;
    for (int64_t x : sizes) n += x;
    Buffers a = make(n, seed), b = make(n, seed);
    const float k[9] = {0.9f, 0.1f, 0.999f, 0.001f, 1e-8f, 1e-5f, 1e-3f, 0.0316f, 0.0f};
    zero::cpu_adamw(pool, spans_of(a, sizes), k, dtype16, false, threads, coef);
    if (coef != 1.0f) {
        // the clipped update is the plain update of the pre-scaled gradient
        Buffers c = make(n, seed);
        for (int64_t i = 0; i < n; ++i) c.g[i] = c.g[i] * coef;
        zero::cpu_adamw(pool, spans_of(c, sizes), k, dtype16, false, threads, 1.0f);
        if (std::memcmp(a.p.data(), c.p.data(), 4 * n) != 0 || std::memcmp(a.v.data(), c.v.data(), 4 * n) != 0 ||
            std::memcmp(a.out.data(), c.out.data(), 2 * n) != 0) {
            std::printf("FAIL: the clipped update differs from the update of scaled gradients\n");
            return 1;
        }
        Buffers u = make(n, seed);                     // and it does change the result
        zero::cpu_adamw(pool, spans_of(u, sizes), k, dtype16, false, threads, 1.0f);
        if (std::memcmp(a.p.data(), u.p.data(), 4 * n) == 0) {
            std::printf("FAIL: the clipping coefficient had no effect\n");
            return 1;
        }
    }
    std::vector<CpuSpan> sb = spans_of(b, sizes);
    std::mt19937 rng(seed + 1);
    int next_group = 0;
    bool order_ok = true;
    std::vector<std::pair<size_t, int64_t>> handed;   // (span, end) of the last range per call
    size_t cur_span = 0;
    int64_t cur_end = 0;
    std::vector<int64_t> covered(n, 0);
    std::vector<int64_t> base(sizes.size(), 0);
    for (size_t i = 1; i < sizes.size(); ++i) base[i] = base[i - 1] + sizes[i - 1];
    const bool ok = zero::cpu_adamw_overlapped(
        pool, sb, groups, k, dtype16, threads, coef,
        [&](int g) {
            order_ok &= g == next_group++;
            std::this_thread::sleep_for(std::chrono::microseconds(rng() % 3000));
            return g != fail_at;
        },
        [&](size_t span, int64_t off, int64_t len) {
            // ranges come in span order, each starting where the previous one ended
            if (span != cur_span) {
                order_ok &= span > cur_span && cur_end == sizes[cur_span];
                for (size_t s2 = cur_span + 1; s2 < span; ++s2) order_ok &= sizes[s2] == 0;
                cur_span = span;
                cur_end = 0;
            }
            order_ok &= off == cur_end && len > 0 && off + len <= sizes[span];
            for (int64_t i = 0; i < len; ++i) covered[base[span] + off + i] += 1;
            cur_end = off + len;
            return true;
        });
    if (fail_at >= 0) {
        if (ok) {
            std::printf("FAIL: a wait that gave up was not reported\n");
            return 1;
        }
        return order_ok ? 0 : 1;
    }
    if (!ok || !order_ok) {
        std::printf("FAIL: ok=%d order=%d\n", (int)ok, (int)order_ok);
        return 1;
    }
    for (int64_t i = 0; i < n; ++i) {
        if (covered[i] != 1) {
            std::printf("FAIL: element %lld handed back %lld times\n", (long long)i, (long long)covered[i]);
            return 1;
        }
    }
    const bool same = std::memcmp(a.p.data(), b.p.data(), 4 * n) == 0 &&
                      std::memcmp(a.m.data(), b.m.data(), 4 * n) == 0 &&
                      std::memcmp(a.v.data(), b.v.data(), 4 * n) == 0 &&
                      std::memcmp(a.out.data(), b.out.data(), 2 * n) == 0;
    if (!same) {
        std::printf("FAIL: overlapped update differs from the plain one\n");
        return 1;
    }
    return 0;
}

}  // namespace

int main()
{
    int bad = 0;
    // One pool of 12 workers for every call, as a plan keeps its pool from step to step: calls
    // with fewer threads leave workers idle, and a call that gave up is followed by others.
    zero::WorkerPool* pool = zero::worker_pool_create(12);
    // (sizes of the spans, group of each span, dtype, threads, wait that gives up)
    bad += check(pool, {5, 70000, 1, 200000, 65536, 3}, {0, 0, 0, 1, 2, 2}, ZERO_BF16, 4, -1, 1);
    bad += check(pool, {1 << 20, 1 << 20, 777777}, {0, 1, 2}, ZERO_FP16, 8, -1, 2);
    bad += check(pool, {300000, 0, 123457}, {0, 1, 1}, ZERO_BF16, 1, -1, 3);
    bad += check(pool, {3000000}, {0}, ZERO_BF16, 16, -1, 4);
    bad += check(pool, {100000, 100000, 100000, 100000}, {0, 1, 2, 3}, ZERO_FP16, 3, 2, 5);
    bad += check(pool, {100000, 100000}, {0, 1}, ZERO_BF16, 2, 0, 6);
    // a clipping coefficient, in the plain and the overlapped update alike
    bad += check(pool, {5, 70000, 1, 200000, 65536, 3}, {0, 0, 0, 1, 2, 2}, ZERO_BF16, 4, -1, 7, 0.37f);
    bad += check(pool, {1 << 20, 777777}, {0, 1}, ZERO_FP16, 8, -1, 8, 1e-3f);
    for (uint32_t r = 0; r < 20; ++r)
        bad += check(pool, {70000 + 1000 * r, 65536, 9}, {0, 1, 1}, r % 2 ? ZERO_FP16 : ZERO_BF16,
                     1 + (int)r % 12, r % 5 == 4 ? 1 : -1, 100 + r);
    zero::worker_pool_destroy(pool);
    std::printf(bad ? "FAILED %d\n" : "ok\n", bad);
    return bad != 0;
}
