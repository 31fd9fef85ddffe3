// Host side of the synthetic input generator: fills host arrays with the
// streams defined in synth_core.h.  Input preparation only; multithreaded.
#include "synth_core.h"

#include <algorithm>
#include <thread>
#include <vector>

extern "C" {

// dst[j] = value(start + j) for j in [0, n).
int syn_fill_host(uint16_t* dst, int64_t n, int64_t start, uint64_t seed, uint64_t workload,
                  uint64_t kind, uint64_t step, uint64_t rank, double sigma, int dtype,
                  int outliers, int64_t inject_index, uint32_t inject_bits, int threads)
{
    if (n < 0 || (n > 0 && dst == nullptr)) return 1;
    const syn_stream_t s = syn_make_stream(seed, workload, kind, step, rank, sigma, dtype,
                                           outliers, inject_index, inject_bits);
    int nt = threads > 0 ? threads : (int)std::max(1u, std::thread::hardware_concurrency());
    if (n < (int64_t)1 << 16) nt = 1;
    auto work = [&](int64_t b, int64_t e) {
        for (int64_t j = b; j < e; ++j) dst[j] = syn_value(&s, (uint64_t)(start + j));
    };
    if (nt == 1) { work(0, n); return 0; }
    std::vector<std::thread> pool;
    int64_t chunk = (n + nt - 1) / nt;
    for (int t = 0; t < nt; ++t) {
        int64_t b = t * chunk, e = std::min(n, b + chunk);
        if (b < e) pool.emplace_back(work, b, e);
    }
    for (auto& th : pool) th.join();
    return 0;
}

// dst[j] = value(idx[j]) for j in [0, n): values at arbitrary stream indices.
int syn_values_at(uint16_t* dst, const int64_t* idx, int64_t n, uint64_t seed, uint64_t workload,
                  uint64_t kind, uint64_t step, uint64_t rank, double sigma, int dtype,
                  int outliers, int64_t inject_index, uint32_t inject_bits)
{
    if (n < 0 || (n > 0 && (dst == nullptr || idx == nullptr))) return 1;
    const syn_stream_t s = syn_make_stream(seed, workload, kind, step, rank, sigma, dtype,
                                           outliers, inject_index, inject_bits);
    for (int64_t j = 0; j < n; ++j) dst[j] = syn_value(&s, (uint64_t)idx[j]);
    return 0;
}

// Raw splitmix64 and key derivation, exported for the generator's own tests
// and for the log-uniform tensor-size list.
uint64_t syn_hash(uint64_t x) { return syn_splitmix64(x); }
uint64_t syn_stream_key(uint64_t seed, uint64_t workload, uint64_t kind, uint64_t step,
                        uint64_t rank)
{
    return syn_key(seed, workload, kind, step, rank);
}
float syn_scale(double sigma) { return syn_scale_for_sigma(sigma); }
uint16_t syn_round_bf16(float f) { return syn_to_bf16(f); }
uint16_t syn_round_fp16(float f) { return syn_to_fp16(f); }

}  // extern "C"
