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
#include <atomic>
#include <chrono>
#include <cmath>
#include <condition_variable>
#include <cstring>
#include <functional>
#include <mutex>
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

// CLIP: the gradient is scaled by the clipping coefficient first (one fp32 multiply, as the
// GPU step does in clip mode).
template <bool FP16, bool CLIP>
void adamw_span(const CpuSpan& s, const float* k, float coef)
{
    const float b1 = k[0], omb1 = k[1], b2 = k[2], omb2 = k[3], eps = k[4], lrwd = k[5];
    const float step = k[6], bc2s = k[7];
    float* __restrict p = s.master;
    float* __restrict m = s.m;
    float* __restrict v = s.v;
    const float* __restrict g = s.grad;
    uint16_t* __restrict out = s.out16;
    for (int64_t i = 0; i < s.n; ++i) {
        const float gi = CLIP ? g[i] * coef : g[i];
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

namespace {

constexpr int64_t kPiece = 1 << 16;          // elements per unit of work of one thread

}  // namespace

// Persistent workers: start(n, fn) runs fn(0) .. fn(n - 1) on n workers and returns at once;
// wait() returns when all of them have returned.  One job at a time.
class WorkerPool {
public:
    explicit WorkerPool(int n)
    {
        for (int i = 0; i < n; ++i) threads_.emplace_back([this, i] { loop(i); });
    }
    ~WorkerPool()
    {
        {
            std::lock_guard<std::mutex> lock(mu_);
            quit_ = true;
        }
        job_cv_.notify_all();
        for (auto& t : threads_) t.join();
    }
    int size() const { return (int)threads_.size(); }
    void start(int n, std::function<void(int)> fn)
    {
        {
            std::lock_guard<std::mutex> lock(mu_);
            fn_ = std::move(fn);
            active_ = std::min(n, size());
            running_ = active_;
            ++generation_;
        }
        job_cv_.notify_all();
    }
    void wait()
    {
        std::unique_lock<std::mutex> lock(mu_);
        done_cv_.wait(lock, [this] { return running_ == 0; });
    }

private:
    void loop(int i)
    {
        uint64_t seen = 0;
        for (;;) {
            std::function<void(int)> fn;
            {
                std::unique_lock<std::mutex> lock(mu_);
                job_cv_.wait(lock, [&] { return quit_ || generation_ != seen; });
                if (quit_) return;
                seen = generation_;
                if (i >= active_) continue;
                fn = fn_;
            }
            fn(i);
            {
                std::lock_guard<std::mutex> lock(mu_);
                if (--running_ == 0) done_cv_.notify_all();
            }
        }
    }
    std::vector<std::thread> threads_;
    std::mutex mu_;
    std::condition_variable job_cv_, done_cv_;
    std::function<void(int)> fn_;
    uint64_t generation_ = 0;
    int active_ = 0, running_ = 0;
    bool quit_ = false;
};

WorkerPool* worker_pool_create(int threads) { return new WorkerPool(std::max(1, threads)); }
void worker_pool_destroy(WorkerPool* pool) { delete pool; }
int worker_pool_size(const WorkerPool* pool) { return pool ? pool->size() : 0; }

// The update of one piece: clip coefficient 1 (no clipping, or a norm within the bound) leaves
// the gradient as it is, exactly as a multiply by 1 would.
void adamw_piece(const CpuSpan& q, const float* k, int dtype16, float coef)
{
    if (coef != 1.0f) {
        if (dtype16 == ZERO_FP16) adamw_span<true, true>(q, k, coef);
        else adamw_span<false, true>(q, k, coef);
    } else if (dtype16 == ZERO_FP16) {
        adamw_span<true, false>(q, k, 1.0f);
    } else {
        adamw_span<false, false>(q, k, 1.0f);
    }
}

void cpu_adamw(WorkerPool* pool, const std::vector<CpuSpan>& spans, const float k[9], int dtype16,
               bool skipped, int threads, float coef)
{
    // Cut the spans into pieces of ~64K elements and deal them to the threads in turn.
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
    const int nt = std::max(1, std::min({threads, (int)pieces.size(), pool->size()}));
    auto work = [&](int tid) {
        for (size_t i = (size_t)tid; i < pieces.size(); i += (size_t)nt) {
            const CpuSpan& q = pieces[i];
            if (skipped) {
                if (dtype16 == ZERO_FP16) recast_span<true>(q);
                else recast_span<false>(q);
            } else {
                adamw_piece(q, k, dtype16, coef);
            }
        }
    };
    pool->start(nt, work);
    pool->wait();
}

bool cpu_adamw_overlapped(WorkerPool* pool, const std::vector<CpuSpan>& spans,
                          const std::vector<int>& group_of_span, const float k[9], int dtype16, int threads,
                          float coef, const std::function<bool(int)>& wait_group,
                          const std::function<bool(size_t, int64_t, int64_t)>& copied)
{
    // Pieces of ~64K elements in span order; the threads take them in that order (one shared
    // counter), each once its group has been released.
    struct Piece {
        size_t span;
        int64_t off, n;
        int group;
    };
    std::vector<Piece> pieces;
    for (size_t i = 0; i < spans.size(); ++i)
        for (int64_t o = 0; o < spans[i].n; o += kPiece)
            pieces.push_back(Piece{i, o, std::min(kPiece, spans[i].n - o), group_of_span[i]});
    const int64_t np = (int64_t)pieces.size();
    const int n_groups = spans.empty() ? 0 : group_of_span.back() + 1;
    std::vector<std::atomic<unsigned char>> done((size_t)np);
    for (auto& d : done) d.store(0, std::memory_order_relaxed);
    std::atomic<int64_t> next{0}, n_done{0};
    std::mutex mu;
    std::condition_variable released_cv, progress_cv;
    int released = -1;              // groups [0, released] may be updated (guarded by mu)
    bool stop = false;              // give up (guarded by mu)

    auto worker = [&](int) {
        for (;;) {
            const int64_t i = next.fetch_add(1);
            if (i >= np) return;
            const Piece& pc = pieces[(size_t)i];
            {
                std::unique_lock<std::mutex> lock(mu);
                released_cv.wait(lock, [&] { return stop || released >= pc.group; });
                if (stop) return;
            }
            CpuSpan q = spans[pc.span];
            q.master += pc.off;
            q.m += pc.off;
            q.v += pc.off;
            q.grad += pc.off;
            q.out16 += pc.off;
            q.n = pc.n;
            adamw_piece(q, k, dtype16, coef);
            done[(size_t)i].store(1, std::memory_order_release);
            n_done.fetch_add(1, std::memory_order_release);
            progress_cv.notify_one();
        }
    };
    const int nt = std::max(1, std::min({threads, (int)std::max<int64_t>(1, np), pool->size()}));
    pool->start(nt, worker);

    // Hand back the finished prefix of pieces, merged into runs of >= 1M elements per span
    // (or the span's end, or everything once `final`).
    int64_t handed = 0;             // pieces handed back
    bool ok = true;
    auto flush = [&](bool final) {
        while (ok && handed < np && done[(size_t)handed].load(std::memory_order_acquire)) {
            const size_t sp = pieces[(size_t)handed].span;
            int64_t end = handed;
            while (end < np && pieces[(size_t)end].span == sp && done[(size_t)end].load(std::memory_order_acquire))
                ++end;
            const int64_t off = pieces[(size_t)handed].off;
            const int64_t n = pieces[(size_t)end - 1].off + pieces[(size_t)end - 1].n - off;
            const bool span_done = end == np || pieces[(size_t)end].span != sp;
            if (!final && !span_done && n < (int64_t)1 << 20) return;
            ok = copied(sp, off, n);
            handed = end;
        }
    };
    auto give_up = [&]() {
        {
            std::lock_guard<std::mutex> lock(mu);
            stop = true;
        }
        released_cv.notify_all();
    };
    for (int g = 0; g < n_groups && ok; ++g) {
        if (!wait_group(g)) {
            ok = false;
            break;
        }
        {
            std::lock_guard<std::mutex> lock(mu);
            released = g;
        }
        released_cv.notify_all();
        flush(false);
    }
    while (ok && handed < np) {
        {
            std::unique_lock<std::mutex> lock(mu);
            progress_cv.wait_for(lock, std::chrono::milliseconds(1));
        }
        flush(n_done.load(std::memory_order_acquire) == np);
    }
    if (!ok) give_up();
    pool->wait();
    return ok;
}

}  // namespace zero
