// zero_internal.h -- plan representation shared by the host planner
// (zero_plan.cpp) and the device side (zero_step.cu).  Not part of the ABI.
#pragma once

#include <cstdint>
#include <functional>
#include <string>
#include <unordered_set>
#include <vector>

#include "../../include/zero.h"

namespace zero {

// One FSDP unit's FlatParameter ("FSDP-1: FlatParameter and Module-Level
// Wrapping"): its tensors are contiguous in the global flat index space,
// followed by tail padding up to a multiple of N_d.
struct Unit {
    int64_t first;       // first tensor
    int64_t count;       // tensors in the unit
    int64_t numel;       // sum of its tensor sizes
    int64_t numel_pad;   // numel rounded up to a multiple of N_d
    int64_t shard;       // numel_pad / N_d
    int64_t base;        // global flat offset of the unit
    int64_t shard_base;  // logical offset of the unit's shard inside a rank's shard
};

// A rank's device buffers (all caller-owned).
struct Rank {
    bool bound = false;          // optimizer state bound: updated by zero_step
    bool peer = false;           // stage 3: 16-bit shard only (optimizer elsewhere)
    float* master[2] = {nullptr, nullptr};
    float* m[2] = {nullptr, nullptr};
    float* v[2] = {nullptr, nullptr};
    uint16_t* shard16 = nullptr; // stage 3
    // ZeRO-Offload: fp32 state and the gradient / 16-bit staging live in host memory
    bool offload = false;
    float* grad_host = nullptr;   // averaged fp32 gradient written by the GPU (pinned)
    uint16_t* param16_host = nullptr;   // 16-bit parameters produced by the CPU (pinned)
};

// A contiguous piece of an offloaded rank's state for the CPU update.
struct CpuSpan {
    float* master;
    float* m;
    float* v;
    const float* grad;
    uint16_t* out16;
    int64_t n;
};

// Host worker threads kept between offloaded steps (creating and joining 16 threads took
// ~0.3 ms a step on the Grace host).  Idle workers sleep on a condition variable.
class WorkerPool;
WorkerPool* worker_pool_create(int threads);
void worker_pool_destroy(WorkerPool* pool);
int worker_pool_size(const WorkerPool* pool);

// CPU AdamW (or, for a skipped step, the re-cast of the unchanged master) over the spans, on
// `threads` workers of `pool` (at most its size); k = the nine fp32 step constants, coef = the
// gradient-clipping coefficient (1: none).
void cpu_adamw(WorkerPool* pool, const std::vector<CpuSpan>& spans, const float k[9], int dtype16,
               bool skipped, int threads, float coef = 1.0f);

// The same update while the gradient is still arriving, in groups of spans (group_of_span,
// non-decreasing): on the calling thread, wait_group(g) is called for g = 0, 1, ... and
// returns once group g's gradient is in host memory (false: give up); the threads update the
// spans of every group released so far, and copied(span, offset, n) is called on the calling
// thread, in span order, for finished ranges of 16-bit parameters (false: give up).  Returns
// false if a callback gave up; every thread has stopped by then.
bool cpu_adamw_overlapped(WorkerPool* pool, const std::vector<CpuSpan>& spans,
                          const std::vector<int>& group_of_span, const float k[9], int dtype16, int threads,
                          float coef, const std::function<bool(int)>& wait_group,
                          const std::function<bool(size_t, int64_t, int64_t)>& copied);

// Elementwise work item of one launch: n elements of one rank's shard.
//   contributions: element c_off of every contribution buffer
//   state:         element s_off of the rank's master/m/v (both halves)
//   16-bit output: element o_off of `out16`
// FSDP-2 per-parameter sharding: rank `rank`'s chunk of tensor `tensor` (rows
// [row0, row0 + rows) of a tensor with `cols` elements per row; the local shard holds
// c_rows * cols elements, rows beyond the tensor being padding).
struct Chunk {
    int64_t rank, unit, tensor, row0, rows, cols, c_rows;
    int64_t contrib_off;  // offset of the owned rows in the unit's gradient buffer
    int64_t state_off;    // logical offset of the local shard in the rank's state
    int64_t phys_off;     // physical offset (16-byte phase of contrib_off)
};

struct Segment {
    int64_t n;
    int64_t c_off;
    int64_t s_off;
    int64_t o_off;
    int rank;
    uint16_t* out16;
};

// Workspace layout: 256 bytes of device-resident step state, then the bias-correction
// table, entry t (t >= 1) = (1 - beta1^t, sqrt(1 - beta2^t)) in double.
constexpr int64_t kStateBytes = 256;
constexpr int64_t kBiasCap = 1 << 16;
// then one double per block of a launch: partial sums of the gradient norm
constexpr int64_t kNormSlots = 4096;
constexpr int64_t kWorkspaceBytes = kStateBytes + 16 * (kBiasCap + 1) + 8 * kNormSlots;

}  // namespace zero

struct zero_plan {
    int n_d = 0;
    int stage = 0;
    int dtype16 = 0;
    int64_t bucket_elems = 0;           // 0 = whole buffer
    std::vector<int64_t> sizes;
    std::vector<int64_t> tensor_offset;
    std::vector<zero::Unit> units;
    int64_t phi = 0;
    int64_t phi_pad = 0;
    int64_t shard_total = 0;
    int64_t n_buckets = 0;
    // Physical state layout: phys_off[r][u] = element offset of unit u's shard in rank r's
    // state buffers; state_elems[r] = their length.
    std::vector<std::vector<int64_t>> phys_off;
    // FSDP-2 per-parameter plans (stage-3 semantics, one chunk per rank and tensor).
    bool per_param = false;
    bool offload = false;               // bound ranks keep their fp32 state in host memory
    std::vector<int64_t> dim0;
    std::vector<zero::Chunk> chunks;    // rank-major, then unit, then tensor
    std::vector<int64_t> state_elems;

    // Bindings (device pointers, caller-owned).
    std::vector<zero::Rank> ranks;
    uint16_t* full16 = nullptr;
    uint32_t* workspace = nullptr;
    int device = -1;

    // Host side of the step lifecycle (the applied-step count, the current ping-pong half
    // and the loss scale live on the device, in the workspace).
    bool in_step = false;
    bool stepped = false;               // a step has been enqueued since the plan was bound
    std::vector<char> covered;          // per bucket / unit in the open step
    std::vector<char> norm_covered;     // per bucket / unit: gradient-norm pre-pass done
    bool norm_open = false;             // a norm pre-pass of the next step has been issued
    float consts[9] = {0};              // fp32 constants that do not depend on t or the scale
    zero_hyper_t step_hyper = {};
    zero_scaler_t scaler = {1.0, 1.0, 1.0, 1.0, 0, 0};
    int scaler_dynamic = 0;
    std::vector<double> bias_host;      // the table last copied into the workspace
    int64_t bias_len = 0;
    int bias_saturates = 0;
    double bias_beta1 = -1.0, bias_beta2 = -1.0;
    std::vector<char> gathered;         // stage 3: per unit
    // Execution options (zero_set_option).
    int staging = ZERO_STAGING_AUTO;    // ZERO_STAGING_*: which step kernel zero_step launches
    int64_t wait_limit_ns = 1000000000; // bound on each barrier wait of the staged kernel
    int64_t bulk_tile = 0;              // elements per staged tile (0: chosen from N_d)
    int bulk_stages = 0;                // ring depth (0: chosen from the tile)
    int last_step_kernel = -1;          // last zero_step launch: 1 staged, 0 register loads
    int last_gather_in_step = -1;       // last zero_step_gather_next: 1 gather inside the step
                                        // launch, 0 launched on its own
    int gather_staging = ZERO_STAGING_AUTO;   // zero_gather_layer's kernel
    int gather_chunk = 0;               // elements per bulk copy of the staged gather (0: default)
    int gather_stages = 0;              // its ring entries (0: default)
    // Overlapped stage-3 schedule: CUDA events (created on first use, released by
    // zero_plan_destroy through the hook the device side installs).
    void* ov_events[5] = {nullptr, nullptr, nullptr, nullptr, nullptr};
    // ZeRO-Offload step in flight: its segments in launch order, the end (index into
    // off_segs) of each reduction group, one CUDA event per group (a pool), the event after
    // the last flag pass, and a side stream that reads the step state once that event is done.
    std::vector<zero::Segment> off_segs;
    std::vector<size_t> off_group_end;
    // ZERO_OPT_OFFLOAD_DEFER: the calls whose writing reduction waits for zero_offload_finish
    struct OffloadCall {
        std::vector<const void*> contribs;
        std::vector<zero::Segment> segs;
    };
    std::vector<OffloadCall> off_deferred;
    int offload_defer = 0;
    int unit_order = 0;                 // zero_step_units_overlapped: 0 first to last, 1 reversed
    std::vector<void*> off_events;
    void* off_flag_event = nullptr;
    void* off_side = nullptr;
    zero::WorkerPool* host_pool = nullptr;   // the host update's threads (created on first use)
    // Steps fed from host memory (zero_step_host): two caller-owned device staging areas, the
    // elements between consecutive ranks' parts of an area, the plan's two copy streams and
    // its events (created on first use: copied[2], used[2], the last copy back), the calls issued so
    // far (call k uses area k % 2), and the open step's device->host copies (repeated after a
    // skipped step's re-cast) with its byte counts.
    struct HostCopy {
        uint16_t* host;
        const uint16_t* dev;
        int64_t n;
    };
    void* host_staging[2] = {nullptr, nullptr};
    int64_t host_rank_stride = 0;
    void* host_h2d = nullptr;
    void* host_d2h = nullptr;
    void* host_events[5] = {nullptr, nullptr, nullptr, nullptr, nullptr};
    std::vector<void*> host_piece_events;   // copied / used of each piece of a split call
    int64_t host_calls = 0;
    bool host_step = false;
    int host_pipeline = 1;
    std::vector<HostCopy> host_outs;
    // host pointers already found to be pinned (cudaPointerGetAttributes costs a driver call;
    // training loops pass the same buffers every step)
    std::unordered_set<const void*> host_pinned;
    int64_t host_h2d_bytes = 0, host_d2h_bytes = 0;             // the open step
    int64_t host_h2d_last = 0, host_d2h_last = 0;               // the last finished host step
    void (*release_hook)(zero_plan*) = nullptr;
};

namespace zero {

// Thread-local last-error text (zero_last_error).
zero_status_t fail(zero_status_t code, const std::string& msg);

// The status of an exception caught at the ABI (every exported function catches all, so none
// crosses it): host memory or thread exhaustion is ZERO_ENOMEM.  Never throws.
zero_status_t exception_status(const char* where) noexcept;

// Bucket b's global flat range [lo, hi) (stages 1/2); b = -1: the whole buffer.
void bucket_range(const zero_plan* p, int64_t b, int64_t* lo, int64_t* hi);

// Work items of one zero_step call over the bound ranks.
std::vector<Segment> step_segments(const zero_plan* p, int64_t which, int cur_out);

// Work items covering every bound rank's whole shard (re-cast of a skipped step).
std::vector<Segment> shard_segments_all(const zero_plan* p);

// fp32 step constants, computed in double and rounded once:
// b1, 1-b1, b2, 1-b2, eps, lr*wd, lr/(1-b1^t), sqrt(1-b2^t), 1/(N_d*scale).
void step_constants(const zero_hyper_t& h, int64_t t, double scale, int n_d, float out[9]);

}  // namespace zero
