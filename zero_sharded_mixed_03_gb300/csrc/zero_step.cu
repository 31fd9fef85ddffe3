// zero_step.cu -- host side of the sharded mixed-precision AdamW step for GB300 (sm_103a):
// kernel choice and launch geometry, the C ABI of include/zero.h (bind, step, finish,
// gathers, norm, offload, options, state) and the no-allocation entry point.  The kernels
// are in zero_kernels.cuh.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <memory>
#include <mutex>
#include <unordered_map>

#include <cuda.h>

#include "zero_kernels.cuh"

namespace zero {
namespace {

// ------------------------------------------------------------------ host helpers

inline bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p % a) == 0; }

// Elements before the first 16-byte boundary of a 16-bit stream starting at p.
inline int head16(const void* p) { return (int)(((16 - ((uintptr_t)p % 16)) % 16) / 2); }

int device_sms(int dev)
{
    static std::mutex mu;
    static int cache[64] = {0};
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 0 || dev >= 64) return 0;
    if (cache[dev] == 0) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev] = sms;
    }
    return cache[dev];
}

// Resident blocks per SM of one kernel, queried once per kernel.  Kernels of one signature
// share this template's statics, so the cache is keyed by the kernel's address.
template <typename K>
int blocks_per_sm(K kernel)
{
    static std::mutex mu;
    static std::unordered_map<const void*, int> cache;
    const void* key = reinterpret_cast<const void*>(kernel);
    std::lock_guard<std::mutex> lock(mu);
    const auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, 0) != cudaSuccess)
        per_sm = 1;
    per_sm = std::max(per_sm, 1);
    cache.emplace(key, per_sm);
    return per_sm;
}

template <typename K>
int grid_for(K kernel, int dev, int64_t work)
{
    const int64_t cap = (int64_t)device_sms(dev) * blocks_per_sm(kernel);
    const int64_t need = std::max<int64_t>(1, (work + kThreads - 1) / kThreads);
    return (int)std::max<int64_t>(1, std::min(cap, need));
}

zero_status_t cuda_fail(cudaError_t e, const char* what)
{
    return fail(ZERO_ECUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

DevState* dev_state(const zero_plan* p) { return reinterpret_cast<DevState*>(p->workspace); }
double* norm_slots(const zero_plan* p)
{
    return reinterpret_cast<double*>(reinterpret_cast<char*>(p->workspace) + kStateBytes +
                                      16 * (kBiasCap + 1));
}
const double* bias_table(const zero_plan* p)
{
    return reinterpret_cast<const double*>(reinterpret_cast<const char*>(p->workspace) + kStateBytes);
}

// Fill one launch's KSeg list from plan segments [b, e), deciding the vector path.
// Returns true when every stream of every segment shares one 16-byte phase.
template <typename PT>
bool build_step_params(const zero_plan* p, const std::vector<Segment>& segs, size_t b, size_t e,
                       const void* const* contribs, PT& P)
{
    bool vec_ok = true;
    P.n_seg = (int)(e - b);
    for (size_t i = b; i < e; ++i) {
        const Segment& sg = segs[i];
        const Rank& R = p->ranks[(size_t)sg.rank];
        KSeg& K = P.seg[i - b];
        for (int h = 0; h < 2; ++h) {
            K.p[h] = R.master[h] + sg.s_off;
            K.m[h] = R.m[h] + sg.s_off;
            K.v[h] = R.v[h] + sg.s_off;
        }
        K.out16 = sg.out16 + sg.o_off;
        K.c_off = sg.c_off;
        K.n = sg.n;
        const int hd = head16(K.out16);
        const int64_t hh = std::min<int64_t>(hd, sg.n);
        // a segment without an 8-element body is all head and tail (scalar): no phase to match
        if (sg.n - hh >= 8) {
            if (contribs)
                for (int r = 0; r < p->n_d; ++r)
                    vec_ok &= head16((const uint16_t*)contribs[r] + sg.c_off) == hd;
            for (int h = 0; h < 2; ++h)
                vec_ok &= aligned(K.p[h] + hh, 16) && aligned(K.m[h] + hh, 16) && aligned(K.v[h] + hh, 16);
        }
        K.head = (int32_t)hh;
        K.nvec = (sg.n - hh) / 8;
        K.tail = (int32_t)(sg.n - hh - 8 * K.nvec);
    }
    return vec_ok;
}

template <typename PT>
void finalize_vectors(PT& P, bool vec)
{
    int64_t acc = 0;
    for (int i = 0; i < P.n_seg; ++i) {
        KSeg& K = P.seg[i];
        if (!vec) {
            K.head = 0;
            K.tail = 0;
            K.nvec = K.n;
        }
        K.vbeg = acc;
        acc += K.nvec;
    }
    P.total_vec = acc;
}

template <typename K, typename PT>
void launch_grid(K kernel, int dev, int64_t work, const PT& P, cudaStream_t st)
{
    int grid = grid_for(kernel, dev, work);
    if (P.partials) grid = (int)std::min<int64_t>(grid, kNormSlots);
    kernel<<<grid, kThreads, 0, st>>>(P);
}

// Register loads keep NB contribution slices in flight per batch: 4, or 16 from N_d = 41 on,
// where the rank loop otherwise serialises on load latency (GB300, ragged ZeRO-2 step: N_d =
// 48 / 64 / 96 / 128 at 0.96 / 0.96 / 0.95 / 0.93 of the copy bandwidth against 0.93 / 0.91 /
// 0.91 / 0.89 with 4; at N_d = 33-40 batches of 16 cost occupancy and lost 2-12 %, below 32
// up to 25 %).
template <int DT, int MODE, typename PT>
void launch_fused_mode(int dev, const PT& P, bool vec, int64_t work, cudaStream_t st)
{
    if (!vec) launch_grid(fused_step_kernel<DT, 1, 1, MODE, PT>, dev, work, P, st);
    else if (P.n_d >= kWideRankBatchFrom) launch_grid(fused_step_kernel<DT, kWideRankBatch, 8, MODE, PT>, dev, work, P, st);
    else launch_grid(fused_step_kernel<DT, kRankBatch, 8, MODE, PT>, dev, work, P, st);
}

// Geometry of the bulk-staged kernel (tile == 0: register-load kernel).  automatic: launch
// it only where its residency pays off (bulk_pays_off), else the register-load kernel.
struct BulkCfg {
    int tile = 0;
    int stages = 0;
    uint64_t wait_ns = 0;
    bool automatic = false;
};

// Units of `unit` elements over the vector bodies of a launch's segments.
template <typename SegT>
int64_t units_over(const SegT* seg, int n_seg, int64_t unit)
{
    int64_t n = 0;
    for (int i = 0; i < n_seg; ++i) n += (8 * seg[i].nvec + unit - 1) / unit;
    return n;
}

// Where the staged kernel beats register loads, from sweeps of N_d = 1 .. 128 on GB300 (ragged
// ZeRO-2 step): with exactly two blocks per SM (8 consumer warps, 75-110 KB rings) and tiles of
// 512 elements or more it won almost everywhere (by up to 7 %; lost 1-2 % at N_d = 10-11);
// with three blocks of 512-element tiles (N_d 22-31) it won by 2-6 %; three blocks of
// 1,024-2,048-element tiles (N_d 1-3, 12) lost 7-14 %, four blocks were a wash, and tiles below
// 512 elements (N_d >= 48: bulk copies of <= 512 B per rank) lost 20-50 % whatever the blocks.
bool bulk_pays_off(int blocks_per_sm, int tile)
{
    return (blocks_per_sm == 2 && tile >= 512) || (blocks_per_sm == 3 && tile == 512);
}

// Dynamic shared memory of one block: alignment slack, barriers, the ring.
int64_t bulk_smem_bytes(int64_t tile, int64_t stages, int64_t n_d)
{
    return 128 + kBulkBarrierBytes + stages * tile * (2 * n_d + 12);
}

// Default geometry: two buffers of the largest tile, a multiple of 512 elements (whole passes
// of the consumer threads over 4-element quads) up to 2048, within 53.5 KB per buffer; for
// N_d >= 48 the largest power of two within that.  Two blocks then share an SM with rings of
// up to 107 KB.  Measured on GB300: two blocks of four consumer warps with 40-53 KB tiles
// beat deeper rings and more, smaller blocks (a 45 KB cap left N_d = 6, 10, 11, 17-20 with
// three or four blocks per SM, 3-7 % slower than this geometry).
int auto_bulk_tile(int n_d)
{
    const int64_t per_elem = 2 * n_d + 12, cap = 54784;
    int64_t tile = std::min<int64_t>(2048, cap / per_elem / 512 * 512);
    if (tile >= 512) return (int)tile;
    // N_d = 47-50: 512-element tiles (1 KB per contribution copy) up to 56 KB per buffer still
    // leave two blocks per SM (0.999 of the copy bandwidth at N_d = 48, against 0.974 with
    // 256-element tiles and 0.946 with register loads)
    if (512 * per_elem <= 57344) return 512;
    tile = 256;
    while (tile > 8 && tile * per_elem > cap) tile /= 2;
    return (int)tile;
}

int auto_bulk_stages(int /*tile*/, int /*n_d*/) { return 2; }

BulkCfg bulk_config(const zero_plan* p)
{
    BulkCfg b;
    if (p->staging == ZERO_STAGING_REGISTER_LOADS) return b;
    b.tile = p->bulk_tile > 0 ? (int)p->bulk_tile : auto_bulk_tile(p->n_d);
    b.stages = p->bulk_stages > 0 ? p->bulk_stages : auto_bulk_stages(b.tile, p->n_d);
    b.wait_ns = (uint64_t)p->wait_limit_ns;
    b.automatic = p->staging == ZERO_STAGING_AUTO;
    return b;
}

int optin_smem(int dev)
{
    static std::mutex mu;
    static int cache[64] = {0};
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 0 || dev >= 64) return 0;
    if (cache[dev] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return 0;
        cache[dev] = v;
    }
    return cache[dev];
}

// Resident blocks per SM of `Kernel` launched with `Threads` threads and `smem` bytes of
// dynamic shared memory (a ring of staged buffers).  The kernel's dynamic shared-memory limit
// only ever grows (so a launch of another plan on another thread never finds it below its own
// ring), and the residency is queried once per device and ring size; both are host calls,
// cached per instantiation.
template <auto Kernel, int Threads>
cudaError_t residency(int dev, int64_t smem, int* per_sm)
{
    static std::mutex mu;
    static int64_t limit_set[64] = {0};
    static std::unordered_map<int64_t, int> per_sm_of[64];
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (limit_set[dev] < smem) {
        const cudaError_t e =
            cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        limit_set[dev] = smem;
    }
    const auto it = per_sm_of[dev].find(smem);
    if (it != per_sm_of[dev].end()) {
        *per_sm = it->second;
        return cudaSuccess;
    }
    int n = 0;
    const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, Kernel, Threads, (size_t)smem);
    if (e != cudaSuccess) return e;
    *per_sm = std::max(n, 1);
    per_sm_of[dev].emplace(smem, *per_sm);
    return cudaSuccess;
}

template <int DT, int MODE, typename PT>
cudaError_t bulk_residency(int dev, int64_t smem, int* per_sm)
{
    return residency<bulk_step_kernel<DT, MODE, PT>, kBulkThreads>(dev, smem, per_sm);
}

// Launch the bulk-staged kernel with `per_sm` resident blocks per SM.
template <int DT, int MODE, typename PT>
cudaError_t launch_bulk_mode(int dev, PT& P, const BulkCfg& B, int per_sm, cudaStream_t st)
{
    auto kernel = bulk_step_kernel<DT, MODE, PT>;
    const int64_t smem = bulk_smem_bytes(B.tile, B.stages, P.n_d);
    int64_t slots = (int64_t)device_sms(dev) * per_sm;
    if (P.partials) slots = std::min<int64_t>(slots, kNormSlots);
    P.tile = B.tile;
    P.stages = B.stages;
    P.wait_ns = B.wait_ns;
    const int64_t tiles = units_over(P.seg, P.n_seg, P.tile);
    P.n_tiles = tiles;
    const int64_t scalar_blocks = ((int64_t)P.n_seg * kScalarSlots + 32 * kBulkConsumers - 1) /
                                  (32 * kBulkConsumers);
    int64_t want = std::max(tiles, scalar_blocks);
    if constexpr (HasGather<PT>::value) {
        const int64_t gscalar = ((int64_t)P.g_n * kScalarSlots + 32 * kBulkConsumers - 1) /
                                (32 * kBulkConsumers);
        want = std::max(want, std::max<int64_t>(P.g_chunks, gscalar));
    }
    int64_t grid = std::min<int64_t>(slots, want);
    grid = std::max<int64_t>(1, grid);
    kernel<<<(int)grid, kBulkThreads, (size_t)smem, st>>>(P);
    return cudaGetLastError();
}

// *used (when given): 1 if the bulk-staged kernel was launched, 0 for register loads.
template <int DT, typename PT>
cudaError_t launch_fused(int dev, PT& P, bool vec, cudaStream_t st, int mode = kPlain,
                         const BulkCfg* bulk = nullptr, int* used = nullptr)
{
    if (used) *used = 0;
    finalize_vectors(P, vec);
    // Norm-report steps keep the register-load kernel: the per-element norm accumulation is a
    // serial chain per thread, which the bulk kernel's few consumer warps do not hide
    // (ragged N_d = 7 workload on GB300: 367 us against 353 us).
    if (bulk && bulk->tile > 0 && vec && P.st && mode != kNormAcc) {
        const int64_t smem = bulk_smem_bytes(bulk->tile, bulk->stages, P.n_d);
        int per_sm = 0;
        const cudaError_t e = mode == kClip ? bulk_residency<DT, kClip, PT>(dev, smem, &per_sm)
                                            : bulk_residency<DT, kPlain, PT>(dev, smem, &per_sm);
        if (e != cudaSuccess) return e;
        if (!bulk->automatic || bulk_pays_off(per_sm, bulk->tile)) {
            if (used) *used = 1;
            if (mode == kClip) return launch_bulk_mode<DT, kClip>(dev, P, *bulk, per_sm, st);
            return launch_bulk_mode<DT, kPlain>(dev, P, *bulk, per_sm, st);
        }
    }
    const int64_t work = std::max<int64_t>(P.total_vec, (int64_t)P.n_seg * kScalarSlots);
    if (mode == kNormAcc) launch_fused_mode<DT, kNormAcc>(dev, P, vec, work, st);
    else if (mode == kClip) launch_fused_mode<DT, kClip>(dev, P, vec, work, st);
    else launch_fused_mode<DT, kPlain>(dev, P, vec, work, st);
    return cudaGetLastError();
}

template <int DT, typename PT>
cudaError_t launch_norm(int dev, PT& P, bool vec, cudaStream_t st)
{
    finalize_vectors(P, vec);
    const int64_t work = std::max<int64_t>(P.total_vec, (int64_t)P.n_seg * kScalarSlots);
    if (!vec) launch_grid(grad_norm_kernel<DT, 1, 1, PT>, dev, work, P, st);
    else if (P.n_d >= kWideNormBatchFrom) launch_grid(grad_norm_kernel<DT, kWideRankBatch, 8, PT>, dev, work, P, st);
    else launch_grid(grad_norm_kernel<DT, kNormRankBatch, 8, PT>, dev, work, P, st);
    return cudaGetLastError();
}

template <int DT, bool STORE, typename PT>
cudaError_t launch_reduce_to_host(int dev, PT& P, bool vec, cudaStream_t st)
{
    finalize_vectors(P, vec);
    const int64_t work = std::max<int64_t>(2 * P.total_vec, (int64_t)P.n_seg * kScalarSlots);
    if (!vec) launch_grid(reduce_to_host_kernel<DT, 1, 1, PT, STORE>, dev, work, P, st);
    else if (P.n_d >= kWideNormBatchFrom) launch_grid(reduce_to_host_kernel<DT, kWideRankBatch, 8, PT, STORE>, dev, work, P, st);
    else launch_grid(reduce_to_host_kernel<DT, kRankBatch, 8, PT, STORE>, dev, work, P, st);
    return cudaGetLastError();
}

// One block per SM at most: the launch does nothing on a clean step (the usual case) except
// read the flag and take the commit ticket, so its cost is the block count; a skipped step's
// re-cast (6 bytes per element) still streams at a good fraction of HBM bandwidth.
template <int DT, typename PT>
cudaError_t launch_recast(int dev, PT& P, bool vec, cudaStream_t st)
{
    finalize_vectors(P, vec);
    const int64_t work = std::max<int64_t>(P.total_vec, (int64_t)P.n_seg * kScalarSlots);
    const int64_t need = std::max<int64_t>(1, (work + kThreads - 1) / kThreads);
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(device_sms(dev), need));
    if (vec) recast_kernel<DT, 8, PT><<<grid, kThreads, 0, st>>>(P);
    else recast_kernel<DT, 1, PT><<<grid, kThreads, 0, st>>>(P);
    return cudaGetLastError();
}

// One copy of a gather: a rank's 16-bit shard (or chunk) into the unit's full buffer.
struct Copy {
    const uint16_t* src;
    uint16_t* dst;
    int64_t n;
};

// The gather kernel of a launch: bulk-staged (with its ring) or register loads.
struct GatherCfg {
    bool bulk = false;
    int chunk = 0;
    int stages = 0;
    uint32_t* err = nullptr;
    uint64_t wait_ns = 0;
};

int64_t gather_smem_bytes(int64_t chunk, int64_t stages) { return 128 + kGatherBarrierBytes + stages * chunk * 2; }

template <typename CP>
cudaError_t launch_bulk_gather(int dev, CP& P, const GatherCfg& g, cudaStream_t s)
{
    const int64_t smem = gather_smem_bytes(g.chunk, g.stages);
    int per_sm = 0;
    const cudaError_t e = residency<bulk_gather_kernel<CP>, kGatherThreads>(dev, smem, &per_sm);
    if (e != cudaSuccess) return e;
    const int64_t slots = (int64_t)device_sms(dev) * per_sm;
    P.err = g.err;
    P.wait_ns = g.wait_ns;
    P.chunk = g.chunk;
    P.stages = g.stages;
    int64_t chunks = 0;
    for (int i = 0; i < P.n_seg; ++i) {
        P.seg[i].cbeg = chunks;
        chunks += (8 * P.seg[i].nvec + P.chunk - 1) / P.chunk;
    }
    P.n_chunks = chunks;
    const int64_t scalar_blocks = ((int64_t)P.n_seg * kScalarSlots + kGatherThreads - 2) / (kGatherThreads - 1);
    int64_t grid = std::min<int64_t>(slots, std::max(chunks, scalar_blocks));
    grid = std::max<int64_t>(1, grid);
    bulk_gather_kernel<CP><<<(int)grid, kGatherThreads, (size_t)smem, s>>>(P);
    return cudaGetLastError();
}

// Launch the gather over `copies`, CP::seg's capacity at a time.
template <typename CP>
cudaError_t launch_gathers(int dev, const std::vector<Copy>& copies, CP& P, const GatherCfg& g,
                           cudaStream_t s)
{
    const size_t cap = sizeof(P.seg) / sizeof(P.seg[0]);
    for (size_t c0 = 0; c0 < copies.size(); c0 += cap) {
        std::memset(&P, 0, sizeof(P));
        bool vec = true;
        const size_t c1 = std::min(copies.size(), c0 + cap);
        P.n_seg = (int)(c1 - c0);
        for (size_t i = c0; i < c1; ++i) {
            CopySeg& K = P.seg[i - c0];
            K.src = copies[i].src;
            K.dst = copies[i].dst;
            K.n = copies[i].n;
            const int h = head16(K.dst);
            K.head = (int32_t)std::min<int64_t>(h, K.n);
            if (K.n - K.head >= 8) vec &= head16(K.src) == h;   // a copy with a vector body
            K.nvec = (K.n - K.head) / 8;
            K.tail = (int32_t)(K.n - K.head - 8 * K.nvec);
        }
        int64_t acc = 0;
        for (int i = 0; i < P.n_seg; ++i) {
            CopySeg& K = P.seg[i];
            if (!vec) {
                K.head = K.tail = 0;
                K.nvec = K.n;
            }
            K.vbeg = acc;
            acc += K.nvec;
        }
        P.total_vec = acc;
        const int64_t work = std::max<int64_t>(acc, (int64_t)P.n_seg * kScalarSlots);
        cudaError_t e;
        if (vec && g.bulk && g.err) {
            e = launch_bulk_gather(dev, P, g, s);
        } else {
            if (vec) gather_kernel<8, CP><<<grid_for(gather_kernel<8, CP>, dev, work), kThreads, 0, s>>>(P);
            else gather_kernel<1, CP><<<grid_for(gather_kernel<1, CP>, dev, work), kThreads, 0, s>>>(P);
            e = cudaGetLastError();
        }
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// Copy list of unit `unit`'s all-gather into full_unit16: (source in a rank's 16-bit shard,
// destination in the unit, length).
std::vector<Copy> gather_copies(const zero_plan* p, int64_t unit, void* full_unit16)
{
    std::vector<Copy> copies;
    const Unit& U = p->units[(size_t)unit];
    if (p->per_param) {
        for (const Chunk& c : p->chunks)
            if (c.unit == unit && c.rows > 0)
                copies.push_back({p->ranks[(size_t)c.rank].shard16 + c.phys_off,
                                  (uint16_t*)full_unit16 + c.contrib_off, c.rows * c.cols});
    } else if (U.shard > 0) {
        for (int r = 0; r < p->n_d; ++r)
            copies.push_back({p->ranks[(size_t)r].shard16 + p->phys_off[(size_t)r][(size_t)unit],
                              (uint16_t*)full_unit16 + r * U.shard, U.shard});
    }
    return copies;
}

// Fill the gather part of a step launch's parameters from `copies` into `dst`.  False when the
// copies do not fit the parameter block or the compact record (32-bit offsets and lengths), or
// when a copy's source and destination are not in one 16-byte phase.
template <typename GPT>
bool build_gather_params(const std::vector<Copy>& copies, uint16_t* dst, GPT& P)
{
    const size_t cap = sizeof(P.gc) / sizeof(P.gc[0]);
    if (copies.empty() || copies.size() > cap) return false;
    P.g_dst = dst;
    P.g_n = (int32_t)copies.size();
    for (size_t i = 0; i < copies.size(); ++i) {
        const Copy& c = copies[i];
        const int64_t off = c.dst - dst;
        if (off < 0 || off > (int64_t)UINT32_MAX || c.n < 0 || c.n > (int64_t)UINT32_MAX) return false;
        const int64_t hd = std::min<int64_t>(head16(c.dst), c.n);
        if (c.n - hd >= 8 && head16(c.src) != head16(c.dst)) return false;
        P.gc[i].src = c.src;
        P.gc[i].dst_off = (uint32_t)off;
        P.gc[i].n = (uint32_t)c.n;
        P.gc[i].cbeg = 0;
        P.gc[i].pad = 0;
    }
    return true;
}

// One step launch (the bulk-staged kernel) that also streams the gather in P's copy list,
// chunked to one ring buffer (at most 32K elements).  *fused = false and nothing launched when
// the staged kernel is not the one this launch would use (automatic choice, norm-report step,
// streams of different phases): the caller then launches the step and the gather separately.
template <int DT, typename GPT>
cudaError_t launch_step_gather(int dev, GPT& P, bool vec, cudaStream_t st, int mode,
                               const BulkCfg& bulk, bool* fused)
{
    *fused = false;
    if (!(bulk.tile > 0 && vec && P.st && mode != kNormAcc)) return cudaSuccess;
    finalize_vectors(P, vec);
    const int64_t smem = bulk_smem_bytes(bulk.tile, bulk.stages, P.n_d);
    int per_sm = 0;
    const cudaError_t e = mode == kClip ? bulk_residency<DT, kClip, GPT>(dev, smem, &per_sm)
                                        : bulk_residency<DT, kPlain, GPT>(dev, smem, &per_sm);
    if (e != cudaSuccess) return e;
    if (bulk.automatic && !bulk_pays_off(per_sm, bulk.tile)) return cudaSuccess;
    const int64_t stage_bytes = (int64_t)bulk.tile * (2 * P.n_d + 12);
    P.g_chunk = (int32_t)std::min<int64_t>(32768, stage_bytes / 16 * 8);
    int64_t chunks = 0;
    for (int i = 0; i < P.g_n; ++i) {
        const uint16_t* d = P.g_dst + P.gc[i].dst_off;
        const int64_t n = P.gc[i].n;
        const int64_t body = (n - std::min<int64_t>(head16(d), n)) / 8 * 8;
        if (chunks > (int64_t)UINT32_MAX) return cudaSuccess;
        P.gc[i].cbeg = (uint32_t)chunks;
        chunks += (body + P.g_chunk - 1) / P.g_chunk;
    }
    P.g_chunks = chunks;
    *fused = true;
    return mode == kClip ? launch_bulk_mode<DT, kClip>(dev, P, bulk, per_sm, st)
                         : launch_bulk_mode<DT, kPlain>(dev, P, bulk, per_sm, st);
}

zero_status_t set_device(const zero_plan* p)
{
    int cur = -1;
    cudaError_t e = cudaGetDevice(&cur);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (p->device >= 0 && cur != p->device) {
        e = cudaSetDevice(p->device);
        if (e != cudaSuccess) return cuda_fail(e, "cudaSetDevice");
    }
    return ZERO_OK;
}

// (Re)build the bias-correction table for (beta1, beta2) and copy it into the workspace.
// Entries run until 1 - beta^t rounds to 1 for both betas (then the table saturates) or
// until kBiasCap entries; beyond a non-saturated table the kernel computes the powers itself.
zero_status_t upload_bias_table(zero_plan* p, double beta1, double beta2, cudaStream_t s)
{
    std::vector<double>& tab = p->bias_host;
    tab.assign(2, 0.0);
    int64_t len = 0;
    bool sat = false;
    for (int64_t t = 1; t <= kBiasCap; ++t) {
        const double bc1 = 1.0 - std::pow(beta1, (double)t);
        const double bc2 = 1.0 - std::pow(beta2, (double)t);
        tab.push_back(bc1);
        tab.push_back(std::sqrt(bc2));
        len = t;
        if (bc1 == 1.0 && bc2 == 1.0) {
            sat = true;
            break;
        }
    }
    const cudaError_t e = cudaMemcpyAsync(reinterpret_cast<char*>(p->workspace) + kStateBytes,
                                          tab.data(), tab.size() * sizeof(double),
                                          cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e, "uploading the bias-correction table");
    p->bias_len = len;
    p->bias_saturates = sat ? 1 : 0;
    p->bias_beta1 = beta1;
    p->bias_beta2 = beta2;
    return ZERO_OK;
}

zero_status_t read_state(zero_plan* p, cudaStream_t s, zero_step_result_t* out)
{
    DevState host;
    cudaError_t e = cudaMemcpyAsync(&host, p->workspace, sizeof(host), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "reading the step state");
    std::memset(out, 0, sizeof(*out));
    out->skipped = (int32_t)host.last_skipped;
    out->current = (int32_t)host.cur;
    out->t = host.t;
    out->scale = host.scale;
    out->good_steps = host.good;
    out->skipped_total = host.skipped;
    out->finished = host.finished;
    out->grad_norm = host.last_norm_valid ? std::sqrt(host.last_norm2) : -1.0;
    if (host.error) {
        e = cudaMemsetAsync(&dev_state(p)->error, 0, sizeof(host.error), s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) return cuda_fail(e, "clearing the error word");
        return fail(ZERO_ETIMEOUT, (host.error & 2u)
                                       ? "a barrier wait and the drain of the bulk-staged step ran out; "
                                         "the steps finished since the last read were discarded"
                                       : "a barrier wait of the bulk-staged step ran out; the steps "
                                         "finished since the last read were discarded");
    }
    return ZERO_OK;
}

// Arguments shared by zero_step and zero_grad_norm.
zero_status_t check_call(const zero_plan_t* p, const void* const* grad_contribs,
                         int64_t n_contribs, int64_t which, const char* fn)
{
    const std::string f(fn);
    if (!p || !grad_contribs) return fail(ZERO_EINVAL, f + ": NULL argument");
    if (n_contribs != p->n_d) return fail(ZERO_EINVAL, f + ": need one contribution per rank");
    if (!p->workspace) return fail(ZERO_ESTATE, f + ": no rank bound");
    bool any = false;
    for (const Rank& R : p->ranks) any |= R.bound;
    if (!any) return fail(ZERO_ESTATE, f + ": no rank bound");
    for (int64_t r = 0; r < n_contribs; ++r) {
        if (!grad_contribs[r]) return fail(ZERO_EINVAL, f + ": NULL contribution");
        if (!aligned(grad_contribs[r], 2))
            return fail(ZERO_EALIGN, f + ": contribution not 2-byte aligned");
    }
    if (p->stage == 3) {
        if (which < 0 || which >= (int64_t)p->units.size())
            return fail(ZERO_EINVAL, f + ": unit out of range");
    } else if (which < -1 || which >= p->n_buckets) {
        return fail(ZERO_EINVAL, f + ": bucket out of range");
    }
    return ZERO_OK;
}

// Fill and launch one chunk of segments [b, e) of a zero_step / zero_grad_norm call.
// Offload work items: the kernel writes the averaged gradient at grad_host + s_off.
template <typename PT>
bool build_offload_params(const zero_plan* p, const std::vector<Segment>& segs, size_t b, size_t e,
                          const void* const* contribs, PT& P)
{
    bool vec_ok = true;
    P.n_seg = (int)(e - b);
    for (size_t i = b; i < e; ++i) {
        const Segment& sg = segs[i];
        const Rank& R = p->ranks[(size_t)sg.rank];
        KSeg& K = P.seg[i - b];
        std::memset(&K, 0, sizeof(K));
        K.p[0] = R.grad_host + sg.s_off;
        K.c_off = sg.c_off;
        K.n = sg.n;
        const int hd = head16((const uint16_t*)contribs[0] + sg.c_off);
        for (int r = 1; r < p->n_d; ++r)
            vec_ok &= head16((const uint16_t*)contribs[r] + sg.c_off) == hd;
        const int64_t hh = std::min<int64_t>(hd, sg.n);
        vec_ok &= aligned(K.p[0] + hh, 16);
        K.head = (int32_t)hh;
        K.nvec = (sg.n - hh) / 8;
        K.tail = (int32_t)(sg.n - hh - 8 * K.nvec);
    }
    return vec_ok;
}

template <typename PT>
void fill_call_params(const zero_plan* p, const void* const* grad_contribs, PT& P)
{
    std::memset(&P, 0, sizeof(P));
    for (int r = 0; r < p->n_d; ++r) P.c[r] = (const uint16_t*)grad_contribs[r];
    std::memcpy(P.k, p->consts, sizeof(P.k));
    P.lr = p->step_hyper.lr;
    P.beta1 = p->step_hyper.beta1;
    P.beta2 = p->step_hyper.beta2;
    P.bias = bias_table(p);
    P.bias_len = p->bias_len;
    P.bias_saturates = p->bias_saturates;
    P.n_d = p->n_d;
    P.st = dev_state(p);
    P.flag = &dev_state(p)->flag;
    P.partials = norm_slots(p);
    P.max_norm = 0.0;
}

// ZeRO-Offload: elements per reduction group (an event after each; the host starts updating
// a group once its gradient has landed): 4M elements, 16 MB of fp32 gradient.
constexpr int64_t kOffloadGroupElems = 1 << 22;

// The CUDA objects and host threads a plan creates on first use, released by
// zero_plan_destroy.
void release_plan_resources(zero_plan* q)
{
    if (q->host_pool) {
        worker_pool_destroy(q->host_pool);
        q->host_pool = nullptr;
    }
    for (void*& ev : q->ov_events)
        if (ev) {
            cudaEventDestroy((cudaEvent_t)ev);
            ev = nullptr;
        }
    for (void*& ev : q->off_events)
        if (ev) {
            cudaEventDestroy((cudaEvent_t)ev);
            ev = nullptr;
        }
    if (q->off_flag_event) {
        cudaEventDestroy((cudaEvent_t)q->off_flag_event);
        q->off_flag_event = nullptr;
    }
    if (q->off_side) {
        cudaStreamDestroy((cudaStream_t)q->off_side);
        q->off_side = nullptr;
    }
    for (void*& ev : q->host_events)
        if (ev) {
            cudaEventDestroy((cudaEvent_t)ev);
            ev = nullptr;
        }
    for (void* ev : q->host_piece_events) cudaEventDestroy((cudaEvent_t)ev);
    q->host_piece_events.clear();
    for (void** st : {&q->host_h2d, &q->host_d2h})
        if (*st) {
            cudaStreamDestroy((cudaStream_t)*st);
            *st = nullptr;
        }
}

// Create the event in *slot unless it exists: no timing, and a host thread that waits for it
// sleeps instead of spinning (the offload update's threads need the cores).
cudaError_t offload_event(zero_plan* p, void** slot)
{
    if (*slot) return cudaSuccess;
    cudaEvent_t ev;
    const cudaError_t e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming | cudaEventBlockingSync);
    if (e != cudaSuccess) return e;
    *slot = ev;
    p->release_hook = release_plan_resources;
    return cudaSuccess;
}

// Everything zero_step checks before it enqueues anything (shared with zero_step_host).
// The hyperparameters every step call accepts.
zero_status_t check_hyper(const zero_hyper_t* hyper, const char* fn)
{
    if (!(hyper->beta1 >= 0.0 && hyper->beta1 < 1.0) || !(hyper->beta2 >= 0.0 && hyper->beta2 < 1.0) ||
        !std::isfinite(hyper->lr) || !std::isfinite(hyper->eps) || !std::isfinite(hyper->weight_decay) ||
        !(hyper->max_grad_norm >= 0.0) || !std::isfinite(hyper->max_grad_norm))
        return fail(ZERO_EINVAL, std::string(fn) + ": betas must lie in [0, 1); lr, eps, wd, max_grad_norm finite");
    return ZERO_OK;
}

zero_status_t check_step(const zero_plan* p, const void* const* grad_contribs, int64_t n_contribs,
                         int64_t which, const zero_hyper_t* hyper, const char* fn)
{
    const std::string f(fn);
    if (!hyper) return fail(ZERO_EINVAL, f + ": NULL argument");
    if (p && p->offload) return fail(ZERO_ESTATE, f + ": offloaded plan (zero_offload_step)");
    zero_status_t cst = check_call(p, grad_contribs, n_contribs, which, fn);
    if (cst != ZERO_OK) return cst;
    cst = check_hyper(hyper, fn);
    if (cst != ZERO_OK) return cst;
    if (hyper->max_grad_norm > 0.0)
        for (int64_t b = 0; b < p->n_buckets; ++b)
            if (!p->norm_covered[(size_t)b])
                return fail(ZERO_ESTATE, f + ": clipping needs zero_grad_norm over every bucket/unit first");
    if (p->in_step && std::memcmp(&p->step_hyper, hyper, sizeof(*hyper)) != 0)
        return fail(ZERO_EINVAL, f + ": hyperparameters changed inside a step");
    if (which == -1) {
        if (p->in_step) return fail(ZERO_ESTATE, f + ": bucket -1 must be the only call of a step");
    } else if (p->covered[(size_t)which]) {
        return fail(ZERO_ESTATE, f + ": bucket/unit already stepped in this step");
    }
    return ZERO_OK;
}

// The gather kernel zero_gather_layer launches for the plan (bulk-staged unless disabled or
// without a workspace, whose error word it needs).
GatherCfg gather_cfg(const zero_plan* p)
{
    GatherCfg g;
    g.bulk = p->gather_staging != ZERO_STAGING_REGISTER_LOADS;
    g.chunk = p->gather_chunk > 0 ? p->gather_chunk : kGatherDefaultChunk;
    g.stages = p->gather_stages > 0 ? p->gather_stages : kGatherDefaultStages;
    g.err = p->workspace ? &dev_state(p)->error : nullptr;   // no workspace: register loads
    g.wait_ns = (uint64_t)p->wait_limit_ns;
    return g;
}

// The gather launches of a copy list (32 copies a launch, or 256 with the wide block).
cudaError_t launch_gather_list(const zero_plan* p, const std::vector<Copy>& copies, cudaStream_t s)
{
    const GatherCfg g = gather_cfg(p);
    if (copies.size() > (size_t)kMaxSegs) {
        CopyParamsWide P;
        return launch_gathers(p->device, copies, P, g, s);
    }
    CopyParams P;
    return launch_gathers(p->device, copies, P, g, s);
}

// The launches of one checked zero_step call (device contribution pointers).  With `gather`
// (a copy list into gather_dst) the call's last launch also streams that all-gather when the
// staged kernel runs it and the list fits the parameter block; otherwise the gather follows
// as its own launch.  *gather_fused (when given) tells which.
zero_status_t enqueue_step(zero_plan* p, const void* const* grad_contribs, int64_t which,
                           const zero_hyper_t* hyper, cudaStream_t s,
                           const std::vector<Copy>* gather = nullptr, uint16_t* gather_dst = nullptr,
                           bool* gather_fused = nullptr, const std::vector<Segment>* only = nullptr,
                           bool mark = true)
{
    zero_status_t st = set_device(p);
    if (st != ZERO_OK) return st;
    if (!p->in_step) {
        if (p->bias_len == 0 || p->bias_beta1 != hyper->beta1 || p->bias_beta2 != hyper->beta2) {
            st = upload_bias_table(p, hyper->beta1, hyper->beta2, s);
            if (st != ZERO_OK) return st;
        }
        // t, the loss scale and the current half are read on the device; the constants that
        // do not depend on them are rounded here once.
        step_constants(*hyper, 1, 1.0, p->n_d, p->consts);
        p->step_hyper = *hyper;
    }
    // clip: the norm is complete on the device; report: accumulate it in this pass
    int mode = kPlain;
    if (hyper->max_grad_norm > 0.0) mode = kClip;
    else if ((hyper->flags & ZERO_REPORT_GRAD_NORM) && !p->norm_open) mode = kNormAcc;
    // only: a part of the call's work items (a host-buffer call split into pieces); mark = false
    // leaves the call open for its remaining pieces
    const std::vector<Segment> segs = only ? *only : step_segments(p, which, 0);
    const BulkCfg bulk = bulk_config(p);
    bool pending = gather && !gather->empty();
    if (gather_fused) *gather_fused = false;
    // the last launch of the call with the gather in its parameters, if that form applies
    auto try_fused = [&](auto& GP, size_t b, size_t e) -> cudaError_t {
        fill_call_params(p, grad_contribs, GP);
        GP.max_norm = mode == kClip ? hyper->max_grad_norm : 0.0;
        const bool vec = build_step_params(p, segs, b, e, grad_contribs, GP);
        if (!build_gather_params(*gather, gather_dst, GP)) return cudaSuccess;
        bool fused = false;
        const cudaError_t err = p->dtype16 == ZERO_BF16
                                    ? launch_step_gather<ZERO_BF16>(p->device, GP, vec, s, mode, bulk, &fused)
                                    : launch_step_gather<ZERO_FP16>(p->device, GP, vec, s, mode, bulk, &fused);
        if (fused) {
            pending = false;
            p->last_step_kernel = 1;
            if (gather_fused) *gather_fused = true;
        }
        return err;
    };
    auto run = [&](auto& P, size_t cap) -> cudaError_t {
        for (size_t b = 0; b < segs.size(); b += cap) {
            const size_t e = std::min(segs.size(), b + cap);
            if (pending && e == segs.size()) {
                const size_t n = std::max(e - b, gather->size());
                cudaError_t err = cudaSuccess;
                if (n <= (size_t)kMaxSegs) {
                    StepGatherParams GP;
                    err = try_fused(GP, b, e);
                } else if (n <= (size_t)kWideSegs) {
                    std::unique_ptr<StepGatherParamsWide> GP(new StepGatherParamsWide);
                    err = try_fused(*GP, b, e);
                }
                if (err != cudaSuccess) return err;
                if (!pending) continue;          // launched with the gather inside
            }
            fill_call_params(p, grad_contribs, P);
            P.max_norm = mode == kClip ? hyper->max_grad_norm : 0.0;
            const bool vec = build_step_params(p, segs, b, e, grad_contribs, P);
            int used = 0;
            const cudaError_t err = p->dtype16 == ZERO_BF16
                                        ? launch_fused<ZERO_BF16>(p->device, P, vec, s, mode, &bulk, &used)
                                        : launch_fused<ZERO_FP16>(p->device, P, vec, s, mode, &bulk, &used);
            p->last_step_kernel = used;
            if (err != cudaSuccess) return err;
        }
        return cudaSuccess;
    };
    cudaError_t lerr;
    if (segs.size() > (size_t)kMaxSegs) {
        std::unique_ptr<StepParamsWide> P(new StepParamsWide);
        lerr = run(*P, kWideSegs);
    } else {
        StepParams P;
        lerr = run(P, kMaxSegs);
    }
    if (lerr == cudaSuccess && pending) lerr = launch_gather_list(p, *gather, s);
    if (lerr != cudaSuccess) return cuda_fail(lerr, "fused step launch");
    if (!mark) return ZERO_OK;
    p->in_step = true;
    if (which == -1) std::fill(p->covered.begin(), p->covered.end(), 1);
    else p->covered[(size_t)which] = 1;
    return ZERO_OK;
}

// Steps fed from host memory: the plan's two copy streams and five events (copied[2],
// used[2], the last device->host copy), created on first use and released with the plan.
cudaError_t host_resources(zero_plan* p)
{
    if (p->host_h2d) return cudaSuccess;
    cudaStream_t st[2] = {nullptr, nullptr};
    cudaEvent_t ev[5] = {nullptr, nullptr, nullptr, nullptr, nullptr};
    cudaError_t e = cudaSuccess;
    for (int i = 0; i < 2 && e == cudaSuccess; ++i) e = cudaStreamCreateWithFlags(&st[i], cudaStreamNonBlocking);
    for (int i = 0; i < 5 && e == cudaSuccess; ++i) e = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming);
    if (e != cudaSuccess) {
        for (cudaEvent_t x : ev)
            if (x) cudaEventDestroy(x);
        for (cudaStream_t x : st)
            if (x) cudaStreamDestroy(x);
        return e;
    }
    p->host_h2d = st[0];
    p->host_d2h = st[1];
    for (int i = 0; i < 5; ++i) p->host_events[i] = ev[i];
    p->release_hook = release_plan_resources;
    return cudaSuccess;
}

bool pinned_host(const void* q)
{
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, q) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    return at.type == cudaMemoryTypeHost;
}

// pinned_host with the plan's cache of pointers already checked (bounded: cleared when full).
// A stale entry (a pinned buffer freed and the address reused by pageable memory) would only
// make that call's copies synchronous with the host; the data copied is the same.
bool pinned_host_cached(zero_plan* p, const void* q)
{
    if (p->host_pinned.count(q)) return true;
    if (!pinned_host(q)) return false;
    if (p->host_pinned.size() >= 4096) p->host_pinned.clear();
    p->host_pinned.insert(q);
    return true;
}

// A host-buffer call that is the step's only call has no neighbour to overlap with; it is cut
// into pieces of its range instead (at least kHostPieceElems elements each, at most
// kHostMaxPieces), so that a piece's step and copy back run while the next piece is copied in.
// (GB300, the 58M-element ragged ZeRO-2 step over 7 ranks: 4.39 ms a step with pieces of at
// least 2^24 elements (3), 4.48 ms with 2^23 (6), 5.0-5.2 ms with 2^22-2^21, 4.8 ms with two.)
constexpr int64_t kHostPieceElems = 1 << 24;
constexpr int kHostMaxPieces = 8;

// The work items of `segs` that fall in [lo, hi) of the call's range, cut at its ends.
std::vector<Segment> segments_in(const std::vector<Segment>& segs, int64_t lo, int64_t hi)
{
    std::vector<Segment> out;
    for (const Segment& sg : segs) {
        const int64_t a = std::max(lo, sg.c_off), e = std::min(hi, sg.c_off + sg.n);
        if (a >= e) continue;
        Segment t = sg;
        const int64_t d = a - sg.c_off;
        t.n = e - a;
        t.c_off = a;
        t.s_off = sg.s_off + d;
        t.o_off = sg.o_off + d;
        out.push_back(t);
    }
    return out;
}

// [lo, hi) element ranges of a call's range that its work items read from every contribution,
// merged where they touch or overlap.
std::vector<std::pair<int64_t, int64_t>> read_runs(const std::vector<Segment>& segs)
{
    std::vector<std::pair<int64_t, int64_t>> r;
    for (const Segment& sg : segs)
        if (sg.n > 0) r.emplace_back(sg.c_off, sg.c_off + sg.n);
    std::sort(r.begin(), r.end());
    std::vector<std::pair<int64_t, int64_t>> out;
    for (const auto& x : r) {
        if (!out.empty() && x.first <= out.back().second) out.back().second = std::max(out.back().second, x.second);
        else out.push_back(x);
    }
    return out;
}

// ZeRO-Offload: reduce segs[b0, e0) of one call (store: the averaged gradient into the
// bound ranks' pinned host buffers; else: the non-finite flag alone), `cap` items a launch.
template <typename PT>
cudaError_t offload_launches(zero_plan* p, const void* const* contribs, const std::vector<Segment>& segs,
                             PT& P, size_t cap, size_t b0, size_t e0, bool store, cudaStream_t s)
{
    for (size_t b = b0; b < e0; b += cap) {
        const size_t e = std::min(e0, b + cap);
        fill_call_params(p, contribs, P);
        const bool vec = build_offload_params(p, segs, b, e, contribs, P);
        cudaError_t err;
        if (p->dtype16 == ZERO_BF16)
            err = store ? launch_reduce_to_host<ZERO_BF16, true>(p->device, P, vec, s)
                        : launch_reduce_to_host<ZERO_BF16, false>(p->device, P, vec, s);
        else
            err = store ? launch_reduce_to_host<ZERO_FP16, true>(p->device, P, vec, s)
                        : launch_reduce_to_host<ZERO_FP16, false>(p->device, P, vec, s);
        if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
}

template <typename F>
cudaError_t with_offload_params(const std::vector<Segment>& segs, F&& f)
{
    if (segs.size() > (size_t)kMaxSegs) {
        std::unique_ptr<StepParamsWide> P(new StepParamsWide);
        return f(*P, (size_t)kWideSegs);
    }
    StepParams P;
    return f(P, (size_t)kMaxSegs);
}

// The flag-only pass over a call (so that, after the step's last call, the host knows the skip
// decision early), then an event the finish waits for.
cudaError_t offload_flag_pass(zero_plan* p, const void* const* contribs, const std::vector<Segment>& segs,
                              cudaStream_t s)
{
    cudaError_t err = with_offload_params(segs, [&](auto& P, size_t cap) {
        return offload_launches(p, contribs, segs, P, cap, 0, segs.size(), false, s);
    });
    if (err == cudaSuccess) err = offload_event(p, &p->off_flag_event);
    if (err == cudaSuccess) err = cudaEventRecord((cudaEvent_t)p->off_flag_event, s);
    return err;
}

// The writing reduction of a call in groups of segments of at least kOffloadGroupElems
// elements, an event after each (the host updates a group as soon as its gradient has
// landed).  first: index in off_segs of the call's first segment.
cudaError_t offload_reduce_groups(zero_plan* p, const void* const* contribs, const std::vector<Segment>& segs,
                                  size_t first, cudaStream_t s)
{
    return with_offload_params(segs, [&](auto& P, size_t cap) {
        cudaError_t err = cudaSuccess;
        size_t b = 0;
        while (err == cudaSuccess && b < segs.size()) {
            size_t e = b;
            int64_t n = 0;
            while (e < segs.size() && n < kOffloadGroupElems) n += segs[e++].n;
            err = offload_launches(p, contribs, segs, P, cap, b, e, true, s);
            const size_t g = p->off_group_end.size();
            if (g >= p->off_events.size()) p->off_events.push_back(nullptr);
            if (err == cudaSuccess) err = offload_event(p, &p->off_events[g]);
            if (err == cudaSuccess) err = cudaEventRecord((cudaEvent_t)p->off_events[g], s);
            p->off_group_end.push_back(first + e);
            b = e;
        }
        return err;
    });
}

// Re-cast + commit of the open step (zero_step_finish without its checks on host calls).
zero_status_t finish_step(zero_plan_t* p, void* stream, zero_step_result_t* out);

}  // namespace
}  // namespace zero

using namespace zero;

extern "C" {

zero_status_t zero_bind(zero_plan_t* p, int rank, float* const master[2], float* const m[2],
                        float* const v[2], void* shard16, void* full16, void* workspace)
try {
    if (!p || !master || !m || !v) return fail(ZERO_EINVAL, "zero_bind: NULL argument");
    if (rank < 0 || rank >= p->n_d) return fail(ZERO_EINVAL, "zero_bind: bad rank");
    if (p->in_step || p->stepped) return fail(ZERO_ESTATE, "zero_bind: bind every rank before the first step");
    if (p->offload) return fail(ZERO_ESTATE, "zero_bind: this plan offloads its ranks (zero_bind_offload)");
    float* bufs[6] = {master[0], master[1], m[0], m[1], v[0], v[1]};
    const int64_t elems = p->state_elems[(size_t)rank];
    if (elems > 0 && (master[0] == master[1] || m[0] == m[1] || v[0] == v[1]))
        return fail(ZERO_EINVAL, "zero_bind: the two halves of a ping-pong pair must differ");
    for (float* b : bufs) {
        if (elems > 0 && !b) return fail(ZERO_EINVAL, "zero_bind: NULL state buffer");
        if (!aligned(b, 4)) return fail(ZERO_EALIGN, "zero_bind: fp32 state not 4-byte aligned");
    }
    if (p->stage == 3) {
        if (elems > 0 && !shard16) return fail(ZERO_EINVAL, "zero_bind: stage 3 needs shard16");
        if (!aligned(shard16, 2)) return fail(ZERO_EALIGN, "zero_bind: shard16 not 2-byte aligned");
    } else {
        if (!full16 && !p->full16 && p->phi_pad > 0)
            return fail(ZERO_EINVAL, "zero_bind: stages 1/2 need the flat 16-bit buffer");
        if (full16 && p->full16 && full16 != p->full16)
            return fail(ZERO_EINVAL, "zero_bind: full16 differs from an earlier bind");
        if (!aligned(full16, 2)) return fail(ZERO_EALIGN, "zero_bind: full16 not 2-byte aligned");
    }
    if (!workspace && !p->workspace) return fail(ZERO_EINVAL, "zero_bind: workspace is NULL");
    if (workspace && p->workspace && workspace != p->workspace)
        return fail(ZERO_EINVAL, "zero_bind: workspace differs from an earlier bind");
    if (!aligned(workspace, 16)) return fail(ZERO_EALIGN, "zero_bind: workspace not 16-byte aligned");

    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "zero_bind: cudaGetDevice");
    if (p->device >= 0 && p->device != dev)
        return fail(ZERO_EINVAL, "zero_bind: buffers of one plan must live on one device");
    if (workspace && !p->workspace) {
        DevState init;
        std::memset(&init, 0, sizeof(init));
        init.scale = 1.0;
        e = cudaMemcpy(workspace, &init, sizeof(init), cudaMemcpyHostToDevice);
        if (e == cudaSuccess) e = cudaDeviceSynchronize();
        if (e != cudaSuccess) return cuda_fail(e, "zero_bind: initialising the workspace");
        p->workspace = (uint32_t*)workspace;
    }
    p->device = dev;
    if (full16) p->full16 = (uint16_t*)full16;
    Rank& R = p->ranks[(size_t)rank];
    R.bound = true;
    R.peer = false;
    for (int h = 0; h < 2; ++h) {
        R.master[h] = master[h];
        R.m[h] = m[h];
        R.v[h] = v[h];
    }
    R.shard16 = (uint16_t*)shard16;
    return ZERO_OK;
}
catch (...) {
    return exception_status("zero_bind");
}

zero_status_t zero_bind_peer(zero_plan_t* p, int rank, const void* shard16)
try {
    if (!p) return fail(ZERO_EINVAL, "zero_bind_peer: NULL plan");
    if (p->stage != 3) return fail(ZERO_EINVAL, "zero_bind_peer: stage 3 only");
    if (rank < 0 || rank >= p->n_d) return fail(ZERO_EINVAL, "zero_bind_peer: bad rank");
    if (!shard16 && p->state_elems[(size_t)rank] > 0)
        return fail(ZERO_EINVAL, "zero_bind_peer: NULL shard16");
    if (!aligned(shard16, 2)) return fail(ZERO_EALIGN, "zero_bind_peer: shard16 not 2-byte aligned");
    Rank& R = p->ranks[(size_t)rank];
    if (R.bound) return fail(ZERO_ESTATE, "zero_bind_peer: rank already bound with state");
    R.peer = true;
    R.shard16 = (uint16_t*)shard16;
    return ZERO_OK;
}
catch (...) {
    return exception_status("zero_bind_peer");
}

zero_status_t zero_set_scaler(zero_plan_t* p, const zero_scaler_t* cfg, void* stream)
try {
    if (!p) return fail(ZERO_EINVAL, "zero_set_scaler: NULL plan");
    if (!p->workspace) return fail(ZERO_ESTATE, "zero_set_scaler: bind a rank first");
    if (p->in_step) return fail(ZERO_ESTATE, "zero_set_scaler: a step is open");
    double scale = 1.0;
    int64_t good = 0;
    if (cfg) {
        if (!(cfg->scale > 0.0) || !std::isfinite(cfg->scale) || !(cfg->backoff_factor > 0.0) ||
            !(cfg->growth_factor > 0.0) || !(cfg->min_scale > 0.0) || cfg->good_steps < 0)
            return fail(ZERO_EINVAL, "zero_set_scaler: bad scaler settings");
        scale = cfg->scale;
        good = cfg->good_steps;
        p->scaler = *cfg;
    }
    p->scaler_dynamic = cfg ? 1 : 0;
    zero_status_t st = set_device(p);
    if (st != ZERO_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    DevState* d = dev_state(p);
    cudaError_t e = cudaMemcpyAsync(&d->scale, &scale, sizeof(scale), cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(&d->good, &good, sizeof(good), cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "zero_set_scaler: writing the loss scale");
    return ZERO_OK;
}
catch (...) {
    return exception_status("zero_set_scaler");
}

zero_status_t zero_set_option(zero_plan_t* p, int option, int64_t value)
try {
    if (!p) return fail(ZERO_EINVAL, "zero_set_option: NULL plan");
    if (p->in_step) return fail(ZERO_ESTATE, "zero_set_option: a step is open");
    int64_t tile = p->bulk_tile, stages = p->bulk_stages;
    switch (option) {
    case ZERO_OPT_STAGING:
        if (value != ZERO_STAGING_REGISTER_LOADS && value != ZERO_STAGING_BULK &&
            value != ZERO_STAGING_AUTO)
            return fail(ZERO_EINVAL, "zero_set_option: staging must be 0, 1 or 2");
        p->staging = (int)value;
        return ZERO_OK;
    case ZERO_OPT_WAIT_LIMIT_NS:
        if (value < 0) return fail(ZERO_EINVAL, "zero_set_option: negative wait limit");
        p->wait_limit_ns = value;
        return ZERO_OK;
    case ZERO_OPT_BULK_TILE:
        if (value != 0 && (value < 8 || value > kBulkMaxTile || value % 8 != 0))
            return fail(ZERO_EINVAL, "zero_set_option: tile must be 0 or a multiple of 8 in [8, 8192]");
        tile = value;
        break;
    case ZERO_OPT_BULK_STAGES:
        if (value != 0 && (value < 2 || value > kBulkMaxStages))
            return fail(ZERO_EINVAL, "zero_set_option: stages must be 0 or in [2, 16]");
        stages = value;
        break;
    case ZERO_OPT_HOST_PIPELINE:
        if (value != 0 && value != 1) return fail(ZERO_EINVAL, "zero_set_option: host pipeline must be 0 or 1");
        p->host_pipeline = (int)value;
        return ZERO_OK;
    case ZERO_OPT_OFFLOAD_DEFER:
        if (value != 0 && value != 1) return fail(ZERO_EINVAL, "zero_set_option: offload defer must be 0 or 1");
        p->offload_defer = (int)value;
        return ZERO_OK;
    case ZERO_OPT_UNIT_ORDER:
        if (value != 0 && value != 1) return fail(ZERO_EINVAL, "zero_set_option: unit order must be 0 or 1");
        p->unit_order = (int)value;
        return ZERO_OK;
    case ZERO_OPT_HOST_H2D_BYTES:
    case ZERO_OPT_HOST_D2H_BYTES:
    case ZERO_OPT_LAST_GATHER_IN_STEP:
        return fail(ZERO_EINVAL, "zero_set_option: read-only option");
    case ZERO_OPT_GATHER_STAGING:
        if (value != ZERO_STAGING_REGISTER_LOADS && value != ZERO_STAGING_BULK &&
            value != ZERO_STAGING_AUTO)
            return fail(ZERO_EINVAL, "zero_set_option: gather staging must be 0, 1 or 2");
        p->gather_staging = (int)value;
        return ZERO_OK;
    case ZERO_OPT_GATHER_CHUNK:
    case ZERO_OPT_GATHER_STAGES: {
        const bool is_chunk = option == ZERO_OPT_GATHER_CHUNK;
        if (is_chunk && value != 0 && (value < 8 || value > kGatherMaxChunk || value % 8 != 0))
            return fail(ZERO_EINVAL, "zero_set_option: gather chunk must be 0 or a multiple of 8 in [8, 32768]");
        if (!is_chunk && value != 0 && (value < kGatherStoresPending + 1 || value > kGatherMaxStages))
            return fail(ZERO_EINVAL, "zero_set_option: gather stages must be 0 or in [3, 32]");
        const int64_t c = is_chunk ? value : p->gather_chunk;
        const int64_t n = is_chunk ? p->gather_stages : value;
        int64_t gcap = 227 * 1024;
        if (p->device >= 0 && optin_smem(p->device) > 0) gcap = std::min<int64_t>(gcap, optin_smem(p->device));
        if (gather_smem_bytes(c > 0 ? c : kGatherDefaultChunk, n > 0 ? n : kGatherDefaultStages) > gcap)
            return fail(ZERO_ERANGE, "zero_set_option: the gather ring does not fit one block's shared memory");
        (is_chunk ? p->gather_chunk : p->gather_stages) = (int)value;
        return ZERO_OK;
    }
    default:
        return fail(ZERO_EINVAL, "zero_set_option: unknown option");
    }
    const int64_t t = tile > 0 ? tile : auto_bulk_tile(p->n_d);
    const int64_t n = stages > 0 ? stages : auto_bulk_stages((int)t, p->n_d);
    // 227 KB: the opt-in shared memory of one block on this architecture (the device's own
    // figure is checked as well once a device is known)
    int64_t cap = 227 * 1024;
    if (p->device >= 0 && optin_smem(p->device) > 0) cap = std::min<int64_t>(cap, optin_smem(p->device));
    if (bulk_smem_bytes(t, n, p->n_d) > cap)
        return fail(ZERO_ERANGE, "zero_set_option: the staging ring does not fit one block's shared memory");
    p->bulk_tile = tile;
    p->bulk_stages = (int)stages;
    return ZERO_OK;
}
catch (...) {
    return exception_status("zero_set_option");
}

zero_status_t zero_get_option(const zero_plan_t* p, int option, int64_t* value)
try {
    if (!p || !value) return fail(ZERO_EINVAL, "zero_get_option: NULL argument");
    switch (option) {
    case ZERO_OPT_STAGING: *value = p->staging; return ZERO_OK;
    case ZERO_OPT_WAIT_LIMIT_NS: *value = p->wait_limit_ns; return ZERO_OK;
    case ZERO_OPT_BULK_TILE: *value = p->bulk_tile > 0 ? p->bulk_tile : auto_bulk_tile(p->n_d); return ZERO_OK;
    case ZERO_OPT_BULK_STAGES:
        *value = p->bulk_stages > 0 ? p->bulk_stages
                                    : auto_bulk_stages((int)(p->bulk_tile > 0 ? p->bulk_tile : auto_bulk_tile(p->n_d)), p->n_d);
        return ZERO_OK;
    case ZERO_OPT_LAST_STEP_KERNEL: *value = p->last_step_kernel; return ZERO_OK;
    case ZERO_OPT_GATHER_STAGING: *value = p->gather_staging; return ZERO_OK;
    case ZERO_OPT_GATHER_CHUNK: *value = p->gather_chunk > 0 ? p->gather_chunk : kGatherDefaultChunk; return ZERO_OK;
    case ZERO_OPT_GATHER_STAGES: *value = p->gather_stages > 0 ? p->gather_stages : kGatherDefaultStages; return ZERO_OK;
    case ZERO_OPT_HOST_PIPELINE: *value = p->host_pipeline; return ZERO_OK;
    case ZERO_OPT_OFFLOAD_DEFER: *value = p->offload_defer; return ZERO_OK;
    case ZERO_OPT_HOST_H2D_BYTES: *value = p->host_h2d_last; return ZERO_OK;
    case ZERO_OPT_HOST_D2H_BYTES: *value = p->host_d2h_last; return ZERO_OK;
    case ZERO_OPT_UNIT_ORDER: *value = p->unit_order; return ZERO_OK;
    case ZERO_OPT_LAST_GATHER_IN_STEP: *value = p->last_gather_in_step; return ZERO_OK;
    default: return fail(ZERO_EINVAL, "zero_get_option: unknown option");
    }
}
catch (...) {
    return exception_status("zero_get_option");
}

}  // extern "C"

namespace zero {
namespace {

// The checks of a gradient-norm pre-pass call (fn: the entry point's name).
zero_status_t check_norm_call(const zero_plan* p, const void* const* grad_contribs, int64_t n_contribs,
                              int64_t which, const char* fn)
{
    const std::string f(fn);
    zero_status_t st = check_call(p, grad_contribs, n_contribs, which, fn);
    if (st != ZERO_OK) return st;
    if (p->in_step) return fail(ZERO_ESTATE, f + ": the norm must precede every zero_step of a step");
    if (which == -1) {
        if (p->norm_open) return fail(ZERO_ESTATE, f + ": bucket -1 must be the only call");
    } else if (p->norm_covered[(size_t)which]) {
        return fail(ZERO_ESTATE, f + ": bucket/unit already included");
    }
    return ZERO_OK;
}

// Launch the norm pre-pass of bucket/unit `which` over device contributions on `s`.
zero_status_t enqueue_norm(zero_plan* p, const void* const* grad_contribs, int64_t which, cudaStream_t s)
{
    zero_status_t st = set_device(p);
    if (st != ZERO_OK) return st;
    const std::vector<Segment> segs = step_segments(p, which, 0);
    auto run = [&](auto& P, size_t cap) -> cudaError_t {
        for (size_t b = 0; b < segs.size(); b += cap) {
            const size_t e = std::min(segs.size(), b + cap);
            fill_call_params(p, grad_contribs, P);
            const bool vec = build_step_params(p, segs, b, e, grad_contribs, P);
            const cudaError_t err = p->dtype16 == ZERO_BF16 ? launch_norm<ZERO_BF16>(p->device, P, vec, s)
                                                            : launch_norm<ZERO_FP16>(p->device, P, vec, s);
            if (err != cudaSuccess) return err;
        }
        return cudaSuccess;
    };
    cudaError_t err;
    if (segs.size() > (size_t)kMaxSegs) {
        StepParamsWide P;
        err = run(P, kWideSegs);
    } else {
        StepParams P;
        err = run(P, kMaxSegs);
    }
    if (err != cudaSuccess) return cuda_fail(err, "gradient-norm launch");
    p->norm_open = true;
    if (which == -1) std::fill(p->norm_covered.begin(), p->norm_covered.end(), 1);
    else p->norm_covered[(size_t)which] = 1;
    return ZERO_OK;
}

}  // namespace
}  // namespace zero

extern "C" {

zero_status_t zero_grad_norm(zero_plan_t* p, const void* const* grad_contribs, int64_t n_contribs,
                             int64_t which, void* stream)
try {
    const zero_status_t st = check_norm_call(p, grad_contribs, n_contribs, which, "zero_grad_norm");
    if (st != ZERO_OK) return st;
    return enqueue_norm(p, grad_contribs, which, (cudaStream_t)stream);
}
catch (...) {
    return exception_status("zero_grad_norm");
}

zero_status_t zero_step(zero_plan_t* p, const void* const* grad_contribs, int64_t n_contribs,
                        int64_t which, const zero_hyper_t* hyper, void* stream)
try {
    const zero_status_t st = check_step(p, grad_contribs, n_contribs, which, hyper, "zero_step");
    if (st != ZERO_OK) return st;
    return enqueue_step(p, grad_contribs, which, hyper, (cudaStream_t)stream);
}
catch (...) {
    return exception_status("zero_step");
}

zero_status_t zero_step_gather_next(zero_plan_t* p, const void* const* grad_contribs,
                                    int64_t n_contribs, int64_t unit, const zero_hyper_t* hyper,
                                    int64_t next_unit, void* next_full16, void* stream)
try {
    zero_status_t st = check_step(p, grad_contribs, n_contribs, unit, hyper, "zero_step_gather_next");
    if (st != ZERO_OK) return st;
    if (p->stage != 3) return fail(ZERO_EINVAL, "zero_step_gather_next: stage 3 only");
    // bucket -1 would update next_unit's shards in the launch that gathers them
    if (unit < 0) return fail(ZERO_EINVAL, "zero_step_gather_next: unit must name one unit (not -1)");
    if (next_unit < 0 || next_unit >= (int64_t)p->units.size() || next_unit == unit)
        return fail(ZERO_EINVAL, "zero_step_gather_next: next_unit out of range or equal to unit");
    if (p->gathered[(size_t)next_unit]) return fail(ZERO_ESTATE, "zero_step_gather_next: next unit not released");
    const Unit& U = p->units[(size_t)next_unit];
    if (U.numel_pad > 0 && !next_full16) return fail(ZERO_EINVAL, "zero_step_gather_next: NULL destination");
    if (!aligned(next_full16, 2)) return fail(ZERO_EALIGN, "zero_step_gather_next: destination not 2-byte aligned");
    for (const Rank& R : p->ranks)
        if (!R.shard16 && U.shard > 0)
            return fail(ZERO_ESTATE, "zero_step_gather_next: a rank has no 16-bit shard bound");
    const std::vector<Copy> copies = gather_copies(p, next_unit, next_full16);
    bool fused = false;
    st = enqueue_step(p, grad_contribs, unit, hyper, (cudaStream_t)stream, &copies,
                      (uint16_t*)next_full16, &fused);
    if (st != ZERO_OK) return st;
    p->gathered[(size_t)next_unit] = 1;
    p->last_gather_in_step = fused ? 1 : 0;
    return ZERO_OK;
}
catch (...) {
    return exception_status("zero_step_gather_next");
}

zero_status_t zero_step_finish(zero_plan_t* p, void* stream, zero_step_result_t* out)
try {
    if (!p) return fail(ZERO_EINVAL, "zero_step_finish: NULL plan");
    if (p->host_step)
        return fail(ZERO_ESTATE, "zero_step_finish: the step has zero_step_host calls (zero_step_host_finish)");
    return finish_step(p, stream, out);
}
catch (...) {
    return exception_status("zero_step_finish");
}

}  // extern "C"

namespace zero {
namespace {

zero_status_t finish_step(zero_plan_t* p, void* stream, zero_step_result_t* out)
{
    if (!p->in_step) return fail(ZERO_ESTATE, "zero_step_finish: no open step");
    for (int64_t b = 0; b < p->n_buckets; ++b)
        if (!p->covered[(size_t)b])
            return fail(ZERO_ESTATE, "zero_step_finish: a bucket/unit was not stepped");
    zero_status_t st = set_device(p);
    if (st != ZERO_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;

    // Re-cast (no-op unless the flag is set), then the one-thread commit.
    const std::vector<Segment> segs = shard_segments_all(p);
    CommitParams C;
    C.st = dev_state(p);
    C.growth = p->scaler.growth_factor;
    C.backoff = p->scaler.backoff_factor;
    C.min_scale = p->scaler.min_scale;
    C.interval = p->scaler.growth_interval;
    C.dynamic = p->scaler_dynamic;
    auto run = [&](auto& P, size_t cap) -> cudaError_t {
        for (size_t b = 0; b < segs.size(); b += cap) {
            const size_t en = std::min(segs.size(), b + cap);
            std::memset(&P, 0, sizeof(P));
            P.n_d = p->n_d;
            P.st = dev_state(p);
            P.commit = C;
            P.do_commit = en == segs.size();
            const bool vec = build_step_params(p, segs, b, en, nullptr, P);
            const cudaError_t err = p->dtype16 == ZERO_BF16 ? launch_recast<ZERO_BF16>(p->device, P, vec, s)
                                                            : launch_recast<ZERO_FP16>(p->device, P, vec, s);
            if (err != cudaSuccess) return err;
        }
        return cudaSuccess;
    };
    cudaError_t rerr;
    if (segs.size() > (size_t)kMaxSegs) {
        StepParamsWide P;
        rerr = run(P, kWideSegs);
    } else {
        StepParams P;
        rerr = run(P, kMaxSegs);
    }
    if (rerr != cudaSuccess) return cuda_fail(rerr, "re-cast launch");
    if (segs.empty()) {                      // nothing to re-cast: commit on its own
        commit_kernel<<<1, 32, 0, s>>>(C);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "commit launch");
    }
    p->in_step = false;
    p->stepped = true;
    p->norm_open = false;
    std::fill(p->covered.begin(), p->covered.end(), 0);
    std::fill(p->norm_covered.begin(), p->norm_covered.end(), 0);
    if (out) return read_state(p, s, out);
    return ZERO_OK;
}

}  // namespace
}  // namespace zero

extern "C" {

zero_status_t zero_read_state(zero_plan_t* p, void* stream, zero_step_result_t* out)
try {
    if (!p || !out) return fail(ZERO_EINVAL, "zero_read_state: NULL argument");
    if (!p->workspace) return fail(ZERO_ESTATE, "zero_read_state: no rank bound");
    zero_status_t st = set_device(p);
    if (st != ZERO_OK) return st;
    return read_state(p, (cudaStream_t)stream, out);
}
catch (...) {
    return exception_status("zero_read_state");
}

zero_status_t zero_restore_state(zero_plan_t* p, const zero_step_result_t* in, void* stream)
try {
    if (!p || !in) return fail(ZERO_EINVAL, "zero_restore_state: NULL argument");
    if (!p->workspace) return fail(ZERO_ESTATE, "zero_restore_state: no rank bound");
    if (p->in_step) return fail(ZERO_ESTATE, "zero_restore_state: a step is open");
    if (in->t < 0 || in->good_steps < 0 || in->skipped_total < 0 || in->finished < 0 ||
        (in->current != 0 && in->current != 1) || !(in->scale > 0.0) || !std::isfinite(in->scale))
        return fail(ZERO_EINVAL, "zero_restore_state: bad state");
    zero_status_t st = set_device(p);
    if (st != ZERO_OK) return st;
    DevState d;
    std::memset(&d, 0, sizeof(d));
    d.cur = (uint32_t)in->current;
    d.last_skipped = in->skipped ? 1u : 0u;
    d.t = in->t;
    d.skipped = in->skipped_total;
    d.good = in->good_steps;
    d.finished = in->finished;
    d.scale = in->scale;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaMemcpyAsync(dev_state(p), &d, sizeof(d), cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "zero_restore_state: writing the state");
    return ZERO_OK;
}
catch (...) {
    return exception_status("zero_restore_state");
}

zero_status_t zero_gather_layer(zero_plan_t* p, int64_t unit, void* full_unit16, void* stream)
try {
    if (!p) return fail(ZERO_EINVAL, "zero_gather_layer: NULL plan");
    if (p->stage != 3) return fail(ZERO_EINVAL, "zero_gather_layer: stage 3 only");
    if (unit < 0 || unit >= (int64_t)p->units.size())
        return fail(ZERO_EINVAL, "zero_gather_layer: unit out of range");
    if (p->gathered[(size_t)unit]) return fail(ZERO_ESTATE, "zero_gather_layer: unit not released");
    const Unit& U = p->units[(size_t)unit];
    if (U.numel_pad > 0 && !full_unit16) return fail(ZERO_EINVAL, "zero_gather_layer: NULL destination");
    if (!aligned(full_unit16, 2)) return fail(ZERO_EALIGN, "zero_gather_layer: destination not 2-byte aligned");
    for (const Rank& R : p->ranks)
        if (!R.shard16 && U.shard > 0)
            return fail(ZERO_ESTATE, "zero_gather_layer: a rank has no 16-bit shard bound");
    zero_status_t st = set_device(p);
    if (st != ZERO_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    const std::vector<Copy> copies = gather_copies(p, unit, full_unit16);
    const cudaError_t gerr = launch_gather_list(p, copies, s);
    if (gerr != cudaSuccess) return cuda_fail(gerr, "gather launch");
    p->gathered[(size_t)unit] = 1;
    return ZERO_OK;
}
catch (...) {
    return exception_status("zero_gather_layer");
}

zero_status_t zero_release_layer(zero_plan_t* p, int64_t unit)
try {
    if (!p) return fail(ZERO_EINVAL, "zero_release_layer: NULL plan");
    if (p->stage != 3) return fail(ZERO_EINVAL, "zero_release_layer: stage 3 only");
    if (unit < 0 || unit >= (int64_t)p->units.size())
        return fail(ZERO_EINVAL, "zero_release_layer: unit out of range");
    if (!p->gathered[(size_t)unit]) return fail(ZERO_ESTATE, "zero_release_layer: unit not gathered");
    p->gathered[(size_t)unit] = 0;
    return ZERO_OK;
}
catch (...) {
    return exception_status("zero_release_layer");
}

zero_status_t zero_bind_offload(zero_plan_t* p, int rank, float* master, float* m, float* v,
                                float* grad_host, void* param16_host, void* shard16, void* full16,
                                void* workspace)
try {
    if (!p) return fail(ZERO_EINVAL, "zero_bind_offload: NULL plan");
    if (rank < 0 || rank >= p->n_d) return fail(ZERO_EINVAL, "zero_bind_offload: bad rank");
    if (p->in_step || p->stepped)
        return fail(ZERO_ESTATE, "zero_bind_offload: bind every rank before the first step");
    for (const Rank& R : p->ranks)
        if (R.bound && !R.offload)
            return fail(ZERO_ESTATE, "zero_bind_offload: the plan already has on-GPU ranks");
    const int64_t elems = p->state_elems[(size_t)rank];
    if (elems > 0 && (!master || !m || !v || !grad_host || !param16_host))
        return fail(ZERO_EINVAL, "zero_bind_offload: NULL host buffer");
    if (!aligned(master, 4) || !aligned(m, 4) || !aligned(v, 4) || !aligned(grad_host, 4) ||
        !aligned(param16_host, 2))
        return fail(ZERO_EALIGN, "zero_bind_offload: host buffers not aligned to their element size");
    if (elems > 0) {
        // the GPU writes grad_host and the copy engines read param16_host: both must be pinned
        const void* pinned[2] = {grad_host, param16_host};
        for (const void* q : pinned) {
            cudaPointerAttributes at;
            const cudaError_t e = cudaPointerGetAttributes(&at, q);
            if (e != cudaSuccess || at.type != cudaMemoryTypeHost)
                return fail(ZERO_EINVAL, "zero_bind_offload: grad_host and param16_host must be "
                                         "pinned host memory (cudaHostAlloc / cudaHostRegister)");
        }
    }
    // the 16-bit destination and the workspace are device memory, as for zero_bind
    if (p->stage == 3) {
        if (elems > 0 && !shard16) return fail(ZERO_EINVAL, "zero_bind_offload: stage 3 needs shard16");
    } else if (!full16 && !p->full16 && p->phi_pad > 0) {
        return fail(ZERO_EINVAL, "zero_bind_offload: stages 1/2 need the flat 16-bit buffer");
    }
    if (!workspace && !p->workspace) return fail(ZERO_EINVAL, "zero_bind_offload: workspace is NULL");
    if (workspace && p->workspace && workspace != p->workspace)
        return fail(ZERO_EINVAL, "zero_bind_offload: workspace differs from an earlier bind");
    if (!aligned(workspace, 16)) return fail(ZERO_EALIGN, "zero_bind_offload: workspace not 16-byte aligned");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "zero_bind_offload: cudaGetDevice");
    if (workspace && !p->workspace) {
        DevState init;
        std::memset(&init, 0, sizeof(init));
        init.scale = 1.0;
        e = cudaMemcpy(workspace, &init, sizeof(init), cudaMemcpyHostToDevice);
        if (e == cudaSuccess) e = cudaDeviceSynchronize();
        if (e != cudaSuccess) return cuda_fail(e, "zero_bind_offload: initialising the workspace");
        p->workspace = (uint32_t*)workspace;
    }
    p->device = dev;
    if (full16) p->full16 = (uint16_t*)full16;
    Rank& R = p->ranks[(size_t)rank];
    R.bound = true;
    R.offload = true;
    R.master[0] = master;
    R.m[0] = m;
    R.v[0] = v;
    R.master[1] = R.m[1] = R.v[1] = nullptr;
    R.grad_host = grad_host;
    R.param16_host = (uint16_t*)param16_host;
    R.shard16 = (uint16_t*)shard16;
    p->offload = true;
    return ZERO_OK;
}
catch (...) {
    return exception_status("zero_bind_offload");
}

zero_status_t zero_offload_step(zero_plan_t* p, const void* const* grad_contribs, int64_t n_contribs,
                                int64_t which, const zero_hyper_t* hyper, void* stream)
try {
    if (!hyper) return fail(ZERO_EINVAL, "zero_offload_step: NULL argument");
    zero_status_t st = check_call(p, grad_contribs, n_contribs, which, "zero_offload_step");
    if (st != ZERO_OK) return st;
    if (!p->offload) return fail(ZERO_ESTATE, "zero_offload_step: no offloaded rank bound");
    if (!(hyper->beta1 >= 0.0 && hyper->beta1 < 1.0) || !(hyper->beta2 >= 0.0 && hyper->beta2 < 1.0) ||
        !std::isfinite(hyper->lr) || !std::isfinite(hyper->eps) || !std::isfinite(hyper->weight_decay))
        return fail(ZERO_EINVAL, "zero_offload_step: betas must lie in [0, 1); lr, eps, wd finite");
    if (hyper->flags != 0) return fail(ZERO_EINVAL, "zero_offload_step: no norm report on the offload path");
    if (!(hyper->max_grad_norm >= 0.0) || !std::isfinite(hyper->max_grad_norm))
        return fail(ZERO_EINVAL, "zero_offload_step: max_grad_norm must be finite and >= 0");
    if (hyper->max_grad_norm > 0.0)
        for (int64_t b = 0; b < p->n_buckets; ++b)
            if (!p->norm_covered[(size_t)b])
                return fail(ZERO_ESTATE, "zero_offload_step: clipping needs zero_grad_norm over every bucket/unit first");
    if (p->in_step && std::memcmp(&p->step_hyper, hyper, sizeof(*hyper)) != 0)
        return fail(ZERO_EINVAL, "zero_offload_step: hyperparameters changed inside a step");
    if (which == -1) {
        if (p->in_step) return fail(ZERO_ESTATE, "zero_offload_step: bucket -1 must be the only call");
    } else if (p->covered[(size_t)which]) {
        return fail(ZERO_ESTATE, "zero_offload_step: bucket/unit already stepped in this step");
    }
    st = set_device(p);
    if (st != ZERO_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    if (!p->in_step) {
        if (p->bias_len == 0 || p->bias_beta1 != hyper->beta1 || p->bias_beta2 != hyper->beta2) {
            st = upload_bias_table(p, hyper->beta1, hyper->beta2, s);
            if (st != ZERO_OK) return st;
        }
        step_constants(*hyper, 1, 1.0, p->n_d, p->consts);
        p->step_hyper = *hyper;
    }
    const std::vector<Segment> segs = step_segments(p, which, 0);
    if (!p->in_step) {
        p->off_segs.clear();
        p->off_group_end.clear();
        p->off_deferred.clear();
    }
    cudaError_t err;
    if (p->offload_defer) {
        // the flag pass now; the writing reduction when zero_offload_finish knows the decision
        err = offload_flag_pass(p, grad_contribs, segs, s);
        if (err == cudaSuccess)
            p->off_deferred.push_back({std::vector<const void*>(grad_contribs, grad_contribs + p->n_d), segs});
    } else {
        err = offload_flag_pass(p, grad_contribs, segs, s);
        if (err == cudaSuccess) err = offload_reduce_groups(p, grad_contribs, segs, p->off_segs.size(), s);
    }
    if (err != cudaSuccess) return cuda_fail(err, "reduce-to-host launch");
    if (!p->offload_defer) p->off_segs.insert(p->off_segs.end(), segs.begin(), segs.end());
    p->in_step = true;
    if (which == -1) std::fill(p->covered.begin(), p->covered.end(), 1);
    else p->covered[(size_t)which] = 1;
    return ZERO_OK;
}
catch (...) {
    return exception_status("zero_offload_step");
}

zero_status_t zero_offload_finish(zero_plan_t* p, int threads, void* stream, zero_step_result_t* out)
try {
    if (!p) return fail(ZERO_EINVAL, "zero_offload_finish: NULL plan");
    if (!p->offload) return fail(ZERO_ESTATE, "zero_offload_finish: no offloaded rank bound");
    if (!p->in_step) return fail(ZERO_ESTATE, "zero_offload_finish: no open step");
    for (int64_t b = 0; b < p->n_buckets; ++b)
        if (!p->covered[(size_t)b])
            return fail(ZERO_ESTATE, "zero_offload_finish: a bucket/unit was not stepped");
    zero_status_t st = set_device(p);
    if (st != ZERO_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    // t and the scale decide the constants, the flag decides between the update and the
    // re-cast: read them on a side stream as soon as the step's last flag pass is done, while
    // the reductions are still streaming the gradients into host memory.
    cudaError_t e = cudaSuccess;
    if (!p->off_side) {
        cudaStream_t side;
        e = cudaStreamCreateWithFlags(&side, cudaStreamNonBlocking);
        if (e != cudaSuccess) return cuda_fail(e, "zero_offload_finish: side stream");
        p->off_side = side;
        p->release_hook = release_plan_resources;
    }
    cudaStream_t side = (cudaStream_t)p->off_side;
    DevState host;
    e = cudaStreamWaitEvent(side, (cudaEvent_t)p->off_flag_event, 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(&host, p->workspace, sizeof(host), cudaMemcpyDeviceToHost, side);
    if (e == cudaSuccess) e = cudaStreamSynchronize(side);
    if (e != cudaSuccess) return cuda_fail(e, "zero_offload_finish: reading the step state");
    float k9[9];
    step_constants(p->step_hyper, host.t + 1, host.scale, p->n_d, k9);
    // clipping: the coefficient from the step's norm, with the double operations of the GPU
    // step's clip mode (correctly rounded sqrt, add, divide; rounded once to fp32)
    float coef = 1.0f;
    if (p->step_hyper.max_grad_norm > 0.0) {
        double c = p->step_hyper.max_grad_norm / (std::sqrt(host.norm2) + 1e-6);
        if (c > 1.0) c = 1.0;
        coef = (float)c;
    }
    // deferred reductions (ZERO_OPT_OFFLOAD_DEFER): the decision is known; a clean step streams
    // every call's gradient to the host now, a skipped one needs none of it
    if (!p->off_deferred.empty()) {
        if (host.flag == 0)
            for (const zero_plan::OffloadCall& c : p->off_deferred) {
                e = offload_reduce_groups(p, c.contribs.data(), c.segs, p->off_segs.size(), s);
                if (e != cudaSuccess) return cuda_fail(e, "zero_offload_finish: reduce-to-host launch");
                p->off_segs.insert(p->off_segs.end(), c.segs.begin(), c.segs.end());
            }
        else
            for (const zero_plan::OffloadCall& c : p->off_deferred)
                p->off_segs.insert(p->off_segs.end(), c.segs.begin(), c.segs.end());
        p->off_deferred.clear();
    }
    const std::vector<Segment>& segs = p->off_segs;
    std::vector<CpuSpan> spans;
    std::vector<int> group_of_span;
    int g = 0;
    for (size_t i = 0; i < segs.size(); ++i) {
        while ((size_t)g < p->off_group_end.size() && i >= p->off_group_end[(size_t)g]) ++g;
        const Segment& sg = segs[i];
        const Rank& R = p->ranks[(size_t)sg.rank];
        spans.push_back(CpuSpan{R.master[0] + sg.s_off, R.m[0] + sg.s_off, R.v[0] + sg.s_off,
                                R.grad_host + sg.s_off, R.param16_host + sg.s_off, sg.n});
        group_of_span.push_back(g);
    }
    // 16-bit parameters [off, off + n) of segment i back to the all-gather destination
    auto copy_back = [&](size_t i, int64_t off, int64_t n) -> cudaError_t {
        const Segment& sg = segs[i];
        const Rank& R = p->ranks[(size_t)sg.rank];
        return cudaMemcpyAsync(sg.out16 + sg.o_off + off, R.param16_host + sg.s_off + off, 2 * (size_t)n,
                               cudaMemcpyHostToDevice, s);
    };
    const int nt = threads > 0 ? threads : 1;
    if (worker_pool_size(p->host_pool) < nt) {
        worker_pool_destroy(p->host_pool);
        p->host_pool = worker_pool_create(nt);
        p->release_hook = release_plan_resources;
    }
    if (host.flag != 0) {
        // skipped step: every gradient lands first, then the re-cast of the unchanged master
        e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) return cuda_fail(e, "zero_offload_finish: waiting for the reductions");
        cpu_adamw(p->host_pool, spans, k9, p->dtype16, true, nt);
        for (size_t i = 0; i < segs.size() && e == cudaSuccess; ++i) e = copy_back(i, 0, segs[i].n);
    } else {
        // the update of each group starts once its gradient has landed; finished ranges of
        // 16-bit parameters are copied back while the rest is still being updated
        const bool ok = cpu_adamw_overlapped(
            p->host_pool, spans, group_of_span, k9, p->dtype16, nt, coef,
            [&](int grp) {
                e = cudaEventSynchronize((cudaEvent_t)p->off_events[(size_t)grp]);
                return e == cudaSuccess;
            },
            [&](size_t i, int64_t off, int64_t n) {
                e = copy_back(i, off, n);
                return e == cudaSuccess;
            });
        if (!ok && e == cudaSuccess) e = cudaErrorUnknown;
    }
    if (e != cudaSuccess) return cuda_fail(e, "zero_offload_finish: the host update or the copy back");
    CommitParams C;
    C.st = dev_state(p);
    C.growth = p->scaler.growth_factor;
    C.backoff = p->scaler.backoff_factor;
    C.min_scale = p->scaler.min_scale;
    C.interval = p->scaler.growth_interval;
    C.dynamic = p->scaler_dynamic;
    commit_kernel<<<1, 32, 0, s>>>(C);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "commit launch");
    p->in_step = false;
    p->stepped = true;
    p->norm_open = false;
    std::fill(p->covered.begin(), p->covered.end(), 0);
    std::fill(p->norm_covered.begin(), p->norm_covered.end(), 0);
    if (out) return read_state(p, s, out);
    return ZERO_OK;
}
catch (...) {
    return exception_status("zero_offload_finish");
}

zero_status_t zero_bind_host_staging(zero_plan_t* p, void* const staging[2], int64_t bytes_each)
try {
    if (!p || !staging || !staging[0] || !staging[1])
        return fail(ZERO_EINVAL, "zero_bind_host_staging: NULL argument");
    if (p->in_step) return fail(ZERO_ESTATE, "zero_bind_host_staging: a step is open");
    if (p->offload) return fail(ZERO_ESTATE, "zero_bind_host_staging: offloaded plan");
    if (p->device < 0 || !p->workspace)
        return fail(ZERO_ESTATE, "zero_bind_host_staging: bind the ranks first");
    zero_plan_info_t info;
    zero_status_t st = zero_plan_info(p, &info);
    if (st != ZERO_OK) return st;
    if (bytes_each < info.host_staging_bytes)
        return fail(ZERO_ERANGE, "zero_bind_host_staging: an area is smaller than info.host_staging_bytes");
    if (!aligned(staging[0], 16) || !aligned(staging[1], 16))
        return fail(ZERO_EALIGN, "zero_bind_host_staging: areas must be 16-byte aligned");
    const uintptr_t a = (uintptr_t)staging[0], b = (uintptr_t)staging[1];
    if (bytes_each > 0 && (a < b ? b - a : a - b) < (uintptr_t)bytes_each)
        return fail(ZERO_EINVAL, "zero_bind_host_staging: the two areas overlap");
    for (int i = 0; i < 2; ++i) {
        cudaPointerAttributes at;
        const cudaError_t e = cudaPointerGetAttributes(&at, staging[i]);
        if (e != cudaSuccess || (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged) ||
            at.device != p->device) {
            (void)cudaGetLastError();
            return fail(ZERO_EINVAL, "zero_bind_host_staging: areas must be device memory of the plan's device");
        }
    }
    p->host_staging[0] = staging[0];
    p->host_staging[1] = staging[1];
    // rank r's part starts r * (bytes_each / N_d, rounded down to 16 bytes) into an area: at
    // least one bucket's or unit's range, whole-buffer calls (bucket -1) given larger areas
    p->host_rank_stride = bytes_each / p->n_d / 16 * 8;
    return ZERO_OK;
}
catch (...) {
    return exception_status("zero_bind_host_staging");
}

zero_status_t zero_grad_norm_host(zero_plan_t* p, const void* const* host_contribs, int64_t n_contribs,
                                  int64_t which, void* stream)
try {
    zero_status_t st = check_norm_call(p, host_contribs, n_contribs, which, "zero_grad_norm_host");
    if (st != ZERO_OK) return st;
    if (!p->host_staging[0])
        return fail(ZERO_ESTATE, "zero_grad_norm_host: no staging bound (zero_bind_host_staging)");
    const std::vector<Segment> segs = step_segments(p, which, 0);
    const auto runs = read_runs(segs);
    if (!runs.empty() && runs.back().second > p->host_rank_stride)
        return fail(ZERO_ERANGE, "zero_grad_norm_host: the call's range exceeds a rank's part of the staging areas");
    if (!segs.empty())
        for (int r = 0; r < p->n_d; ++r)
            if (!pinned_host_cached(p, host_contribs[r]))
                return fail(ZERO_EINVAL, "zero_grad_norm_host: a contribution is not pinned host memory");
    st = set_device(p);
    if (st != ZERO_OK) return st;
    cudaError_t e = host_resources(p);
    if (e != cudaSuccess) return cuda_fail(e, "zero_grad_norm_host: copy streams");
    cudaStream_t s = (cudaStream_t)stream, h2d = (cudaStream_t)p->host_h2d;
    const int b = (int)(p->host_calls % 2);
    cudaEvent_t copied = (cudaEvent_t)p->host_events[b], used = (cudaEvent_t)p->host_events[2 + b];
    cudaEvent_t out_done = (cudaEvent_t)p->host_events[4];
    // the same staging rotation and ordering as zero_step_host
    e = cudaStreamWaitEvent(h2d, p->host_pipeline ? used : out_done, 0);
    std::vector<const void*> dev(p->n_d);
    int64_t h2d_bytes = 0;
    for (int r = 0; r < p->n_d && e == cudaSuccess; ++r) {
        dev[(size_t)r] = (uint16_t*)p->host_staging[b] + (int64_t)r * p->host_rank_stride;
        for (const auto& run : runs) {
            const size_t bytes = 2 * (size_t)(run.second - run.first);
            e = cudaMemcpyAsync((uint16_t*)dev[(size_t)r] + run.first, (const uint16_t*)host_contribs[r] + run.first,
                                bytes, cudaMemcpyHostToDevice, h2d);
            if (e != cudaSuccess) break;
            h2d_bytes += (int64_t)bytes;
        }
    }
    if (e == cudaSuccess) e = cudaEventRecord(copied, h2d);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, copied, 0);
    if (e != cudaSuccess) return cuda_fail(e, "zero_grad_norm_host: host-to-device copies");
    st = enqueue_norm(p, dev.data(), which, s);
    if (st != ZERO_OK) return st;
    // the area is free again once the pass has read it (serial: the next call waits for it)
    e = cudaEventRecord(used, s);
    if (e == cudaSuccess) e = cudaEventRecord(out_done, s);
    if (e != cudaSuccess) return cuda_fail(e, "zero_grad_norm_host: ordering the copies");
    p->host_h2d_bytes += h2d_bytes;
    ++p->host_calls;
    return ZERO_OK;
}
catch (...) {
    return exception_status("zero_grad_norm_host");
}

zero_status_t zero_step_host(zero_plan_t* p, const void* const* host_contribs, int64_t n_contribs,
                             int64_t which, const zero_hyper_t* hyper, void* host_out16, void* stream)
try {
    zero_status_t st = check_step(p, host_contribs, n_contribs, which, hyper, "zero_step_host");
    if (st != ZERO_OK) return st;
    if (!p->host_staging[0]) return fail(ZERO_ESTATE, "zero_step_host: no staging bound (zero_bind_host_staging)");
    if (!host_out16) return fail(ZERO_EINVAL, "zero_step_host: NULL host_out16");
    if (!aligned(host_out16, 2)) return fail(ZERO_EALIGN, "zero_step_host: host_out16 not 2-byte aligned");
    const std::vector<Segment> segs = step_segments(p, which, 0);
    const auto runs = read_runs(segs);
    if (!runs.empty() && runs.back().second > p->host_rank_stride)
        return fail(ZERO_ERANGE, "zero_step_host: the call's range exceeds a rank's part of the staging areas "
                                 "(bucket -1 needs areas of N_d * 2 * phi_pad bytes, phi_pad rounded up to 8)");
    if (!segs.empty()) {
        if (!pinned_host_cached(p, host_out16))
            return fail(ZERO_EINVAL, "zero_step_host: host_out16 is not pinned host memory");
        for (int r = 0; r < p->n_d; ++r)
            if (!pinned_host_cached(p, host_contribs[r]))
                return fail(ZERO_EINVAL, "zero_step_host: a contribution is not pinned host memory");
    }
    st = set_device(p);
    if (st != ZERO_OK) return st;
    cudaError_t e = host_resources(p);
    if (e != cudaSuccess) return cuda_fail(e, "zero_step_host: copy streams");
    cudaStream_t s = (cudaStream_t)stream, h2d = (cudaStream_t)p->host_h2d, d2h = (cudaStream_t)p->host_d2h;
    const int b = (int)(p->host_calls % 2);
    cudaEvent_t copied = (cudaEvent_t)p->host_events[b], used = (cudaEvent_t)p->host_events[2 + b];
    cudaEvent_t out_done = (cudaEvent_t)p->host_events[4];
    // pieces: the call alone makes the step (nothing before or after it to overlap with)
    // (runs are sorted and disjoint: the call reads [front.first, back.second))
    const int64_t lo = runs.empty() ? 0 : runs.front().first;
    const int64_t hi = runs.empty() ? 0 : runs.back().second;
    int pieces = 1;
    if (p->host_pipeline && !p->in_step && (which == -1 || p->n_buckets == 1))
        pieces = (int)std::max<int64_t>(1, std::min<int64_t>(kHostMaxPieces, (hi - lo) / kHostPieceElems));
    while (pieces > 1 && p->host_piece_events.size() < (size_t)(2 * pieces)) {
        cudaEvent_t ev;
        e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
        if (e != cudaSuccess) return cuda_fail(e, "zero_step_host: events");
        p->host_piece_events.push_back(ev);
        p->release_hook = release_plan_resources;
    }
    // host -> device: after the step that last read this area (pipelined), or after everything
    // the previous call did, its device -> host copies included (serial)
    e = cudaStreamWaitEvent(h2d, p->host_pipeline ? used : out_done, 0);
    if (e != cudaSuccess) return cuda_fail(e, "zero_step_host: ordering the copies");
    std::vector<const void*> dev(p->n_d);
    for (int r = 0; r < p->n_d; ++r)
        dev[(size_t)r] = (uint16_t*)p->host_staging[b] + (int64_t)r * p->host_rank_stride;
    int64_t h2d_bytes = 0, d2h_bytes = 0;
    std::vector<zero_plan::HostCopy> outs;
    for (int i = 0; i < pieces; ++i) {
        // piece i: [plo, phi) of the call's range, cut at a multiple of 8 elements
        const int64_t plo = i == 0 ? lo : (lo + (hi - lo) * i / pieces) / 8 * 8;
        const int64_t phi = i + 1 == pieces ? hi : (lo + (hi - lo) * (i + 1) / pieces) / 8 * 8;
        const std::vector<Segment> part = pieces == 1 ? segs : segments_in(segs, plo, phi);
        const auto part_runs = pieces == 1 ? runs : read_runs(part);
        cudaEvent_t pc = pieces == 1 ? copied : (cudaEvent_t)p->host_piece_events[(size_t)(2 * i)];
        cudaEvent_t pu = pieces == 1 ? used : (cudaEvent_t)p->host_piece_events[(size_t)(2 * i + 1)];
        for (int r = 0; r < p->n_d && e == cudaSuccess; ++r) {
            uint16_t* area = (uint16_t*)dev[(size_t)r];
            for (const auto& run : part_runs) {
                const size_t bytes = 2 * (size_t)(run.second - run.first);
                e = cudaMemcpyAsync(area + run.first, (const uint16_t*)host_contribs[r] + run.first, bytes,
                                    cudaMemcpyHostToDevice, h2d);
                if (e != cudaSuccess) break;
                h2d_bytes += (int64_t)bytes;
            }
        }
        if (e == cudaSuccess) e = cudaEventRecord(pc, h2d);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s, pc, 0);
        if (e != cudaSuccess) return cuda_fail(e, "zero_step_host: host-to-device copies");
        st = enqueue_step(p, dev.data(), which, hyper, s, nullptr, nullptr, nullptr,
                          pieces == 1 ? nullptr : &part, i + 1 == pieces);
        if (st != ZERO_OK) return st;
        // device -> host: the piece's 16-bit results, merged where both sides are contiguous
        e = cudaEventRecord(pu, s);
        if (e == cudaSuccess && pieces > 1 && i + 1 == pieces) e = cudaEventRecord(used, s);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(d2h, pu, 0);
        const size_t first_out = outs.size();
        for (const Segment& sg : part) {
            if (sg.n <= 0) continue;
            uint16_t* h = (uint16_t*)host_out16 + sg.c_off;
            const uint16_t* d = sg.out16 + sg.o_off;
            if (outs.size() > first_out && outs.back().host + outs.back().n == h && outs.back().dev + outs.back().n == d)
                outs.back().n += sg.n;
            else
                outs.push_back({h, d, sg.n});
        }
        for (size_t j = first_out; j < outs.size() && e == cudaSuccess; ++j) {
            e = cudaMemcpyAsync(outs[j].host, outs[j].dev, 2 * (size_t)outs[j].n, cudaMemcpyDeviceToHost, d2h);
            d2h_bytes += 2 * outs[j].n;
        }
        if (e != cudaSuccess) return cuda_fail(e, "zero_step_host: device-to-host copies");
    }
    e = cudaEventRecord(out_done, d2h);
    if (e != cudaSuccess) return cuda_fail(e, "zero_step_host: device-to-host copies");
    p->host_outs.insert(p->host_outs.end(), outs.begin(), outs.end());
    p->host_h2d_bytes += h2d_bytes;
    p->host_d2h_bytes += d2h_bytes;
    p->host_step = true;
    ++p->host_calls;
    return ZERO_OK;
}
catch (...) {
    return exception_status("zero_step_host");
}

zero_status_t zero_step_host_finish(zero_plan_t* p, void* stream, zero_step_result_t* out)
try {
    if (!p) return fail(ZERO_EINVAL, "zero_step_host_finish: NULL plan");
    if (!p->host_step) return fail(ZERO_ESTATE, "zero_step_host_finish: no zero_step_host call in the open step");
    zero_status_t st = set_device(p);
    if (st != ZERO_OK) return st;
    zero_step_result_t res;
    st = finish_step(p, stream, &res);                 // synchronises `stream`
    if (st == ZERO_ESTATE || st == ZERO_EINVAL) return st;   // nothing was enqueued
    const std::string finish_msg = st != ZERO_OK ? zero_last_error() : "";
    cudaStream_t d2h = (cudaStream_t)p->host_d2h;
    cudaError_t e = cudaStreamSynchronize(d2h);
    // a skipped or discarded step re-cast its 16-bit parameters after they were copied
    if (e == cudaSuccess && (st == ZERO_ETIMEOUT || (st == ZERO_OK && res.skipped))) {
        for (const zero_plan::HostCopy& c : p->host_outs) {
            e = cudaMemcpyAsync(c.host, c.dev, 2 * (size_t)c.n, cudaMemcpyDeviceToHost, d2h);
            if (e != cudaSuccess) break;
            p->host_d2h_bytes += 2 * c.n;
        }
        if (e == cudaSuccess) e = cudaStreamSynchronize(d2h);
    }
    p->host_h2d_last = p->host_h2d_bytes;
    p->host_d2h_last = p->host_d2h_bytes;
    p->host_h2d_bytes = p->host_d2h_bytes = 0;
    p->host_outs.clear();
    p->host_step = false;
    if (e != cudaSuccess) return cuda_fail(e, "zero_step_host_finish: device-to-host copies");
    if (out) *out = res;
    if (st != ZERO_OK) return fail(st, finish_msg);
    return ZERO_OK;
}
catch (...) {
    return exception_status("zero_step_host_finish");
}

zero_status_t zero_step_units_overlapped(zero_plan_t* p, const void* const* unit_contribs,
                                         int64_t n_ptrs, void* const* gather_bufs,
                                         const zero_hyper_t* hyper, void* compute_stream,
                                         void* comm_stream, zero_step_result_t* out)
try {
    if (!p || !unit_contribs || !gather_bufs || !hyper)
        return fail(ZERO_EINVAL, "zero_step_units_overlapped: NULL argument");
    if (p->stage != 3) return fail(ZERO_EINVAL, "zero_step_units_overlapped: stage 3 only");
    const int64_t nu = (int64_t)p->units.size();
    if (n_ptrs != nu * p->n_d)
        return fail(ZERO_EINVAL, "zero_step_units_overlapped: need n_units * N_d contributions");
    if (comm_stream && compute_stream == comm_stream)
        return fail(ZERO_EINVAL, "zero_step_units_overlapped: the two streams must differ");
    if (p->in_step) return fail(ZERO_ESTATE, "zero_step_units_overlapped: a step is open");
    const int64_t nd = p->n_d;
    // the units in the order of the schedule: first to last, or last to first
    std::vector<int64_t> seq((size_t)nu);
    for (int64_t i = 0; i < nu; ++i) seq[(size_t)i] = p->unit_order ? nu - 1 - i : i;
    // every argument the calls below check, checked before the first is enqueued, so a refused
    // call leaves no step open and no unit gathered
    zero_status_t st = check_hyper(hyper, "zero_step_units_overlapped");
    if (st != ZERO_OK) return st;
    for (int64_t u = 0; u < nu; ++u) {
        st = check_call(p, unit_contribs + u * nd, nd, u, "zero_step_units_overlapped");
        if (st != ZERO_OK) return st;
        if (p->gathered[(size_t)u]) return fail(ZERO_ESTATE, "zero_step_units_overlapped: a unit is gathered");
    }
    for (int64_t i = 0; i < nu; ++i) {
        const Unit& U = p->units[(size_t)seq[(size_t)i]];
        void* buf = gather_bufs[i % 2];
        if (U.numel_pad > 0 && !buf) return fail(ZERO_EINVAL, "zero_step_units_overlapped: NULL gather buffer");
        if (!aligned(buf, 2))
            return fail(ZERO_EALIGN, "zero_step_units_overlapped: gather buffer not 2-byte aligned");
        for (const Rank& R : p->ranks)
            if (!R.shard16 && U.shard > 0)
                return fail(ZERO_ESTATE, "zero_step_units_overlapped: a rank has no 16-bit shard bound");
    }
    st = set_device(p);
    if (st != ZERO_OK) return st;
    if (!comm_stream) {
        // one stream: the next unit's all-gather streams inside each unit's step launch
        if (hyper->max_grad_norm > 0.0)
            for (int64_t u = 0; u < nu; ++u) {
                st = zero_grad_norm(p, unit_contribs + u * nd, nd, u, compute_stream);
                if (st != ZERO_OK) return st;
            }
        if (nu > 0) {
            st = zero_gather_layer(p, seq[0], gather_bufs[0], compute_stream);
            if (st != ZERO_OK) return st;
        }
        for (int64_t i = 0; i < nu; ++i) {
            const int64_t u = seq[(size_t)i];
            // (a layer's forward/backward would consume gather_bufs[i % 2] here)
            st = zero_release_layer(p, u);
            if (st != ZERO_OK) return st;
            st = i + 1 < nu ? zero_step_gather_next(p, unit_contribs + u * nd, nd, u, hyper, seq[(size_t)i + 1],
                                                    gather_bufs[(i + 1) % 2], compute_stream)
                            : zero_step(p, unit_contribs + u * nd, nd, u, hyper, compute_stream);
            if (st != ZERO_OK) return st;
        }
        return zero_step_finish(p, compute_stream, out);
    }
    if (!p->ov_events[0]) {
        for (int i = 0; i < 5; ++i) {
            cudaEvent_t ev;
            const cudaError_t e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
            if (e != cudaSuccess) return cuda_fail(e, "zero_step_units_overlapped: event");
            p->ov_events[i] = ev;
        }
        p->release_hook = release_plan_resources;
    }
    cudaStream_t cs = (cudaStream_t)compute_stream, ms = (cudaStream_t)comm_stream;
    cudaEvent_t start = (cudaEvent_t)p->ov_events[0];
    cudaEvent_t gathered[2] = {(cudaEvent_t)p->ov_events[1], (cudaEvent_t)p->ov_events[2]};
    cudaEvent_t released[2] = {(cudaEvent_t)p->ov_events[3], (cudaEvent_t)p->ov_events[4]};
    if (hyper->max_grad_norm > 0.0)
        for (int64_t u = 0; u < nu; ++u) {
            st = zero_grad_norm(p, unit_contribs + u * nd, nd, u, compute_stream);
            if (st != ZERO_OK) return st;
        }
    cudaError_t e = cudaEventRecord(start, cs);           // the previous step's shards are final
    if (e == cudaSuccess) e = cudaStreamWaitEvent(ms, start, 0);
    if (e != cudaSuccess) return cuda_fail(e, "zero_step_units_overlapped: ordering the streams");
    for (int64_t i = 0; i < nu; ++i) {
        const int64_t u = seq[(size_t)i];
        const int b = (int)(i % 2);
        if (i >= 2) {
            e = cudaStreamWaitEvent(ms, released[b], 0);
            if (e != cudaSuccess) return cuda_fail(e, "zero_step_units_overlapped: wait release");
        }
        st = zero_gather_layer(p, u, gather_bufs[b], comm_stream);
        if (st != ZERO_OK) return st;
        e = cudaEventRecord(gathered[b], ms);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, gathered[b], 0);
        if (e != cudaSuccess) return cuda_fail(e, "zero_step_units_overlapped: wait gather");
        // (a layer's forward/backward would consume gather_bufs[b] here)
        st = zero_release_layer(p, u);
        if (st != ZERO_OK) return st;
        e = cudaEventRecord(released[b], cs);
        if (e != cudaSuccess) return cuda_fail(e, "zero_step_units_overlapped: record release");
        st = zero_step(p, unit_contribs + u * nd, nd, u, hyper, compute_stream);
        if (st != ZERO_OK) return st;
    }
    return zero_step_finish(p, compute_stream, out);
}
catch (...) {
    return exception_status("zero_step_units_overlapped");
}

// ---------------------------------------------------------------------------------------
// No-allocation variant: the fused step over one flat range with its scratch (the non-finite
// flag) in a library-owned static device array instead of a caller workspace.
// ---------------------------------------------------------------------------------------

}  // extern "C"

static __device__ __align__(256) uint32_t g_noalloc_scratch[ZERO_NOALLOC_SCRATCH_BYTES / 4];

namespace zero {
namespace {

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
struct NoallocAddr {
    unsigned long long ctx = 0;   // unique ID of the CUDA context the address belongs to
    void* addr = nullptr;
};
NoallocAddr g_noalloc_addr[kMaxDevices];

// Unique ID of the calling thread's current CUDA context (0 when none is current or the
// driver cannot say).  Context IDs are never reused within a process, so a device reset,
// which replaces the primary context and reloads the module, changes the ID.
unsigned long long current_context_id()
{
    using GetCurrent = CUresult (*)(CUcontext*);
    using GetId = CUresult (*)(CUcontext, unsigned long long*);
    static GetCurrent get_current = nullptr;
    static GetId get_id = nullptr;
    static bool resolved = false;
    if (!resolved) {            // under g_noalloc_mu
        cudaDriverEntryPointQueryResult q1, q2;
        void *f1 = nullptr, *f2 = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) == cudaSuccess &&
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) == cudaSuccess &&
            q1 == cudaDriverEntryPointSuccess && q2 == cudaDriverEntryPointSuccess) {
            get_current = (GetCurrent)f1;
            get_id = (GetId)f2;
        }
        (void)cudaGetLastError();
        resolved = true;
    }
    if (!get_current || !get_id) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Device address of g_noalloc_scratch for the current device.  In host code the array's name
// is only a host-side handle, never a device address.  The address is looked up with the
// device current the first time a device (in a given CUDA context) is used, and cached.
zero_status_t noalloc_scratch(void** out)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "zero_step_range_noalloc: cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices)
        return fail(ZERO_ERANGE, "zero_step_range_noalloc: device index beyond the supported range");
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    NoallocAddr& c = g_noalloc_addr[dev];
    const unsigned long long ctx = current_context_id();
    if (!c.addr || ctx == 0 || c.ctx != ctx) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);   // makes the context current
        if (e != cudaSuccess || !p)
            return cuda_fail(e, "zero_step_range_noalloc: cudaGetSymbolAddress of the scratch");
        c.addr = p;
        c.ctx = current_context_id();
    }
    *out = c.addr;
    return ZERO_OK;
}

}  // namespace
}  // namespace zero

extern "C" {

zero_status_t zero_step_range_noalloc(const void* const* grad_contribs, int n_d, int64_t n,
                                      int dtype16, const float* master_in, const float* m_in,
                                      const float* v_in, float* master_out, float* m_out,
                                      float* v_out, void* out16, const zero_hyper_t* hyper,
                                      int64_t t, double loss_scale, void* stream,
                                      int32_t* nonfinite)
try {
    static_assert(sizeof(uint32_t) <= ZERO_NOALLOC_SCRATCH_BYTES, "flag must fit the scratch");
    if (!grad_contribs || !hyper || !nonfinite)
        return fail(ZERO_EINVAL, "zero_step_range_noalloc: NULL argument");
    if (n_d < 1) return fail(ZERO_EINVAL, "zero_step_range_noalloc: n_d must be >= 1");
    if (n_d > ZERO_MAX_RANKS)
        return fail(ZERO_ERANGE, "zero_step_range_noalloc: n_d exceeds ZERO_MAX_RANKS");
    if (n < 0) return fail(ZERO_EINVAL, "zero_step_range_noalloc: n < 0");
    if (dtype16 != ZERO_BF16 && dtype16 != ZERO_FP16)
        return fail(ZERO_EINVAL, "zero_step_range_noalloc: bad dtype16");
    if (t < 1) return fail(ZERO_EINVAL, "zero_step_range_noalloc: t must be >= 1");
    if (hyper->max_grad_norm != 0.0 || hyper->flags != 0)
        return fail(ZERO_EINVAL, "zero_step_range_noalloc: no gradient-norm options here");
    if (!(loss_scale > 0.0) || !std::isfinite(loss_scale))
        return fail(ZERO_EINVAL, "zero_step_range_noalloc: bad loss scale");
    const float* fin[3] = {master_in, m_in, v_in};
    float* fout[3] = {master_out, m_out, v_out};
    if (n > 0) {
        for (int i = 0; i < 3; ++i) {
            if (!fin[i] || !fout[i]) return fail(ZERO_EINVAL, "zero_step_range_noalloc: NULL state");
            if (fin[i] == fout[i])
                return fail(ZERO_EINVAL, "zero_step_range_noalloc: output state aliases its input");
            if (!aligned(fin[i], 4) || !aligned(fout[i], 4))
                return fail(ZERO_EALIGN, "zero_step_range_noalloc: fp32 state not 4-byte aligned");
        }
        if (!out16) return fail(ZERO_EINVAL, "zero_step_range_noalloc: NULL out16");
        if (!aligned(out16, 2)) return fail(ZERO_EALIGN, "zero_step_range_noalloc: out16 not 2-byte aligned");
        for (int r = 0; r < n_d; ++r) {
            if (!grad_contribs[r]) return fail(ZERO_EINVAL, "zero_step_range_noalloc: NULL contribution");
            if (!aligned(grad_contribs[r], 2))
                return fail(ZERO_EALIGN, "zero_step_range_noalloc: contribution not 2-byte aligned");
        }
    }
    void* scratch = nullptr;
    zero_status_t st = noalloc_scratch(&scratch);
    if (st != ZERO_OK) return st;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "zero_step_range_noalloc: cudaGetDevice");
    cudaStream_t s = (cudaStream_t)stream;
    e = cudaMemsetAsync(scratch, 0, sizeof(uint32_t), s);   // the flag must start at zero
    if (e != cudaSuccess) return cuda_fail(e, "zero_step_range_noalloc: clearing the flag");
    if (n > 0) {
        // Host mode of the fused kernel: all constants from the host, half 0 read, half 1 written.
        StepParams P;
        std::memset(&P, 0, sizeof(P));
        for (int r = 0; r < n_d; ++r) P.c[r] = (const uint16_t*)grad_contribs[r];
        step_constants(*hyper, t, loss_scale, n_d, P.k);
        P.n_d = n_d;
        P.n_seg = 1;
        P.flag = (uint32_t*)scratch;
        P.st = nullptr;
        KSeg& K = P.seg[0];
        K.p[0] = const_cast<float*>(master_in);
        K.m[0] = const_cast<float*>(m_in);
        K.v[0] = const_cast<float*>(v_in);
        K.p[1] = master_out;
        K.m[1] = m_out;
        K.v[1] = v_out;
        K.out16 = (uint16_t*)out16;
        K.c_off = 0;
        K.n = n;
        const int h = head16(K.out16);
        bool vec = true;
        for (int r = 0; r < n_d; ++r) vec &= head16(P.c[r]) == h;
        const int64_t hh = std::min<int64_t>(h, n);
        for (int i = 0; i < 2; ++i)
            vec &= aligned(K.p[i] + hh, 16) && aligned(K.m[i] + hh, 16) && aligned(K.v[i] + hh, 16);
        K.head = (int32_t)hh;
        K.nvec = (n - hh) / 8;
        K.tail = (int32_t)(n - hh - 8 * K.nvec);
        e = dtype16 == ZERO_BF16 ? launch_fused<ZERO_BF16>(dev, P, vec, s)
                                 : launch_fused<ZERO_FP16>(dev, P, vec, s);
        if (e != cudaSuccess) return cuda_fail(e, "zero_step_range_noalloc: launch");
    }
    uint32_t flag = 0;
    e = cudaMemcpyAsync(&flag, scratch, sizeof(flag), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "zero_step_range_noalloc: reading the flag");
    *nonfinite = flag ? 1 : 0;
    return ZERO_OK;
}
catch (...) {
    return exception_status("zero_step_range_noalloc");
}

}  // extern "C"
