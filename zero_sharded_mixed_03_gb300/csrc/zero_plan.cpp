// zero_plan.cpp -- host planner of the sharded step: flat-buffer partition,
// bucket and shard tables, the physical state layout, and the memory /
// communication accounting.  Pure host code (no CUDA calls), so every entry
// point here also works on a machine without a GPU.
//
// Page: "Zero Redundancy Optimizer (ZeRO) and Fully Sharded Data Parallelism
// (FSDP): Mathematical Foundations ..." (llms.blog).
#include <algorithm>
#include <cmath>
#include <cstring>
#include <exception>
#include <memory>
#include <new>

#include "zero_internal.h"

namespace zero {

namespace {
thread_local std::string g_last_error;

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
}  // namespace

zero_status_t fail(zero_status_t code, const std::string& msg)
{
    g_last_error = msg;
    return code;
}

zero_status_t exception_status(const char* where) noexcept
{
    const char* what = "unknown exception";
    try {
        throw;
    } catch (const std::exception& e) {
        what = e.what();
    } catch (...) {
    }
    try {
        g_last_error = std::string(where) + ": host resource exhausted (" + what + ")";
    } catch (...) {
        // the message itself could not be stored: the status still reports the failure
    }
    return ZERO_ENOMEM;
}

void bucket_range(const zero_plan* p, int64_t b, int64_t* lo, int64_t* hi)
{
    if (b < 0) {
        *lo = 0;
        *hi = p->phi_pad;
        return;
    }
    const int64_t B = p->bucket_elems ? p->bucket_elems : p->phi_pad;
    *lo = b * B;
    *hi = std::min(p->phi_pad, *lo + B);
}

std::vector<Segment> step_segments(const zero_plan* p, int64_t which, int cur_out)
{
    (void)cur_out;
    std::vector<Segment> segs;
    if (p->per_param) {
        for (const Chunk& c : p->chunks) {
            if (c.unit != which || c.rows == 0 || !p->ranks[(size_t)c.rank].bound) continue;
            segs.push_back(Segment{c.rows * c.cols, c.contrib_off, c.phys_off, c.phys_off,
                                   (int)c.rank, p->ranks[(size_t)c.rank].shard16});
        }
        return segs;
    }
    if (p->stage == 3) {
        const Unit& U = p->units[(size_t)which];
        for (int r = 0; r < p->n_d; ++r) {
            if (!p->ranks[(size_t)r].bound || U.shard == 0) continue;
            const int64_t off = p->phys_off[(size_t)r][(size_t)which];
            segs.push_back(Segment{U.shard, r * U.shard, off, off, r, p->ranks[(size_t)r].shard16});
        }
        return segs;
    }
    int64_t lo, hi;
    bucket_range(p, which, &lo, &hi);
    const int64_t S = p->units[0].shard;
    for (int r = 0; r < p->n_d; ++r) {
        if (!p->ranks[(size_t)r].bound) continue;
        const int64_t s_lo = r * S, s_hi = s_lo + S;
        const int64_t a = std::max(lo, s_lo), e = std::min(hi, s_hi);
        if (a >= e) continue;
        segs.push_back(Segment{e - a, a - lo, p->phys_off[(size_t)r][0] + (a - s_lo), a, r,
                               p->full16});
    }
    return segs;
}

std::vector<Segment> shard_segments_all(const zero_plan* p)
{
    std::vector<Segment> segs;
    if (p->per_param) {
        for (const Chunk& c : p->chunks) {
            if (c.rows == 0 || !p->ranks[(size_t)c.rank].bound) continue;
            segs.push_back(Segment{c.rows * c.cols, 0, c.phys_off, c.phys_off, (int)c.rank,
                                   p->ranks[(size_t)c.rank].shard16});
        }
        return segs;
    }
    for (int r = 0; r < p->n_d; ++r) {
        if (!p->ranks[(size_t)r].bound) continue;
        for (size_t u = 0; u < p->units.size(); ++u) {
            const Unit& U = p->units[u];
            if (U.shard == 0) continue;
            const int64_t off = p->phys_off[(size_t)r][u];
            if (p->stage == 3)
                segs.push_back(Segment{U.shard, 0, off, off, r, p->ranks[(size_t)r].shard16});
            else
                segs.push_back(Segment{U.shard, 0, off, U.base + r * U.shard, r, p->full16});
        }
    }
    return segs;
}

void step_constants(const zero_hyper_t& h, int64_t t, double scale, int n_d, float out[9])
{
    const double one_minus_b1t = 1.0 - std::pow(h.beta1, (double)t);
    const double one_minus_b2t = 1.0 - std::pow(h.beta2, (double)t);
    out[0] = (float)h.beta1;
    out[1] = (float)(1.0 - h.beta1);
    out[2] = (float)h.beta2;
    out[3] = (float)(1.0 - h.beta2);
    out[4] = (float)h.eps;
    out[5] = (float)(h.lr * h.weight_decay);
    out[6] = (float)(h.lr / one_minus_b1t);
    out[7] = (float)std::sqrt(one_minus_b2t);
    out[8] = (float)(1.0 / ((double)n_d * scale));
}

}  // namespace zero

using namespace zero;

extern "C" {

const char* zero_last_error(void) { return g_last_error.c_str(); }

zero_status_t zero_plan_create(const int64_t* tensor_sizes, int64_t n_tensors, int n_d, int stage,
                               int64_t bucket_elems, const int64_t* unit_first, int64_t n_units,
                               int dtype16, zero_plan_t** out)
try {
    if (out == nullptr) return fail(ZERO_EINVAL, "zero_plan_create: out is NULL");
    *out = nullptr;
    if (n_tensors < 0 || (n_tensors > 0 && tensor_sizes == nullptr))
        return fail(ZERO_EINVAL, "zero_plan_create: bad tensor list");
    if (n_d < 1) return fail(ZERO_EINVAL, "zero_plan_create: n_d must be >= 1");
    if (n_d > ZERO_MAX_RANKS) return fail(ZERO_ERANGE, "zero_plan_create: n_d > ZERO_MAX_RANKS");
    if (stage < 1 || stage > 3) return fail(ZERO_EINVAL, "zero_plan_create: stage must be 1, 2 or 3");
    if (dtype16 != ZERO_BF16 && dtype16 != ZERO_FP16)
        return fail(ZERO_EINVAL, "zero_plan_create: dtype16 must be ZERO_BF16 or ZERO_FP16");
    if (bucket_elems < 0) return fail(ZERO_EINVAL, "zero_plan_create: bucket_elems < 0");
    const bool has_units = unit_first != nullptr && n_units > 0;
    if (stage == 3 && bucket_elems != 0)
        return fail(ZERO_EINVAL, "zero_plan_create: stage 3 reduces per unit; bucket_elems must be 0");
    if (stage != 3 && has_units)
        return fail(ZERO_EINVAL, "zero_plan_create: units are a stage-3 notion");
    for (int64_t i = 0; i < n_tensors; ++i)
        if (tensor_sizes[i] < 0) return fail(ZERO_EINVAL, "zero_plan_create: negative tensor size");

    // owned here until it is handed out, so that a failure (or an exception) part way frees it
    std::unique_ptr<zero_plan> owner(new (std::nothrow) zero_plan);
    if (!owner) return fail(ZERO_ENOMEM, "zero_plan_create: out of host memory");
    zero_plan* p = owner.get();
    p->n_d = n_d;
    p->stage = stage;
    p->dtype16 = dtype16;
    p->bucket_elems = bucket_elems;
    p->sizes.assign(tensor_sizes, tensor_sizes + n_tensors);
    p->tensor_offset.assign((size_t)n_tensors, 0);

    std::vector<int64_t> starts;
    if (has_units) {
        starts.assign(unit_first, unit_first + n_units);
        bool ok = starts[0] == 0;
        for (size_t u = 1; ok && u < starts.size(); ++u)
            ok = starts[u] > starts[u - 1] && starts[u] <= n_tensors;
        if (!ok || (n_tensors == 0 && starts.size() > 1))
            return fail(ZERO_EINVAL, "zero_plan_create: unit_first must start at 0 and increase");
    } else {
        starts.push_back(0);
    }

    int64_t base = 0, shard_base = 0, phi = 0;
    for (size_t u = 0; u < starts.size(); ++u) {
        Unit U;
        U.first = starts[u];
        U.count = (u + 1 < starts.size() ? starts[u + 1] : n_tensors) - U.first;
        U.numel = 0;
        for (int64_t k = U.first; k < U.first + U.count; ++k) {
            p->tensor_offset[(size_t)k] = base + U.numel;
            U.numel += p->sizes[(size_t)k];
        }
        U.numel_pad = ceil_div(U.numel, n_d) * n_d;
        U.shard = U.numel_pad / n_d;
        U.base = base;
        U.shard_base = shard_base;
        base += U.numel_pad;
        shard_base += U.shard;
        phi += U.numel;
        p->units.push_back(U);
    }
    p->phi = phi;
    p->phi_pad = base;
    p->shard_total = shard_base;
    if (stage == 3) {
        p->n_buckets = (int64_t)p->units.size();
    } else {
        const int64_t B = bucket_elems ? bucket_elems : p->phi_pad;
        p->n_buckets = p->phi_pad == 0 ? 0 : ceil_div(p->phi_pad, B);
    }

    // Physical state layout: unit u's shard of rank r starts at an offset congruent to
    // r * S_u modulo 8, the element phase of that shard inside the 16-bit buffers.
    p->phys_off.assign((size_t)n_d, std::vector<int64_t>(p->units.size(), 0));
    p->state_elems.assign((size_t)n_d, 0);
    for (int r = 0; r < n_d; ++r) {
        int64_t cursor = 0;
        for (size_t u = 0; u < p->units.size(); ++u) {
            const int64_t want = (r * p->units[u].shard) % 8;
            const int64_t off = cursor + (((want - cursor) % 8) + 8) % 8;
            p->phys_off[(size_t)r][u] = off;
            cursor = off + p->units[u].shard;
        }
        p->state_elems[(size_t)r] = ceil_div(cursor, 8) * 8;
    }
    p->ranks.assign((size_t)n_d, Rank());
    p->covered.assign((size_t)std::max<int64_t>(p->n_buckets, 1), 0);
    p->norm_covered.assign((size_t)std::max<int64_t>(p->n_buckets, 1), 0);
    p->gathered.assign(p->units.size(), 0);
    *out = owner.release();
    return ZERO_OK;
}
catch (...) {
    return exception_status("zero_plan_create");
}

zero_status_t zero_plan_create_per_param(const int64_t* tensor_sizes, const int64_t* dim0,
                                         int64_t n_tensors, int n_d, const int64_t* unit_first,
                                         int64_t n_units, int dtype16, zero_plan_t** out)
try {
    if (out == nullptr) return fail(ZERO_EINVAL, "zero_plan_create_per_param: out is NULL");
    *out = nullptr;
    if (n_tensors > 0 && dim0 == nullptr)
        return fail(ZERO_EINVAL, "zero_plan_create_per_param: dim0 is NULL");
    for (int64_t t = 0; t < n_tensors; ++t) {
        if (tensor_sizes && (dim0[t] < 0 || (dim0[t] == 0 && tensor_sizes[t] != 0) ||
                             (dim0[t] > 0 && tensor_sizes[t] % dim0[t] != 0)))
            return fail(ZERO_EINVAL, "zero_plan_create_per_param: size is not a multiple of dim0");
    }
    zero_plan_t* made = nullptr;
    zero_status_t st = zero_plan_create(tensor_sizes, n_tensors, n_d, 3, 0, unit_first, n_units,
                                        dtype16, &made);
    if (st != ZERO_OK) return st;
    // destroyed here if anything below fails (or throws) before it is handed out
    std::unique_ptr<zero_plan, void (*)(zero_plan*)> owner(made, zero_plan_destroy);
    zero_plan* p = owner.get();
    p->per_param = true;
    p->dim0.assign(dim0, dim0 + n_tensors);
    // units: unpadded gradient buffers; a rank's unit shard = its padded local chunks
    int64_t base = 0, shard_base = 0;
    for (Unit& U : p->units) {
        U.numel_pad = U.numel;
        U.base = base;
        int64_t off = 0;
        U.shard = 0;
        for (int64_t t = U.first; t < U.first + U.count; ++t) {
            p->tensor_offset[(size_t)t] = base + off;
            off += p->sizes[(size_t)t];
            const int64_t rows_t = p->dim0[(size_t)t];
            const int64_t cols = rows_t > 0 ? p->sizes[(size_t)t] / rows_t : 0;
            U.shard += ceil_div(rows_t, n_d) * cols;
        }
        U.shard_base = shard_base;
        base += U.numel;
        shard_base += U.shard;
    }
    p->phi_pad = base;
    p->shard_total = shard_base;
    p->chunks.clear();
    for (int r = 0; r < n_d; ++r) {
        int64_t logical = 0, cursor = 0;
        for (size_t u = 0; u < p->units.size(); ++u) {
            const Unit& U = p->units[u];
            int64_t off = 0;
            for (int64_t t = U.first; t < U.first + U.count; ++t) {
                Chunk c;
                c.rank = r;
                c.unit = (int64_t)u;
                c.tensor = t;
                const int64_t rows_t = p->dim0[(size_t)t];
                c.cols = rows_t > 0 ? p->sizes[(size_t)t] / rows_t : 0;
                c.c_rows = ceil_div(rows_t, n_d);
                c.row0 = r * c.c_rows;
                c.rows = std::max<int64_t>(0, std::min(c.row0 + c.c_rows, rows_t) - c.row0);
                c.contrib_off = off + c.row0 * c.cols;
                c.state_off = logical;
                const int64_t want = c.contrib_off % 8;
                c.phys_off = cursor + (((want - cursor) % 8) + 8) % 8;
                if (t == U.first) p->phys_off[(size_t)r][u] = c.phys_off;
                cursor = c.phys_off + c.c_rows * c.cols;
                logical += c.c_rows * c.cols;
                off += p->sizes[(size_t)t];
                p->chunks.push_back(c);
            }
        }
        p->state_elems[(size_t)r] = ceil_div(cursor, 8) * 8;
    }
    *out = owner.release();
    return ZERO_OK;
}
catch (...) {
    return exception_status("zero_plan_create_per_param");
}

void zero_plan_destroy(zero_plan_t* plan)
try {
    if (plan && plan->release_hook) plan->release_hook(plan);
    delete plan;
}
catch (...) {
    (void)exception_status("zero_plan_destroy");
}

zero_status_t zero_plan_info(const zero_plan_t* p, zero_plan_info_t* out)
try {
    if (!p || !out) return fail(ZERO_EINVAL, "zero_plan_info: NULL argument");
    std::memset(out, 0, sizeof(*out));
    out->n_tensors = (int64_t)p->sizes.size();
    out->n_units = (int64_t)p->units.size();
    out->n_buckets = p->n_buckets;
    out->phi = p->phi;
    out->phi_pad = p->phi_pad;
    out->shard = p->shard_total;
    int64_t maxc = 0, maxu = 0;
    if (p->stage == 3) {
        for (const Unit& U : p->units) maxu = std::max(maxu, U.numel_pad);
        maxc = maxu;
    } else {
        maxc = p->bucket_elems ? std::min(p->bucket_elems, p->phi_pad) : p->phi_pad;
    }
    out->max_contrib_elems = maxc;
    out->max_unit_pad = maxu;
    out->host_staging_bytes = (int64_t)p->n_d * ((maxc + 7) / 8 * 8) * 2;
    out->workspace_bytes = kWorkspaceBytes;
    out->n_d = p->n_d;
    out->stage = p->stage;
    out->dtype16 = p->dtype16;
    return ZERO_OK;
}
catch (...) {
    return exception_status("zero_plan_info");
}

zero_status_t zero_rank_state_elems(const zero_plan_t* p, int rank, int64_t* elems)
try {
    if (!p || !elems) return fail(ZERO_EINVAL, "zero_rank_state_elems: NULL argument");
    if (rank < 0 || rank >= p->n_d) return fail(ZERO_EINVAL, "zero_rank_state_elems: bad rank");
    *elems = p->state_elems[(size_t)rank];
    return ZERO_OK;
}
catch (...) {
    return exception_status("zero_rank_state_elems");
}

zero_status_t zero_plan_tables(const zero_plan_t* p, int which, int64_t* dst, int64_t cap,
                               int64_t* n_rows)
try {
    if (!p || !n_rows) return fail(ZERO_EINVAL, "zero_plan_tables: NULL argument");
    std::vector<int64_t> rows;
    int cols = 0;
    switch (which) {
    case ZERO_TABLE_TENSOR_OFFSET:
        cols = 1;
        rows = p->tensor_offset;
        break;
    case ZERO_TABLE_UNITS:
        cols = 7;
        for (const Unit& U : p->units)
            rows.insert(rows.end(), {U.first, U.count, U.numel, U.numel_pad, U.shard, U.base,
                                     U.shard_base});
        break;
    case ZERO_TABLE_PARAM_CHUNKS:
        if (!p->per_param) return fail(ZERO_EINVAL, "zero_plan_tables: not a per-parameter plan");
        cols = 10;
        for (const Chunk& c : p->chunks)
            rows.insert(rows.end(), {c.rank, c.unit, c.tensor, c.row0, c.rows, c.cols, c.c_rows,
                                     c.contrib_off, c.state_off, c.phys_off});
        break;
    case ZERO_TABLE_SHARD_SEGMENTS:
        if (p->per_param) return fail(ZERO_EINVAL, "zero_plan_tables: flat-buffer table of a per-parameter plan");
        cols = 6;
        // Per (rank, unit): the shard interval cut at tensor boundaries, then the tail padding.
        for (int r = 0; r < p->n_d; ++r)
            for (size_t u = 0; u < p->units.size(); ++u) {
                const Unit& U = p->units[u];
                const int64_t lo = U.base + r * U.shard, hi = lo + U.shard;
                // first tensor whose end lies beyond lo (tensor offsets are non-decreasing)
                const int64_t t0 = U.first, t1 = U.first + U.count;
                int64_t k = std::lower_bound(p->tensor_offset.begin() + t0,
                                             p->tensor_offset.begin() + t1, lo + 1) -
                            p->tensor_offset.begin();
                k = std::max(t0, k - 1);
                for (; k < t1; ++k) {
                    const int64_t a = std::max(lo, p->tensor_offset[(size_t)k]);
                    const int64_t e = std::min(hi, p->tensor_offset[(size_t)k] + p->sizes[(size_t)k]);
                    if (p->tensor_offset[(size_t)k] >= hi) break;
                    if (a < e)
                        rows.insert(rows.end(), {r, (int64_t)u, k, a - p->tensor_offset[(size_t)k],
                                                 U.shard_base + (a - lo), e - a});
                }
                const int64_t pad_lo = U.base + U.numel, pad_hi = U.base + U.numel_pad;
                const int64_t a = std::max(lo, pad_lo), e = std::min(hi, pad_hi);
                if (a < e)
                    rows.insert(rows.end(), {r, (int64_t)u, -1, a - pad_lo, U.shard_base + (a - lo),
                                             e - a});
            }
        break;
    case ZERO_TABLE_BUCKET_SEGMENTS:
        if (p->per_param) return fail(ZERO_EINVAL, "zero_plan_tables: flat-buffer table of a per-parameter plan");
        cols = 5;
        if (p->stage != 3) {
            const int64_t S = p->units[0].shard;
            for (int64_t b = 0; b < p->n_buckets; ++b) {
                int64_t lo, hi;
                bucket_range(p, b, &lo, &hi);
                for (int r = 0; r < p->n_d; ++r) {
                    const int64_t a = std::max(lo, r * S), e = std::min(hi, (r + 1) * S);
                    if (a < e) rows.insert(rows.end(), {b, (int64_t)r, a, a - r * S, e - a});
                }
            }
        }
        break;
    case ZERO_TABLE_STATE_LAYOUT:
        if (p->per_param) return fail(ZERO_EINVAL, "zero_plan_tables: use ZERO_TABLE_PARAM_CHUNKS");
        cols = 4;
        for (int r = 0; r < p->n_d; ++r)
            for (size_t u = 0; u < p->units.size(); ++u)
                rows.insert(rows.end(), {(int64_t)r, (int64_t)u, p->phys_off[(size_t)r][u],
                                         p->units[u].shard});
        break;
    default:
        return fail(ZERO_EINVAL, "zero_plan_tables: unknown table");
    }
    *n_rows = (int64_t)rows.size() / cols;
    if ((int64_t)rows.size() > cap) {
        if (dst == nullptr && cap == 0) return ZERO_OK;  // size query
        return fail(ZERO_ERANGE, "zero_plan_tables: destination too small");
    }
    if (!rows.empty()) {
        if (!dst) return fail(ZERO_EINVAL, "zero_plan_tables: dst is NULL");
        std::memcpy(dst, rows.data(), rows.size() * sizeof(int64_t));
    }
    return ZERO_OK;
}
catch (...) {
    return exception_status("zero_plan_tables");
}

zero_status_t zero_memory_report(const zero_plan_t* p, zero_mem_report_t* out)
try {
    if (!p || !out) return fail(ZERO_EINVAL, "zero_memory_report: NULL argument");
    std::memset(out, 0, sizeof(*out));
    const int64_t F = p->phi_pad, S = p->shard_total;
    // "Memory Partitioning Stages Comparison": (params, grads, optimizer) per stage.
    const int64_t tab[4][3] = {{2 * F, 2 * F, 12 * F},
                               {2 * F, 2 * F, 12 * S},
                               {2 * F, 2 * S, 12 * S},
                               {2 * S, 2 * S, 12 * S}};
    for (int s = 0; s < 4; ++s) {
        out->logical_total[s] = 0;
        for (int c = 0; c < 3; ++c) {
            out->logical[s][c] = tab[s][c];
            out->logical_total[s] += tab[s][c];
        }
    }
    out->logical_ddp_fp32_grads = 2 * F + 4 * F + 12 * F;
    int64_t state = 0;
    for (int r = 0; r < p->n_d; ++r)
        if (p->ranks[(size_t)r].bound) state = std::max(state, p->state_elems[(size_t)r]);
    if (state == 0)
        for (int r = 0; r < p->n_d; ++r) state = std::max(state, p->state_elems[(size_t)r]);
    out->physical_state_bytes = state * 4 * 3 * 2;
    out->physical_param16_bytes = p->stage == 3 ? state * 2 : F * 2;
    zero_plan_info_t info;
    zero_plan_info(p, &info);
    out->physical_contrib_bytes = (int64_t)p->n_d * info.max_contrib_elems * 2;
    out->physical_gather_bytes = info.max_unit_pad * 2;
    out->workspace_bytes = info.workspace_bytes;
    return ZERO_OK;
}
catch (...) {
    return exception_status("zero_memory_report");
}

zero_status_t zero_comm_report(const zero_plan_t* p, zero_comm_report_t* out)
try {
    if (!p || !out) return fail(ZERO_EINVAL, "zero_comm_report: NULL argument");
    std::memset(out, 0, sizeof(*out));
    const int64_t one = (int64_t)(p->n_d - 1) * p->shard_total;  // (N-1)/N * phi_pad
    out->per_collective = one;
    out->ddp = 2 * one;
    out->zero1 = 2 * one;
    out->zero2 = 2 * one;
    out->zero3 = 3 * one;
    out->this_stage = p->stage == 1 ? out->zero1 : p->stage == 2 ? out->zero2 : out->zero3;
    out->bytes_per_elem = 2;
    out->collectives_per_step =
        p->stage == 3 ? 3 * (int64_t)p->units.size() : 2 * p->n_buckets;
    return ZERO_OK;
}
catch (...) {
    return exception_status("zero_comm_report");
}

}  // extern "C"
