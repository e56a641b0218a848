// Reshard planning ("boxing"): from a source layout and a destination layout,
// the list of rectangular regions to move. Every destination piece is the
// union of its intersections with the source pieces (OneFlow page: boxing
// inserted between mismatched SBPs; ONNX page: execution semantics, "reshard
// inputs"). Partial sources (OneFlow SBP definition of partial sum) become
// regions read from every member of a partial group and summed.
//
// Each source byte is planned to be read once per destination group of equal
// pieces: broadcast destinations with the same box are written from the same
// registers (one read, many writes), which keeps all-gather and all-reduce
// traffic at its algorithmic minimum.
#include <algorithm>
#include <cstring>
#include <map>
#include <string>
#include <unordered_map>

#include "rtp_internal.h"

namespace rtp {

namespace {

struct SrcGroup {
    Box box;
    std::vector<std::pair<int64_t, int>> members;  // (partial index, rank)
};

struct DstGroup {
    Box box;
    std::vector<int> ranks;
};

bool same_box(int ndim, const Box& a, const Box& b)
{
    for (int d = 0; d < ndim; ++d)
        if (a.lo[d] != b.lo[d] || a.hi[d] != b.hi[d]) return false;
    return true;
}

void row_major_strides(int ndim, const Box& b, int64_t* st)
{
    int64_t s = 1;
    for (int a = ndim - 1; a >= 0; --a) {
        st[a] = s;
        s *= b.hi[a] - b.lo[a];
    }
}

// Region [lo, hi) of the logical tensor, read from pieces with box sbox and
// written to pieces with box dbox.
int make_task(int ndim, const int64_t* lo, const int64_t* hi, const Box& sbox, const Box& dbox, PlanTask* t,
              int64_t* soff, int64_t* doff)
{
    int64_t e[RTP_MAX_NDIM] = {}, ss[RTP_MAX_NDIM] = {}, ds[RTP_MAX_NDIM] = {};
    row_major_strides(ndim, sbox, ss);
    row_major_strides(ndim, dbox, ds);
    *soff = 0;
    *doff = 0;
    for (int a = 0; a < ndim; ++a) {
        e[a] = hi[a] - lo[a];
        *soff += (lo[a] - sbox.lo[a]) * ss[a];
        *doff += (lo[a] - dbox.lo[a]) * ds[a];
    }
    // innermost run: the last axis, grown outward while the region covers
    // whole rows of both pieces
    int a = ndim - 1;
    int64_t cols = e[a];
    while (a > 0 && ss[a - 1] == cols && ds[a - 1] == cols) {
        --a;
        cols *= e[a];
    }
    // outer dims, unit extents dropped, contiguous neighbours merged
    int64_t oe[RTP_MAX_NDIM], os[RTP_MAX_NDIM], od[RTP_MAX_NDIM];
    int n = 0;
    for (int b = 0; b < a; ++b) {
        if (e[b] == 1) continue;
        if (n > 0 && os[n - 1] == e[b] * ss[b] && od[n - 1] == e[b] * ds[b]) {
            oe[n - 1] *= e[b];
            os[n - 1] = ss[b];
            od[n - 1] = ds[b];
            continue;
        }
        oe[n] = e[b];
        os[n] = ss[b];
        od[n] = ds[b];
        ++n;
    }
    if (n > kMaxOuter) return fail(RTP_EUNSUPPORTED, "reshard: region needs %d outer dims (max %d)", n, kMaxOuter);
    t->cols = cols;
    t->n_outer = n;
    t->rows = 1;
    for (int k = 0; k < n; ++k) {
        t->ext[k] = oe[k];
        t->sstr[k] = os[k];
        t->dstr[k] = od[k];
        t->rows *= oe[k];
    }
    return RTP_OK;
}

// One-shot test hooks of the calling thread (rtp_test_hook).
thread_local int g_hook = RTP_HOOK_NONE;
thread_local int64_t g_hook_arg = 0;

}  // namespace

void inject_alloc_fault()
{
    if (g_hook == RTP_HOOK_FAIL_ALLOC) {
        g_hook = RTP_HOOK_NONE;
        throw std::bad_alloc();
    }
}

int check_task_bounds(const char* fn, const std::vector<PlanTask>& tasks, const std::vector<int64_t>& src_vol,
                      const std::vector<int64_t>& dst_vol)
{
    for (size_t i = 0; i < tasks.size(); ++i) {
        const PlanTask& t = tasks[i];
        if (t.rows < 1 || t.cols < 1 || t.n_outer < 0 || t.n_outer > kMaxOuter)
            return fail(RTP_EINVAL, "%s: planned task %zu has an empty or malformed region", fn, i);
        int64_t rows = 1, sspan = 0, dspan = 0;  // offsets of the last row's first element
        for (int k = 0; k < t.n_outer; ++k) {
            if (t.ext[k] < 1 || t.sstr[k] < 0 || t.dstr[k] < 0)
                return fail(RTP_EINVAL, "%s: planned task %zu has a malformed outer dim %d", fn, i, k);
            rows *= t.ext[k];
            sspan += (t.ext[k] - 1) * t.sstr[k];
            dspan += (t.ext[k] - 1) * t.dstr[k];
        }
        if (rows != t.rows) return fail(RTP_EINVAL, "%s: planned task %zu has %lld rows, its dims %lld", fn, i,
                                        (long long)t.rows, (long long)rows);
        for (int side = 0; side < 2; ++side) {
            const std::vector<Ref>& refs = side == 0 ? t.src : t.dst;
            const std::vector<int64_t>& vol = side == 0 ? src_vol : dst_vol;
            const int64_t span = (side == 0 ? sspan : dspan) + t.cols;
            for (const Ref& r : refs) {
                if (r.rank < 0 || (size_t)r.rank >= vol.size())
                    return fail(RTP_EINVAL, "%s: planned task %zu names %s rank %d", fn, i, side ? "destination" : "source",
                                r.rank);
                if (r.offset < 0 || r.offset + span > vol[(size_t)r.rank])
                    return fail(RTP_EINVAL,
                                "%s: planned task %zu would %s elements [%lld, %lld) of %s piece %d, which holds %lld",
                                fn, i, side ? "write" : "read", (long long)r.offset, (long long)(r.offset + span),
                                side ? "destination" : "source", r.rank, (long long)vol[(size_t)r.rank]);
            }
        }
    }
    return RTP_OK;
}

int plan_reshard(int ndim, const int64_t* shape, const rtp_spec& src, const rtp_spec& dst,
                 std::vector<PlanTask>* tasks)
{
    inject_alloc_fault();
    tasks->clear();
    int64_t sc[RTP_MAX_RANKS * RTP_MAX_MESH_NDIM], dc[RTP_MAX_RANKS * RTP_MAX_MESH_NDIM];
    rank_coords(src, sc);
    rank_coords(dst, dc);
    int64_t nsrc = num_ranks(src), ndst = num_ranks(dst);

    // Source pieces grouped by box; within a group, one member per partial index.
    std::vector<SrcGroup> sg;
    for (int r = 0; r < nsrc; ++r) {
        Box b = rank_box(ndim, shape, src, sc + r * RTP_MAX_MESH_NDIM);
        if (!b.b_rep || box_volume(ndim, b) == 0) continue;
        auto it = std::find_if(sg.begin(), sg.end(), [&](const SrcGroup& g) { return same_box(ndim, g.box, b); });
        if (it == sg.end()) {
            sg.push_back(SrcGroup{b, {}});
            it = sg.end() - 1;
        }
        it->members.emplace_back(b.pidx, r);
    }
    for (auto& g : sg) std::sort(g.members.begin(), g.members.end());

    // Destination pieces grouped by box and by whether they hold values.
    std::vector<DstGroup> dval, dzero;
    for (int r = 0; r < ndst; ++r) {
        Box b = rank_box(ndim, shape, dst, dc + r * RTP_MAX_MESH_NDIM);
        if (box_volume(ndim, b) == 0) continue;
        auto& list = b.holds_value ? dval : dzero;
        auto it = std::find_if(list.begin(), list.end(), [&](const DstGroup& g) { return same_box(ndim, g.box, b); });
        if (it == list.end()) {
            list.push_back(DstGroup{b, {}});
            it = list.end() - 1;
        }
        it->ranks.push_back(r);
    }

    for (const auto& dg : dval) {
        for (const auto& g : sg) {
            int64_t lo[RTP_MAX_NDIM], hi[RTP_MAX_NDIM];
            bool empty = false;
            for (int a = 0; a < ndim; ++a) {
                lo[a] = std::max(dg.box.lo[a], g.box.lo[a]);
                hi[a] = std::min(dg.box.hi[a], g.box.hi[a]);
                if (hi[a] <= lo[a]) empty = true;
            }
            if (empty) continue;
            PlanTask t;
            int64_t so, dof;
            int st = make_task(ndim, lo, hi, g.box, dg.box, &t, &so, &dof);
            if (st) return st;
            for (auto& m : g.members) t.src.push_back(Ref{m.second, so});
            for (int r : dg.ranks) t.dst.push_back(Ref{r, dof});
            t.op = partial_reduction(src);
            tasks->push_back(std::move(t));
        }
    }
    for (const auto& dg : dzero) {
        PlanTask t;
        int64_t so, dof;
        int st = make_task(ndim, dg.box.lo, dg.box.hi, dg.box, dg.box, &t, &so, &dof);
        if (st) return st;
        for (int r : dg.ranks) t.dst.push_back(Ref{r, dof});
        t.op = partial_reduction(dst);  // filled with the identity of the destination's reduction
        tasks->push_back(std::move(t));
    }
    return RTP_OK;
}

}  // namespace rtp

using namespace rtp;

namespace {

int element_size(int dtype) { return dtype == RTP_F32 ? 4 : 2; }

int check_common(const char* fn, int dtype, int ndim, const int64_t* shape)
{
    if (dtype != RTP_F32 && dtype != RTP_BF16) return fail(RTP_EINVAL, "%s: unknown dtype %d", fn, dtype);
    if (!shape) return fail(RTP_EINVAL, "%s: shape is NULL", fn);
    if (ndim < 1 || ndim > RTP_MAX_NDIM) return fail(RTP_EINVAL, "%s: ndim %d outside [1, %d]", fn, ndim, RTP_MAX_NDIM);
    for (int a = 0; a < ndim; ++a)
        if (shape[a] < 0) return fail(RTP_ESHAPE, "%s: extent %d is negative", fn, a);
    return RTP_OK;
}

int check_pointers(const char* fn, const char* which, const std::vector<PlanTask>& tasks, const void* const* bufs,
                   bool src, int es)
{
    for (const auto& t : tasks)
        for (const auto& r : (src ? t.src : t.dst)) {
            const void* p = bufs[r.rank];
            if (!p) return fail(RTP_EINVAL, "%s: %s buffer of rank %d is NULL", fn, which, r.rank);
            if ((uintptr_t)p % es) return fail(RTP_EINVAL, "%s: %s buffer of rank %d is not %d-byte aligned", fn, which, r.rank, es);
        }
    return RTP_OK;
}

// Byte ranges [begin, end) of the non-empty pieces of `spec`, one per rank.
void piece_ranges(int ndim, const int64_t* shape, const rtp_spec& spec, const void* const* bufs, int es, bool src,
                  std::vector<std::pair<uintptr_t, uintptr_t>>* out)
{
    int64_t coords[RTP_MAX_RANKS * RTP_MAX_MESH_NDIM];
    rank_coords(spec, coords);
    for (int64_t r = 0; r < num_ranks(spec); ++r) {
        const Box b = rank_box(ndim, shape, spec, coords + r * RTP_MAX_MESH_NDIM);
        const int64_t v = box_volume(ndim, b);
        if (v == 0 || !bufs[r] || (src && !b.b_rep)) continue;
        const uintptr_t p = (uintptr_t)bufs[r];
        out->emplace_back(p, p + (uintptr_t)v * (uintptr_t)es);
    }
}

// Source and destination pieces must not share memory: the kernel reads
// sources while it writes destinations, in no fixed order.
int check_no_overlap(const char* fn, std::vector<std::pair<uintptr_t, uintptr_t>> srcs,
                     std::vector<std::pair<uintptr_t, uintptr_t>> dsts)
{
    std::sort(srcs.begin(), srcs.end());
    std::sort(dsts.begin(), dsts.end());
    size_t i = 0, j = 0;
    while (i < srcs.size() && j < dsts.size()) {
        if (srcs[i].first < dsts[j].second && dsts[j].first < srcs[i].second)
            return fail(RTP_EINVAL, "%s: a source buffer overlaps a destination buffer", fn);
        if (srcs[i].second <= dsts[j].second) ++i;
        else ++j;
    }
    return RTP_OK;
}

// The planner reads, of each spec, the mesh shape, the rank of every mesh
// position and each mesh dim's kind and axis; the key holds exactly those
// (unused array slots may hold anything and are left out).
void append_spec(std::string* k, const rtp_spec& s)
{
    const int64_t n = num_ranks(s);
    k->append(reinterpret_cast<const char*>(&s.mesh_ndim), sizeof s.mesh_ndim);
    k->append(reinterpret_cast<const char*>(s.mesh_shape), sizeof(int64_t) * (size_t)s.mesh_ndim);
    k->append(reinterpret_cast<const char*>(s.rank_ids), sizeof(int32_t) * (size_t)n);
    k->append(reinterpret_cast<const char*>(s.sbp_kind), sizeof(int32_t) * (size_t)s.mesh_ndim);
    k->append(reinterpret_cast<const char*>(s.sbp_axis), sizeof(int32_t) * (size_t)s.mesh_ndim);
}

// Element count of every rank's piece (0 for pieces a reshard never touches).
std::vector<int64_t> piece_volumes(int ndim, const int64_t* shape, const rtp_spec& spec)
{
    int64_t coords[RTP_MAX_RANKS * RTP_MAX_MESH_NDIM];
    rank_coords(spec, coords);
    std::vector<int64_t> v((size_t)num_ranks(spec));
    for (size_t r = 0; r < v.size(); ++r)
        v[r] = box_volume(ndim, rank_box(ndim, shape, spec, coords + r * RTP_MAX_MESH_NDIM));
    return v;
}

// Per thread, like the rest of the launch state (no locking).
thread_local std::unordered_map<std::string, std::vector<PlanTask>> g_plan_cache;

// plan_reshard with a per-thread cache: a repeated (shape, src, dst) reuses its
// task list (planning 64 region intersections takes about 13 us on the host).
// A new plan is checked against both layouts' piece extents before it is used
// or cached (check_task_bounds), so no planned access leaves its piece. Specs
// must have passed check_spec. The list stays valid until this thread's next
// call.
int cached_plan(const char* fn, int ndim, const int64_t* shape, const rtp_spec& src, const rtp_spec& dst,
                const std::vector<PlanTask>** out)
{
    auto& cache = g_plan_cache;
    std::string key(reinterpret_cast<const char*>(&ndim), sizeof ndim);
    key.append(reinterpret_cast<const char*>(shape), sizeof(int64_t) * (size_t)ndim);
    append_spec(&key, src);
    append_spec(&key, dst);
    auto it = cache.find(key);
    if (it == cache.end()) {
        std::vector<PlanTask> tasks;
        int st = plan_reshard(ndim, shape, src, dst, &tasks);
        if (st) return st;
        if (g_hook == RTP_HOOK_PLAN_SHIFT) {  // a planted planning mistake (tests only)
            g_hook = RTP_HOOK_NONE;
            if (!tasks.empty() && !tasks[0].dst.empty()) tasks[0].dst[0].offset += g_hook_arg;
        }
        if ((st = check_task_bounds(fn, tasks, piece_volumes(ndim, shape, src), piece_volumes(ndim, shape, dst))))
            return st;
        if (cache.size() >= 256) cache.clear();
        it = cache.emplace(std::move(key), std::move(tasks)).first;
    }
    *out = &it->second;
    return RTP_OK;
}

int reshard_impl(rtp_dtype dtype, int ndim, const int64_t* shape, const void* const* src_dev, const rtp_spec* src,
                 void* const* dst_dev, const rtp_spec* dst, rtp_stream stream)
{
    const char* fn = "rtp_reshard";
    int st = check_common(fn, dtype, ndim, shape);
    if (st) return st;
    if (!src || !dst || !src_dev || !dst_dev) return fail(RTP_EINVAL, "%s: NULL spec or buffer array", fn);
    if ((st = check_spec(ndim, *src, "rtp_reshard (src)"))) return st;
    if ((st = check_spec(ndim, *dst, "rtp_reshard (dst)"))) return st;
    const std::vector<PlanTask>* plan = nullptr;
    if ((st = cached_plan(fn, ndim, shape, *src, *dst, &plan))) return st;
    const std::vector<PlanTask>& tasks = *plan;
    int es = element_size(dtype);
    if ((st = check_pointers(fn, "source", tasks, src_dev, true, es))) return st;
    if ((st = check_pointers(fn, "destination", tasks, (const void* const*)dst_dev, false, es))) return st;
    std::vector<std::pair<uintptr_t, uintptr_t>> sr, dr;
    piece_ranges(ndim, shape, *src, src_dev, es, true, &sr);
    piece_ranges(ndim, shape, *dst, (const void* const*)dst_dev, es, false, &dr);
    if ((st = check_no_overlap(fn, std::move(sr), std::move(dr)))) return st;
    return launch_tasks(dtype, tasks, src_dev, dst_dev, stream, nullptr);
}

int shard_impl(rtp_dtype dtype, int ndim, const int64_t* shape, const void* full, const rtp_spec* spec,
               void* const* shard_dev, rtp_stream stream)
{
    const char* fn = "rtp_shard";
    int st = check_common(fn, dtype, ndim, shape);
    if (st) return st;
    if (!spec || !shard_dev) return fail(RTP_EINVAL, "%s: NULL spec or buffer array", fn);
    if ((st = check_spec(ndim, *spec, fn))) return st;
    rtp_spec whole = whole_tensor_spec();
    const std::vector<PlanTask>* plan = nullptr;
    if ((st = cached_plan(fn, ndim, shape, whole, *spec, &plan))) return st;
    const std::vector<PlanTask>& tasks = *plan;
    const void* srcs[1] = {full};
    int es = element_size(dtype);
    if ((st = check_pointers(fn, "full-tensor", tasks, srcs, true, es))) return st;
    if ((st = check_pointers(fn, "shard", tasks, (const void* const*)shard_dev, false, es))) return st;
    std::vector<std::pair<uintptr_t, uintptr_t>> sr, dr;
    piece_ranges(ndim, shape, whole, srcs, es, true, &sr);
    piece_ranges(ndim, shape, *spec, (const void* const*)shard_dev, es, false, &dr);
    if ((st = check_no_overlap(fn, std::move(sr), std::move(dr)))) return st;
    return launch_tasks(dtype, tasks, srcs, shard_dev, stream, nullptr);
}

int reshard_cost_impl(rtp_dtype dtype, int ndim, const int64_t* shape, const rtp_spec* src, const rtp_spec* dst,
                      int64_t* bytes_read, int64_t* bytes_written, int32_t* n_tasks, int32_t* n_launches)
{
    const char* fn = "rtp_reshard_cost";
    int st = check_common(fn, dtype, ndim, shape);
    if (st) return st;
    if (!src || !dst) return fail(RTP_EINVAL, "%s: NULL spec", fn);
    if ((st = check_spec(ndim, *src, "rtp_reshard_cost (src)"))) return st;
    if ((st = check_spec(ndim, *dst, "rtp_reshard_cost (dst)"))) return st;
    const std::vector<PlanTask>* plan = nullptr;
    if ((st = cached_plan(fn, ndim, shape, *src, *dst, &plan))) return st;
    const std::vector<PlanTask>& tasks = *plan;
    int64_t rd = 0, wr = 0, es = element_size(dtype);
    for (const auto& t : tasks) {
        int64_t v = t.rows * t.cols * es;
        rd += v * (int64_t)t.src.size();
        wr += v * (int64_t)t.dst.size();
    }
    if (bytes_read) *bytes_read = rd;
    if (bytes_written) *bytes_written = wr;
    if (n_tasks) *n_tasks = (int32_t)tasks.size();
    if (n_launches) *n_launches = count_launches(tasks);
    return RTP_OK;
}

int reshard_forms_impl(rtp_dtype dtype, int ndim, const int64_t* shape, const rtp_spec* src, const rtp_spec* dst,
                       int32_t* counts)
{
    const char* fn = "rtp_reshard_forms";
    int st = check_common(fn, dtype, ndim, shape);
    if (st) return st;
    if (!src || !dst || !counts) return fail(RTP_EINVAL, "%s: NULL argument", fn);
    if ((st = check_spec(ndim, *src, "rtp_reshard_forms (src)"))) return st;
    if ((st = check_spec(ndim, *dst, "rtp_reshard_forms (dst)"))) return st;
    const std::vector<PlanTask>* plan = nullptr;
    if ((st = cached_plan(fn, ndim, shape, *src, *dst, &plan))) return st;
    const std::vector<PlanTask>& tasks = *plan;
    return classify_tasks(dtype, tasks, counts);
}

}  // namespace

extern "C" {

int rtp_reshard(rtp_dtype dtype, int ndim, const int64_t* shape, const void* const* src_dev, const rtp_spec* src,
                void* const* dst_dev, const rtp_spec* dst, rtp_stream stream)
{
    return guarded("rtp_reshard", [&] { return reshard_impl(dtype, ndim, shape, src_dev, src, dst_dev, dst, stream); });
}

int rtp_shard(rtp_dtype dtype, int ndim, const int64_t* shape, const void* full, const rtp_spec* spec,
              void* const* shard_dev, rtp_stream stream)
{
    return guarded("rtp_shard", [&] { return shard_impl(dtype, ndim, shape, full, spec, shard_dev, stream); });
}

int rtp_reshard_cost(rtp_dtype dtype, int ndim, const int64_t* shape, const rtp_spec* src, const rtp_spec* dst,
                     int64_t* bytes_read, int64_t* bytes_written, int32_t* n_tasks, int32_t* n_launches)
{
    return guarded("rtp_reshard_cost", [&] {
        return reshard_cost_impl(dtype, ndim, shape, src, dst, bytes_read, bytes_written, n_tasks, n_launches);
    });
}

int rtp_reshard_forms(rtp_dtype dtype, int ndim, const int64_t* shape, const rtp_spec* src, const rtp_spec* dst,
                      int32_t* counts)
{
    return guarded("rtp_reshard_forms", [&] { return reshard_forms_impl(dtype, ndim, shape, src, dst, counts); });
}

int rtp_test_hook(int hook, int64_t arg)
{
    if (hook != RTP_HOOK_NONE && hook != RTP_HOOK_PLAN_SHIFT && hook != RTP_HOOK_FAIL_ALLOC)
        return fail(RTP_EINVAL, "rtp_test_hook: unknown hook %d", hook);
    g_hook = hook;
    g_hook_arg = arg;
    g_plan_cache.clear();  // the next reshard or shard plans afresh
    return RTP_OK;
}

}  // extern "C"
