// Layout specs: error reporting, the Paddle and ONNX front-ends, and the
// geometry of each rank's piece.
//
// Geometry follows the split rule of the "ONNX multi-device proposal" page
// (index rule for multi-axis splits: the first split is the outer loop) and
// the OneFlow 2D SBP example (mesh dim 0 is the outer level). Uneven extents,
// which that page leaves to the backend, are cut into ceil-sized pieces level
// by level.
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "rtp_internal.h"

namespace rtp {

namespace {
// A fixed buffer, so that reporting an error (an allocation failure among
// them) never allocates.
thread_local char g_last_error[1024];
}

int fail(int status, const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return status;
}

void clear_error() { g_last_error[0] = 0; }

int64_t num_ranks(const rtp_spec& s)
{
    int64_t n = 1;
    for (int d = 0; d < s.mesh_ndim; ++d) n *= s.mesh_shape[d];
    return n;
}

int check_spec(int ndim, const rtp_spec& s, const char* what)
{
    if (ndim < 1 || ndim > RTP_MAX_NDIM) return fail(RTP_EINVAL, "%s: tensor rank %d outside [1, %d]", what, ndim, RTP_MAX_NDIM);
    if (s.mesh_ndim < 1 || s.mesh_ndim > RTP_MAX_MESH_NDIM)
        return fail(RTP_EINVAL, "%s: mesh_ndim %d outside [1, %d]", what, s.mesh_ndim, RTP_MAX_MESH_NDIM);
    int64_t n = 1;
    for (int d = 0; d < s.mesh_ndim; ++d) {
        if (s.mesh_shape[d] < 1) return fail(RTP_EINVAL, "%s: mesh dim %d has size %lld", what, d, (long long)s.mesh_shape[d]);
        n *= s.mesh_shape[d];
        if (n > RTP_MAX_RANKS) return fail(RTP_EUNSUPPORTED, "%s: more than %d ranks", what, RTP_MAX_RANKS);
    }
    bool seen[RTP_MAX_RANKS] = {};
    for (int64_t p = 0; p < n; ++p) {
        int r = s.rank_ids[p];
        if (r < 0 || r >= n || seen[r])
            return fail(RTP_EINVAL, "%s: rank_ids must be a permutation of 0..%lld", what, (long long)(n - 1));
        seen[r] = true;
    }
    for (int d = 0; d < s.mesh_ndim; ++d) {
        int k = s.sbp_kind[d];
        if (k != RTP_SBP_SPLIT && k != RTP_SBP_BROADCAST && !is_partial(k))
            return fail(RTP_EINVAL, "%s: mesh dim %d has unknown sbp kind %d", what, d, k);
        for (int e = 0; e < d; ++e)
            if (is_partial(k) && is_partial(s.sbp_kind[e]) && s.sbp_kind[e] != k)
                return fail(RTP_EUNSUPPORTED, "%s: mesh dims %d and %d are partial with different reductions", what, e, d);
        if (k == RTP_SBP_SPLIT && (s.sbp_axis[d] < 0 || s.sbp_axis[d] >= ndim))
            return fail(RTP_EINVAL, "%s: mesh dim %d splits axis %d of a rank-%d tensor", what, d, s.sbp_axis[d], ndim);
    }
    return RTP_OK;
}

bool is_partial(int k) { return k == RTP_SBP_PARTIAL_SUM || k == RTP_SBP_PARTIAL_MIN || k == RTP_SBP_PARTIAL_MAX; }

int partial_reduction(const rtp_spec& s)
{
    for (int d = 0; d < s.mesh_ndim; ++d) {
        if (s.sbp_kind[d] == RTP_SBP_PARTIAL_MIN) return RED_MIN;
        if (s.sbp_kind[d] == RTP_SBP_PARTIAL_MAX) return RED_MAX;
    }
    return RED_SUM;
}

void rank_coords(const rtp_spec& s, int64_t* coords)
{
    int64_t n = num_ranks(s);
    for (int64_t p = 0; p < n; ++p) {
        int r = s.rank_ids[p];
        int64_t rem = p;
        for (int d = s.mesh_ndim - 1; d >= 0; --d) {
            coords[r * RTP_MAX_MESH_NDIM + d] = rem % s.mesh_shape[d];
            rem /= s.mesh_shape[d];
        }
    }
}

Box rank_box(int ndim, const int64_t* shape, const rtp_spec& s, const int64_t* c)
{
    Box b;
    for (int a = 0; a < ndim; ++a) {
        b.lo[a] = 0;
        b.hi[a] = shape[a];
    }
    b.holds_value = true;
    b.b_rep = true;
    b.pidx = 0;
    for (int d = 0; d < s.mesh_ndim; ++d) {
        switch (s.sbp_kind[d]) {
        case RTP_SBP_SPLIT: {
            int a = s.sbp_axis[d];
            int64_t len = b.hi[a] - b.lo[a], n = s.mesh_shape[d];
            int64_t w = (len + n - 1) / n;
            int64_t first = c[d] * w < len ? c[d] * w : len;
            int64_t last = (c[d] + 1) * w < len ? (c[d] + 1) * w : len;
            b.hi[a] = b.lo[a] + last;
            b.lo[a] += first;
            break;
        }
        case RTP_SBP_BROADCAST:
            if (c[d] != 0) b.b_rep = false;
            break;
        default:  // partial (sum, min or max)
            if (c[d] != 0) b.holds_value = false;
            b.pidx = b.pidx * s.mesh_shape[d] + c[d];
            break;
        }
    }
    return b;
}

int64_t box_volume(int ndim, const Box& b)
{
    int64_t v = 1;
    for (int a = 0; a < ndim; ++a) v *= b.hi[a] - b.lo[a];
    return v;
}

rtp_spec whole_tensor_spec()
{
    rtp_spec s;
    std::memset(&s, 0, sizeof s);
    s.mesh_ndim = 1;
    s.mesh_shape[0] = 1;
    s.rank_ids[0] = 0;
    s.sbp_kind[0] = RTP_SBP_BROADCAST;
    s.sbp_axis[0] = -1;
    return s;
}

}  // namespace rtp

using namespace rtp;

extern "C" {

const char* rtp_last_error(void) { return g_last_error; }

const char* rtp_version(void) { return "rtp 0.1 (sm_103a)"; }

int rtp_spec_check(int ndim, const rtp_spec* spec)
{
    if (!spec) return fail(RTP_EINVAL, "rtp_spec_check: spec is NULL");
    return check_spec(ndim, *spec, "rtp_spec_check");
}

int rtp_spec_from_dims_mapping(int ndim, const int32_t* dims_mapping, int mesh_ndim, const int64_t* mesh_shape,
                               const int32_t* rank_ids, uint32_t partial_mask, rtp_spec* out)
{
    if (!dims_mapping || !mesh_shape || !out) return fail(RTP_EINVAL, "rtp_spec_from_dims_mapping: NULL argument");
    if (mesh_ndim < 1 || mesh_ndim > RTP_MAX_MESH_NDIM)
        return fail(RTP_EINVAL, "rtp_spec_from_dims_mapping: mesh_ndim %d outside [1, %d]", mesh_ndim, RTP_MAX_MESH_NDIM);
    if (ndim < 1 || ndim > RTP_MAX_NDIM) return fail(RTP_EINVAL, "rtp_spec_from_dims_mapping: ndim %d", ndim);
    if (partial_mask >> mesh_ndim) return fail(RTP_EINVAL, "rtp_spec_from_dims_mapping: partial_mask names a missing mesh dim");
    rtp_spec s;
    std::memset(&s, 0, sizeof s);
    s.mesh_ndim = mesh_ndim;
    int64_t n = 1;
    for (int d = 0; d < mesh_ndim; ++d) {
        s.mesh_shape[d] = mesh_shape[d];
        if (mesh_shape[d] < 1) return fail(RTP_EINVAL, "rtp_spec_from_dims_mapping: mesh dim %d has size %lld", d, (long long)mesh_shape[d]);
        n *= mesh_shape[d];
        if (n > RTP_MAX_RANKS) return fail(RTP_EUNSUPPORTED, "rtp_spec_from_dims_mapping: more than %d ranks", RTP_MAX_RANKS);
        s.sbp_kind[d] = (partial_mask >> d) & 1u ? RTP_SBP_PARTIAL_SUM : RTP_SBP_BROADCAST;
        s.sbp_axis[d] = -1;
    }
    for (int64_t p = 0; p < n; ++p) s.rank_ids[p] = rank_ids ? rank_ids[p] : (int32_t)p;
    for (int i = 0; i < ndim; ++i) {
        int j = dims_mapping[i];
        if (j == -1) continue;
        if (j < -1 || j >= mesh_ndim) return fail(RTP_EINVAL, "rtp_spec_from_dims_mapping: dims_mapping[%d] = %d", i, j);
        if (s.sbp_kind[j] == RTP_SBP_PARTIAL_SUM)
            return fail(RTP_EINVAL, "rtp_spec_from_dims_mapping: mesh dim %d is both split and partial", j);
        if (s.sbp_kind[j] == RTP_SBP_SPLIT)
            return fail(RTP_EINVAL, "rtp_spec_from_dims_mapping: tensor dims %d and %d both on mesh dim %d", s.sbp_axis[j], i, j);
        s.sbp_kind[j] = RTP_SBP_SPLIT;
        s.sbp_axis[j] = i;
    }
    int st = check_spec(ndim, s, "rtp_spec_from_dims_mapping");
    if (st) return st;
    *out = s;
    return RTP_OK;
}

static int rtp_spec_from_onnx_body(int ndim, int n_device, const int64_t* device, int n_groups, const int64_t* group_keys,
                                   const int32_t* group_sizes, const int64_t* group_devices, int n_sharded, const int64_t* axes,
                                   const int64_t* num_shards, rtp_spec* out)
{
    const char* fn = "rtp_spec_from_onnx";
    if (!device || !out || n_device < 1) return fail(RTP_EINVAL, "%s: empty device list", fn);
    if (n_groups < 0 || (n_groups > 0 && (!group_keys || !group_sizes || !group_devices)))
        return fail(RTP_EINVAL, "%s: malformed device_map", fn);
    if (n_sharded < 0 || (n_sharded > 0 && (!axes || !num_shards))) return fail(RTP_EINVAL, "%s: malformed sharded_dim", fn);
    if (n_sharded + 1 > RTP_MAX_MESH_NDIM) return fail(RTP_EUNSUPPORTED, "%s: more than %d sharded dims", fn, RTP_MAX_MESH_NDIM - 1);
    if (ndim < 1 || ndim > RTP_MAX_NDIM) return fail(RTP_EINVAL, "%s: ndim %d", fn, ndim);
    // Resolve every entry of `device` to its list of ranks.
    std::vector<std::vector<int64_t>> members(n_device);
    for (int s = 0; s < n_device; ++s) {
        if (device[s] >= 0) {
            members[s].push_back(device[s]);
            continue;
        }
        int64_t off = 0;
        bool found = false;
        for (int g = 0; g < n_groups; ++g) {
            if (group_sizes[g] < 1) return fail(RTP_EINVAL, "%s: group %lld is empty", fn, (long long)group_keys[g]);
            if (group_keys[g] == device[s]) {
                members[s].assign(group_devices + off, group_devices + off + group_sizes[g]);
                found = true;
                break;
            }
            off += group_sizes[g];
        }
        if (!found) return fail(RTP_EINVAL, "%s: device key %lld not in device_map", fn, (long long)device[s]);
    }
    for (int s = 1; s < n_device; ++s)
        if (members[s].size() != members[0].size())
            return fail(RTP_EUNSUPPORTED, "%s: device groups of unequal size (%zu vs %zu)", fn, members[s].size(), members[0].size());
    int64_t pieces = 1;
    for (int k = 0; k < n_sharded; ++k) {
        if (num_shards[k] < 1) return fail(RTP_EINVAL, "%s: num_shards %lld", fn, (long long)num_shards[k]);
        pieces *= num_shards[k];
        if (pieces > RTP_MAX_RANKS) return fail(RTP_EUNSUPPORTED, "%s: more than %d pieces", fn, RTP_MAX_RANKS);
    }
    if (pieces != n_device)
        return fail(RTP_ESHAPE, "%s: %lld pieces for %d device entries", fn, (long long)pieces, n_device);
    rtp_spec sp;
    std::memset(&sp, 0, sizeof sp);
    int md = 0;
    bool axis_used[RTP_MAX_NDIM] = {};
    for (int k = 0; k < n_sharded; ++k) {
        int64_t a = axes[k];
        if (a < -ndim || a >= ndim) return fail(RTP_EINVAL, "%s: axis %lld outside [-%d, %d]", fn, (long long)a, ndim, ndim - 1);
        if (a < 0) a += ndim;
        if (axis_used[a]) return fail(RTP_EUNSUPPORTED, "%s: axis %lld listed twice", fn, (long long)a);
        axis_used[a] = true;
        sp.mesh_shape[md] = num_shards[k];
        sp.sbp_kind[md] = RTP_SBP_SPLIT;
        sp.sbp_axis[md] = (int32_t)a;
        ++md;
    }
    int64_t g = (int64_t)members[0].size();
    if (g > 1 || md == 0) {
        sp.mesh_shape[md] = g;
        sp.sbp_kind[md] = RTP_SBP_BROADCAST;
        sp.sbp_axis[md] = -1;
        ++md;
    }
    sp.mesh_ndim = md;
    if (pieces * g > RTP_MAX_RANKS) return fail(RTP_EUNSUPPORTED, "%s: more than %d ranks", fn, RTP_MAX_RANKS);
    for (int s = 0; s < n_device; ++s)
        for (int64_t t = 0; t < g; ++t) {
            int64_t r = members[s][t];
            if (r < 0 || r >= pieces * g) return fail(RTP_EINVAL, "%s: rank id %lld outside 0..%lld", fn, (long long)r, (long long)(pieces * g - 1));
            sp.rank_ids[s * g + t] = (int32_t)r;
        }
    int st = check_spec(ndim, sp, fn);
    if (st) return st;
    *out = sp;
    return RTP_OK;
}

int rtp_spec_from_onnx(int ndim, int n_device, const int64_t* device, int n_groups, const int64_t* group_keys,
                       const int32_t* group_sizes, const int64_t* group_devices, int n_sharded, const int64_t* axes,
                       const int64_t* num_shards, rtp_spec* out)
{
    return guarded("rtp_spec_from_onnx", [&] {
        return rtp_spec_from_onnx_body(ndim, n_device, device, n_groups, group_keys, group_sizes, group_devices,
                                       n_sharded, axes, num_shards, out);
    });
}

int rtp_shard_box(int ndim, const int64_t* shape, const rtp_spec* spec, int rank, int64_t* lo, int64_t* hi,
                  int32_t* holds_value)
{
    if (!shape || !spec || !lo || !hi) return fail(RTP_EINVAL, "rtp_shard_box: NULL argument");
    int st = check_spec(ndim, *spec, "rtp_shard_box");
    if (st) return st;
    for (int a = 0; a < ndim; ++a)
        if (shape[a] < 0) return fail(RTP_ESHAPE, "rtp_shard_box: negative extent");
    if (rank < 0 || rank >= num_ranks(*spec)) return fail(RTP_EINVAL, "rtp_shard_box: rank %d outside the mesh", rank);
    int64_t coords[RTP_MAX_RANKS * RTP_MAX_MESH_NDIM];
    rank_coords(*spec, coords);
    Box b = rank_box(ndim, shape, *spec, coords + rank * RTP_MAX_MESH_NDIM);
    for (int a = 0; a < ndim; ++a) {
        lo[a] = b.lo[a];
        hi[a] = b.hi[a];
    }
    if (holds_value) *holds_value = b.holds_value ? 1 : 0;
    return RTP_OK;
}

int rtp_shard_shape(int ndim, const int64_t* shape, const rtp_spec* spec, int rank, int64_t* out_shape)
{
    int64_t lo[RTP_MAX_NDIM], hi[RTP_MAX_NDIM];
    if (!out_shape) return fail(RTP_EINVAL, "rtp_shard_shape: NULL argument");
    int st = rtp_shard_box(ndim, shape, spec, rank, lo, hi, nullptr);
    if (st) return st;
    for (int a = 0; a < ndim; ++a) out_shape[a] = hi[a] - lo[a];
    return RTP_OK;
}

}  // extern "C"
