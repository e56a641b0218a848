// Host-side sharding inference.
//
// infer_spmd follows the einsum-based rule of the Paddle "SPMD rules" design
// note: (1) the op as an einsum, (2) merge the inputs' dims_mappings per
// einsum letter (ShardingMergeForTensors), (3) read the output's mapping off
// the merged letters (GetDimsMappingForAxes). A letter that is summed away
// while sharded leaves the output partial over that mesh dim (ONNX sharding
// formalism, reduction operators: a local reduction followed by a
// cross-device one).
//
// The reshape rule follows the same note's DimTrans table (InputDim, Flatten,
// Split, Singleton).
//
// rtp_infer_sbp_signature follows the OneFlow page's walk-through of SBP
// signature inference for add_n: candidate set (split on every axis, partial
// sum, broadcast), filters, and the sort by OrderValue then CopyCost.
#include <algorithm>
#include <cstring>
#include <string>

#include "rtp_internal.h"

using namespace rtp;

namespace {

struct Parsed {
    int n_in = 0;
    std::string in[8];
    std::string out;
};

int parse_einsum(const char* s, int n_in, Parsed* p)
{
    if (!s) return fail(RTP_EINVAL, "rtp_infer_spmd: einsum is NULL");
    const char* arrow = std::strstr(s, "->");
    if (!arrow) return fail(RTP_EINVAL, "rtp_infer_spmd: einsum \"%s\" has no \"->\"", s);
    int k = 0;
    for (const char* c = s; c < arrow; ++c) {
        if (*c == ',') {
            if (++k >= 8) return fail(RTP_EUNSUPPORTED, "rtp_infer_spmd: more than 8 inputs");
            continue;
        }
        if (*c < 'a' || *c > 'z') return fail(RTP_EINVAL, "rtp_infer_spmd: bad character '%c' in \"%s\"", *c, s);
        if (p->in[k].find(*c) != std::string::npos)
            return fail(RTP_EUNSUPPORTED, "rtp_infer_spmd: letter '%c' repeated within one operand", *c);
        p->in[k].push_back(*c);
    }
    p->n_in = k + 1;
    if (p->n_in != n_in) return fail(RTP_EINVAL, "rtp_infer_spmd: einsum has %d inputs, %d mappings given", p->n_in, n_in);
    for (const char* c = arrow + 2; *c; ++c) {
        if (*c < 'a' || *c > 'z') return fail(RTP_EINVAL, "rtp_infer_spmd: bad character '%c' in \"%s\"", *c, s);
        if (p->out.find(*c) != std::string::npos) return fail(RTP_EINVAL, "rtp_infer_spmd: output letter '%c' repeated", *c);
        bool found = false;
        for (int j = 0; j < p->n_in; ++j) found = found || p->in[j].find(*c) != std::string::npos;
        if (!found) return fail(RTP_EINVAL, "rtp_infer_spmd: output letter '%c' is in no input", *c);
        p->out.push_back(*c);
    }
    return RTP_OK;
}

}  // namespace

extern "C" {

static int rtp_infer_spmd_body(const char* einsum, int n_in, const int32_t* const* in_dims_mappings, int mesh_ndim,
                               int32_t* out_dims_mapping, uint32_t* out_partial_mask, uint32_t* in_needs_reshard_mask,
                               int32_t* const* in_inferred)
{
    if (!in_dims_mappings || !out_dims_mapping || !out_partial_mask || !in_needs_reshard_mask)
        return fail(RTP_EINVAL, "rtp_infer_spmd: NULL argument");
    if (mesh_ndim < 1 || mesh_ndim > 32) return fail(RTP_EINVAL, "rtp_infer_spmd: mesh_ndim %d", mesh_ndim);
    Parsed p;
    int st = parse_einsum(einsum, n_in, &p);
    if (st) return st;
    for (int j = 0; j < n_in; ++j) {
        if (!in_dims_mappings[j] && !p.in[j].empty()) return fail(RTP_EINVAL, "rtp_infer_spmd: mapping %d is NULL", j);
        uint32_t used = 0;
        for (size_t i = 0; i < p.in[j].size(); ++i) {
            int v = in_dims_mappings[j][i];
            if (v < -1 || v >= mesh_ndim) return fail(RTP_EINVAL, "rtp_infer_spmd: input %d dim %zu maps to mesh dim %d", j, i, v);
            if (v >= 0 && ((used >> v) & 1u)) return fail(RTP_EINVAL, "rtp_infer_spmd: input %d uses mesh dim %d twice", j, v);
            if (v >= 0) used |= 1u << v;
        }
    }
    // Letters in the order they first appear in the einsum string.
    std::string order;
    for (const char* c = einsum; *c; ++c)
        if (*c >= 'a' && *c <= 'z' && order.find(*c) == std::string::npos) order.push_back(*c);
    int dim_of[26];
    for (int& d : dim_of) d = -1;
    // Step 2: merge. First sharded occurrence wins; later disagreeing inputs reshard.
    for (char L : order)
        for (int j = 0; j < n_in && dim_of[L - 'a'] == -1; ++j) {
            size_t pos = p.in[j].find(L);
            if (pos != std::string::npos) dim_of[L - 'a'] = in_dims_mappings[j][pos];
        }
    // A mesh dim shards one letter only: the earliest letter keeps it.
    uint32_t claimed = 0;
    for (char L : order) {
        int d = dim_of[L - 'a'];
        if (d < 0) continue;
        if ((claimed >> d) & 1u) dim_of[L - 'a'] = -1;
        else claimed |= 1u << d;
    }
    uint32_t needs = 0;
    for (int j = 0; j < n_in; ++j)
        for (size_t i = 0; i < p.in[j].size(); ++i) {
            int m = dim_of[p.in[j][i] - 'a'];
            if (in_dims_mappings[j][i] != m) needs |= 1u << j;
            if (in_inferred && in_inferred[j]) in_inferred[j][i] = m;
        }
    // Step 3: output mapping; contracted sharded letters leave partial sums.
    for (size_t i = 0; i < p.out.size(); ++i) out_dims_mapping[i] = dim_of[p.out[i] - 'a'];
    uint32_t partial = 0;
    for (char L : order)
        if (p.out.find(L) == std::string::npos && dim_of[L - 'a'] >= 0) partial |= 1u << dim_of[L - 'a'];
    *out_partial_mask = partial;
    *in_needs_reshard_mask = needs;
    return RTP_OK;
}

int rtp_infer_spmd(const char* einsum, int n_in, const int32_t* const* in_dims_mappings, int mesh_ndim,
                   int32_t* out_dims_mapping, uint32_t* out_partial_mask, uint32_t* in_needs_reshard_mask,
                   int32_t* const* in_inferred)
{
    return guarded("rtp_infer_spmd", [&] {
        return rtp_infer_spmd_body(einsum, n_in, in_dims_mappings, mesh_ndim, out_dims_mapping, out_partial_mask,
                                   in_needs_reshard_mask, in_inferred);
    });
}

static int rtp_infer_reshape_body(int in_ndim, const int64_t* in_shape, const int32_t* in_dims_mapping, int out_ndim,
                                  const int64_t* out_shape, int mesh_ndim, const int64_t* mesh_shape, int32_t* in_after,
                                  int32_t* out_dims_mapping)
{
    const char* fn = "rtp_infer_reshape";
    if (!in_shape || !in_dims_mapping || !out_shape || !mesh_shape || !in_after || !out_dims_mapping)
        return fail(RTP_EINVAL, "%s: NULL argument", fn);
    if (in_ndim < 1 || in_ndim > RTP_MAX_NDIM || out_ndim < 1 || out_ndim > RTP_MAX_NDIM)
        return fail(RTP_EINVAL, "%s: ranks %d -> %d", fn, in_ndim, out_ndim);
    if (mesh_ndim < 1 || mesh_ndim > RTP_MAX_MESH_NDIM) return fail(RTP_EINVAL, "%s: mesh_ndim %d", fn, mesh_ndim);
    int64_t ni = 1, no = 1;
    for (int i = 0; i < in_ndim; ++i) {
        if (in_shape[i] < 1) return fail(RTP_ESHAPE, "%s: input extent %d is %lld", fn, i, (long long)in_shape[i]);
        int v = in_dims_mapping[i];
        if (v < -1 || v >= mesh_ndim) return fail(RTP_EINVAL, "%s: dims_mapping[%d] = %d", fn, i, v);
        ni *= in_shape[i];
        in_after[i] = v;
    }
    for (int o = 0; o < out_ndim; ++o) {
        if (out_shape[o] < 1) return fail(RTP_ESHAPE, "%s: output extent %d is %lld", fn, o, (long long)out_shape[o]);
        no *= out_shape[o];
        out_dims_mapping[o] = -1;
    }
    if (ni != no) return fail(RTP_ESHAPE, "%s: %lld elements cannot become %lld", fn, (long long)ni, (long long)no);
    int i = 0, o = 0;
    while (i < in_ndim || o < out_ndim) {
        const bool out_unit = o < out_ndim && out_shape[o] == 1;
        const bool in_unit = i < in_ndim && in_shape[i] == 1;
        if (out_unit && !in_unit) {  // Singleton output dim
            ++o;
            continue;
        }
        if (in_unit && !out_unit) {  // unit input dim disappears with its split
            in_after[i++] = -1;
            continue;
        }
        // A group of input dims and output dims with equal products.
        const int gi = i, go = o;
        int64_t a = in_shape[i++], b = out_shape[o++];
        while (a != b) {
            if (a < b) a *= in_shape[i++];
            else b *= out_shape[o++];
        }
        int lead_in = gi, lead_out = go;
        while (lead_in + 1 < i && in_shape[lead_in] == 1) ++lead_in;
        while (lead_out + 1 < o && out_shape[lead_out] == 1) ++lead_out;
        for (int k = gi; k < i; ++k)
            if (k != lead_in) in_after[k] = -1;
        const int d = in_after[lead_in];
        if (d < 0) continue;
        const int64_t n = mesh_shape[d];
        int64_t inner_in = 1, inner_out = 1;
        for (int k = lead_in + 1; k < i; ++k) inner_in *= in_shape[k];
        for (int k = lead_out + 1; k < o; ++k) inner_out *= out_shape[k];
        // Each rank's run of the flattened group, before and after.
        const int64_t L = in_shape[lead_in], E = out_shape[lead_out];
        const int64_t wl = (L + n - 1) / n, we = (E + n - 1) / n;
        bool keep = true;
        for (int64_t r = 0; r < n && keep; ++r) {
            const int64_t x0 = (r * wl < L ? r * wl : L) * inner_in, x1 = ((r + 1) * wl < L ? (r + 1) * wl : L) * inner_in;
            const int64_t y0 = (r * we < E ? r * we : E) * inner_out, y1 = ((r + 1) * we < E ? (r + 1) * we : E) * inner_out;
            keep = x0 == y0 && x1 == y1;
        }
        if (keep) out_dims_mapping[lead_out] = d;
        else in_after[lead_in] = -1;
    }
    return RTP_OK;
}

int rtp_infer_reshape(int in_ndim, const int64_t* in_shape, const int32_t* in_dims_mapping, int out_ndim,
                      const int64_t* out_shape, int mesh_ndim, const int64_t* mesh_shape, int32_t* in_after,
                      int32_t* out_dims_mapping)
{
    return guarded("rtp_infer_reshape", [&] {
        return rtp_infer_reshape_body(in_ndim, in_shape, in_dims_mapping, out_ndim, out_shape, mesh_ndim, mesh_shape,
                                      in_after, out_dims_mapping);
    });
}

}  // extern "C"

static int rtp_infer_sbp_signature_body(int n_in, int ndim, const int64_t* shape, int elem_bytes, int mesh_ndim,
                                        const int32_t* in_kinds, const int32_t* in_axes, const int32_t* constraint_kinds,
                                        const int32_t* constraint_axes, int32_t* out_kinds, int32_t* out_axes,
                                        double* out_cost, int32_t* out_order)
{
    const char* fn = "rtp_infer_sbp_signature";
    if (!shape || !in_kinds || !in_axes || !out_kinds || !out_axes) return fail(RTP_EINVAL, "%s: NULL argument", fn);
    if (n_in < 1 || ndim < 1 || ndim > RTP_MAX_NDIM || elem_bytes < 1)
        return fail(RTP_EINVAL, "%s: n_in %d, ndim %d, elem_bytes %d", fn, n_in, ndim, elem_bytes);
    if (mesh_ndim < 1 || mesh_ndim > RTP_MAX_MESH_NDIM) return fail(RTP_EINVAL, "%s: mesh_ndim %d", fn, mesh_ndim);
    if ((constraint_kinds == nullptr) != (constraint_axes == nullptr))
        return fail(RTP_EINVAL, "%s: constraint kinds and axes go together", fn);
    int64_t bytes = elem_bytes;
    for (int a = 0; a < ndim; ++a) bytes *= shape[a];
    // per input: kind/axis per mesh dim; "same" compares whole ND-SBPs
    auto entry_ok = [&](int k, int ax) {
        return k == RTP_SBP_BROADCAST || k == RTP_SBP_PARTIAL_SUM || k == RTP_SBP_PARTIAL_MIN ||
               k == RTP_SBP_PARTIAL_MAX || (k == RTP_SBP_SPLIT && ax >= 0);
    };
    for (int j = 0; j < n_in; ++j)
        for (int d = 0; d < mesh_ndim; ++d)
            if (!entry_ok(in_kinds[j * mesh_ndim + d], in_axes[j * mesh_ndim + d]))
                return fail(RTP_EINVAL, "%s: input %d mesh dim %d has a bad SBP", fn, j, d);
    // 1D candidates: S(0..ndim-1), P, B
    const int n1 = ndim + 2;
    auto kind_of = [&](int c) { return c < ndim ? RTP_SBP_SPLIT : (c == ndim ? RTP_SBP_PARTIAL_SUM : RTP_SBP_BROADCAST); };
    auto axis_of = [&](int c) { return c < ndim ? c : -1; };
    int64_t total = 1;
    for (int d = 0; d < mesh_ndim; ++d) total *= n1;
    bool found = false;
    int64_t best = -1;
    int best_order = 0;
    double best_cost = 0;
    for (int64_t cand = 0; cand < total; ++cand) {
        int ck[RTP_MAX_MESH_NDIM], ca[RTP_MAX_MESH_NDIM];
        int64_t rem = cand;
        for (int d = mesh_ndim - 1; d >= 0; --d) {
            int c = (int)(rem % n1);
            rem /= n1;
            ck[d] = kind_of(c);
            ca[d] = axis_of(c);
        }
        // filter: split axes must be axes of the tensor (always true for these
        // candidates); and the constraint, when given
        bool keep = true;
        for (int d = 0; d < mesh_ndim && keep; ++d) {
            if (ck[d] == RTP_SBP_SPLIT && ca[d] >= ndim) keep = false;
            if (constraint_kinds && (constraint_kinds[d] != ck[d] || (ck[d] == RTP_SBP_SPLIT && constraint_axes[d] != ca[d])))
                keep = false;
        }
        if (!keep) continue;
        int order = 0;
        double cost = 0;
        for (int j = 0; j < n_in; ++j) {
            bool same = true, pb = false;
            for (int d = 0; d < mesh_ndim; ++d) {
                const int k = in_kinds[j * mesh_ndim + d], ax = in_axes[j * mesh_ndim + d];
                if (k != ck[d] || (k == RTP_SBP_SPLIT && ax != ca[d])) same = false;
                if (k != RTP_SBP_SPLIT) pb = true;  // broadcast or partial
            }
            if (same) {
                if (!constraint_kinds) order -= 10;
                continue;
            }
            cost += pb ? 1e30 : (double)bytes;
        }
        if (!found || order < best_order || (order == best_order && cost < best_cost)) {
            found = true;
            best = cand;
            best_order = order;
            best_cost = cost;
        }
    }
    if (!found) return fail(RTP_ECONFLICT, "%s: no candidate signature satisfies the constraint", fn);
    int64_t rem = best;
    for (int d = mesh_ndim - 1; d >= 0; --d) {
        int c = (int)(rem % n1);
        rem /= n1;
        out_kinds[d] = kind_of(c);
        out_axes[d] = axis_of(c);
    }
    if (out_cost) *out_cost = best_cost;
    if (out_order) *out_order = best_order;
    return RTP_OK;
}

extern "C" int rtp_infer_sbp_signature(int n_in, int ndim, const int64_t* shape, int elem_bytes, int mesh_ndim,
                                       const int32_t* in_kinds, const int32_t* in_axes, const int32_t* constraint_kinds,
                                       const int32_t* constraint_axes, int32_t* out_kinds, int32_t* out_axes,
                                       double* out_cost, int32_t* out_order)
{
    return guarded("rtp_infer_sbp_signature", [&] {
        return rtp_infer_sbp_signature_body(n_in, ndim, shape, elem_bytes, mesh_ndim, in_kinds, in_axes,
                                            constraint_kinds, constraint_axes, out_kinds, out_axes, out_cost,
                                            out_order);
    });
}

// ---- ONNX sharding checker: broadcast n-ary element-wise operators ----------------
//
// "ONNX multi-device proposal", operator groups, broadcast n-ary element-wise
// operators: inputs must agree on every non-broadcast axis, a broadcast axis
// of extent 1 must be held whole wherever it is used, and the output shard of
// a device is what it can compute from the input shards it holds; with two or
// more broadcast axes a shard's devices are the intersection of the devices of
// the input shards it reads (the Add([M,1],[1,N]) example).

namespace {

struct Interval {
    int64_t lo, hi;
    bool operator<(const Interval& o) const { return lo < o.lo || (lo == o.lo && hi < o.hi); }
    bool operator==(const Interval& o) const { return lo == o.lo && hi == o.hi; }
};

}  // namespace

static int rtp_infer_broadcast_body(int n_in, const int32_t* in_ndims, const int64_t* const* in_shapes,
                                    const rtp_spec* in_specs, int* out_ndim, int64_t* out_shape, rtp_spec* out_spec)
{
    using namespace rtp;
    const char* fn = "rtp_infer_broadcast";
    if (n_in < 1 || !in_ndims || !in_shapes || !in_specs || !out_ndim || !out_shape || !out_spec)
        return fail(RTP_EINVAL, "%s: NULL argument or no input", fn);
    int nd = 0;
    for (int k = 0; k < n_in; ++k) {
        if (in_ndims[k] < 1 || in_ndims[k] > RTP_MAX_NDIM || !in_shapes[k])
            return fail(RTP_EINVAL, "%s: input %d has rank %d", fn, k, in_ndims[k]);
        if (in_ndims[k] > nd) nd = in_ndims[k];
        int st = check_spec(in_ndims[k], in_specs[k], "input");
        if (st) return st;
        for (int d = 0; d < in_specs[k].mesh_ndim; ++d)
            if (is_partial(in_specs[k].sbp_kind[d]))
                return fail(RTP_EUNSUPPORTED, "%s: input %d is partial; the ONNX operator rules have no partial "
                            "layouts", fn, k);
    }
    const int64_t R = num_ranks(in_specs[0]);
    for (int k = 1; k < n_in; ++k)
        if (num_ranks(in_specs[k]) != R)
            return fail(RTP_EINVAL, "%s: inputs live on %lld and %lld ranks", fn, (long long)R,
                        (long long)num_ranks(in_specs[k]));
    // multidirectional broadcast of the shapes (trailing dims aligned)
    int64_t shape[RTP_MAX_NDIM];
    for (int d = 0; d < nd; ++d) {
        int64_t e = 1;
        for (int k = 0; k < n_in; ++k) {
            const int dk = d - (nd - in_ndims[k]);
            if (dk < 0) continue;
            const int64_t x = in_shapes[k][dk];
            if (x < 1) return fail(RTP_ESHAPE, "%s: extent %lld (must be >= 1)", fn, (long long)x);
            if (x == 1) continue;
            if (e != 1 && e != x)
                return fail(RTP_ESHAPE, "%s: extents %lld and %lld on output dim %d do not broadcast", fn, (long long)e,
                            (long long)x, d);
            e = x;
        }
        shape[d] = e;  // 1 when every input has extent 1 there
    }
    // each rank's output box: the intersection over inputs of what its pieces allow
    std::vector<Box> box((size_t)R);
    std::vector<bool> empty((size_t)R, false);
    std::vector<int64_t> coords((size_t)R * RTP_MAX_MESH_NDIM);
    for (int64_t r = 0; r < R; ++r) {
        for (int d = 0; d < nd; ++d) {
            box[r].lo[d] = 0;
            box[r].hi[d] = shape[d];
        }
    }
    for (int k = 0; k < n_in; ++k) {
        rank_coords(in_specs[k], coords.data());
        for (int64_t r = 0; r < R; ++r) {
            const Box b = rank_box(in_ndims[k], in_shapes[k], in_specs[k], coords.data() + r * RTP_MAX_MESH_NDIM);
            for (int dk = 0; dk < in_ndims[k]; ++dk) {
                const int d = dk + (nd - in_ndims[k]);
                if (in_shapes[k][dk] == shape[d]) {  // a non-broadcast axis: intersect
                    box[r].lo[d] = std::max(box[r].lo[d], b.lo[dk]);
                    box[r].hi[d] = std::min(box[r].hi[d], b.hi[dk]);
                } else if (b.hi[dk] <= b.lo[dk]) {   // extent 1 broadcast, but this rank holds none of it
                    empty[r] = true;
                }
            }
        }
    }
    for (int64_t r = 0; r < R; ++r)
        for (int d = 0; d < nd; ++d)
            if (box[r].hi[d] <= box[r].lo[d] && shape[d] > 0) empty[r] = true;
    // an input laid out over the whole output shape whose pieces are exactly the
    // boxes is the answer as it stands (the usual case: inputs sharded alike)
    for (int k = 0; k < n_in; ++k) {
        if (in_ndims[k] != nd || !std::equal(shape, shape + nd, in_shapes[k])) continue;
        rank_coords(in_specs[k], coords.data());
        bool same = true;
        for (int64_t r = 0; r < R && same; ++r) {
            const Box b = rank_box(nd, shape, in_specs[k], coords.data() + r * RTP_MAX_MESH_NDIM);
            // a rank that computes nothing must hold an empty piece; the others the same box
            const bool none = empty[r] || box_volume(nd, box[r]) == 0;
            if (none) {
                same = box_volume(nd, b) == 0;
            } else {
                for (int d = 0; d < nd; ++d)
                    if (b.lo[d] != box[r].lo[d] || b.hi[d] != box[r].hi[d]) same = false;
            }
        }
        if (same) {
            *out_ndim = nd;
            for (int d = 0; d < nd; ++d) out_shape[d] = shape[d];
            *out_spec = in_specs[k];
            clear_error();
            return RTP_OK;
        }
    }
    auto same_box = [&](int64_t x, int64_t y) {
        for (int d = 0; d < nd; ++d)
            if (box[x].lo[d] != box[y].lo[d] || box[x].hi[d] != box[y].hi[d]) return false;
        return true;
    };
    // distinct boxes must not overlap (else no layout describes them)
    std::vector<int64_t> distinct;
    for (int64_t r = 0; r < R; ++r) {
        if (empty[r]) continue;
        bool seen = false;
        for (int64_t x : distinct) seen |= same_box(x, r);
        if (!seen) distinct.push_back(r);
    }
    for (size_t i = 0; i < distinct.size(); ++i)
        for (size_t j = i + 1; j < distinct.size(); ++j) {
            bool meet = true;
            for (int d = 0; d < nd; ++d)
                meet &= std::max(box[distinct[i]].lo[d], box[distinct[j]].lo[d]) <
                        std::min(box[distinct[i]].hi[d], box[distinct[j]].hi[d]);
            if (meet)
                return fail(RTP_EUNSUPPORTED, "%s: the output pieces of ranks %lld and %lld overlap without being "
                            "equal", fn, (long long)distinct[i], (long long)distinct[j]);
        }
    // disjoint pieces cover the output iff their volumes add up
    int64_t total = 1, covered = 0;
    for (int d = 0; d < nd; ++d) total *= shape[d];
    for (int64_t x : distinct) covered += box_volume(nd, box[x]);
    if (covered != total)
        return fail(RTP_ECONFLICT, "%s: some output elements have no device holding all of their inputs (the inputs "
                    "are sharded incompatibly)", fn);
    for (int64_t r = 0; r < R; ++r)
        if (empty[r]) return fail(RTP_EUNSUPPORTED, "%s: rank %lld computes nothing", fn, (long long)r);
    // a grid of cells, each on the same number of ranks
    std::vector<std::vector<Interval>> cuts((size_t)nd);
    int64_t cells = 1;
    for (int d = 0; d < nd; ++d) {
        for (int64_t r = 0; r < R; ++r) cuts[d].push_back({box[r].lo[d], box[r].hi[d]});
        std::sort(cuts[d].begin(), cuts[d].end());
        cuts[d].erase(std::unique(cuts[d].begin(), cuts[d].end()), cuts[d].end());
        cells *= (int64_t)cuts[d].size();
    }
    if (cells != (int64_t)distinct.size())
        return fail(RTP_EUNSUPPORTED, "%s: the output pieces do not form a grid", fn);
    std::vector<std::vector<int>> holders((size_t)cells);
    for (int64_t r = 0; r < R; ++r) {
        int64_t cell = 0;
        for (int d = 0; d < nd; ++d) {
            const int64_t i = std::lower_bound(cuts[d].begin(), cuts[d].end(), Interval{box[r].lo[d], box[r].hi[d]}) -
                              cuts[d].begin();
            cell = cell * (int64_t)cuts[d].size() + i;
        }
        holders[cell].push_back((int)r);
    }
    const size_t rep = holders[0].size();
    for (const auto& h : holders)
        if (h.size() != rep)
            return fail(RTP_EUNSUPPORTED, "%s: output pieces are held by unequal numbers of ranks", fn);
    // the output layout: split mesh dims (output axes in order, outer first), then
    // one broadcast mesh dim for the replicas
    rtp_spec o;
    std::memset(&o, 0, sizeof o);
    for (int d = 0; d < nd; ++d) {
        if (cuts[d].size() <= 1) continue;
        if (o.mesh_ndim == RTP_MAX_MESH_NDIM)
            return fail(RTP_EUNSUPPORTED, "%s: more than %d split output axes", fn, RTP_MAX_MESH_NDIM);
        o.mesh_shape[o.mesh_ndim] = (int64_t)cuts[d].size();
        o.sbp_kind[o.mesh_ndim] = RTP_SBP_SPLIT;
        o.sbp_axis[o.mesh_ndim] = d;
        ++o.mesh_ndim;
    }
    if (rep > 1 || o.mesh_ndim == 0) {
        if (o.mesh_ndim == RTP_MAX_MESH_NDIM)
            return fail(RTP_EUNSUPPORTED, "%s: too many mesh dims for the output", fn);
        o.mesh_shape[o.mesh_ndim] = (int64_t)rep;
        o.sbp_kind[o.mesh_ndim] = RTP_SBP_BROADCAST;
        ++o.mesh_ndim;
    }
    for (int64_t c = 0; c < cells; ++c) {
        std::vector<int> h = holders[c];
        std::sort(h.begin(), h.end());
        for (size_t t = 0; t < rep; ++t) o.rank_ids[c * rep + t] = h[t];
    }
    // the spec must reproduce the boxes (the cuts follow this library's split rule)
    rank_coords(o, coords.data());
    for (int64_t r = 0; r < R; ++r) {
        const Box b = rank_box(nd, shape, o, coords.data() + r * RTP_MAX_MESH_NDIM);
        for (int d = 0; d < nd; ++d)
            if (b.lo[d] != box[r].lo[d] || b.hi[d] != box[r].hi[d])
                return fail(RTP_EUNSUPPORTED, "%s: the output cuts of dim %d are not the even split this library "
                            "uses", fn, d);
    }
    *out_ndim = nd;
    for (int d = 0; d < nd; ++d) out_shape[d] = shape[d];
    *out_spec = o;
    clear_error();
    return RTP_OK;
}

extern "C" int rtp_infer_broadcast(int n_in, const int32_t* in_ndims, const int64_t* const* in_shapes,
                                   const rtp_spec* in_specs, int* out_ndim, int64_t* out_shape, rtp_spec* out_spec)
{
    return guarded("rtp_infer_broadcast", [&] {
        return rtp_infer_broadcast_body(n_in, in_ndims, in_shapes, in_specs, out_ndim, out_shape, out_spec);
    });
}
