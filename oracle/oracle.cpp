// Oracle: a plain, slow, single-threaded CPU statement of what the resharding
// library computes. It is test infrastructure. Only the tests, the smoke check
// and the benchmark's CPU-baseline leg load it. It shares no code, header or
// table with the CUDA library and must stay that way.
//
// What each function follows (page title, section):
//   * shard geometry: "ONNX multi-device proposal ... ShardingSpec" (zskr.cn),
//     sections "Sharding as a Split" and "index rule for multi-axis splits"
//     (the nested loop: axis a outer, axis b inner, shards appended in that
//     order); "Sharding as a Broadcast" and "mixing split and broadcast"
//     (device_map groups); OneFlow SBP page (szpsdzdm.com), 2D SBP
//     (broadcast, split(0)) on ranks [[0,1],[2,3]]: mesh dim 0 is the outer
//     level, mesh dim 1 the inner one.
//   * partial sum: OneFlow SBP page, definition of partial: the logical tensor
//     is the element-wise sum of the per-device tensors.
//   * infer_spmd: Paddle "SPMD rules" page (contextqmd.com), steps 1-3 of the
//     einsum-based rule (einsum, ShardingMergeForTensors,
//     GetDimsMappingForAxes); reductions over a sharded axis leave a partial
//     result: ONNX page, section on reduction operators.
//   * reshape rule: Paddle page, DimTrans table (InputDim, Flatten, Split,
//     Singleton) and its sharding rule.
//   * TP-MLP: ColossalAI 1D tensor parallelism page (mhpq.cn) section 2 and
//     2.1: Y_i = X A_i, Z = sum_i Y_i B_i; GELU between the GEMMs from the
//     Domino page (mzlw.cn), forward section ("GeMM GeLU GeMM").
//   * TP-MLP backward: ColossalAI page section 2.2: each rank's input
//     gradient is dY_i A_i^T and the full one is their sum; the weight
//     gradients are the usual products of the layer input and the output
//     gradient, on each rank's own shard.
//
// Readings where the pages are silent (each is listed in the design notes):
//   * uneven extents: ceil-sized leading shards, applied level by level;
//   * shard() of a partial layout: the device whose partial coordinates are
//     all zero holds the tensor, the others hold the reduction's identity
//     (0 for sum, +inf for min, -inf for max);
//   * GELU is the exact erf form; Y is rounded to bf16 before the second GEMM.
//   * backward: the saved pre-activation H and the gradient dH are bf16
//     tensors (the compute type), so they may be rounded (flags below).
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <string>
#include <vector>

namespace {

constexpr int kMaxMesh = 8;
constexpr int kMaxDev = 256;
constexpr int kMaxDim = 8;

}  // namespace

extern "C" {

// A layout in the ND-SBP form: a row-major mesh of device ids and one entry per
// mesh dim: 'S' (split tensor axis `axis`), 'B' (broadcast), or a partial
// reduction: 'P' (sum), 'N' (min) or 'X' (max). The OneFlow SBP page defines
// partial by sum and notes that min and max work the same way.
struct OracleLayout {
    int32_t mesh_ndim;
    int64_t mesh_shape[kMaxMesh];
    int32_t devices[kMaxDev];
    int8_t kind[kMaxMesh];
    int32_t axis[kMaxMesh];
};

}  // extern "C"

namespace {

int64_t num_devices(const OracleLayout& L)
{
    int64_t n = 1;
    for (int d = 0; d < L.mesh_ndim; ++d) n *= L.mesh_shape[d];
    return n;
}

// Mesh coordinates of device `dev`, or false if it is not on the mesh.
bool coords_of(const OracleLayout& L, int dev, int64_t* c)
{
    int64_t n = num_devices(L);
    for (int64_t p = 0; p < n; ++p) {
        if (L.devices[p] != dev) continue;
        int64_t rem = p;
        for (int d = L.mesh_ndim - 1; d >= 0; --d) {
            c[d] = rem % L.mesh_shape[d];
            rem /= L.mesh_shape[d];
        }
        return true;
    }
    return false;
}

// The slice [lo, hi) of every tensor axis held by a device at mesh coords c.
// For each axis, the mesh dims that split it are visited outer first; each
// level cuts the current interval into num_shards pieces of width
// ceil(len / num_shards) (the last piece is short, possibly empty).
void slice_of(const OracleLayout& L, int ndim, const int64_t* shape, const int64_t* c, int64_t* lo,
              int64_t* hi)
{
    for (int a = 0; a < ndim; ++a) {
        lo[a] = 0;
        hi[a] = shape[a];
    }
    for (int d = 0; d < L.mesh_ndim; ++d) {
        if (L.kind[d] != 'S') continue;
        int a = L.axis[d];
        int64_t len = hi[a] - lo[a];
        int64_t n = L.mesh_shape[d];
        int64_t width = (len + n - 1) / n;
        int64_t b = std::min(c[d] * width, len);
        int64_t e = std::min((c[d] + 1) * width, len);
        hi[a] = lo[a] + e;
        lo[a] = lo[a] + b;
    }
}

bool is_partial_kind(int8_t k) { return k == 'P' || k == 'N' || k == 'X'; }

// The partial reduction of a layout ('P', 'N' or 'X'; 'P' when there is none).
int8_t reduction_of(const OracleLayout& L)
{
    for (int d = 0; d < L.mesh_ndim; ++d)
        if (is_partial_kind(L.kind[d])) return L.kind[d];
    return 'P';
}

// What members of a partial group that do not hold the tensor contain: the
// value that leaves the reduction unchanged.
double identity_of(int8_t reduction)
{
    if (reduction == 'N') return INFINITY;
    if (reduction == 'X') return -INFINITY;
    return 0.0;
}

bool holds_partial_value(const OracleLayout& L, const int64_t* c)
{
    for (int d = 0; d < L.mesh_ndim; ++d)
        if (is_partial_kind(L.kind[d]) && c[d] != 0) return false;
    return true;
}

bool is_b_representative(const OracleLayout& L, const int64_t* c)
{
    for (int d = 0; d < L.mesh_ndim; ++d)
        if (L.kind[d] == 'B' && c[d] != 0) return false;
    return true;
}

int check_layout(const OracleLayout& L, int ndim)
{
    if (L.mesh_ndim < 1 || L.mesh_ndim > kMaxMesh || ndim < 0 || ndim > kMaxDim) return -1;
    int64_t n = num_devices(L);
    if (n < 1 || n > kMaxDev) return -1;
    std::vector<int> seen(n, 0);
    for (int64_t p = 0; p < n; ++p) {
        int v = L.devices[p];
        if (v < 0 || v >= n || seen[v]) return -1;
        seen[v] = 1;
    }
    for (int d = 0; d < L.mesh_ndim; ++d) {
        if (L.kind[d] != 'S' && L.kind[d] != 'B' && !is_partial_kind(L.kind[d])) return -1;
        if (L.kind[d] == 'S' && (L.axis[d] < 0 || L.axis[d] >= ndim)) return -1;
        for (int e = 0; e < d; ++e)  // one reduction per layout
            if (is_partial_kind(L.kind[d]) && is_partial_kind(L.kind[e]) && L.kind[d] != L.kind[e]) return -1;
    }
    return 0;
}

// ---- scalar conversions -------------------------------------------------

double bf16_bits_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return (double)f;
}

// Round a double to the nearest bfloat16 (8 significant bits, float's exponent
// range, subnormals down to 2^-133), ties to even.
uint16_t double_to_bf16_bits(double x)
{
    if (std::isnan(x)) return 0x7FC0;
    float f;
    if (x == 0.0 || std::isinf(x)) {
        f = (float)x;
    } else {
        int ex;
        std::frexp(x, &ex);  // |x| in [2^(ex-1), 2^ex)
        int qexp = std::max(ex - 8, -133);
        double q = std::ldexp(1.0, qexp);
        double r = std::nearbyint(x / q) * q;  // default rounding mode: ties to even
        if (std::fabs(r) >= std::ldexp(1.0, 128)) r = std::copysign(INFINITY, x);
        f = (float)r;  // exact: r has at most 8 significant bits
    }
    uint32_t u;
    std::memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

double load(int dtype, const void* p, int64_t i)
{
    if (dtype == 0) return (double)((const float*)p)[i];
    return bf16_bits_to_double(((const uint16_t*)p)[i]);
}

void store(int dtype, void* p, int64_t i, double v)
{
    if (dtype == 0) ((float*)p)[i] = (float)v;
    else ((uint16_t*)p)[i] = double_to_bf16_bits(v);
}

// Row-major successor of index idx within extents ext; false when done.
bool next_index(int ndim, const int64_t* ext, int64_t* idx)
{
    for (int a = ndim - 1; a >= 0; --a) {
        if (++idx[a] < ext[a]) return true;
        idx[a] = 0;
    }
    return false;
}

int64_t linear(int ndim, const int64_t* ext, const int64_t* idx)
{
    int64_t off = 0;
    for (int a = 0; a < ndim; ++a) off = off * ext[a] + idx[a];
    return off;
}

}  // namespace

extern "C" {

// Shape of the piece held by `device`; returns 0, or -1 on a malformed layout.
int oracle_shard_box(int ndim, const int64_t* shape, const OracleLayout* L, int device, int64_t* lo, int64_t* hi,
                     int32_t* holds_value)
{
    if (check_layout(*L, ndim)) return -1;
    int64_t c[kMaxMesh];
    if (!coords_of(*L, device, c)) return -1;
    slice_of(*L, ndim, shape, c, lo, hi);
    *holds_value = holds_partial_value(*L, c) ? 1 : 0;
    return 0;
}

// shard: the per-device pieces of the logical tensor `full`.
// out[dev] receives the row-major piece of device dev.
int oracle_shard(int dtype, int ndim, const int64_t* shape, const void* full, const OracleLayout* L, void* const* out)
{
    if (check_layout(*L, ndim)) return -1;
    int64_t n = num_devices(*L);
    for (int dev = 0; dev < n; ++dev) {
        int64_t c[kMaxMesh], lo[kMaxDim], hi[kMaxDim], ext[kMaxDim], e[kMaxDim], g[kMaxDim];
        coords_of(*L, dev, c);
        slice_of(*L, ndim, shape, c, lo, hi);
        bool value = holds_partial_value(*L, c);
        int64_t count = 1;
        for (int a = 0; a < ndim; ++a) {
            ext[a] = hi[a] - lo[a];
            count *= ext[a];
            e[a] = 0;
        }
        if (count == 0) continue;
        int64_t k = 0;
        do {
            for (int a = 0; a < ndim; ++a) g[a] = lo[a] + e[a];
            double v = value ? load(dtype, full, linear(ndim, shape, g)) : identity_of(reduction_of(*L));
            store(dtype, out[dev], k++, v);
        } while (next_index(ndim, ext, e));
    }
    return 0;
}

// The logical tensor (in double) described by per-device pieces `in` laid out
// by L: pieces of B replicas other than coordinate 0 are skipped, partial
// pieces are combined by the layout's reduction (sum in double; min / max
// with the IEEE minNum / maxNum of std::fmin / std::fmax).
int oracle_gather(int dtype, int ndim, const int64_t* shape, const void* const* in, const OracleLayout* L,
                  double* logical)
{
    if (check_layout(*L, ndim)) return -1;
    int64_t total = 1;
    for (int a = 0; a < ndim; ++a) total *= shape[a];
    const int8_t red = reduction_of(*L);
    for (int64_t i = 0; i < total; ++i) logical[i] = identity_of(red);
    int64_t n = num_devices(*L);
    for (int dev = 0; dev < n; ++dev) {
        int64_t c[kMaxMesh], lo[kMaxDim], hi[kMaxDim], ext[kMaxDim], e[kMaxDim], g[kMaxDim];
        coords_of(*L, dev, c);
        if (!is_b_representative(*L, c)) continue;
        slice_of(*L, ndim, shape, c, lo, hi);
        int64_t count = 1;
        for (int a = 0; a < ndim; ++a) {
            ext[a] = hi[a] - lo[a];
            count *= ext[a];
            e[a] = 0;
        }
        if (count == 0) continue;
        int64_t k = 0;
        do {
            for (int a = 0; a < ndim; ++a) g[a] = lo[a] + e[a];
            double& acc = logical[linear(ndim, shape, g)];
            const double v = load(dtype, in[dev], k++);
            if (red == 'N') acc = std::fmin(acc, v);
            else if (red == 'X') acc = std::fmax(acc, v);
            else acc += v;
        } while (next_index(ndim, ext, e));
    }
    return 0;
}

// reshard: gather the logical tensor from the source pieces (summing partial
// pieces in double), then cut it by the destination layout, rounding once to
// the element type.
int oracle_reshard(int dtype, int ndim, const int64_t* shape, const void* const* src, const OracleLayout* Ls,
                   void* const* dst, const OracleLayout* Ld)
{
    if (check_layout(*Ls, ndim) || check_layout(*Ld, ndim)) return -1;
    int64_t total = 1;
    for (int a = 0; a < ndim; ++a) total *= shape[a];
    std::vector<double> logical((size_t)std::max<int64_t>(total, 1));
    oracle_gather(dtype, ndim, shape, src, Ls, logical.data());
    int64_t n = num_devices(*Ld);
    for (int dev = 0; dev < n; ++dev) {
        int64_t c[kMaxMesh], lo[kMaxDim], hi[kMaxDim], ext[kMaxDim], e[kMaxDim], g[kMaxDim];
        coords_of(*Ld, dev, c);
        slice_of(*Ld, ndim, shape, c, lo, hi);
        bool value = holds_partial_value(*Ld, c);
        int64_t count = 1;
        for (int a = 0; a < ndim; ++a) {
            ext[a] = hi[a] - lo[a];
            count *= ext[a];
            e[a] = 0;
        }
        if (count == 0) continue;
        int64_t k = 0;
        do {
            for (int a = 0; a < ndim; ++a) g[a] = lo[a] + e[a];
            store(dtype, dst[dev], k++, value ? logical[linear(ndim, shape, g)] : identity_of(reduction_of(*Ld)));
        } while (next_index(ndim, ext, e));
    }
    return 0;
}

// ---- front-ends -----------------------------------------------------------

// Paddle dims_mapping: dims_mapping[i] = j splits tensor dim i along mesh dim j,
// -1 leaves it whole. Mesh dims named by no tensor dim are broadcast, or
// partial when their bit is set in partial_mask.
int oracle_layout_from_dims_mapping(int ndim, const int32_t* dims_mapping, int mesh_ndim, const int64_t* mesh_shape,
                                    const int32_t* devices, uint32_t partial_mask, OracleLayout* out)
{
    if (mesh_ndim < 1 || mesh_ndim > kMaxMesh || ndim < 0 || ndim > kMaxDim) return -1;
    OracleLayout L;
    std::memset(&L, 0, sizeof L);
    L.mesh_ndim = mesh_ndim;
    int64_t n = 1;
    for (int d = 0; d < mesh_ndim; ++d) {
        L.mesh_shape[d] = mesh_shape[d];
        L.kind[d] = (partial_mask >> d) & 1u ? 'P' : 'B';
        L.axis[d] = -1;
        n *= mesh_shape[d];
    }
    if (n < 1 || n > kMaxDev) return -1;
    for (int64_t p = 0; p < n; ++p) L.devices[p] = devices ? devices[p] : (int32_t)p;
    for (int i = 0; i < ndim; ++i) {
        int j = dims_mapping[i];
        if (j == -1) continue;
        if (j < 0 || j >= mesh_ndim) return -1;
        if ((partial_mask >> j) & 1u) return -1;  // a mesh dim cannot both split and hold partials
        if (L.kind[j] == 'S') return -1;         // two tensor dims on one mesh dim
        L.kind[j] = 'S';
        L.axis[j] = i;
    }
    if (check_layout(L, ndim)) return -1;
    *out = L;
    return 0;
}

// ONNX ShardingSpecProto: `device` lists device ids, or negative keys into
// device_map (index_to_device_group_map). The sharded_dim entries split their
// axes in the listed order (first = outer); split piece s goes to device[s],
// or to every device of group device_map[device[s]]. The product of the
// num_shards must equal the length of `device`; all groups must be the same
// size. The result is a mesh [num_shards..., group size] whose last dim, when
// the groups have more than one device, is broadcast.
int oracle_layout_from_onnx(int ndim, int n_device, const int64_t* device, int n_groups, const int64_t* group_keys,
                            const int32_t* group_sizes, const int64_t* group_devices, int n_sharded,
                            const int64_t* axes, const int64_t* num_shards, OracleLayout* out)
{
    if (n_device < 1 || n_sharded < 0 || n_sharded + 1 > kMaxMesh) return -1;
    // Expand each device entry into its list of devices.
    std::vector<std::vector<int64_t>> members;
    for (int s = 0; s < n_device; ++s) {
        std::vector<int64_t> m;
        if (device[s] >= 0) {
            m.push_back(device[s]);
        } else {
            int64_t off = 0;
            bool found = false;
            for (int g = 0; g < n_groups; ++g) {
                if (group_keys[g] == device[s]) {
                    for (int t = 0; t < group_sizes[g]; ++t) m.push_back(group_devices[off + t]);
                    found = true;
                    break;
                }
                off += group_sizes[g];
            }
            if (!found || m.empty()) return -1;
        }
        if (!members.empty() && m.size() != members[0].size()) return -1;
        members.push_back(m);
    }
    int64_t splits = 1;
    for (int k = 0; k < n_sharded; ++k) {
        if (num_shards[k] < 1) return -1;
        splits *= num_shards[k];
    }
    if (splits != n_device) return -1;
    OracleLayout L;
    std::memset(&L, 0, sizeof L);
    int md = 0;
    for (int k = 0; k < n_sharded; ++k) {
        int64_t a = axes[k];
        if (a < -ndim || a >= ndim) return -1;
        if (a < 0) a += ndim;
        L.mesh_shape[md] = num_shards[k];
        L.kind[md] = 'S';
        L.axis[md] = (int32_t)a;
        ++md;
    }
    int64_t gsize = (int64_t)members[0].size();
    if (gsize > 1 || md == 0) {
        L.mesh_shape[md] = gsize;
        L.kind[md] = 'B';
        L.axis[md] = -1;
        ++md;
    }
    L.mesh_ndim = md;
    int64_t n = splits * gsize;
    if (n > kMaxDev) return -1;
    for (int s = 0; s < n_device; ++s)
        for (int64_t t = 0; t < gsize; ++t) L.devices[s * gsize + t] = (int32_t)members[s][t];
    if (check_layout(L, ndim)) return -1;
    *out = L;
    return 0;
}

// ---- infer_spmd (einsum rule) ---------------------------------------------

// Step 1: the einsum ("mk,kn->mn") names every axis of every input and of the
// output by a letter. Step 2 (merge): each letter takes the first mesh dim that
// some input gives it; an input that gives it another mesh dim conflicts and
// must be resharded. A mesh dim may shard one letter only: the letter that
// comes first in the einsum keeps it. Step 3: the output dims_mapping lists
// the merged mesh dims of the output letters; a letter that is summed away
// (present in the inputs, absent from the output) and sharded leaves the
// output partial over that mesh dim.
//   merged_in[j][i]: dims_mapping that input j must be resharded to.
// Returns 0, or -1 on a malformed einsum / mapping.
int oracle_infer_spmd(const char* einsum, int n_in, const int32_t* const* in_dims_mapping, int mesh_ndim,
                      int32_t* out_dims_mapping, uint32_t* out_partial_mask, uint32_t* in_needs_reshard_mask,
                      int32_t* const* merged_in)
{
    std::string s(einsum ? einsum : "");
    size_t arrow = s.find("->");
    if (arrow == std::string::npos || n_in < 1 || n_in > 8 || mesh_ndim < 1 || mesh_ndim > kMaxMesh) return -1;
    std::vector<std::string> ins;
    {
        std::string lhs = s.substr(0, arrow), cur;
        for (char ch : lhs) {
            if (ch == ',') {
                ins.push_back(cur);
                cur.clear();
            } else {
                cur.push_back(ch);
            }
        }
        ins.push_back(cur);
    }
    std::string outs = s.substr(arrow + 2);
    if ((int)ins.size() != n_in) return -1;
    for (auto& t : ins)
        for (size_t i = 0; i < t.size(); ++i) {
            if (t[i] < 'a' || t[i] > 'z' || t.find(t[i]) != i) return -1;
        }
    for (size_t i = 0; i < outs.size(); ++i) {
        char ch = outs[i];
        if (ch < 'a' || ch > 'z' || outs.find(ch) != i) return -1;
        bool present = false;
        for (auto& t : ins) present = present || t.find(ch) != std::string::npos;
        if (!present) return -1;
    }
    for (int j = 0; j < n_in; ++j)
        for (size_t i = 0; i < ins[j].size(); ++i) {
            int v = in_dims_mapping[j][i];
            if (v < -1 || v >= mesh_ndim) return -1;
            for (size_t k = 0; k < i; ++k)
                if (v != -1 && in_dims_mapping[j][k] == v) return -1;
        }
    // letters in order of first appearance in the einsum string
    std::string order;
    for (char ch : s)
        if (ch >= 'a' && ch <= 'z' && order.find(ch) == std::string::npos) order.push_back(ch);
    int letter_dim[26];
    for (int i = 0; i < 26; ++i) letter_dim[i] = -1;
    for (char ch : order)
        for (int j = 0; j < n_in; ++j) {
            size_t pos = ins[j].find(ch);
            if (pos == std::string::npos) continue;
            int v = in_dims_mapping[j][pos];
            if (v != -1 && letter_dim[ch - 'a'] == -1) letter_dim[ch - 'a'] = v;
        }
    for (int d = 0; d < mesh_ndim; ++d) {
        bool taken = false;
        for (char ch : order) {
            if (letter_dim[ch - 'a'] != d) continue;
            if (taken) letter_dim[ch - 'a'] = -1;
            taken = true;
        }
    }
    uint32_t needs = 0;
    for (int j = 0; j < n_in; ++j)
        for (size_t i = 0; i < ins[j].size(); ++i) {
            int m = letter_dim[ins[j][i] - 'a'];
            if (merged_in && merged_in[j]) merged_in[j][i] = m;
            if (in_dims_mapping[j][i] != m) needs |= 1u << j;
        }
    for (size_t i = 0; i < outs.size(); ++i) out_dims_mapping[i] = letter_dim[outs[i] - 'a'];
    uint32_t partial = 0;
    for (char ch : order)
        if (outs.find(ch) == std::string::npos && letter_dim[ch - 'a'] != -1) partial |= 1u << letter_dim[ch - 'a'];
    *out_partial_mask = partial;
    *in_needs_reshard_mask = needs;
    return 0;
}

// ---- reshape rule (DimTrans) ----------------------------------------------

// Describes each output dim of a reshape by the Paddle DimTrans kinds:
//   0 InputDim(i), 1 Flatten(dims), 2 Split(input dim, sizes, idx),
//   3 Singleton, 4 Split(Flatten(dims), sizes, idx).
// in_first/in_count: the input dims feeding the output dim; piece/npieces: its
// index among the output dims cut from the same input group.
// Then the sharding rule: in a group, only the leading member (first with
// extent > 1) may carry a split, and it survives the reshape iff each device's
// contiguous run of the flattened group is the same before and after (ceil
// pieces of the leading input member scaled by the rest of the input group
// equal ceil pieces of the leading output member scaled by the rest of the
// output group). Otherwise the input must first be resharded to drop it.
int oracle_reshape_spmd(int in_ndim, const int64_t* in_shape, const int32_t* in_dims_mapping, int out_ndim,
                        const int64_t* out_shape, int mesh_ndim, const int64_t* mesh_shape, int32_t* in_dims_after,
                        int32_t* out_dims_mapping, int32_t* dt_kind, int32_t* dt_in_first, int32_t* dt_in_count,
                        int32_t* dt_piece, int32_t* dt_npieces)
{
    if (in_ndim < 0 || in_ndim > kMaxDim || out_ndim < 0 || out_ndim > kMaxDim || mesh_ndim < 1 ||
        mesh_ndim > kMaxMesh)
        return -1;
    int64_t pi = 1, po = 1;
    for (int i = 0; i < in_ndim; ++i) {
        if (in_shape[i] < 1) return -1;
        pi *= in_shape[i];
        int v = in_dims_mapping[i];
        if (v < -1 || v >= mesh_ndim) return -1;
        in_dims_after[i] = v;
    }
    for (int o = 0; o < out_ndim; ++o) {
        if (out_shape[o] < 1) return -1;
        po *= out_shape[o];
        out_dims_mapping[o] = -1;
        dt_kind[o] = 3;
        dt_in_first[o] = -1;
        dt_in_count[o] = 0;
        dt_piece[o] = 0;
        dt_npieces[o] = 1;
    }
    if (pi != po) return -1;
    int i = 0, o = 0;
    while (i < in_ndim || o < out_ndim) {
        if (o < out_ndim && out_shape[o] == 1 && (i >= in_ndim || in_shape[i] != 1)) {
            ++o;  // Singleton
            continue;
        }
        if (i < in_ndim && in_shape[i] == 1 && (o >= out_ndim || out_shape[o] != 1)) {
            in_dims_after[i] = -1;  // a size-1 input dim vanishes; its split cannot survive
            ++i;
            continue;
        }
        int i0 = i, o0 = o;
        int64_t a = in_shape[i++], b = out_shape[o++];
        while (a != b) {
            if (a < b) a *= in_shape[i++];
            else b *= out_shape[o++];
        }
        int ni = i - i0, no = o - o0;
        for (int k = 0; k < no; ++k) {
            dt_kind[o0 + k] = ni == 1 && no == 1 ? 0 : (no == 1 ? 1 : (ni == 1 ? 2 : 4));
            dt_in_first[o0 + k] = i0;
            dt_in_count[o0 + k] = ni;
            dt_piece[o0 + k] = k;
            dt_npieces[o0 + k] = no;
        }
        // leading members
        int li = i0, lo = o0;
        while (li < i - 1 && in_shape[li] == 1) ++li;
        while (lo < o - 1 && out_shape[lo] == 1) ++lo;
        for (int k = i0; k < i; ++k)
            if (k != li) in_dims_after[k] = -1;
        int d = in_dims_after[li];
        if (d == -1) continue;
        int64_t n = mesh_shape[d];
        int64_t L0 = in_shape[li], E0 = out_shape[lo], I = 1, J = 1;
        for (int k = li + 1; k < i; ++k) I *= in_shape[k];
        for (int k = lo + 1; k < o; ++k) J *= out_shape[k];
        int64_t wi = (L0 + n - 1) / n, wo = (E0 + n - 1) / n;
        bool same = true;
        for (int64_t r = 0; r < n; ++r) {
            int64_t b1 = std::min(r * wi, L0) * I, e1 = std::min((r + 1) * wi, L0) * I;
            int64_t b2 = std::min(r * wo, E0) * J, e2 = std::min((r + 1) * wo, E0) * J;
            if (b1 != b2 || e1 != e2) same = false;
        }
        if (same) out_dims_mapping[lo] = d;
        else in_dims_after[li] = -1;
    }
    return 0;
}

// ---- SBP signature inference (OneFlow page, add_n walk-through) -------------

// A signature: one (kind, axis) per mesh dim, shared by every input and the
// output of an element-wise op. kind: 'S' split(axis), 'P' partial sum,
// 'B' broadcast (inputs may also be 'N' / 'X', partial min / max).
struct Sig {
    std::vector<std::pair<char, int>> dims;
    int order = 0;
    double cost = 0;
};

// Step 1: candidates. For one mesh dim the op offers split(i) for every axis
// i of the input shape, then partial sum; broadcast is added by default. On an
// ND mesh every slot takes any 1D candidate: the direct product, built with
// mesh dim 0 varying slowest.
// Step 2: filters: a split axis must be an axis of the tensor; a required
// signature (constraint), when given, must match.
// Step 3: sort by OrderValue (-10 per input already in the candidate's SBP,
// 0 for all when a constraint is given), then by CopyCost (per input: 0 if
// equal; a huge number when the input is partial or broadcast; else its
// bytes), keeping the candidate order among equals; the first one wins.
int oracle_infer_sbp_signature(int n_in, int ndim, const int64_t* shape, int elem_bytes, int mesh_ndim,
                               const int8_t* in_kinds, const int32_t* in_axes, const int8_t* constraint_kinds,
                               const int32_t* constraint_axes, int8_t* out_kinds, int32_t* out_axes, double* out_cost,
                               int32_t* out_order, int32_t* n_candidates)
{
    if (n_in < 1 || ndim < 1 || mesh_ndim < 1 || mesh_ndim > kMaxMesh) return -1;
    std::vector<std::pair<char, int>> one;
    for (int i = 0; i < ndim; ++i) one.push_back({'S', i});
    one.push_back({'P', -1});
    one.push_back({'B', -1});
    std::vector<Sig> cands(1);
    for (int d = 0; d < mesh_ndim; ++d) {
        std::vector<Sig> next;
        for (const Sig& c : cands)
            for (const auto& e : one) {
                Sig n = c;
                n.dims.push_back(e);
                next.push_back(n);
            }
        cands = next;
    }
    std::vector<Sig> kept;
    for (const Sig& c : cands) {
        bool ok = true;
        for (int d = 0; d < mesh_ndim; ++d) {
            if (c.dims[d].first == 'S' && c.dims[d].second >= ndim) ok = false;
            if (constraint_kinds && (constraint_kinds[d] != c.dims[d].first ||
                                     (c.dims[d].first == 'S' && constraint_axes[d] != c.dims[d].second)))
                ok = false;
        }
        if (ok) kept.push_back(c);
    }
    if (n_candidates) *n_candidates = (int32_t)kept.size();
    if (kept.empty()) return -2;
    double bytes = elem_bytes;
    for (int a = 0; a < ndim; ++a) bytes *= (double)shape[a];
    for (Sig& c : kept) {
        for (int j = 0; j < n_in; ++j) {
            bool same = true, partial_or_broadcast = false;
            for (int d = 0; d < mesh_ndim; ++d) {
                char k = (char)in_kinds[j * mesh_ndim + d];
                int ax = in_axes[j * mesh_ndim + d];
                if (k != 'S') partial_or_broadcast = true;
                if (k != c.dims[d].first || (k == 'S' && ax != c.dims[d].second)) same = false;
            }
            if (same && !constraint_kinds) c.order -= 10;
            if (!same) c.cost += partial_or_broadcast ? 1e30 : bytes;
        }
    }
    std::stable_sort(kept.begin(), kept.end(), [](const Sig& a, const Sig& b) {
        if (a.order != b.order) return a.order < b.order;
        return a.cost < b.cost;
    });
    for (int d = 0; d < mesh_ndim; ++d) {
        out_kinds[d] = (int8_t)kept[0].dims[d].first;
        out_axes[d] = kept[0].dims[d].second;
    }
    *out_cost = kept[0].cost;
    *out_order = kept[0].order;
    return 0;
}

// ---- ONNX broadcast n-ary element-wise rule -----------------------------------

// "ONNX multi-device proposal", operator groups: for a broadcast n-ary
// element-wise operator a device computes the output elements whose inputs it
// all holds; a shard's devices are the intersection of the devices of the input
// shards it reads (the Add([M,1],[1,N]) example). Done per element here.
// Inputs: n_in tensors (shapes right-aligned for broadcasting) on the same
// n_dev devices. Result: *status = 0 and, per device, the box [lo, hi) of the
// output it computes (out_lo/out_hi[dev * kMaxDim + axis]; empty = lo == hi on
// some axis), plus a layout that yields those boxes; *status = 1 when some
// output element has no device; *status = 2 when the boxes are not a layout
// (two devices' boxes overlap without being equal, they do not form a grid,
// the grid cells have unequal numbers of devices, or the cuts are not the even
// split). An input whose own layout already gives exactly the boxes is
// returned as the layout.
int oracle_infer_broadcast(int n_in, const int32_t* in_ndims, const int64_t* const* in_shapes,
                           const OracleLayout* in_layouts, int* out_ndim, int64_t* out_shape, int64_t* out_lo,
                           int64_t* out_hi, OracleLayout* out_layout, int* status)
{
    if (n_in < 1) return -1;
    int nd = 0;
    for (int k = 0; k < n_in; ++k) {
        if (in_ndims[k] < 1 || in_ndims[k] > kMaxDim) return -1;
        if (check_layout(in_layouts[k], in_ndims[k])) return -1;
        for (int d = 0; d < in_layouts[k].mesh_ndim; ++d)
            if (is_partial_kind(in_layouts[k].kind[d])) return -1;
        nd = std::max(nd, (int)in_ndims[k]);
    }
    const int64_t n_dev = num_devices(in_layouts[0]);
    for (int k = 1; k < n_in; ++k)
        if (num_devices(in_layouts[k]) != n_dev) return -1;
    int64_t shape[kMaxDim];
    for (int d = 0; d < nd; ++d) {
        int64_t e = 1;
        for (int k = 0; k < n_in; ++k) {
            int dk = d - (nd - in_ndims[k]);
            if (dk < 0) continue;
            int64_t x = in_shapes[k][dk];
            if (x < 1) return -1;  // empty tensors are not handled by this rule
            if (x == 1) continue;
            if (e != 1 && e != x) return -1;
            e = x;
        }
        shape[d] = e;
    }
    int64_t total = 1;
    for (int d = 0; d < nd; ++d) total *= shape[d];
    // input pieces of every device
    std::vector<int64_t> plo((size_t)n_in * n_dev * kMaxDim), phi((size_t)n_in * n_dev * kMaxDim);
    for (int k = 0; k < n_in; ++k)
        for (int64_t dev = 0; dev < n_dev; ++dev) {
            int64_t c[kMaxMesh];
            if (!coords_of(in_layouts[k], (int)dev, c)) return -1;
            slice_of(in_layouts[k], in_ndims[k], in_shapes[k], c, &plo[(k * n_dev + dev) * kMaxDim],
                     &phi[(k * n_dev + dev) * kMaxDim]);
        }
    // per device: which output elements it can compute (bounding box + count)
    std::vector<int64_t> lo((size_t)n_dev * kMaxDim), hi((size_t)n_dev * kMaxDim), count((size_t)n_dev, 0);
    std::vector<int> covered((size_t)total, 0);
    for (int64_t dev = 0; dev < n_dev; ++dev) {
        for (int d = 0; d < nd; ++d) {
            lo[dev * kMaxDim + d] = shape[d];
            hi[dev * kMaxDim + d] = 0;
        }
        int64_t e[kMaxDim];
        for (int64_t flat = 0; flat < total; ++flat) {
            int64_t rem = flat;
            for (int d = nd - 1; d >= 0; --d) {
                e[d] = rem % shape[d];
                rem /= shape[d];
            }
            bool ok = true;
            for (int k = 0; k < n_in && ok; ++k)
                for (int dk = 0; dk < in_ndims[k] && ok; ++dk) {
                    int d = dk + (nd - in_ndims[k]);
                    int64_t i = in_shapes[k][dk] == 1 ? 0 : e[d];  // a broadcast axis reads element 0
                    const int64_t* L = &plo[(k * n_dev + dev) * kMaxDim];
                    const int64_t* H = &phi[(k * n_dev + dev) * kMaxDim];
                    if (i < L[dk] || i >= H[dk]) ok = false;
                }
            if (!ok) continue;
            ++count[dev];
            ++covered[flat];
            for (int d = 0; d < nd; ++d) {
                lo[dev * kMaxDim + d] = std::min(lo[dev * kMaxDim + d], e[d]);
                hi[dev * kMaxDim + d] = std::max(hi[dev * kMaxDim + d], e[d] + 1);
            }
        }
        if (count[dev] == 0)
            for (int d = 0; d < nd; ++d) lo[dev * kMaxDim + d] = hi[dev * kMaxDim + d] = 0;
        int64_t vol = 1;
        for (int d = 0; d < nd; ++d) vol *= hi[dev * kMaxDim + d] - lo[dev * kMaxDim + d];
        if (count[dev] > 0 && vol != count[dev]) return -1;  // cannot happen: intersections of boxes are boxes
    }
    *out_ndim = nd;
    for (int d = 0; d < nd; ++d) out_shape[d] = shape[d];
    for (int64_t i = 0; i < n_dev * kMaxDim; ++i) {
        out_lo[i] = lo[i];
        out_hi[i] = hi[i];
    }
    auto same_box = [&](int64_t a, int64_t b) {
        for (int d = 0; d < nd; ++d)
            if (lo[a * kMaxDim + d] != lo[b * kMaxDim + d] || hi[a * kMaxDim + d] != hi[b * kMaxDim + d]) return false;
        return true;
    };
    // an input whose own pieces are these boxes
    for (int k = 0; k < n_in; ++k) {
        if (in_ndims[k] != nd) continue;
        bool full = true;
        for (int d = 0; d < nd; ++d) full &= in_shapes[k][d] == shape[d];
        if (!full) continue;
        bool match = true;
        for (int64_t dev = 0; dev < n_dev && match; ++dev) {
            const int64_t* L = &plo[(k * n_dev + dev) * kMaxDim];
            const int64_t* H = &phi[(k * n_dev + dev) * kMaxDim];
            int64_t vol = 1;
            for (int d = 0; d < nd; ++d) vol *= H[d] - L[d];
            if (vol != count[dev]) match = false;
            for (int d = 0; d < nd && match && count[dev] > 0; ++d)
                if (L[d] != lo[dev * kMaxDim + d] || H[d] != hi[dev * kMaxDim + d]) match = false;
        }
        if (match) {
            *out_layout = in_layouts[k];
            *status = 0;
            return 0;
        }
    }
    // overlapping boxes that differ
    for (int64_t a = 0; a < n_dev; ++a)
        for (int64_t b = a + 1; b < n_dev; ++b) {
            if (!count[a] || !count[b] || same_box(a, b)) continue;
            bool meet = true;
            for (int d = 0; d < nd; ++d)
                meet &= std::max(lo[a * kMaxDim + d], lo[b * kMaxDim + d]) <
                        std::min(hi[a * kMaxDim + d], hi[b * kMaxDim + d]);
            if (meet) {
                *status = 2;
                return 0;
            }
        }
    for (int64_t f = 0; f < total; ++f)
        if (!covered[f]) {
            *status = 1;
            return 0;
        }
    // a grid of cells, each on the same number of devices
    std::vector<std::vector<std::pair<int64_t, int64_t>>> cuts((size_t)nd);
    for (int d = 0; d < nd; ++d) {
        for (int64_t dev = 0; dev < n_dev; ++dev)
            if (count[dev]) cuts[d].push_back({lo[dev * kMaxDim + d], hi[dev * kMaxDim + d]});
        std::sort(cuts[d].begin(), cuts[d].end());
        cuts[d].erase(std::unique(cuts[d].begin(), cuts[d].end()), cuts[d].end());
    }
    int64_t cells = 1;
    for (int d = 0; d < nd; ++d) cells *= (int64_t)cuts[d].size();
    std::vector<std::vector<int>> holders((size_t)std::max<int64_t>(cells, 1));
    int64_t distinct = 0;
    for (int64_t dev = 0; dev < n_dev; ++dev) {
        if (!count[dev]) {
            *status = 2;  // a device with nothing to compute
            return 0;
        }
        bool first = true;
        for (int64_t o = 0; o < dev; ++o)
            if (count[o] && same_box(o, dev)) first = false;
        distinct += first ? 1 : 0;
        int64_t cell = 0;
        for (int d = 0; d < nd; ++d) {
            int64_t i = std::find(cuts[d].begin(), cuts[d].end(),
                                  std::make_pair(lo[dev * kMaxDim + d], hi[dev * kMaxDim + d])) - cuts[d].begin();
            cell = cell * (int64_t)cuts[d].size() + i;
        }
        holders[cell].push_back((int)dev);
    }
    if (distinct != cells) {
        *status = 2;
        return 0;
    }
    size_t rep = holders[0].size();
    for (auto& h : holders)
        if (h.size() != rep) {
            *status = 2;
            return 0;
        }
    OracleLayout L;
    std::memset(&L, 0, sizeof L);
    for (int d = 0; d < nd; ++d) {
        if (cuts[d].size() <= 1) continue;
        if (L.mesh_ndim == kMaxMesh) return -1;
        L.mesh_shape[L.mesh_ndim] = (int64_t)cuts[d].size();
        L.kind[L.mesh_ndim] = 'S';
        L.axis[L.mesh_ndim] = d;
        ++L.mesh_ndim;
    }
    if (rep > 1 || L.mesh_ndim == 0) {
        L.mesh_shape[L.mesh_ndim] = (int64_t)rep;
        L.kind[L.mesh_ndim] = 'B';
        ++L.mesh_ndim;
    }
    for (int64_t c = 0; c < cells; ++c) {
        std::vector<int> h = holders[c];
        std::sort(h.begin(), h.end());
        for (size_t t = 0; t < rep; ++t) L.devices[c * rep + t] = h[t];
    }
    for (int64_t dev = 0; dev < n_dev; ++dev) {
        int64_t c[kMaxMesh], l2[kMaxDim], h2[kMaxDim];
        coords_of(L, (int)dev, c);
        slice_of(L, nd, shape, c, l2, h2);
        for (int d = 0; d < nd; ++d)
            if (l2[d] != lo[dev * kMaxDim + d] || h2[d] != hi[dev * kMaxDim + d]) {
                *status = 2;  // not the even split
                return 0;
            }
    }
    *out_layout = L;
    *status = 0;
    return 0;
}

// ---- scalar helpers exposed for pins -----------------------------------------

uint16_t oracle_bf16_round(double x) { return double_to_bf16_bits(x); }

double oracle_gelu(double x) { return 0.5 * x * (1.0 + std::erf(x / std::sqrt(2.0))); }

// Derivative of the exact GELU x Phi(x): Phi(x) + x phi(x).
double oracle_gelu_grad(double x)
{
    const double pi = 3.14159265358979323846;
    return 0.5 * (1.0 + std::erf(x / std::sqrt(2.0))) + x * std::exp(-0.5 * x * x) / std::sqrt(2.0 * pi);
}

// ---- TP-MLP -------------------------------------------------------------------

// Megatron 1D tensor-parallel MLP on P virtual devices, for the listed rows of X:
//   Y_i = act(X A_i)      (column-parallel: A = [A_1 ... A_P], A_i is [K, F/P])
//   Z   = sum_i Y_i B_i   (row-parallel: B = [B_1; ...; B_P], B_i is [F/P, N])
// X, A_i, B_i are bf16 bit patterns, row-major. Products are summed in double;
// Y is rounded to bf16 before the second product (it is a bf16 tensor).
// act: 0 identity, 1 GELU (exact erf form).
// y_out (optional): [n_rows, F] with shard i in columns [i F/P, (i+1) F/P);
// z_out: [n_rows, N].
int oracle_tp_mlp(int64_t P, int64_t M, int64_t K, int64_t F, int64_t N, const uint16_t* X,
                  const uint16_t* const* A, const uint16_t* const* B, int act, int round_y, int64_t n_rows,
                  const int64_t* rows, double* y_out, double* z_out)
{
    if (P < 1 || F % P != 0 || M < 0 || K < 1 || N < 1) return -1;
    int64_t Fp = F / P;
    std::vector<double> x((size_t)K), y((size_t)Fp);
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t m = rows[r];
        if (m < 0 || m >= M) return -1;
        for (int64_t k = 0; k < K; ++k) x[k] = bf16_bits_to_double(X[m * K + k]);
        double* z = z_out + r * N;
        for (int64_t n = 0; n < N; ++n) z[n] = 0.0;
        for (int64_t i = 0; i < P; ++i) {
            for (int64_t f = 0; f < Fp; ++f) y[f] = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                const uint16_t* arow = A[i] + k * Fp;
                for (int64_t f = 0; f < Fp; ++f) y[f] += x[k] * bf16_bits_to_double(arow[f]);
            }
            for (int64_t f = 0; f < Fp; ++f) {
                double v = act == 1 ? oracle_gelu(y[f]) : y[f];
                if (round_y) v = bf16_bits_to_double(double_to_bf16_bits(v));
                y[f] = v;
                if (y_out) y_out[r * F + i * Fp + f] = v;
            }
            for (int64_t f = 0; f < Fp; ++f) {
                const uint16_t* brow = B[i] + f * N;
                for (int64_t n = 0; n < N; ++n) z[n] += y[f] * bf16_bits_to_double(brow[n]);
            }
        }
    }
    return 0;
}

// Backward of the TP-MLP above (act = GELU) for the loss L = sum(dZ * Z),
// i.e. dZ is the gradient arriving at Z. With H_i = X A_i, Y_i = GELU(H_i):
//   dY_i = dZ B_i^T,  dH_i = dY_i * GELU'(H_i),
//   dX   = sum_i dH_i A_i^T,  dA_i = X^T dH_i,  dB_i = Y_i^T dZ.
// All products are summed in double. flags select the bf16 roundings of the
// stored tensors: 1 = H rounded before GELU', 2 = Y rounded (as the forward
// stores it), 4 = dH rounded before the products that read it. flags = 0 gives
// the exact gradient.
// Rows (of X, dX): for each listed row m
//   dx_out [n_rows, K] = row m of dX; dh_out / dy_out / h_out (optional,
//   [n_rows, F], shard i in columns [i F/P, (i+1) F/P)) = row m of dH (before
//   rounding), dY and H (after rounding if flag 1).
// Columns (of the hidden dimension): for each listed f in [0, F) (rank
//   i = f / (F/P), local column f - i F/P)
//   da_out [n_cols, K] = column f of A's gradient (dA_i[:, local f]),
//   db_out [n_cols, N] = row f of B's gradient (dB_i[local f, :]).
int oracle_tp_mlp_backward(int64_t P, int64_t M, int64_t K, int64_t F, int64_t N, const uint16_t* X,
                           const uint16_t* const* A, const uint16_t* const* B, const uint16_t* dZ, int flags,
                           int64_t n_rows, const int64_t* rows, double* dx_out, double* dh_out, double* dy_out,
                           double* h_out, int64_t n_cols, const int64_t* cols, double* da_out, double* db_out)
{
    if (P < 1 || F % P != 0 || M < 0 || K < 1 || N < 1 || n_rows < 0 || n_cols < 0) return -1;
    const int64_t Fp = F / P;
    const bool round_h = flags & 1, round_y = flags & 2, round_dh = flags & 4;
    auto rnd = [](double v) { return bf16_bits_to_double(double_to_bf16_bits(v)); };
    auto a_at = [&](int64_t k, int64_t f) { return bf16_bits_to_double(A[f / Fp][k * Fp + f % Fp]); };
    auto b_at = [&](int64_t f, int64_t n) { return bf16_bits_to_double(B[f / Fp][(f % Fp) * N + n]); };
    std::vector<double> x((size_t)K), dz((size_t)N), dh((size_t)F);
    for (int64_t r = 0; r < n_rows; ++r) {
        const int64_t m = rows[r];
        if (m < 0 || m >= M) return -1;
        for (int64_t k = 0; k < K; ++k) x[k] = bf16_bits_to_double(X[m * K + k]);
        for (int64_t n = 0; n < N; ++n) dz[n] = bf16_bits_to_double(dZ[m * N + n]);
        for (int64_t f = 0; f < F; ++f) {
            double h = 0.0, dy = 0.0;
            for (int64_t k = 0; k < K; ++k) h += x[k] * a_at(k, f);
            for (int64_t n = 0; n < N; ++n) dy += dz[n] * b_at(f, n);
            if (round_h) h = rnd(h);
            const double g = dy * oracle_gelu_grad(h);
            if (dh_out) dh_out[r * F + f] = g;
            if (dy_out) dy_out[r * F + f] = dy;
            if (h_out) h_out[r * F + f] = h;
            dh[f] = round_dh ? rnd(g) : g;
        }
        for (int64_t k = 0; k < K; ++k) {
            double acc = 0.0;
            for (int64_t f = 0; f < F; ++f) acc += dh[f] * a_at(k, f);
            dx_out[r * K + k] = acc;
        }
    }
    for (int64_t c = 0; c < n_cols; ++c) {
        const int64_t f = cols[c];
        if (f < 0 || f >= F) return -1;
        double* da = da_out + c * K;
        double* db = db_out + c * N;
        for (int64_t k = 0; k < K; ++k) da[k] = 0.0;
        for (int64_t n = 0; n < N; ++n) db[n] = 0.0;
        for (int64_t m = 0; m < M; ++m) {
            double h = 0.0, dy = 0.0;
            for (int64_t k = 0; k < K; ++k) h += bf16_bits_to_double(X[m * K + k]) * a_at(k, f);
            for (int64_t n = 0; n < N; ++n) dy += bf16_bits_to_double(dZ[m * N + n]) * b_at(f, n);
            double y = oracle_gelu(h);
            if (round_y) y = rnd(y);
            if (round_h) h = rnd(h);
            double g = dy * oracle_gelu_grad(h);
            if (round_dh) g = rnd(g);
            for (int64_t k = 0; k < K; ++k) da[k] += bf16_bits_to_double(X[m * K + k]) * g;
            for (int64_t n = 0; n < N; ++n) db[n] += y * bf16_bits_to_double(dZ[m * N + n]);
        }
    }
    return 0;
}

}  // extern "C"
