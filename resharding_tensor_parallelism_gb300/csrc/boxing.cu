// Boxing kernel: executes planned reshard tasks (copies, partial sums, zero
// fills) for shard() and reshard().
//
// Design for GB300 (HBM-bound, no tensor-core work):
//   * the task table travels in the kernel parameters (up to ~26 KB per
//     launch, __grid_constant__), so no device memory is allocated or copied
//     per call and the launch can be captured in a CUDA graph;
//   * a persistent grid (8 blocks of 256 threads per SM, a multiple of the SM
//     count) walks ~32 KB chunks of work; long rows are cut into segments
//     that a whole block streams, short rows are handed one per warp;
//   * loads and stores are 16-byte vectors whenever every pointer, stride and
//     run length allows it (else 8, 4 or 2 bytes), with streaming cache hints
//     since every byte is touched once;
//   * a task with several destinations (broadcast pieces) reads its source
//     once and writes every destination from registers;
//   * a task with several sources (partial sums) adds them in float32 in a
//     fixed order (partial coordinates row-major) and rounds once.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>

#include "rtp_internal.h"

namespace rtp {

namespace {

constexpr int kBlock = 256;
constexpr int kWarps = kBlock / 32;
constexpr int kUnroll = 4;
constexpr int kBlocksPerSm = 8;
constexpr int64_t kChunkBytes = 32 * 1024;
constexpr int kMaxTasks = 96;
constexpr int kMaxPtrs = 640;

struct KTask {
    int64_t chunk_begin;  // first chunk index of this task within the launch
    int64_t rows, cols;   // region: rows runs of cols contiguous elements
    int64_t seg, nseg;    // block mode: elements per segment, segments per row
    int64_t rpc;          // warp mode: rows per chunk
    int32_t mode;         // 1: block streams one row segment; 0: one row per warp
    int32_t vec;          // bytes per vector access
    int32_t n_outer, n_src, n_dst, ptr0;
    int32_t ext[kMaxOuter];
    int32_t pad_;
    int64_t sstr[kMaxOuter], dstr[kMaxOuter];
};

struct KParams {
    int32_t n_tasks;
    int32_t dtype;
    int64_t total_chunks;
    KTask tasks[kMaxTasks];
    const void* ptrs[kMaxPtrs];  // per task: n_src source bases, then n_dst destination bases
};
static_assert(sizeof(KParams) <= 32000, "kernel parameter block too large");

template <int VB>
struct Raw;
template <>
struct Raw<16> {
    using T = uint4;
};
template <>
struct Raw<8> {
    using T = uint2;
};
template <>
struct Raw<4> {
    using T = unsigned int;
};
template <>
struct Raw<2> {
    using T = unsigned short;
};

template <int VB>
union Lanes {
    typename Raw<VB>::T v;
    uint32_t w[VB >= 4 ? VB / 4 : 1];
    uint16_t h[VB / 2];
};

__device__ __forceinline__ int find_task(const KParams& p, int64_t c)
{
    int lo = 0, hi = p.n_tasks - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (p.tasks[mid].chunk_begin <= c) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ void row_offsets(const KTask& t, int64_t row, int64_t& so, int64_t& dof)
{
    so = 0;
    dof = 0;
    uint32_t r = (uint32_t)row;
    for (int k = t.n_outer - 1; k >= 0; --k) {
        uint32_t e = (uint32_t)t.ext[k];
        uint32_t q = r / e;
        uint32_t i = r - q * e;
        so += (int64_t)i * t.sstr[k];
        dof += (int64_t)i * t.dstr[k];
        r = q;
    }
}

// One contiguous run of nvec vectors: source(s) at element offset so, every
// destination at element offset dof. `lane`/`stride` split it among threads.
template <int VB>
__device__ __forceinline__ void run_copy(const KParams& p, const KTask& t, int es, int64_t so, int64_t dof,
                                         int64_t nvec, int lane, int stride)
{
    using V = typename Raw<VB>::T;
    const V* s = reinterpret_cast<const V*>(static_cast<const char*>(p.ptrs[t.ptr0]) + so * es);
    const int nd = t.n_dst;
    const void* const* dp = p.ptrs + t.ptr0 + 1;
    int64_t i = lane;
    for (; i + (int64_t)(kUnroll - 1) * stride < nvec; i += (int64_t)kUnroll * stride) {
        V v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) v[u] = __ldcs(s + i + u * stride);
        for (int j = 0; j < nd; ++j) {
            V* d = reinterpret_cast<V*>(static_cast<char*>(const_cast<void*>(dp[j])) + dof * es);
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) __stcs(d + i + u * stride, v[u]);
        }
    }
    for (; i < nvec; i += stride) {
        V v = __ldcs(s + i);
        for (int j = 0; j < nd; ++j) {
            V* d = reinterpret_cast<V*>(static_cast<char*>(const_cast<void*>(dp[j])) + dof * es);
            __stcs(d + i, v);
        }
    }
}

template <int VB>
__device__ __forceinline__ void run_zero(const KParams& p, const KTask& t, int es, int64_t dof, int64_t nvec,
                                         int lane, int stride)
{
    using V = typename Raw<VB>::T;
    Lanes<VB> z;
#pragma unroll
    for (int k = 0; k < VB / 2; ++k) z.h[k] = 0;
    const void* const* dp = p.ptrs + t.ptr0;
    for (int j = 0; j < t.n_dst; ++j) {
        V* d = reinterpret_cast<V*>(static_cast<char*>(const_cast<void*>(dp[j])) + dof * es);
        for (int64_t i = lane; i < nvec; i += stride) __stcs(d + i, z.v);
    }
}

// Sum of n_src sources. ES: element size (4 = float32, 2 = bf16).
template <int VB, int ES>
__device__ __forceinline__ void run_sum(const KParams& p, const KTask& t, int64_t so, int64_t dof, int64_t nvec,
                                        int lane, int stride)
{
    using V = typename Raw<VB>::T;
    constexpr int NE = VB / ES;  // elements per vector
    const int ns = t.n_src, nd = t.n_dst;
    const void* const* sp = p.ptrs + t.ptr0;
    const void* const* dp = sp + ns;
    for (int64_t i0 = lane; i0 < nvec; i0 += (int64_t)kUnroll * stride) {
        float acc[kUnroll][NE];
        bool live[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            live[u] = i0 + (int64_t)u * stride < nvec;
#pragma unroll
            for (int e = 0; e < NE; ++e) acc[u][e] = 0.f;
        }
        for (int j = 0; j < ns; ++j) {
            const V* s = reinterpret_cast<const V*>(static_cast<const char*>(sp[j]) + so * ES);
            Lanes<VB> in[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
                if (live[u]) in[u].v = __ldcs(s + i0 + u * stride);
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
#pragma unroll
                for (int e = 0; e < NE; ++e) {
                    float x;
                    if (ES == 4) x = __uint_as_float(in[u].w[e]);
                    else x = __uint_as_float((uint32_t)in[u].h[e] << 16);
                    acc[u][e] = j == 0 ? x : acc[u][e] + x;
                }
            }
        }
        Lanes<VB> out[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
#pragma unroll
            for (int e = 0; e < NE; ++e) {
                if (ES == 4) out[u].w[e] = __float_as_uint(acc[u][e]);
                else out[u].h[e] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[u][e]));
            }
        for (int j = 0; j < nd; ++j) {
            V* d = reinterpret_cast<V*>(static_cast<char*>(const_cast<void*>(dp[j])) + dof * ES);
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
                if (live[u]) __stcs(d + i0 + u * stride, out[u].v);
        }
    }
}

template <int VB>
__device__ __forceinline__ void run_any(const KParams& p, const KTask& t, int64_t so, int64_t dof, int64_t n,
                                        int lane, int stride)
{
    const int es = p.dtype == RTP_F32 ? 4 : 2;
    const int64_t nvec = n * es / VB;
    if (t.n_src == 1) {
        run_copy<VB>(p, t, es, so, dof, nvec, lane, stride);
    } else if (t.n_src == 0) {
        run_zero<VB>(p, t, es, dof, nvec, lane, stride);
    } else if (p.dtype == RTP_F32) {
        if constexpr (VB >= 4) run_sum<VB, 4>(p, t, so, dof, nvec, lane, stride);
    } else {
        run_sum<VB, 2>(p, t, so, dof, nvec, lane, stride);
    }
}

__device__ __forceinline__ void run(const KParams& p, const KTask& t, int64_t so, int64_t dof, int64_t n, int lane,
                                    int stride)
{
    switch (t.vec) {
    case 16: run_any<16>(p, t, so, dof, n, lane, stride); break;
    case 8: run_any<8>(p, t, so, dof, n, lane, stride); break;
    case 4: run_any<4>(p, t, so, dof, n, lane, stride); break;
    default: run_any<2>(p, t, so, dof, n, lane, stride); break;
    }
}

__global__ void __launch_bounds__(kBlock) boxing_kernel(const __grid_constant__ KParams p)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int64_t c = blockIdx.x; c < p.total_chunks; c += gridDim.x) {
        const KTask& t = p.tasks[find_task(p, c)];
        const int64_t lc = c - t.chunk_begin;
        int64_t so, dof;
        if (t.mode == 1) {
            const int64_t row = lc / t.nseg;
            const int64_t c0 = (lc - row * t.nseg) * t.seg;
            const int64_t n = min(t.seg, t.cols - c0);
            row_offsets(t, row, so, dof);
            run(p, t, so + c0, dof + c0, n, threadIdx.x, kBlock);
        } else {
            const int64_t r0 = lc * t.rpc;
            const int64_t r1 = min(r0 + t.rpc, t.rows);
            for (int64_t row = r0 + warp; row < r1; row += kWarps) {
                row_offsets(t, row, so, dof);
                run(p, t, so, dof, t.cols, lane, 32);
            }
        }
    }
}

int sm_count()
{
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (!cached[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        cached[dev] = n;
    }
    return cached[dev];
}

int pick_vec(const PlanTask& t, const void* const* src, void* const* dst, int es)
{
    for (int v = 16; v > es; v >>= 1) {
        bool ok = (t.cols * es) % v == 0;
        for (int k = 0; ok && k < t.n_outer; ++k)
            ok = t.ext[k] == 1 || ((t.sstr[k] * es) % v == 0 && (t.dstr[k] * es) % v == 0);
        for (const auto& r : t.src) ok = ok && ((uintptr_t)src[r.rank] + (uintptr_t)(r.offset * es)) % v == 0;
        for (const auto& r : t.dst) ok = ok && ((uintptr_t)dst[r.rank] + (uintptr_t)(r.offset * es)) % v == 0;
        if (ok) return v;
    }
    return es;
}

int64_t fill_task(KTask& k, const PlanTask& t, int vec, int es)
{
    std::memset(&k, 0, sizeof k);
    k.rows = t.rows;
    k.cols = t.cols;
    k.vec = vec;
    k.n_outer = t.n_outer;
    for (int i = 0; i < t.n_outer; ++i) {
        k.ext[i] = (int32_t)t.ext[i];
        k.sstr[i] = t.sstr[i];
        k.dstr[i] = t.dstr[i];
    }
    k.n_src = (int32_t)t.src.size();
    k.n_dst = (int32_t)t.dst.size();
    const int64_t row_bytes = t.cols * es;
    if (row_bytes >= (int64_t)kBlock * vec) {
        const int64_t epv = vec / es;
        int64_t seg = std::max<int64_t>(epv, (kChunkBytes / es) / epv * epv);
        seg = std::min(seg, t.cols);
        k.mode = 1;
        k.seg = seg;
        k.nseg = (t.cols + seg - 1) / seg;
        return t.rows * k.nseg;
    }
    k.mode = 0;
    int64_t rpc = std::max<int64_t>(kWarps, kChunkBytes / std::max<int64_t>(row_bytes, 1));
    rpc = std::min(rpc, t.rows);
    k.rpc = rpc;
    return (t.rows + rpc - 1) / rpc;
}

}  // namespace

int count_launches(const std::vector<PlanTask>& tasks)
{
    int launches = 0, nt = 0, np = 0;
    for (const auto& t : tasks) {
        int need = (int)(t.src.size() + t.dst.size());
        if (nt == kMaxTasks || np + need > kMaxPtrs) {
            ++launches;
            nt = 0;
            np = 0;
        }
        ++nt;
        np += need;
    }
    return launches + (nt > 0 ? 1 : 0);
}

int launch_tasks(int dtype, const std::vector<PlanTask>& tasks, const void* const* src, void* const* dst,
                 void* stream, int* n_launches_out)
{
    const int es = dtype == RTP_F32 ? 4 : 2;
    for (const auto& t : tasks) {
        if (t.rows >= (int64_t)1 << 31) return fail(RTP_EUNSUPPORTED, "reshard: region with 2^31 or more rows");
        for (int k = 0; k < t.n_outer; ++k)
            if (t.ext[k] >= (int64_t)1 << 31) return fail(RTP_EUNSUPPORTED, "reshard: extent of 2^31 or more");
        if (t.src.size() + t.dst.size() > (size_t)kMaxPtrs) return fail(RTP_EUNSUPPORTED, "reshard: too many buffers");
    }
    static thread_local KParams prm;  // large: keep it off the stack
    const int max_grid = sm_count() * kBlocksPerSm;
    int launches = 0;
    size_t i = 0;
    while (i < tasks.size()) {
        std::memset(&prm, 0, offsetof(KParams, tasks));
        prm.dtype = dtype;
        int np = 0;
        int64_t chunks = 0;
        int nt = 0;
        for (; i < tasks.size() && nt < kMaxTasks; ++i) {
            const PlanTask& t = tasks[i];
            const int need = (int)(t.src.size() + t.dst.size());
            if (np + need > kMaxPtrs) break;
            KTask& k = prm.tasks[nt];
            int64_t nc = fill_task(k, t, pick_vec(t, src, dst, es), es);
            k.chunk_begin = chunks;
            k.ptr0 = np;
            for (const auto& r : t.src) prm.ptrs[np++] = static_cast<const char*>(src[r.rank]) + r.offset * es;
            for (const auto& r : t.dst) prm.ptrs[np++] = static_cast<char*>(dst[r.rank]) + r.offset * es;
            chunks += nc;
            ++nt;
        }
        prm.n_tasks = nt;
        prm.total_chunks = chunks;
        if (chunks == 0) continue;
        const int grid = (int)std::min<int64_t>(chunks, max_grid);
        boxing_kernel<<<grid, kBlock, 0, static_cast<cudaStream_t>(stream)>>>(prm);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return fail(RTP_ECUDA, "boxing kernel launch failed: %s", cudaGetErrorString(e));
        ++launches;
    }
    if (n_launches_out) *n_launches_out = launches;
    return RTP_OK;
}

}  // namespace rtp
