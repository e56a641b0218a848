// Boxing kernel: executes planned reshard tasks (copies, partial sums, zero
// fills) for shard() and reshard().
//
// Design for GB300 (HBM-bound, no tensor-core work):
//   * the task table travels in the kernel parameters (3 to 26 KB per launch,
//     __grid_constant__, sized to the launch's tasks), so no device memory is
//     allocated or copied per call and the launch can be captured in a CUDA
//     graph;
//   * blocks of 256 threads (up to 4 resident per SM) each take one chunk of
//     a task. Alone on the GPU the grid has one block per chunk; beside another
//     kernel it is a persistent grid of a few blocks per SM;
//   * three forms, chosen per task on the host:
//       - bulk staging: runs of 4 KB or more are loaded into shared memory
//         with cp.async.bulk (the TMA engine, no tensor map) and stored from
//         there, or summed from there;
//       - TMA tiles: shorter rows whose one side is contiguous move the strided
//         side as one cp.async.bulk.tensor tile of a 3D / 4D tensor map per
//         source (or destination) and chunk (the axis-changing S(i) -> S(j)
//         moves, the P -> S reduce-scatter); a launch of single-destination
//         tile copies only runs in small blocks of 128 threads, more of them
//         per SM;
//       - registers: every other task; the block stages each row's offsets in
//         shared memory and spreads (row, vector) items over its threads, so
//         every thread keeps several loads in flight even for short rows;
//   * 16-byte vectors whenever every pointer, stride and run length allows it
//     (else 8, 4 or 2 bytes), streaming cache hints since every byte is
//     touched once;
//   * a task with several destinations (broadcast pieces) reads its source
//     once and writes every destination from the same registers or shared
//     memory;
//   * a task with several sources (partial sums) adds them in float32 in a
//     fixed order (partial coordinates row-major) and rounds once; partial
//     min / max members combine with fminf / fmaxf (exact);
//   * a task with no source fills its destinations with the identity of the
//     destination's partial reduction (0, +inf or -inf);
//   * every wait on a bulk or tile copy is bounded (about 2 s); a wait that
//     gives up records a code in a device word and the block returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <unordered_map>

#include "rtp_internal.h"

namespace rtp {

namespace {

constexpr int kBlock = 256;
constexpr int64_t kChunkBytes = 32 * 1024;
constexpr int kMaxTasks = 96;
constexpr int kMaxPtrs = 640;
constexpr int kBulkMinRowBytes = 4096;        // shorter rows take the register path (measured: bulk copies of 1-2 KB rows are slower)
constexpr int64_t kBulkStageBytes = 64 * 1024;  // shared staging of a reduction chunk (all sources)
constexpr int kBulkDynSmem = 64 * 1024;       // dynamic shared memory a launch may request
// Shared staging of a tile-form sum chunk (all sources): 48 KB lets four
// 256-thread blocks share an SM (measured: the bf16 P-sum of 8 -> S(2), whose
// 1 KB rows filled 56 KB at 7 rows a source, 2-3 % faster at 6 rows).
constexpr int64_t kTileSumStageBytes = 48 * 1024;
constexpr unsigned long long kBulkWaitNs = 2000000000ull;
constexpr uint32_t kErrBulkWait = 16;         // device error code: a bulk copy never completed

__device__ unsigned int g_box_error;

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint64_t now_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait for phase `parity` of an mbarrier; false (and the error word
// set) when it does not complete within kBulkWaitNs.
__device__ __noinline__ bool bar_wait(uint32_t bar, uint32_t parity, unsigned long long limit_ns = kBulkWaitNs)
{
    const uint64_t t0 = now_ns();
    for (uint32_t i = 0;; ++i) {
        uint32_t done;
        asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
                     : "=r"(done)
                     : "r"(bar), "r"(parity)
                     : "memory");
        if (done) return true;
        if ((i & 15u) == 15u && now_ns() - t0 > limit_ns) {
            atomicCAS(&g_box_error, 0u, kErrBulkWait);
            return false;
        }
    }
}

// Self-test of the bounded wait above: every thread of one block waits (as a
// staged chunk does) on an mbarrier whose transaction bytes never arrive; the
// waits give up after limit_ns, record kErrBulkWait, and the block agrees to
// stop. out[0] = 1 when the block stopped on the failed wait.
__global__ void bulk_wait_selftest_kernel(unsigned long long limit_ns, uint32_t* out)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&bar)) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        // 16 bytes announced, none sent: the phase cannot complete
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(&bar)), "r"(16u) : "memory");
    }
    __syncthreads();
    const int ok = __syncthreads_and(bar_wait(su32(&bar), 0, limit_ns) ? 1 : 0);
    if (threadIdx.x == 0) out[0] = ok ? 0u : 1u;
}

// Bulk copies (cp.async.bulk, no tensor map): 16-byte aligned addresses, sizes
// multiple of 16. Loads complete on an mbarrier; stores form a bulk group.
__device__ __forceinline__ void bulk_load(uint32_t dst_smem, const void* src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst_smem), "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}
__device__ __forceinline__ void bulk_store(void* dst, uint32_t src_smem, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src_smem), "r"(bytes)
                 : "memory");
}

// TMA tiles over a view [outer][rows][mid][inner] of a strided row region (4D;
// 3D without the outer dim); the box is rows-per-chunk x mid x inner of one
// outer index, i.e. whole rows, dense in shared memory. Rows past the region
// are zero-filled on load (and count toward the bytes) and skipped on store.
template <int R>
__device__ __forceinline__ void tile_load(uint32_t dst_smem, const CUtensorMap* map, int n_outer, int row, int outer,
                                          uint32_t bar)
{
    const uint64_t m = reinterpret_cast<uint64_t>(map);
    if (R == 3 || n_outer == 1)
        asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
                     ::"r"(dst_smem), "l"(m), "r"(0), "r"(0), "r"(row), "r"(bar)
                     : "memory");
    else
        asm volatile("cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], [%6];"
                     ::"r"(dst_smem), "l"(m), "r"(0), "r"(0), "r"(row), "r"(outer), "r"(bar)
                     : "memory");
}
template <int R>
__device__ __forceinline__ void tile_store(const CUtensorMap* map, int n_outer, int row, int outer, uint32_t src_smem)
{
    const uint64_t m = reinterpret_cast<uint64_t>(map);
    if (R == 3 || n_outer == 1)
        asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];"
                     ::"l"(m), "r"(0), "r"(0), "r"(row), "r"(src_smem)
                     : "memory");
    else
        asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3, %4}], [%5];"
                     ::"l"(m), "r"(0), "r"(0), "r"(row), "r"(outer), "r"(src_smem)
                     : "memory");
}

struct KTask {
    int64_t chunk_begin;  // first chunk index of this task within the launch
    int64_t rows, cols;   // region: rows runs of cols contiguous elements
    int64_t seg, nseg;    // column segment (elements) and segments per row
    int32_t rpc;          // rows per chunk (1 when rows are cut into segments)
    int32_t vec;          // bytes per vector access
    int32_t n_outer, n_src, n_dst, ptr0;
    int32_t ext[kMaxOuter];
    int32_t op;           // RED_SUM / RED_MIN / RED_MAX: how several sources combine
    uint32_t fill;        // with no source: the element pattern written (the op's identity),
                          // repeated to 32 bits for 16-bit elements
    int32_t bulk;         // 1: staged through shared memory with bulk (TMA) copies
    int32_t tile;         // 1: sources read as TMA tiles (rows strided), destination rows contiguous;
                          // 2: source rows contiguous, destinations written as TMA tiles
    int32_t map0;         // first tensor map of the task (sources for tile 1, destinations for tile 2)
    int64_t sstr[kMaxOuter], dstr[kMaxOuter];
};

// The parameter block of one launch. A launch copies the whole declared block,
// so launches with few tasks use a smaller form (about 3 KB or 11 KB instead
// of 26 KB): measured, that saves microseconds on every short reshard.
template <int MT, int MP>
struct KParamsT {
    int32_t n_tasks;
    int32_t dtype;
    int64_t total_chunks;
    KTask tasks[MT];
    const void* ptrs[MP];  // per task: n_src source bases, then n_dst destination bases
    static constexpr int kMaps = 0;
};
using KParams = KParamsT<kMaxTasks, kMaxPtrs>;

// The form for launches with TMA-tile tasks: the tensor maps of their strided
// sides travel with the tasks.
// R = 3: every tile task has one outer dim (3D maps); R = 4: some have two.
constexpr int kTileTasks = 64, kTilePtrs = 256, kTileMaps = 64;
template <int R>
struct KParamsTileT {
    int32_t n_tasks;
    int32_t dtype;
    int64_t total_chunks;
    KTask tasks[kTileTasks];
    const void* ptrs[kTilePtrs];
    CUtensorMap maps[kTileMaps];
    static constexpr int kMaps = kTileMaps;
    static constexpr int kTileRank = R;
};
using KParamsTile3 = KParamsTileT<3>;
using KParamsTile4 = KParamsTileT<4>;
static_assert(sizeof(KParamsTile4) <= 32000, "kernel parameter block too large");
constexpr int kSmallTasks = 16, kSmallPtrs = 128, kMediumTasks = 64, kMediumPtrs = 256;
using KParamsSmall = KParamsT<kSmallTasks, kSmallPtrs>;
using KParamsMedium = KParamsT<kMediumTasks, kMediumPtrs>;
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

template <class PP>
__device__ __forceinline__ int find_task(const PP& p, int64_t c)
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

// jj = q * nv + r with 0 <= r < nv, for jj < 2^24: a float estimate, then one correction.
__device__ __forceinline__ void divmod(int jj, int nv, float inv, int& q, int& r)
{
    q = (int)((float)jj * inv);
    r = jj - q * nv;
    if (r < 0) {
        --q;
        r += nv;
    } else if (r >= nv) {
        ++q;
        r -= nv;
    }
}

// Items (row, vector) of one chunk are spread over the block, U per thread per
// pass: item j is vector j % nv of row j / nv; s_off / d_off hold each row's
// first element offset (relative to the task's buffers).
template <int VB, int ES, int U>
struct Items {
    using V = typename Raw<VB>::T;
    int q[U], r[U];  // row and vector of each item; r < 0 marks a dead item
    const int64_t* s_off;
    const int64_t* d_off;
    __device__ __forceinline__ void at(int j0, int total, int nv, float inv)
    {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int jj = j0 + u * kBlock;
            q[u] = 0;
            r[u] = -1;
            if (jj < total) divmod(jj, nv, inv, q[u], r[u]);
        }
    }
    __device__ __forceinline__ const V* src(const void* base, int u) const
    {
        return reinterpret_cast<const V*>(static_cast<const char*>(base) + s_off[q[u]] * ES) + r[u];
    }
    __device__ __forceinline__ V* dst(const void* base, int u) const
    {
        return reinterpret_cast<V*>(static_cast<char*>(const_cast<void*>(base)) + d_off[q[u]] * ES) + r[u];
    }
};

// No source: every destination gets the fill pattern (the identity of the
// destination's partial reduction).
template <int VB, int ES>
__device__ __forceinline__ void fill_chunk(const void* const* ptrs, const KTask& t, int total, int nv, const int64_t* s_off,
                                           const int64_t* d_off)
{
    constexpr int U = 4;
    Items<VB, ES, U> it{{}, {}, s_off, d_off};
    Lanes<VB> z;
#pragma unroll
    for (int k = 0; k < VB / 2; ++k) z.h[k] = (uint16_t)(t.fill >> (16 * (k & 1)));
    const float inv = 1.0f / (float)nv;
    const void* const* dp = ptrs + t.ptr0;
    for (int j0 = threadIdx.x; j0 < total; j0 += kBlock * U) {
        it.at(j0, total, nv, inv);
        for (int j = 0; j < t.n_dst; ++j)
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (it.r[u] >= 0) __stcs(it.dst(dp[j], u), z.v);
    }
}

// One source: its bits go to every destination (read once).
template <int VB, int ES>
__device__ __forceinline__ void copy_chunk(const void* const* ptrs, const KTask& t, int total, int nv, const int64_t* s_off,
                                           const int64_t* d_off)
{
    constexpr int U = 4;
    using V = typename Raw<VB>::T;
    Items<VB, ES, U> it{{}, {}, s_off, d_off};
    const float inv = 1.0f / (float)nv;
    const void* const* sp = ptrs + t.ptr0;
    const void* const* dp = sp + 1;
    for (int j0 = threadIdx.x; j0 < total; j0 += kBlock * U) {
        it.at(j0, total, nv, inv);
        V x[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (it.r[u] >= 0) x[u] = __ldcs(it.src(sp[0], u));
        for (int j = 0; j < t.n_dst; ++j)
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (it.r[u] >= 0) __stcs(it.dst(dp[j], u), x[u]);
    }
}

// One source, float32, narrow vectors (8 or 4 bytes: a row or pointer not
// 16-byte aligned) and long rows: the block walks the chunk row by row, each thread
// moving UR vectors of a row (strided by the block size) per pass, loads
// first, so that 8 vectors a thread are in flight with no per-item row table
// (copy_chunk's (row, vector) items keep 4 a thread); the row's end goes in
// one pass of 4, then one vector at a time. Not inlined: its registers stay
// out of the allocation of the kernel's other paths.
template <int VB, int ES>
__device__ __noinline__ void copy_rows(const void* const* ptrs, const KTask& t, int nr, int nv, const int64_t* s_off,
                                       const int64_t* d_off)
{
    constexpr int UR = 8;
    using V = typename Raw<VB>::T;
    const char* sb = static_cast<const char*>(ptrs[t.ptr0]);
    const void* const* dp = ptrs + t.ptr0 + 1;
    for (int q = 0; q < nr; ++q) {
        const V* src = reinterpret_cast<const V*>(sb + s_off[q] * ES);
        int v0 = threadIdx.x;
        for (; v0 + (UR - 1) * kBlock < nv; v0 += kBlock * UR) {
            V x[UR];
#pragma unroll
            for (int u = 0; u < UR; ++u) x[u] = __ldcs(src + v0 + u * kBlock);
            for (int j = 0; j < t.n_dst; ++j) {
                V* dst = reinterpret_cast<V*>(static_cast<char*>(const_cast<void*>(dp[j])) + d_off[q] * ES) + v0;
#pragma unroll
                for (int u = 0; u < UR; ++u) __stcs(dst + u * kBlock, x[u]);
            }
        }
        if (v0 + 3 * kBlock < nv) {  // a pass of 4
            V x[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) x[u] = __ldcs(src + v0 + u * kBlock);
            for (int j = 0; j < t.n_dst; ++j) {
                V* dst = reinterpret_cast<V*>(static_cast<char*>(const_cast<void*>(dp[j])) + d_off[q] * ES) + v0;
#pragma unroll
                for (int u = 0; u < 4; ++u) __stcs(dst + u * kBlock, x[u]);
            }
            v0 += 4 * kBlock;
        }
        for (; v0 < nv; v0 += kBlock) {
            const V x = __ldcs(src + v0);
            for (int j = 0; j < t.n_dst; ++j)
                __stcs(reinterpret_cast<V*>(static_cast<char*>(const_cast<void*>(dp[j])) + d_off[q] * ES) + v0, x);
        }
    }
}

template <int OP>
__device__ __forceinline__ float combine(float acc, float x)
{
    if constexpr (OP == RED_SUM) return acc + x;
    else if constexpr (OP == RED_MIN) return fminf(acc, x);
    else return fmaxf(acc, x);
}

// Several sources combined element-wise in float32 in source order (partial
// coordinates row-major), starting from the reduction's identity, rounded once
// to the element type.
template <int VB, int ES, int OP>
__device__ __forceinline__ void reduce_chunk(const void* const* ptrs, const KTask& t, int total, int nv, const int64_t* s_off,
                                             const int64_t* d_off)
{
    constexpr int U = 2;
    constexpr int NE = VB / ES;  // elements per vector
    using V = typename Raw<VB>::T;
    Items<VB, ES, U> it{{}, {}, s_off, d_off};
    const float inv = 1.0f / (float)nv;
    const int ns = t.n_src;
    const void* const* sp = ptrs + t.ptr0;
    const void* const* dp = sp + ns;
    const float ident = OP == RED_SUM ? 0.0f : (OP == RED_MIN ? __int_as_float(0x7F800000) : __int_as_float(0xFF800000));
    for (int j0 = threadIdx.x; j0 < total; j0 += kBlock * U) {
        it.at(j0, total, nv, inv);
        float acc[U][NE];
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int e = 0; e < NE; ++e) acc[u][e] = ident;
#pragma unroll 8
        for (int j = 0; j < ns; ++j) {
            Lanes<VB> in[U];
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (it.r[u] >= 0) in[u].v = __ldcs(it.src(sp[j], u));
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int e = 0; e < NE; ++e) {
                    float x;
                    if constexpr (ES == 4) x = __uint_as_float(in[u].w[e]);
                    else x = __uint_as_float((uint32_t)in[u].h[e] << 16);
                    acc[u][e] = combine<OP>(acc[u][e], x);
                }
        }
        Lanes<VB> out[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int e = 0; e < NE; ++e) {
                if constexpr (ES == 4) out[u].w[e] = __float_as_uint(acc[u][e]);
                else out[u].h[e] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[u][e]));
            }
        for (int j = 0; j < t.n_dst; ++j)
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (it.r[u] >= 0) __stcs(it.dst(dp[j], u), out[u].v);
    }
}

template <int VB, int ES, bool SUM, int OP>
__device__ __forceinline__ void run_chunk(const void* const* ptrs, const KTask& t, int nr, int nv, const int64_t* s_off,
                                          const int64_t* d_off)
{
    const int total = nr * nv;
    if (t.n_src == 0) {
        fill_chunk<VB, ES>(ptrs, t, total, nv, s_off, d_off);
    } else if (ES == 4 && VB < 16 && (!SUM || t.n_src == 1) && nv >= 4 * kBlock) {
        if constexpr (ES == 4 && VB < 16) copy_rows<VB, ES>(ptrs, t, nr, nv, s_off, d_off);
    } else if (!SUM || t.n_src == 1) {
        copy_chunk<VB, ES>(ptrs, t, total, nv, s_off, d_off);
    } else if constexpr (SUM) {
        reduce_chunk<VB, ES, OP>(ptrs, t, total, nv, s_off, d_off);
    }
}

// A chunk staged through shared memory: warp 0 bulk-loads every source's rows
// (source j, row r at (j nr + r) rowbytes), all threads wait on the block's
// mbarrier, then a copy is bulk-stored from shared memory to every destination
// (the same bytes, read once), or a reduction is added up by all threads in
// float32 in source order and stored with streaming stores. False when a wait
// gave up (the error word is set).
template <bool SUM, int ES, int OP>
__device__ __forceinline__ bool bulk_chunk(const void* const* ptrs, const KTask& t, int nr, uint32_t rowbytes,
                                           const int64_t* s_off, const int64_t* d_off, uint8_t* stage, uint32_t bar,
                                           uint32_t parity)
{
    const int ns = t.n_src;
    const void* const* sp = ptrs + t.ptr0;
    const void* const* dp = sp + ns;
    const uint32_t st0 = su32(stage);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == 0) {
        if (lane == 0)
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                         "r"((uint32_t)ns * (uint32_t)nr * rowbytes)
                         : "memory");
        __syncwarp();
        for (int j = 0; j < ns; ++j)
            for (int r = lane; r < nr; r += 32)
                bulk_load(st0 + (uint32_t)(j * nr + r) * rowbytes, static_cast<const char*>(sp[j]) + s_off[r] * ES,
                          rowbytes, bar);
    }
    if (!__syncthreads_and(bar_wait(bar, parity) ? 1 : 0)) return false;
    if (ns == 1) {
        if (warp == 0) {
            for (int k = 0; k < t.n_dst; ++k)
                for (int r = lane; r < nr; r += 32)
                    bulk_store(static_cast<char*>(const_cast<void*>(dp[k])) + d_off[r] * ES, st0 + (uint32_t)r * rowbytes,
                               rowbytes);
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");  // shared memory read before reuse
        }
        return true;
    }
    if constexpr (SUM) {
        constexpr int NE = 16 / ES;
        const int vpr = (int)(rowbytes / 16);
        const int total = nr * vpr;
        const float inv = 1.0f / (float)vpr;
        const size_t src_stride = (size_t)nr * rowbytes;  // a source's rows are dense in the staging
        const float ident = OP == RED_SUM ? 0.0f : (OP == RED_MIN ? __int_as_float(0x7F800000) : __int_as_float(0xFF800000));
        for (int i = threadIdx.x; i < total; i += kBlock) {
            int r = 0, v = i;
            if (nr > 1) divmod(i, vpr, inv, r, v);  // block-uniform: segments have one row
            float acc[NE];
#pragma unroll
            for (int e = 0; e < NE; ++e) acc[e] = ident;
#pragma unroll 8
            for (int j = 0; j < ns; ++j) {
                Lanes<16> x;
                x.v = *reinterpret_cast<const uint4*>(stage + (size_t)j * src_stride + (size_t)i * 16);
#pragma unroll
                for (int e = 0; e < NE; ++e) {
                    float y;
                    if constexpr (ES == 4) y = __uint_as_float(x.w[e]);
                    else y = __uint_as_float((uint32_t)x.h[e] << 16);
                    acc[e] = combine<OP>(acc[e], y);
                }
            }
            Lanes<16> out;
#pragma unroll
            for (int e = 0; e < NE; ++e) {
                if constexpr (ES == 4) out.w[e] = __float_as_uint(acc[e]);
                else out.h[e] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[e]));
            }
            for (int k = 0; k < t.n_dst; ++k)
                __stcs(reinterpret_cast<uint4*>(static_cast<char*>(const_cast<void*>(dp[k])) + d_off[r] * ES) + v, out.v);
        }
    }
    return true;
}

// Staging bytes of one source's box in shared memory (128-byte aligned slots).
__device__ __host__ __forceinline__ uint32_t tile_slot(int64_t rpc, int64_t row_bytes)
{
    return (uint32_t)((rpc * row_bytes + 127) / 128 * 128);
}

// Chunk `lc` of a region with one or two outer dims: rows r1 .. r1+nr of the
// inner row dim at outer index o (o = 0 with one outer dim), staged through
// shared memory. tile 1: each source's rows arrive as one TMA tile (its rows
// are strided), the destination rows are contiguous within an outer index: a
// copy is one bulk store per destination, a reduction is added up by all
// threads and stored with streaming stores. tile 2 (copies): the source rows
// are contiguous (one bulk load), each destination is written as one TMA
// tile. False when a wait gave up (the error word is set).
template <class PP, bool SUM, int ES, int OP>
__device__ __forceinline__ bool tile_chunk(const PP& p, const KTask& t, int64_t lc, uint32_t row_bytes, uint8_t* stage,
                                           uint32_t bar, uint32_t parity)
{
    constexpr int R = PP::kTileRank;
    const int inn = R == 3 ? 0 : t.n_outer - 1;  // the inner row dim
    const int64_t ext_in = t.ext[inn];
    int64_t o = 0, r1 = lc * t.rpc;
    if (R == 4 && inn > 0) {  // chunks never straddle two outer indices
        const int64_t nb = (ext_in + t.rpc - 1) / t.rpc;
        o = lc / nb;
        r1 = (lc - o * nb) * t.rpc;
    }
    const int nr = (int)min((int64_t)t.rpc, ext_in - r1);
    // element offsets of the chunk's first row on the contiguous sides
    const int64_t soff = (R == 4 && inn > 0 ? o * t.sstr[0] : 0) + r1 * t.sstr[inn];
    const int64_t doff = (R == 4 && inn > 0 ? o * t.dstr[0] : 0) + r1 * t.dstr[inn];
    const int ns = t.n_src;
    const void* const* sp = p.ptrs + t.ptr0;
    const void* const* dp = sp + ns;
    const uint32_t st0 = su32(stage);
    const uint32_t slot = tile_slot(t.rpc, row_bytes);
    const bool first = threadIdx.x == 0;
    if (first) {
        if (t.tile == 1) {
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                         "r"((uint32_t)ns * (uint32_t)t.rpc * row_bytes)
                         : "memory");
            for (int j = 0; j < ns; ++j)
                tile_load<R>(st0 + (uint32_t)j * slot, &p.maps[t.map0 + j], t.n_outer, (int)r1, (int)o, bar);
        } else {
            const uint32_t bytes = (uint32_t)nr * row_bytes;
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
            bulk_load(st0, static_cast<const char*>(sp[0]) + soff * ES, bytes, bar);
        }
    }
    if (!__syncthreads_and(bar_wait(bar, parity) ? 1 : 0)) return false;
    if (ns == 1) {
        if (first) {
            for (int k = 0; k < t.n_dst; ++k) {
                if (t.tile == 1)
                    bulk_store(static_cast<char*>(const_cast<void*>(dp[k])) + doff * ES, st0, (uint32_t)nr * row_bytes);
                else
                    tile_store<R>(&p.maps[t.map0 + k], t.n_outer, (int)r1, (int)o, st0);
            }
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
        }
        return true;
    }
    if constexpr (SUM) {
        constexpr int NE = 16 / ES;
        const int total = (int)((uint32_t)nr * row_bytes / 16);  // vectors; destination rows are contiguous
        const float ident = OP == RED_SUM ? 0.0f : (OP == RED_MIN ? __int_as_float(0x7F800000) : __int_as_float(0xFF800000));
        for (int i = threadIdx.x; i < total; i += kBlock) {
            float acc[NE];
#pragma unroll
            for (int e = 0; e < NE; ++e) acc[e] = ident;
#pragma unroll 8
            for (int j = 0; j < ns; ++j) {
                Lanes<16> x;
                x.v = *reinterpret_cast<const uint4*>(stage + (size_t)j * slot + (size_t)i * 16);
#pragma unroll
                for (int e = 0; e < NE; ++e) {
                    float y;
                    if constexpr (ES == 4) y = __uint_as_float(x.w[e]);
                    else y = __uint_as_float((uint32_t)x.h[e] << 16);
                    acc[e] = combine<OP>(acc[e], y);
                }
            }
            Lanes<16> out;
#pragma unroll
            for (int e = 0; e < NE; ++e) {
                if constexpr (ES == 4) out.w[e] = __float_as_uint(acc[e]);
                else out.h[e] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[e]));
            }
            for (int k = 0; k < t.n_dst; ++k)
                __stcs(reinterpret_cast<uint4*>(static_cast<char*>(const_cast<void*>(dp[k])) + doff * ES) + i, out.v);
        }
    }
    return true;
}

// SUM = false: copies and fills only; SUM = true: also multi-source
// reductions with OP (every reduction of one launch has the same op, that of
// the source spec). ES: element size in bytes.
template <class PP, bool SUM, int ES, int OP>
__global__ void __launch_bounds__(kBlock, 4) boxing_kernel(const __grid_constant__ PP p)
{
    __shared__ int64_t s_off[kBlock], d_off[kBlock];
    __shared__ __align__(8) uint64_t bar;
    extern __shared__ __align__(128) uint8_t stage[];  // bulk staging; sized by the launch
    if (threadIdx.x == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&bar)) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    uint32_t parity = 0;  // phase of `bar` for the next bulk chunk of this block
    for (int64_t c = blockIdx.x; c < p.total_chunks; c += gridDim.x) {
        const KTask& t = p.tasks[find_task(p, c)];
        const int64_t lc = c - t.chunk_begin;
        const int64_t rb = lc / t.nseg;
        const int64_t c0 = (lc - rb * t.nseg) * t.seg;
        const int64_t r0 = rb * t.rpc;
        const int nr = (int)min((int64_t)t.rpc, t.rows - r0);
        const int64_t len = min(t.seg, t.cols - c0);
        if (t.bulk && nr == 1) {  // one segment: every thread derives its offsets, no row table
            int64_t so, dof;
            row_offsets(t, r0, so, dof);
            so += c0;
            dof += c0;
            if (!bulk_chunk<SUM, ES, OP>(p.ptrs, t, 1, (uint32_t)(len * ES), &so, &dof, stage, su32(&bar), parity))
                return;  // a bulk copy never completed: the error word is set
            parity ^= 1u;
            __syncthreads();
            continue;
        }
        if constexpr (PP::kMaps > 0) {
            if (t.tile) {  // block-uniform
                if (!tile_chunk<PP, SUM, ES, OP>(p, t, lc, (uint32_t)(t.cols * ES), stage, su32(&bar), parity))
                    return;  // a bulk copy never completed: the error word is set
                parity ^= 1u;
                __syncthreads();
                continue;
            }
        }
        if ((int)threadIdx.x < nr) {
            int64_t so, dof;
            row_offsets(t, r0 + threadIdx.x, so, dof);
            s_off[threadIdx.x] = so + c0;
            d_off[threadIdx.x] = dof + c0;
        }
        __syncthreads();
        if (t.bulk) {  // block-uniform
            if (!bulk_chunk<SUM, ES, OP>(p.ptrs, t, nr, (uint32_t)(len * ES), s_off, d_off, stage, su32(&bar), parity))
                return;  // a bulk copy never completed: the error word is set
            parity ^= 1u;
            __syncthreads();
            continue;
        }
        const int nv = (int)(len * ES / t.vec);
        switch (t.vec) {
        case 16: run_chunk<16, ES, SUM, OP>(p.ptrs, t, nr, nv, s_off, d_off); break;
        case 8: run_chunk<8, ES, SUM, OP>(p.ptrs, t, nr, nv, s_off, d_off); break;
        case 4: run_chunk<4, ES, SUM, OP>(p.ptrs, t, nr, nv, s_off, d_off); break;
        default:
            if constexpr (ES == 2) run_chunk<2, ES, SUM, OP>(p.ptrs, t, nr, nv, s_off, d_off);
            break;
        }
        __syncthreads();
    }
}

// Launches whose every task is a TMA-tile copy to one destination: thread 0
// of a block moves a chunk (one bulk or tile load, then one tile or bulk
// store) and the other threads only wait, so the block is small and has no
// row tables: 6 blocks (6 chunks in flight) fit on an SM where 4 of
// boxing_kernel's do. Measured on the bf16 S(2) -> S(1) move of the
// [8,2048,4096] sweep on a 1x8 mesh (4D tiles): 6.30 -> 6.61 TB/s.
constexpr int kTileBlock = 128;

template <class PP, int ES>
__global__ void __launch_bounds__(kTileBlock, 8) tile_copy_kernel(const __grid_constant__ PP p)
{
    __shared__ __align__(8) uint64_t bar;
    extern __shared__ __align__(128) uint8_t stage[];  // sized by the launch
    if (threadIdx.x == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&bar)) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    uint32_t parity = 0;
    for (int64_t c = blockIdx.x; c < p.total_chunks; c += gridDim.x) {
        const KTask& t = p.tasks[find_task(p, c)];
        if (!tile_chunk<PP, false, ES, RED_SUM>(p, t, c - t.chunk_begin, (uint32_t)(t.cols * ES), stage, su32(&bar),
                                                 parity))
            return;  // a copy never completed: the error word is set
        parity ^= 1u;
        __syncthreads();
    }
}

int sm_count()
{
    static std::atomic<int> cached[64];  // 0 = not yet queried
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    int n = cached[dev].load(std::memory_order_relaxed);
    if (!n) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        cached[dev].store(n, std::memory_order_relaxed);
    }
    return n;
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

// Inner extent of the 3D tile view [rows][cols / inner][inner] of a row of
// `cols` elements: the largest divisor of cols of at most 256 elements whose
// bytes are a multiple of 16, with cols / inner at most 256 (0: none).
int64_t tile_inner(int64_t cols, int es)
{
    for (int64_t d = std::min<int64_t>(cols, 256); d >= 1; --d)
        if (cols % d == 0 && (d * es) % 16 == 0) return cols / d <= 256 ? d : 0;
    return 0;
}

// Everything a tile map is encoded from (the rank follows from dims[3]).
struct MapKey {
    uintptr_t ptr;
    uint64_t dims[4];
    uint64_t strides[3];
    uint32_t rpc;
    int es;
    bool operator==(const MapKey& o) const
    {
        return ptr == o.ptr && std::memcmp(dims, o.dims, sizeof dims) == 0 &&
               std::memcmp(strides, o.strides, sizeof strides) == 0 && rpc == o.rpc && es == o.es;
    }
};
struct MapKeyHash {
    size_t operator()(const MapKey& k) const
    {
        uint64_t h = k.ptr * 0x9E3779B97F4A7C15ull;
        for (uint64_t v : k.dims) h = (h ^ v) * 0x100000001B3ull;
        for (uint64_t v : k.strides) h = (h ^ v) * 0x100000001B3ull;
        return (size_t)(h ^ ((uint64_t)k.rpc << 3) ^ (uint64_t)k.es);
    }
};

// Per thread, like the rest of the launch state (no locking).
std::unordered_map<MapKey, CUtensorMap, MapKeyHash>& map_cache()
{
    static thread_local std::unordered_map<MapKey, CUtensorMap, MapKeyHash> cache;
    return cache;
}

// The tensor map of a tile task's strided side: base `ptr`, rows of `cols`
// elements in n_outer (1 or 2) outer dims of extents ext and element strides
// str (outer first); box: rpc whole rows of one outer index.
int encode_tile_map(CUtensorMap* m, const void* ptr, int n_outer, const int32_t* ext, const int64_t* str, int64_t cols,
                    int64_t rpc, int es)
{
    auto fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encoder());
    if (!fn) return fail(RTP_ECUDA, "reshard: cuTensorMapEncodeTiled is unavailable");
    const int64_t inner = tile_inner(cols, es);
    const int rank = 2 + n_outer;
    cuuint64_t dims[4] = {(cuuint64_t)inner, (cuuint64_t)(cols / inner), (cuuint64_t)ext[n_outer - 1],
                          n_outer == 2 ? (cuuint64_t)ext[0] : 1u};
    cuuint64_t strides[3] = {(cuuint64_t)(inner * es), (cuuint64_t)(str[n_outer - 1] * es),
                             n_outer == 2 ? (cuuint64_t)(str[0] * es) : 0u};
    cuuint32_t box[4] = {(cuuint32_t)inner, (cuuint32_t)(cols / inner), (cuuint32_t)rpc, 1u};
    cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    // Repeated reshards of the same buffers reuse their maps (encoding one takes
    // a fraction of a microsecond; a 64-task launch needs 64).
    MapKey key{reinterpret_cast<uintptr_t>(ptr), {dims[0], dims[1], dims[2], dims[3]}, {strides[0], strides[1], strides[2]},
               (uint32_t)rpc, es};
    auto& cache = map_cache();
    auto it = cache.find(key);
    if (it != cache.end()) {
        *m = it->second;
        return RTP_OK;
    }
    CUresult r = fn(m, es == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank,
                    const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(RTP_ECUDA, "reshard: cuTensorMapEncodeTiled failed (%d)", (int)r);
    if (cache.size() >= 4096) cache.clear();
    cache.emplace(key, *m);
    return RTP_OK;
}

// Chunking: rows longer than a chunk are cut into segments (one row per
// chunk); shorter rows are grouped, up to one row per thread of the block.
int64_t fill_task(KTask& k, const PlanTask& t, int vec, int es, bool allow_bulk)
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
    k.op = t.op;
    // identity of the reduction: 0 (sum), +inf (min), -inf (max)
    if (es == 4) k.fill = t.op == RED_MIN ? 0x7F800000u : t.op == RED_MAX ? 0xFF800000u : 0u;
    else k.fill = t.op == RED_MIN ? 0x7F807F80u : t.op == RED_MAX ? 0xFF80FF80u : 0u;
    const int64_t row_bytes = t.cols * es;
    const int64_t epv = vec / es;
    const int64_t ns = (int64_t)t.src.size();
    // Staged through shared memory (bulk copies) when vectors are 16 bytes, the
    // rows or segments are long, and every source's chunk fits the staging.
    const int64_t bulk_chunk_bytes = ns <= 1 ? kChunkBytes : std::max<int64_t>(4096, kBulkStageBytes / std::max<int64_t>(ns, 1));
    k.bulk = allow_bulk && vec == 16 && ns >= 1 && ns * bulk_chunk_bytes <= kBulkStageBytes &&
             std::min(row_bytes, bulk_chunk_bytes) >= kBulkMinRowBytes;
    // Shorter rows of a one-outer-dim region whose destination rows (or, for a
    // copy, source rows) are contiguous: TMA tiles for the strided side.
    int64_t inner = 0;
    const int inn = t.n_outer - 1;  // the inner row dim
    if (allow_bulk && !k.bulk && vec == 16 && ns >= 1 && (t.n_outer == 1 || t.n_outer == 2) && row_bytes <= 4096 &&
        (t.dstr[inn] == t.cols || (ns == 1 && t.sstr[inn] == t.cols)))
        inner = tile_inner(t.cols, es);
    // a multiple of 128 bytes, so that the rounded slots of all sources fit too
    const int64_t budget = ns <= 1 ? kChunkBytes : kTileSumStageBytes / std::max<int64_t>(ns, 1) / 128 * 128;
    if (inner > 0 && budget >= row_bytes) {
        k.tile = t.dstr[inn] == t.cols ? 1 : 2;
        k.seg = t.cols;
        k.nseg = 1;
        k.rpc = (int32_t)std::min<int64_t>({(int64_t)kBlock, budget / row_bytes, t.ext[inn]});
        const int64_t nb = (t.ext[inn] + k.rpc - 1) / k.rpc;
        return (inn > 0 ? t.ext[0] : 1) * nb;
    }
    // Register path: a copy to several destinations writes each chunk several
    // times, so its chunks shrink to keep the bytes a block moves near 2 x 32 KB
    // (4 KB at least). A float32 copy of 8- or 4-byte vectors takes 64 KB
    // chunks whatever its destinations: long rows go row by row there, and
    // more rows a chunk spread the chunk's set-up over more bytes (measured:
    // 12 KB rows to two destinations 5.15 -> 5.79 TB/s).
    const int64_t chunk_bytes = k.bulk ? bulk_chunk_bytes
                                : (ns == 1 && es == 4 && vec < 16) ? 2 * kChunkBytes
                                : ns <= 1 ? std::max<int64_t>(4096, 2 * kChunkBytes / (int64_t)(1 + t.dst.size()))
                                          : kChunkBytes;
    if (row_bytes >= chunk_bytes) {
        const int64_t seg = std::min(t.cols, std::max<int64_t>(epv, (chunk_bytes / es) / epv * epv));
        k.seg = seg;
        k.nseg = (t.cols + seg - 1) / seg;
        k.rpc = 1;
    } else {
        k.seg = t.cols;
        k.nseg = 1;
        k.rpc = (int32_t)std::min<int64_t>({(int64_t)kBlock, std::max<int64_t>(1, chunk_bytes / std::max<int64_t>(row_bytes, 1)),
                                            t.rows});
    }
    return (t.rows + k.rpc - 1) / k.rpc * k.nseg;
}

// Shared staging a bulk or tile task's chunk needs (0 for the register path).
int64_t stage_bytes(const KTask& k, int es)
{
    if (k.tile) return (int64_t)std::max(1, k.n_src) * tile_slot(k.rpc, k.cols * es);
    if (!k.bulk) return 0;
    return (int64_t)k.n_src * (k.rpc == 1 ? k.seg * es : (int64_t)k.rpc * k.cols * es);
}

// Copies the used part of a full parameter block into a smaller form.
template <class PP>
const PP& shrink(const KParams& full, int nt, int np, PP* out)
{
    out->n_tasks = full.n_tasks;
    out->dtype = full.dtype;
    out->total_chunks = full.total_chunks;
    std::memcpy(out->tasks, full.tasks, sizeof(KTask) * (size_t)nt);
    std::memcpy(out->ptrs, full.ptrs, sizeof(void*) * (size_t)np);
    return *out;
}

template <class PP, bool SUM, int ES, int OP>
int launch_one(const PP& prm, int grid, int smem, cudaStream_t st)
{
    static std::atomic<bool> configured[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return fail(RTP_ECUDA, "reshard: no CUDA device");
    if (smem > 0 && !configured[dev].load(std::memory_order_acquire)) {
        if (cudaFuncSetAttribute(boxing_kernel<PP, SUM, ES, OP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kBulkDynSmem) != cudaSuccess)
            return fail(RTP_ECUDA, "reshard: cudaFuncSetAttribute failed");
        configured[dev].store(true, std::memory_order_release);
    }
    boxing_kernel<PP, SUM, ES, OP><<<grid, kBlock, smem, st>>>(prm);
    return RTP_OK;
}

template <class PP>
int launch_boxing(const PP& prm, int grid, int smem, cudaStream_t st, bool any_sum, int sum_op, int es)
{
    if (!any_sum) {
        if (es == 4) return launch_one<PP, false, 4, RED_SUM>(prm, grid, smem, st);
        return launch_one<PP, false, 2, RED_SUM>(prm, grid, smem, st);
    }
    if (es == 4) {
        if (sum_op == RED_MIN) return launch_one<PP, true, 4, RED_MIN>(prm, grid, smem, st);
        if (sum_op == RED_MAX) return launch_one<PP, true, 4, RED_MAX>(prm, grid, smem, st);
        return launch_one<PP, true, 4, RED_SUM>(prm, grid, smem, st);
    }
    if (sum_op == RED_MIN) return launch_one<PP, true, 2, RED_MIN>(prm, grid, smem, st);
    if (sum_op == RED_MAX) return launch_one<PP, true, 2, RED_MAX>(prm, grid, smem, st);
    return launch_one<PP, true, 2, RED_SUM>(prm, grid, smem, st);
}

template <class PP, int ES>
int launch_tile_copy(const PP& prm, int grid, int smem, cudaStream_t st)
{
    static std::atomic<bool> configured[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return fail(RTP_ECUDA, "reshard: no CUDA device");
    if (smem > 0 && !configured[dev].load(std::memory_order_acquire)) {
        if (cudaFuncSetAttribute(tile_copy_kernel<PP, ES>, cudaFuncAttributeMaxDynamicSharedMemorySize, kBulkDynSmem) !=
            cudaSuccess)
            return fail(RTP_ECUDA, "reshard: cudaFuncSetAttribute failed");
        configured[dev].store(true, std::memory_order_release);
    }
    tile_copy_kernel<PP, ES><<<grid, kTileBlock, smem, st>>>(prm);
    return RTP_OK;
}

// Fills a tile-form parameter block from the full one, encodes the tensor maps
// of the tile tasks' strided sides, and launches.
template <class PP>
int launch_tiles(const KParams& prm, int nt, int np, int es, PP* tp, int grid, int smem, cudaStream_t st, bool any_sum,
                 int sum_op)
{
    shrink(prm, nt, np, tp);
    int m = 0, rc;
    for (int k = 0; k < nt; ++k) {
        KTask& kt = tp->tasks[k];
        if (!kt.tile) continue;
        kt.map0 = m;
        const int n = kt.tile == 1 ? kt.n_src : kt.n_dst;
        const int base = kt.tile == 1 ? kt.ptr0 : kt.ptr0 + kt.n_src;
        const int64_t* str = kt.tile == 1 ? kt.sstr : kt.dstr;
        for (int j = 0; j < n; ++j)
            if ((rc = encode_tile_map(&tp->maps[m++], tp->ptrs[base + j], kt.n_outer, kt.ext, str, kt.cols, kt.rpc, es)))
                return rc;
    }
    // Every task a tile copy to one destination: the small-block kernel.
    // (Copies to several destinations, a broadcast's pieces, stay on
    // boxing_kernel: measured 1-1.5 % slower in the small blocks.)
    bool tile_copies = !any_sum;
    for (int k = 0; k < nt; ++k) tile_copies = tile_copies && tp->tasks[k].tile && tp->tasks[k].n_dst == 1;
    if (tile_copies)
        return es == 4 ? launch_tile_copy<PP, 4>(*tp, grid, smem, st) : launch_tile_copy<PP, 2>(*tp, grid, smem, st);
    return launch_boxing(*tp, grid, smem, st, any_sum, sum_op, es);
}

}  // namespace

void* tensor_map_encoder()
{
    static std::atomic<void*> fn{nullptr};
    void* f = fn.load(std::memory_order_acquire);
    if (!f) {
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn.store(f, std::memory_order_release);
    }
    return f;
}

int bulk_wait_selftest(unsigned long long limit_ns, uint32_t* out, void* stream)
{
    bulk_wait_selftest_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(limit_ns, out);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(RTP_ECUDA, "rtp_wait_selftest: launch failed: %s", cudaGetErrorString(e));
    return RTP_OK;
}

int classify_tasks(int dtype, const std::vector<PlanTask>& tasks, int32_t* counts)
{
    const int es = dtype == RTP_F32 ? 4 : 2;
    for (int f = 0; f < 4; ++f) counts[f] = 0;
    // buffers as cudaMalloc returns them: 256-byte aligned bases
    std::vector<const void*> fake(RTP_MAX_RANKS, reinterpret_cast<const void*>(uintptr_t(256)));
    size_t i = 0;
    while (i < tasks.size()) {
        KTask ks[kMaxTasks];
        int nt = 0, np = 0, n_maps = 0;
        for (; i < tasks.size() && nt < kMaxTasks; ++i) {
            const PlanTask& t = tasks[i];
            const int need = (int)(t.src.size() + t.dst.size());
            if (np + need > kMaxPtrs) break;
            fill_task(ks[nt], t, pick_vec(t, fake.data(), const_cast<void* const*>(fake.data()), es), es, true);
            if (ks[nt].tile) n_maps += ks[nt].tile == 1 ? ks[nt].n_src : ks[nt].n_dst;
            np += need;
            ++nt;
        }
        const bool tiles = n_maps > 0 && nt <= kTileTasks && np <= kTilePtrs && n_maps <= kTileMaps;
        for (int k = 0; k < nt; ++k) {
            if (ks[k].tile && tiles) ++counts[ks[k].n_outer == 2 ? 3 : 2];
            else if (ks[k].bulk) ++counts[1];
            else ++counts[0];
        }
    }
    return RTP_OK;
}

int take_boxing_error(void* stream, uint32_t* code)
{
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_box_error, sizeof v, 0, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemcpyToSymbolAsync(g_box_error, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return fail(RTP_ECUDA, "rtp_device_error: %s", cudaGetErrorString(cudaGetLastError()));
    *code = v;
    return RTP_OK;
}

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
                 void* stream, int* n_launches_out, int blocks_per_sm)
{
    const int es = dtype == RTP_F32 ? 4 : 2;
    for (const auto& t : tasks) {
        if (t.rows >= (int64_t)1 << 31) return fail(RTP_EUNSUPPORTED, "reshard: region with 2^31 or more rows");
        for (int k = 0; k < t.n_outer; ++k)
            if (t.ext[k] >= (int64_t)1 << 31) return fail(RTP_EUNSUPPORTED, "reshard: extent of 2^31 or more");
        if (t.src.size() + t.dst.size() > (size_t)kMaxPtrs) return fail(RTP_EUNSUPPORTED, "reshard: too many buffers");
    }
    static thread_local KParams prm;  // large: keep it off the stack
    const int max_grid = sm_count() * (blocks_per_sm < 1 ? 1 : blocks_per_sm > 4 ? 4 : blocks_per_sm);
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
            // beside another kernel the staging would keep the blocks off its SMs
            int64_t nc = fill_task(k, t, pick_vec(t, src, dst, es), es, blocks_per_sm >= 4);
            k.chunk_begin = chunks;
            k.ptr0 = np;
            for (const auto& r : t.src) prm.ptrs[np++] = static_cast<const char*>(src[r.rank]) + r.offset * es;
            for (const auto& r : t.dst) prm.ptrs[np++] = static_cast<char*>(dst[r.rank]) + r.offset * es;
            chunks += nc;
            ++nt;
        }
        prm.n_tasks = nt;
        prm.total_chunks = chunks;
        bool any_sum = false;
        int sum_op = RED_SUM;
        for (int k = 0; k < nt; ++k)
            if (prm.tasks[k].n_src > 1) {
                if (any_sum && prm.tasks[k].op != sum_op)
                    return fail(RTP_EUNSUPPORTED, "reshard: reductions of different kinds in one launch");
                any_sum = true;
                sum_op = prm.tasks[k].op;
            }
        if (chunks == 0) continue;
        // One block per chunk when the kernel has the GPU to itself: blocks then
        // start in chunk order, so the chunks in flight stay close in memory
        // (measured: 4% more bandwidth than a persistent grid on the resharding
        // sweep). Beside another kernel, a persistent grid of blocks_per_sm
        // blocks per SM limits how much of each SM the copy takes.
        const int64_t grid64 = blocks_per_sm >= 4 ? std::min<int64_t>(chunks, 0x7fffffff) : std::min<int64_t>(chunks, max_grid);
        const int grid = (int)grid64;
        cudaStream_t st = static_cast<cudaStream_t>(stream);
        // TMA-tile tasks need their tensor maps in the launch's parameters
        int n_maps = 0;
        for (int k = 0; k < nt; ++k)
            if (prm.tasks[k].tile) n_maps += prm.tasks[k].tile == 1 ? prm.tasks[k].n_src : prm.tasks[k].n_dst;
        const bool tiles = n_maps > 0 && nt <= kTileTasks && np <= kTilePtrs && n_maps <= kTileMaps;
        if (!tiles)
            for (int k = 0; k < nt; ++k) prm.tasks[k].tile = 0;  // their chunks also suit the register path
        int64_t smem = 0;
        for (int k = 0; k < nt; ++k) smem = std::max(smem, stage_bytes(prm.tasks[k], es));
        int st_ok;
        bool rank4 = false;
        for (int k = 0; k < nt; ++k) rank4 |= prm.tasks[k].tile && prm.tasks[k].n_outer == 2;
        if (tiles) {
            if (rank4) {
                static thread_local KParamsTile4 tp4;
                st_ok = launch_tiles(prm, nt, np, es, &tp4, grid, (int)smem, st, any_sum, sum_op);
            } else {
                static thread_local KParamsTile3 tp3;
                st_ok = launch_tiles(prm, nt, np, es, &tp3, grid, (int)smem, st, any_sum, sum_op);
            }
        } else if (nt <= kSmallTasks && np <= kSmallPtrs) {
            static thread_local KParamsSmall small;
            st_ok = launch_boxing(shrink(prm, nt, np, &small), grid, (int)smem, st, any_sum, sum_op, es);
        } else if (nt <= kMediumTasks && np <= kMediumPtrs) {
            static thread_local KParamsMedium medium;
            st_ok = launch_boxing(shrink(prm, nt, np, &medium), grid, (int)smem, st, any_sum, sum_op, es);
        } else {
            st_ok = launch_boxing(prm, grid, (int)smem, st, any_sum, sum_op, es);
        }
        if (st_ok) return st_ok;
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return fail(RTP_ECUDA, "boxing kernel launch failed: %s", cudaGetErrorString(e));
        ++launches;
    }
    if (n_launches_out) *n_launches_out = launches;
    return RTP_OK;
}

}  // namespace rtp
