// Megatron 1D tensor-parallel MLP on a virtual mesh of P ranks held in one GPU
// (ColossalAI "1D tensor parallelism" page, sections 2 and 2.1; GELU between
// the GEMMs from the Domino page, forward section).
//
//   column-parallel:  Y_i = GELU(X A_i)          X [M,K], A_i [K,F/P]
//   row-parallel:     Z   = sum_i Y_i B_i        Y_i [M,F/P], B_i [F/P,N]
//
// Both GEMMs run on one persistent, warp-specialised tcgen05 kernel in which a
// cluster of 2 CTAs (2 SMs) computes one 256x256 output tile per step:
//   warp 0     TMA producer, in each CTA: its 128 rows of the K-major operand
//              (X or Y_i, 128x64 per stage) and its 128 columns of the N-major
//              operand (A_i or B_i, two 64x64 boxes), 128-byte swizzled, into
//              a 6-stage ring of 32 KB stages;
//   warp 1     one thread of the leader CTA issues tcgen05.mma.cta_group::2
//              (M=256, N=256, K=16, bf16 in, float32 accumulate in TMEM), which
//              reads both CTAs' operands and writes each CTA's 128 rows to that
//              CTA's TMEM; 2 accumulators of 256 columns let the epilogue of one
//              tile overlap the next tile's K loop;
//   warps 2-5  epilogue, in each CTA: tcgen05.ld of its accumulator rows, GELU
//              and bf16 rounding (GEMM1) or float32 (GEMM2), staged 32 x 32 at
//              a time in swizzled shared memory and written by TMA tensor
//              stores clipped to the launch's output window.
// Consecutive GEMM launches overlap their set-up with the previous kernel's end
// (programmatic dependent launch); a kernel waits for its predecessor before
// touching global memory.
// Per SM the pair tile halves the operand bytes fetched from L2 and staged in
// shared memory per FLOP compared with a 128x256 single-SM tile. Tiles are
// walked in groups of 16 M-tiles so that the pairs running at one time share
// operand panels in L2.
//
// The row-parallel GEMM has two forms. Separate: each rank's Y_i B_i is a
// float32 partial, and a multi-source kernel sums the partials (the
// all-reduce of the pages), or, optionally, the epilogue that writes a
// partial tile also adds it to Z in rank order (one cluster takes every
// rank's tile of an output tile in turn; the same bits as the separate sum).
// Fused: the K loop of one output tile walks every rank's K range in turn, so
// the sum of ranks happens in the TMEM accumulator and no partial is ever
// written.
//
// Sequence parallelism (ColossalAI page, section 5.3: the column layer
// all-gathers its sequence-split input, the row layer reduce-scatters its
// output) is fused too: the column-parallel GEMM loads each 128-row block of X
// from the rank that holds it, and the rank-summing row-parallel GEMM writes
// each output row to the rank that owns it.
//
// The Domino schedule (Domino page, row split of X and column split of B)
// cuts X into row chunks (and B_i into column blocks): the reduction of
// chunk c runs on a second stream while the GEMMs of chunk c+1 run.
//
// Every mbarrier wait is bounded: after a few seconds without progress the
// waiting thread records an error code in a device word, raises a CTA-wide
// abort flag and every role leaves its loop; the CTA then frees its TMEM and
// exits. rtp_device_error() reads and clears that word.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstring>
#include <unordered_map>
#include <vector>

#include "rtp_internal.h"

namespace rtp {

namespace {

constexpr int BN = 256, BK = 64;
constexpr uint32_t B_SUB = 64 * BK * 2;  // one 64(N) x 64(K) box, 8 KB
// Warps: 0 TMA producer, 1 MMA issuer, then EPI_WARPS epilogue warps. An
// epilogue warp reaches the TMEM lane quarter (warp % 4); with 8 of them, two
// warps share each quarter and take half of the tile's columns each.
constexpr int EPI_WARPS = 4;
constexpr int THREADS = 64 + 32 * EPI_WARPS;
constexpr int EPI_CHUNKS = BN / 32 / (EPI_WARPS / 4);  // 32-column chunks per epilogue warp
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr int GROUP_M = 16;        // M tiles per raster block when K < 8192
constexpr int GROUP_M_LONG_K = 8;  // ... and when K >= 8192
// Reduction blocks per SM while a GEMM runs beside it: 2 is the most that stay
// resident next to a GEMM CTA (registers: 192 x 133 for the GEMM, 2 x 256 x 64
// for the reductions, of 64 K). Measured on the Llama-70B MLP, Domino with 2
// chunks: 2.40 ms with 2 per SM, 2.50 with 1, 2.69 with one per 2 SMs.
constexpr int kOverlapBlocksPerSm = 2;
constexpr int MAX_GROUPS = 8;
constexpr unsigned long long WAIT_LIMIT_NS = 4000000000ull;

enum : uint32_t { ERR_PRODUCER = 1, ERR_MMA_STAGE = 2, ERR_MMA_ACC = 3, ERR_EPILOGUE = 4, ERR_SELFTEST = 5 };
enum { EPI_GELU_BF16 = 0, EPI_F32 = 1, EPI_DGELU_BF16 = 2 };
// Kernel configuration (a compile-time template parameter):
//   CFG_SP_A    rows of the A operand come from per-shard maps (sequence parallel)
//   CFG_SP_OUT  output rows go to per-shard buffers (sequence parallel)
//   CFG_A_MN    A is M-major in memory (a transposed operand: X^T, Y^T)
//   CFG_B_K     B is K-major in memory (a transposed operand: A_i^T, B_i^T)
//   bits 4-5    the epilogue (EPI_*)
enum : int { CFG_SP_A = 1, CFG_SP_OUT = 2, CFG_A_MN = 4, CFG_B_K = 8, CFG_EPI_SHIFT = 4 };
enum : int { RANKS_OUTER = 0, RANKS_IN_N = 1 };


struct GemmArgs {
    CUtensorMap ta[MAX_GROUPS];  // A operand of each group ([M rows, K] K-major, or [K rows, M] M-major)
    CUtensorMap tb[MAX_GROUPS];  // B operand of each group ([K rows, N] N-major, or [N rows, K] K-major)
    // Output of each group (to[0] when fused; of each row shard with
    // out_rows_per_ptr > 0), as a tensor map of the launch's window: rows
    // [0, m_end) and columns [0, n_end) of the buffer, box 32 x 32. TMA stores
    // write only inside the map, so the window's edges clip every store.
    CUtensorMap to[MAX_GROUPS];
    CUtensorMap to2[MAX_GROUPS]; // GELU epilogue with store_h: the pre-activation's outputs
    const void* aux[MAX_GROUPS]; // GELU-gradient epilogue: the pre-activation H read at each output
    int32_t store_h;             // GELU epilogue: also store the bf16 pre-activation (to2)
    int64_t ldo;                 // output row stride, elements
    int32_t groups, fused, epi;
    int32_t m_tiles, n_tiles, kb_per_group;
    int32_t m0, n0;              // window of the problem (Domino chunk / column block)
    int32_t m_end, n_end;        // exclusive bounds of the output window
    int32_t total_tiles;
    // Sequence parallelism (rows sharded over the ranks): when > 0, the
    // K-major operand of row r comes from map ta[r / a_rows_per_map] at row
    // r % a_rows_per_map (an all-gather fused into the loads), and/or output
    // row r goes to out[r / out_rows_per_ptr] at row r % out_rows_per_ptr (a
    // reduce-scatter fused into the epilogue of the rank-summing GEMM).
    int32_t a_rows_per_map, a_maps;
    int32_t out_rows_per_ptr, out_ptrs;
    int32_t cfg;                 // kernel configuration (CFG_* operand bits), chosen by the host
    // Tile order of a non-fused launch over several groups (ranks):
    //   RANKS_OUTER  group by group;
    //   RANKS_IN_N   the groups' N tiles form one N range. For groups with the
    //                same A operand (X in X A_i): each block of group_m A row
    //                tiles then stays in L2 while every group's B columns stream
    //                past it, instead of being fetched again for every group.
    int32_t rank_fold;
    // M tiles per raster block (set at launch from the K extent): the tiles in
    // flight at once cover group_m rows of tiles and about 76 / group_m
    // columns of tiles.
    int32_t group_m;
    // Rank sum in the epilogue (mode 0 of the row-parallel GEMMs): the
    // groups' tiles of one output tile go to one cluster, rank after rank,
    // and its epilogue, besides writing rank g's partial, adds it to sum_dst
    // (row stride ldo): sum_dst = ((0 + p_0) + p_1) + ... in float32, the same
    // bits as summing the finished partials in rank order.
    int32_t sum_into;
    float* sum_dst;
};

__device__ unsigned int g_tp_error;

// ---- PTX wrappers ------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Slow path of wait_bar, kept out of line.
__device__ __noinline__ bool wait_bar_slow(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag, uint32_t code,
                                           unsigned long long limit_ns)
{
    const uint64_t t0 = global_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 0) {
            if (*abort_flag) return false;
            if (global_ns() - t0 > limit_ns) {
                *abort_flag = 1;
                atomicCAS(&g_tp_error, 0u, code);
                return false;
            }
        }
    }
}

// Bounded wait. False: this wait gave up, or another role already did.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag, uint32_t code,
                                         unsigned long long limit_ns = WAIT_LIMIT_NS)
{
    if (mbar_try_wait(bar, parity)) return true;
    return wait_bar_slow(bar, parity, abort_flag, code, limit_ns);
}

// Self-test of the bounded wait: two threads wait on an mbarrier that nothing
// completes. The first gives up after limit_ns, records ERR_SELFTEST and raises
// the abort flag; the second leaves on the flag. out[w] = 1 if waiter w gave up.
// The mbarrier is never armed or awaited again, so nothing is left in flight.
__global__ void wait_selftest_kernel(unsigned long long limit_ns, uint32_t* out)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t abort_word;
    volatile uint32_t* abort_flag = &abort_word;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) {
        // waiter 1's own limit is 4x longer: it should leave on waiter 0's abort
        // flag, so the kernel lasts about limit_ns (4 limit_ns at most)
        const bool ok = wait_bar(smem_u32(&bar), 0, abort_flag, ERR_SELFTEST, w == 0 ? limit_ns : 4 * limit_ns);
        out[w] = ok ? 0u : 1u;
    }
}

// Bounded wait used only while tearing down after an abort: it ignores the
// abort flag so that copies and MMAs already in flight can land.
__device__ __noinline__ void drain_wait(uint32_t bar, uint32_t parity)
{
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > 200000000ull) break;
}

__device__ __forceinline__ void prefetch_map(const CUtensorMap* map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor (tcgen05): start >> 4 (bits 0-13), leading
// byte offset >> 4 (16-29), stride byte offset >> 4 (32-45), version 1 (46-48),
// base offset 0, swizzle mode 2 = 128-byte swizzle (61-63).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo)
{
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

__device__ __forceinline__ void tmem_ld_32cols(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// Waits for this thread's outstanding tcgen05.ld. The registers of the load
// whose results are used next pass through the asm as read-write operands, so
// the compiler cannot move their uses above the wait.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                   "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                   "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

// Tile index -> (group, M tile, N tile). Within an (M range, N range) the
// tiles go in blocks of group_m M tiles, N tile after N tile within a block,
// so the tiles in flight at once share their A rows and B columns in L2. The
// group is the outermost index, or part of the N range (rank_fold). Both maps
// are bijections of [0, groups * m_tiles * n_tiles).
__device__ __forceinline__ void tile_coords(const GemmArgs& a, int tile, int& g, int& mt, int& nt)
{
    const bool in_n = !a.fused && !a.sum_into && a.rank_fold == RANKS_IN_N;
    const int per_group = a.fused || in_n || a.sum_into ? 0 : a.m_tiles * a.n_tiles;
    g = per_group ? tile / per_group : 0;
    int r = tile - g * per_group;
    if (a.sum_into) {  // rank innermost: tile = output tile * groups + rank
        g = tile % a.groups;
        r = tile / a.groups;
    }
    const int ntiles = in_n ? a.groups * a.n_tiles : a.n_tiles;
    const int span = a.group_m * ntiles;
    const int first_m = (r / span) * a.group_m;
    const int rows = min(a.m_tiles - first_m, a.group_m);
    const int w = r % span;
    mt = first_m + w % rows;
    nt = w / rows;
    if (in_n) {
        g = nt / a.n_tiles;
        nt -= g * a.n_tiles;
    }
}

// The k-th tile of cluster `pair` of `npairs`, or -1 when it has no more.
// Clusters take tiles in turn; with the rank sum in the epilogue they take
// whole groups (every rank's tile of one output tile, rank after rank), so one
// cluster adds up each output tile's partials in rank order.
__device__ __forceinline__ int nth_tile(const GemmArgs& a, int pair, int npairs, int k)
{
    if (!a.sum_into) {
        const int t = pair + k * npairs;
        return t < a.total_tiles ? t : -1;
    }
    const int grp = pair + (k / a.groups) * npairs;
    return grp < a.total_tiles / a.groups ? grp * a.groups + k % a.groups : -1;
}

__device__ __forceinline__ float gelu(float x) { return 0.5f * x * (1.0f + erff(x * 0.70710678118654752440f)); }

// d GELU(h) / dh = Phi(h) + h phi(h) for the exact erf form.
__device__ __forceinline__ float gelu_grad(float h)
{
    const float cdf = 0.5f * (1.0f + erff(h * 0.70710678118654752440f));
    const float pdf = 0.39894228040143267794f * expf(-0.5f * h * h);
    return cdf + h * pdf;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi)
{
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
}

// ---- the kernel ----------------------------------------------------------------------
//
// CTA r of the pair holds rows [128r, 128r+128) of the K-major operand and
// columns [128r, 128r+128) of the N-major operand. Barriers:
//   full[s]      in the leader: expects both CTAs' TMA bytes (one arrival, the
//                leader's expect_tx); each CTA's loads signal it (cta_group::2)
//   empty[s]     in both CTAs: one arrival from the leader's commit (multicast)
//   acc_full[x]  in both CTAs: the leader's commit after a tile's last MMA
//   acc_empty[x] in the leader: 8 arrivals, the 4 epilogue warps of each CTA

constexpr int BM2 = 256;
constexpr int STAGES2 = 6;
constexpr uint32_t A2_BYTES = 128 * BK * 2;           // 16 KB
constexpr uint32_t B2_BYTES = 128 * BK * 2;           // 16 KB: 2 boxes of 64(N) x 64(K)
constexpr uint32_t STAGE2_BYTES = A2_BYTES + B2_BYTES;  // 32 KB
// Epilogue staging: per epilogue warp two 4 KB buffers, each one 32 x 32 output
// chunk (float32, or bf16 Y and H side by side), swizzled as its TMA store
// reads it.
constexpr uint32_t EPI_STAGE_BYTES = 4096;
constexpr uint32_t EPI_WARP_BYTES = 2 * EPI_STAGE_BYTES;
constexpr size_t SMEM2_BYTES =
    STAGES2 * STAGE2_BYTES + 1024 + EPI_WARPS * EPI_WARP_BYTES + 1024;  // ring, barriers, staging, alignment
static_assert(SMEM2_BYTES <= 232448, "at most 227 KB of shared memory per CTA");
// Instruction descriptor of tcgen05.mma kind::f16: D float32 (bits 4-5 = 1),
// A and B bf16 (bits 7-9 = 1, 10-12 = 1), bit 15 = A M-major, bit 16 = B
// N-major, N >> 3 in bits 17-22, M >> 4 in bits 24-28 (M = 256 for the pair).
__host__ __device__ constexpr uint32_t idesc2(bool a_mn, bool b_k)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_k ? 0u : 1u) << 16) |
           ((uint32_t)(256 >> 3) << 17) | ((uint32_t)(BM2 >> 4) << 24);
}

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_id()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t num_clusters()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}
// Address in the shared::cluster window of the same variable in CTA `rank`.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster, int x, int y)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y)
        : "memory");
}
// TMA tile store shared -> global (bulk async group of the issuing thread).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Until at most one of this thread's bulk groups still reads shared memory.
__device__ __forceinline__ void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
// Until every bulk group of this thread has completed (its writes performed).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Makes this thread's shared-memory writes visible to the TMA (async proxy).
__device__ __forceinline__ void fence_async_shared() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t x, uint32_t y, uint32_t z, uint32_t w)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(x), "r"(y), "r"(z), "r"(w) : "memory");
}

__device__ __forceinline__ void mma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_commit_pair(uint32_t bar)
{
    const uint16_t both = 3;
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
                 "h"(both)
                 : "memory");
}
__device__ __forceinline__ void mma_commit_pair_local(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// CFG (CFG_* bits) is compile-time, so each configuration's loops carry no
// work for the others.
template <int CFG>
__global__ void __launch_bounds__(THREADS, 1) tp_gemm_kernel(const __grid_constant__ GemmArgs a)
{
    constexpr bool SP_A = (CFG & CFG_SP_A) != 0, SP_OUT = (CFG & CFG_SP_OUT) != 0;
    constexpr bool A_MN = (CFG & CFG_A_MN) != 0, B_K = (CFG & CFG_B_K) != 0;
    constexpr int EPI = (CFG >> CFG_EPI_SHIFT) & 3;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES2 * STAGE2_BYTES);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES2 + 5);
    volatile uint32_t* abort_flag = tmem_slot + 1;
    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * (uint32_t)s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (uint32_t)(STAGES2 + s); };
    auto acc_full = [&](int x) { return bar0 + 8u * (uint32_t)(2 * STAGES2 + x); };
    auto acc_empty = [&](int x) { return bar0 + 8u * (uint32_t)(2 * STAGES2 + 2 + x); };
    const uint32_t drain_bar = bar0 + 8u * (uint32_t)(2 * STAGES2 + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t cta = cluster_rank();
    const int pair = (int)cluster_id(), npairs = (int)num_clusters();
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES2; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(acc_full(x), 1);
            mbar_init(acc_empty(x), 2 * EPI_WARPS);  // every epilogue warp of both CTAs
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        for (int g = 0; g < a.groups; ++g) {
            prefetch_map(&a.ta[g]);
            prefetch_map(&a.tb[g]);
        }
    }
    if (warp == 2 && lane == 0) {
        const int nout = SP_OUT ? a.out_ptrs : (a.fused ? 1 : a.groups);
        for (int g = 0; g < nout; ++g) {
            prefetch_map(&a.to[g]);
            if (EPI == EPI_GELU_BF16 && a.store_h) prefetch_map(&a.to2[g]);
        }
    }
    if (warp == 1) {
        // one warp in each CTA of the pair allocates collectively
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the peer's barriers are initialised before any remote use
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // Launched as a programmatic dependent of the previous kernel in the
    // stream, this CTA may have started (and run the set-up above) while that
    // kernel was finishing: wait for it to complete, and its writes to be
    // visible, before any global memory access. Without such a launch this
    // returns at once.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int kbs = a.fused ? a.groups * a.kb_per_group : a.kb_per_group;

    if (warp == 0) {
        // ---------------- TMA producer (one lane per CTA) ----------------
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0, issued_parity = 0;
            bool ok = true;
            const uint32_t smem0 = smem_u32(smem);
            const uint32_t leader_full0 = map_to_rank(full_bar(0), 0);  // barriers are 8 bytes apart
            for (int k = 0, tile; ok && (tile = nth_tile(a, pair, npairs, k)) >= 0; ++k) {
                int g, mt, nt;
                tile_coords(a, tile, g, mt, nt);
                const int row = a.m0 + mt * BM2 + (int)cta * 128, col = a.n0 + nt * BN + (int)cta * 128;
                const CUtensorMap* amap_sp = nullptr;
                int arow = row;
                if constexpr (SP_A) {
                    // the 128-row block lies in one shard (shards are multiples of 128
                    // rows); rows past the last shard read as zeros
                    const int sh = min(row / a.a_rows_per_map, a.a_maps - 1);
                    amap_sp = &a.ta[sh];
                    arow = row - sh * a.a_rows_per_map;
                }
                int gg = a.fused ? 0 : g, kk = 0;
                for (int kb = 0; kb < kbs; ++kb) {
                    if (!wait_bar(empty_bar(stage), phase ^ 1u, abort_flag, ERR_PRODUCER)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = smem0 + (uint32_t)stage * STAGE2_BYTES;
                    const uint32_t sb = sa + A2_BYTES;
                    const uint32_t fb = leader_full0 + 8u * (uint32_t)stage;
                    if (cta == 0) mbar_expect_tx(full_bar(stage), 2 * STAGE2_BYTES);
                    const CUtensorMap* am = SP_A ? amap_sp : &a.ta[gg];
                    if constexpr (A_MN) {  // two 64(M) x 64(K) boxes
                        tma_load_2d_pair(sa, am, fb, arow, kk * BK);
                        tma_load_2d_pair(sa + B_SUB, am, fb, arow + 64, kk * BK);
                    } else {  // one 128(M) x 64(K) box
                        tma_load_2d_pair(sa, am, fb, kk * BK, arow);
                    }
                    if constexpr (B_K) {  // one 128(N) x 64(K) box
                        tma_load_2d_pair(sb, &a.tb[gg], fb, kk * BK, col);
                    } else {  // two 64(N) x 64(K) boxes
                        tma_load_2d_pair(sb, &a.tb[gg], fb, col, kk * BK);
                        tma_load_2d_pair(sb + B_SUB, &a.tb[gg], fb, col + 64, kk * BK);
                    }
                    issued |= 1u << stage;
                    issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    if (++kk == a.kb_per_group) {  // next rank's K range (fused reduction)
                        kk = 0;
                        ++gg;
                    }
                    if (++stage == STAGES2) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                if (cta == 0) {
                    for (int s = 0; s < STAGES2; ++s)
                        if ((issued >> s) & 1u) drain_wait(full_bar(s), (issued_parity >> s) & 1u);
                } else {
                    // the follower cannot wait on the leader's barrier: give its
                    // last loads (microseconds) time to land
                    const uint64_t t0 = global_ns();
                    while (global_ns() - t0 < 2000000ull) {
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- MMA issuer (one lane of the leader) ----------------
        if (lane == 0 && cta == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            // K-major operand: 32-byte steps (16 bf16) inside the 128-byte swizzle
            // row, 8-row groups 1024 bytes apart. M/N-major operand: 16 K-rows = 2
            // groups of 8 rows of 128 bytes (2048-byte steps); its two 64-wide boxes
            // are B_SUB bytes apart.
            constexpr uint32_t a_step = A_MN ? 2048u : 32u, b_step = B_K ? 32u : 2048u;
            constexpr uint32_t idesc = idesc2(A_MN, B_K);
            const uint64_t desc_a0 = smem_desc(smem_u32(smem), A_MN ? B_SUB : 16u, 1024u);
            const uint64_t desc_b0 = smem_desc(smem_u32(smem) + A2_BYTES, B_K ? 16u : B_SUB, 1024u);
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int k = 0, tile; ok && (tile = nth_tile(a, pair, npairs, k)) >= 0; ++k) {
                if (!wait_bar(acc_empty(acc), acc_phase ^ 1u, abort_flag, ERR_MMA_ACC)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int kb = 0; kb < kbs; ++kb) {
                    if (!wait_bar(full_bar(stage), phase, abort_flag, ERR_MMA_STAGE)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // descriptors are affine in the start address (bits 0-13 hold addr >> 4)
                    const uint64_t off = (uint64_t)((uint32_t)stage * STAGE2_BYTES >> 4);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k) {
                        const uint64_t da = desc_a0 + off + (uint64_t)(a_step * k >> 4);
                        const uint64_t db = desc_b0 + off + (uint64_t)(b_step * k >> 4);
                        mma_bf16_pair(d_tmem, da, db, idesc, (kb > 0 || k > 0) ? 1u : 0u);
                    }
                    mma_commit_pair(empty_bar(stage));
                    if (++stage == STAGES2) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit_pair(acc_full(acc));
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            if (!ok || *abort_flag) {
                mma_commit_pair_local(drain_bar);
                drain_wait(drain_bar, 0);
            }
        }
        __syncwarp();
    } else {
        // ---------------- epilogue (both CTAs) ----------------
        const uint32_t stage_epi = smem_u32(smem) + STAGES2 * STAGE2_BYTES + 1024u + (uint32_t)(warp - 2) * EPI_WARP_BYTES;
        const int quarter = warp & 3;
        const int c_begin = ((warp - 2) >> 2) * EPI_CHUNKS;
        int acc = 0;
        uint32_t acc_phase = 0;
        // TMA stores this warp has issued (warp-uniform). The two staging
        // buffers alternate by store, not by chunk: a tile cut by the window's
        // column edge stores fewer chunks, and by chunk parity the next tile's
        // first chunk could reuse the buffer of the store issued just before.
        uint32_t stores = 0;
        for (int k = 0, tile; (tile = nth_tile(a, pair, npairs, k)) >= 0; ++k) {
            int g, mt, nt;
            tile_coords(a, tile, g, mt, nt);
            int ok = 1;
            if (lane == 0) ok = wait_bar(acc_full(acc), acc_phase, abort_flag, ERR_EPILOGUE) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after();
            // this warp's 32 rows: lane l holds row row0 + l of the accumulator
            const int64_t row0 = a.m0 + (int64_t)mt * BM2 + cta * 128 + quarter * 32;
            const int64_t row = row0 + lane;
            const int64_t col = a.n0 + (int64_t)nt * BN;
            const bool row_ok = row < a.m_end;
            int om = g;  // output map
            int64_t orow0 = row0;
            if constexpr (SP_OUT) {  // the warp's rows lie in one shard (shards are multiples of 128 rows)
                om = min((int)(row0 / a.out_rows_per_ptr), a.out_ptrs - 1);
                orow0 = row0 - (int64_t)om * a.out_rows_per_ptr;
            }
            const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
            const __nv_bfloat16* hrow = nullptr;
            if constexpr (EPI == EPI_DGELU_BF16) hrow = static_cast<const __nv_bfloat16*>(a.aux[g]) + row * a.ldo;
            // H of chunk c (GELU-gradient epilogue only)
            auto load_h = [&](int c, uint4 (&h)[4]) {
                if constexpr (EPI == EPI_DGELU_BF16) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int64_t cq = col + 32 * c + 8 * q;
                        h[q] = (row_ok && cq < a.n_end) ? __ldg(reinterpret_cast<const uint4*>(hrow + cq))
                                                         : make_uint4(0u, 0u, 0u, 0u);
                    }
                }
            };
            // Chunk c (32 columns of the warp's 32 rows): each lane writes its row
            // to a staging buffer in the TMA's swizzled layout (16-byte unit u of
            // row r at unit u ^ (r / 2 % 4) of a 64-byte bf16 row, u ^ (r % 8) of a
            // 128-byte float32 row: the 8 lanes of each store phase hit distinct
            // banks), then one lane stores the 32 x 32 tile. The map's window
            // clips rows past m_end and columns past n_end.
            auto emit = [&](int c, const uint32_t (&r)[32], const uint4 (&h)[4]) {
                const int64_t c0 = col + 32 * c;
                if (c0 >= a.n_end || row0 >= a.m_end) return;  // warp-uniform: nothing of the window here
                const uint32_t buf = stage_epi + (stores & 1u) * EPI_STAGE_BYTES;
                if (lane == 0) bulk_wait_read_1();  // the store two stores back has read this buffer
                __syncwarp();
                if constexpr (EPI == EPI_F32) {
                    const uint32_t rb = buf + (uint32_t)lane * 128u;
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        st_shared_v4(rb + 16u * (uint32_t)(q ^ (lane & 7)), r[4 * q + 0], r[4 * q + 1], r[4 * q + 2],
                                     r[4 * q + 3]);
                } else {
                    const uint32_t rb = buf + (uint32_t)lane * 64u;
                    const int sw = (lane >> 1) & 3;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint32_t w[4];
                        if constexpr (EPI == EPI_DGELU_BF16) {
                            // dH = dY * GELU'(H): the accumulator is dY, H was read at the same place
                            w[0] = pack_bf16(__uint_as_float(r[8 * q + 0]) * gelu_grad(bf16_lo(h[q].x)),
                                             __uint_as_float(r[8 * q + 1]) * gelu_grad(bf16_hi(h[q].x)));
                            w[1] = pack_bf16(__uint_as_float(r[8 * q + 2]) * gelu_grad(bf16_lo(h[q].y)),
                                             __uint_as_float(r[8 * q + 3]) * gelu_grad(bf16_hi(h[q].y)));
                            w[2] = pack_bf16(__uint_as_float(r[8 * q + 4]) * gelu_grad(bf16_lo(h[q].z)),
                                             __uint_as_float(r[8 * q + 5]) * gelu_grad(bf16_hi(h[q].z)));
                            w[3] = pack_bf16(__uint_as_float(r[8 * q + 6]) * gelu_grad(bf16_lo(h[q].w)),
                                             __uint_as_float(r[8 * q + 7]) * gelu_grad(bf16_hi(h[q].w)));
                        } else {
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                w[e] = pack_bf16(gelu(__uint_as_float(r[8 * q + 2 * e])),
                                                 gelu(__uint_as_float(r[8 * q + 2 * e + 1])));
                        }
                        st_shared_v4(rb + 16u * (uint32_t)(q ^ sw), w[0], w[1], w[2], w[3]);
                        if (EPI == EPI_GELU_BF16 && a.store_h) {  // the pre-activation, for the backward pass
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                w[e] = pack_bf16(__uint_as_float(r[8 * q + 2 * e]), __uint_as_float(r[8 * q + 2 * e + 1]));
                            st_shared_v4(rb + 2048u + 16u * (uint32_t)(q ^ sw), w[0], w[1], w[2], w[3]);
                        }
                    }
                }
                fence_async_shared();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(&a.to[om], buf, (int)c0, (int)orow0);
                    if (EPI == EPI_GELU_BF16 && a.store_h) tma_store_2d(&a.to2[om], buf + 2048u, (int)c0, (int)orow0);
                    bulk_commit();
                }
                ++stores;
                if constexpr (EPI == EPI_F32) {
                    if (a.sum_into) {
                        // sum_dst[rows, c0 + lane] += the staged chunk's column `lane`, rank g after
                        // rank g - 1 (the same lane of the same warp added those: program order);
                        // rank 0 starts from +0. Each access of the warp is one 128-byte row.
                        const bool col_in = c0 + lane < a.n_end;
                        float* zc = a.sum_dst + row0 * a.ldo + c0 + lane;
                        const uint32_t sbase = buf + 4u * (uint32_t)(lane & 3);
                        float prev[32];
#pragma unroll
                        for (int rr = 0; rr < 32; ++rr)
                            prev[rr] = (g > 0 && col_in && row0 + rr < a.m_end) ? __ldcg(zc + rr * a.ldo) : 0.0f;
#pragma unroll
                        for (int rr = 0; rr < 32; ++rr) {
                            float v;
                            asm volatile("ld.shared.f32 %0, [%1];"
                                         : "=f"(v)
                                         : "r"(sbase + (uint32_t)rr * 128u + 16u * (uint32_t)((lane >> 2) ^ (rr & 7))));
                            if (col_in && row0 + rr < a.m_end) __stcg(zc + rr * a.ldo, prev[rr] + v);
                        }
                    }
                }
            };
            // the TMEM load (and H load) of the next chunk is in flight while a
            // chunk is computed and stored (the loads are warp-wide: all lanes)
            static_assert(EPI_CHUNKS % 2 == 0, "chunks are processed in pairs");
            const int c_end = c_begin + EPI_CHUNKS;
            uint32_t ra[32], rb[32];
            uint4 ha[4], hb[4];
            load_h(c_begin, ha);
            tmem_ld_32cols(taddr + 32u * c_begin, ra);
            tmem_ld_wait(ra);
            for (int c = c_begin; c < c_end; c += 2) {
                tmem_ld_32cols(taddr + 32u * (c + 1), rb);
                load_h(c + 1, hb);
                emit(c, ra, ha);
                tmem_ld_wait(rb);
                if (c + 2 < c_end) {
                    tmem_ld_32cols(taddr + 32u * (c + 2), ra);
                    load_h(c + 2, ha);
                }
                emit(c + 1, rb, hb);
                if (c + 2 < c_end) tmem_ld_wait(ra);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(map_to_rank(acc_empty(acc), 0));
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        if (lane == 0) bulk_wait_all();  // every output tile written before the CTA leaves
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    // This CTA's work is done: the next kernel of the stream may be scheduled
    // once every CTA of this grid has come here (or exited). Every CTA of this
    // grid is then resident or done, so the next kernel's CTAs only take SMs
    // this grid no longer needs.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    cluster_sync();  // no CTA leaves while its peer may still signal or read it
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS) : "memory");
}

// ---- host side --------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encoder());
}

// 2D bf16 tensor map over a row-major [rows, cols] matrix, box [box_rows, 64],
// 128-byte swizzle (64 bf16 per box row).
int make_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int box_rows)
{
    auto fn = encode_fn();
    if (!fn) return fail(RTP_ECUDA, "tp_mlp: cuTensorMapEncodeTiled is unavailable");
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(cols * 2)};
    cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(RTP_ECUDA, "tp_mlp: cuTensorMapEncodeTiled failed (%d)", (int)r);
    return RTP_OK;
}

// Everything an output map is encoded from.
struct OutKey {
    uintptr_t ptr;
    int64_t rows, cols, ld;
    bool f32;
    bool operator==(const OutKey& o) const
    {
        return ptr == o.ptr && rows == o.rows && cols == o.cols && ld == o.ld && f32 == o.f32;
    }
};
struct OutKeyHash {
    size_t operator()(const OutKey& k) const
    {
        uint64_t h = k.ptr * 0x9E3779B97F4A7C15ull;
        for (uint64_t v : {(uint64_t)k.rows, (uint64_t)k.cols, (uint64_t)k.ld, (uint64_t)k.f32}) h = (h ^ v) * 0x100000001B3ull;
        return (size_t)h;
    }
};

// Tensor map of an output window: rows [0, rows) and columns [0, cols) of a
// row-major buffer with a row stride of ld elements, box 32 x 32 (one
// epilogue warp's chunk), swizzled like the staging buffer: 64-byte swizzle
// for bf16 (64-byte box rows), 128-byte for float32. Repeated calls with the
// same buffers reuse their maps (cached per thread).
int make_out_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int64_t ld, bool f32)
{
    static thread_local std::unordered_map<OutKey, CUtensorMap, OutKeyHash> cache;
    const OutKey key{reinterpret_cast<uintptr_t>(ptr), rows, cols, ld, f32};
    auto it = cache.find(key);
    if (it != cache.end()) {
        *m = it->second;
        return RTP_OK;
    }
    auto fn = encode_fn();
    if (!fn) return fail(RTP_ECUDA, "tp_mlp: cuTensorMapEncodeTiled is unavailable");
    const int es = f32 ? 4 : 2;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(ld * es)};
    cuuint32_t box[2] = {32u, 32u};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr),
                    dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    f32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(RTP_ECUDA, "tp_mlp: cuTensorMapEncodeTiled (output) failed (%d)", (int)r);
    if (cache.size() >= 4096) cache.clear();
    cache.emplace(key, *m);
    return RTP_OK;
}

template <int CFG>
int launch_gemm_t(GemmArgs& args, cudaStream_t stream)
{
    // per device: resident 2-SM clusters (0 = not yet queried); racing first
    // calls compute the same value
    static std::atomic<int> max_clusters[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return fail(RTP_ECUDA, "tp_mlp: no CUDA device");
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // Programmatic dependent launch: the kernel may be set up while the
    // previous kernel of the stream finishes; it waits for that kernel's
    // completion (griddepcontrol.wait) before touching global memory.
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = SMEM2_BYTES;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int nclusters = max_clusters[dev].load(std::memory_order_acquire);
    if (!nclusters) {
        cudaError_t e = cudaFuncSetAttribute(tp_gemm_kernel<CFG>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM2_BYTES);
        if (e != cudaSuccess) return fail(RTP_ECUDA, "tp_mlp: cudaFuncSetAttribute: %s", cudaGetErrorString(e));
        cfg.gridDim = dim3(2 * 64);
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, tp_gemm_kernel<CFG>, &cfg);
        if (e != cudaSuccess || n <= 0) return fail(RTP_ECUDA, "tp_mlp: cudaOccupancyMaxActiveClusters: %s", cudaGetErrorString(e));
        max_clusters[dev].store(n, std::memory_order_release);
        nclusters = n;
    }
    args.total_tiles = (args.fused ? 1 : args.groups) * args.m_tiles * args.n_tiles;
    // With a short K a block of group_m A row tiles stays in L2 while the B
    // columns stream past it, so tall blocks pay. With a long K no operand
    // panel survives in L2 from one wave of tiles to the next, and each wave
    // reads every row and column panel it covers: near-square waves (8 x 9.5
    // tiles instead of 16 x 4.75) read the fewest.
    const int64_t k_extent = (int64_t)(args.fused ? args.groups : 1) * args.kb_per_group * BK;
    args.group_m = k_extent >= 8192 ? GROUP_M_LONG_K : GROUP_M;
    // clusters take tiles (or, with the rank sum in the epilogue, whole groups
    // of every rank's tile of one output tile) in turn
    const int units = args.sum_into ? args.total_tiles / args.groups : args.total_tiles;
    const int clusters = units < nclusters ? units : nclusters;
    if (clusters <= 0) return RTP_OK;
    cfg.gridDim = dim3(2 * clusters);
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelEx(&cfg, tp_gemm_kernel<CFG>, args);
    if (e != cudaSuccess) return fail(RTP_ECUDA, "tp_mlp: GEMM launch failed: %s", cudaGetErrorString(e));
    return RTP_OK;
}

int launch_gemm(GemmArgs& args, cudaStream_t stream)
{
    constexpr int GELU = EPI_GELU_BF16 << CFG_EPI_SHIFT, F32 = EPI_F32 << CFG_EPI_SHIFT,
                  DGELU = EPI_DGELU_BF16 << CFG_EPI_SHIFT;
    switch (args.cfg | (args.epi << CFG_EPI_SHIFT)) {
    case GELU: return launch_gemm_t<GELU>(args, stream);
    case F32: return launch_gemm_t<F32>(args, stream);
    case CFG_SP_A | GELU: return launch_gemm_t<CFG_SP_A | GELU>(args, stream);
    case CFG_SP_OUT | F32: return launch_gemm_t<CFG_SP_OUT | F32>(args, stream);
    case CFG_A_MN | F32: return launch_gemm_t<CFG_A_MN | F32>(args, stream);
    case CFG_B_K | DGELU: return launch_gemm_t<CFG_B_K | DGELU>(args, stream);
    case CFG_B_K | F32: return launch_gemm_t<CFG_B_K | F32>(args, stream);
    default:
        return fail(RTP_EUNSUPPORTED, "tp_mlp: no GEMM kernel for configuration %d, epilogue %d", args.cfg, args.epi);
    }
}

struct Events {
    cudaEvent_t fwd = nullptr, back = nullptr;
};

// One pair per host thread and device: a call records an event on its own s0
// and makes its own s1 wait on it, so two threads calling at once (on their
// own streams) must not share the event, or one would wait on the other's
// record. The events live until the process exits.
int events(Events** out)
{
    static thread_local Events ev[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return fail(RTP_ECUDA, "tp_mlp: no CUDA device");
    Events& e = ev[dev];
    if (!e.fwd) {
        if (cudaEventCreateWithFlags(&e.fwd, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&e.back, cudaEventDisableTiming) != cudaSuccess)
            return fail(RTP_ECUDA, "tp_mlp: cudaEventCreate failed");
    }
    *out = &e;
    return RTP_OK;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Where the row-parallel GEMMs of mode 0 sum their partials, per host thread
// (rtp_tp_mlp_overlap): 0 (the default) in kernels of their own, 1 in the
// GEMM's epilogue. The epilogue sum needs every rank's tile of an output tile
// on one cluster, rank after rank; with that order the ranks' operand panels
// stop sharing L2 and the partials' stream evicts the running sums, so on the
// Llama-70B MLP shape the GEMM took as long as the summing kernel it replaces
// (1205 against 1051 us, DRAM reads 2.6 against 1.0 GB).
thread_local int g_sum_in_epilogue = 0;

}  // namespace

}  // namespace rtp

using namespace rtp;

namespace {

// Forward MLP; H (may be NULL) receives the bf16 pre-activations X A_i.
int tp_mlp_impl(const char* fn, int P, int64_t M, int64_t K, int64_t F, int64_t N, const void* X,
                const void* const* A_shards, const void* const* B_shards, void* const* Y, void* const* H,
                void* const* partials, float* Z, int mode, int chunks, int col_blocks, rtp_stream s0_, rtp_stream s1_)
{
    if (P < 1 || P > MAX_GROUPS) return fail(RTP_EUNSUPPORTED, "%s: P = %d outside [1, %d]", fn, P, MAX_GROUPS);
    if (!A_shards || !B_shards || !Y) return fail(RTP_EINVAL, "%s: NULL argument", fn);
    if (mode != 0 && mode != 1) return fail(RTP_EINVAL, "%s: mode %d", fn, mode);
    if (mode == 0 && !partials) return fail(RTP_EINVAL, "%s: mode 0 needs partial buffers", fn);
    if (chunks != 1 && chunks != 2 && chunks != 4) return fail(RTP_EINVAL, "%s: chunks %d not in {1,2,4}", fn, chunks);
    if (col_blocks != 1 && col_blocks != 2) return fail(RTP_EINVAL, "%s: col_blocks %d not in {1,2}", fn, col_blocks);
    if (mode == 1 && col_blocks != 1) return fail(RTP_EINVAL, "%s: column blocks apply to mode 0", fn);
    if (M < 0 || K < 1 || F < 1 || N < 1) return fail(RTP_ESHAPE, "%s: sizes M=%lld K=%lld F=%lld N=%lld", fn, (long long)M,
                                                      (long long)K, (long long)F, (long long)N);
    if (F % P) return fail(RTP_ESHAPE, "%s: F=%lld is not divisible by P=%d", fn, (long long)F, P);
    const int64_t Fp = F / P;
    if (M % chunks) return fail(RTP_ESHAPE, "%s: M=%lld is not divisible by chunks=%d", fn, (long long)M, chunks);
    if (K % 8 || Fp % 8) return fail(RTP_ESHAPE, "%s: K and F/P must be multiples of 8 (16-byte rows)", fn);
    if (N % (8 * col_blocks)) return fail(RTP_ESHAPE, "%s: N must be a multiple of %d", fn, 8 * col_blocks);
    if (M >= ((int64_t)1 << 31) || K >= ((int64_t)1 << 31) || Fp >= ((int64_t)1 << 31) || N >= ((int64_t)1 << 31))
        return fail(RTP_ESHAPE, "%s: extents must stay below 2^31", fn);
    // Buffers with M rows (X, Y, H, partials, Z) are empty, and may be NULL,
    // when M == 0: then nothing is launched.
    if (M > 0 && (!X || !Z)) return fail(RTP_EINVAL, "%s: NULL argument", fn);
    if (!aligned16(X) || !aligned16(Z)) return fail(RTP_EINVAL, "%s: X and Z must be 16-byte aligned", fn);
    for (int i = 0; i < P; ++i) {
        if (!A_shards[i] || !B_shards[i] || (M > 0 && (!Y[i] || (mode == 0 && !partials[i]) || (H && !H[i]))))
            return fail(RTP_EINVAL, "%s: NULL buffer for rank %d", fn, i);
        if (!aligned16(A_shards[i]) || !aligned16(B_shards[i]) || !aligned16(Y[i]) ||
            (mode == 0 && !aligned16(partials[i])) || (H && !aligned16(H[i])))
            return fail(RTP_EINVAL, "%s: buffers of rank %d must be 16-byte aligned", fn, i);
    }
    if (M == 0) return RTP_OK;
    cudaStream_t s0 = static_cast<cudaStream_t>(s0_), s1 = static_cast<cudaStream_t>(s1_);
    const bool two_streams = s1 != s0;
    Events* ev = nullptr;
    if (mode == 0 && two_streams) {
        int st = events(&ev);
        if (st) return st;
    }
    const int64_t Mc = M / chunks;
    const int64_t Nb = N / col_blocks;
    // mode 0: the partials' rank sum in the row-parallel GEMM's epilogue, or
    // in kernels of their own (on s1 beside the next GEMMs when given)
    const bool sum_in_gemm = mode == 0 && g_sum_in_epilogue;

    // GEMM1 arguments (tensor maps shared by every chunk)
    static thread_local GemmArgs g1, g2;
    std::memset(&g1, 0, sizeof g1);
    std::memset(&g2, 0, sizeof g2);
    int st;
    for (int i = 0; i < P; ++i) {
        if ((st = make_map(&g1.ta[i], X, M, K, 128))) return st;
        if ((st = make_map(&g1.tb[i], A_shards[i], K, Fp, BK))) return st;
        if ((st = make_map(&g2.ta[i], Y[i], M, Fp, 128))) return st;
        if ((st = make_map(&g2.tb[i], B_shards[i], Fp, N, BK))) return st;
    }
    g1.store_h = H != nullptr;
    g1.ldo = Fp;
    g1.groups = P;
    g1.fused = 0;
    g1.rank_fold = RANKS_IN_N;  // every rank multiplies the same X
    g1.epi = EPI_GELU_BF16;
    const int bm = BM2;
    g1.m_tiles = (int)((Mc + bm - 1) / bm);
    g1.n_tiles = (int)((Fp + BN - 1) / BN);
    g1.kb_per_group = (int)((K + BK - 1) / BK);
    g1.n0 = 0;
    g1.n_end = (int)Fp;
    g2.ldo = N;
    g2.groups = P;
    g2.fused = mode == 1;
    g2.epi = EPI_F32;
    g2.m_tiles = (int)((Mc + bm - 1) / bm);
    g2.n_tiles = (int)((Nb + BN - 1) / BN);
    g2.kb_per_group = (int)((Fp + BK - 1) / BK);

    // The launches in order: per chunk c, GEMM1 (all ranks), then per column
    // block b the row-parallel GEMM of window (c, b) (rows of chunk c, columns
    // of block b of Z). In mode 0 a window's partials are complete once its
    // GEMM2 has run, and Z's window is their sum: computed in that GEMM's
    // epilogue as the ranks' tiles finish (sum_in_gemm), or by a kernel of its
    // own that runs on s1 beside the next window's GEMMs.
    struct Launch {
        bool gemm2;
        int c, b;
    };
    std::vector<Launch> ls;  // host allocations all happen before the first launch
    for (int c = 0; c < chunks; ++c) {
        ls.push_back(Launch{false, c, 0});
        for (int b = 0; b < (mode == 0 ? col_blocks : 1); ++b) ls.push_back(Launch{true, c, b});
    }
    const int nwin = mode == 0 ? chunks * col_blocks : 0;
    // Window sums as kernels of their own: one boxing task each,
    // Z[rows, cols] = sum_i partial_i[rows, cols].
    std::vector<std::vector<PlanTask>> red_tasks(sum_in_gemm ? 0 : (size_t)nwin);
    if (!red_tasks.empty()) {
        inject_alloc_fault();
        const std::vector<int64_t> vol_src((size_t)P, M * N), vol_dst(1, M * N);
        for (int w = 0; w < nwin; ++w) {
            const int c = w / col_blocks, b = w % col_blocks;
            PlanTask t;
            t.cols = Nb;
            t.rows = Mc;
            t.n_outer = 1;
            t.ext[0] = Mc;
            t.sstr[0] = N;
            t.dstr[0] = N;
            if (col_blocks == 1) {  // whole rows: one contiguous run
                t.cols = Mc * N;
                t.rows = 1;
                t.n_outer = 0;
            }
            const int64_t off = c * Mc * N + b * Nb;
            for (int i = 0; i < P; ++i) t.src.push_back(Ref{i, off});
            t.dst.push_back(Ref{0, off});
            red_tasks[(size_t)w].push_back(std::move(t));
            if ((st = check_task_bounds(fn, red_tasks[(size_t)w], vol_src, vol_dst))) return st;
        }
    }
    // Output maps of every launch, encoded before the first launch: each
    // covers the launch's window, so its TMA stores stay inside it.
    std::vector<CUtensorMap> omaps(ls.size() * 2 * MAX_GROUPS);
    for (size_t j = 0; j < ls.size(); ++j) {
        const Launch& L = ls[j];
        CUtensorMap* o = &omaps[j * 2 * MAX_GROUPS];
        const int64_t m_end = (L.c + 1) * Mc, n_end = (L.b + 1) * Nb;
        for (int i = 0; i < P; ++i) {
            if (!L.gemm2) {
                if ((st = make_out_map(&o[i], Y[i], m_end, Fp, Fp, false))) return st;
                if (H && (st = make_out_map(&o[MAX_GROUPS + i], H[i], m_end, Fp, Fp, false))) return st;
            } else if (mode == 0) {
                if ((st = make_out_map(&o[i], partials[i], m_end, n_end, N, true))) return st;
            } else if (i == 0) {
                if ((st = make_out_map(&o[0], Z, m_end, N, N, true))) return st;
            }
        }
    }
    g2.sum_into = sum_in_gemm;
    g2.sum_dst = sum_in_gemm ? Z : nullptr;

    void* zdst[1] = {Z};
    for (size_t j = 0; j < ls.size(); ++j) {
        const Launch& L = ls[j];
        GemmArgs& g = L.gemm2 ? g2 : g1;
        g.m0 = (int)(L.c * Mc);
        g.m_end = (int)((L.c + 1) * Mc);
        if (L.gemm2) {
            g.n0 = (int)(L.b * Nb);
            g.n_end = (int)((L.b + 1) * Nb);
        }
        std::memcpy(g.to, &omaps[j * 2 * MAX_GROUPS], sizeof g.to);
        std::memcpy(g.to2, &omaps[j * 2 * MAX_GROUPS + MAX_GROUPS], sizeof g.to2);
        if ((st = launch_gemm(g, s0))) return st;
        if (!L.gemm2 || mode == 1 || sum_in_gemm) continue;
        const int w = L.c * col_blocks + L.b;
        cudaStream_t rs = s0;
        if (two_streams) {
            if (cudaEventRecord(ev->fwd, s0) != cudaSuccess || cudaStreamWaitEvent(s1, ev->fwd, 0) != cudaSuccess)
                return fail(RTP_ECUDA, "tp_mlp: event ordering failed");
            rs = s1;
        }
        // Beside the next chunk's GEMM (one CTA per SM), a sum on s1 runs
        // kOverlapBlocksPerSm blocks per SM so that both fit on every SM at
        // once; the last window's sum has nothing to overlap and takes the
        // whole GPU.
        const bool last = w == nwin - 1;
        const int bps = rs != s0 && !last ? kOverlapBlocksPerSm : 4;
        if ((st = launch_tasks(RTP_F32, red_tasks[(size_t)w], (const void* const*)partials, zdst, rs, nullptr, bps)))
            return st;
    }
    if (mode == 0 && two_streams && !sum_in_gemm) {
        if (cudaEventRecord(ev->back, s1) != cudaSuccess || cudaStreamWaitEvent(s0, ev->back, 0) != cudaSuccess)
            return fail(RTP_ECUDA, "tp_mlp: event ordering failed");
    }
    return RTP_OK;
}

}  // namespace

extern "C" {

int rtp_tp_mlp(int P, int64_t M, int64_t K, int64_t F, int64_t N, const void* X, const void* const* A_shards,
               const void* const* B_shards, void* const* Y, void* const* partials, float* Z, int mode, int chunks,
               int col_blocks, rtp_stream s0, rtp_stream s1)
{
    return guarded("rtp_tp_mlp", [&] {
        return tp_mlp_impl("rtp_tp_mlp", P, M, K, F, N, X, A_shards, B_shards, Y, nullptr, partials, Z, mode, chunks,
                           col_blocks, s0, s1);
    });
}

int rtp_tp_mlp_train_forward(int P, int64_t M, int64_t K, int64_t F, int64_t N, const void* X,
                             const void* const* A_shards, const void* const* B_shards, void* const* Y, void* const* H,
                             float* Z, rtp_stream stream)
{
    if (!H) return fail(RTP_EINVAL, "rtp_tp_mlp_train_forward: NULL H");
    return guarded("rtp_tp_mlp_train_forward", [&] {
        return tp_mlp_impl("rtp_tp_mlp_train_forward", P, M, K, F, N, X, A_shards, B_shards, Y, H, nullptr, Z, 1, 1, 1,
                           stream, stream);
    });
}

int rtp_tp_mlp_overlap(int sum_in_epilogue, int* previous)
{
    if (sum_in_epilogue != 0 && sum_in_epilogue != 1)
        return fail(RTP_EINVAL, "rtp_tp_mlp_overlap: %d is not 0 or 1", sum_in_epilogue);
    if (previous) *previous = g_sum_in_epilogue;
    g_sum_in_epilogue = sum_in_epilogue;
    return RTP_OK;
}

static int tp_mlp_backward_body(int P, int64_t M, int64_t K, int64_t F, int64_t N, const void* X,
                                const void* const* A_shards, const void* const* B_shards, const void* const* H,
                                const void* const* Y, const void* dZ, void* const* dH, void* const* dX_partials,
                                float* dX, float* const* dA, float* const* dB, int mode, rtp_stream s0_,
                                rtp_stream s1_)
{
    const char* fn = "rtp_tp_mlp_backward";
    if (P < 1 || P > MAX_GROUPS) return fail(RTP_EUNSUPPORTED, "%s: P = %d outside [1, %d]", fn, P, MAX_GROUPS);
    if (!A_shards || !B_shards || !H || !Y || !dH || !dA || !dB) return fail(RTP_EINVAL, "%s: NULL argument", fn);
    if (M > 0 && (!X || !dZ || !dX)) return fail(RTP_EINVAL, "%s: NULL argument", fn);
    if (mode != 0 && mode != 1) return fail(RTP_EINVAL, "%s: mode %d", fn, mode);
    if (mode == 0 && !dX_partials) return fail(RTP_EINVAL, "%s: mode 0 needs partial buffers", fn);
    if (M < 0 || K < 1 || F < 1 || N < 1) return fail(RTP_ESHAPE, "%s: sizes M=%lld K=%lld F=%lld N=%lld", fn, (long long)M,
                                                      (long long)K, (long long)F, (long long)N);
    if (F % P) return fail(RTP_ESHAPE, "%s: F=%lld is not divisible by P=%d", fn, (long long)F, P);
    const int64_t Fp = F / P;
    if (K % 8 || Fp % 8 || N % 8) return fail(RTP_ESHAPE, "%s: K, F/P and N must be multiples of 8 (16-byte rows)", fn);
    if (M >= ((int64_t)1 << 31) || K >= ((int64_t)1 << 31) || Fp >= ((int64_t)1 << 31) || N >= ((int64_t)1 << 31))
        return fail(RTP_ESHAPE, "%s: extents must stay below 2^31", fn);
    if (!aligned16(X) || !aligned16(dZ) || !aligned16(dX))
        return fail(RTP_EINVAL, "%s: X, dZ and dX must be 16-byte aligned", fn);
    for (int i = 0; i < P; ++i) {
        // buffers with M rows are empty (and may be NULL) when M == 0
        const void* bufs[8] = {A_shards[i], B_shards[i], dA[i], dB[i], H[i], Y[i], dH[i],
                               mode == 0 ? dX_partials[i] : (const void*)dX};
        for (int b = 0; b < (M > 0 ? 8 : 4); ++b) {
            if (!bufs[b]) return fail(RTP_EINVAL, "%s: NULL buffer for rank %d", fn, i);
            if (!aligned16(bufs[b])) return fail(RTP_EINVAL, "%s: buffers of rank %d must be 16-byte aligned", fn, i);
        }
    }
    cudaStream_t s0 = static_cast<cudaStream_t>(s0_), s1 = static_cast<cudaStream_t>(s1_);
    if (M == 0) {  // no tokens: the weight gradients are zero, dX is empty
        for (int i = 0; i < P; ++i) {
            if (cudaMemsetAsync(dA[i], 0, (size_t)(K * Fp * 4), s0) != cudaSuccess ||
                cudaMemsetAsync(dB[i], 0, (size_t)(Fp * N * 4), s0) != cudaSuccess)
                return fail(RTP_ECUDA, "%s: cudaMemsetAsync failed", fn);
        }
        return RTP_OK;
    }
    const bool two_streams = mode == 0 && s1 != s0;
    Events* ev = nullptr;
    if (two_streams) {
        int st = events(&ev);
        if (st) return st;
    }
    static thread_local GemmArgs gh, gx, ga, gb;
    std::memset(&gh, 0, sizeof gh);
    std::memset(&gx, 0, sizeof gx);
    std::memset(&ga, 0, sizeof ga);
    std::memset(&gb, 0, sizeof gb);
    int st;
    for (int i = 0; i < P; ++i) {
        // dH_i = (dZ B_i^T) * GELU'(H_i): dZ K-major [M, N], B_i^T read K-major from B_i [F/P, N]
        if ((st = make_map(&gh.ta[i], dZ, M, N, 128))) return st;
        if ((st = make_map(&gh.tb[i], B_shards[i], Fp, N, 128))) return st;
        if ((st = make_out_map(&gh.to[i], dH[i], M, Fp, Fp, false))) return st;
        gh.aux[i] = H[i];
        // dX (+)= dH_i A_i^T: dH_i K-major [M, F/P], A_i^T read K-major from A_i [K, F/P]
        if ((st = make_map(&gx.ta[i], dH[i], M, Fp, 128))) return st;
        if ((st = make_map(&gx.tb[i], A_shards[i], K, Fp, 128))) return st;
        if (mode == 0 && (st = make_out_map(&gx.to[i], dX_partials[i], M, K, K, true))) return st;
        if (mode == 1 && i == 0 && (st = make_out_map(&gx.to[0], dX, M, K, K, true))) return st;
        // dA_i = X^T dH_i: X^T read M-major from X [M, K], dH_i N-major
        if ((st = make_map(&ga.ta[i], X, M, K, 64))) return st;
        if ((st = make_map(&ga.tb[i], dH[i], M, Fp, BK))) return st;
        if ((st = make_out_map(&ga.to[i], dA[i], K, Fp, Fp, true))) return st;
        // dB_i = Y_i^T dZ: Y_i^T read M-major from Y_i [M, F/P], dZ N-major
        if ((st = make_map(&gb.ta[i], Y[i], M, Fp, 64))) return st;
        if ((st = make_map(&gb.tb[i], dZ, M, N, BK))) return st;
        if ((st = make_out_map(&gb.to[i], dB[i], Fp, N, N, true))) return st;
    }
    auto shape = [&](GemmArgs& g, int64_t rows, int64_t cols, int64_t kdim, int epi, int cfg, int fused) {
        g.groups = P;
        g.fused = fused;
        g.epi = epi;
        g.cfg = cfg;
        g.ldo = cols;
        g.m_tiles = (int)((rows + BM2 - 1) / BM2);
        g.n_tiles = (int)((cols + BN - 1) / BN);
        g.kb_per_group = (int)((kdim + BK - 1) / BK);
        g.m_end = (int)rows;
        g.n_end = (int)cols;
    };
    shape(gh, M, Fp, N, EPI_DGELU_BF16, CFG_B_K, 0);
    shape(gx, M, K, Fp, EPI_F32, CFG_B_K, mode == 1);
    shape(ga, K, Fp, M, EPI_F32, CFG_A_MN, 0);
    shape(gb, Fp, N, M, EPI_F32, CFG_A_MN, 0);
    // dZ and X^T are the A operands of every rank's dH and dA. dB (long K,
    // shared B operand) keeps the rank-outer order: with K = M its operand
    // panels do not survive in L2 between waves, and rank by rank its waves
    // are already near square (8 x 9.5 tiles on the 8192x4096x16384x4096 MLP).
    gh.rank_fold = RANKS_IN_N;
    ga.rank_fold = RANKS_IN_N;
    // Mode 0: the dX partials' rank sum. By default the dX GEMM adds each
    // output tile's partials up in its epilogue as the ranks' tiles finish;
    // otherwise it is a kernel of its own, on s1 beside the weight-gradient
    // GEMMs when a second stream is given (the Domino backward).
    const bool sum_in_gemm = mode == 0 && g_sum_in_epilogue;
    std::vector<PlanTask> dx_tasks;  // host allocations before the first launch
    if (mode == 0 && !sum_in_gemm) {
        inject_alloc_fault();
        PlanTask t;
        t.cols = M * K;
        t.rows = 1;
        t.n_outer = 0;
        for (int i = 0; i < P; ++i) t.src.push_back(Ref{i, 0});
        t.dst.push_back(Ref{0, 0});
        dx_tasks.push_back(std::move(t));
        if ((st = check_task_bounds(fn, dx_tasks, std::vector<int64_t>((size_t)P, M * K), std::vector<int64_t>(1, M * K))))
            return st;
    }
    gx.sum_into = sum_in_gemm;
    gx.sum_dst = sum_in_gemm ? dX : nullptr;
    if ((st = launch_gemm(gh, s0)) || (st = launch_gemm(gx, s0))) return st;
    if (mode == 0 && !sum_in_gemm) {
        cudaStream_t rs = s0;
        if (two_streams) {
            if (cudaEventRecord(ev->fwd, s0) != cudaSuccess || cudaStreamWaitEvent(s1, ev->fwd, 0) != cudaSuccess)
                return fail(RTP_ECUDA, "%s: event ordering failed", fn);
            rs = s1;
        }
        void* d[1] = {dX};
        if ((st = launch_tasks(RTP_F32, dx_tasks, (const void* const*)dX_partials, d, rs, nullptr,
                               two_streams ? kOverlapBlocksPerSm : 4)))
            return st;
    }
    if ((st = launch_gemm(ga, s0)) || (st = launch_gemm(gb, s0))) return st;
    if (two_streams && !sum_in_gemm) {
        if (cudaEventRecord(ev->back, s1) != cudaSuccess || cudaStreamWaitEvent(s0, ev->back, 0) != cudaSuccess)
            return fail(RTP_ECUDA, "%s: event ordering failed", fn);
    }
    return RTP_OK;
}

int rtp_tp_mlp_backward(int P, int64_t M, int64_t K, int64_t F, int64_t N, const void* X, const void* const* A_shards,
                        const void* const* B_shards, const void* const* H, const void* const* Y, const void* dZ,
                        void* const* dH, void* const* dX_partials, float* dX, float* const* dA, float* const* dB,
                        int mode, rtp_stream s0_, rtp_stream s1_)
{
    return guarded("rtp_tp_mlp_backward", [&] {
        return tp_mlp_backward_body(P, M, K, F, N, X, A_shards, B_shards, H, Y, dZ, dH, dX_partials, dX, dA, dB, mode,
                                    s0_, s1_);
    });
}

int rtp_tp_mlp_sp(int P, int64_t M, int64_t K, int64_t F, int64_t N, const void* const* X_shards,
                  const void* const* A_shards, const void* const* B_shards, void* const* Y, float* const* Z_shards,
                  rtp_stream stream_)
{
    const char* fn = "rtp_tp_mlp_sp";
    if (P < 1 || P > MAX_GROUPS) return fail(RTP_EUNSUPPORTED, "%s: P = %d outside [1, %d]", fn, P, MAX_GROUPS);
    if (!X_shards || !A_shards || !B_shards || !Y || !Z_shards) return fail(RTP_EINVAL, "%s: NULL argument", fn);
    if (M < 0 || K < 1 || F < 1 || N < 1) return fail(RTP_ESHAPE, "%s: sizes M=%lld K=%lld F=%lld N=%lld", fn,
                                                      (long long)M, (long long)K, (long long)F, (long long)N);
    if (F % P || M % P) return fail(RTP_ESHAPE, "%s: F=%lld and M=%lld must be divisible by P=%d", fn, (long long)F, (long long)M, P);
    const int64_t Fp = F / P, Mr = M / P;
    if (Mr % 128) return fail(RTP_ESHAPE, "%s: M/P=%lld must be a multiple of 128 (one row block per shard)", fn, (long long)Mr);
    if (K % 8 || Fp % 8 || N % 8) return fail(RTP_ESHAPE, "%s: K, F/P and N must be multiples of 8 (16-byte rows)", fn);
    if (M >= ((int64_t)1 << 31) || K >= ((int64_t)1 << 31) || Fp >= ((int64_t)1 << 31) || N >= ((int64_t)1 << 31))
        return fail(RTP_ESHAPE, "%s: extents must stay below 2^31", fn);
    for (int i = 0; i < P; ++i) {
        // X_shards, Y and Z_shards have rows of the M tokens: empty, and possibly NULL, when M == 0
        if (!A_shards[i] || !B_shards[i] || (M > 0 && (!X_shards[i] || !Y[i] || !Z_shards[i])))
            return fail(RTP_EINVAL, "%s: NULL buffer for rank %d", fn, i);
        if (!aligned16(X_shards[i]) || !aligned16(A_shards[i]) || !aligned16(B_shards[i]) || !aligned16(Y[i]) || !aligned16(Z_shards[i]))
            return fail(RTP_EINVAL, "%s: buffers of rank %d must be 16-byte aligned", fn, i);
    }
    if (M == 0) return RTP_OK;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    static thread_local GemmArgs g1, g2;
    std::memset(&g1, 0, sizeof g1);
    std::memset(&g2, 0, sizeof g2);
    int st;
    for (int i = 0; i < P; ++i) {
        if ((st = make_map(&g1.ta[i], X_shards[i], Mr, K, 128))) return st;  // X rows by shard
        if ((st = make_map(&g1.tb[i], A_shards[i], K, Fp, BK))) return st;
        if ((st = make_out_map(&g1.to[i], Y[i], M, Fp, Fp, false))) return st;
        if ((st = make_map(&g2.ta[i], Y[i], M, Fp, 128))) return st;
        if ((st = make_map(&g2.tb[i], B_shards[i], Fp, N, BK))) return st;
        if ((st = make_out_map(&g2.to[i], Z_shards[i], Mr, N, N, true))) return st;  // Z rows by shard
    }
    // column-parallel GEMM with the all-gather of X fused into its loads
    g1.ldo = Fp;
    g1.groups = P;
    g1.fused = 0;
    g1.epi = EPI_GELU_BF16;
    g1.m_tiles = (int)((M + BM2 - 1) / BM2);
    g1.n_tiles = (int)((Fp + BN - 1) / BN);
    g1.kb_per_group = (int)((K + BK - 1) / BK);
    g1.m_end = (int)M;
    g1.n_end = (int)Fp;
    g1.a_rows_per_map = (int)Mr;
    g1.a_maps = P;
    g1.cfg = CFG_SP_A;
    g1.rank_fold = RANKS_IN_N;  // every rank multiplies the same (gathered) X
    if ((st = launch_gemm(g1, stream))) return st;
    // row-parallel GEMM: ranks summed in TMEM, rows scattered to their shard
    g2.ldo = N;
    g2.groups = P;
    g2.fused = 1;
    g2.epi = EPI_F32;
    g2.m_tiles = (int)((M + BM2 - 1) / BM2);
    g2.n_tiles = (int)((N + BN - 1) / BN);
    g2.kb_per_group = (int)((Fp + BK - 1) / BK);
    g2.m_end = (int)M;
    g2.n_end = (int)N;
    g2.out_rows_per_ptr = (int)Mr;
    g2.out_ptrs = P;
    g2.cfg = CFG_SP_OUT;
    return launch_gemm(g2, stream);
}

int rtp_wait_selftest(int kernel, unsigned long long limit_ns, uint32_t* out, rtp_stream stream)
{
    if (kernel != 0 && kernel != 1) return fail(RTP_EINVAL, "rtp_wait_selftest: kernel %d not 0 or 1", kernel);
    if (!out) return fail(RTP_EINVAL, "rtp_wait_selftest: NULL out");
    if (limit_ns < 1000000ull || limit_ns > 1000000000ull)
        return fail(RTP_EINVAL, "rtp_wait_selftest: limit %llu ns outside [1 ms, 1 s]", limit_ns);
    if (!aligned16(out)) return fail(RTP_EINVAL, "rtp_wait_selftest: out must be 16-byte aligned");
    if (kernel == 1) return bulk_wait_selftest(limit_ns, out, stream);
    wait_selftest_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(limit_ns, out);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(RTP_ECUDA, "rtp_wait_selftest: launch failed: %s", cudaGetErrorString(e));
    return RTP_OK;
}

int rtp_device_error(rtp_stream stream, uint32_t* code)
{
    if (!code) return fail(RTP_EINVAL, "rtp_device_error: NULL argument");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_tp_error, sizeof v, 0, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemcpyToSymbolAsync(g_tp_error, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return fail(RTP_ECUDA, "rtp_device_error: %s", cudaGetErrorString(cudaGetLastError()));
    uint32_t box = 0;
    int st = take_boxing_error(stream, &box);
    if (st) return st;
    *code = v ? v : box;
    return RTP_OK;
}

}  // extern "C"
