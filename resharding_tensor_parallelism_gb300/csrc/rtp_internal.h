// Internal declarations of the rtp library (host side). Not installed.
#pragma once

#include <cstdint>
#include <exception>
#include <new>
#include <string>
#include <vector>

#include "rtp.h"

namespace rtp {

// ---- errors ------------------------------------------------------------------
// Records a message for rtp_last_error() on this thread and returns `status`.
int fail(int status, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
void clear_error();

// Runs the body of an entry point that allocates host memory: a failed
// allocation (std::bad_alloc) becomes RTP_ENOMEM, and no exception crosses the
// C ABI.
template <class F>
int guarded(const char* fn, F&& body) noexcept
{
    try {
        return body();
    } catch (const std::bad_alloc&) {
        return fail(RTP_ENOMEM, "%s: a host allocation failed", fn);
    } catch (const std::exception& e) {
        return fail(RTP_EUNSUPPORTED, "%s: internal error: %s", fn, e.what());
    }
}

// ---- spec geometry -------------------------------------------------------------
int64_t num_ranks(const rtp_spec& s);
// RTP_OK or an error (message recorded) if the spec cannot describe a tensor of rank ndim.
int check_spec(int ndim, const rtp_spec& s, const char* what);
// Reduction of a spec's partial mesh dims: RED_SUM (also when there are none), RED_MIN, RED_MAX.
enum { RED_SUM = 0, RED_MIN = 1, RED_MAX = 2 };
int partial_reduction(const rtp_spec& s);
bool is_partial(int sbp_kind);
// Mesh coordinates of every rank: coords[r * RTP_MAX_MESH_NDIM + d].
void rank_coords(const rtp_spec& s, int64_t* coords);

struct Box {
    int64_t lo[RTP_MAX_NDIM];
    int64_t hi[RTP_MAX_NDIM];
    bool holds_value;  // false: member of a partial group that holds the reduction's identity
    bool b_rep;        // coordinate 0 on every broadcast mesh dim
    int64_t pidx;      // index of the partial coordinates (row-major), 0 if no P dim
};
// Piece of rank r (caller validated the spec).
Box rank_box(int ndim, const int64_t* shape, const rtp_spec& s, const int64_t* coords_of_r);
int64_t box_volume(int ndim, const Box& b);

// ---- copy plan -------------------------------------------------------------------
// One rectangular region moved from n_src source pieces (summed when n_src > 1,
// zeros when n_src == 0) to n_dst destination pieces. After merging, the region
// is rows x cols: `cols` consecutive elements in every buffer, rows indexed by
// the mixed radix ext[0..n_outer) with per-buffer element strides.
constexpr int kMaxOuter = 7;
struct Ref {
    int rank;        // buffer index
    int64_t offset;  // element offset of the region's first element
};
struct PlanTask {
    int64_t rows = 1, cols = 1;
    int n_outer = 0;
    int64_t ext[kMaxOuter] = {};
    int64_t sstr[kMaxOuter] = {};
    int64_t dstr[kMaxOuter] = {};
    std::vector<Ref> src;
    std::vector<Ref> dst;
    int op = RED_SUM;  // how several sources combine; with no source, dst is filled with op's identity
};
// Plans moving a tensor laid out by `src` into the layout `dst`.
int plan_reshard(int ndim, const int64_t* shape, const rtp_spec& src, const rtp_spec& dst,
                 std::vector<PlanTask>* tasks);

// The single-rank, broadcast spec of an unsharded tensor.
rtp_spec whole_tensor_spec();

// Every element a task touches lies inside the piece it reads or writes: for
// each source (destination) reference, its first element offset is >= 0 and
// its last is below src_vol[rank] (dst_vol[rank]), the piece's element count.
// RTP_EINVAL (message names fn, the task and the piece) otherwise.
int check_task_bounds(const char* fn, const std::vector<PlanTask>& tasks, const std::vector<int64_t>& src_vol,
                      const std::vector<int64_t>& dst_vol);

// Test hooks (rtp_test_hook), one-shot and per thread. inject_alloc_fault()
// throws std::bad_alloc when the allocation-failure hook is armed (and
// disarms it); it marks the host allocations of planning.
void inject_alloc_fault();

// ---- launches (boxing.cu) --------------------------------------------------------------
// Executes planned tasks on `stream`; src/dst buffer arrays are indexed by Ref::rank.
// blocks_per_sm caps the persistent grid (default 4 = full occupancy); a
// reduction that should run beside another kernel uses 1.
int launch_tasks(int dtype, const std::vector<PlanTask>& tasks, const void* const* src, void* const* dst,
                 void* stream, int* n_launches_out, int blocks_per_sm = 4);
// Number of launches the tasks need (host only).
int count_launches(const std::vector<PlanTask>& tasks);
// How many of the tasks a reshard would run in each form of the boxing kernel:
// counts[0] registers, [1] bulk staging, [2] TMA tiles (3D), [3] TMA tiles (4D),
// for 256-byte aligned buffers and the kernel alone on the GPU (host only).
int classify_tasks(int dtype, const std::vector<PlanTask>& tasks, int32_t* counts);
// Reads and clears the boxing kernel's device error word (synchronises `stream`).
int take_boxing_error(void* stream, uint32_t* code);
// Launches the resharding kernel's bounded-wait self-test (a wait that never
// completes, given up after limit_ns); out[0] = 1 when the block stopped on it.
int bulk_wait_selftest(unsigned long long limit_ns, uint32_t* out, void* stream);
// The driver's cuTensorMapEncodeTiled (a PFN_cuTensorMapEncodeTiled_v12000), or NULL.
void* tensor_map_encoder();

}  // namespace rtp
