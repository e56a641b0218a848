/*
 * rtp.h - resharding and 1D tensor parallelism on a virtual device mesh held
 * inside one GPU (NVIDIA GB300, sm_103a).
 *
 * The virtual "devices" (ranks) of a mesh are separate buffers in the memory
 * of one GPU. Every rank buffer, and every other buffer passed here, is
 * allocated and owned by the caller; the library never allocates memory that
 * the caller sees and never frees a caller pointer.
 *
 * Conventions for every call:
 *   - Return value: RTP_OK (0) or a negative rtp_status. On failure,
 *     rtp_last_error() returns a text for the calling thread, and nothing
 *     was launched (arguments are checked on the host before any launch).
 *     RTP_ECUDA means that a CUDA call failed; its message names the call.
 *   - Tensors are dense and row-major (C order). Shapes are int64 arrays of
 *     length ndim (0 < ndim <= RTP_MAX_NDIM). Element types: rtp_dtype.
 *   - "device pointer" means memory of the current CUDA device; calls that
 *     take a stream are asynchronous with respect to the host and ordered on
 *     that stream (NULL = the legacy default stream). Host-only calls (the
 *     front-ends, shapes, inference) touch no GPU state.
 *   - Source and destination buffers must not overlap: rtp_shard and
 *     rtp_reshard return RTP_EINVAL, before any launch, when a source piece
 *     they would read and a destination piece share bytes.
 *   - Calls may come from several host threads at once. Launch parameters,
 *     cached tensor maps and the events that order a call's two streams are
 *     kept per thread, so concurrent calls on their own streams do not wait
 *     on, or overwrite, each other's state. Buffers that two concurrent calls
 *     both write are the caller's to order.
 *
 * Readings of the pages that the semantics rely on (pages are cited by title
 * and section):
 *   - split order: "ONNX multi-device proposal", section on the index rule for
 *     multi-axis splits: the first sharded axis is the outer loop, so shards
 *     are produced in (a outer, b inner) order; for an ND-SBP on a mesh, mesh
 *     dim 0 is the outer level (OneFlow 2D SBP example on ranks [[0,1],[2,3]]).
 *   - uneven extents are left to the backend by the ONNX page (note on
 *     divisibility). Here every split level cuts its interval into pieces of
 *     ceil(len/n) with a short (possibly empty) last piece; two mesh dims
 *     splitting one axis cut it level by level, outer mesh dim first.
 *   - partial (OneFlow SBP definition): the logical tensor is the element-wise
 *     sum of the rank tensors. When a logical tensor is *sharded* to a
 *     partial layout, the rank whose partial coordinates are all zero holds
 *     the value and the other ranks hold zeros.
 */
#ifndef RTP_H_
#define RTP_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define RTP_MAX_NDIM 8
#define RTP_MAX_MESH_NDIM 4
#define RTP_MAX_RANKS 64

typedef enum { RTP_F32 = 0, RTP_BF16 = 1 } rtp_dtype;

typedef enum {
    RTP_OK = 0,
    RTP_EINVAL = -1,       /* malformed argument (NULL pointer, bad spec, bad axis) */
    RTP_ESHAPE = -2,       /* sizes that do not fit the operation (e.g. F % P != 0) */
    RTP_EUNSUPPORTED = -3, /* legal-looking request outside what is implemented */
    RTP_ECONFLICT = -4,    /* inference found no consistent result */
    RTP_ECUDA = -5,        /* a CUDA runtime/driver call failed */
    RTP_ENOMEM = -6        /* host-side allocation failed */
} rtp_status;

/*
 * Per-mesh-dim distribution (OneFlow SBP page: split, broadcast, partial; the
 * page notes that besides sum, min and max also work as partial reductions).
 * All partial mesh dims of one spec use the same reduction (else
 * RTP_EUNSUPPORTED). When a logical tensor is sharded to a partial layout,
 * the rank whose partial coordinates are all zero holds the tensor and the
 * others hold the reduction's identity: 0 (sum), +inf (min), -inf (max).
 * Min and max are exact, so their reshards are bit-exact; they follow IEEE
 * minNum/maxNum (a NaN member is ignored unless all members are NaN) and may
 * return either zero for min/max of +0 and -0.
 */
typedef enum {
    RTP_SBP_SPLIT = 0,
    RTP_SBP_BROADCAST = 1,
    RTP_SBP_PARTIAL_SUM = 2,
    RTP_SBP_PARTIAL_MIN = 3,
    RTP_SBP_PARTIAL_MAX = 4
} rtp_sbp;

/* A CUDA stream (cudaStream_t) passed as an opaque pointer; NULL = default stream. */
typedef void* rtp_stream;

/*
 * Canonical layout of a tensor on a virtual mesh (the ND-SBP form of the
 * OneFlow page; the Paddle dims_mapping and ONNX ShardingSpec forms are
 * converted to it by the front-ends below).
 *   mesh_ndim     number of mesh dims, 1..RTP_MAX_MESH_NDIM
 *   mesh_shape    size of each mesh dim (>= 1); R = product <= RTP_MAX_RANKS
 *   rank_ids      the mesh, row-major: rank_ids[p] is the rank at flat mesh
 *                 position p. Must be a permutation of 0..R-1; rank r's buffer
 *                 is entry r of the buffer arrays passed to shard/reshard.
 *   sbp_kind      per mesh dim, an rtp_sbp value
 *   sbp_axis      per mesh dim with RTP_SBP_SPLIT: the tensor axis it splits,
 *                 in [0, ndim); ignored otherwise
 */
typedef struct {
    int32_t mesh_ndim;
    int64_t mesh_shape[RTP_MAX_MESH_NDIM];
    int32_t rank_ids[RTP_MAX_RANKS];
    int32_t sbp_kind[RTP_MAX_MESH_NDIM];
    int32_t sbp_axis[RTP_MAX_MESH_NDIM];
} rtp_spec;

/* ---- front-ends and geometry (host only) ----------------------------------- */

/*
 * Paddle form ("SPMD rules" design note, ProcessMesh and dims_mapping):
 * dims_mapping[i] = j splits tensor dim i along mesh dim j; -1 keeps it whole.
 * Mesh dims that no tensor dim names are broadcast, or partial-sum when their
 * bit is set in partial_mask. rank_ids: the ProcessMesh ids, row-major (NULL
 * means 0..R-1). Two tensor dims on one mesh dim, or a mesh dim both split
 * and partial, give RTP_EINVAL.
 */
int rtp_spec_from_dims_mapping(int ndim, const int32_t* dims_mapping, int mesh_ndim, const int64_t* mesh_shape,
                               const int32_t* rank_ids, uint32_t partial_mask, rtp_spec* out);

/*
 * ONNX form ("ONNX multi-device proposal", ShardingSpecProto, ShardedDimProto,
 * SimpleShardedDimProto and device_map = index_to_device_group_map):
 *   device[n_device]     rank ids, or negative keys into the group map
 *   group_keys[n_groups] the negative keys; group k holds group_sizes[k]
 *                        ranks, listed consecutively in group_devices
 *   axes[n_sharded], num_shards[n_sharded]
 *                        one simple_sharding per sharded_dim (axis may be
 *                        negative, counted from the end)
 * Split piece s (row-major over the sharded dims, first listed = outer) goes
 * to device[s], or to every rank of its group. Requires the product of
 * num_shards to equal n_device. Result: mesh [num_shards..., group size],
 * the last dim broadcast when groups hold more than one rank.
 * RTP_EUNSUPPORTED: groups of unequal size.
 */
int rtp_spec_from_onnx(int ndim, int n_device, const int64_t* device, int n_groups, const int64_t* group_keys,
                       const int32_t* group_sizes, const int64_t* group_devices, int n_sharded, const int64_t* axes,
                       const int64_t* num_shards, rtp_spec* out);

/*
 * Checks a spec against a tensor rank; RTP_OK if usable, else the reason
 * ("ONNX multi-device proposal", validity check: a sharding spec the backend
 * cannot honour is reported with its reason).
 */
int rtp_spec_check(int ndim, const rtp_spec* spec);

/*
 * Shape of rank `rank`'s piece of a tensor of shape `shape` (out_shape[ndim]),
 * by the split rule of the ONNX page (index rule for multi-axis splits, outer
 * axis first; uneven extents as in the note on divisibility, read as ceil-sized
 * leading pieces).
 */
int rtp_shard_shape(int ndim, const int64_t* shape, const rtp_spec* spec, int rank, int64_t* out_shape);

/*
 * Box [lo, hi) of the logical tensor covered by rank `rank`, and whether the
 * rank holds values (0 only for a non-zero partial coordinate when sharding).
 * The split rule as in rtp_shard_shape; a broadcast mesh dim gives every rank
 * of its group the same box (ONNX page, sharding as broadcast); the members of
 * a partial group share one box (OneFlow page, partial sum).
 */
int rtp_shard_box(int ndim, const int64_t* shape, const rtp_spec* spec, int rank, int64_t* lo, int64_t* hi,
                  int32_t* holds_value);

/* ---- the four calls -------------------------------------------------------- */

/*
 * shard(tensor, spec): materialises every rank's piece of a logical tensor
 * ("ONNX multi-device proposal": sharding as a split, as a broadcast, and
 * split plus broadcast; OneFlow page: split, broadcast, partial).
 *   full       device pointer, the logical tensor [shape]
 *   shard_dev  R device pointers; shard_dev[r] receives rank r's piece, of
 *              shape rtp_shard_shape(r) (empty pieces may pass NULL)
 * Data movement is bit-exact.
 */
int rtp_shard(rtp_dtype dtype, int ndim, const int64_t* shape, const void* full, const rtp_spec* spec,
              void* const* shard_dev, rtp_stream stream);

/*
 * reshard(shards, src_spec, dst_spec): converts rank pieces from one layout to
 * another ("boxing" in the OneFlow page; "reshard inputs" step of the ONNX
 * execution semantics): S(i)->S(j) (all-to-all), S->B (all-gather), B->S
 * (slice), P->B (all-reduce), P->S (reduce-scatter), and any mix on an ND mesh.
 *   src_dev  R_src device pointers laid out by `src`
 *   dst_dev  R_dst device pointers laid out by `dst` (meshes may differ)
 * Without partial sources the result is bit-exact. Partial sources are
 * summed in float32 in a fixed order (partial coordinates row-major), then
 * rounded once to the element type; results are identical run to run.
 */
int rtp_reshard(rtp_dtype dtype, int ndim, const int64_t* shape, const void* const* src_dev, const rtp_spec* src,
                void* const* dst_dev, const rtp_spec* dst, rtp_stream stream);

/*
 * Algorithmic traffic of a reshard (host only): bytes read (each distinct
 * source byte once; every partial read) and bytes written (every destination
 * byte), and the number of copy tasks and kernel launches it plans. The pages
 * have no counterpart to this query: it reports the bytes that the
 * measurements of this library divide by.
 */
int rtp_reshard_cost(rtp_dtype dtype, int ndim, const int64_t* shape, const rtp_spec* src, const rtp_spec* dst,
                     int64_t* bytes_read, int64_t* bytes_written, int32_t* n_tasks, int32_t* n_launches);

/*
 * How rtp_reshard would run the same request: counts[4] receives the number of
 * planned tasks in each form of the resharding kernel: [0] registers
 * (16-byte or narrower vectors), [1] bulk staging through shared memory (runs
 * of 4 KB or more), [2] TMA tiles of a 3D tensor map, [3] TMA tiles of a 4D
 * tensor map (short strided rows). Host only; assumes 256-byte aligned rank
 * buffers (as cudaMalloc returns) and the kernel alone on the GPU (beside
 * another kernel every task takes the register form). Same errors as
 * rtp_reshard_cost. The pages have no counterpart: it describes this
 * library's kernel.
 */
int rtp_reshard_forms(rtp_dtype dtype, int ndim, const int64_t* shape, const rtp_spec* src, const rtp_spec* dst,
                      int32_t* counts);

/*
 * infer_spmd(einsum, dims_mappings) (Paddle "SPMD rules" note, steps 1-3:
 * einsum notation, ShardingMergeForTensors, GetDimsMappingForAxes; ONNX
 * sharding formalism, reduction operators). Host only.
 *   einsum            e.g. "mk,kn->mn": one letter per axis, inputs separated
 *                     by ',', output after "->" (letters a-z, none repeated
 *                     within one operand)
 *   in_dims_mappings  n_in arrays, one entry per letter of that input
 *   out_dims_mapping  receives one entry per output letter
 *   out_partial_mask  bit d set: the output is a partial sum over mesh dim d
 *                     (a sharded letter summed away)
 *   in_needs_reshard_mask  bit j set: input j must be resharded to its
 *                     inferred mapping (written to in_inferred[j] if given)
 * Merge rule: a letter takes the first mesh dim any input gives it (inputs in
 * order); a mesh dim shards one letter only, the one that comes first in the
 * einsum string.
 */
int rtp_infer_spmd(const char* einsum, int n_in, const int32_t* const* in_dims_mappings, int mesh_ndim,
                   int32_t* out_dims_mapping, uint32_t* out_partial_mask, uint32_t* in_needs_reshard_mask,
                   int32_t* const* in_inferred);

/*
 * SBP-signature inference for an element-wise n-ary op (OneFlow page, the
 * add_n walk-through: candidate set, filters, sort by OrderValue then
 * CopyCost). Host only.
 *   n_in inputs of one logical shape [ndim] with element size elem_bytes;
 *   in_kinds / in_axes: [n_in * mesh_ndim], input j's ND-SBP (rtp_sbp kind
 *   and split axis per mesh dim; mesh_ndim = 1 is the 1D case)
 *   constraint_kinds / constraint_axes: [mesh_ndim] required ND-SBP of the
 *   signature, or NULL for none
 *   out_kinds / out_axes: [mesh_ndim] the chosen signature (every input and
 *   the output take it); out_cost: its CopyCost; out_order: its OrderValue
 * Candidates per mesh dim: split(i) for every axis i, partial-sum, broadcast
 * (in that order); on an ND mesh, every combination (mesh dim 0 varies
 * slowest). A candidate whose split axis is not an axis of the tensor is
 * dropped, and so is one that differs from the constraint.
 * OrderValue: -10 for every input already in the candidate's SBP (0 for all
 * candidates when a constraint is given). CopyCost, summed over inputs: 0 if
 * the input's SBP equals the candidate's; otherwise a huge number (1e30) if
 * the input is partial-sum or broadcast on some mesh dim, else the input's
 * bytes. The least (OrderValue, CopyCost) wins; ties keep candidate order.
 * Reading: "partial_sum and broadcast cost a huge number" refers to the input's
 * current SBP; the page's example (split + broadcast inputs infer broadcast)
 * only holds under that reading.
 */
int rtp_infer_sbp_signature(int n_in, int ndim, const int64_t* shape, int elem_bytes, int mesh_ndim,
                            const int32_t* in_kinds, const int32_t* in_axes, const int32_t* constraint_kinds,
                            const int32_t* constraint_axes, int32_t* out_kinds, int32_t* out_axes, double* out_cost,
                            int32_t* out_order);

/*
 * Reshape rule (Paddle note, DimTrans: InputDim, Flatten, Split, Singleton).
 * Host only. A split survives a reshape only on the leading (first non-unit)
 * member of a group of dims that map onto each other, and only if every
 * rank's contiguous run of that group is the same before and after; other
 * splits are dropped (in_after = the mapping the input must be resharded to).
 */
int rtp_infer_reshape(int in_ndim, const int64_t* in_shape, const int32_t* in_dims_mapping, int out_ndim,
                      const int64_t* out_shape, int mesh_ndim, const int64_t* mesh_shape, int32_t* in_after,
                      int32_t* out_dims_mapping);

/*
 * Sharding checker and output inference for broadcast n-ary element-wise
 * operators (Add, Mul, Sub, Where, ...): "ONNX multi-device proposal", sections
 * on the validity check and on operator groups. A device computes the output
 * elements whose inputs it holds; with broadcast axes a shard's devices are the
 * intersection of the devices of the input shards it reads (the page's
 * Add([M,1],[1,N]) example: output shard [i,j] lives where input-1 shard i and
 * input-2 shard j both are). Host only.
 *   in_ndims[k], in_shapes[k]  input k's rank and shape (extents >= 1); shapes
 *                              broadcast with trailing dims aligned (else
 *                              RTP_ESHAPE)
 *   in_specs[k]                input k's layout; all on the same number of
 *                              ranks, no partial mesh dims (RTP_EUNSUPPORTED:
 *                              the ONNX rules have no partial layouts)
 *   out_ndim, out_shape        the broadcast output shape (out_shape holds
 *                              RTP_MAX_NDIM entries)
 *   out_spec                   the output layout: an input's own spec when its
 *                              pieces are exactly the computable boxes, else
 *                              split mesh dims for the cut output axes (in axis
 *                              order, outer first) and one broadcast mesh dim for
 *                              replicas, ranks in ascending order within a piece
 * RTP_ECONFLICT: some output element has no rank holding all of its inputs
 * (e.g. one input split on axis 0 and the other on axis 1). RTP_EUNSUPPORTED:
 * the computable pieces are not a layout (overlapping, not a grid, held by
 * unequal numbers of ranks, a rank with nothing, or cuts other than the even
 * split).
 */
int rtp_infer_broadcast(int n_in, const int32_t* in_ndims, const int64_t* const* in_shapes, const rtp_spec* in_specs,
                        int* out_ndim, int64_t* out_shape, rtp_spec* out_spec);

/*
 * tp_mlp(X, A_shards, B_shards): the Megatron 1D tensor-parallel MLP on P
 * virtual ranks (ColossalAI "1D tensor parallelism" page, sections 2 and 2.1:
 * column-parallel Y_i = X A_i, row-parallel Z = sum_i Y_i B_i; GELU between
 * the GEMMs as in the Domino page's "GeMM GeLU GeMM").
 *   X         bf16 [M, K] device pointer
 *   A_shards  P bf16 [K, F/P] device pointers (column blocks of A)
 *   B_shards  P bf16 [F/P, N] device pointers (row blocks of B)
 *   Y         P bf16 [M, F/P] device pointers; receives Y_i = GELU(X A_i)
 *             (exact erf GELU on the float32 accumulator, rounded once)
 *   partials  P float32 [M, N] device pointers for mode 0 (receive Y_i B_i);
 *             may be NULL in mode 1
 *   Z         float32 [M, N] device pointer; receives sum_i Y_i B_i
 *   mode      0: row-parallel GEMM writes per-rank partials, a separate
 *             kernel sums them (the all-reduce); 1: the row-parallel GEMM
 *             walks all ranks' K ranges in one accumulator (fused reduction)
 *   chunks    1, 2 or 4: Domino row split of X (and Z) (DeepSpeed Domino page,
 *             row split of the input X); in mode 0 the sum of chunk c overlaps
 *             chunk c+1's GEMMs
 *   col_blocks 1 or 2: Domino column split of B_i (mode 0) (Domino page,
 *             column split of the weight B); the sum of column block 0
 *             overlaps the GEMM of block 1
 *   s0, s1    streams; all work is ordered after prior work on s0 and the
 *             call's completion is ordered on s0 (s1 is joined back)
 * Mode 0 sums the partials (the all-reduce) in one of two ways
 * (rtp_tp_mlp_overlap). By default every window (one chunk and one column
 * block) is summed by a kernel of its own after its row-parallel GEMM, on s1
 * beside the next window's GEMMs when s1 != s0 (the Domino schedule as the
 * page draws it). Otherwise the row-parallel GEMM's clusters take every
 * rank's tile of one output tile in turn, and the epilogue that writes rank
 * i's partial tile also adds it into Z (the reduction fused into the GEMM's
 * epilogue, beside the GEMM of the other tiles). Either way
 * Z = ((0 + p_0) + p_1) + ... in float32 in rank order, so Z is
 * bit-identical across chunks, column blocks and both ways.
 * Requirements (else RTP_ESHAPE, like the ValueError on out_features %
 * tp_size in ColossalAI's Linear1D_Col): F % P == 0, M % chunks == 0, K, F/P
 * and N / col_blocks multiples of 8 (16-byte rows); P <= 8 (else
 * RTP_EUNSUPPORTED); all pointers 16-byte aligned (else RTP_EINVAL).
 * M == 0 (no tokens) launches nothing; the buffers with M rows (X, Y,
 * partials, Z) may then be NULL.
 * Errors leave nothing launched. The kernels allocate nothing; the first call
 * on a device sets the GEMM kernel's shared-memory limit and, per host thread,
 * creates two events used to order s0 and s1. The GEMM kernels are launched
 * as programmatic dependents of the previous kernel in their stream: they may
 * start their set-up early but wait for that kernel to complete before they
 * touch global memory, so stream order is kept; a caller's own kernel launched
 * the same way after them must wait likewise (griddepcontrol.wait) before
 * reading their outputs.
 */
int rtp_tp_mlp(int P, int64_t M, int64_t K, int64_t F, int64_t N, const void* X, const void* const* A_shards,
               const void* const* B_shards, void* const* Y, void* const* partials, float* Z, int mode, int chunks,
               int col_blocks, rtp_stream s0, rtp_stream s1);

/*
 * The fused forward of rtp_tp_mlp (mode 1, one chunk) that also keeps what the
 * backward pass needs: H_i = X A_i, the pre-activation, rounded to bf16 (the
 * forward of the ColossalAI "1D tensor parallelism" page, sections 2 and 2.1,
 * keeping the input of the GELU for the backward of section 2.2).
 *   H         P bf16 [M, F/P] device pointers (caller-owned, 16-byte aligned)
 *   the rest  as in rtp_tp_mlp; Y_i = GELU of the float32 accumulator (not of
 *             the rounded H_i), so Y and Z are bit-identical to rtp_tp_mlp's
 * Same requirements and errors as rtp_tp_mlp; H NULL is RTP_EINVAL.
 */
int rtp_tp_mlp_train_forward(int P, int64_t M, int64_t K, int64_t F, int64_t N, const void* X,
                             const void* const* A_shards, const void* const* B_shards, void* const* Y, void* const* H,
                             float* Z, rtp_stream stream);

/*
 * Backward pass of the tensor-parallel MLP (ColossalAI "1D tensor
 * parallelism" page, section 2.2: each rank's column-parallel layer yields a
 * partial input gradient dY_i A_i^T and the full one is their all-reduced sum;
 * the row-parallel layer's input Y_i is already split the way its gradient is
 * needed, so dZ reaches every rank unchanged). Per rank i:
 *   dH_i = bf16( (dZ B_i^T) * GELU'(H_i) )     GELU'(h) = Phi(h) + h phi(h)
 *   dA_i = X^T dH_i         dB_i = Y_i^T dZ    dX = sum_i dH_i A_i^T
 *   X, A_shards, B_shards  as in rtp_tp_mlp (bf16 [M,K], [K,F/P], [F/P,N])
 *   H, Y      P bf16 [M, F/P]: what rtp_tp_mlp_train_forward kept
 *   dZ        bf16 [M, N]: gradient of the loss with respect to Z
 *   dH        P bf16 [M, F/P] device scratch (receives dH_i)
 *   dX_partials P float32 [M, K] device scratch for mode 0; may be NULL in mode 1
 *   dX        float32 [M, K]; dA: P float32 [K, F/P]; dB: P float32 [F/P, N]
 *   mode      1: the input-gradient GEMM walks all ranks' F/P ranges in one
 *             accumulator (the all-reduce fused); 0: it writes per-rank
 *             partials and their rank sum: by default a kernel of its own,
 *             on s1 beside the weight-gradient GEMMs on s0 when s1 != s0 (the
 *             DeepSpeed Domino page, backward: the all-reduce of the input
 *             gradient overlaps the same micro-batch's weight-gradient GEMMs);
 *             or in the dX GEMM's epilogue (rtp_tp_mlp_overlap)
 *   s0, s1    streams; the call's completion is ordered on s0
 * float32 accumulation of bf16 products throughout; GELU' is evaluated in
 * float32 on the bf16 H_i. Requirements: F % P == 0, K, F/P, N multiples of 8,
 * P <= 8, pointers 16-byte aligned (RTP_ESHAPE / RTP_EUNSUPPORTED /
 * RTP_EINVAL). M == 0 zeroes dA and dB. Errors leave nothing launched.
 */
int rtp_tp_mlp_backward(int P, int64_t M, int64_t K, int64_t F, int64_t N, const void* X, const void* const* A_shards,
                        const void* const* B_shards, const void* const* H, const void* const* Y, const void* dZ,
                        void* const* dH, void* const* dX_partials, float* dX, float* const* dA, float* const* dB,
                        int mode, rtp_stream s0, rtp_stream s1);

/*
 * Where mode 0 of rtp_tp_mlp and rtp_tp_mlp_backward sums the partials, for
 * later calls from the calling thread (no page counterpart: it chooses how
 * this library places the all-reduce on one GPU). sum_in_epilogue = 0 (the
 * default): in kernels of their own, on s1 beside the next GEMMs when a
 * second stream is given; 1: in the epilogue of the GEMM that writes them, as
 * each output tile's rank partials finish. Results are bit-identical.
 * *previous (if not NULL) receives the setting it replaces. RTP_EINVAL for a
 * value other than 0 or 1.
 */
int rtp_tp_mlp_overlap(int sum_in_epilogue, int* previous);

/*
 * The tensor-parallel MLP with sequence parallelism (ColossalAI "1D tensor
 * parallelism" page, section 5.3: with sequence parallelism the column-parallel
 * layer all-gathers its input in the forward pass and the row-parallel layer
 * reduce-scatters its output instead of all-reducing it).
 *   X_shards  P bf16 [M/P, K]: rank r holds rows [r M/P, (r+1) M/P) of X
 *   A_shards, B_shards, Y: as in rtp_tp_mlp (Y_i [M, F/P] covers all rows)
 *   Z_shards  P float32 [M/P, N]: rank r receives rows [r M/P, (r+1) M/P) of
 *             Z = sum_i GELU(X A_i) B_i
 * Both collectives are fused into the GEMMs: the column-parallel GEMM reads X
 * from the shards directly and the row-parallel GEMM sums the ranks in its
 * accumulator and writes each row to its shard. Requires M % P == 0 and
 * (M/P) % 128 == 0, K, F/P and N multiples of 8, P <= 8 (else RTP_ESHAPE /
 * RTP_EUNSUPPORTED); pointers 16-byte aligned. M == 0 launches nothing, and
 * X_shards, Y and Z_shards may then be NULL.
 */
int rtp_tp_mlp_sp(int P, int64_t M, int64_t K, int64_t F, int64_t N, const void* const* X_shards,
                  const void* const* A_shards, const void* const* B_shards, void* const* Y, float* const* Z_shards,
                  rtp_stream stream);

/*
 * tp_mlp for callers that cannot allocate device memory (code running inside
 * another runtime's memory pool, or a serving loop whose memory plan is fixed
 * at start-up). The pages have no counterpart to this call; it is a service
 * of this library.
 *   X, A_shards, B_shards, Z: as in rtp_tp_mlp (caller-owned, 16-byte aligned)
 *   stream: the stream that orders the work
 * Computes Z = sum_i GELU(X A_i) B_i with the reduction fused into the
 * row-parallel GEMM. The activations Y live in a static device array of the
 * library (16 MiB), so the call allocates nothing. It returns RTP_ESHAPE when
 * P * round_up(M * F/P * 2 bytes, 256) exceeds 16 MiB (about M * F <= 8 Mi
 * elements), and the other errors of rtp_tp_mlp.
 * The first call on a device finds the array's device address (with that
 * device current); make that first call before any stream capture. A device
 * reset (cudaDeviceReset) after that first call is not supported: the array
 * may then live at another address.
 * Every call uses the same array: calls that overlap on the GPU (on several
 * streams, or from several threads) race on it and must be ordered by the
 * caller.
 */
int rtp_tp_mlp_noalloc(int P, int64_t M, int64_t K, int64_t F, int64_t N, const void* X, const void* const* A_shards,
                       const void* const* B_shards, float* Z, rtp_stream stream);

/*
 * Reads and clears the device words in which the tensor-core kernels of
 * rtp_tp_mlp record a wait that gave up (no progress for about 4 seconds; the
 * kernel then stops, frees its tensor memory and returns instead of hanging),
 * and in which the resharding kernel records a bulk copy that never completed.
 * Synchronises `stream`. *code == 0: no such event since the last check;
 * otherwise the results of the launches since then are invalid
 * (1 producer, 2 MMA waiting for operands, 3 MMA waiting for an accumulator,
 * 4 epilogue, 5 rtp_wait_selftest; 16: a bulk copy of the resharding kernel
 * did not complete within about 2 seconds, so that launch stopped early).
 * The pages have no counterpart: this is the library's failure detection.
 */
int rtp_device_error(rtp_stream stream, uint32_t* code);

/*
 * Self-test of the bounded waits of this library's kernels (no page
 * counterpart: it checks failure detection without a fault). A wait on an
 * mbarrier that nothing completes gives up after limit_ns of %globaltimer and
 * records a code in the device word that rtp_device_error reads; the kernel
 * then returns normally and the context stays usable.
 *   kernel    0: the wait of rtp_tp_mlp's tensor-core kernel. One block, two
 *             waiting threads: the first gives up after limit_ns, records code
 *             5 and raises the block's abort flag; the second (own limit
 *             4 x limit_ns) leaves on that flag. out[w] = 1 when waiter w gave
 *             up (both, when the test works).
 *             1: the wait of the resharding kernel's staged copies. One block
 *             of 64 threads waits for 16 announced bytes that never arrive; the
 *             waits give up, record code 16 and the block stops: out[0] = 1.
 *   limit_ns  in [1e6, 1e9] (1 ms to 1 s), else RTP_EINVAL
 *   out       device pointer to 2 uint32 (16-byte aligned, caller-owned)
 * Asynchronous on `stream`.
 */
int rtp_wait_selftest(int kernel, unsigned long long limit_ns, uint32_t* out, rtp_stream stream);

/*
 * Fault injection for tests of the host-side checks (no page counterpart: it
 * exercises this library's own failure reporting without touching a GPU).
 * Arms a one-shot fault on the calling thread and clears that thread's cache of
 * reshard plans, so its next rtp_shard / rtp_reshard / rtp_reshard_cost /
 * rtp_reshard_forms plans afresh:
 *   RTP_HOOK_NONE        disarms;
 *   RTP_HOOK_PLAN_SHIFT  the next plan built has the first destination offset
 *                        of its first task moved by `arg` elements (a planted
 *                        planning mistake). Every new plan is checked against
 *                        both layouts' piece extents before use, so a shift that
 *                        leaves the piece returns RTP_EINVAL, nothing launched;
 *   RTP_HOOK_FAIL_ALLOC  the next planning step fails as if host memory ran
 *                        out: the call returns RTP_ENOMEM, nothing launched.
 * RTP_EINVAL for an unknown hook.
 */
enum { RTP_HOOK_NONE = 0, RTP_HOOK_PLAN_SHIFT = 1, RTP_HOOK_FAIL_ALLOC = 2 };
int rtp_test_hook(int hook, int64_t arg);

/*
 * Text of the last error on the calling thread ("" if none): the reason the
 * ONNX page's validity check asks an implementation to report.
 */
const char* rtp_last_error(void);

/* Library version string (no page counterpart). */
const char* rtp_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RTP_H_ */
