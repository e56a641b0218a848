"""Python binding of librtp (resharding and 1D tensor parallelism on a virtual
mesh inside one GB300).

Argument marshalling and buffer checks only: every step of the path runs in the library's CUDA
kernels. PyTorch supplies device memory and streams. Loading fails loudly if
the compiled library is missing; there is no fallback.

Names mirror the C ABI in ``include/rtp.h``:
  spec_from_dims_mapping, spec_from_onnx, spec_nd_sbp (the ND-SBP form filled
  directly), shard_shape, shard_box, shard, reshard, reshard_cost,
  infer_spmd, infer_reshape, tp_mlp, last_error.
"""
from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Sequence, Tuple, Union

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "librtp.so")

MAX_NDIM = 8
MAX_MESH_NDIM = 4
MAX_RANKS = 64
F32, BF16 = 0, 1
SPLIT, BROADCAST, PARTIAL, PARTIAL_MIN, PARTIAL_MAX = 0, 1, 2, 3, 4
STATUS = {0: "RTP_OK", -1: "RTP_EINVAL", -2: "RTP_ESHAPE", -3: "RTP_EUNSUPPORTED", -4: "RTP_ECONFLICT",
          -5: "RTP_ECUDA", -6: "RTP_ENOMEM"}


class RtpError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__("%s: %s" % (STATUS.get(status, status), message))
        self.status = status


class Spec(ctypes.Structure):
    """rtp_spec: the canonical (ND-SBP) layout of a tensor on a virtual mesh."""

    _fields_ = [
        ("mesh_ndim", ctypes.c_int32),
        ("mesh_shape", ctypes.c_int64 * MAX_MESH_NDIM),
        ("rank_ids", ctypes.c_int32 * MAX_RANKS),
        ("sbp_kind", ctypes.c_int32 * MAX_MESH_NDIM),
        ("sbp_axis", ctypes.c_int32 * MAX_MESH_NDIM),
    ]

    @property
    def num_ranks(self) -> int:
        n = 1
        for d in range(self.mesh_ndim):
            n *= self.mesh_shape[d]
        return n

    def describe(self):
        ents = []
        for d in range(self.mesh_ndim):
            k = self.sbp_kind[d]
            ents.append(("S", self.sbp_axis[d]) if k == SPLIT else
                        {BROADCAST: "B", PARTIAL: "P", PARTIAL_MIN: "Pmin", PARTIAL_MAX: "Pmax"}[k])
        mesh = tuple(self.mesh_shape[d] for d in range(self.mesh_ndim))
        return mesh, tuple(ents), tuple(self.rank_ids[p] for p in range(self.num_ranks))

    def __repr__(self):
        mesh, ents, ranks = self.describe()
        return "Spec(mesh=%s, sbp=%s, ranks=%s)" % (mesh, ents, ranks)


_lib = None


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError("librtp.so is not built (%s); run `python -c \"import __graft_entry__ as g; g.build()\"`"
                          % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER
    i64p, i32p, u32p, vp = P(ctypes.c_int64), P(ctypes.c_int32), P(ctypes.c_uint32), ctypes.c_void_p
    vpp = P(ctypes.c_void_p)
    c_int = ctypes.c_int
    sig = {
        "rtp_spec_from_dims_mapping": [c_int, i32p, c_int, i64p, i32p, ctypes.c_uint32, P(Spec)],
        "rtp_spec_from_onnx": [c_int, c_int, i64p, c_int, i64p, i32p, i64p, c_int, i64p, i64p, P(Spec)],
        "rtp_spec_check": [c_int, P(Spec)],
        "rtp_shard_shape": [c_int, i64p, P(Spec), c_int, i64p],
        "rtp_shard_box": [c_int, i64p, P(Spec), c_int, i64p, i64p, i32p],
        "rtp_shard": [c_int, c_int, i64p, vp, P(Spec), vpp, vp],
        "rtp_reshard": [c_int, c_int, i64p, vpp, P(Spec), vpp, P(Spec), vp],
        "rtp_reshard_cost": [c_int, c_int, i64p, P(Spec), P(Spec), i64p, i64p, i32p, i32p],
        "rtp_reshard_forms": [c_int, c_int, i64p, P(Spec), P(Spec), i32p],
        "rtp_infer_spmd": [ctypes.c_char_p, c_int, P(i32p), c_int, i32p, u32p, u32p, P(i32p)],
        "rtp_infer_reshape": [c_int, i64p, i32p, c_int, i64p, c_int, i64p, i32p, i32p],
        "rtp_infer_sbp_signature": [c_int, c_int, i64p, c_int, c_int, i32p, i32p, i32p, i32p, i32p, i32p,
                                    P(ctypes.c_double), i32p],
        "rtp_infer_broadcast": [c_int, i32p, P(i64p), P(Spec), P(c_int), i64p, P(Spec)],
        "rtp_device_error": [vp, u32p],
        "rtp_wait_selftest": [c_int, ctypes.c_ulonglong, vp, vp],
        "rtp_test_hook": [c_int, ctypes.c_int64],
        "rtp_tp_mlp_overlap": [c_int, P(c_int)],
        "rtp_tp_mlp_sp": [c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, vpp, vpp, vpp, vpp,
                          vpp, vp],
        "rtp_tp_mlp_noalloc": [c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, vp, vpp, vpp,
                               vp, vp],
        "rtp_tp_mlp": [c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, vp, vpp, vpp, vpp,
                       vpp, vp, c_int, c_int, c_int, vp, vp],
        "rtp_tp_mlp_train_forward": [c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, vp, vpp,
                                     vpp, vpp, vpp, vp, vp],
        "rtp_tp_mlp_backward": [c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, vp, vpp, vpp,
                                vpp, vpp, vp, vpp, vpp, vp, vpp, vpp, c_int, vp, vp],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = c_int
    lib.rtp_last_error.restype = ctypes.c_char_p
    lib.rtp_last_error.argtypes = []
    lib.rtp_version.restype = ctypes.c_char_p
    lib.rtp_version.argtypes = []
    _lib = lib
    return lib


def lib():
    """The loaded ctypes library (loads it on first use)."""
    return _load()


def last_error() -> str:
    return _load().rtp_last_error().decode()


def _check(rc: int) -> None:
    if rc != 0:
        raise RtpError(rc, last_error())


def _i64(xs) -> ctypes.Array:
    xs = [int(x) for x in xs]
    return (ctypes.c_int64 * max(1, len(xs)))(*xs)


def _i32(xs) -> ctypes.Array:
    xs = [int(x) for x in xs]
    return (ctypes.c_int32 * max(1, len(xs)))(*xs)


def _ptrs(ptrs) -> ctypes.Array:
    return (ctypes.c_void_p * max(1, len(ptrs)))(*[p if p else None for p in ptrs])


# ---- specs ------------------------------------------------------------------------

Entry = Union[str, Tuple[str, int]]


def spec_nd_sbp(mesh: Sequence[int], entries: Sequence[Entry], rank_ids: Sequence[int] = ()) -> Spec:
    """ND-SBP form: one entry per mesh dim, ("S", axis), "B", "P" (partial sum),
    "Pmin" or "Pmax" (partial min / max) (OneFlow page)."""
    s = Spec()
    s.mesh_ndim = len(mesh)
    n = 1
    for d, m in enumerate(mesh):
        s.mesh_shape[d] = int(m)
        n *= int(m)
    ranks = list(rank_ids) if rank_ids else list(range(n))
    if len(ranks) > MAX_RANKS:
        raise RtpError(-3, "more than %d ranks" % MAX_RANKS)
    for p, r in enumerate(ranks):
        s.rank_ids[p] = int(r)
    for d, e in enumerate(entries):
        if e == "B":
            s.sbp_kind[d], s.sbp_axis[d] = BROADCAST, -1
        elif e in ("P", "Pmin", "Pmax"):
            s.sbp_kind[d], s.sbp_axis[d] = {"P": PARTIAL, "Pmin": PARTIAL_MIN, "Pmax": PARTIAL_MAX}[e], -1
        else:
            s.sbp_kind[d], s.sbp_axis[d] = SPLIT, int(e[1])
    return s


def spec_from_dims_mapping(dims_mapping: Sequence[int], mesh: Sequence[int], rank_ids: Sequence[int] = (),
                           partial: Sequence[int] = ()) -> Spec:
    mask = 0
    for d in partial:
        mask |= 1 << int(d)
    out = Spec()
    _check(_load().rtp_spec_from_dims_mapping(len(dims_mapping), _i32(dims_mapping), len(mesh), _i64(mesh),
                                              _i32(rank_ids) if rank_ids else None, mask, ctypes.byref(out)))
    return out


def spec_from_onnx(ndim: int, device: Sequence[int], device_map: dict, sharded_dim: Sequence[Tuple[int, int]]
                   ) -> Spec:
    """device: ids or negative keys; device_map: {key: [ids]}; sharded_dim: [(axis, num_shards)]."""
    keys = list(device_map.keys())
    sizes = [len(device_map[k]) for k in keys]
    flat = [d for k in keys for d in device_map[k]]
    out = Spec()
    _check(_load().rtp_spec_from_onnx(ndim, len(device), _i64(device), len(keys), _i64(keys), _i32(sizes),
                                      _i64(flat), len(sharded_dim), _i64([a for a, _ in sharded_dim]),
                                      _i64([s for _, s in sharded_dim]), ctypes.byref(out)))
    return out


def spec_check(ndim: int, spec: Spec) -> None:
    _check(_load().rtp_spec_check(ndim, ctypes.byref(spec)))


def shard_shape(shape: Sequence[int], spec: Spec, rank: int) -> Tuple[int, ...]:
    out = _i64([0] * len(shape))
    _check(_load().rtp_shard_shape(len(shape), _i64(shape), ctypes.byref(spec), rank, out))
    return tuple(out[a] for a in range(len(shape)))


def shard_box(shape: Sequence[int], spec: Spec, rank: int):
    nd = len(shape)
    lo, hi, hv = _i64([0] * nd), _i64([0] * nd), ctypes.c_int32()
    _check(_load().rtp_shard_box(nd, _i64(shape), ctypes.byref(spec), rank, lo, hi, ctypes.byref(hv)))
    return tuple(lo[a] for a in range(nd)), tuple(hi[a] for a in range(nd)), bool(hv.value)


# ---- data movement ----------------------------------------------------------------

def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError("rtp tensors are float32 or bfloat16, got %s" % t.dtype)


def _stream_ptr(stream) -> Optional[int]:
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return stream or None
    return stream.cuda_stream or None


_PIECE_SHAPES: dict = {}


def piece_shapes(shape: Sequence[int], spec: Spec) -> List[Tuple[int, ...]]:
    """shard_shape of every rank, cached per (shape, spec)."""
    key = (tuple(shape), bytes(spec))
    got = _PIECE_SHAPES.get(key)
    if got is None:
        got = [shard_shape(shape, spec, r) for r in range(spec.num_ranks)]
        if len(_PIECE_SHAPES) > 4096:
            _PIECE_SHAPES.clear()
        _PIECE_SHAPES[key] = got
    return got


def _alloc_pieces(shapes, like, out):
    torch = _torch()
    if out is not None:
        return list(out)
    return [torch.empty(s, dtype=like.dtype, device=like.device) for s in shapes]


def _check_cuda(ts, what):
    for t in ts:
        if t is not None and t.numel() > 0:
            if not t.is_cuda:
                raise RtpError(-1, "%s: tensors must live on the GPU" % what)
            if not t.is_contiguous():
                raise RtpError(-1, "%s: tensors must be contiguous (row-major)" % what)


def _check_buffers(what, device: int, groups):
    """The library gets raw pointers and cannot see buffer sizes, so every
    buffer is checked here against the shape and dtype the call will read or
    write: a wrong buffer raises instead of reaching the GPU. device: the CUDA
    device index the call runs on. groups: (name, tensors, shape, dtype), shape
    one tuple for all the tensors or a list of one tuple per tensor (which also
    fixes their count)."""
    for name, ts, shape, dtype in groups:
        per = isinstance(shape, list)
        if per and len(ts) != len(shape):
            raise RtpError(-1, "%s: %d %s buffers given, %d expected" % (what, len(ts), name, len(shape)))
        for i, t in enumerate(ts):
            s = shape[i] if per else shape
            if t.dtype is not dtype or t.shape != s or not t.is_contiguous() or t.get_device() != device:
                _buffer_error(what, name, i, t, s, dtype, device)


def _buffer_error(what, name, i, t, shape, dtype, device):
    if t.dtype is not dtype or tuple(t.shape) != tuple(shape):
        raise RtpError(-2, "%s: %s[%d] is %s %s, expected %s %s" % (
            what, name, i, t.dtype, tuple(t.shape), dtype, tuple(shape)))
    if t.numel() == 0:
        return  # an empty piece is never touched, wherever it lives
    if not t.is_contiguous():
        raise RtpError(-1, "%s: %s[%d] must be contiguous (row-major)" % (what, name, i))
    raise RtpError(-1, "%s: %s[%d] is on %s, the call runs on device %d" % (what, name, i, t.device, device))


def _device_of(t) -> int:
    """Index of the current CUDA device, which must hold `t`."""
    torch = _torch()
    if not t.is_cuda:
        raise RtpError(-1, "tensors must live on the GPU")
    if t.get_device() != torch.cuda.current_device():
        raise RtpError(-1, "tensors are on %s but the current CUDA device is %d" % (t.device,
                                                                                  torch.cuda.current_device()))
    return t.get_device()


def shard(full, spec: Spec, out=None, stream=None):
    """Rank pieces of the logical tensor `full` (a CUDA tensor) under `spec`."""
    shape = tuple(full.shape)
    shapes = piece_shapes(shape, spec)
    code = _dtype_code(full)
    pieces = _alloc_pieces(shapes, full, out)
    _check_buffers("shard", _device_of(full), [("full", [full], shape, full.dtype),
                                               ("out", pieces, shapes, full.dtype)])
    _check(_load().rtp_shard(code, len(shape), _i64(shape), full.data_ptr(), ctypes.byref(spec),
                             _ptrs([p.data_ptr() for p in pieces]), _stream_ptr(stream)))
    return pieces


def reshard(pieces, shape: Sequence[int], src: Spec, dst: Spec, out=None, stream=None):
    """Pieces laid out by `dst`, from `pieces` laid out by `src`."""
    shape = tuple(int(s) for s in shape)
    like = pieces[0]
    dshapes = piece_shapes(shape, dst)
    code = _dtype_code(like)
    outs = _alloc_pieces(dshapes, like, out)
    _check_buffers("reshard", _device_of(like), [("pieces", pieces, piece_shapes(shape, src), like.dtype),
                                                 ("out", outs, dshapes, like.dtype)])
    _check(_load().rtp_reshard(code, len(shape), _i64(shape), _ptrs([p.data_ptr() for p in pieces]),
                               ctypes.byref(src), _ptrs([o.data_ptr() for o in outs]), ctypes.byref(dst),
                               _stream_ptr(stream)))
    return outs


def reshard_forms(dtype_code: int, shape: Sequence[int], src: Spec, dst: Spec):
    """Tasks per kernel form a reshard would use: (registers, bulk staging,
    TMA tiles 3D, TMA tiles 4D), for 256-byte aligned buffers."""
    c = (ctypes.c_int32 * 4)()
    _check(_load().rtp_reshard_forms(dtype_code, len(shape), _i64(shape), ctypes.byref(src), ctypes.byref(dst), c))
    return tuple(c)


def reshard_cost(dtype_code: int, shape: Sequence[int], src: Spec, dst: Spec):
    """(bytes_read, bytes_written, n_tasks, n_launches) planned for a reshard."""
    rd, wr, nt, nl = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int32(), ctypes.c_int32()
    _check(_load().rtp_reshard_cost(dtype_code, len(shape), _i64(shape), ctypes.byref(src), ctypes.byref(dst),
                                    ctypes.byref(rd), ctypes.byref(wr), ctypes.byref(nt), ctypes.byref(nl)))
    return rd.value, wr.value, nt.value, nl.value


# ---- inference --------------------------------------------------------------------

def infer_spmd(einsum: str, dims_mappings: Sequence[Sequence[int]], mesh_ndim: int):
    """(out_dims_mapping, partial_mesh_dims, inputs_needing_reshard, inferred_input_mappings)."""
    lhs, rhs = einsum.split("->") if "->" in einsum else (einsum, "")
    ins = lhs.split(",")
    P = ctypes.POINTER(ctypes.c_int32)
    arrs = [_i32(dm) for dm in dims_mappings]
    merged = [_i32([0] * max(1, len(t))) for t in ins]
    inp = (P * max(1, len(arrs)))(*[ctypes.cast(a, P) for a in arrs])
    mp = (P * max(1, len(merged)))(*[ctypes.cast(a, P) for a in merged])
    out = _i32([0] * max(1, len(rhs)))
    pm, rm = ctypes.c_uint32(), ctypes.c_uint32()
    _check(_load().rtp_infer_spmd(einsum.encode(), len(dims_mappings), inp, mesh_ndim, out, ctypes.byref(pm),
                                  ctypes.byref(rm), mp))
    return ([out[i] for i in range(len(rhs))], [d for d in range(32) if (pm.value >> d) & 1],
            [j for j in range(len(ins)) if (rm.value >> j) & 1],
            [[merged[j][i] for i in range(len(ins[j]))] for j in range(len(ins))])


def infer_reshape(in_shape, in_dims_mapping, out_shape, mesh):
    """(in_dims_after, out_dims_mapping) for a reshape."""
    ni, no = len(in_shape), len(out_shape)
    after, outm = _i32([0] * ni), _i32([0] * no)
    _check(_load().rtp_infer_reshape(ni, _i64(in_shape), _i32(in_dims_mapping), no, _i64(out_shape), len(mesh),
                                     _i64(mesh), after, outm))
    return [after[i] for i in range(ni)], [outm[o] for o in range(no)]


def _sbp_entry(e):
    if e == "B":
        return BROADCAST, -1
    if e in ("P", "Pmin", "Pmax"):
        return {"P": PARTIAL, "Pmin": PARTIAL_MIN, "Pmax": PARTIAL_MAX}[e], -1
    return SPLIT, int(e[1])


def infer_sbp_signature(shape, elem_bytes, inputs, constraint=None):
    """OneFlow-style SBP signature of an element-wise op. inputs: per input its
    ND-SBP (entries ("S", axis) / "B" / "P" per mesh dim). Returns
    (signature entries, CopyCost, OrderValue)."""
    md = len(inputs[0])
    kinds, axes = [], []
    for sbp in inputs:
        for e in sbp:
            k, a = _sbp_entry(e)
            kinds.append(k)
            axes.append(a)
    ck = ca = None
    if constraint is not None:
        c = [_sbp_entry(e) for e in constraint]
        ck, ca = _i32([k for k, _ in c]), _i32([a for _, a in c])
    okind, oaxis = _i32([0] * md), _i32([0] * md)
    cost, order = ctypes.c_double(), ctypes.c_int32()
    _check(_load().rtp_infer_sbp_signature(len(inputs), len(shape), _i64(shape), elem_bytes, md, _i32(kinds),
                                           _i32(axes), ck, ca, okind, oaxis, ctypes.byref(cost), ctypes.byref(order)))
    sig = []
    for d in range(md):
        k = okind[d]
        sig.append(("S", oaxis[d]) if k == SPLIT else {BROADCAST: "B", PARTIAL: "P"}[k])
    return sig, cost.value, order.value


def infer_broadcast(shapes, specs):
    """ONNX broadcast n-ary element-wise rule: (output shape, output Spec) for
    inputs of the given shapes and layouts; RtpError -4 when the inputs are
    sharded incompatibly."""
    n = len(shapes)
    nds = (ctypes.c_int32 * n)(*[len(sh) for sh in shapes])
    arrs = [_i64(sh) for sh in shapes]
    shp = (ctypes.POINTER(ctypes.c_int64) * n)(*[ctypes.cast(a, ctypes.POINTER(ctypes.c_int64)) for a in arrs])
    sp = (Spec * n)(*specs)
    out_nd, oshape, out = ctypes.c_int(), _i64([0] * 8), Spec()
    _check(_load().rtp_infer_broadcast(n, nds, shp, sp, ctypes.byref(out_nd), oshape, ctypes.byref(out)))
    return tuple(oshape[d] for d in range(out_nd.value)), out


# ---- tensor-parallel MLP ------------------------------------------------------------

def tp_mlp(X, A_shards, B_shards, Y=None, partials=None, Z=None, mode: int = 1, chunks: int = 1,
           col_blocks: int = 1, s0=None, s1=None):
    """Z = sum_i GELU(X A_i) B_i on P = len(A_shards) virtual ranks (bf16 in, float32 Z).
    Returns (Z, Y). Buffers not given are allocated with torch."""
    torch = _torch()
    P = len(A_shards)
    M, K = X.shape
    Fp = A_shards[0].shape[1]
    N = B_shards[0].shape[1]
    F = Fp * P
    dev = X.device
    if Y is None:
        Y = [torch.empty((M, Fp), dtype=torch.bfloat16, device=dev) for _ in range(P)]
    if Z is None:
        Z = torch.empty((M, N), dtype=torch.float32, device=dev)
    if mode == 0 and partials is None:
        partials = [torch.empty((M, N), dtype=torch.float32, device=dev) for _ in range(P)]
    bf16, f32 = torch.bfloat16, torch.float32
    _check_buffers("tp_mlp", _device_of(X), [
        ("X", [X], (M, K), bf16), ("A_shards", A_shards, (K, Fp), bf16), ("B_shards", B_shards, [(Fp, N)] * P, bf16),
        ("Y", Y, [(M, Fp)] * P, bf16), ("partials", partials or [], [(M, N)] * (P if partials is not None else 0), f32),
        ("Z", [Z], (M, N), f32)])
    if s0 is None:
        s0 = torch.cuda.current_stream()
    if s1 is None:
        s1 = s0
    pp = _ptrs([p.data_ptr() for p in partials]) if partials is not None else None
    _check(_load().rtp_tp_mlp(P, M, K, F, N, X.data_ptr(), _ptrs([a.data_ptr() for a in A_shards]),
                              _ptrs([b.data_ptr() for b in B_shards]), _ptrs([y.data_ptr() for y in Y]), pp,
                              Z.data_ptr(), mode, chunks, col_blocks, _stream_ptr(s0), _stream_ptr(s1)))
    return Z, Y


def tp_mlp_overlap(sum_in_epilogue: int) -> int:
    """Where mode 0 sums the rank partials, for later calls from this thread:
    0 (the default) in kernels of their own (on s1 beside the next GEMMs when
    given), 1 in the epilogue of the GEMM that writes them. Returns the
    previous setting."""
    prev = ctypes.c_int()
    _check(_load().rtp_tp_mlp_overlap(int(sum_in_epilogue), ctypes.byref(prev)))
    return prev.value


def tp_mlp_train_forward(X, A_shards, B_shards, Y=None, H=None, Z=None, stream=None):
    """The fused forward that also keeps the bf16 pre-activations H_i = X A_i
    for the backward pass. Returns (Z, Y, H)."""
    torch = _torch()
    P = len(A_shards)
    M, K = X.shape
    Fp = A_shards[0].shape[1]
    N = B_shards[0].shape[1]
    dev = X.device
    if Y is None:
        Y = [torch.empty((M, Fp), dtype=torch.bfloat16, device=dev) for _ in range(P)]
    if H is None:
        H = [torch.empty((M, Fp), dtype=torch.bfloat16, device=dev) for _ in range(P)]
    if Z is None:
        Z = torch.empty((M, N), dtype=torch.float32, device=dev)
    bf16, f32 = torch.bfloat16, torch.float32
    _check_buffers("tp_mlp_train_forward", _device_of(X), [
        ("X", [X], (M, K), bf16), ("A_shards", A_shards, (K, Fp), bf16), ("B_shards", B_shards, [(Fp, N)] * P, bf16),
        ("Y", Y, [(M, Fp)] * P, bf16), ("H", H, [(M, Fp)] * P, bf16), ("Z", [Z], (M, N), f32)])
    _check(_load().rtp_tp_mlp_train_forward(P, M, K, Fp * P, N, X.data_ptr(), _ptrs([a.data_ptr() for a in A_shards]),
                                            _ptrs([b.data_ptr() for b in B_shards]), _ptrs([y.data_ptr() for y in Y]),
                                            _ptrs([h.data_ptr() for h in H]), Z.data_ptr(), _stream_ptr(stream)))
    return Z, Y, H


def tp_mlp_backward(X, A_shards, B_shards, H, Y, dZ, dH=None, dX_partials=None, dX=None, dA=None, dB=None,
                    mode: int = 1, s0=None, s1=None):
    """Gradients of Z = sum_i GELU(X A_i) B_i given dZ (bf16 [M, N]):
    returns (dX, dA, dB, dH) with dX float32 [M, K], dA[i] float32 [K, F/P],
    dB[i] float32 [F/P, N] and dH[i] = bf16(dZ B_i^T * GELU'(H_i))."""
    torch = _torch()
    P = len(A_shards)
    M, K = X.shape
    Fp = A_shards[0].shape[1]
    N = B_shards[0].shape[1]
    dev = X.device
    f32, bf16 = torch.float32, torch.bfloat16
    if dH is None:
        dH = [torch.empty((M, Fp), dtype=bf16, device=dev) for _ in range(P)]
    if dX is None:
        dX = torch.empty((M, K), dtype=f32, device=dev)
    if dA is None:
        dA = [torch.empty((K, Fp), dtype=f32, device=dev) for _ in range(P)]
    if dB is None:
        dB = [torch.empty((Fp, N), dtype=f32, device=dev) for _ in range(P)]
    if mode == 0 and dX_partials is None:
        dX_partials = [torch.empty((M, K), dtype=f32, device=dev) for _ in range(P)]
    nparts = P if dX_partials is not None else 0
    _check_buffers("tp_mlp_backward", _device_of(X), [
        ("X", [X], (M, K), bf16), ("A_shards", A_shards, (K, Fp), bf16), ("B_shards", B_shards, [(Fp, N)] * P, bf16),
        ("H", H, [(M, Fp)] * P, bf16), ("Y", Y, [(M, Fp)] * P, bf16), ("dZ", [dZ], (M, N), bf16),
        ("dH", dH, [(M, Fp)] * P, bf16), ("dX_partials", dX_partials or [], [(M, K)] * nparts, f32),
        ("dX", [dX], (M, K), f32), ("dA", dA, [(K, Fp)] * P, f32), ("dB", dB, [(Fp, N)] * P, f32)])
    if s0 is None:
        s0 = torch.cuda.current_stream()
    if s1 is None:
        s1 = s0
    ptrs = lambda ts: _ptrs([t.data_ptr() for t in ts])
    pp = ptrs(dX_partials) if dX_partials is not None else None
    _check(_load().rtp_tp_mlp_backward(P, M, K, Fp * P, N, X.data_ptr(), ptrs(A_shards), ptrs(B_shards), ptrs(H),
                                       ptrs(Y), dZ.data_ptr(), ptrs(dH), pp, dX.data_ptr(), ptrs(dA), ptrs(dB), mode,
                                       _stream_ptr(s0), _stream_ptr(s1)))
    return dX, dA, dB, dH


def tp_mlp_sp(X_shards, A_shards, B_shards, Y=None, Z_shards=None, stream=None):
    """Sequence-parallel TP-MLP: X_shards[r] holds rows r*M/P.. of X; returns
    (Z_shards, Y) with Z_shards[r] the same rows of sum_i GELU(X A_i) B_i."""
    torch = _torch()
    P = len(A_shards)
    Mr, K = X_shards[0].shape
    M = Mr * P
    Fp = A_shards[0].shape[1]
    N = B_shards[0].shape[1]
    dev = X_shards[0].device
    if Y is None:
        Y = [torch.empty((M, Fp), dtype=torch.bfloat16, device=dev) for _ in range(P)]
    if Z_shards is None:
        Z_shards = [torch.empty((Mr, N), dtype=torch.float32, device=dev) for _ in range(P)]
    bf16, f32 = torch.bfloat16, torch.float32
    _check_buffers("tp_mlp_sp", _device_of(X_shards[0]), [
        ("X_shards", X_shards, [(Mr, K)] * P, bf16), ("A_shards", A_shards, (K, Fp), bf16),
        ("B_shards", B_shards, [(Fp, N)] * P, bf16), ("Y", Y, [(M, Fp)] * P, bf16),
        ("Z_shards", Z_shards, [(Mr, N)] * P, f32)])
    _check(_load().rtp_tp_mlp_sp(P, M, K, Fp * P, N, _ptrs([x.data_ptr() for x in X_shards]),
                                 _ptrs([a.data_ptr() for a in A_shards]), _ptrs([b.data_ptr() for b in B_shards]),
                                 _ptrs([y.data_ptr() for y in Y]), _ptrs([z.data_ptr() for z in Z_shards]),
                                 _stream_ptr(stream)))
    return Z_shards, Y


def tp_mlp_noalloc(X, A_shards, B_shards, Z=None, stream=None):
    """Z = sum_i GELU(X A_i) B_i with the activations in the library's static
    device scratch (for callers that cannot allocate). Returns Z.

    Every call shares that one static array (16 MiB per device): calls that
    overlap on the GPU, on several streams or from several threads, race on it
    and must be ordered by the caller. The first call on a device finds the
    array's address; make it before any stream capture, and do not reset the
    device after it."""
    torch = _torch()
    P = len(A_shards)
    M, K = X.shape
    Fp = A_shards[0].shape[1]
    N = B_shards[0].shape[1]
    if Z is None:
        Z = torch.empty((M, N), dtype=torch.float32, device=X.device)
    bf16 = torch.bfloat16
    _check_buffers("tp_mlp_noalloc", _device_of(X), [
        ("X", [X], (M, K), bf16), ("A_shards", A_shards, (K, Fp), bf16), ("B_shards", B_shards, [(Fp, N)] * P, bf16),
        ("Z", [Z], (M, N), torch.float32)])
    _check(_load().rtp_tp_mlp_noalloc(P, M, K, Fp * P, N, X.data_ptr(), _ptrs([a.data_ptr() for a in A_shards]),
                                      _ptrs([b.data_ptr() for b in B_shards]), Z.data_ptr(), _stream_ptr(stream)))
    return Z


def device_error(stream=None) -> int:
    """Reads and clears the device word set when a tensor-core kernel's bounded wait gave up."""
    code = ctypes.c_uint32()
    _check(_load().rtp_device_error(_stream_ptr(stream), ctypes.byref(code)))
    return code.value


def wait_selftest(limit_ns: int, out=None, stream=None, kernel: int = 0):
    """Runs a bounded-wait self-test kernel (a wait on a barrier that nothing
    completes, given up after limit_ns): kernel 0 the tensor-core kernel's
    wait, 1 the resharding kernel's. Returns the uint32 device tensor of
    outcomes (1 = that waiter gave up)."""
    torch = _torch()
    if out is None:
        out = torch.zeros(4, dtype=torch.int32, device="cuda")
    if out.numel() < 2 or out.element_size() != 4 or out.dtype.is_floating_point:
        raise RtpError(-1, "wait_selftest: out must hold at least 2 int32 values")
    _check_cuda([out], "wait_selftest")
    _check(_load().rtp_wait_selftest(int(kernel), int(limit_ns), out.data_ptr(), _stream_ptr(stream)))
    return out


HOOK_NONE, HOOK_PLAN_SHIFT, HOOK_FAIL_ALLOC = 0, 1, 2


def test_hook(hook: int, arg: int = 0) -> None:
    """Arms a one-shot host-side fault for this thread's next reshard plan
    (rtp_test_hook): HOOK_PLAN_SHIFT moves a planned destination offset by
    `arg` elements, HOOK_FAIL_ALLOC fails the planner's next allocation."""
    _check(_load().rtp_test_hook(int(hook), int(arg)))


def version() -> str:
    return _load().rtp_version().decode()
