"""CPU oracle for the resharding library (test infrastructure only).

A plain, slow, single-threaded C++ statement of what the library computes
(``oracle.cpp``), with this ctypes wrapper. Only ``tests/``, the smoke check in
``__graft_entry__`` and the benchmark's CPU-baseline leg may import it. It
shares no code with the CUDA library; the only common dependency is the
seeded input generator in ``synth``.

Layouts are passed in the ND-SBP form: a mesh shape, a row-major list of
device ids on the mesh, and per mesh dim one of ``("S", axis)``, ``"B"``,
``"P"`` (partial sum), ``"Pmin"`` or ``"Pmax"`` (partial min / max). ``layout_from_dims_mapping`` and ``layout_from_onnx`` turn the Paddle
and ONNX descriptions into that form.

Parity status: every function here is pinned by tests in
``tests/test_oracle_pins.py`` against values printed on the pages, closed
forms, invariants or brute force (nothing is "parity unpinned").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field
from typing import List, Sequence, Tuple, Union

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB = os.path.join(_HERE, "_oracle.so")
_lib = None

MAX_MESH = 8
MAX_DEV = 256
F32, BF16 = 0, 1


class _Layout(ctypes.Structure):
    _fields_ = [
        ("mesh_ndim", ctypes.c_int32),
        ("mesh_shape", ctypes.c_int64 * MAX_MESH),
        ("devices", ctypes.c_int32 * MAX_DEV),
        ("kind", ctypes.c_int8 * MAX_MESH),
        ("axis", ctypes.c_int32 * MAX_MESH),
    ]


Entry = Union[str, Tuple[str, int]]


@dataclass
class Layout:
    """ND-SBP layout: mesh shape, device ids (row-major), one entry per mesh dim."""

    mesh: Tuple[int, ...]
    entries: Tuple[Entry, ...]
    devices: Tuple[int, ...] = field(default=())

    def __post_init__(self):
        self.mesh = tuple(int(m) for m in self.mesh)
        self.entries = tuple(self.entries)
        if not self.devices:
            self.devices = tuple(range(int(np.prod(self.mesh))))
        self.devices = tuple(int(d) for d in self.devices)

    @property
    def num_devices(self) -> int:
        return int(np.prod(self.mesh))

    def _c(self) -> _Layout:
        L = _Layout()
        L.mesh_ndim = len(self.mesh)
        for d, m in enumerate(self.mesh):
            L.mesh_shape[d] = m
        for p, dev in enumerate(self.devices):
            L.devices[p] = dev
        for d, e in enumerate(self.entries):
            if e == "B":
                L.kind[d], L.axis[d] = ord("B"), -1
            elif e in ("P", "Pmin", "Pmax"):
                L.kind[d], L.axis[d] = ord({"P": "P", "Pmin": "N", "Pmax": "X"}[e]), -1
            else:
                L.kind[d], L.axis[d] = ord("S"), int(e[1])
        return L

    @staticmethod
    def _from_c(L: _Layout) -> "Layout":
        mesh = tuple(L.mesh_shape[d] for d in range(L.mesh_ndim))
        entries = []
        for d in range(L.mesh_ndim):
            k = chr(L.kind[d])
            entries.append(("S", L.axis[d]) if k == "S" else {"N": "Pmin", "X": "Pmax"}.get(k, k))
        n = int(np.prod(mesh))
        return Layout(mesh, tuple(entries), tuple(L.devices[p] for p in range(n)))


def build(force: bool = False) -> str:
    """Compile the oracle (building the checker is not running it)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", _SRC, "-o", tmp])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P = ctypes.POINTER
    i64p, i32p, u32p, dblp = P(ctypes.c_int64), P(ctypes.c_int32), P(ctypes.c_uint32), P(ctypes.c_double)
    vpp = P(ctypes.c_void_p)
    lib.oracle_shard_box.argtypes = [ctypes.c_int, i64p, P(_Layout), ctypes.c_int, i64p, i64p, i32p]
    lib.oracle_shard.argtypes = [ctypes.c_int, ctypes.c_int, i64p, ctypes.c_void_p, P(_Layout), vpp]
    lib.oracle_gather.argtypes = [ctypes.c_int, ctypes.c_int, i64p, vpp, P(_Layout), dblp]
    lib.oracle_reshard.argtypes = [ctypes.c_int, ctypes.c_int, i64p, vpp, P(_Layout), vpp, P(_Layout)]
    lib.oracle_layout_from_dims_mapping.argtypes = [ctypes.c_int, i32p, ctypes.c_int, i64p, i32p,
                                                    ctypes.c_uint32, P(_Layout)]
    lib.oracle_layout_from_onnx.argtypes = [ctypes.c_int, ctypes.c_int, i64p, ctypes.c_int, i64p, i32p, i64p,
                                            ctypes.c_int, i64p, i64p, P(_Layout)]
    lib.oracle_infer_spmd.argtypes = [ctypes.c_char_p, ctypes.c_int, P(i32p), ctypes.c_int, i32p, u32p, u32p,
                                      P(i32p)]
    lib.oracle_reshape_spmd.argtypes = [ctypes.c_int, i64p, i32p, ctypes.c_int, i64p, ctypes.c_int, i64p, i32p,
                                        i32p, i32p, i32p, i32p, i32p, i32p]
    i8p = P(ctypes.c_int8)
    lib.oracle_infer_sbp_signature.argtypes = [ctypes.c_int, ctypes.c_int, i64p, ctypes.c_int, ctypes.c_int, i8p,
                                               i32p, i8p, i32p, i8p, i32p, dblp, i32p, i32p]
    lib.oracle_infer_sbp_signature.restype = ctypes.c_int
    lib.oracle_bf16_round.argtypes = [ctypes.c_double]
    lib.oracle_bf16_round.restype = ctypes.c_uint16
    lib.oracle_gelu.argtypes = [ctypes.c_double]
    lib.oracle_gelu.restype = ctypes.c_double
    lib.oracle_tp_mlp.argtypes = [ctypes.c_int64] * 5 + [P(ctypes.c_uint16), vpp, vpp, ctypes.c_int, ctypes.c_int,
                                                         ctypes.c_int64, i64p, dblp, dblp]
    lib.oracle_gelu_grad.argtypes = [ctypes.c_double]
    lib.oracle_gelu_grad.restype = ctypes.c_double
    lib.oracle_tp_mlp_backward.argtypes = ([ctypes.c_int64] * 5 + [P(ctypes.c_uint16), vpp, vpp, P(ctypes.c_uint16),
                                           ctypes.c_int, ctypes.c_int64, i64p, dblp, dblp, dblp, dblp,
                                           ctypes.c_int64, i64p, dblp, dblp])
    lib.oracle_infer_broadcast.argtypes = [ctypes.c_int, i32p, P(i64p), P(_Layout), P(ctypes.c_int), i64p, i64p, i64p,
                                           P(_Layout), P(ctypes.c_int)]
    for f in ("oracle_infer_broadcast", "oracle_shard_box", "oracle_shard", "oracle_gather", "oracle_reshard",
              "oracle_layout_from_dims_mapping", "oracle_layout_from_onnx", "oracle_infer_spmd",
              "oracle_reshape_spmd", "oracle_tp_mlp", "oracle_tp_mlp_backward"):
        getattr(lib, f).restype = ctypes.c_int
    _lib = lib
    return lib


def _i64(xs) -> ctypes.Array:
    xs = list(xs)
    return (ctypes.c_int64 * max(1, len(xs)))(*xs)


def _i32(xs) -> ctypes.Array:
    xs = list(xs)
    return (ctypes.c_int32 * max(1, len(xs)))(*xs)


def _dtype_code(arr: np.ndarray) -> int:
    if arr.dtype == np.float32:
        return F32
    if arr.dtype == np.uint16:
        return BF16
    raise TypeError("oracle tensors are float32 or bf16 bit patterns (uint16)")


class OracleError(RuntimeError):
    pass


def _ok(rc: int, what: str) -> None:
    if rc != 0:
        raise OracleError("%s rejected its arguments" % what)


# ---- layouts ------------------------------------------------------------------

def layout_from_dims_mapping(dims_mapping: Sequence[int], mesh: Sequence[int], devices: Sequence[int] = (),
                             partial: Sequence[int] = ()) -> Layout:
    mesh = list(mesh)
    n = int(np.prod(mesh))
    devs = list(devices) if devices else list(range(n))
    mask = 0
    for d in partial:
        mask |= 1 << d
    out = _Layout()
    _ok(_load().oracle_layout_from_dims_mapping(len(dims_mapping), _i32(dims_mapping), len(mesh), _i64(mesh),
                                                _i32(devs), mask, ctypes.byref(out)), "layout_from_dims_mapping")
    return Layout._from_c(out)


def layout_from_onnx(ndim: int, device: Sequence[int], device_map: dict, sharded_dim: Sequence[Tuple[int, int]]
                     ) -> Layout:
    """device: ids or negative keys; device_map: {key: [ids]}; sharded_dim: [(axis, num_shards)]."""
    keys = list(device_map.keys())
    sizes = [len(device_map[k]) for k in keys]
    flat = [d for k in keys for d in device_map[k]]
    out = _Layout()
    _ok(_load().oracle_layout_from_onnx(ndim, len(device), _i64(device), len(keys), _i64(keys), _i32(sizes),
                                        _i64(flat), len(sharded_dim), _i64([a for a, _ in sharded_dim]),
                                        _i64([s for _, s in sharded_dim]), ctypes.byref(out)), "layout_from_onnx")
    return Layout._from_c(out)


def shard_box(shape: Sequence[int], layout: Layout, device: int):
    """(lo, hi, holds_value) of the piece held by `device`."""
    nd = len(shape)
    lo, hi, hv = _i64([0] * nd), _i64([0] * nd), ctypes.c_int32()
    L = layout._c()
    _ok(_load().oracle_shard_box(nd, _i64(shape), ctypes.byref(L), device, lo, hi, ctypes.byref(hv)), "shard_box")
    return tuple(lo[a] for a in range(nd)), tuple(hi[a] for a in range(nd)), bool(hv.value)


def infer_broadcast(shapes: Sequence[Sequence[int]], layouts: Sequence[Layout]):
    """ONNX broadcast n-ary element-wise rule, per element. Returns
    (status, out_shape, boxes, layout): status 0 = a layout (boxes[dev] =
    (lo, hi) of the output each device computes), 1 = some output element has
    no device, 2 = the pieces are not a layout."""
    n = len(shapes)
    nds = (ctypes.c_int32 * n)(*[len(sh) for sh in shapes])
    arrs = [_i64(sh) for sh in shapes]
    shp = (ctypes.POINTER(ctypes.c_int64) * n)(*[ctypes.cast(a, ctypes.POINTER(ctypes.c_int64)) for a in arrs])
    Ls = (_Layout * n)(*[L._c() for L in layouts])
    ndev = layouts[0].num_devices
    out_nd, st = ctypes.c_int(), ctypes.c_int()
    oshape = _i64([0] * 8)
    lo, hi = _i64([0] * (8 * ndev)), _i64([0] * (8 * ndev))
    outL = _Layout()
    _ok(_load().oracle_infer_broadcast(n, nds, shp, Ls, ctypes.byref(out_nd), oshape, lo, hi, ctypes.byref(outL),
                                       ctypes.byref(st)), "infer_broadcast")
    nd = out_nd.value
    shape = tuple(oshape[d] for d in range(nd))
    if st.value != 0:
        return st.value, shape, None, None
    boxes = [(tuple(lo[v * 8 + d] for d in range(nd)), tuple(hi[v * 8 + d] for d in range(nd))) for v in range(ndev)]
    return 0, shape, boxes, Layout._from_c(outL)


def shard_shape(shape: Sequence[int], layout: Layout, device: int) -> Tuple[int, ...]:
    lo, hi, _ = shard_box(shape, layout, device)
    return tuple(h - l for l, h in zip(lo, hi))


# ---- data movement -----------------------------------------------------------

def shard(full: np.ndarray, layout: Layout) -> List[np.ndarray]:
    full = np.ascontiguousarray(full)
    code = _dtype_code(full)
    shape = full.shape
    outs = [np.zeros(shard_shape(shape, layout, d), dtype=full.dtype) for d in range(layout.num_devices)]
    ptrs = (ctypes.c_void_p * len(outs))(*[o.ctypes.data for o in outs])
    L = layout._c()
    _ok(_load().oracle_shard(code, len(shape), _i64(shape), full.ctypes.data, ctypes.byref(L), ptrs), "shard")
    return outs


def gather(pieces: Sequence[np.ndarray], shape: Sequence[int], layout: Layout) -> np.ndarray:
    """The logical tensor in float64 (partials summed in float64)."""
    pieces = [np.ascontiguousarray(p) for p in pieces]
    code = _dtype_code(pieces[0])
    out = np.zeros(tuple(shape), dtype=np.float64)
    ptrs = (ctypes.c_void_p * len(pieces))(*[p.ctypes.data for p in pieces])
    L = layout._c()
    _ok(_load().oracle_gather(code, len(shape), _i64(shape), ptrs, ctypes.byref(L),
                              out.ctypes.data_as(ctypes.POINTER(ctypes.c_double))), "gather")
    return out


def reshard(pieces: Sequence[np.ndarray], shape: Sequence[int], src: Layout, dst: Layout) -> List[np.ndarray]:
    pieces = [np.ascontiguousarray(p) for p in pieces]
    code = _dtype_code(pieces[0])
    dt = pieces[0].dtype
    outs = [np.zeros(shard_shape(shape, dst, d), dtype=dt) for d in range(dst.num_devices)]
    sp = (ctypes.c_void_p * len(pieces))(*[p.ctypes.data for p in pieces])
    dp = (ctypes.c_void_p * len(outs))(*[o.ctypes.data for o in outs])
    Ls, Ld = src._c(), dst._c()
    _ok(_load().oracle_reshard(code, len(shape), _i64(shape), sp, ctypes.byref(Ls), dp, ctypes.byref(Ld)),
        "reshard")
    return outs


# ---- inference ---------------------------------------------------------------

def infer_spmd(einsum: str, dims_mappings: Sequence[Sequence[int]], mesh_ndim: int):
    """Returns (out_dims_mapping, partial_mesh_dims, needs_reshard_inputs, inferred_input_mappings)."""
    lhs, rhs = einsum.split("->")
    ins = lhs.split(",")
    arrs = [_i32(dm) for dm in dims_mappings]
    merged = [_i32([0] * max(1, len(t))) for t in ins]
    P = ctypes.POINTER(ctypes.c_int32)
    inp = (P * len(arrs))(*[ctypes.cast(a, P) for a in arrs])
    mp = (P * len(merged))(*[ctypes.cast(a, P) for a in merged])
    out = _i32([0] * max(1, len(rhs)))
    pm, rm = ctypes.c_uint32(), ctypes.c_uint32()
    _ok(_load().oracle_infer_spmd(einsum.encode(), len(dims_mappings), inp, mesh_ndim, out, ctypes.byref(pm),
                                  ctypes.byref(rm), mp), "infer_spmd")
    partial = [d for d in range(32) if (pm.value >> d) & 1]
    needs = [j for j in range(len(ins)) if (rm.value >> j) & 1]
    return ([out[i] for i in range(len(rhs))], partial, needs,
            [[merged[j][i] for i in range(len(ins[j]))] for j in range(len(ins))])


DIMTRANS = {0: "InputDim", 1: "Flatten", 2: "Split", 3: "Singleton", 4: "SplitFlatten"}


def reshape_spmd(in_shape, in_dims_mapping, out_shape, mesh):
    """Returns (in_dims_after, out_dims_mapping, dimtrans) where dimtrans[o] =
    (kind, first input dim, number of input dims, piece, number of pieces)."""
    ni, no = len(in_shape), len(out_shape)
    after, outm = _i32([0] * ni), _i32([0] * no)
    k, f, c, p, n = (_i32([0] * no) for _ in range(5))
    _ok(_load().oracle_reshape_spmd(ni, _i64(in_shape), _i32(in_dims_mapping), no, _i64(out_shape), len(mesh),
                                    _i64(mesh), after, outm, k, f, c, p, n), "reshape_spmd")
    dts = [(DIMTRANS[k[o]], f[o], c[o], p[o], n[o]) for o in range(no)]
    return [after[i] for i in range(ni)], [outm[o] for o in range(no)], dts


def _sbp_code(e):
    if e in ("B", "P"):
        return ord(e), -1
    if e in ("Pmin", "Pmax"):
        return ord("N" if e == "Pmin" else "X"), -1
    return ord("S"), int(e[1])


def infer_sbp_signature(shape, elem_bytes, inputs, constraint=None):
    """inputs: per input, its ND-SBP as a list of entries ("S", axis) / "B" / "P"
    (one per mesh dim). Returns (signature entries, CopyCost, OrderValue,
    number of candidates kept)."""
    n_in = len(inputs)
    md = len(inputs[0])
    kinds, axes = [], []
    for sbp in inputs:
        for e in sbp:
            k, a = _sbp_code(e)
            kinds.append(k)
            axes.append(a)
    I8 = ctypes.c_int8
    ck = ca = None
    if constraint is not None:
        c = [_sbp_code(e) for e in constraint]
        ck = (I8 * md)(*[k for k, _ in c])
        ca = _i32([a for _, a in c])
    ok_, oa = (I8 * md)(), _i32([0] * md)
    cost, order, ncand = ctypes.c_double(), ctypes.c_int32(), ctypes.c_int32()
    rc = _load().oracle_infer_sbp_signature(n_in, len(shape), _i64(shape), elem_bytes, md,
                                            (I8 * len(kinds))(*kinds), _i32(axes), ck, ca, ok_, oa,
                                            ctypes.byref(cost), ctypes.byref(order), ctypes.byref(ncand))
    if rc == -2:
        raise OracleError("no candidate satisfies the constraint")
    _ok(rc, "infer_sbp_signature")
    sig = []
    for d in range(md):
        k = chr(ok_[d])
        sig.append(("S", oa[d]) if k == "S" else k)
    return sig, cost.value, order.value, ncand.value


# ---- scalars and the TP-MLP -----------------------------------------------------

def bf16_round(x: float) -> int:
    return int(_load().oracle_bf16_round(float(x)))


def gelu(x: float) -> float:
    return float(_load().oracle_gelu(float(x)))


def gelu_grad(x: float) -> float:
    return float(_load().oracle_gelu_grad(float(x)))


def tp_mlp_backward(X, A_shards, B_shards, dZ, rows=(), cols=(), flags: int = 7):
    """Gradients of sum(dZ * Z) for Z = sum_i GELU(X A_i) B_i (all bf16 bit
    patterns), in float64. flags: 1 round H, 2 round Y, 4 round dH to bf16
    (7 = what a bf16 pipeline stores; 0 = the exact gradient).
    Returns a dict with, for the listed rows m: dX [r, K], dH (before its own
    rounding), dY and H [r, F]; for the listed hidden columns f in [0, F):
    dA [c, K] = dA_{f // (F/P)}[:, f % (F/P)] and dB [c, N] = the matching row of dB."""
    X = np.ascontiguousarray(X, dtype=np.uint16)
    dZ = np.ascontiguousarray(dZ, dtype=np.uint16)
    A_shards = [np.ascontiguousarray(a, dtype=np.uint16) for a in A_shards]
    B_shards = [np.ascontiguousarray(b, dtype=np.uint16) for b in B_shards]
    P = len(A_shards)
    M, K = X.shape
    Fp = A_shards[0].shape[1]
    N = B_shards[0].shape[1]
    F = Fp * P
    rows = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1)
    cols = np.ascontiguousarray(cols, dtype=np.int64).reshape(-1)
    out = {"dX": np.zeros((len(rows), K)), "dH": np.zeros((len(rows), F)), "dY": np.zeros((len(rows), F)),
           "H": np.zeros((len(rows), F)), "dA": np.zeros((len(cols), K)), "dB": np.zeros((len(cols), N))}
    ap = (ctypes.c_void_p * P)(*[a.ctypes.data for a in A_shards])
    bp = (ctypes.c_void_p * P)(*[b.ctypes.data for b in B_shards])
    dbl = ctypes.POINTER(ctypes.c_double)
    u16 = ctypes.POINTER(ctypes.c_uint16)
    i64 = ctypes.POINTER(ctypes.c_int64)
    d = {k: v.ctypes.data_as(dbl) for k, v in out.items()}
    _ok(_load().oracle_tp_mlp_backward(P, M, K, F, N, X.ctypes.data_as(u16), ap, bp, dZ.ctypes.data_as(u16), flags,
                                       len(rows), rows.ctypes.data_as(i64), d["dX"], d["dH"], d["dY"], d["H"],
                                       len(cols), cols.ctypes.data_as(i64), d["dA"], d["dB"]), "tp_mlp_backward")
    return out


def tp_mlp(X: np.ndarray, A_shards: Sequence[np.ndarray], B_shards: Sequence[np.ndarray], rows=None,
           act: str = "gelu", round_y: bool = True):
    """Z rows (float64) of sum_i act(X A_i) B_i and the bf16-rounded Y rows.
    X, A_i, B_i are bf16 bit patterns (uint16)."""
    X = np.ascontiguousarray(X, dtype=np.uint16)
    A_shards = [np.ascontiguousarray(a, dtype=np.uint16) for a in A_shards]
    B_shards = [np.ascontiguousarray(b, dtype=np.uint16) for b in B_shards]
    P = len(A_shards)
    M, K = X.shape
    Fp = A_shards[0].shape[1]
    N = B_shards[0].shape[1]
    F = Fp * P
    rows = np.arange(M, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    y = np.zeros((len(rows), F), dtype=np.float64)
    z = np.zeros((len(rows), N), dtype=np.float64)
    ap = (ctypes.c_void_p * P)(*[a.ctypes.data for a in A_shards])
    bp = (ctypes.c_void_p * P)(*[b.ctypes.data for b in B_shards])
    dbl = ctypes.POINTER(ctypes.c_double)
    _ok(_load().oracle_tp_mlp(P, M, K, F, N, X.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)), ap, bp,
                              1 if act == "gelu" else 0, 1 if round_y else 0, len(rows),
                              rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), y.ctypes.data_as(dbl),
                              z.ctypes.data_as(dbl)), "tp_mlp")
    return z, y
