"""Pins of the CPU oracle to things other than itself.

Each test ties an oracle function to values the pages print (fixtures under
tests/golden, each with its citation), to closed forms, to invariants, to
independent library routines (numpy, scipy, torch) or to brute force on tiny
inputs. A plausible slip in the oracle (a transposed mesh order, inner-first
splits, a dropped partial, a wrong rounding) fails at least one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import Layout


def _golden(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


# ---- pages' worked examples ---------------------------------------------------

def test_onnx_sharding_examples(golden_dir):
    g = _golden(golden_dir, "onnx_sharding_examples.json")
    T = np.array(g["tensor"], dtype=np.float32)
    for case in g["cases"]:
        dmap = {int(k): v for k, v in case["device_map"].items()}
        L = oracle.layout_from_onnx(2, case["device"], dmap, [tuple(s) for s in case["sharded_dim"]])
        pieces = oracle.shard(T, L)
        assert [p.tolist() for p in pieces] == case["expected"], case["name"]


def test_split_broadcast_follows_rule_not_printed_value(golden_dir):
    g = _golden(golden_dir, "onnx_sharding_examples.json")
    case = g["cases"][-1]
    T = np.array(g["tensor"], dtype=np.float32)
    L = oracle.layout_from_onnx(2, case["device"], {-1: [0, 1], -2: [2, 3]}, [(0, 2)])
    pieces = oracle.shard(T, L)
    # the rule: piece 1 of axis 0 is the second row
    assert pieces[2].tolist() == [T[1].tolist()] == pieces[3].tolist()
    assert pieces[2].tolist() != case["printed_on_page_for_devices_2_and_3"]


def test_oneflow_add_infers_split0_and_computes(golden_dir):
    g = _golden(golden_dir, "oneflow_sbp_examples.json")["add_example"]
    T = np.array(g["tensor"], dtype=np.float32)
    out, partial, needs, merged = oracle.infer_spmd(g["einsum"], [g["t1_dims_mapping"], g["t2_dims_mapping"]], 1)
    assert out == g["expected_t3_dims_mapping"] and partial == []
    assert needs == [1]  # t1 already matches; t2 must be resharded
    mesh = [2]
    L1 = oracle.layout_from_dims_mapping(g["t1_dims_mapping"], mesh)
    L2 = oracle.layout_from_dims_mapping(g["t2_dims_mapping"], mesh)
    L3 = oracle.layout_from_dims_mapping(out, mesh)
    assert L3.entries == (("S", 0),) and L3.devices == tuple(g["printed_t3_placement_ranks"])
    t1, t2 = oracle.shard(T, L1), oracle.shard(T, L2)
    t2r = oracle.reshard(t2, T.shape, L2, oracle.layout_from_dims_mapping(merged[1], mesh))
    t3 = [a + b for a, b in zip(t1, t2r)]
    assert [p.tolist() for p in t3] == g["expected_t3_pieces"]
    np.testing.assert_array_equal(oracle.gather(t3, T.shape, L3), 2 * T)


def test_oneflow_nd_sbp_broadcast_then_split(golden_dir):
    g = _golden(golden_dir, "oneflow_sbp_examples.json")
    nd = g["nd_sbp_example"]
    T = np.array(nd["tensor"], dtype=np.float32)
    ents = tuple(e if isinstance(e, str) else (e[0], e[1]) for e in nd["nd_sbp"])
    L = Layout((2, 2), ents, tuple(sum(nd["ranks"], [])))
    assert [p.tolist() for p in oracle.shard(T, L)] == nd["expected"]
    for h in g["hierarchy"]:
        ranks = np.array(h["ranks"])
        assert list(ranks.shape) == h["hierarchy"]
        L = oracle.layout_from_dims_mapping([-1], list(ranks.shape), list(ranks.reshape(-1)))
        assert L.mesh == tuple(h["hierarchy"]) and L.devices == tuple(ranks.reshape(-1).tolist())


def test_paddle_matmul_merge(golden_dir):
    g = _golden(golden_dir, "paddle_spmd_examples.json")["matmul"]
    out, partial, needs, merged = oracle.infer_spmd(g["einsum"], [g["x"], g["y"]], g["mesh_ndim"])
    assert out == g["expected_out"] and partial == [] and needs == []
    assert merged == [[g["merged"]["m"], g["merged"]["k"]], [g["merged"]["k"], g["merged"]["n"]]]


def test_paddle_bsh_dims_mapping(golden_dir):
    g = _golden(golden_dir, "paddle_spmd_examples.json")["bsh"]
    shape = (4, 3, 6)
    L = oracle.layout_from_dims_mapping(g["dims_mapping"], [2, 2])
    T = np.arange(np.prod(shape), dtype=np.float32).reshape(shape)
    pieces = oracle.shard(T, L)
    for x in range(2):
        for y in range(2):
            np.testing.assert_array_equal(pieces[2 * x + y], T[2 * x:2 * x + 2, :, 3 * y:3 * y + 3])


def test_paddle_dimtrans_examples(golden_dir):
    for case in _golden(golden_dir, "paddle_spmd_examples.json")["dimtrans"]:
        _, _, dts = oracle.reshape_spmd(case["in"], [-1] * len(case["in"]), case["out"], [2])
        for dt, exp in zip(dts, case["expected"]):
            kind, first, count, piece, npieces = dt
            assert kind == exp[0]
            if kind == "InputDim":
                assert first == exp[1] and count == 1
            elif kind == "Flatten":
                assert list(range(first, first + count)) == exp[1:]
            elif kind == "Split":
                assert first == exp[1] and piece == exp[2] and count == 1


# ---- geometry invariants ------------------------------------------------------

MESHES = [(1,), (2,), (3,), (4,), (2, 2), (2, 3)]


def _layouts(ndim, mesh):
    """Every assignment of S(axis)/B/P to the mesh dims."""
    opts = [("S", a) for a in range(ndim)] + ["B", "P"]
    for ents in itertools.product(opts, repeat=len(mesh)):
        yield Layout(mesh, ents)


def test_pieces_tile_tensor_in_device_order():
    """S pieces of the B-representative devices cover every element once, are
    boxes, follow the outer-first order, and have ceil-sized leading pieces."""
    for shape in [(L,) for L in range(1, 18)] + [(a, b) for a in (1, 2, 3, 5) for b in (1, 4, 7)]:
        T = np.arange(int(np.prod(shape)), dtype=np.float32).reshape(shape)
        for mesh in MESHES:
            for L in _layouts(len(shape), mesh):
                if "P" in L.entries:
                    continue
                pieces = oracle.shard(T, L)
                reps = []
                for dev in range(L.num_devices):
                    pos = L.devices.index(dev)
                    coords = np.unravel_index(pos, mesh)
                    if all(c == 0 for c, e in zip(coords, L.entries) if e == "B"):
                        reps.append(pieces[dev])
                    lo, hi, _ = oracle.shard_box(shape, L, dev)
                    np.testing.assert_array_equal(pieces[dev], T[tuple(slice(l, h) for l, h in zip(lo, hi))])
                vals = np.sort(np.concatenate([p.reshape(-1) for p in reps]))
                np.testing.assert_array_equal(vals, T.reshape(-1))


def test_uneven_split_sizes_and_nesting():
    # one level: ceil-sized leading pieces, short (possibly empty) tail
    for Lx in range(1, 18):
        for n in (2, 3, 4):
            L = Layout((n,), (("S", 0),))
            sizes = [oracle.shard_shape((Lx,), L, d)[0] for d in range(n)]
            c = math.ceil(Lx / n)
            assert sum(sizes) == Lx and max(sizes) == c
            assert sizes == sorted(sizes, reverse=True)
            assert all(s == c for s in sizes[:Lx // c])
    # nested: (S(0), S(0)) on 2x2 cuts level by level, outer first
    L = Layout((2, 2), (("S", 0), ("S", 0)))
    boxes = [oracle.shard_box((5,), L, d)[:2] for d in range(4)]
    assert boxes == [((0,), (2,)), ((2,), (3,)), ((3,), (4,)), ((4,), (5,))]
    # the uneven configuration: [12289, 6143] on a 2x2 mesh as (S(0), S(1))
    L = Layout((2, 2), (("S", 0), ("S", 1)))
    assert [oracle.shard_shape((12289, 6143), L, d) for d in range(4)] == [
        (6145, 3072), (6145, 3071), (6144, 3072), (6144, 3071)]


def test_partial_shard_is_exact_and_sums_back():
    T = synth.normal(3, (5, 7), "f32")
    for mesh in [(2,), (4,), (2, 2)]:
        for ents in [("P",) * len(mesh), ("P", ("S", 1))[:len(mesh)], (("S", 0), "P")[:len(mesh)]]:
            L = Layout(mesh, ents)
            pieces = oracle.shard(T, L)
            np.testing.assert_array_equal(oracle.gather(pieces, T.shape, L), T.astype(np.float64))
            # P -> B of a sharded-P tensor gives B exactly
            B = Layout(mesh, ("B",) * len(mesh))
            for p in oracle.reshard(pieces, T.shape, L, B):
                np.testing.assert_array_equal(p, T)


def test_reshard_round_trip_and_definition():
    rng = np.random.default_rng(0)
    shape = (5, 6, 3)
    T = synth.uniform(4, shape, "f32")
    Tb = synth.uniform(4, shape, "bf16")
    meshes = [(2,), (3,), (2, 2), (2, 3)]
    for _ in range(120):
        mesh = meshes[rng.integers(len(meshes))]
        opts = [("S", a) for a in range(3)] + ["B"]
        a = Layout(mesh, tuple(opts[i] for i in rng.integers(len(opts), size=len(mesh))))
        b = Layout(mesh, tuple(opts[i] for i in rng.integers(len(opts), size=len(mesh))))
        for X in (T, Tb):
            pa = oracle.shard(X, a)
            pb = oracle.reshard(pa, shape, a, b)
            for got, exp in zip(pb, oracle.shard(X, b)):
                np.testing.assert_array_equal(got, exp)
            for got, exp in zip(oracle.reshard(pb, shape, b, a), pa):
                np.testing.assert_array_equal(got, exp)


def test_partial_sum_against_numpy():
    """P -> B / P -> S of 4 N(0,1) [4,6] partials against numpy's float64 sum."""
    parts = [synth.normal(100 + k, (4, 6), "f32") for k in range(4)]
    ref = np.sum(np.stack(parts).astype(np.float64), axis=0)
    P = Layout((4,), ("P",))
    for out in oracle.reshard(parts, (4, 6), P, Layout((4,), ("B",))):
        np.testing.assert_array_equal(out, ref.astype(np.float32))
    outs = oracle.reshard(parts, (4, 6), P, Layout((4,), (("S", 1),)))
    np.testing.assert_array_equal(np.concatenate(outs, axis=1), ref.astype(np.float32))
    # bf16 partials: one rounding of the exact sum
    pb = [synth.normal(200 + k, (4, 6), "bf16") for k in range(4)]
    refb = np.sum(np.stack([synth.bf16_bits_to_f32(p) for p in pb]).astype(np.float64), axis=0)
    want = torch.from_numpy(refb.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.reshard(pb, (4, 6), P, Layout((4,), ("B",)))[0]
    # float64 -> float32 -> bf16 can differ from a direct rounding only at ties
    assert np.count_nonzero(got != want) <= 1


# ---- scalars ------------------------------------------------------------------

def test_bf16_rounding_special_values():
    cases = [(1.0, 0x3F80), (1 + 2 ** -8, 0x3F80), (1 + 3 * 2 ** -8, 0x3F82), (1 + 2 ** -8 + 2 ** -30, 0x3F81),
             (-2.5, 0xC020), (0.0, 0x0000), (-0.0, 0x8000), (2.0 ** -133, 0x0001), (2.0 ** -134, 0x0000),
             (1.5 * 2.0 ** -134, 0x0001), (2.0 ** -126, 0x0080), (2.0 ** 128, 0x7F80),
             ((2 - 2 ** -8) * 2.0 ** 127, 0x7F80), ((2 - 2 ** -7) * 2.0 ** 127, 0x7F7F), (float("inf"), 0x7F80)]
    for x, bits in cases:
        assert oracle.bf16_round(x) == bits, x


def test_bf16_rounding_matches_torch_on_floats():
    x = np.concatenate([synth.normal(7, (4000,), "f32", std=10.0), synth.uniform(8, (4000,), "f32", -1e-38, 1e-38)])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_round(float(v)) for v in x], dtype=np.uint16)
    np.testing.assert_array_equal(got, want)


def test_gelu_closed_forms():
    from scipy.special import ndtr
    assert oracle.gelu(0.0) == 0.0
    assert abs(oracle.gelu(1.0) - 0.8413447460685429) < 1e-15  # Phi(1)
    assert abs(oracle.gelu(2.0) - 2 * 0.9772498680518208) < 1e-15
    for x in np.linspace(-8, 8, 161):
        assert abs(oracle.gelu(x) - x * ndtr(x)) <= 1e-14 * max(1.0, abs(x))
        assert abs(oracle.gelu(x) - oracle.gelu(-x) - x) <= 1e-14 * max(1.0, abs(x))


# ---- inference: brute-force execution -----------------------------------------

EINSUMS = ["mk,kn->mn", "mn,mn->mn", "bmk,bkn->bmn", "mn->mn", "mk,k->m"]


def _dim_sizes(einsum, rng):
    letters = sorted(set(c for c in einsum if c.isalpha()))
    return {c: int(rng.choice([2, 4, 6])) for c in letters}


def test_infer_spmd_by_execution():
    """Reshard inputs to the inferred mappings, run the einsum on each device,
    and check that the inferred output layout describes the true result."""
    rng = np.random.default_rng(1)
    for einsum in EINSUMS:
        lhs, rhs = einsum.split("->")
        ins = lhs.split(",")
        for mesh in [(2,), (2, 2)]:
            for _ in range(25):
                sizes = _dim_sizes(einsum, rng)
                dms = []
                for t in ins:
                    dm = [-1] * len(t)
                    for d in range(len(mesh)):
                        if rng.random() < 0.6:
                            i = int(rng.integers(len(t)))
                            if dm[i] == -1:
                                dm[i] = d
                    dms.append(dm)
                out, partial, needs, merged = oracle.infer_spmd(einsum, dms, len(mesh))
                for j in range(len(ins)):
                    assert (j in needs) == (merged[j] != dms[j])
                tensors = [synth.uniform(10 + j, [sizes[c] for c in t], "f32") for j, t in enumerate(ins)]
                exact = np.einsum(einsum, *[x.astype(np.float64) for x in tensors])
                locs = [oracle.shard(x, oracle.layout_from_dims_mapping(m, mesh)) for x, m in zip(tensors, merged)]
                pieces = [np.einsum(einsum, *[l[dev].astype(np.float64) for l in locs]).astype(np.float32)
                          for dev in range(int(np.prod(mesh)))]
                Lout = oracle.layout_from_dims_mapping(out, mesh, partial=partial)
                got = oracle.gather(pieces, exact.shape, Lout)
                np.testing.assert_allclose(got, exact, rtol=1e-5, atol=1e-5)


def test_infer_spmd_contraction_leaves_partial():
    out, partial, needs, merged = oracle.infer_spmd("mk,kn->mn", [[-1, 0], [0, -1]], 1)
    assert out == [-1, -1] and partial == [0] and needs == []


# ---- reshape rule: brute force ------------------------------------------------

def _factorisations(total, max_dims=3):
    res = []
    def rec(rem, cur):
        if len(cur) and rem == 1:
            res.append(tuple(cur))
        if len(cur) == max_dims:
            return
        for f in range(2, rem + 1):
            if rem % f == 0:
                rec(rem // f, cur + [f])
    rec(total, [])
    return res


def _reshape_ok(T, in_dm, out_shape, out_dm, mesh):
    Lin = oracle.layout_from_dims_mapping(in_dm, mesh)
    Lout = oracle.layout_from_dims_mapping(out_dm, mesh)
    pin = oracle.shard(T, Lin)
    pout = oracle.shard(T.reshape(out_shape), Lout)
    return all(a.size == b.size and np.array_equal(a.reshape(-1), b.reshape(-1)) for a, b in zip(pin, pout))


def test_reshape_rule_by_brute_force():
    checked = 0
    for total in (6, 8, 12):
        shapes = _factorisations(total)
        for ishape in shapes:
            T = np.arange(total, dtype=np.float32).reshape(ishape)
            for oshape in shapes:
                for mesh in [(2,), (3,)]:
                    for i in range(-1, len(ishape)):
                        in_dm = [-1] * len(ishape)
                        if i >= 0:
                            in_dm[i] = 0
                        after, out_dm, _ = oracle.reshape_spmd(ishape, in_dm, oshape, mesh)
                        # the resharded input, reshaped locally, is the output layout
                        assert _reshape_ok(T, after, oshape, out_dm, mesh), (ishape, in_dm, oshape, mesh)
                        # nothing is dropped that could have been kept
                        if i >= 0 and after[i] == -1:
                            for o in range(len(oshape)):
                                alt = [-1] * len(oshape)
                                alt[o] = 0
                                assert not _reshape_ok(T, in_dm, oshape, alt, mesh)
                        checked += 1
    assert checked > 300


def test_reshape_configuration_cases():
    # [2,3,4096] -> [6,4096]: a split of the leading member survives ...
    assert oracle.reshape_spmd([2, 3, 4096], [0, -1, -1], [6, 4096], [2])[:2] == ([0, -1, -1], [0, -1])
    # ... a split of the inner member of the flattened group cannot ...
    assert oracle.reshape_spmd([2, 3, 4096], [-1, 0, -1], [6, 4096], [2])[:2] == ([-1, -1, -1], [-1, -1])
    # ... and the axis outside the group keeps its split
    assert oracle.reshape_spmd([2, 3, 4096], [-1, -1, 0], [6, 4096], [2])[:2] == ([-1, -1, 0], [-1, 0])
    # [6144,4096] -> [2,3072,4096]: the split lands on the leading piece
    assert oracle.reshape_spmd([6144, 4096], [0, -1], [2, 3072, 4096], [2])[:2] == ([0, -1], [0, -1, -1])


# ---- TP-MLP ---------------------------------------------------------------------

def _bf16(x):
    return synth.bf16_bits_to_f32(x).astype(np.float64)


def _split_cols(A, P):
    return [np.ascontiguousarray(a) for a in np.split(A, P, axis=1)]


def _split_rows(B, P):
    return [np.ascontiguousarray(b) for b in np.split(B, P, axis=0)]


@pytest.mark.parametrize("shape", [(4, 8, 16, 8, 2), (5, 12, 24, 7, 3), (3, 16, 32, 10, 8)])
def test_tp_mlp_identity_equals_xab(shape):
    """sum_i (X A_i) B_i == X A B (column split of A, row split of B)."""
    M, K, F, N, P = shape
    X = synth.normal(0, (M, K), "bf16")
    A = synth.normal(1, (K, F), "bf16")
    B = synth.normal(2, (F, N), "bf16")
    z, y = oracle.tp_mlp(X, _split_cols(A, P), _split_rows(B, P), act="identity", round_y=False)
    ref = _bf16(X) @ _bf16(A) @ _bf16(B)
    np.testing.assert_allclose(z, ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(y, _bf16(X) @ _bf16(A), rtol=1e-12, atol=1e-12)


def test_tp_mlp_gelu_commutes_with_column_split():
    """sum_i GELU(X A_i) B_i == GELU(X A) B, and Y is the bf16 rounding of GELU(X A)."""
    from scipy.special import ndtr
    M, K, F, N, P = 4, 8, 16, 8, 2  # the tiny configuration, seed 0, N(0,1)
    X = synth.normal(0, (M, K), "bf16")
    A = synth.normal(1, (K, F), "bf16")
    B = synth.normal(2, (F, N), "bf16")
    H = _bf16(X) @ _bf16(A)
    G = H * ndtr(H)
    z, y = oracle.tp_mlp(X, _split_cols(A, P), _split_rows(B, P), act="gelu", round_y=False)
    np.testing.assert_allclose(z, G @ _bf16(B), rtol=1e-12, atol=1e-12)
    z2, y2 = oracle.tp_mlp(X, _split_cols(A, P), _split_rows(B, P), act="gelu", round_y=True)
    Gb = torch.from_numpy(G).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(y2, Gb)
    np.testing.assert_allclose(z2, Gb @ _bf16(B), rtol=1e-12, atol=1e-12)


def test_tp_mlp_row_subset_matches_full():
    M, K, F, N, P = 9, 16, 32, 8, 4
    X = synth.normal(5, (M, K), "bf16")
    A = synth.normal(6, (K, F), "bf16", std=0.02)
    B = synth.normal(7, (F, N), "bf16", std=0.02)
    zf, yf = oracle.tp_mlp(X, _split_cols(A, P), _split_rows(B, P))
    rows = np.array([8, 0, 3])
    zs, ys = oracle.tp_mlp(X, _split_cols(A, P), _split_rows(B, P), rows=rows)
    np.testing.assert_array_equal(zs, zf[rows])
    np.testing.assert_array_equal(ys, yf[rows])


# ---- TP-MLP backward (ColossalAI page, section 2.2) ---------------------------------

def test_gelu_grad_is_the_derivative_of_gelu():
    """GELU'(0) = 1/2, the limits 0 and 1, the minimum at -sqrt(2) (where
    GELU'' = phi(x) (2 - x^2) vanishes), and central differences of GELU."""
    from scipy.special import ndtr
    assert oracle.gelu_grad(0.0) == 0.5
    assert abs(oracle.gelu_grad(9.0) - 1.0) < 1e-15 and abs(oracle.gelu_grad(-9.0)) < 1e-15
    xm = -np.sqrt(2.0)
    gm = oracle.gelu_grad(xm)
    assert gm < oracle.gelu_grad(xm - 1e-3) and gm < oracle.gelu_grad(xm + 1e-3)
    for x in (-3.1, -0.7, 0.25, 1.0, 2.5):
        h = 1e-5
        fd = ((x + h) * ndtr(x + h) - (x - h) * ndtr(x - h)) / (2 * h)
        assert abs(oracle.gelu_grad(x) - fd) < 1e-9
        fo = (oracle.gelu(x + h) - oracle.gelu(x - h)) / (2 * h)
        assert abs(oracle.gelu_grad(x) - fo) < 1e-9


def test_tp_mlp_backward_matches_finite_differences():
    """flags = 0: dX, dA_i, dB_i are the gradient of L = sum(dZ * Z) with
    Z = GELU(X A) B; checked by central differences of a float64 numpy
    forward on every input element."""
    from scipy.special import ndtr
    M, K, F, N, P = 5, 6, 8, 7, 2
    X = synth.normal(11, (M, K), "bf16")
    A = synth.normal(12, (K, F), "bf16", std=0.5)
    B = synth.normal(13, (F, N), "bf16", std=0.5)
    dZ = synth.normal(14, (M, N), "bf16")
    x, a, b, dz = _bf16(X), _bf16(A), _bf16(B), _bf16(dZ)

    def loss(x, a, b):
        h = x @ a
        return float(np.sum(dz * ((h * ndtr(h)) @ b)))

    g = oracle.tp_mlp_backward(X, _split_cols(A, P), _split_rows(B, P), dZ, rows=np.arange(M), cols=np.arange(F),
                               flags=0)
    eps = 1e-6
    for name, base, got in (("X", x, g["dX"]), ("A", a, g["dA"].T), ("B", b, g["dB"])):
        fd = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            args = {"X": x, "A": a, "B": b}
            up, dn = base.copy(), base.copy()
            up[idx] += eps
            dn[idx] -= eps
            args[name] = up
            lu = loss(args["X"], args["A"], args["B"])
            args[name] = dn
            ld = loss(args["X"], args["A"], args["B"])
            fd[idx] = (lu - ld) / (2 * eps)
        np.testing.assert_allclose(got, fd, rtol=1e-6, atol=1e-7, err_msg="d" + name)


def test_tp_mlp_backward_independent_of_rank_count():
    """The gradients of the full A and B do not depend on how many ranks hold
    their shards, with or without the bf16 roundings (each is elementwise)."""
    M, K, F, N = 6, 16, 32, 8
    X = synth.normal(21, (M, K), "bf16")
    A = synth.normal(22, (K, F), "bf16", std=0.1)
    B = synth.normal(23, (F, N), "bf16", std=0.1)
    dZ = synth.normal(24, (M, N), "bf16")
    for flags in (0, 7):
        g1 = oracle.tp_mlp_backward(X, [A], [B], dZ, rows=np.arange(M), cols=np.arange(F), flags=flags)
        g4 = oracle.tp_mlp_backward(X, _split_cols(A, 4), _split_rows(B, 4), dZ, rows=np.arange(M),
                                    cols=np.arange(F), flags=flags)
        for k in ("dX", "dH", "dA", "dB"):
            np.testing.assert_array_equal(g1[k], g4[k], err_msg="%s flags %d" % (k, flags))


def test_tp_mlp_backward_row_and_column_paths_agree():
    """dA and dB come from a per-column pass over all rows; with every rounding
    on they equal X^T round(dH) and round(GELU(X A))^T dZ formed from the
    per-row pass (dH, H) and the forward oracle (Y)."""
    M, K, F, N, P = 7, 8, 16, 8, 2
    X = synth.normal(31, (M, K), "bf16")
    A = synth.normal(32, (K, F), "bf16", std=0.3)
    B = synth.normal(33, (F, N), "bf16", std=0.3)
    dZ = synth.normal(34, (M, N), "bf16")
    As, Bs = _split_cols(A, P), _split_rows(B, P)
    g = oracle.tp_mlp_backward(X, As, Bs, dZ, rows=np.arange(M), cols=np.arange(F), flags=7)
    dh = torch.from_numpy(g["dH"]).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_allclose(g["dA"], (_bf16(X).T @ dh).T, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g["dX"], dh @ _bf16(A).T, rtol=1e-12, atol=1e-12)
    _, y = oracle.tp_mlp(X, As, Bs)
    np.testing.assert_allclose(g["dB"], y.T @ _bf16(dZ), rtol=1e-12, atol=1e-12)
    # H is rounded to bf16 with flag 1, and dH = dY * GELU'(H)
    hb = torch.from_numpy(_bf16(X) @ _bf16(A)).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(g["H"], hb)
    np.testing.assert_allclose(g["dY"], _bf16(dZ) @ _bf16(B).T, rtol=1e-12, atol=1e-12)
    gg = np.vectorize(oracle.gelu_grad)(hb)
    np.testing.assert_allclose(g["dH"], g["dY"] * gg, rtol=1e-12, atol=1e-15)


# ---- partial min / max (OneFlow page: min and max also work as partial reductions) ----

def test_partial_min_max_against_numpy():
    parts = [synth.normal(300 + k, (5, 7), "f32") for k in range(4)]
    stack = np.stack(parts)
    for red, fn in (("Pmin", np.minimum.reduce), ("Pmax", np.maximum.reduce)):
        L = Layout((4,), (red,))
        np.testing.assert_array_equal(oracle.gather(parts, (5, 7), L), fn(stack).astype(np.float64))
        for out in oracle.reshard(parts, (5, 7), L, Layout((4,), ("B",))):
            np.testing.assert_array_equal(out, fn(stack))
        outs = oracle.reshard(parts, (5, 7), L, Layout((4,), (("S", 1),)))
        np.testing.assert_array_equal(np.concatenate(outs, axis=1), fn(stack))
    # bf16 members: min / max are exact
    pb = [synth.normal(400 + k, (3, 9), "bf16") for k in range(3)]
    got = oracle.reshard(pb, (3, 9), Layout((3,), ("Pmax",)), Layout((3,), ("B",)))[0]
    want_f = np.maximum.reduce([synth.bf16_bits_to_f32(p) for p in pb])
    np.testing.assert_array_equal(synth.bf16_bits_to_f32(got), want_f)


def test_shard_to_partial_min_max_holds_identity():
    T = synth.normal(5, (4, 6), "f32")
    for red, ident in (("Pmin", np.inf), ("Pmax", -np.inf), ("P", 0.0)):
        L = Layout((2, 2), (red, ("S", 1)))
        pieces = oracle.shard(T, L)
        np.testing.assert_array_equal(pieces[0], T[:, :3])
        np.testing.assert_array_equal(pieces[1], T[:, 3:])
        assert np.all(pieces[2] == ident) and np.all(pieces[3] == ident)
        np.testing.assert_array_equal(oracle.gather(pieces, T.shape, L), T.astype(np.float64))


def test_mixed_partial_reductions_rejected():
    with pytest.raises(oracle.OracleError):
        oracle.shard(np.zeros((2, 2), np.float32), Layout((2, 2), ("P", "Pmax")))


# ---- SBP signature inference (OneFlow add_n walk-through) ------------------------

def _ent(e):
    return e if isinstance(e, str) else (e[0], e[1])


def test_sbp_signature_page_examples(golden_dir):
    g = _golden(golden_dir, "oneflow_sbp_examples.json")["signature_inference"]
    shape = tuple(g["shape"])
    for case in g["cases"]:
        inputs = [[_ent(e) for e in sbp] for sbp in case["inputs"]]
        sig, cost, order, ncand = oracle.infer_sbp_signature(shape, g["elem_bytes"], inputs)
        assert sig == [_ent(e) for e in case["expected"]]
        assert ncand == len(g["candidates_1d_in_order"])
    # the candidate order: with no input matching any candidate's SBP except
    # through ties, the first candidate wins (two partial-min inputs: every
    # candidate costs the same huge amount)
    sig, cost, order, _ = oracle.infer_sbp_signature(shape, 4, [["Pmin"], ["Pmin"]])
    assert sig == [_ent(g["candidates_1d_in_order"][0])] and order == 0


def test_sbp_signature_invariants():
    rng = np.random.default_rng(7)
    for ndim in (1, 2, 3):
        shape = tuple(int(x) for x in rng.integers(1, 5, size=ndim))
        opts = [("S", a) for a in range(ndim)] + ["P", "B"]
        for md in (1, 2):
            for _ in range(20):
                common = [opts[i] for i in rng.integers(len(opts), size=md)]
                n_in = int(rng.integers(1, 4))
                # all inputs already agree: that signature, order -10 n, no cost
                sig, cost, order, ncand = oracle.infer_sbp_signature(shape, 2, [common] * n_in)
                assert sig == common and cost == 0 and order == -10 * n_in
                assert ncand == (ndim + 2) ** md
                # a constraint is obeyed and disables the order value
                other = [opts[i] for i in rng.integers(len(opts), size=md)]
                sig, cost, order, ncand = oracle.infer_sbp_signature(shape, 2, [common] * n_in, constraint=other)
                assert sig == other and order == 0 and ncand == 1
    # a split input moved to another split costs its bytes; a broadcast one is "huge"
    sig, cost, order, _ = oracle.infer_sbp_signature((4, 4), 4, [[("S", 0)], [("S", 1)], [("S", 1)]])
    assert sig == [("S", 1)] and cost == 64 and order == -20
    with pytest.raises(oracle.OracleError):
        oracle.infer_sbp_signature((4,), 4, [[("S", 0)]], constraint=[("S", 3)])


# ---- ONNX broadcast n-ary element-wise rule (ONNX page, operator groups) ----------

def _onnx_layout(inp):
    dm = {int(k): v for k, v in inp["device_map"].items()}
    return oracle.layout_from_onnx(len(inp["shape"]), inp["device"], dm, [tuple(x) for x in inp["sharded_dim"]])


def test_broadcast_rule_page_examples(golden_dir):
    cases = json.load(open(os.path.join(golden_dir, "onnx_broadcast_rule_examples.json")))["cases"]
    comp, bad = cases
    st, shape, boxes, _ = oracle.infer_broadcast([c["shape"] for c in comp["inputs"]],
                                                 [_onnx_layout(c) for c in comp["inputs"]])
    assert st == 0 and list(shape) == comp["expected_shape"]
    for dev, (i, j) in enumerate(comp["expected_shard_of_device"]):
        rows, cols = shape[0] // 2, shape[1] // 2
        assert boxes[dev] == ((i * rows, j * cols), ((i + 1) * rows, (j + 1) * cols))
    st, _, _, _ = oracle.infer_broadcast([c["shape"] for c in bad["inputs"]], [_onnx_layout(c) for c in bad["inputs"]])
    assert st == 1


def _random_broadcast_case(rng):
    nd = int(rng.integers(1, 4))
    out = [int(rng.integers(1, 7)) for _ in range(nd)]
    meshes = {2: [(2,)], 3: [(3,)], 4: [(4,), (2, 2)], 6: [(6,), (2, 3), (3, 2)]}
    R = int(rng.choice([2, 3, 4, 6]))
    shapes, layouts = [], []
    for _ in range(int(rng.integers(2, 4))):
        drop = int(rng.integers(0, nd))  # leading dims absent
        sh = [1 if rng.random() < 0.3 else x for x in out[drop:]]
        mesh = meshes[R][int(rng.integers(0, len(meshes[R])))]
        ents = []
        for _m in mesh:
            if rng.random() < 0.6:
                ents.append(("S", int(rng.integers(0, len(sh)))))
            else:
                ents.append("B")
        shapes.append(tuple(sh))
        layouts.append(Layout(mesh, tuple(ents), tuple(int(v) for v in rng.permutation(R))))
    return shapes, layouts


def test_broadcast_rule_by_execution():
    """Where the rule infers a layout, every device computes its output box
    from its own input pieces alone (numpy broadcasting on the local slices) and
    gets the slice of the global result; where it reports a conflict, some
    output element is read from input pieces no single device holds together
    (found by a direct search over elements and devices)."""
    rng = np.random.default_rng(7)
    seen = {0: 0, 1: 0, 2: 0}
    for _ in range(150):
        shapes, layouts = _random_broadcast_case(rng)
        st, oshape, boxes, lay = oracle.infer_broadcast(shapes, layouts)
        seen[st] += 1
        xs = [rng.standard_normal(sh) for sh in shapes]
        full = sum((k + 1) * x for k, x in enumerate(xs)) * np.ones(oshape)
        nd = len(oshape)
        if st == 0:
            for dev, (lo, hi) in enumerate(boxes):
                assert lay is not None
                llo, lhi, _ = oracle.shard_box(oshape, lay, dev)
                if any(h <= l for l, h in zip(lo, hi)):  # computes nothing: an empty piece
                    assert any(h <= l for l, h in zip(llo, lhi))
                    continue
                assert (llo, lhi) == (lo, hi)
                acc = np.zeros([h - l for l, h in zip(lo, hi)])
                for k, (x, L) in enumerate(zip(xs, layouts)):
                    plo, phi, _ = oracle.shard_box(x.shape, L, dev)
                    piece = x[tuple(slice(a, b) for a, b in zip(plo, phi))]
                    off = nd - x.ndim
                    sl = []
                    for dk in range(x.ndim):
                        d = dk + off
                        if x.shape[dk] == 1:
                            assert phi[dk] - plo[dk] == 1
                            sl.append(slice(0, 1))
                        else:
                            assert plo[dk] <= lo[d] and hi[d] <= phi[dk]
                            sl.append(slice(lo[d] - plo[dk], hi[d] - plo[dk]))
                    acc = acc + (k + 1) * piece[tuple(sl)]
                np.testing.assert_array_equal(acc, full[tuple(slice(l, h) for l, h in zip(lo, hi))])
        elif st == 1:
            # some element has no device holding every input element it reads
            found = False
            for e in np.ndindex(*oshape):
                ok_any = False
                for dev in range(layouts[0].num_devices):
                    ok = True
                    for x, L in zip(xs, layouts):
                        plo, phi, _ = oracle.shard_box(x.shape, L, dev)
                        off = nd - x.ndim
                        for dk in range(x.ndim):
                            i = 0 if x.shape[dk] == 1 else e[dk + off]
                            ok &= plo[dk] <= i < phi[dk]
                    ok_any |= ok
                if not ok_any:
                    found = True
                    break
            assert found
    assert seen[0] > 20 and seen[1] > 10, seen
