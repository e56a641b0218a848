"""GPU parity of shard() and reshard() against the CPU oracle.

Data movement must be bit-exact. Partial sums (P -> B, P -> S) must be within
the bound of gpu_util.assert_psum. Every case goes through the C ABI via the
Python binding; inputs come from the seeded generator and never from the GPU.
"""
import itertools
import json
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import Guarded, as_f64, assert_psum, to_dev, to_host

pytestmark = pytest.mark.gpu

rtp = None


@pytest.fixture(scope="module", autouse=True)
def lib():
    global rtp
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from resharding_tensor_parallelism_gb300 import _build
    _build.build()
    import resharding_tensor_parallelism_gb300 as m
    rtp = m
    yield


def _both(mesh, entries, ranks=()):
    return rtp.spec_nd_sbp(mesh, entries, ranks), oracle.Layout(mesh, entries, tuple(ranks))


def _gpu_shard(T, spec):
    """rtp.shard into guarded pieces (every write outside a piece is caught)."""
    x = to_dev(T)
    g = Guarded()
    out = rtp.shard(x, spec, out=g.many([rtp.shard_shape(T.shape, spec, r) for r in range(spec.num_ranks)], x.dtype))
    g.check("shard")
    return [to_host(p) for p in out]


def _gpu_reshard(pieces, shape, s_src, s_dst):
    """rtp.reshard into guarded pieces (every write outside a piece is caught)."""
    ins = [to_dev(p) for p in pieces]
    g = Guarded()
    out = rtp.reshard(ins, shape, s_src, s_dst,
                      out=g.many([rtp.shard_shape(shape, s_dst, r) for r in range(s_dst.num_ranks)], ins[0].dtype))
    g.check("reshard")
    return [to_host(p) for p in out]


def _check_reshard(pieces, shape, src_spec, src_lay, dst_spec, dst_lay, what=""):
    got = _gpu_reshard(pieces, shape, src_spec, dst_spec)
    want = oracle.reshard(pieces, shape, src_lay, dst_lay)
    if "P" not in src_lay.entries:  # copies, and exact partial min / max

        for r, (g, w) in enumerate(zip(got, want)):
            assert g.shape == w.shape and g.dtype == w.dtype
            np.testing.assert_array_equal(g, w, err_msg="%s rank %d" % (what, r))
        return
    # partial sources: the exact sum and sum |x| per element, from the oracle
    ref = oracle.gather(pieces, shape, src_lay)
    abs_pieces = [np.abs(as_f64(p)).astype(np.float32) for p in pieces]
    abs_sum = oracle.gather(abs_pieces, shape, src_lay)
    for r, g in enumerate(got):
        lo, hi, hv = oracle.shard_box(shape, dst_lay, r)
        sl = tuple(slice(l, h) for l, h in zip(lo, hi))
        if hv:
            assert_psum(g, ref[sl], abs_sum[sl], "%s rank %d" % (what, r))
        else:  # the identity of the destination's partial reduction
            np.testing.assert_array_equal(g, want[r], err_msg="%s rank %d" % (what, r))


# ---- the pages' tiny examples -------------------------------------------------

def test_onnx_examples(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "onnx_sharding_examples.json")))
    T = np.array(g["tensor"], dtype=np.float32)
    for case in g["cases"]:
        dmap = {int(k): v for k, v in case["device_map"].items()}
        spec = rtp.spec_from_onnx(2, case["device"], dmap, [tuple(s) for s in case["sharded_dim"]])
        assert [p.tolist() for p in _gpu_shard(T, spec)] == case["expected"], case["name"]


def test_oneflow_examples(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "oneflow_sbp_examples.json")))
    nd = g["nd_sbp_example"]
    spec = rtp.spec_nd_sbp((2, 2), ("B", ("S", 0)), sum(nd["ranks"], []))
    assert [p.tolist() for p in _gpu_shard(np.array(nd["tensor"], np.float32), spec)] == nd["expected"]
    ex = g["add_example"]
    T = np.array(ex["tensor"], dtype=np.float32)
    out, partial, needs, merged = rtp.infer_spmd(ex["einsum"], [ex["t1_dims_mapping"], ex["t2_dims_mapping"]], 1)
    s1 = rtp.spec_from_dims_mapping(ex["t1_dims_mapping"], [2])
    s2 = rtp.spec_from_dims_mapping(ex["t2_dims_mapping"], [2])
    t1 = rtp.shard(to_dev(T), s1)
    t2 = rtp.reshard(rtp.shard(to_dev(T), s2), T.shape, s2, rtp.spec_from_dims_mapping(merged[1], [2]))
    t3 = [to_host(a + b) for a, b in zip(t1, t2)]
    assert out == ex["expected_t3_dims_mapping"] and [p.tolist() for p in t3] == ex["expected_t3_pieces"]


def test_psum_of_four_to_broadcast():
    """The tiny P-sum: 4 seeded N(0,1) [4,6] partials reduced to B."""
    parts = [synth.normal(100 + k, (4, 6), "f32") for k in range(4)]
    for mesh, src_e, dst_e in [((4,), ("P",), ("B",)), ((2, 2), ("P", "P"), ("B", "B")),
                               ((4,), ("P",), (("S", 1),)), ((2, 2), ("P", "P"), (("S", 0), ("S", 1)))]:
        s, L = _both(mesh, src_e)
        d, Ld = _both(mesh, dst_e)
        _check_reshard(parts, (4, 6), s, L, d, Ld, str((mesh, src_e, dst_e)))


# ---- random cases against the oracle ----------------------------------------------

MESHES = [(1,), (2,), (3,), (4,), (2, 2), (2, 3), (3, 2), (2, 2, 2), (1, 4), (8,)]


def _rand_entries(rng, ndim, mdim, allow_p=True):
    red = ("P", "Pmin", "Pmax")[int(rng.integers(3))]  # one partial reduction per layout
    opts = [("S", a) for a in range(ndim)] + ["B"] + ([red] if allow_p else [])
    return tuple(opts[i] for i in rng.integers(len(opts), size=mdim))


def _rand_tensor(rng, shape, dt, seed):
    if dt == "f32":
        return synth.normal(seed, shape, "f32")
    return synth.normal(seed, shape, "bf16")


def test_shard_random_vs_oracle():
    rng = np.random.default_rng(11)
    for case in range(150):
        ndim = int(rng.integers(1, 5))
        shape = tuple(int(x) for x in rng.integers(1, 10, size=ndim))
        mesh = MESHES[rng.integers(len(MESHES))]
        ranks = tuple(int(x) for x in rng.permutation(int(np.prod(mesh))))
        ents = _rand_entries(rng, ndim, len(mesh))
        dt = ("f32", "bf16")[case % 2]
        T = _rand_tensor(rng, shape, dt, case)
        spec, lay = _both(mesh, ents, ranks)
        for r, (g, w) in enumerate(zip(_gpu_shard(T, spec), oracle.shard(T, lay))):
            np.testing.assert_array_equal(g, w, err_msg="case %d %s %s %s rank %d" % (case, shape, mesh, ents, r))


def test_reshard_random_vs_oracle():
    rng = np.random.default_rng(12)
    for case in range(300):
        ndim = int(rng.integers(1, 5))
        shape = tuple(int(x) for x in rng.integers(1, 10, size=ndim))
        m1 = MESHES[rng.integers(len(MESHES))]
        m2 = MESHES[rng.integers(len(MESHES))]
        r1 = tuple(int(x) for x in rng.permutation(int(np.prod(m1))))
        r2 = tuple(int(x) for x in rng.permutation(int(np.prod(m2))))
        e1 = _rand_entries(rng, ndim, len(m1))
        e2 = _rand_entries(rng, ndim, len(m2))
        dt = ("f32", "bf16")[case % 2]
        s1, L1 = _both(m1, e1, r1)
        s2, L2 = _both(m2, e2, r2)
        # source pieces straight from the generator (partials are independent draws)
        pieces = [_rand_tensor(rng, oracle.shard_shape(shape, L1, r), dt, 1000 * case + r) for r in range(len(r1))]
        if not any(e in ("P", "Pmin", "Pmax") for e in e1):
            pieces = oracle.shard(_rand_tensor(rng, shape, dt, case), L1)
        _check_reshard(pieces, shape, s1, L1, s2, L2, "case %d %s %s%s -> %s%s" % (case, shape, m1, e1, m2, e2))


def test_edge_cases():
    # zero-size tensors launch nothing and succeed
    s, _ = _both((2,), (("S", 0),))
    out = rtp.shard(torch.empty((0, 5), device="cuda"), s)
    assert [tuple(o.shape) for o in out] == [(0, 5), (0, 5)]
    # more ranks than rows: trailing pieces are empty
    T = synth.normal(1, (3, 4), "f32")
    s, L = _both((8,), (("S", 0),))
    got = _gpu_shard(T, s)
    assert [g.shape for g in got] == [(1, 4), (1, 4), (1, 4)] + [(0, 4)] * 5
    for g, w in zip(got, oracle.shard(T, L)):
        np.testing.assert_array_equal(g, w)
    # the maximum rank (8 dims) and the maximum mesh (64 ranks)
    T = synth.normal(2, (2, 3, 1, 2, 3, 2, 1, 3), "bf16")
    s, L = _both((4, 4, 4), (("S", 1), ("S", 4), ("S", 7)))
    for g, w in zip(_gpu_shard(T, s), oracle.shard(T, L)):
        np.testing.assert_array_equal(g, w)
    s2, L2 = _both((4, 4, 4), ("B", ("S", 0), "B"))
    _check_reshard(oracle.shard(T, L), T.shape, s, L, s2, L2, "64 ranks")
    # unaligned base pointers force narrow vectors
    T = synth.normal(3, (7, 33), "f32")
    base = to_dev(np.concatenate([np.zeros(1, np.float32), T.reshape(-1)]))
    full = base[1:].view(7, 33)
    s, L = _both((2,), (("S", 1),))
    got = [to_host(p) for p in rtp.shard(full, s)]
    for g, w in zip(got, oracle.shard(T, L)):
        np.testing.assert_array_equal(g, w)


def test_errors_launch_nothing():
    s, _ = _both((2,), (("S", 0),))
    x = torch.zeros((4, 4), device="cuda")
    with pytest.raises(rtp.RtpError):
        rtp.shard(x, s, out=[torch.zeros((2, 4), device="cuda"), torch.zeros((0,), device="cuda")])
    bad = rtp.spec_nd_sbp((2,), (("S", 5),))
    with pytest.raises(rtp.RtpError):
        rtp.shard(x, bad)


# ---- full-size configurations ---------------------------------------------------

def _slice(T, shape, lay, r):
    lo, hi, hv = oracle.shard_box(shape, lay, r)
    return T[tuple(slice(l, h) for l, h in zip(lo, hi))], hv


def test_uneven_configuration_full_size():
    """[12289, 6143] fp32 U[-1,1) on 2x2: (S0,S1) -> (S1,S0) and -> (B,S1)."""
    shape = (12289, 6143)
    T = synth.uniform(7, shape, "f32")
    s01, L01 = _both((2, 2), (("S", 0), ("S", 1)))
    got = _gpu_shard(T, s01)
    want = oracle.shard(T, L01)
    assert [g.shape for g in got] == [(6145, 3072), (6145, 3071), (6144, 3072), (6144, 3071)]
    for g, w in zip(got, want):
        np.testing.assert_array_equal(g, w)
    for ents in [(("S", 1), ("S", 0)), ("B", ("S", 1))]:
        sd, Ld = _both((2, 2), ents)
        for g, w in zip(_gpu_reshard(want, shape, s01, sd), oracle.reshard(want, shape, L01, Ld)):
            np.testing.assert_array_equal(g, w)


SWEEP = [
    ("S0->S2", [0, -1, -1], [], [-1, -1, 0], []),
    ("S2->S1", [-1, -1, 0], [], [-1, 0, -1], []),
    ("S0S2->B", [0, -1, 1], [], [-1, -1, -1], []),
    ("P->B", [-1, -1, -1], "all", [-1, -1, -1], []),
    ("P->S2", [-1, -1, -1], "all", [-1, -1, 0], []),
    ("B->S0", [-1, -1, -1], [], [0, -1, -1], []),
]


def _sweep_specs(mesh, sdm, spart, ddm):
    """dims_mapping transitions of the sweep; on 2x4, 'P-sum of 8' is partial
    over both mesh dims, and S on one mapping uses both mesh dims (nested)."""
    if mesh == (1, 8) or mesh == (8,):
        m = (1, 8) if 1 in sdm else (8,)
    else:
        m = mesh
    nd = len(m)
    if spart == "all":
        src = rtp.spec_nd_sbp(m, ("P",) * nd)
        lsrc = oracle.Layout(m, ("P",) * nd)
    else:
        src = rtp.spec_from_dims_mapping(sdm, m)
        lsrc = oracle.layout_from_dims_mapping(sdm, m)
    if spart == "all" and nd == 2 and any(v >= 0 for v in ddm):
        ax = [i for i, v in enumerate(ddm) if v >= 0][0]
        dst = rtp.spec_nd_sbp(m, (("S", ax), ("S", ax)))
        ldst = oracle.Layout(m, (("S", ax), ("S", ax)))
    elif sdm == [-1, -1, -1] and spart != "all" and nd == 2:
        ax = [i for i, v in enumerate(ddm) if v >= 0][0]
        src = rtp.spec_nd_sbp(m, ("B", "B"))
        lsrc = oracle.Layout(m, ("B", "B"))
        dst = rtp.spec_nd_sbp(m, (("S", ax), ("S", ax)))
        ldst = oracle.Layout(m, (("S", ax), ("S", ax)))
    else:
        dst = rtp.spec_from_dims_mapping(ddm, m)
        ldst = oracle.layout_from_dims_mapping(ddm, m)
    return src, lsrc, dst, ldst


@pytest.fixture(scope="module")
def sweep_inputs():
    shape = (8, 2048, 4096)
    data = {}
    for dt in ("f32", "bf16"):
        data[dt] = (synth.normal(20, shape, dt), [synth.normal(30 + k, shape, dt) for k in range(8)])
    return shape, data


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("mesh", [(8,), (2, 4)])
@pytest.mark.parametrize("name,sdm,spart,ddm,dpart", SWEEP)
def test_sweep_full_size(sweep_inputs, dt, mesh, name, sdm, spart, ddm, dpart):
    shape, data = sweep_inputs
    T, parts = data[dt]
    src, lsrc, dst, ldst = _sweep_specs(mesh, sdm, spart, ddm)
    if spart == "all":
        pieces = parts
    else:
        pieces = [np.ascontiguousarray(_slice(T, shape, lsrc, r)[0]) for r in range(src.num_ranks)]
    dev_in = [to_dev(p) for p in pieces]
    guard = Guarded()
    outs = rtp.reshard(dev_in, shape, src, dst,
                       out=guard.many([rtp.shard_shape(shape, dst, r) for r in range(dst.num_ranks)], dev_in[0].dtype))
    guard.check(name)
    if spart != "all":
        for r, o in enumerate(outs):
            want, hv = _slice(T, shape, ldst, r)
            np.testing.assert_array_equal(to_host(o), want, err_msg="%s rank %d" % (name, r))
        return
    ref = np.zeros(shape, np.float64)
    abs_sum = np.zeros(shape, np.float64)
    for p in parts:
        x = as_f64(p)
        ref += x
        abs_sum += np.abs(x)
    for r, o in enumerate(outs):
        lo, hi, hv = oracle.shard_box(shape, ldst, r)
        sl = tuple(slice(l, h) for l, h in zip(lo, hi))
        assert_psum(to_host(o), ref[sl], abs_sum[sl], "%s rank %d" % (name, r))
    # deterministic: the same bits on every run
    first = [to_host(o) for o in outs]
    for _ in range(2):
        again = rtp.reshard(dev_in, shape, src, dst)
        torch.cuda.synchronize()
        for a, b in zip(first, again):
            np.testing.assert_array_equal(a, to_host(b))


# ---- beyond 2^31 elements -------------------------------------------------------

def test_more_than_2_to_the_31_elements():
    """Tensors of more than 2^31 elements (offsets past 4 GiB and 8 GiB): a
    ragged S(0) -> S(1) -> S(0) round trip in bf16, and a P-sum of two float32
    partials to B. Too large for the oracle, so the checks are properties that
    hold at any size: each piece is its slice of the logical tensor (bit for
    bit), the round trip is the identity, the B replicas are identical, and
    sampled sums (including the last elements) are within the P-sum bound."""
    g = torch.Generator(device="cuda")
    g.manual_seed(31)
    shape = (65537, 32771)  # 2,147,713,027 elements > 2^31; both splits ragged
    assert shape[0] * shape[1] > 2 ** 31
    T = torch.randn(shape, generator=g, device="cuda", dtype=torch.float32).to(torch.bfloat16)
    s0, s1 = rtp.spec_nd_sbp((2,), (("S", 0),)), rtp.spec_nd_sbp((2,), (("S", 1),))
    a = rtp.shard(T, s0)
    assert torch.equal(a[0], T[:32769]) and torch.equal(a[1], T[32769:])
    b = rtp.reshard(a, shape, s0, s1)
    assert torch.equal(b[0], T[:, :16386]) and torch.equal(b[1], T[:, 16386:])
    c = rtp.reshard(b, shape, s1, s0)
    assert all(torch.equal(x, y) for x, y in zip(c, a))
    del T, a, b, c
    torch.cuda.empty_cache()

    shape = (46341, 46341)  # 2,147,488,281 float32 elements (8.6 GB) per partial
    parts = [torch.randn(shape, generator=g, device="cuda") for _ in range(2)]
    outs = rtp.reshard(parts, shape, rtp.spec_nd_sbp((2,), ("P",)), rtp.spec_nd_sbp((2,), ("B",)))
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1])
    n = shape[0] * shape[1]
    idx = torch.cat([torch.randint(0, n, (1 << 20,), generator=g, device="cuda"),
                     torch.arange(n - 4096, n, device="cuda")])
    x = [p.view(-1)[idx].double().cpu().numpy() for p in parts]
    got = outs[0].view(-1)[idx].double().cpu().numpy()
    assert np.all(np.abs(got - (x[0] + x[1])) <= 1e-6 * (np.abs(x[0]) + np.abs(x[1])))
    assert rtp.device_error() == 0
