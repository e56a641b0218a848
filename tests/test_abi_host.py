"""The C-ABI library loads, exports what include/rtp.h declares, and its
host-only logic (front-ends, shard geometry, inference, reshape rule, planned
traffic) agrees with the oracle. No GPU needed: nothing here launches work."""
import itertools
import json
import os
import re

import numpy as np
import pytest

import oracle
import resharding_tensor_parallelism_gb300 as rtp
from resharding_tensor_parallelism_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()


def _declared():
    text = open(os.path.join(ROOT, "include", "rtp.h")).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(rtp_\w+)\s*\(", text, flags=re.M)))


def test_exports_every_declared_symbol():
    names = _declared()
    assert len(names) >= 13
    lib = rtp.lib()
    for n in names:
        assert hasattr(lib, n), n
    out = os.popen("nm -D --defined-only %s" % rtp.LIB_PATH).read()
    for n in names:
        assert re.search(r"\bT %s\b" % n, out), n


def test_version_and_errors():
    assert "sm_103a" in rtp.version()
    with pytest.raises(rtp.RtpError) as e:
        rtp.spec_from_dims_mapping([0, 0], [2])
    assert e.value.status == -1 and "mesh dim 0" in rtp.last_error()
    with pytest.raises(rtp.RtpError) as e:
        rtp.spec_from_onnx(2, [-1, -2], {-1: [0, 1], -2: [2]}, [(0, 2)])
    assert e.value.status == -3  # unequal groups
    with pytest.raises(rtp.RtpError):
        rtp.spec_from_onnx(2, [0, 1, 2], {}, [(0, 2)])  # 2 pieces, 3 devices
    with pytest.raises(rtp.RtpError):
        rtp.spec_from_onnx(2, [0, 1], {}, [(2, 2)])  # axis out of range
    with pytest.raises(rtp.RtpError):
        rtp.spec_check(2, rtp.spec_nd_sbp((2,), (("S", 2),)))
    with pytest.raises(rtp.RtpError):
        rtp.spec_check(2, rtp.spec_nd_sbp((2,), ("B",), (0, 0)))
    with pytest.raises(rtp.RtpError):
        rtp.infer_spmd("mk,kn->mz", [[0, -1], [-1, -1]], 1)
    with pytest.raises(rtp.RtpError):
        rtp.infer_reshape([2, 3], [0, -1], [7], [2])
    # the wait self-test checks its limit on the host, before any launch
    lib = rtp.lib()
    for kernel in (0, 1):
        for bad in (0, 999_999, 1_000_000_001):
            assert lib.rtp_wait_selftest(kernel, bad, 16, None) == -1
        assert lib.rtp_wait_selftest(kernel, 5_000_000, None, None) == -1
    assert lib.rtp_wait_selftest(2, 5_000_000, 16, None) == -1


def _same_layout(spec, lay, shape):
    for r in range(spec.num_ranks):
        assert rtp.shard_box(shape, spec, r) == oracle.shard_box(shape, lay, r)


def test_front_ends_match_oracle():
    shape = (5, 7, 3)
    rng = np.random.default_rng(0)
    for mesh in [(2,), (3,), (2, 2), (2, 3), (1, 4)]:
        n = int(np.prod(mesh))
        for _ in range(20):
            dm = [-1] * 3
            for d in range(len(mesh)):
                if rng.random() < 0.7:
                    i = int(rng.integers(3))
                    if dm[i] == -1:
                        dm[i] = d
            free = [d for d in range(len(mesh)) if d not in dm]
            partial = [d for d in free if rng.random() < 0.5]
            ranks = list(rng.permutation(n))
            s = rtp.spec_from_dims_mapping(dm, mesh, ranks, partial)
            L = oracle.layout_from_dims_mapping(dm, mesh, ranks, partial)
            _same_layout(s, L, shape)
    cases = [
        ([0, 1], {}, [(0, 2)]), ([0, 1], {}, [(1, 2)]), ([0, 1, 2, 3], {}, [(0, 2), (1, 2)]),
        ([-1], {-1: [0, 1]}, []), ([-1, -2], {-1: [0, 1], -2: [2, 3]}, [(0, 2)]),
        ([-1, -2], {-1: [0, 2], -2: [1, 3]}, [(-1, 2)]), ([3, 1, 0, 2], {}, [(1, 4)]),
    ]
    for device, dmap, sd in cases:
        s = rtp.spec_from_onnx(2, device, dmap, sd)
        L = oracle.layout_from_onnx(2, device, dmap, sd)
        _same_layout(s, L, (4, 6))
        _same_layout(s, L, (3, 5))


def test_nd_sbp_geometry_matches_oracle():
    opts = lambda nd: [("S", a) for a in range(nd)] + ["B", "P", "Pmax"]
    for shape in [(7,), (5, 4), (3, 1, 9)]:
        for mesh in [(2,), (4,), (2, 2), (2, 3), (3, 2)]:
            for ents in itertools.product(opts(len(shape)), repeat=len(mesh)):
                if "P" in ents and "Pmax" in ents:  # one reduction per layout
                    with pytest.raises(rtp.RtpError) as e:
                        rtp.spec_check(len(shape), rtp.spec_nd_sbp(mesh, ents))
                    assert e.value.status == -3
                    continue
                _same_layout(rtp.spec_nd_sbp(mesh, ents), oracle.Layout(mesh, ents), shape)


EINSUMS = ["mk,kn->mn", "mn,mn->mn", "bmk,bkn->bmn", "mn->mn", "mk,k->m", "ij,jk,kl->il", "mn->m"]


def test_infer_spmd_matches_oracle():
    rng = np.random.default_rng(2)
    for einsum in EINSUMS:
        ins = einsum.split("->")[0].split(",")
        for mesh_ndim in (1, 2, 3):
            for _ in range(60):
                dms = []
                for t in ins:
                    dm = [-1] * len(t)
                    for d in range(mesh_ndim):
                        if rng.random() < 0.6:
                            i = int(rng.integers(len(t)))
                            if dm[i] == -1:
                                dm[i] = d
                    dms.append(dm)
                assert rtp.infer_spmd(einsum, dms, mesh_ndim) == oracle.infer_spmd(einsum, dms, mesh_ndim), (einsum, dms)


def test_infer_spmd_page_examples():
    assert rtp.infer_spmd("mk,kn->mn", [[0, -1], [-1, 1]], 2)[:3] == ([0, 1], [], [])
    assert rtp.infer_spmd("mn,mn->mn", [[0, -1], [-1, 0]], 1)[:3] == ([0, -1], [], [1])
    assert rtp.infer_spmd("mk,kn->mn", [[-1, 0], [0, -1]], 1)[:3] == ([-1, -1], [0], [])


def test_infer_reshape_matches_oracle():
    shapes = {6: [(6,), (2, 3), (3, 2), (1, 6), (6, 1), (2, 1, 3)], 12: [(12,), (2, 6), (6, 2), (3, 4), (2, 2, 3),
                                                                           (4, 3), (2, 3, 2)]}
    for total, group in shapes.items():
        for a in group:
            for b in group:
                for mesh in [(2,), (3,), (2, 2)]:
                    for dm in itertools.product(range(-1, len(mesh)), repeat=len(a)):
                        used = [d for d in dm if d >= 0]
                        if len(used) != len(set(used)):
                            continue
                        got = rtp.infer_reshape(a, list(dm), b, mesh)
                        want = oracle.reshape_spmd(a, list(dm), b, mesh)[:2]
                        assert got == (want[0], want[1]), (a, dm, b, mesh)
    assert rtp.infer_reshape([2, 3, 4096], [0, -1, -1], [6, 4096], [2]) == ([0, -1, -1], [0, -1])
    assert rtp.infer_reshape([6144, 4096], [0, -1], [2, 3072, 4096], [2]) == ([0, -1], [0, -1, -1])


def _dm(dm, mesh, partial=()):
    return rtp.spec_from_dims_mapping(dm, mesh, partial=partial)


def test_planned_traffic_matches_algorithmic_bytes():
    """Bytes planned for the resharding sweep on [8,2048,4096] (each source
    byte read once, every destination byte written)."""
    shape = (8, 2048, 4096)
    N = int(np.prod(shape))
    for es, code in ((4, rtp.F32), (2, rtp.BF16)):
        m1, m2 = (8,), (2, 4)
        cases = [
            (_dm([0, -1, -1], m1), _dm([-1, -1, 0], m1), 2),
            (_dm([-1, -1, 0], m1), _dm([-1, 0, -1], m1), 2),
            (_dm([0, -1, 1], (1, 8)), _dm([-1, -1, -1], (1, 8)), 9),
            (_dm([-1, -1, -1], m1, [0]), _dm([-1, -1, -1], m1), 16),
            (_dm([-1, -1, -1], m1, [0]), _dm([-1, -1, 0], m1), 9),
            (_dm([-1, -1, -1], m1), _dm([0, -1, -1], m1), 2),
            (_dm([0, -1, -1], m2), _dm([-1, -1, 0], m2), 5),
            (_dm([-1, -1, 0], m2), _dm([-1, 0, -1], m2), 5),
            (_dm([0, -1, 1], m2), _dm([-1, -1, -1], m2), 9),
            (_dm([-1, -1, -1], m2, [0, 1]), _dm([-1, -1, -1], m2), 16),
            (rtp.spec_nd_sbp(m2, ("P", "P")), rtp.spec_nd_sbp(m2, (("S", 2), ("S", 2))), 9),
            (rtp.spec_nd_sbp(m2, ("B", "B")), rtp.spec_nd_sbp(m2, (("S", 0), ("S", 0))), 2),
        ]
        for src, dst, mult in cases:
            rd, wr, nt, nl = rtp.reshard_cost(code, shape, src, dst)
            assert rd + wr == mult * N * es, (src, dst, rd, wr)
            assert nl == 1
    # the uneven configuration
    shape = (12289, 6143)
    N = 12289 * 6143
    s01 = rtp.spec_nd_sbp((2, 2), (("S", 0), ("S", 1)))
    assert sum(rtp.reshard_cost(rtp.F32, shape, s01, rtp.spec_nd_sbp((2, 2), (("S", 1), ("S", 0))))[:2]) == 2 * N * 4
    assert sum(rtp.reshard_cost(rtp.F32, shape, s01, rtp.spec_nd_sbp((2, 2), ("B", ("S", 1))))[:2]) == 3 * N * 4


def test_sbp_signature_matches_oracle():
    rng = np.random.default_rng(9)
    for ndim in (1, 2, 3):
        opts = [("S", a) for a in range(ndim)] + ["P", "B", "Pmax"]
        for md in (1, 2, 3):
            for _ in range(40):
                shape = tuple(int(x) for x in rng.integers(1, 7, size=ndim))
                n_in = int(rng.integers(1, 4))
                inputs = [[opts[i] for i in rng.integers(len(opts), size=md)] for _ in range(n_in)]
                want = oracle.infer_sbp_signature(shape, 2, inputs)
                got = rtp.infer_sbp_signature(shape, 2, inputs)
                assert got == tuple(want[:3]), (shape, inputs)
                cons = [opts[i] for i in rng.integers(len(opts) - 1, size=md)]
                want = oracle.infer_sbp_signature(shape, 2, inputs, constraint=cons)
                assert rtp.infer_sbp_signature(shape, 2, inputs, constraint=cons) == tuple(want[:3])
    assert rtp.infer_sbp_signature((2, 4), 4, [[("S", 0)], [("S", 1)]])[0] == [("S", 0)]
    assert rtp.infer_sbp_signature((2, 4), 4, [[("S", 0)], ["B"]])[0] == ["B"]


def test_infer_broadcast_matches_oracle():
    """ONNX broadcast n-ary rule: the library (box intersection) and the oracle
    (per element) agree on the status and on every rank's output piece."""
    import sys
    sys.path.insert(0, os.path.dirname(__file__))
    from test_oracle_pins import _random_broadcast_case

    rng = np.random.default_rng(11)
    counts = {0: 0, 1: 0, 2: 0}
    for _ in range(300):
        shapes, layouts = _random_broadcast_case(rng)
        st, oshape, boxes, _ = oracle.infer_broadcast(shapes, layouts)
        counts[st] += 1
        specs = [rtp.spec_nd_sbp(L.mesh, L.entries, L.devices) for L in layouts]
        if st != 0:
            with pytest.raises(rtp.RtpError) as e:
                rtp.infer_broadcast(shapes, specs)
            assert e.value.status == {1: -4, 2: -3}[st], (shapes, layouts, rtp.last_error())
            continue
        shape, spec = rtp.infer_broadcast(shapes, specs)
        assert shape == oshape
        for r, (lo, hi) in enumerate(boxes):
            llo, lhi, _ = rtp.shard_box(shape, spec, r)
            if any(h <= l for l, h in zip(lo, hi)):
                assert any(h <= l for l, h in zip(llo, lhi))
            else:
                assert (tuple(llo), tuple(lhi)) == (lo, hi)
    assert min(counts.values()) > 20, counts


def test_infer_broadcast_page_examples(golden_dir):
    cases = json.load(open(os.path.join(golden_dir, "onnx_broadcast_rule_examples.json")))["cases"]
    comp, bad = cases

    def spec(inp):
        dm = {int(k): v for k, v in inp["device_map"].items()}
        return rtp.spec_from_onnx(len(inp["shape"]), inp["device"], dm, [tuple(x) for x in inp["sharded_dim"]])

    shape, o = rtp.infer_broadcast([c["shape"] for c in comp["inputs"]], [spec(c) for c in comp["inputs"]])
    assert list(shape) == comp["expected_shape"]
    for dev, (i, j) in enumerate(comp["expected_shard_of_device"]):
        lo, hi, _ = rtp.shard_box(shape, o, dev)
        assert tuple(lo) == (2 * i, 3 * j) and tuple(hi) == (2 * i + 2, 3 * j + 3)
    with pytest.raises(rtp.RtpError) as e:
        rtp.infer_broadcast([c["shape"] for c in bad["inputs"]], [spec(c) for c in bad["inputs"]])
    assert e.value.status == -4
    # partial inputs and shapes that do not broadcast are refused
    with pytest.raises(rtp.RtpError) as e:
        rtp.infer_broadcast([(4, 4), (4, 4)], [rtp.spec_nd_sbp((2,), ("P",)), rtp.spec_nd_sbp((2,), ("B",))])
    assert e.value.status == -3
    with pytest.raises(rtp.RtpError) as e:
        rtp.infer_broadcast([(4, 3), (4, 5)], [rtp.spec_nd_sbp((2,), ("B",))] * 2)
    assert e.value.status == -2


def test_forms_cover_the_sweep():
    """The resharding sweep needs no register form on 256-byte aligned buffers:
    long runs are staged by bulk copies, short strided rows move as TMA tiles
    (3D and 4D tensor maps)."""
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    seen = [0, 0, 0, 0]
    for mesh in ("1x8", "2x4"):
        for _, src, dst, _ in bench.sweep_specs(rtp, mesh):
            for code in (rtp.F32, rtp.BF16):
                c = rtp.reshard_forms(code, bench.SWEEP_SHAPE, src, dst)
                assert c[0] == 0 and sum(c) == rtp.reshard_cost(code, bench.SWEEP_SHAPE, src, dst)[2]
                seen = [a + b for a, b in zip(seen, c)]
    assert seen[1] > 0 and seen[2] > 0 and seen[3] > 0
    # narrow rows and 8-byte vectors take the register form
    s, d = rtp.spec_nd_sbp((4,), (("S", 0),)), rtp.spec_nd_sbp((4,), (("S", 1),))
    assert rtp.reshard_forms(rtp.F32, (64, 36), s, d)[0] > 0


def test_form_test_cases_take_their_form():
    """Each case of the GPU form tests is carried by the form it names, on the
    host planner alone (no GPU): registers, including the float32 rows that
    go row by row, bulk staging, 3D and 4D TMA tiles."""
    import sys
    sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
    import test_gpu_boxing_forms as tf
    for name, shape, mesh, src, dst, form in tf.CASES:
        for code in (rtp.F32, rtp.BF16):
            c = rtp.reshard_forms(code, shape, rtp.spec_nd_sbp(mesh, src), rtp.spec_nd_sbp(mesh, dst))
            assert c[form] > 0 and sum(c) == c[form], (name, code, c)


def test_binding_checks_buffers_before_any_launch():
    """The library sees raw pointers only, so the binding checks every buffer's
    count, shape, dtype and device against what the call will touch; a wrong
    buffer raises RtpError and nothing reaches the GPU."""
    import torch

    spec = rtp.spec_nd_sbp((3,), (("S", 0),))
    shapes = rtp.piece_shapes((13, 7), spec)
    assert shapes == [rtp.shard_shape((13, 7), spec, r) for r in range(3)] == [(5, 7), (5, 7), (3, 7)]
    assert rtp.piece_shapes((13, 7), spec) is shapes  # cached per (shape, spec)

    cpu, f32 = -1, torch.float32  # get_device() of a host tensor
    good = [torch.zeros(s) for s in shapes]
    rtp._check_buffers("t", cpu, [("out", good, shapes, f32)])
    cases = [
        (good[:2], -1),                                                # one piece missing
        ([good[0], torch.zeros((5, 7)), torch.zeros((5, 7))], -2),     # last piece too large
        ([good[0], good[1], torch.zeros((3, 7), dtype=torch.bfloat16)], -2),  # wrong dtype
        ([good[0], good[1], torch.zeros((7, 3)).t()], -1),              # right shape, not row-major
    ]
    for pieces, status in cases:
        with pytest.raises(rtp.RtpError) as e:
            rtp._check_buffers("t", cpu, [("out", pieces, shapes, f32)])
        assert e.value.status == status
    # the public calls refuse host tensors before launching anything
    with pytest.raises(rtp.RtpError):
        rtp.shard(torch.zeros((13, 7)), spec)
    with pytest.raises(rtp.RtpError):
        rtp.reshard(good, (13, 7), spec, rtp.spec_nd_sbp((3,), (("S", 1),)))
    with pytest.raises(TypeError):
        rtp.shard(torch.zeros((13, 7), dtype=torch.float64), spec)


def test_overlapping_source_and_destination_are_rejected():
    """rtp_shard / rtp_reshard refuse buffers where a source piece and a
    destination piece share bytes (the kernel reads and writes them in no fixed
    order). The check runs on the host before any launch, so fake, never
    dereferenced addresses serve here."""
    import ctypes

    lib = rtp.lib()
    shape = rtp._i64([4, 4])
    s0 = rtp.spec_nd_sbp((2,), (("S", 0),))
    s1 = rtp.spec_nd_sbp((2,), (("S", 1),))
    src = rtp._ptrs([0x10000, 0x10100])  # two [2,4] float32 pieces: 32 bytes each
    dst = rtp._ptrs([0x20000, 0x10110])  # rank 1's [4,2] piece starts inside source piece 1
    rc = lib.rtp_reshard(rtp.F32, 2, shape, src, ctypes.byref(s0), dst, ctypes.byref(s1), None)
    assert rc == -1 and "overlaps" in rtp.last_error()
    full = ctypes.c_void_p(0x30000)      # the whole [4,4] tensor: 64 bytes
    pieces = rtp._ptrs([0x30020, 0x40000])  # rank 0's piece inside the full tensor
    rc = lib.rtp_shard(rtp.F32, 2, shape, full, ctypes.byref(s0), pieces, None)
    assert rc == -1 and "overlaps" in rtp.last_error()


def test_missing_library_fails_loudly(tmp_path):
    """Without librtp.so the binding raises on first use: there is no CPU or
    library fallback behind any call. Run in a fresh interpreter whose copy of
    the package has no compiled library next to it."""
    import shutil
    import subprocess
    import sys

    pkg = tmp_path / "resharding_tensor_parallelism_gb300"
    pkg.mkdir()
    src = os.path.join(ROOT, "resharding_tensor_parallelism_gb300")
    for f in ("__init__.py", "_build.py"):
        shutil.copy(os.path.join(src, f), pkg / f)
    code = ("import resharding_tensor_parallelism_gb300 as rtp\n"
            "for call in (lambda: rtp.lib(), lambda: rtp.spec_from_dims_mapping([0, -1], [2]),\n"
            "             lambda: rtp.version()):\n"
            "    try:\n"
            "        call()\n"
            "    except ImportError as e:\n"
            "        assert 'librtp.so is not built' in str(e)\n"
            "    else:\n"
            "        raise SystemExit('no error without the library')\n"
            "print(rtp.__file__)\n")
    out = subprocess.run([sys.executable, "-c", code], cwd=str(tmp_path), capture_output=True, text=True)
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip().startswith(str(tmp_path)), out.stdout  # the copy without a library was imported


def test_plan_cache_returns_each_layouts_own_plan():
    """shard / reshard and the cost and form queries reuse a per-thread cache
    of planned tasks, keyed by the shape and both layouts. Over interleaved
    repeats of many (shape, src, dst) triples, more than the cache holds (it
    is then cleared), the planned bytes stay those the oracle's piece geometry
    gives (every destination piece written; each distinct value-holding
    destination box read once per partial member), the form counts stay the
    first call's, and a layout whose unused array slots hold other values
    finds the same plan."""
    import random

    def expected(shape, mesh, src_e, dst_e):
        src_l, dst_l = oracle.Layout(mesh, src_e), oracle.Layout(mesh, dst_e)
        n = int(np.prod(mesh))
        vol = lambda lo, hi: int(np.prod([h - l for l, h in zip(lo, hi)]))
        members = int(np.prod([m for m, e in zip(mesh, src_e) if e == "P"]))
        wr, boxes = 0, set()
        for r in range(n):
            lo, hi, hv = oracle.shard_box(shape, dst_l, r)
            wr += vol(lo, hi) * 4
            if hv and vol(lo, hi):
                boxes.add((tuple(lo), tuple(hi)))
        rd = sum(vol(lo, hi) for lo, hi in boxes) * 4 * members
        return rd, wr

    meshes = [(2,), (4,), (2, 2), (8,), (2, 4)]
    rng = random.Random(5)
    cases = []
    for _ in range(300):
        mesh = meshes[rng.randrange(len(meshes))]
        shape = tuple(rng.randint(1, 40) for _ in range(rng.randint(1, 3)))
        opts = [("S", a) for a in range(len(shape))] + ["B", "P"]
        src_e = tuple(opts[rng.randrange(len(opts))] for _ in mesh)
        dst_e = tuple(opts[rng.randrange(len(opts) - 1)] for _ in mesh)
        cases.append((shape, rtp.spec_nd_sbp(mesh, src_e), rtp.spec_nd_sbp(mesh, dst_e),
                      expected(shape, mesh, src_e, dst_e)))
    forms = {}
    for _ in range(3):
        order = list(range(len(cases)))
        rng.shuffle(order)
        for i in order:
            sh, s, d, want = cases[i]
            assert rtp.reshard_cost(rtp.F32, sh, s, d)[:2] == want, (sh, s, d)
            assert forms.setdefault(i, rtp.reshard_forms(rtp.F32, sh, s, d)) == rtp.reshard_forms(rtp.F32, sh, s, d)
    # values beyond the used slots of each array: the same plan
    sh, s, d, want = cases[0]
    noisy = rtp.Spec.from_buffer_copy(bytes(s))
    for p in range(s.num_ranks, rtp.MAX_RANKS):
        noisy.rank_ids[p] = 77
    for m in range(s.mesh_ndim, rtp.MAX_MESH_NDIM):
        noisy.mesh_shape[m], noisy.sbp_kind[m], noisy.sbp_axis[m] = 9, 5, 3
    assert rtp.reshard_cost(rtp.F32, sh, noisy, d)[:2] == want


def test_planted_plan_mistake_is_rejected_before_any_launch():
    """A planning mistake (a destination offset moved past its piece) is caught
    by the host-side bounds check that every new plan passes before use: the
    call fails with RTP_EINVAL and nothing is launched (the buffers are fake
    host addresses that must never be touched). The layouts are chosen so that
    the first task fills its destination piece exactly: any shift leaves it."""
    shape = (4, 6)
    whole, dst = rtp.spec_nd_sbp((1,), ("B",)), rtp.spec_nd_sbp((2,), (("S", 0),))
    assert rtp.reshard_cost(rtp.F32, shape, whole, dst)[:2] == (96, 96)
    for shift in (1, -1, 1000):
        rtp.test_hook(rtp.HOOK_PLAN_SHIFT, shift)
        with pytest.raises(rtp.RtpError) as e:
            rtp.reshard_cost(rtp.F32, shape, whole, dst)
        assert e.value.status == -1 and "planned task 0" in rtp.last_error()
    rtp.test_hook(rtp.HOOK_PLAN_SHIFT, 0)  # a shift of 0 leaves the plan correct
    assert rtp.reshard_cost(rtp.F32, shape, whole, dst)[:2] == (96, 96)
    # through rtp_reshard and rtp_shard themselves, with fake pointers
    lib = rtp.lib()
    rtp.test_hook(rtp.HOOK_PLAN_SHIFT, 1)
    rc = lib.rtp_reshard(rtp.F32, 2, rtp._i64(shape), rtp._ptrs([4096]), whole, rtp._ptrs([16384, 20480]), dst, None)
    assert rc == -1 and "would write elements [1, 13) of destination piece 0, which holds 12" in rtp.last_error()
    rtp.test_hook(rtp.HOOK_PLAN_SHIFT, -1)
    rc = lib.rtp_shard(rtp.F32, 2, rtp._i64(shape), 4096, dst, rtp._ptrs([16384, 20480]), None)
    assert rc == -1 and "planned task 0" in rtp.last_error()
    # the rejected plans were not cached: a clean plan of the same layouts works
    assert rtp.reshard_cost(rtp.F32, shape, whole, dst)[:2] == (96, 96)


def test_injected_allocation_failure_returns_enomem():
    """A host allocation that fails while planning becomes RTP_ENOMEM (no
    exception crosses the C ABI) and nothing is launched; the next call
    plans normally."""
    shape = (8, 8)
    src, dst = rtp.spec_nd_sbp((4,), ("P",)), rtp.spec_nd_sbp((2, 2), (("S", 0), ("S", 1)))
    rtp.test_hook(rtp.HOOK_FAIL_ALLOC)
    with pytest.raises(rtp.RtpError) as e:
        rtp.reshard_cost(rtp.F32, shape, src, dst)
    assert e.value.status == -6 and "allocation failed" in rtp.last_error()
    assert rtp.reshard_cost(rtp.F32, shape, src, dst)[0] == 4 * 8 * 8 * 4
    lib = rtp.lib()
    rtp.test_hook(rtp.HOOK_FAIL_ALLOC)
    rc = lib.rtp_reshard(rtp.F32, 2, rtp._i64(shape), rtp._ptrs([4096] * 4), src, rtp._ptrs([8192] * 4), dst, None)
    assert rc == -6
    rtp.test_hook(rtp.HOOK_FAIL_ALLOC)
    rtp.test_hook(rtp.HOOK_NONE)  # disarmed before use
    assert rtp.reshard_cost(rtp.F32, shape, src, dst)[0] == 4 * 8 * 8 * 4
    assert rtp.lib().rtp_test_hook(7, 0) == -1


def test_noalloc_size_check_cannot_wrap():
    """Sizes whose activation bytes would wrap a 64-bit product are rejected on
    the host (RTP_ESHAPE) before any CUDA call; the pointers are fake."""
    lib = rtp.lib()
    fake = rtp._ptrs([4096] * 8)
    for (P, M, Fp) in [(1, 2 ** 30, 2 ** 30), (8, 2 ** 30, 2 ** 30), (8, 2 ** 31 - 1, 8), (2, 8, 2 ** 31 - 8),
                       (8, 4096, 512)]:
        rc = lib.rtp_tp_mlp_noalloc(P, M, 64, P * Fp, 64, 4096, fake, fake, 8192, None)
        assert rc == -2 and "static scratch" in rtp.last_error(), (P, M, Fp, rc, rtp.last_error())


def test_bounds_check_accepts_every_correct_plan():
    """The host-side bounds check runs on every new plan: over random shapes
    (ragged, some empty pieces), meshes and layouts of every kind, it passes
    each correct plan (no call is refused) and the planned bytes still equal
    the oracle's piece sizes."""
    rng = np.random.default_rng(21)
    meshes = [(1,), (2,), (3,), (4,), (2, 2), (2, 3), (3, 2), (2, 2, 2), (1, 4), (8,)]
    for case in range(400):
        ndim = int(rng.integers(1, 5))
        shape = tuple(int(x) for x in rng.integers(1, 12, size=ndim))
        m1, m2 = meshes[rng.integers(len(meshes))], meshes[rng.integers(len(meshes))]
        red = ("P", "Pmin", "Pmax")[case % 3]
        opts = [("S", a) for a in range(ndim)] + ["B", red]
        e1 = tuple(opts[i] for i in rng.integers(len(opts), size=len(m1)))
        e2 = tuple(opts[i] for i in rng.integers(len(opts), size=len(m2)))
        r1 = tuple(int(x) for x in rng.permutation(int(np.prod(m1))))
        r2 = tuple(int(x) for x in rng.permutation(int(np.prod(m2))))
        src, dst = rtp.spec_nd_sbp(m1, e1, r1), rtp.spec_nd_sbp(m2, e2, r2)
        rd, wr, nt, nl = rtp.reshard_cost(rtp.F32, shape, src, dst)
        ldst = oracle.Layout(m2, e2, r2)
        written = sum(int(np.prod(oracle.shard_shape(shape, ldst, r))) for r in range(len(r2)))
        assert wr == 4 * written, (case, shape, m1, e1, m2, e2)
