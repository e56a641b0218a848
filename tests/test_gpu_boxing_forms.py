"""GPU parity of each form of the resharding kernel on ragged cases.

The kernel runs a task in registers (float32 rows of 1024 vectors or more
that only allow 8- or 4-byte vectors go row by row, the rest as (row, vector)
items spread over the block), staged through shared memory by bulk
copies, or with TMA tiles of a 3D / 4D tensor map (rtp.reshard_forms tells
which). Each case below is chosen so that one form carries it, with a ragged
last chunk (or segment), in float32 and bf16, for copies and for sum, min and
max reductions; results are compared with the oracle: bit-exact for copies
and min / max, within the partial-sum bound for sums.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import test_gpu_boxing as tb

pytestmark = pytest.mark.gpu

REG, BULK, TILE3, TILE4 = 0, 1, 2, 3


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from resharding_tensor_parallelism_gb300 import _build
    _build.build()
    import resharding_tensor_parallelism_gb300 as m
    tb.rtp = m
    yield
    assert m.device_error() == 0


# (name, shape, mesh, src entries, dst entries, form that carries every task)
CASES = [
    ("registers, long rows of 4- and 8-byte vectors", (40, 8195), (2,), (("S", 1),), (("S", 0),), REG),
    ("registers, long rows, to a split of columns", (40, 8195), (2,), (("S", 0),), (("S", 1),), REG),
    ("bulk copy, ragged rows", (10, 2048), (4,), ("B",), (("S", 0),), BULK),
    ("bulk sum, ragged segment", (5, 3000), (4,), ("P",), ("B",), BULK),
    ("bulk min", (7, 5000), (4,), ("Pmin",), ("B",), BULK),
    ("bulk max to a split", (6, 4096), (2,), ("Pmax",), (("S", 0),), BULK),
    ("3D tiles copy S(0)->S(2), ragged chunk", (2, 300, 512), (8,), (("S", 0),), (("S", 2),), TILE3),
    ("3D tiles sum P->S(1), ragged chunk", (300, 512), (4,), ("P",), (("S", 1),), TILE3),
    ("3D tiles max P->S(1)", (100, 1024), (4,), ("Pmax",), (("S", 1),), TILE3),
    ("4D tiles copy S(2)->S(1), ragged rows", (3, 100, 512), (8,), (("S", 2),), (("S", 1),), TILE4),
]


def _pieces(shape, lay, dtype, seed):
    if any(e in ("P", "Pmin", "Pmax") for e in lay.entries):
        return [synth.normal(seed + k, shape, dtype) for k in range(lay.num_devices)]
    return oracle.shard(synth.normal(seed, shape, dtype), lay)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("name,shape,mesh,src,dst,form", CASES, ids=[c[0] for c in CASES])
def test_form_matches_oracle(name, shape, mesh, src, dst, form, dtype):
    code = tb.rtp.F32 if dtype == "f32" else tb.rtp.BF16
    s_spec, s_lay = tb._both(mesh, src)
    d_spec, d_lay = tb._both(mesh, dst)
    counts = tb.rtp.reshard_forms(code, shape, s_spec, d_spec)
    assert counts[form] > 0 and sum(counts) == counts[form], (name, dtype, counts)
    pieces = _pieces(shape, s_lay, dtype, seed=sum(shape) + form)
    tb._check_reshard(pieces, shape, s_spec, s_lay, d_spec, d_lay, "%s %s" % (name, dtype))

