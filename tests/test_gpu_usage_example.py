"""The usage example of the README, run as written: the shapes it states, and
values checked by properties (each piece is its slice of the logical tensor,
the all-reduce gives equal replicas within the partial-sum bound, the MLP
matches the oracle on sampled rows within the Z bound)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rtp():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from resharding_tensor_parallelism_gb300 import _build
    _build.build()
    import resharding_tensor_parallelism_gb300 as m
    return m


def test_readme_example(rtp):
    torch.manual_seed(0)
    x = torch.randn(8, 2048, 4096, device="cuda")
    s0 = rtp.spec_from_dims_mapping([0, -1, -1], [8])
    s2 = rtp.spec_from_dims_mapping([-1, -1, 0], [8])
    pieces = rtp.shard(x, s0)
    assert [tuple(p.shape) for p in pieces] == [(1, 2048, 4096)] * 8
    moved = rtp.reshard(pieces, x.shape, s0, s2)
    assert [tuple(p.shape) for p in moved] == [(8, 2048, 512)] * 8
    for r in range(8):
        assert torch.equal(pieces[r], x[r:r + 1]) and torch.equal(moved[r], x[:, :, 512 * r:512 * (r + 1)])

    partials = [torch.randn_like(x) for _ in range(8)]
    p, b = rtp.spec_nd_sbp((8,), ("P",)), rtp.spec_nd_sbp((8,), ("B",))
    summed = rtp.reshard(partials, x.shape, p, b)
    assert len(summed) == 8 and all(torch.equal(s, summed[0]) for s in summed)
    exact = sum(q.double() for q in partials)
    bound = 1e-6 * sum(q.double().abs() for q in partials)
    assert bool(((summed[0].double() - exact).abs() <= bound).all())

    P = 8
    X = torch.randn(8192, 4096, device="cuda").bfloat16()
    A = [(0.02 * torch.randn(4096, 2048, device="cuda")).bfloat16() for _ in range(P)]
    B = [(0.02 * torch.randn(2048, 4096, device="cuda")).bfloat16() for _ in range(P)]
    Z, Y = rtp.tp_mlp(X, A, B)
    assert tuple(Z.shape) == (8192, 4096) and Z.dtype == torch.float32
    assert [tuple(y.shape) for y in Y] == [(8192, 2048)] * P
    rows = np.array([0, 1, 4095, 8191])
    zref, _ = oracle.tp_mlp(to_host(X), [to_host(a) for a in A], [to_host(q) for q in B], rows=rows)
    err = np.abs(to_host(Z)[rows].astype(np.float64) - zref).max()
    assert err <= 2e-2 * np.sqrt(16384 / 4096) * np.sqrt(np.mean(zref ** 2))
    assert rtp.device_error() == 0
