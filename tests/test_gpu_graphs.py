"""The library's launches can be captured in a CUDA graph: reshard and the
TP-MLP allocate no device memory and take their task tables and tensor maps as
kernel parameters, so a captured sequence replays with the results of direct
calls, without host-side planning."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import to_dev, to_host

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
    assert m.device_error() == 0


def test_reshard_sequence_replays_in_a_graph():
    shape = (8, 256, 512)
    T = synth.normal(3, shape, "f32")
    s0 = rtp.spec_nd_sbp((8,), (("S", 0),))
    s2 = rtp.spec_nd_sbp((8,), (("S", 2),))
    s1 = rtp.spec_nd_sbp((8,), (("S", 1),))
    src = [p.contiguous() for p in rtp.shard(to_dev(T), s0)]
    mid = [torch.empty(rtp.shard_shape(shape, s2, r), device="cuda") for r in range(8)]
    out = [torch.empty(rtp.shard_shape(shape, s1, r), device="cuda") for r in range(8)]
    stream = torch.cuda.Stream()
    # warm up (first launches set kernel attributes), then capture S(0) -> S(2) -> S(1)
    with torch.cuda.stream(stream):
        rtp.reshard(src, shape, s0, s2, out=mid, stream=stream)
        rtp.reshard(mid, shape, s2, s1, out=out, stream=stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        rtp.reshard(src, shape, s0, s2, out=mid, stream=stream)
        rtp.reshard(mid, shape, s2, s1, out=out, stream=stream)
    for o in out:
        o.zero_()
    for p, new in zip(src, rtp.shard(to_dev(T * 2.0), s0)):  # new inputs, same buffers
        p.copy_(new)
    g.replay()
    torch.cuda.synchronize()
    want = oracle.shard(T * 2.0, oracle.Layout((8,), (("S", 1),)))
    for r in range(8):
        np.testing.assert_array_equal(to_host(out[r]), want[r])


def test_tp_mlp_replays_in_a_graph():
    M, K, F, N, P = 256, 128, 512, 256, 2
    X = to_dev(synth.normal(0, (M, K), "bf16"))
    A = [to_dev(a) for a in np.split(synth.normal(1, (K, F), "bf16", std=0.02), P, axis=1)]
    B = [to_dev(b) for b in np.split(synth.normal(2, (F, N), "bf16", std=0.02), P, axis=0)]
    A = [a.contiguous() for a in A]
    Y = [torch.empty((M, F // P), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    Z = torch.empty((M, N), dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        rtp.tp_mlp(X, A, B, Y=Y, Z=Z, mode=1, s0=stream)
    torch.cuda.synchronize()
    direct = Z.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        rtp.tp_mlp(X, A, B, Y=Y, Z=Z, mode=1, s0=stream)
    Z.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(Z, direct)
