"""Two host threads reshard at once, each on its own stream, through the
library's per-thread launch state (parameter blocks, cached tensor maps and
cached plans): every result stays bit-identical to the single-threaded one."""
import threading

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rtp():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from resharding_tensor_parallelism_gb300 import _build
    _build.build()
    import resharding_tensor_parallelism_gb300 as m
    return m


def test_reshard_from_two_host_threads(rtp):
    g = torch.Generator(device="cuda")
    g.manual_seed(7)
    shape = (8, 256, 1001)  # the 8-way split of the last axis is ragged (126 x 7 + 119)
    mesh = (8,)
    chains = [  # each thread walks its own chain of layouts (copies, a P-sum, TMA-tile moves)
        [(("S", 0),), (("S", 2),), (("S", 1),), ("B",), (("S", 0),)],
        [("P",), (("S", 2),), (("S", 0),), (("S", 2),), ("B",)],
    ]
    specs = [[rtp.spec_nd_sbp(mesh, e) for e in chain] for chain in chains]
    T = torch.randn(shape, generator=g, device="cuda")
    parts = [torch.randn(shape, generator=g, device="cuda") for _ in range(8)]
    starts = [rtp.shard(T, specs[0][0]), parts]

    def run(k, stream):
        cur = starts[k]
        outs = []
        with torch.cuda.stream(stream):
            for a, b in zip(specs[k], specs[k][1:]):
                cur = rtp.reshard(cur, shape, a, b, stream=stream)
                outs.append(cur)
        stream.synchronize()
        return outs

    want = [run(k, torch.cuda.current_stream()) for k in range(2)]
    errors = []

    def worker(k):
        try:
            torch.cuda.set_device(0)
            s = torch.cuda.Stream()
            for it in range(25):
                got = run(k, s)
                for step, (x, y) in enumerate(zip(got, want[k])):
                    if not all(torch.equal(p, q) for p, q in zip(x, y)):
                        errors.append("thread %d, pass %d, step %d differs" % (k, it, step))
                        return
        except Exception as e:  # reported by the main thread
            errors.append("thread %d: %r" % (k, e))

    threads = [threading.Thread(target=worker, args=(k,)) for k in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    assert rtp.device_error() == 0
