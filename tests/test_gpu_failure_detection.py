"""Failure detection on the GPU without a fault: a bounded wait on an mbarrier
that nothing completes must give up, report through rtp_device_error, and leave
the context usable (the same wait code the tensor-core kernels use)."""
import numpy as np
import pytest
import torch

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
    # first launch loads the kernel (lazy module loading); keep that out of the timings
    m.wait_selftest(1_000_000)
    torch.cuda.synchronize()
    assert m.device_error() == 5
    yield


@pytest.mark.parametrize("limit_ms", [5, 50])
def test_wait_on_unset_barrier_gives_up_and_reports(limit_ms):
    assert rtp.device_error() == 0
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    out = rtp.wait_selftest(limit_ms * 1_000_000)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    got = out.cpu().numpy()[:2]
    np.testing.assert_array_equal(got, [1, 1])  # both waiters gave up
    assert rtp.device_error() == 5               # the first one recorded the self-test code
    assert rtp.device_error() == 0               # reading cleared it
    # the first waiter's limit, not the second's (4x): the second left on the abort flag
    assert limit_ms <= ms < 2.5 * limit_ms + 2, ms


def test_context_usable_after_the_timeout():
    rtp.wait_selftest(10_000_000)
    assert rtp.device_error() == 5
    X = torch.ones((256, 64), dtype=torch.bfloat16, device="cuda")
    As = [torch.full((64, 128), 0.125, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    Bs = [torch.full((128, 64), 0.5, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    Z, _ = rtp.tp_mlp(X, As, Bs)
    torch.cuda.synchronize()
    # h = 64 * 0.125 = 8 everywhere, GELU(8) rounds to 8 in bf16, Z = 256 * 8 * 0.5
    assert float(Z.min()) == float(Z.max()) == 1024.0
    assert rtp.device_error() == 0


@pytest.mark.parametrize("limit_ms", [5, 50])
def test_staged_copy_wait_gives_up_and_reports(limit_ms):
    """The resharding kernel's bounded wait (staged bulk copies): 16 bytes
    announced on the block's mbarrier never arrive; the wait gives up, records
    code 16, and the block stops."""
    assert rtp.device_error() == 0
    out = torch.zeros(4, dtype=torch.int32, device="cuda")
    rtp.wait_selftest(1_000_000, out=out, kernel=1)  # first launch loads the kernel
    torch.cuda.synchronize()
    assert rtp.device_error() == 16
    out.zero_()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    rtp.wait_selftest(limit_ms * 1_000_000, out=out, kernel=1)
    e1.record()
    torch.cuda.synchronize()
    assert int(out[0]) == 1
    assert rtp.device_error() == 16
    assert rtp.device_error() == 0
    assert limit_ms <= e0.elapsed_time(e1) < 2.5 * limit_ms + 2
    # a reshard right after runs correctly
    x = torch.arange(64 * 1024, dtype=torch.float32, device="cuda").view(64, 1024)
    s0, s1 = rtp.spec_nd_sbp((4,), (("S", 0),)), rtp.spec_nd_sbp((4,), (("S", 1),))
    back = rtp.reshard(rtp.reshard(rtp.shard(x, s0), x.shape, s0, s1), x.shape, s1, s0)
    torch.cuda.synchronize()
    assert torch.equal(torch.cat(back, 0), x)
    assert rtp.device_error() == 0


def test_limit_outside_range_is_rejected():
    out = torch.zeros(4, dtype=torch.int32, device="cuda")
    for bad in (0, 999_999, 1_000_000_001):
        with pytest.raises(rtp.RtpError) as e:
            rtp.wait_selftest(bad, out=out)
        assert e.value.status == -1
