"""GPU parity of the tensor-parallel MLP (tcgen05 GEMMs) against the CPU oracle.

Bounds (bf16 inputs, float32 accumulation):
  * Z: max |Z - Z_ref| <= 2e-2 * sqrt(F / 4096) * RMS(Z_ref)   (K_eff = F)
  * Y: max |Y - Y_ref| <= 2e-2 * sqrt(K / 4096) * RMS(Y_ref) on the rounded
    values, and per element |Y - y| <= ulp_bf16(y) + 1.2 K 2^-24 sum_k |x_k a_k|
    against the unrounded float64 y (one rounding plus float32 accumulation).
The same seeded inputs feed both sides; Y_ref and Z_ref come from the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import Guarded, as_f64, bf16_ulp, to_dev, to_host

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


def _inputs(M, K, F, N, P, seed=0, wstd=0.02):
    X = synth.normal(seed, (M, K), "bf16")
    A = synth.normal(seed + 1, (K, F), "bf16", std=wstd)
    B = synth.normal(seed + 2, (F, N), "bf16", std=wstd)
    As = [np.ascontiguousarray(a) for a in np.split(A, P, axis=1)]
    Bs = [np.ascontiguousarray(b) for b in np.split(B, P, axis=0)]
    return X, As, Bs


def _gpu(X, As, Bs, mode, chunks=1, col_blocks=1, second_stream=False):
    """rtp.tp_mlp with Y, the partials and Z in guarded buffers (every write
    outside them is caught)."""
    s1 = torch.cuda.Stream() if second_stream else None
    P, (M, _), Fp, N = len(As), X.shape, As[0].shape[1], Bs[0].shape[1]
    g = Guarded()
    Y = g.many([(M, Fp)] * P, torch.bfloat16, "Y")
    parts = g.many([(M, N)] * P, torch.float32, "partials") if mode == 0 else None
    Z = g.empty((M, N), torch.float32, "Z")
    rtp.tp_mlp(to_dev(X), [to_dev(a) for a in As], [to_dev(b) for b in Bs], Y=Y, partials=parts, Z=Z, mode=mode,
               chunks=chunks, col_blocks=col_blocks, s1=s1)
    g.check("tp_mlp mode %d, %d chunks x %d blocks" % (mode, chunks, col_blocks))
    return to_host(Z), [to_host(y) for y in Y]


def _check(X, As, Bs, Z, Ys, rows, what=""):
    P = len(As)
    K = X.shape[1]
    F = sum(a.shape[1] for a in As)
    z_ref, y_ref = oracle.tp_mlp(X, As, Bs, rows=rows)
    # unrounded y and sum_k |x a| for the per-element bound
    _, y64 = oracle.tp_mlp(X, As, Bs, rows=rows, round_y=False)
    absX = X & np.uint16(0x7FFF)
    _, s_abs = oracle.tp_mlp(absX, [a & np.uint16(0x7FFF) for a in As], [b & np.uint16(0x7FFF) for b in Bs],
                             rows=rows, act="identity", round_y=False)
    y_gpu = np.concatenate([as_f64(y[rows]) for y in Ys], axis=1)
    z_gpu = Z[rows].astype(np.float64)
    z_err = np.abs(z_gpu - z_ref).max()
    z_tol = 2e-2 * np.sqrt(F / 4096) * np.sqrt(np.mean(z_ref ** 2))
    assert z_err <= z_tol, "%s: Z error %.3g > %.3g" % (what, z_err, z_tol)
    y_err = np.abs(y_gpu - y_ref).max()
    y_tol = 2e-2 * np.sqrt(K / 4096) * np.sqrt(np.mean(y_ref ** 2))
    bound = bf16_ulp(y64) + 1.2 * K * 2.0 ** -24 * s_abs
    bad = np.abs(y_gpu - y64) > bound
    assert not bad.any(), "%s: %d Y elements outside the per-element bound" % (what, bad.sum())
    assert y_err <= max(y_tol, np.max(bound)), "%s: Y error %.3g > %.3g" % (what, y_err, y_tol)
    return z_err / np.sqrt(np.mean(z_ref ** 2))


def test_tiny_configuration():
    """X[4,8] @ A[8,16] in 2 column shards, GELU, @ B[16,8] in 2 row shards; seed 0, N(0,1)."""
    X, As, Bs = _inputs(4, 8, 16, 8, 2, seed=0, wstd=1.0)
    for mode in (0, 1):
        Z, Ys = _gpu(X, As, Bs, mode)
        _check(X, As, Bs, Z, Ys, np.arange(4), "tiny mode %d" % mode)


@pytest.mark.parametrize("M,K,F,N,P", [(300, 200, 528, 520, 2), (128, 64, 2048, 256, 8), (384, 136, 288, 264, 3),
                                       (257, 1024, 1024, 512, 4), (520, 264, 392, 136, 1)])
def test_ragged_multi_tile(M, K, F, N, P):
    X, As, Bs = _inputs(M, K, F, N, P, seed=M + K)
    rows = np.arange(M)
    for mode in (0, 1):
        Z, Ys = _gpu(X, As, Bs, mode)
        _check(X, As, Bs, Z, Ys, rows, "mode %d" % mode)
    if M % 2 == 0 and N % 16 == 0:
        Z, Ys = _gpu(X, As, Bs, 0, chunks=2, col_blocks=2, second_stream=True)
        _check(X, As, Bs, Z, Ys, rows, "domino 2x2")


def _sample_rows(M, n):
    base = [0, 1, 127, 128, 129, M // 2, M - 129, M - 128, M - 1]
    rng = np.random.default_rng(M)
    extra = list(rng.integers(0, M, size=max(0, n - len(base))))
    return np.array(sorted(set(int(r) for r in base + extra)))


def test_column_edge_with_odd_chunk_count_is_stable():
    """Every output tile at the window's column edge stores an odd number of
    32-column chunks (F/P = 200: 7 chunks; N = 912: 5 in the last N tile), and
    each cluster takes several such tiles in a row (GEMM1 512 tiles, the mode 0
    partials 2048, for 76 clusters) with a one-block K loop, so the epilogue's
    staging buffers turn over as fast as they can. The buffers alternate by
    store, so a tile's first chunk never reuses the buffer of the store issued
    just before it. Every repetition is bit-identical to the first, and sampled
    rows match the oracle."""
    M, K, F, N, P = 16384, 64, 1600, 912, 8
    X, As, Bs = _inputs(M, K, F, N, P, seed=41)
    rows = _sample_rows(M, 12)
    for mode in (1, 0):
        Z0, Y0 = _gpu(X, As, Bs, mode)
        _check(X, As, Bs, Z0, Y0, rows, "odd column edge, mode %d" % mode)
        for rep in range(4):
            Z, Ys = _gpu(X, As, Bs, mode)
            assert np.array_equal(Z, Z0), "mode %d repetition %d: Z differs" % (mode, rep)
            assert all(np.array_equal(a, b) for a, b in zip(Ys, Y0)), "mode %d repetition %d: Y differs" % (mode, rep)


@pytest.fixture(scope="module")
def cfg4():
    return _inputs(8192, 4096, 16384, 4096, 8, seed=40)


def test_tp_mlp_configuration_full_size(cfg4):
    """X [8192,4096], A [4096,16384] and B [16384,4096] N(0,0.02), P = 8."""
    X, As, Bs = cfg4
    rows = _sample_rows(8192, 16)
    Zs = {}
    for mode in (1, 0):
        Z, Ys = _gpu(X, As, Bs, mode)
        _check(X, As, Bs, Z, Ys, rows, "full mode %d" % mode)
        Zs[mode] = Z
    # the Domino schedules sum the same partials in the same order: same bits
    for chunks, cb in ((2, 1), (4, 2)):
        Z, _ = _gpu(X, As, Bs, 0, chunks=chunks, col_blocks=cb, second_stream=True)
        np.testing.assert_array_equal(Z, Zs[0])
    # deterministic
    Z, _ = _gpu(X, As, Bs, 1)
    np.testing.assert_array_equal(Z, Zs[1])


def test_domino_configuration_full_size():
    """Llama-70B MLP shape: tokens 4096, hidden 8192, ffn 28672, P = 8; fused, and
    the Domino row split (2 and 4 chunks) with the 2D column split."""
    X, As, Bs = _inputs(4096, 8192, 28672, 8192, 8, seed=50)
    rows = _sample_rows(4096, 10)
    Z1, Ys = _gpu(X, As, Bs, 1)
    _check(X, As, Bs, Z1, Ys, rows, "fused")
    Z2, Ys2 = _gpu(X, As, Bs, 0, chunks=2, col_blocks=2, second_stream=True)
    _check(X, As, Bs, Z2, Ys2, rows, "domino 2 chunks, 2 column blocks")
    Z4, _ = _gpu(X, As, Bs, 0, chunks=4, col_blocks=1, second_stream=True)
    np.testing.assert_array_equal(Z4, Z2)


@pytest.mark.parametrize("M,K,F,N,P", [(520, 264, 400, 144, 2), (1024, 512, 2048, 1024, 8), (4096, 8192, 28672, 8192, 8)])
def test_domino_overlap_settings_give_identical_bits(M, K, F, N, P):
    """Mode 0 sums the rank partials in kernels of their own after each Domino
    window (overlap 0, the default), on the same or a second stream, or in the
    row-parallel GEMM's epilogue (each output tile's ranks in turn on one
    cluster).
    Every way adds the same float32 partials in rank order, so Z is
    bit-identical to the serial schedule (one chunk, one summing kernel after
    the GEMMs), whose Z is checked against the oracle, and the partials are
    the same everywhere."""
    X, As, Bs = _inputs(M, K, F, N, P, seed=M + N + 7)
    Xd, Ad, Bd = to_dev(X), [to_dev(a) for a in As], [to_dev(b) for b in Bs]
    prev = rtp.tp_mlp_overlap(0)
    try:
        parts0 = [torch.empty((M, N), dtype=torch.float32, device="cuda") for _ in range(P)]
        Zs, Ys = rtp.tp_mlp(Xd, Ad, Bd, partials=parts0, mode=0, chunks=1)
        torch.cuda.synchronize()
        want = to_host(Zs)
        want_parts = [to_host(p) for p in parts0]
        _check(X, As, Bs, want, [to_host(y) for y in Ys], _sample_rows(M, 8), "serial")
        for setting in (1, 0):
            rtp.tp_mlp_overlap(setting)
            for chunks, cb in ((1, 1), (2, 1), (2, 2), (4, 1), (4, 2)):
                for s1 in (None, torch.cuda.Stream()):
                    g = Guarded()  # every write stays inside Z and the partials
                    Z = g.empty((M, N), torch.float32, "Z")
                    parts = g.many([(M, N)] * P, torch.float32, "partials")
                    rtp.tp_mlp(Xd, Ad, Bd, Z=Z, partials=parts, mode=0, chunks=chunks, col_blocks=cb, s1=s1)
                    what = "sum in epilogue %d, %d chunks x %d blocks" % (setting, chunks, cb)
                    g.check(what)
                    np.testing.assert_array_equal(to_host(Z), want, err_msg=what)
                    for p, w in zip(parts, want_parts):
                        np.testing.assert_array_equal(to_host(p), w, err_msg=what + " partials")
    finally:
        rtp.tp_mlp_overlap(prev)
    assert rtp.device_error() == 0


def test_domino_overlap_setting_errors():
    with pytest.raises(rtp.RtpError) as e:
        rtp.tp_mlp_overlap(2)
    assert e.value.status == -1
    with pytest.raises(rtp.RtpError):
        rtp.tp_mlp_overlap(-1)
    assert rtp.tp_mlp_overlap(1) == 0  # the default: kernels of their own
    assert rtp.tp_mlp_overlap(0) == 1


def test_domino_from_two_host_threads():
    """Two host threads run the two-stream Domino schedule at once, each on its
    own pair of streams: each call orders its own second stream after its own
    GEMMs (the ordering events are per thread), so both keep producing the
    single-threaded result bit for bit."""
    import threading

    cases = [_inputs(512, 256, 1024, 512, 4, seed=s) for s in (500, 600)]
    dev_cases = [(to_dev(X), [to_dev(a) for a in As], [to_dev(b) for b in Bs]) for X, As, Bs in cases]
    want = []
    for X, As, Bs in dev_cases:
        Z, _ = rtp.tp_mlp(X, As, Bs, mode=0, chunks=2, col_blocks=2, s1=torch.cuda.Stream())
        torch.cuda.synchronize()
        want.append(Z.clone())
    errors = []

    def worker(k):
        try:
            torch.cuda.set_device(0)
            X, As, Bs = dev_cases[k]
            s0, s1 = torch.cuda.Stream(), torch.cuda.Stream()
            M, N = X.shape[0], Bs[0].shape[1]
            with torch.cuda.stream(s0):  # every allocation, fill and comparison ordered on s0
                Y = [torch.empty((M, As[0].shape[1]), dtype=torch.bfloat16, device="cuda") for _ in As]
                parts = [torch.empty((M, N), dtype=torch.float32, device="cuda") for _ in As]
                for it in range(40):
                    Z = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
                    rtp.tp_mlp(X, As, Bs, Y=Y, partials=parts, Z=Z, mode=0, chunks=2, col_blocks=2, s0=s0, s1=s1)
                    if not torch.equal(Z, want[k]):
                        errors.append("thread %d, call %d: Z differs" % (k, it))
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


def test_no_tokens():
    """M == 0: every form of the forward launches nothing and succeeds, with
    the token-row buffers empty (their data pointers are NULL)."""
    dev = lambda *s: torch.zeros(s, dtype=torch.bfloat16, device="cuda")
    As, Bs = [dev(64, 128) for _ in range(2)], [dev(128, 64) for _ in range(2)]
    for mode, chunks in ((1, 1), (0, 1), (0, 2)):
        Z, Y = rtp.tp_mlp(dev(0, 64), As, Bs, mode=mode, chunks=chunks, s1=torch.cuda.Stream())
        assert tuple(Z.shape) == (0, 64) and [tuple(y.shape) for y in Y] == [(0, 128)] * 2
    Zs, Y = rtp.tp_mlp_sp([dev(0, 64)] * 2, As, Bs)
    assert [tuple(z.shape) for z in Zs] == [(0, 64)] * 2
    assert tuple(rtp.tp_mlp_noalloc(dev(0, 64), As, Bs).shape) == (0, 64)
    torch.cuda.synchronize()
    assert rtp.device_error() == 0


def test_argument_errors():
    dev = lambda *s: torch.zeros(s, dtype=torch.bfloat16, device="cuda")
    X = dev(256, 64)
    As = [dev(64, 128) for _ in range(2)]
    Bs = [dev(128, 64) for _ in range(2)]
    with pytest.raises(rtp.RtpError) as e:  # M not divisible by chunks
        rtp.tp_mlp(dev(255, 64), As, Bs, mode=0, chunks=2)
    assert e.value.status == -2
    with pytest.raises(rtp.RtpError) as e:  # K not a multiple of 8
        rtp.tp_mlp(dev(256, 60), [dev(60, 128)] * 2, Bs)
    assert e.value.status == -2
    with pytest.raises(rtp.RtpError) as e:  # misaligned X
        rtp.tp_mlp(dev(256 * 64 + 1)[1:].view(256, 64), As, Bs)
    assert e.value.status == -1
    with pytest.raises(rtp.RtpError):  # 9 ranks
        rtp.tp_mlp(X, [dev(64, 8)] * 9, [dev(8, 64)] * 9)
    with pytest.raises(rtp.RtpError):  # column blocks need mode 0
        rtp.tp_mlp(X, As, Bs, mode=1, col_blocks=2)
    Z, _ = rtp.tp_mlp(X, As, Bs)
    torch.cuda.synchronize()
    assert float(Z.abs().max()) == 0.0


# ---- sequence parallelism (ColossalAI page, section 5.3) --------------------------

@pytest.mark.parametrize("M,K,F,N,P", [(256, 64, 512, 256, 2), (512, 200, 1056, 264, 4), (1024, 512, 2048, 512, 8),
                                       (128, 96, 264, 136, 1)])
def test_sequence_parallel_matches_oracle_and_fused(M, K, F, N, P):
    """X split by rows over the ranks in, Z split by rows over the ranks out;
    the all-gather and reduce-scatter are fused into the GEMMs."""
    X, As, Bs = _inputs(M, K, F, N, P, seed=M + 3 * K)
    Mr = M // P
    Xs = [np.ascontiguousarray(X[r * Mr:(r + 1) * Mr]) for r in range(P)]
    g = Guarded()  # every write outside Y and the Z shards is caught
    Zs, Ys = rtp.tp_mlp_sp([to_dev(x) for x in Xs], [to_dev(a) for a in As], [to_dev(b) for b in Bs],
                           Y=g.many([(M, F // P)] * P, torch.bfloat16, "Y"),
                           Z_shards=g.many([(Mr, N)] * P, torch.float32, "Z_shards"))
    g.check("sequence parallel")
    Z = np.concatenate([to_host(z) for z in Zs], axis=0)
    _check(X, As, Bs, Z, [to_host(y) for y in Ys], np.arange(M), "sequence parallel")
    # the same accumulation as the fused MLP on the gathered X: identical bits
    Zf, Yf = _gpu(X, As, Bs, 1)
    np.testing.assert_array_equal(Z, Zf)
    for a, b in zip(Ys, Yf):
        np.testing.assert_array_equal(to_host(a), b)


def test_sequence_parallel_full_size(cfg4):
    X, As, Bs = cfg4
    P, M = 8, 8192
    Mr = M // P
    Zs, Ys = rtp.tp_mlp_sp([to_dev(np.ascontiguousarray(X[r * Mr:(r + 1) * Mr])) for r in range(P)],
                           [to_dev(a) for a in As], [to_dev(b) for b in Bs])
    torch.cuda.synchronize()
    Z = np.concatenate([to_host(z) for z in Zs], axis=0)
    rows = _sample_rows(M, 12)
    _check(X, As, Bs, Z, [to_host(y) for y in Ys], rows, "sequence parallel full size")


def test_sequence_parallel_errors():
    dev = lambda *s: torch.zeros(s, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(rtp.RtpError) as e:  # M/P = 100 rows is not a multiple of 128
        rtp.tp_mlp_sp([dev(100, 64)] * 2, [dev(64, 256)] * 2, [dev(256, 64)] * 2)
    assert e.value.status == -2
