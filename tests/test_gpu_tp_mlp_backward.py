"""GPU parity of the tensor-parallel MLP backward pass (ColossalAI "1D tensor
parallelism" page, section 2.2) against the CPU oracle.

The training forward keeps H_i = bf16(X A_i); the backward forms
dH_i = bf16(dZ B_i^T * GELU'(H_i)), dX = sum_i dH_i A_i^T, dA_i = X^T dH_i and
dB_i = Y_i^T dZ with float32 accumulation. The oracle works in float64 from the
same bf16 inputs and rounds H, Y and dH to bf16 where the kernels store them.

Bounds:
  * H: one bf16 spacing of the float64 pre-activation h plus the float32
    accumulation bound 1.2 K 2^-24 sum_k |x a| (call the total eH);
  * dH, per element: one bf16 spacing of the float64 value, plus
    |dY| * 0.8 * (eH + spacing(H)) (the kernel's H and the oracle's rounded H
    differ by at most that, and |GELU''| <= 0.8), plus |GELU'(H)| * 1.2 N 2^-24 sum_n |dz b| (float32
    accumulation of dY);
  * dX, dA, dB: max |got - ref| <= TOL * max(1, sqrt(K_eff / 4096)) * RMS(ref),
    with K_eff the length of the contraction (the form of the forward's Z
    bound). The error comes mostly from elements of dH or Y that rounded to the
    neighbouring bf16 value: float32 sums of N terms with random signs carry a
    relative error of order N 2^-24, so a few percent of them land across a
    bf16 rounding boundary; each such element moves one term by one bf16
    spacing. Measured: 1e-7 (tiny case) to 4e-3 of RMS. A dropped K-block or
    a wrong GELU' term costs far more than the tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import Guarded, as_f64, bf16_ulp, to_dev, to_host

pytestmark = pytest.mark.gpu

TOL = 2e-2

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
    dZ = synth.normal(seed + 3, (M, N), "bf16")
    As = [np.ascontiguousarray(a) for a in np.split(A, P, axis=1)]
    Bs = [np.ascontiguousarray(b) for b in np.split(B, P, axis=0)]
    return X, As, Bs, dZ


def _run(X, As, Bs, dZ, mode=1, second_stream=False):
    """Training forward then backward on the GPU, every output in a guarded
    buffer (writes outside them are caught); everything back on the host."""
    Xd, Ad, Bd, dZd = to_dev(X), [to_dev(a) for a in As], [to_dev(b) for b in Bs], to_dev(dZ)
    P, (M, K), Fp, N = len(As), X.shape, As[0].shape[1], Bs[0].shape[1]
    g = Guarded()
    bf, f32 = torch.bfloat16, torch.float32
    Z, Y, H = rtp.tp_mlp_train_forward(Xd, Ad, Bd, Y=g.many([(M, Fp)] * P, bf, "Y"), H=g.many([(M, Fp)] * P, bf, "H"),
                                       Z=g.empty((M, N), f32, "Z"))
    s1 = torch.cuda.Stream() if second_stream else None
    dX, dA, dB, dH = rtp.tp_mlp_backward(
        Xd, Ad, Bd, H, Y, dZd, dH=g.many([(M, Fp)] * P, bf, "dH"),
        dX_partials=g.many([(M, K)] * P, f32, "dX_partials") if mode == 0 else None, dX=g.empty((M, K), f32, "dX"),
        dA=g.many([(K, Fp)] * P, f32, "dA"), dB=g.many([(Fp, N)] * P, f32, "dB"), mode=mode, s1=s1)
    g.check("training forward and backward, mode %d" % mode)
    h = lambda ts: [to_host(t) for t in ts]
    return {"Z": to_host(Z), "Y": h(Y), "H": h(H), "dX": to_host(dX), "dA": h(dA), "dB": h(dB), "dH": h(dH)}


def _rel_check(got, ref, k_eff, what):
    rms = np.sqrt(np.mean(ref ** 2))
    err = np.abs(got - ref).max()
    tol = TOL * max(1.0, np.sqrt(k_eff / 4096)) * rms
    assert err <= tol, "%s: max error %.3g > %.3g (RMS %.3g)" % (what, err, tol, rms)
    return err / rms


def _check(X, As, Bs, dZ, g, rows, cols, what=""):
    P = len(As)
    M, K = X.shape
    Fp = As[0].shape[1]
    N = Bs[0].shape[1]
    F = Fp * P
    ref = oracle.tp_mlp_backward(X, As, Bs, dZ, rows=rows, cols=cols, flags=7)
    # H: one bf16 spacing of the float64 pre-activation plus float32 accumulation
    ex = oracle.tp_mlp_backward(X, As, Bs, dZ, rows=rows, flags=6)  # H not rounded
    h_gpu = np.concatenate([as_f64(h[rows]) for h in g["H"]], axis=1)
    a_abs = np.abs(np.concatenate([as_f64(a) for a in As], axis=1))  # [K, F]
    e_h = bf16_ulp(ex["H"]) + 1.2 * K * 2.0 ** -24 * (np.abs(as_f64(X[rows])) @ a_abs)
    bad = np.abs(h_gpu - ex["H"]) > e_h
    assert not bad.any(), "%s: %d H elements outside the bound" % (what, bad.sum())
    # dH per element
    dh_gpu = np.concatenate([as_f64(d[rows]) for d in g["dH"]], axis=1)
    dz = np.abs(as_f64(dZ[rows]))
    b_abs = np.abs(np.concatenate([as_f64(b) for b in Bs], axis=0))  # [F, N]
    s_abs = dz @ b_abs.T
    gg = np.vectorize(oracle.gelu_grad)(ref["H"])
    bound = (bf16_ulp(ref["dH"]) + 0.8 * np.abs(ref["dY"]) * (e_h + bf16_ulp(ref["H"])) +
             np.abs(gg) * 1.2 * N * 2.0 ** -24 * s_abs + 1e-30)
    bad = np.abs(dh_gpu - ref["dH"]) > bound
    assert not bad.any(), "%s: %d dH elements outside the per-element bound" % (what, bad.sum())
    # dX rows, dA columns, dB rows of the sampled hidden units
    rx = _rel_check(g["dX"][rows].astype(np.float64), ref["dX"], F, what + " dX")
    da = np.stack([g["dA"][f // Fp][:, f % Fp] for f in cols]).astype(np.float64)
    db = np.stack([g["dB"][f // Fp][f % Fp, :] for f in cols]).astype(np.float64)
    ra = _rel_check(da, ref["dA"], M, what + " dA")
    rb = _rel_check(db, ref["dB"], M, what + " dB")
    return rx, ra, rb


def _cols(F, n, seed):
    base = [0, 1, 63, 64, 255, 256, F // 2, F - 1]
    rng = np.random.default_rng(seed)
    extra = list(rng.integers(0, F, size=max(0, n - len(base))))
    return np.array(sorted(set(int(c) for c in base + extra if c < F)))


def _rows(M, n, seed):
    base = [0, 1, 127, 128, 129, M // 2, M - 129, M - 128, M - 1]
    rng = np.random.default_rng(seed)
    extra = list(rng.integers(0, M, size=max(0, n - len(base))))
    return np.array(sorted(set(int(r) for r in base + extra if 0 <= r < M)))


def test_tiny_configuration():
    """X[4,8], A[8,16] in 2 column shards, B[16,8] in 2 row shards, dZ[4,8]; N(0,1)."""
    X, As, Bs, dZ = _inputs(4, 8, 16, 8, 2, seed=0, wstd=1.0)
    for mode in (1, 0):
        g = _run(X, As, Bs, dZ, mode)
        _check(X, As, Bs, dZ, g, np.arange(4), np.arange(16), "tiny mode %d" % mode)


@pytest.mark.parametrize("M,K,F,N,P", [(300, 200, 528, 520, 2), (128, 64, 2048, 256, 8), (384, 136, 288, 264, 3),
                                       (257, 1024, 1024, 512, 4), (64, 8, 16, 8, 1)])
def test_ragged_multi_tile(M, K, F, N, P):
    X, As, Bs, dZ = _inputs(M, K, F, N, P, seed=M + K, wstd=0.05)
    for mode, two in ((1, False), (0, False), (0, True)):
        g = _run(X, As, Bs, dZ, mode, second_stream=two)
        _check(X, As, Bs, dZ, g, np.arange(M), np.arange(F), "mode %d%s" % (mode, " two streams" if two else ""))


def test_train_forward_matches_inference_forward():
    """The training forward's Y and Z are the inference forward's, bit for bit."""
    X, As, Bs, _ = _inputs(300, 200, 528, 520, 2, seed=9)
    g = _run(X, As, Bs, np.zeros((300, 520), np.uint16))
    Z, Y = rtp.tp_mlp(to_dev(X), [to_dev(a) for a in As], [to_dev(b) for b in Bs], mode=1)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(g["Z"], to_host(Z))
    for a, b in zip(g["Y"], Y):
        np.testing.assert_array_equal(a, to_host(b))
    # dZ = 0: every gradient is zero
    assert not np.any(g["dX"]) and not any(np.any(d) for d in g["dA"] + g["dB"])
    assert not any(np.any(as_f64(d)) for d in g["dH"])


def test_no_tokens():
    """M = 0: dA and dB are zero (they are sums over no rows)."""
    dev = lambda *s: torch.zeros(s, dtype=torch.bfloat16, device="cuda")
    As, Bs = [dev(64, 32) for _ in range(2)], [dev(32, 16) for _ in range(2)]
    dA = [torch.full((64, 32), 7.0, device="cuda") for _ in range(2)]
    dB = [torch.full((32, 16), 7.0, device="cuda") for _ in range(2)]
    rtp.tp_mlp_backward(dev(0, 64), As, Bs, [dev(0, 32)] * 2, [dev(0, 32)] * 2, dev(0, 16), dA=dA, dB=dB)
    torch.cuda.synchronize()
    assert all(float(t.abs().max()) == 0.0 for t in dA + dB)


@pytest.fixture(scope="module")
def cfg4():
    return _inputs(8192, 4096, 16384, 4096, 8, seed=60)


def test_backward_configuration_full_size(cfg4):
    """X [8192,4096], A [4096,16384], B [16384,4096] N(0,0.02), dZ N(0,1), P = 8:
    sampled rows of dX and dH, sampled hidden units of dA and dB."""
    X, As, Bs, dZ = cfg4
    rows, cols = _rows(8192, 12, 1), _cols(16384, 12, 2)
    g1 = _run(X, As, Bs, dZ, 1)
    _check(X, As, Bs, dZ, g1, rows, cols, "full fused")
    g0 = _run(X, As, Bs, dZ, 0, second_stream=True)
    _check(X, As, Bs, dZ, g0, rows, cols, "full separate, overlapped")
    # the weight gradients do not depend on how dX is reduced; reruns are deterministic
    for k in ("dA", "dB", "dH"):
        for a, b in zip(g0[k], g1[k]):
            np.testing.assert_array_equal(a, b)
    g1b = _run(X, As, Bs, dZ, 1)
    np.testing.assert_array_equal(g1b["dX"], g1["dX"])


@pytest.mark.parametrize("M,K,F,N,P", [(520, 264, 400, 144, 2), (1024, 512, 2048, 1024, 8)])
def test_overlapped_dx_sum_settings_give_identical_bits(M, K, F, N, P):
    """Mode 0 sums the dX partials in a kernel of its own beside the
    weight-gradient GEMMs on the same or a second stream (overlap 0, the
    default), or in the dX GEMM's epilogue (each output tile's ranks in turn
    on one cluster). The same
    float32 partials are added in rank order, so every way gives the same
    bits, and the weight gradients do not depend on it."""
    X, As, Bs, dZ = _inputs(M, K, F, N, P, seed=M + 11)
    rows, cols = _rows(M, 8, 3), _cols(F, 8, 4)
    base = None
    prev = rtp.tp_mlp_overlap(0)
    try:
        for setting in (0, 1):
            rtp.tp_mlp_overlap(setting)
            for second in (False, True):
                g = _run(X, As, Bs, dZ, 0, second_stream=second)
                if base is None:
                    _check(X, As, Bs, dZ, g, rows, cols, "separate dX sum")
                    base = g
                for k in ("dX", "dA", "dB", "dH"):
                    got, want = (g[k], base[k]) if k == "dX" else (np.stack(g[k]), np.stack(base[k]))
                    np.testing.assert_array_equal(got, want, err_msg="%s, sum in epilogue %d" % (k, setting))
    finally:
        rtp.tp_mlp_overlap(prev)


def test_argument_errors():
    dev = lambda *s: torch.zeros(s, dtype=torch.bfloat16, device="cuda")
    X = dev(256, 64)
    As, Bs = [dev(64, 128) for _ in range(2)], [dev(128, 64) for _ in range(2)]
    Hs = [dev(256, 128) for _ in range(2)]
    with pytest.raises(rtp.RtpError) as e:  # N not a multiple of 8
        rtp.tp_mlp_backward(X, As, [dev(128, 60)] * 2, Hs, Hs, dev(256, 60))
    assert e.value.status == -2
    with pytest.raises(rtp.RtpError) as e:  # misaligned dZ
        rtp.tp_mlp_backward(X, As, Bs, Hs, Hs, dev(256 * 64 + 1)[1:].view(256, 64))
    assert e.value.status == -1
    with pytest.raises(rtp.RtpError) as e:  # 9 ranks
        rtp.tp_mlp_backward(X, [dev(64, 8)] * 9, [dev(8, 64)] * 9, [dev(256, 8)] * 9, [dev(256, 8)] * 9,
                            dev(256, 64))
    assert e.value.status == -3
    with pytest.raises(rtp.RtpError) as e:  # mode 2
        rtp.tp_mlp_backward(X, As, Bs, Hs, Hs, dev(256, 64), mode=2)
    assert e.value.status == -1
