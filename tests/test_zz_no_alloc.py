"""rtp_tp_mlp_noalloc: the tensor-parallel MLP for callers that cannot allocate
device memory (code inside another runtime's memory pool, or a serving loop
with a fixed memory plan). The activations live in a static device array of
the library; the caller passes only X, the weight shards and Z.

The new entry point is called through the C ABI (ctypes, raw device pointers)
and compared, on two calls in a row with different sizes, with rtp_tp_mlp on
the same inputs and with the CPU oracle on sampled rows, both within the Z
bound the other MLP tests use (max |Z - Z_ref| <= 2e-2 sqrt(F/4096) RMS(Z_ref)).
It must pass in a fresh process and after the other tests (this file is
collected last).
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rtp():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from resharding_tensor_parallelism_gb300 import _build
    _build.build()
    import resharding_tensor_parallelism_gb300 as m
    return m


def _host_inputs(M, K, F, N, P, seed):
    X = synth.normal(seed, (M, K), "bf16")
    A = synth.normal(seed + 1, (K, F), "bf16", std=0.02)
    B = synth.normal(seed + 2, (F, N), "bf16", std=0.02)
    As = [np.ascontiguousarray(a) for a in np.split(A, P, axis=1)]
    Bs = [np.ascontiguousarray(b) for b in np.split(B, P, axis=0)]
    return X, As, Bs


def _inputs(M, K, F, N, P, seed):
    X, As, Bs = _host_inputs(M, K, F, N, P, seed)
    return to_dev(X), [to_dev(a) for a in As], [to_dev(b) for b in Bs]


def _noalloc_via_cabi(rtp, X, As, Bs, Z):
    lib = rtp.lib()
    P = len(As)
    M, K = X.shape
    F = As[0].shape[1] * P
    N = Bs[0].shape[1]
    ap = (ctypes.c_void_p * P)(*[a.data_ptr() for a in As])
    bp = (ctypes.c_void_p * P)(*[b.data_ptr() for b in Bs])
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream or None)
    return lib.rtp_tp_mlp_noalloc(P, M, K, F, N, ctypes.c_void_p(X.data_ptr()), ap, bp,
                                  ctypes.c_void_p(Z.data_ptr()), stream)


def test_noalloc_matches_tp_mlp_and_oracle_on_two_calls(rtp):
    for (M, K, F, N, P, seed) in [(512, 1024, 8192, 1024, 8, 70), (300, 256, 2048, 520, 4, 80)]:
        Xh, Ash, Bsh = _host_inputs(M, K, F, N, P, seed)
        X, As, Bs = to_dev(Xh), [to_dev(a) for a in Ash], [to_dev(b) for b in Bsh]
        Z_lib, _ = rtp.tp_mlp(X, As, Bs, mode=1)
        Z = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        rc = _noalloc_via_cabi(rtp, X, As, Bs, Z)
        assert rc == 0, rtp.last_error()
        torch.cuda.synchronize()
        z, zl = Z.double().cpu().numpy(), Z_lib.double().cpu().numpy()
        assert np.isfinite(z).all()
        tol = 2e-2 * np.sqrt(F / 4096) * np.sqrt(np.mean(zl ** 2))
        assert np.abs(z - zl).max() <= tol
        # the oracle (float64 from the same bf16 inputs, Y rounded to bf16) on
        # sampled rows: the first and last of each 128-row tile and a few more
        rows = np.array(sorted({0, 1, 127, 128, M // 2, M - 2, M - 1} | set(range(5, M, 37))))
        z_ref, _ = oracle.tp_mlp(Xh, Ash, Bsh, rows=rows)
        tol_ref = 2e-2 * np.sqrt(F / 4096) * np.sqrt(np.mean(z_ref ** 2))
        err = np.abs(z[rows] - z_ref).max()
        assert err <= tol_ref, "Z error %.3g against the oracle > %.3g" % (err, tol_ref)
    assert rtp.device_error() == 0


def test_noalloc_rejects_sizes_beyond_the_scratch(rtp):
    X, As, Bs = _inputs(1024, 64, 16384, 64, 8, 90)  # Y would need 32 MiB
    Z = torch.zeros((1024, 64), dtype=torch.float32, device="cuda")
    rc = _noalloc_via_cabi(rtp, X, As, Bs, Z)
    assert rc == -2 and "static scratch" in rtp.last_error()
    torch.cuda.synchronize()
    assert float(Z.abs().max()) == 0.0  # nothing was launched
