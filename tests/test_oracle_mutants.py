"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a copy of the oracle's source (on the CPU,
never in the CUDA path): the split order, the uneven-split rule, a dropped
partial, a lost partial mesh dim, the GELU scale, a dropped GELU' term, a
transposed operand, the wrong gradient in a product, a dropped rank, the
broadcast rule's intersection, the reshape rule's surviving member, the bf16
tie rule, the partial-max identity, whose SBP the CopyCost reads, and the
ONNX device placement. It builds that copy, points the oracle module at
it, and checks that at least one of the named pin tests fails.
"""
import os
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.cpp")

MUTANTS = [
    ("inner mesh dim split first",
     "    for (int d = 0; d < L.mesh_ndim; ++d) {\n        if (L.kind[d] != 'S') continue;",
     "    for (int d = L.mesh_ndim - 1; d >= 0; --d) {\n        if (L.kind[d] != 'S') continue;",
     ["test_uneven_split_sizes_and_nesting", "test_onnx_sharding_examples"]),
    ("floor-sized pieces",
     "        int64_t width = (len + n - 1) / n;",
     "        int64_t width = std::max<int64_t>(1, len / n);",
     ["test_uneven_split_sizes_and_nesting", "test_pieces_tile_tensor_in_device_order"]),
    ("a partial member dropped",
     "            else acc += v;",
     "            else if (dev > 0) acc += v;",
     ["test_partial_sum_against_numpy", "test_partial_shard_is_exact_and_sums_back"]),
    ("contraction leaves no partial",
     "        if (outs.find(ch) == std::string::npos && letter_dim[ch - 'a'] != -1) partial |= 1u << letter_dim[ch - 'a'];",
     "        if (outs.find(ch) == std::string::npos && letter_dim[ch - 'a'] != -1) partial |= 0u;",
     ["test_infer_spmd_contraction_leaves_partial", "test_infer_spmd_by_execution"]),
    ("GELU without the 1/sqrt(2)",
     "double oracle_gelu(double x) { return 0.5 * x * (1.0 + std::erf(x / std::sqrt(2.0))); }",
     "double oracle_gelu(double x) { return 0.5 * x * (1.0 + std::erf(x)); }",
     ["test_gelu_closed_forms", "test_tp_mlp_gelu_commutes_with_column_split"]),
    ("GELU' without h phi(h)",
     "+ x * std::exp(-0.5 * x * x) / std::sqrt(2.0 * pi);",
     "+ 0.0 * x;",
     ["test_gelu_grad_is_the_derivative_of_gelu", "test_tp_mlp_backward_matches_finite_differences"]),
    ("A read transposed in the forward",
     "                for (int64_t f = 0; f < Fp; ++f) y[f] += x[k] * bf16_bits_to_double(arow[f]);",
     "                for (int64_t f = 0; f < Fp; ++f) y[f] += x[k] * bf16_bits_to_double(A[i][f * K + k]);",
     ["test_tp_mlp_identity_equals_xab"]),
    ("dA built from dY instead of dH",
     "            for (int64_t k = 0; k < K; ++k) da[k] += bf16_bits_to_double(X[m * K + k]) * g;",
     "            for (int64_t k = 0; k < K; ++k) da[k] += bf16_bits_to_double(X[m * K + k]) * dy;",
     ["test_tp_mlp_backward_matches_finite_differences"]),
    ("dX misses the last rank",
     "            for (int64_t f = 0; f < F; ++f) acc += dh[f] * a_at(k, f);",
     "            for (int64_t f = 0; f < F - Fp; ++f) acc += dh[f] * a_at(k, f);",
     ["test_tp_mlp_backward_matches_finite_differences"]),
    ("broadcast rule ignores what a device holds",
     "                    if (i < L[dk] || i >= H[dk]) ok = false;",
     "                    if (i < L[dk] && i >= H[dk]) ok = false;",
     ["test_broadcast_rule_page_examples", "test_broadcast_rule_by_execution"]),
    ("reshape keeps the innermost member's split",
     "        int li = i0, lo = o0;\n        while (li < i - 1 && in_shape[li] == 1) ++li;\n"
     "        while (lo < o - 1 && out_shape[lo] == 1) ++lo;",
     "        int li = i - 1, lo = o - 1;",
     ["test_reshape_rule_by_brute_force", "test_reshape_configuration_cases", "test_paddle_dimtrans_examples"]),
    ("bf16 ties rounded away from zero",
     "        double r = std::nearbyint(x / q) * q;",
     "        double r = std::round(x / q) * q;",
     ["test_bf16_rounding_special_values", "test_bf16_rounding_matches_torch_on_floats"]),
    ("partial max padded with +inf",
     "    if (reduction == 'X') return -INFINITY;",
     "    if (reduction == 'X') return INFINITY;",
     ["test_shard_to_partial_min_max_holds_identity", "test_partial_min_max_against_numpy"]),
    ("CopyCost read from the candidate, not the input",
     "                if (k != 'S') partial_or_broadcast = true;",
     "                if (c.dims[d].first != 'S') partial_or_broadcast = true;",
     ["test_sbp_signature_page_examples", "test_sbp_signature_invariants"]),
    ("ONNX devices placed group by group transposed",
     "        for (int64_t t = 0; t < gsize; ++t) L.devices[s * gsize + t] = (int32_t)members[s][t];",
     "        for (int64_t t = 0; t < gsize; ++t) L.devices[t * n_device + s] = (int32_t)members[s][t];",
     ["test_onnx_sharding_examples", "test_split_broadcast_follows_rule_not_printed_value"]),
]


@pytest.fixture(scope="module")
def restore_oracle():
    saved = (oracle._SRC, oracle._LIB, oracle._lib)
    yield
    oracle._SRC, oracle._LIB, oracle._lib = saved


def _run_pin(name, golden_dir):
    fn = getattr(pins, name)
    args = {"golden_dir": golden_dir} if "golden_dir" in fn.__code__.co_varnames[:fn.__code__.co_argcount] else {}
    for mark in getattr(fn, "pytestmark", []):  # a parametrized pin: run every parameter set
        if mark.name == "parametrize":
            for params in mark.args[1]:
                fn(params, **args)
            return
    fn(**args)


@pytest.mark.parametrize("what,old,new,tests", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(what, old, new, tests, tmp_path, golden_dir, restore_oracle):
    src = open(SRC).read()
    assert src.count(old) == 1, "mutation site not found: " + what
    mutant = tmp_path / "oracle_mutant.cpp"
    mutant.write_text(src.replace(old, new))
    lib = tmp_path / "oracle_mutant.so"
    subprocess.check_call(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", str(mutant), "-o", str(lib)])
    oracle._SRC, oracle._LIB, oracle._lib = str(mutant), str(lib), None
    caught = []
    for name in tests:
        try:
            _run_pin(name, golden_dir)
        except (AssertionError, RuntimeError, ValueError, IndexError) as e:
            caught.append((name, type(e).__name__))
    oracle._lib = None
    assert caught, "no pin caught: " + what
