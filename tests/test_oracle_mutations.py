"""The oracle's pins must catch plausible mistakes (CPU only).

Each case plants one mistake in a copy of the oracle's C source, compiles the
copy, and runs the pins of ``test_oracle.py`` against it: at least one pin
must fail.  Nothing here touches a GPU.
"""
import os
import tempfile

import pytest

import oracle
import test_oracle as pins
from conftest import read_golden

SRC = os.path.join(os.path.dirname(oracle.__file__), "vq_oracle.c")

MUTATIONS = {
    # fused multiply-add instead of a separate multiply and add
    "fma": ("float sq = d * d;\n        dist = dist + sq;",
            "dist = fmaf(d, d, dist);"),
    # sum the squares in descending i
    "descending_sum": ("for (int32_t i = 0; i < sub_dim; ++i) {\n        float d",
                       "for (int32_t i = sub_dim - 1; i >= 0; --i) {\n        float d"),
    # ties go to the highest index
    "tie_rule": ("if (dist < best) {", "if (dist <= best) {"),
    # one coordinate dropped from the distance
    "dropped_term": ("for (int32_t i = 0; i < sub_dim; ++i) {\n        float d",
                     "for (int32_t i = 1; i < sub_dim; ++i) {\n        float d"),
    # codebook read with a transposed stride
    "transposed_codebook": ("cb + (size_t)c * (size_t)sub_dim * es",
                            "cb + (size_t)c * es"),
    # wrong group for grouped rows
    "wrong_group": ("const int64_t g = n / n_per_group;",
                    "const int64_t g = n % (n_per_group ? n_per_group : 1) % 2;"),
    # fp16 exponent bias off by one
    "f16_bias": ("(int)e - 25", "(int)e - 24"),
    # bf16 read from the wrong half
    "bf16_half": ("(uint32_t)b << 16", "(uint32_t)b << 15"),
    # the running best starts at a finite value
    "finite_init": ("float best = INFINITY;", "float best = 1e30f;"),
    # squared difference replaced by absolute difference
    "abs_distance": ("float sq = d * d;", "float sq = fabsf(d);"),
    # smoothing multiplies instead of dividing
    "smooth_multiply": ("xs[i] = load_elem(xn, dtype, i) / f[i];",
                        "xs[i] = load_elem(xn, dtype, i) * f[i];"),
    # smoothing reads the factors of the wrong channel block
    "smooth_block": ("% (head_dim / sub_dim);", "/ (head_dim / sub_dim) % (head_dim / sub_dim);"),
    # every group smoothed with group 0's factors
    "smooth_group": ("smooth + (size_t)g * (size_t)head_dim", "smooth + 0 * (size_t)g"),
}


def _pins(lib):
    """Every pin of test_oracle.py, bound to one oracle library."""
    yield lambda: pins.test_f16_decode_matches_numpy_for_every_bit_pattern(lib)
    yield lambda: pins.test_bf16_decode_matches_torch_for_every_bit_pattern(lib)
    for row in read_golden("distance_rounding.txt"):
        yield lambda row=row: pins.test_distance_golden_rounding(lib, row)
    yield lambda: pins.test_distance_exact_on_small_integers(lib)
    yield lambda: pins.test_distance_within_fp32_error_bound_of_exact(lib)
    yield lambda: pins.test_encode_exact_integers_with_ties(lib)
    for dt in ("f16", "bf16", "f32"):
        yield lambda dt=dt: pins.test_encode_brute_force_float64(lib, dt, 4)
    yield lambda: pins.test_exact_copies_map_to_first_equal_row(lib)
    yield lambda: pins.test_duplicated_rows_resolve_to_lower_index(lib)
    yield lambda: pins.test_single_centroid_encodes_everything_to_zero(lib)
    yield lambda: pins.test_sub_dim_one_reduces_to_boundary_count(lib)
    yield lambda: pins.test_permuting_codebook_rows_permutes_indices(lib)
    yield lambda: pins.test_chunking_grouping_and_threads_do_not_change_results(lib)
    yield lambda: pins.test_special_values(lib)
    yield lambda: pins.test_smooth_ones_is_the_plain_encode(lib)
    yield lambda: pins.test_smooth_equals_encoding_numpy_divided_rows(lib)
    yield lambda: pins.test_smooth_by_powers_of_two_scales_the_codebook(lib)
    yield lambda: pins.test_smooth_factors_are_per_group(lib)


def test_unmutated_source_passes_every_pin():
    lib = oracle.default()
    for pin in _pins(lib):
        pin()


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name):
    before, after = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(before) == 1, f"mutation anchor for {name} not found exactly once"
    with tempfile.TemporaryDirectory() as tmp:
        path = os.path.join(tmp, "mutant.c")
        with open(path, "w") as f:
            f.write(src.replace(before, after))
        lib = oracle.OracleLib(oracle.compile_source(path, os.path.join(tmp, "mutant.so")))
        caught = 0
        for pin in _pins(lib):
            try:
                pin()
            except (AssertionError, RuntimeError, ValueError):
                caught += 1
                break
        assert caught, f"no pin caught the '{name}' mutation"


# ---- decode attention (Python oracle): mutate the function's source, run the
# pins of test_oracle_attention.py against the mutant

ATTENTION_MUTATIONS = {
    # query head h reads KV head h % Hkv instead of h // (Hq / Hkv)
    "gqa_interleave": ("out[bi, h * qpk + g] =", "out[bi, g * hkv + h] ="),
    # the first `window` tokens instead of the last
    "window_first": ("first = t - window if", "first = window if"),
    # default scale 1/D instead of 1/sqrt(D)
    "scale_default": ("1.0 / np.sqrt(d)", "1.0 / d"),
    # softmax without the maximum subtracted
    "no_max_shift": ("np.exp(logits - logits.max())", "np.exp(logits)"),
    # weights not normalised
    "no_normalise": ("(p / p.sum()) @ vals", "p @ vals"),
    # scores against the values
    "keys_values_swapped": ("logits = scale * (keys @ q", "logits = scale * (vals @ q"),
    # keys decoded with the value codebook
    "key_codebook": ("np.asarray(k_codebooks)[h:h + 1]", "np.asarray(v_codebooks)[h:h + 1]"),
}


def _mutant_attention(before, after):
    import inspect
    import textwrap

    src = textwrap.dedent(inspect.getsource(oracle.attention_decode))
    assert src.count(before) == 1, f"mutation anchor {before!r} not found exactly once"
    namespace = dict(vars(oracle))
    exec(compile(src.replace(before, after), "<mutant>", "exec"), namespace)
    return namespace["attention_decode"]


def test_unmutated_attention_passes_every_pin():
    import test_oracle_attention as apins

    for pin in apins.PINS:
        pin(oracle.attention_decode)


@pytest.mark.parametrize("name", sorted(ATTENTION_MUTATIONS))
def test_attention_mutation_is_caught(name):
    import test_oracle_attention as apins

    fn = _mutant_attention(*ATTENTION_MUTATIONS[name])
    caught = 0
    for pin in apins.PINS:
        try:
            pin(fn)
        except (AssertionError, FloatingPointError, ValueError, IndexError):
            caught += 1
            break
    assert caught, f"no pin caught the '{name}' mutation"


# ---- sibling encoders (scalar quantize, Hadamard rotation) in the C source

SIBLING_MUTATIONS = {
    # ties go to the higher index
    "scalar_tie": ("if (dist < best_dist) {", "if (dist <= best_dist) {"),
    # the value is rounded to fp16 precision before the subtraction
    "scalar_half": ("float d = val - centroids[j];",
                    "float d = (float)(_Float16)val - centroids[j];"),
    # butterfly with the difference the wrong way round
    "butterfly_sign": ("v[e + stride] = a - b;", "v[e + stride] = b - a;"),
    # the random sign flip dropped
    "no_diag": ("load_elem(x, dtype, row * dim + e) * diag[e];",
                "load_elem(x, dtype, row * dim + e);"),
    # the butterfly pairs elements one stride too far
    "butterfly_partner": ("const float a = v[e], b = v[e + stride];",
                          "const float a = v[e], b = v[(e + 2 * stride) % dim];"),
    # scaling skipped
    "no_scale": ("v[e] = v[e] * scale;", "v[e] = v[e];"),
}


@pytest.mark.parametrize("name", sorted(SIBLING_MUTATIONS))
def test_sibling_mutation_is_caught(name):
    import test_oracle_siblings as spins

    before, after = SIBLING_MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(before) == 1, f"mutation anchor for {name} not found exactly once"
    with tempfile.TemporaryDirectory() as tmp:
        path = os.path.join(tmp, "mutant.c")
        with open(path, "w") as f:
            f.write(src.replace(before, after))
        lib = oracle.OracleLib(oracle.compile_source(path, os.path.join(tmp, "mutant.so")))
        caught = 0
        for pin in spins.PINS:
            try:
                pin(lib)
            except (AssertionError, RuntimeError, ValueError):
                caught += 1
                break
        assert caught, f"no pin caught the '{name}' mutation"


def test_unmutated_sibling_source_passes_every_pin():
    import test_oracle_siblings as spins

    lib = oracle.default()
    for pin in spins.PINS:
        pin(lib)
