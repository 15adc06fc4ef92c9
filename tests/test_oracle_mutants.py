"""Each plausible slip, planted into a temporary copy of the oracle source, must
make at least one pin in test_oracle_pins fail.  The committed oracle is never
modified; the mutants are compiled into a temporary directory on the CPU."""

import ctypes
import os
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "rvq_oracle.cpp")

MUTANTS = {
    "residual_sign": ("residual[i] -= s;", "residual[i] += s;"),
    "transposed_w_in": ("s += (double)row[i] * residual[i];", "s += (double)Win[(size_t)i * d + j] * residual[i];"),
    "tie_to_highest": ("if (dist < d1) {", "if (dist <= d1) {"),
    "l1_metric": ("dist += t * t;", "dist += (t < 0 ? -t : t);"),
    "encode_drops_b_in": ("if (W.b_in) s +=", "if (false) s +="),
    "encode_drops_b_out": ("if (W.b_out) s +=", "if (false) s +="),
    "decode_drops_b_out": ("if (b_out) s +=", "if (false) s +="),
    "decode_stage_zero_weights": ("const float *Wout = w_out + (size_t)k * D * d;",
                                  "const float *Wout = w_out;"),
    "gap_over_d1": ("(d2 - d1) / d2", "(d2 - d1) / d1"),
    "second_best_not_tracked": ("} else if (dist < d2) {", "} else if (false) {"),
    "codeword_from_wrong_stage": ("const float *c = embed + (size_t)best * d;",
                                  "const float *c = W.codebook + (size_t)best * d;"),
    # the normalised metric
    "cosine_query_not_normalised": ("if (metric == 1) l2_normalise(e);", "(void)0;"),
    "cosine_codebook_not_normalised": ("if (metric == 1) l2_normalise(c_n);", "(void)0;"),
    "cosine_eps_added_to_norm": ("std::max(std::sqrt(ss), kNormEps)", "(std::sqrt(ss) + kNormEps)"),
    "cosine_residual_uses_normalised_codeword": (
        "for (int j = 0; j < d; ++j) s += (double)row[j] * (double)c[j];\n      if (W.b_out)",
        "double nn = 0; for (int j = 0; j < d; ++j) nn += (double)c[j] * c[j];\n"
        "      for (int j = 0; j < d; ++j) s += (double)row[j] * (double)c[j] / (metric == 1 ? std::sqrt(nn) : 1.0);\n"
        "      if (W.b_out)"),
    # the Linear layers around the quantizer
    "fc_bias_dropped": ("if (fc_b) s += (double)fc_b[i];", "if (false) s += (double)fc_b[i];"),
    "fc_transposed": ("for (int j = 0; j < D_in; ++j) s += (double)row[j] * (double)xn[j];",
                      "for (int j = 0; j < D_in; ++j) s += (double)fc_w[(size_t)j * D + i] * (double)xn[j];"),
    "fc2_bias_dropped": ("if (fc2_b) t += (double)fc2_b[i];", "if (false) t += (double)fc2_b[i];"),
    "fc2_transposed": ("for (int j = 0; j < D; ++j) t += (double)row[j] * acc[j];",
                       "for (int j = 0; j < D; ++j) t += (double)fc2_w[(size_t)j * D_out + i] * acc[j];"),
    # a stage index dropped (every stage reads stage 0's weights), the update skipped
    "encode_w_in_of_stage_zero": ("const float *Win = W.w_in + (size_t)k * d * D;", "const float *Win = W.w_in;"),
    "encode_b_in_of_stage_zero": ("s += (double)W.b_in[(size_t)k * d + j];", "s += (double)W.b_in[j];"),
    "encode_b_out_of_stage_zero": ("if (W.b_out) s += (double)W.b_out[(size_t)k * D + i];",
                                   "if (W.b_out) s += (double)W.b_out[i];"),
    "residual_not_updated": ("residual[i] -= s;", "(void)s;"),
    "decode_codebook_of_stage_zero": ("const float *e = codebook + ((size_t)k * K + code) * d;",
                                      "const float *e = codebook + (size_t)code * d;"),
    "decode_b_out_of_stage_zero": ("if (b_out) s += (double)b_out[(size_t)k * D + i];",
                                   "if (b_out) s += (double)b_out[i];"),
    # bad decode codes: read as row 0 instead of skipped, or skipped without counting
    "decode_bad_code_read_as_row_zero": ("bad_per_frame[(size_t)n] += 1;\n          continue;",
                                         "bad_per_frame[(size_t)n] += 1;\n          code = 0;"),
    "decode_bad_code_not_counted": ("bad_per_frame[(size_t)n] += 1;", "(void)0;"),
    # the reported best distance is the runner-up's
    "best_dist_is_second": ("if (best_dist) best_dist[k] = d1;", "if (best_dist) best_dist[k] = d2;"),
}

PINS = [
    pins.test_balanced_ternary_digits_closed_form,
    pins.test_gap_and_distance_closed_form,
    lambda: pins.test_planted_recovery_exact(True),
    pins.test_planted_recovery_with_noise,
    pins.test_single_stage_identity_is_nearest_neighbour,
    lambda: pins.test_integer_instances_argmin_certificate(0),
    lambda: pins.test_integer_instances_argmin_certificate(1),
    pins.test_duplicate_rows_take_lowest_index,
    pins.test_decode_is_sum_of_single_stage_decodes,
    pins.test_decode_scaling_bias_and_prefix,
    pins.test_decode_counts_and_skips_bad_codes,
    pins.test_input_bias_is_a_codebook_shift,
    pins.test_cosine_closed_form_2d,
    pins.test_cosine_eps_clamps_small_vectors,
    pins.test_cosine_single_stage_is_scipy_cosine_neighbour,
    pins.test_cosine_scale_invariance_of_one_stage,
    pins.test_cosine_planted_recovery_exact,
    pins.test_fc_maps_frames_before_the_loop,
    pins.test_fc2_maps_the_decoded_sum,
]


def _build_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutated = src.replace(old, new)
    path = tmp_path / f"{name}.cpp"
    path.write_text(mutated)
    lib = tmp_path / f"lib{name}.so"
    subprocess.run(["g++", "-O1", "-std=c++17", "-shared", "-fPIC", "-pthread", "-ffp-contract=off",
                    "-o", str(lib), str(path)], check=True)
    return str(lib)


def _configure(lib):
    f = ctypes.c_void_p
    lib.rvq_oracle_encode.argtypes = [ctypes.c_int] * 4 + [f] * 6 + [ctypes.c_int64, ctypes.c_int] + [f] * 4 + [ctypes.c_int]
    lib.rvq_oracle_encode.restype = ctypes.c_int
    lib.rvq_oracle_encode_metric.argtypes = ([ctypes.c_int] * 4 + [f] * 6 + [ctypes.c_int64, ctypes.c_int] + [f] * 4
                                             + [ctypes.c_int, ctypes.c_int])
    lib.rvq_oracle_encode_metric.restype = ctypes.c_int
    lib.rvq_oracle_encode_ex.argtypes = ([ctypes.c_int] * 5 + [f] * 8 + [ctypes.c_int64, ctypes.c_int] + [f] * 4
                                         + [ctypes.c_int, ctypes.c_int])
    lib.rvq_oracle_encode_ex.restype = ctypes.c_int
    lib.rvq_oracle_decode_ex.argtypes = [ctypes.c_int] * 5 + [f] * 6 + [ctypes.c_int64, ctypes.c_int, f, f, ctypes.c_int]
    lib.rvq_oracle_decode_ex.restype = ctypes.c_int
    lib.rvq_oracle_decode.argtypes = [ctypes.c_int] * 4 + [f] * 4 + [ctypes.c_int64, ctypes.c_int, f, f, ctypes.c_int]
    lib.rvq_oracle_decode.restype = ctypes.c_int
    lib.rvq_oracle_version.restype = ctypes.c_char_p
    return lib


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path, monkeypatch):
    old, new = MUTANTS[name]
    lib = _configure(ctypes.CDLL(_build_mutant(tmp_path, name, old, new)))
    monkeypatch.setattr(oracle, "_lib", lib)
    failures = 0
    for pin in PINS:
        try:
            pin()
        except AssertionError:
            failures += 1
    assert failures > 0, f"no pin caught mutant {name}"


def test_unmutated_copy_passes_every_pin(tmp_path, monkeypatch):
    lib = _configure(ctypes.CDLL(_build_mutant(tmp_path, "identity", "rvq-oracle f64 3", "rvq-oracle f64 3")))
    monkeypatch.setattr(oracle, "_lib", lib)
    for pin in PINS:
        pin()
