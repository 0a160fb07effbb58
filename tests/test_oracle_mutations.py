"""Plant plausible mistakes in copies of the oracle's C source and check that
the pins catch every one of them (no GPU needed).  The copies are compiled
into a temporary directory; the real oracle is untouched."""
import os

import pytest

import oracle
from oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "ssu_oracle.c")

# (name, text in ssu_oracle.c, replacement)
MUTATIONS = [
    ("drop_D_term", "y += Dh * xv;", "y += 0.0 * xv;"),
    ("y_from_old_state",
     "S[n] = S[n] * dA + d * xv * load_elem(pr->B, bc + n, pr->io_dtype);\n"
     "                        y += S[n] * load_elem(pr->C, bc + n, pr->io_dtype);",
     "y += S[n] * load_elem(pr->C, bc + n, pr->io_dtype);\n"
     "                        S[n] = S[n] * dA + d * xv * load_elem(pr->B, bc + n, pr->io_dtype);"),
    ("decay_sign", "exp(A * d)", "exp(-A * d)"),
    ("swap_B_C", "d * xv * load_elem(pr->B, bc + n", "d * xv * load_elem(pr->C, bc + n"),
    ("drop_x", "d * xv * load_elem", "d * load_elem"),
    ("softplus_sign", "log1p(exp(-fabs(v)))", "log1p(exp(fabs(v)))"),
    ("gate_sigmoid", "return z / (1.0 + exp(-z));", "return 1.0 / (1.0 + exp(-z));"),
    ("seed_off_by_one", "t_seed = pr->num_accepted[b] - 1;", "t_seed = pr->num_accepted[b];"),
    ("group_modulo", "const int64_t g = h / heads_per_group;", "const int64_t g = h % G;"),
    ("drop_bias", "+ bias;", "+ 0.0 * bias;"),
    ("pad_written",
     "if (!pr->disable_state_update && wslot[r] != pr->pad_slot_id)",
     "if (!pr->disable_state_update && wslot[r] >= 0)"),
    ("disable_ignored", "if (!pr->disable_state_update && wslot[r]", "if (wslot[r]"),
    ("per_row_as_strided", "return row_start + step;", "return b + step;"),
    ("per_row_seed_past_sequence", "rtab->mode == ORC_SLOTS_PER_ROW && t_seed >= len)",
     "rtab->mode == ORC_SLOTS_PER_ROW && t_seed >= len + 8)"),
    ("publish_seed_entry", "if (resolve(wtab, b, t, start[b], &w) != 0)",
     "if (resolve(wtab, b, 0, start[b], &w) != 0)"),
    ("bf16_truncates", "double r = round_to_format(v, 7, -126, 127);", "double r = trunc(v * 128.0) / 128.0;"),
    ("pad_reads_state", "S[n] = (seed[b] == pr->pad_slot_id)", "S[n] = (seed[b] < 0)"),
    ("replay_gamma_skips_current", "hist += w * d * xv * kq;\n                    w *= exp(A * d);",
     "hist += w * d * xv * kq;"),
    ("replay_fold_skips_buffer", "for (int64_t j = 0; j < c; ++j) {", "for (int64_t j = 0; j < 0; ++j) {"),
    ("replay_append_position", "const int64_t e = ((slot * Lb + c) * H + h) * P + p;",
     "const int64_t e = ((slot * Lb + c + 1) * H + h) * P + p;"),
    ("replay_count_not_reset", "pr->count_out[b] = (pad || fold) ? 0 : c + 1;",
     "pr->count_out[b] = pad ? 0 : c + 1;"),
    ("replay_decay_before_term", "hist += w * dj * xj * kq;\n                        w *= exp(A * dj);",
     "w *= exp(A * dj);\n                        hist += w * dj * xj * kq;"),
    ("dt_per_head_wrong_head", "const int64_t dti = pr->dt_per_head ? (r * H + h) : xi;",
     "const int64_t dti = pr->dt_per_head ? (r * H) : xi;"),
    # the low-precision read copy of the checkpoint
    ("read_copy_ignored", "sq += (pr->shadow_format != ORC_SHADOW_NONE", "sq += (0"),
    ("e4m3_scale_240", "round_to_format(amax / 448.0, 23", "round_to_format(amax / 240.0, 23"),
    ("e4m3_factor_240", "v[i] * 448.0 / amax", "v[i] * 240.0 / amax"),
    ("e4m3_signed_amax", "if (fabs(v[i]) > amax)\n            amax = fabs(v[i]);",
     "if (v[i] > amax)\n            amax = v[i];"),
    ("e4m3_two_fraction_bits", "double r = fabs(round_to_format(v, 3, -6, 8));",
     "double r = fabs(round_to_format(v, 2, -6, 8));"),
    ("fold_skips_read_copy",
     "if (pr->shadow_format != ORC_SHADOW_NONE) {\n                            /* the read copy",
     "if (0) {\n                            /* the read copy"),
    ("e4m3_no_saturation", "if (isinf(r) || r > 448.0)\n        r = 448.0;", ""),
    ("e4m3_exponent_bias", "ldexp((double)(f + 8), e - 10)", "ldexp((double)(f + 8), e - 11)"),
    # the NVFP4 read copy
    ("e2m1_exponent_bias", "ldexp(1.0 + 0.5 * f, e - 1)", "ldexp(1.0 + 0.5 * f, e - 2)"),
    ("e2m1_no_saturation", "if (isinf(r) || r > 6.0)\n        r = 6.0;", ""),
    ("e2m1_ties_away", "double r = fabs(round_to_format(v, 1, 0, 2));",
     "double r = fabs(round_to_format(v * (1.0 + 1e-12), 1, 0, 2));"),
    ("nvfp4_row_scale_448", "round_to_format(amax / (6.0 * 448.0), 23", "round_to_format(amax / 448.0, 23"),
    ("nvfp4_block_scale_undivided", "orc_e4m3_encode(bmax / (6.0 * (double)s))", "orc_e4m3_encode(bmax / (double)s)"),
    ("nvfp4_blocks_of_32", "for (int64_t k = 0; k < n / 16; ++k) {", "for (int64_t k = 0; k < n / 32; ++k) {"),
    ("nvfp4_nibble_order", "                if (i % 2 == 0)\n                    out[i / 2] = c;",
     "                if (i % 2 == 1)\n                    out[i / 2] = c;"),
    ("nvfp4_signed_block_max", "if (fabs(v[i]) > bmax)\n                    bmax = fabs(v[i]);",
     "if (v[i] > bmax)\n                    bmax = v[i];"),
    ("nvfp4_read_ignores_block_scale", "return orc_e2m1_decode(c) * orc_e4m3_decode(((const uint8_t *)(rec + 1))[i / 16]) * (double)rec[0];",
     "return orc_e2m1_decode(c) * 448.0 * (double)rec[0];"),
    # SSD prefill
    ("ssd_seq_idx_ignored", "if (c == 0 || pr->seq_idx[c] != pr->seq_idx[c - 1]) {", "if (c == 0) {"),
    ("ssd_dt_limit_dropped", "d = fmin(fmax(d, pr->dt_lo), pr->dt_hi);", "d = d;"),
    ("ssd_initial_ignored", "S[n] = pr->initial_states\n", "S[n] = 0 && pr->initial_states\n"),
    # speculative decoding on checkpoint + buffer
    ("verify_late_flush", "const int fold = !pad && c_in + 2 * T >= Lb;", "const int fold = !pad && c_in + T >= Lb;"),
    ("verify_commits_drafts", "        pr->count_out[b] = c;\n", "        pr->count_out[b] = c + T;\n"),
    ("verify_append_at_start", "const int64_t e = ((slot * Lb + c + k) * H + h) * P + p;",
     "const int64_t e = ((slot * Lb + k) * H + h) * P + p;"),
    ("verify_y_before_step",
     "S[n] = S[n] * a + d * xv * load_elem(pr->B, bc + n, pr->io_dtype);\n"
     "                        y += S[n] * load_elem(pr->C, bc + n, pr->io_dtype);",
     "y += S[n] * load_elem(pr->C, bc + n, pr->io_dtype);\n"
     "                        S[n] = S[n] * a + d * xv * load_elem(pr->B, bc + n, pr->io_dtype);"),
    ("verify_drafts_from_old_checkpoint", "load_elem(fold ? pr->ckpt_out : pr->ckpt_in, row * N + n",
     "load_elem(pr->ckpt_in, row * N + n"),
    ("ssd_decay_after_input",
     "S[n] = S[n] * a + d * xv * load_elem(pr->B, (t * G + g) * N + n, pr->io_dtype);",
     "S[n] = (S[n] + d * xv * load_elem(pr->B, (t * G + g) * N + n, pr->io_dtype)) * a;"),
]


@pytest.fixture(scope="module")
def src_text():
    with open(SRC) as f:
        return f.read()


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_mutation(name, old, new, src_text, tmp_path):
    assert src_text.count(old) >= 1, f"mutation {name}: pattern not found in the oracle source"
    mutated = src_text.replace(old, new)
    path = tmp_path / f"orc_{name}.c"
    path.write_text(mutated)
    lib = oracle.load_library(oracle.compile_source(str(path), str(tmp_path / f"lib_{name}.so")))
    caught = []
    for pin in ALL_PINS:
        try:
            pin(lib)
        except Exception as e:            # AssertionError, OracleError, ...
            caught.append(f"{pin.__name__}: {str(e)[:80]}")
    assert caught, f"no pin caught the planted mistake {name}"
