"""Plant plausible mistakes in a copy of the oracle (on the CPU) and check
that the pins catch every one of them.

Each mutant is a one-place edit of ``oracle/moe_oracle.c`` built into a
temporary library; at least one ``check_*`` in ``oracle_pins.py`` must fail on
it. This shows the pins constrain each step of the oracle (routing, dispatch,
gather, experts, combine, norm, dtype rounding), not only its happy path.
Mutants run inside the test process, so none may touch memory outside a
buffer: the mutated C code itself stays in bounds, and the oracle's Python
wrappers check every index array (dispatch maps, offsets) against the buffer
it indexes, so a mutant whose maps disagree with its offsets raises
ValueError instead of reading or writing past a buffer.
"""

import ctypes
import os
import subprocess

import pytest

import oracle
from oracle_pins import ALL_CHECKS

SRC = os.path.join(os.path.dirname(oracle.__file__), "moe_oracle.c")

# (name, text in moe_oracle.c, replacement)
MUTANTS = [
    ("tie_to_higher_id", "if (best < 0 || l[e] > l[best]) best = e;",
     "if (best < 0 || l[e] >= l[best]) best = e;"),
    ("no_renormalise", "sel[j] = sel[j] / z;", "sel[j] = sel[j];"),
    ("softmax_no_denominator", "p[e] = expf(l[e] - m) / s;",
     "p[e] = expf(l[e] - m);"),
    ("all_ninf_row_valid", "if (has_nan_or_pinf || all_ninf) {",
     "if (has_nan_or_pinf) {"),
    ("pinf_row_valid", "if (isnan(l[e]) || (isinf(l[e]) && l[e] > 0.0f))",
     "if (isnan(l[e]))"),
    ("silu_wrong_sign", "hv[i] = g / (1.0 + exp(-g)) * u;",
     "hv[i] = g / (1.0 + exp(g)) * u;"),
    ("gate_up_swapped", "hv[i] = g / (1.0 + exp(-g)) * u;",
     "hv[i] = u / (1.0 + exp(-u)) * g;"),
    ("silu_dropped_gate", "hv[i] = g / (1.0 + exp(-g)) * u;",
     "hv[i] = 1.0 / (1.0 + exp(-g)) * u;"),
    ("gate_transposed", "g += load_elem(gate, dt, wrow + k) * xr[k];",
     "g += load_elem(gate, dt, (e * H + k) * I + i) * xr[k];"),
    ("down_transposed", "acc += load_elem(down, dt, wrow + i) * hv[i];",
     "acc += load_elem(down, dt, (e * I + i) * H + o) * hv[i];"),
    ("combine_drops_first_slot",
     "for (int64_t j = 0; j < top_k; ++j) {\n                int64_t r",
     "for (int64_t j = 1; j < top_k; ++j) {\n                int64_t r"),
    ("combine_ignores_weight",
     "acc += load_elem(w, wdt, t * top_k + j) * load_elem(out_disp",
     "acc += 1.0 * load_elem(out_disp"),
    ("dispatch_src_is_token", "src_of[r] = (int32_t)a;",
     "src_of[r] = (int32_t)(a / top_k);"),
    ("gather_wrong_token", "int64_t t = src_of[r] / top_k;",
     "int64_t t = src_of[r] % top_k;"),
    ("offsets_short_by_one", "offsets[e + 1] = offsets[e] + counts[e];\n        next[e] = offsets[e];",
     "offsets[e + 1] = offsets[e] + counts[e] - (e + 1 == E);\n        next[e] = offsets[e];"),
    ("rows_reversed_in_expert", "int64_t r = next[e]++;",
     "int64_t r = offsets[e + 1] - 1 - (next[e]++ - offsets[e]);"),
    ("rms_mean_off_by_one", "ss / (double)H + (double)eps", "ss / (double)(H + 1) + (double)eps"),
    ("rms_eps_dropped", "ss / (double)H + (double)eps", "ss / (double)H"),
    ("rms_not_reciprocal", "double r = 1.0 / sqrt(", "double r = sqrt("),
    ("add_residual_dropped",
     "combine[t * H + h] + load_elem(residual, rdt, t * H + h)",
     "combine[t * H + h]"),
    ("bf16_truncates", "u += 0x7fffu + keep_lsb;", "u += 0u * keep_lsb;"),
    # group-limited sigmoid routing
    ("sg_weight_uses_corrected_score", "pick[j] = sc[best];", "pick[j] = c[best];"),
    ("sg_bias_subtracted", "c[e] = sc[e] + (bias ? bias[e] : 0.0f);",
     "c[e] = sc[e] - (bias ? bias[e] : 0.0f);"),
    ("sg_top_two_ignored", "gscore[g] = group_top_two ? first + second : first;",
     "gscore[g] = first;"),
    ("sg_top_two_always", "gscore[g] = group_top_two ? first + second : first;",
     "gscore[g] = first + second;"),
    ("sg_second_best_missed", "else if (c[e] > second) second = c[e];", "else second = second;"),
    ("sg_group_tie_to_higher_id", "if (best < 0 || gscore[g] > gscore[best]) best = g;",
     "if (best < 0 || gscore[g] >= gscore[best]) best = g;"),
    ("sg_expert_tie_to_higher_id", "if (best < 0 || c[e] > c[best]) best = e;",
     "if (best < 0 || c[e] >= c[best]) best = e;"),
    ("sg_groups_ignored", "if (taken[e] || !gkept[e / gs]) continue;", "if (taken[e]) continue;"),
    ("sg_scale_dropped", "(double)(pick[j] * scale)", "(double)(pick[j])"),
    ("sg_no_renormalise", "pick[j] = pick[j] / zsum;", "pick[j] = pick[j];"),
    ("sg_nan_row_valid", "if (isnan(c[e])) has_nan = 1;", "if (isnan(c[e])) has_nan = 0;"),
    # combine with special experts, shared expert and active mask
    ("cv2_zero_is_copy", "        } else if (id < E + zero_n) {\n                    o = 0.0;",
     "        } else if (id < E + zero_n) {\n                    o = load_elem(ori_x ? ori_x : out_disp, ori_x ? xdt : odt, t * H + h);"),
    ("cv2_copy_is_zero", "o = load_elem(ori_x, xdt, t * H + h);\n                } else if",
     "o = 0.0;\n                } else if"),
    ("cv2_const_alphas_swapped",
     "o = load_elem(alpha1, xdt, c) * load_elem(ori_x, xdt, t * H + h) +\n                        load_elem(alpha2, xdt, c)",
     "o = load_elem(alpha2, xdt, c) * load_elem(ori_x, xdt, t * H + h) +\n                        load_elem(alpha1, xdt, c)"),
    ("cv2_const_index_off", "const int64_t c = id - E - zero_n - copy_n;",
     "const int64_t c = (id - E - zero_n - copy_n + 1) % const_n;"),
    ("cv2_shared_unscaled", "if (shared_x) acc += sc * load_elem(shared_x, xdt, t * H + h);",
     "if (shared_x && j == 0) acc += load_elem(shared_x, xdt, t * H + h);"),
    ("cv2_mask2_ignored", "if (mask_dims == 2 && !mask[a]) continue;", "if (mask_dims == 3) continue;"),
    ("cv2_mask1_ignored", "if (mask_dims == 1 && !mask[t]) continue;", "if (mask_dims == 3) continue;"),
    ("cv2_invalid_id_is_zero", "                } else {\n                    acc = NAN;\n                    break;\n                }",
     "                } else {\n                    o = 0.0;\n                }"),
    ("sg_sigmoid_wrong_sign", "return (float)(1.0 / (1.0 + exp(-(double)x)));",
     "return (float)(1.0 / (1.0 + exp((double)x)));"),
    # first-order training
    ("rw_renorm_dropped", "double v = renormalize ? sel[j] / z : sel[j];", "double v = sel[j];"),
    ("rw_scale_dropped", "store_elem(w, wdt, t * top_k + j, v * scale);",
     "store_elem(w, wdt, t * top_k + j, v);"),
    ("rw_illegal_id_ignored",
     "if (e < 0 || e >= E) ok = 0;\n            else sel[j] = p[e];\n        }\n        if (!ok) {\n"
     "            for (int64_t j = 0; j < top_k; ++j) store_elem(w,",
     "if (e < 0 || e >= E) sel[j] = 0.0;\n            else sel[j] = p[e];\n        }\n        if (!ok) {\n"
     "            for (int64_t j = 0; j < top_k; ++j) store_elem(w,"),
    ("rw_sigmoid_wrong_sign", "p[e] = 1.0 / (1.0 + exp(-load_elem(logits, ldt, t * E + e)));",
     "p[e] = 1.0 / (1.0 + exp(load_elem(logits, ldt, t * E + e)));"),
    ("rw_softmax_unnormalised", "for (int64_t e = 0; e < E; ++e) p[e] /= s;",
     "for (int64_t e = 0; e < E; ++e) p[e] /= 1.0;"),
    ("rb_softmax_not_centred", "store_elem(dl, dldt, t * E + e, p[e] * (G[e] - c));",
     "store_elem(dl, dldt, t * E + e, p[e] * G[e]);"),
    ("rb_renorm_mean_dropped", "ds[j] = scale * (load_elem(gw, gwdt, t * top_k + j) - gbar) / z;",
     "ds[j] = scale * load_elem(gw, gwdt, t * top_k + j) / z;"),
    ("rb_renorm_not_divided", "ds[j] = scale * (load_elem(gw, gwdt, t * top_k + j) - gbar) / z;",
     "ds[j] = scale * (load_elem(gw, gwdt, t * top_k + j) - gbar);"),
    ("rb_sigmoid_derivative_short", "store_elem(dl, dldt, t * E + e, G[e] * p[e] * (1.0 - p[e]));",
     "store_elem(dl, dldt, t * E + e, G[e] * p[e]);"),
    ("rb_sigmoid_unselected_nan", "for (int64_t e = 0; e < E; ++e) store_elem(dl, dldt, t * E + e, 0.0);",
     "for (int64_t e = 0; e < E; ++e) store_elem(dl, dldt, t * E + e, 0.0 * p[e]);"),
    ("rb_scale_dropped", "ds[j] = scale * load_elem(gw, gwdt, t * top_k + j);",
     "ds[j] = load_elem(gw, gwdt, t * top_k + j);"),
    ("rb_repeat_overwrites", "G[idx[t * top_k + j]] += ds[j];", "G[idx[t * top_k + j]] = ds[j];"),
    ("cb_dw_uses_weight", "acc += g * load_elem(out_disp, odt, r * H + h);", "acc += g * wj;"),
    ("cb_dexpert_unweighted", "dexpert[r * H + h] = wj * g;", "dexpert[r * H + h] = g;"),
    ("sb_dsilu_short", "dgv[i] = dh * u * s * (1.0 + g * (1.0 - s));", "dgv[i] = dh * u * s;"),
    ("sb_du_sigmoid_only", "duv[i] = dh * g * s;", "duv[i] = dh * s;"),
    ("sb_gate_up_grads_swapped", "dgate[(e * I + i) * H + k] += dgv[i] * xr[k];",
     "dgate[(e * I + i) * H + k] += duv[i] * xr[k];"),
    ("sb_ddown_uses_dg", "ddown[(e * H + o) * I + i] += dor[o] * hv[i];",
     "ddown[(e * H + o) * I + i] += dor[o] * dgv[i];"),
    ("sb_dx_up_term_dropped",
     "acc += load_elem(gate, dt, (e * I + i) * H + k) * dgv[i] +\n"
     "                       load_elem(up, dt, (e * I + i) * H + k) * duv[i];",
     "acc += load_elem(gate, dt, (e * I + i) * H + k) * dgv[i];"),
    ("sb_dh_transposed", "dh += load_elem(down, dt, (e * H + o) * I + i) * dor[o];",
     "dh += load_elem(down, dt, ((e * H + o) * I + i + 1) % (E * H * I)) * dor[o];"),
    ("db_last_slot_only", "if (r >= 0) acc += load_elem(dinput, dt, r * H + h);",
     "if (r >= 0) acc = load_elem(dinput, dt, r * H + h);"),
]


def _build(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    c = tmp_path / f"{name}.c"
    c.write_text(src.replace(old, new))
    so = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", str(c), "-o",
                    str(so), "-lm"], check=True)
    return oracle.load_library(str(so))


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    lib = _build(tmp_path, name, old, new)
    caught = []
    for check in ALL_CHECKS:
        try:
            check(lib)
        except (AssertionError, ValueError, IndexError):
            caught.append(check.__name__)
    assert caught, f"no pin catches mutant {name}"


def test_wrappers_reject_out_of_range_indices():
    """Index arrays that point past their buffers are refused before any C
    code runs (the shape of the short-offsets mutant's maps)."""
    import numpy as np
    rows, H, k = 5, 4, 2
    out = np.zeros((rows, H))
    w = np.full((3, k), 0.5)
    gy = np.zeros((3, H))
    bad_row_of = np.array([0, 1, 2, 3, 4, rows], dtype=np.int32)
    with pytest.raises(ValueError):
        oracle.combine(out, "f64", w, "f64", bad_row_of, k)
    with pytest.raises(ValueError):
        oracle.combine_backward(out, "f64", w, "f64", bad_row_of, gy, "f64", k)
    with pytest.raises(ValueError):
        oracle.dispatch_backward(out, "f64", bad_row_of, k)
    with pytest.raises(ValueError):
        oracle.gather(np.zeros((2, H), np.float32), "f32", k, np.array([0, 1, 4], np.int32), 3)
    gate = np.zeros((2, 3, H), np.float32)
    down = np.zeros((2, H, 3), np.float32)
    with pytest.raises(ValueError):
        oracle.experts_dispatched(np.zeros((4, H), np.float32), "f32",
                                  np.array([0, 3, 5], np.int32), gate, gate, down)
    with pytest.raises(ValueError):
        oracle.experts_cache_dispatched(np.zeros((4, H), np.float32), "f32",
                                        np.array([0, 3, 2], np.int32), gate, gate)
