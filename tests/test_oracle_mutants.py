"""Mutation check of the oracle's pins.

Each case plants one plausible mistake in a copy of the C oracle (a dropped
term, a wrong operand, a missing clamp), builds that copy with the oracle's
own flags under ``oracle/_build/mutants``, and runs the oracle's pin tests
against it through ``FP8OPT_ORACLE_LIB``.  Every case must make at least one
pin fail; a mistake that no pin catches would be a hole in the pins.  The
unchanged source, built the same way, must pass them all, so a failure is
the planted mistake's and not the harness's.  CPU only.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "fp8opt_oracle.c")
OUT = os.path.join(ROOT, "oracle", "_build", "mutants")

PINS = ("codec", "cast", "step", "reduce", "clip")

# (name, text in the oracle, planted replacement, pin file tried first)
MUTANTS = [
    # OCP 8-bit formats (TransformerEngine issue #131; the formats' definition)
    ("round_half_away", "return rint(a / q) * q;", "return floor(a / q + 0.5) * q;",
     "codec"),
    ("no_saturation", "if (r > f->maxval) r = f->maxval;", "(void)0;", "codec"),
    ("e4m3_max_480", "{3, 7, 448.0, 0},", "{3, 7, 480.0, 0},", "codec"),
    ("subnormal_exponent", "v = ldexp((double)m, 1 - f->bias - f->mbits);",
     "v = ldexp((double)m, -f->bias - f->mbits);", "codec"),
    ("f16_overflow_saturates", "bits = (r > OR_HALF.maxval) ? 0x7C00u",
     "bits = (r > OR_HALF.maxval) ? 0x7BFFu", "codec"),
    ("e5m2_inf_to_nan", "return f->has_inf ? (neg ? 0xFC : 0x7C) : 0x7F;",
     "return 0x7F;", "codec"),
    ("e4m3_inf_saturates", "return f->has_inf ? (neg ? 0xFC : 0x7C) : 0x7F;",
     "return f->has_inf ? (neg ? 0xFC : 0x7C) : (neg ? 0xFE : 0x7E);", "codec"),
    ("e5m2_nan_decodes_inf",
     "if (m != 0) return or_bits_f32(0x7FC00000u);\n        v = INFINITY;",
     "v = INFINITY;", "codec"),
    ("negative_zero_unsigned", "int neg = signbit(x) != 0;\n    if (isinf(x))",
     "int neg = x < 0;\n    if (isinf(x))", "codec"),
    ("f16_subnormal_unclamped",
     "        lead = e - 1;\n        if (lead < emin) lead = emin;",
     "        lead = e - 1;", "codec"),
    ("f16_decode_subnormal", "v = ldexp((double)m, -24);", "v = ldexp((double)m, -25);",
     "codec"),
    ("f16_max_is_inf", "bits = (r > OR_HALF.maxval) ? 0x7C00u",
     "bits = (r >= OR_HALF.maxval) ? 0x7C00u", "codec"),
    ("e4m3_decode_top_codes_nan",
     "if (!f->has_inf && e == eall && m == (1 << f->mbits) - 1)",
     "if (!f->has_inf && e == eall && m >= (1 << f->mbits) - 2)", "codec"),
    ("fields_exponent_off", "return ((uint32_t)(lead + f->bias) << f->mbits) | M;",
     "return ((uint32_t)(lead + f->bias + 1) << f->mbits) | M;", "codec"),
    ("decode_exponent_off",
     "v = ldexp(1.0 + ldexp((double)m, -f->mbits), e - f->bias);\n    }\n    return (float)(s ? -v : v);   /* exact",
     "v = ldexp(1.0 + ldexp((double)m, -f->mbits), e - f->bias + 1);\n    }\n    return (float)(s ? -v : v);   /* exact",
     "codec"),
    ("e5m2_max_61440", "{2, 15, 57344.0, 1},", "{2, 15, 61440.0, 1},", "codec"),
    ("f16_decode_nan_as_inf",
     "if (m) return or_bits_f32(0x7FC00000u);\n        v = INFINITY;\n    } else if (e == 0) {\n        v = ldexp((double)m, -24);",
     "v = INFINITY;\n    } else if (e == 0) {\n        v = ldexp((double)m, -24);", "codec"),
    # scaled cast, just-in-time per-tensor scale (MS-AMP O1)
    ("amax_signed", "else if (fabsf(x) > a->fin) a->fin = fabsf(x);",
     "else if (x > a->fin) a->fin = x;", "cast"),
    ("scale_inverted", "float q = (float)OR_FMT[fmt].maxval / amax;",
     "float q = amax / (float)OR_FMT[fmt].maxval;", "cast"),
    ("nan_below_inf", "if (a->nan) return or_bits_f32(0x7FC00000u);\n    if (a->inf)",
     "if (a->inf) return INFINITY;\n    if (a->nan)", "cast"),
    ("cast_unscaled", "float t = x * scale;", "float t = x;", "cast"),
    ("tiny_amax_scale_unguarded", "if (!isfinite(q)) return 1.0f;\n    return q;",
     "return q;", "cast"),
    ("f16_source_as_bf16",
     "default: return oracle_f16_to_f32(((const uint16_t *)src)[i]);",
     "default: return oracle_bf16_to_f32(((const uint16_t *)src)[i]);", "cast"),
    ("cast_nonfinite_all_nan",
     "if (!isfinite(x)) { codes[i] = oracle_fp8_encode(x, fmt); continue; }",
     "if (!isfinite(x)) { codes[i] = 0x7F; continue; }", "cast"),
    ("amax_ignores_inf", "else if (isinf(x)) a->inf = 1;", "else if (isinf(x)) (void)0;",
     "cast"),
    ("bf16_shift_15", "return or_bits_f32((uint32_t)h << 16); }",
     "return or_bits_f32((uint32_t)h << 15); }", "cast"),
    # AdamW / Adam step with FP8 m and FP16 v (MS-AMP O2 / O3; torch AdamW)
    ("eps_inside_root", "float denom = fmaf(sqrtf(v), s.inv_sbc2, eps);",
     "float denom = sqrtf(v * s.inv_sbc2 * s.inv_sbc2 + eps);", "step"),
    ("no_sqrt", "float denom = fmaf(sqrtf(v), s.inv_sbc2, eps);",
     "float denom = fmaf(v, s.inv_sbc2, eps);", "step"),
    ("no_weight_decay", "float w = fmaf(-s.step_size, upd, wp * s.decay);",
     "float w = fmaf(-s.step_size, upd, wp);", "step"),
    ("no_first_bias_correction", "s.step_size = (float)((double)lr / bc1);",
     "s.step_size = lr; (void)bc1;", "step"),
    ("no_second_bias_correction", "s.inv_sbc2 = (float)(1.0 / sqrt(bc2));",
     "s.inv_sbc2 = 1.0f; (void)bc2;", "step"),
    ("bias_power_every_bit", "if (t & 1) r = r * b;", "r = r * b;", "step"),
    ("no_unscale", "return inv_loss_scale / p->g_scale;",
     "(void)inv_loss_scale; return 1.0f / p->g_scale;", "step"),
    ("m_with_beta2", "return fmaf(beta1, mp, s->omb1 * g);",
     "return fmaf(1.0f - s->omb2, mp, s->omb1 * g);", "step"),
    ("v_with_beta1", "float v = fmaf(beta2, vp, s.omb2 * (g * g));",
     "float v = fmaf(beta1, vp, s.omb1 * (g * g));", "step"),
    ("m_not_dequantized", "float mp = oracle_fp8_decode(p->m[i], OR_E4M3) * minv;",
     "float mp = oracle_fp8_decode(p->m[i], OR_E4M3); (void)minv;", "step"),
    ("m_encoded_unscaled", "q->m[i] = oracle_fp8_encode(m * m_scale_new, OR_E4M3);",
     "q->m[i] = oracle_fp8_encode(m, OR_E4M3);", "step"),
    ("copy_amax_from_fp32", "if (q->w8) or_amax_add(&aw, oracle_f16_to_f32(q->w[i]));",
     "if (q->w8) or_amax_add(&aw, w);", "step"),
    ("found_inf_ignored", "if (!isfinite(or_grad(&p[t], k, i))) return 1;",
     "(void)0;", "step"),
    ("l2_term_dropped", "return l2 ? fmaf(wd, oracle_f16_to_f32(p->w[i]), g) : g;",
     "(void)wd; return g;", "step"),
    ("l2_also_decays", "s.decay = l2 ? 1.0f : 1.0f - lr * wd;",
     "s.decay = 1.0f - lr * wd;", "step"),
    ("scaled_v_not_rescaled", "if (scaled_v) vp = vp * vinv;", "(void)vinv;", "step"),
    ("scaled_v_bound_forgets", "b_new = fmaf(beta2, *q->v_bound, s.omb2 * (gmax * gmax));",
     "b_new = s.omb2 * (gmax * gmax);", "step"),
    ("m_scale_not_stored", "*q->m_scale = m_scale_new;", "(void)0;", "step"),
    ("v_bound_not_stored", "if (scaled_v) *q->v_bound = b_new;", "(void)0;", "step"),
    ("scaled_v_stored_unscaled",
     "q->v[i] = oracle_f32_to_f16(scaled_v ? v * v_scale_new : v);",
     "q->v[i] = oracle_f32_to_f16(v); (void)v_scale_new;", "step"),
    ("w8_amax_reports_scale", "*q->w8_amax = amax_w;", "*q->w8_amax = w8_scale;", "step"),
    ("w8_off_by_a_ulp",
     "q->w8[i] = oracle_fp8_encode(oracle_f16_to_f32(q->w[i]) * w8_scale,",
     "q->w8[i] = oracle_fp8_encode(oracle_f16_to_f32(q->w[i]) * w8_scale * 1.0009765625f,",
     "step"),
    ("l2_found_inf_after_decay", "if (!isfinite(or_grad(&p[t], k, i))) return 1;",
     "if (!isfinite(or_grad_l2(&p[t], or_grad(&p[t], k, i), l2, wd, i))) return 1;",
     "step"),
    ("decay_without_lr", "s.decay = l2 ? 1.0f : 1.0f - lr * wd;",
     "s.decay = l2 ? 1.0f : 1.0f - wd;", "step"),
    ("v_abs_not_square", "float v = fmaf(beta2, vp, s.omb2 * (g * g));",
     "float v = fmaf(beta2, vp, s.omb2 * fabsf(g));", "step"),
    ("m_amax_over_g", "or_amax_add(&am, or_m_new(q, minv, g, beta1, &s, i));",
     "or_amax_add(&am, g);", "step"),
    ("state_bytes_fp32_v",
     "case 2: case 3: return (int)(sizeof(uint8_t) + sizeof(uint16_t));",
     "case 2: case 3: return (int)(sizeof(uint8_t) + sizeof(float));", "step"),
    ("scaled_v_gmax_before_l2", "if (scaled_v) or_amax_add(&ag, g);",
     "if (scaled_v) or_amax_add(&ag, or_grad(q, k, i));", "step"),
    ("m_scale_from_e5m2_max",
     "float m_scale_new = oracle_scale_from_amax(amax_m, OR_E4M3);",
     "float m_scale_new = oracle_scale_from_amax(amax_m, OR_E5M2);", "step"),
    ("w8_scale_from_e5m2_max", "float w8_scale = oracle_scale_from_amax(amax_w, OR_E4M3);",
     "float w8_scale = oracle_scale_from_amax(amax_w, OR_E5M2);", "step"),
    ("v_target_2_15", "#define OR_V_TARGET 16384.0f", "#define OR_V_TARGET 32768.0f",
     "step"),
    ("vinv_2_15", "vinv = *q->v_bound * 0x1p-14f;", "vinv = *q->v_bound * 0x1p-15f;",
     "step"),
    ("grad_factor_times_scale", "return inv_loss_scale / p->g_scale;",
     "return inv_loss_scale * p->g_scale;", "step"),
    ("bias_power_squares_first", "if (t & 1) r = r * b;\n        b = b * b;",
     "b = b * b;\n        if (t & 1) r = r * b;", "step"),
    ("eps_scaled_by_correction", "float denom = fmaf(sqrtf(v), s.inv_sbc2, eps);",
     "float denom = (sqrtf(v) + eps) * s.inv_sbc2;", "step"),
    ("step_zero_allowed", "return n < 0 || step < 1;", "return n < 0 || step < 0;",
     "step"),
    ("first_bias_step_off_by_one",
     "double bc1 = 1.0 - oracle_bias_power((double)beta1, step);",
     "double bc1 = 1.0 - oracle_bias_power((double)beta1, step + 1);", "step"),
    ("second_bias_step_off_by_one",
     "double bc2 = 1.0 - oracle_bias_power((double)beta2, step);",
     "double bc2 = 1.0 - oracle_bias_power((double)beta2, step + 1);", "step"),
    ("second_correction_not_rooted", "s.inv_sbc2 = (float)(1.0 / sqrt(bc2));",
     "s.inv_sbc2 = (float)(1.0 / bc2);", "step"),
    ("w_store_truncates", "q->w[i] = oracle_f32_to_f16(w);",
     "q->w[i] = (uint16_t)(oracle_f32_to_f16(w) & 0xFFFEu);", "step"),
    ("v_store_truncates",
     "q->v[i] = oracle_f32_to_f16(scaled_v ? v * v_scale_new : v);",
     "q->v[i] = (uint16_t)(oracle_f32_to_f16(scaled_v ? v * v_scale_new : v) & 0xFFFEu);",
     "step"),
    ("m_scale_stale",
     "float m_scale_new = oracle_scale_from_amax(amax_m, OR_E4M3);",
     "float m_scale_new = *q->m_scale; (void)amax_m;", "step"),
    ("v_scale_unguarded", "float q = OR_V_TARGET / b;\n    return isfinite(q) ? q : 1.0f;",
     "float q = OR_V_TARGET / b;\n    return q;", "step"),
    ("fp32_state_bytes_6", "case 0: case 1: return (int)(sizeof(float) + sizeof(float));",
     "case 0: case 1: return (int)(sizeof(float) + sizeof(uint16_t));", "step"),
    # the step by phases: pieces of a tensor with the tensor's maxima
    ("copy_uses_first_record_amax",
     "if (p[t].w8) or_tensor_copy(&p[t], master_amax[t]);",
     "if (p[t].w8) or_tensor_copy(&p[t], master_amax[0]);", "step"),
    ("update_master_amax_not_reported",
     "if (master_amax != NULL) master_amax[t] = aw;",
     "if (master_amax != NULL) master_amax[t] = 0.0f * aw;", "step"),
    # local reduction of FP8 shards (MS-AMP O1, FP8 all-reduce)
    ("reduce_divides", "acc = acc + oracle_fp8_decode(src[(int64_t)j * stride + i], in_fmt) * r[j];",
     "acc = acc + oracle_fp8_decode(src[(int64_t)j * stride + i], in_fmt) / scales[j];",
     "reduce"),
    ("reduce_one_scale", "acc = acc + oracle_fp8_decode(src[(int64_t)j * stride + i], in_fmt) * r[j];",
     "acc = acc + oracle_fp8_decode(src[(int64_t)j * stride + i], in_fmt) * r[0];",
     "reduce"),
    ("reduce_no_post", "y[i] = acc * post;", "y[i] = acc; (void)post;", "reduce"),
    ("reduce_stride_as_numel", "src[(int64_t)j * stride + i]", "src[(int64_t)j * numel + i]",
     "reduce"),
    ("reduce_drops_last_shard", "for (int j = 1; j < k; ++j)\n            acc",
     "for (int j = 1; j < k - 1; ++j)\n            acc", "reduce"),
    ("reduce_encodes_in_input_format",
     "rc = oracle_cast_scaled(y, OR_F32, numel, out_fmt,",
     "rc = oracle_cast_scaled(y, OR_F32, numel, in_fmt,", "reduce"),
    ("reduce_post_squared", "y[i] = acc * post;", "y[i] = acc * post * post;", "reduce"),
    ("reduce_first_shard_skipped",
     "float acc = oracle_fp8_decode(src[i], in_fmt) * r[0];", "float acc = 0.0f * r[0];",
     "reduce"),
    ("reduce_accepts_short_stride",
     "if (numel < 0 || k < 1 || k > 64 || stride < numel || in_fmt < 0 ||",
     "if (numel < 0 || k < 1 || k > 64 || in_fmt < 0 ||", "reduce"),
    ("reduce_accepts_no_shard",
     "if (numel < 0 || k < 1 || k > 64 || stride < numel || in_fmt < 0 ||",
     "if (numel < 0 || k < 0 || k > 64 || stride < numel || in_fmt < 0 ||", "reduce"),
    ("cast_accepts_bad_dtype",
     "if (numel < 0 || fmt < 0 || fmt > 1 || dtype < 0 || dtype > 2) return -1;",
     "if (numel < 0 || fmt < 0 || fmt > 1 || dtype < 0) return -1;", "reduce"),
    ("reduce_given_amax_ignored", "*scale_out = oracle_scale_from_amax(amax, out_fmt);",
     "*scale_out = oracle_scale_from_amax(448.0f, out_fmt); (void)amax;", "reduce"),
    # global gradient norm and clipping (torch clip_grad_norm_)
    ("sq_sum_not_squared", "acc += (unsigned __int128)r * r;",
     "acc += (unsigned __int128)r * 65536u;", "clip"),
    ("sq_sum_unit_halved", "uint64_t r = (uint64_t)ldexp(fabs((double)x), 16);",
     "uint64_t r = (uint64_t)ldexp(fabs((double)x), 15);", "clip"),
    ("norm_sum_not_squared", "sum += (unsigned __int128)q * q;",
     "sum += (unsigned __int128)q * 65536u;", "clip"),
    ("norm_k_not_squared", "double kk = (double)k * (double)k;", "double kk = (double)k;",
     "clip"),
    ("norm_unit_dropped", "terms[t] = kk * ldexp((double)sum, -32);",
     "terms[t] = kk * (double)sum;", "clip"),
    ("clip_no_epsilon", "double c = (double)max_norm / (norm + 1e-6);",
     "double c = (double)max_norm / norm;", "clip"),
    ("clip_unclamped", "return c < 1.0 ? (float)c : 1.0f;", "return (float)c;", "clip"),
    ("clip_unused", "if (clip != 1.0f) k = k * clip;", "(void)clip;", "clip"),
    ("norm_found_dropped",
     "if (!isfinite(or_grad(&p[t], k, i))) { found = 1; continue; }",
     "if (!isfinite(or_grad(&p[t], k, i))) { continue; }", "clip"),
    ("norm_last_tensor_only", "for (int t = 0; t < n; ++t) total = total + terms[t];",
     "for (int t = 0; t < n; ++t) total = terms[t];", "clip"),
    ("clip_nonpositive_max", "if (!(max_norm > 0.0f)) return 1.0f;\n    double c",
     "double c", "clip"),
    ("found_inf_on_clipped_gradient",
     "float k = or_grad_factor(&p[t], inv_loss_scale);\n        for (int64_t i = 0; i < p[t].numel; ++i)\n            if (!isfinite",
     "float k = or_grad_factor(&p[t], inv_loss_scale) * clip;\n        for (int64_t i = 0; i < p[t].numel; ++i)\n            if (!isfinite",
     "clip"),
    ("norm_code_unit_halved", "uint64_t q = (uint64_t)ldexp(d, 16);",
     "uint64_t q = (uint64_t)ldexp(d, 15);", "clip"),
    ("norm_not_rooted", "*norm = sqrt(total);", "*norm = total;", "clip"),
    ("norm_k_squared_in_float", "double kk = (double)k * (double)k;",
     "double kk = (double)(k * k);", "clip"),
    ("norm_terms_in_float", "terms[t] = kk * ldexp((double)sum, -32);",
     "terms[t] = (float)(kk * ldexp((double)sum, -32));", "clip"),
    ("norm_total_in_float", "for (int t = 0; t < n; ++t) total = total + terms[t];",
     "for (int t = 0; t < n; ++t) total = (float)(total + terms[t]);", "clip"),
    ("clip_coef_in_float", "double c = (double)max_norm / (norm + 1e-6);",
     "double c = (double)(max_norm / (float)(norm + 1e-6));", "clip"),
    ("norm_finite_on_found", "if (found != 0) { *norm = INFINITY; return found; }",
     "if (found != 0) { *norm = sqrt(total); return found; }", "clip"),
]


def _mutant_source(text, old, new):
    assert text.count(old) == 1, f"planted text not unique in the oracle: {old!r}"
    return text.replace(old, new)


def _run_pins(lib_path, first):
    order = [first] + [p for p in PINS if p != first]
    files = [os.path.join("tests", f"test_oracle_{p}.py") for p in order]
    env = dict(os.environ, FP8OPT_ORACLE_LIB=lib_path)
    r = subprocess.run([sys.executable, "-m", "pytest", *files, "-x", "-q",
                        "-p", "no:cacheprovider", "-m", "not gpu"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout[-1500:] + r.stderr[-500:]


def _build_and_run(name, text, first):
    import oracle
    src = os.path.join(OUT, f"{name}.c")
    with open(src, "w") as f:
        f.write(text)
    lib = oracle.compile_library(src, os.path.join(OUT, f"lib{name}.so"))
    return name, _run_pins(lib, first)


def test_mutant_names_are_unique():
    names = [m[0] for m in MUTANTS]
    assert len(set(names)) == len(names)
    assert all(m[3] in PINS for m in MUTANTS)


def test_every_planted_mistake_fails_a_pin():
    text = open(SRC).read()
    jobs = [("control", text, "codec")]
    jobs += [(name, _mutant_source(text, old, new), first)
             for name, old, new, first in MUTANTS]
    os.makedirs(OUT, exist_ok=True)
    workers = max(1, min(8, os.cpu_count() or 1))
    with ThreadPoolExecutor(workers) as ex:
        results = dict(ex.map(lambda j: _build_and_run(*j), jobs))
    rc, out = results.pop("control")
    assert rc == 0, f"the unchanged oracle fails its pins:\n{out}"
    survivors = {n: out for n, (rc, out) in results.items() if rc != 1}
    assert not survivors, "planted mistakes no pin caught (or a harness error):\n" + \
        "\n".join(f"--- {n} (rc {results[n][0]})\n{o}" for n, o in survivors.items())
