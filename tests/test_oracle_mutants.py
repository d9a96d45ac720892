"""Plant plausible mistakes in a copy of the oracle and check that the pins catch
each one.  The real oracle source is never modified: every mutant is a textual
edit of a temporary copy, compiled into a temporary directory.  CPU only."""
import os

import pytest

import oracle
from oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "dsa_oracle.c")

MUTANTS = {
    "relu_dropped": ("double relu = dot > 0.0 ? dot : 0.0;", "double relu = dot;"),
    "head_weight_dropped": ("score += bf(w[j]) * relu;", "score += relu;"),
    "causal_excludes_self": ("/* every causal key s <= t is scored */\n  for (int64_t s = 0; s <= t; ++s) {",
                             "/* every causal key s <= t is scored */\n  for (int64_t s = 0; s < t; ++s) {"),
    "fp8_causal_excludes_self": ("const float* ksb = c->ks + (int64_t)b * c->S_max;\n  for (int64_t s = 0; s <= t; ++s) {",
                                 "const float* ksb = c->ks + (int64_t)b * c->S_max;\n  for (int64_t s = 0; s < t; ++s) {"),
    "tie_break_reversed": ("return (x->s < y->s) ? -1 : (x->s > y->s);",
                           "return (x->s > y->s) ? -1 : (x->s < y->s);"),
    "short_rows_sorted_not_all": ("if (n <= c->topk) {", "if (n < 0) {"),
    "rope_dims_dropped": ("for (int d = 0; d < RLAT; ++d) dot += bf(q[d]) * bf(row[d]);",
                          "for (int d = 0; d < VLAT; ++d) dot += bf(q[d]) * bf(row[d]);"),
    "scale_dropped": ("z[j] = dot * c->scale;", "z[j] = dot;"),
    "value_shifted_into_rope": ("oh[d] += p * bf(row[d]); /* value",
                                "oh[d] += p * bf(row[d + 64]); /* value"),
    "lse_without_max": ("lse[h] = m + log(l);", "lse[h] = log(l);"),
    "softmax_not_normalised": ("for (int d = 0; d < VLAT; ++d) oh[d] /= l;", ""),
    "gate_without_sigmoid": ("o[col] = u / (1.0 + exp(-g));", "o[col] = u * g;"),
    "gate_sign_flipped": ("o[col] = u / (1.0 + exp(-g));", "o[col] = u / (1.0 + exp(g));"),
    "explicit_value_uses_key_weight": ("acc += Wv[(int64_t)e * c->R + d] * ck[d];",
                                       "acc += Wk[(int64_t)e * c->R + d] * ck[d];"),
    "sparse_ignores_minus_one_wrongly": ("int32_t s = ix[j];\n    if (s < 0) continue;\n    if (s > t",
                                         "int32_t s = ix[j];\n    if (s < 0) s = 0;\n    if (s > t"),
    "dense_excludes_self": ("const int64_t nk = t + 1;", "const int64_t nk = t > 0 ? t : 1;"),
    "dense_rope_dims_dropped": ("for (int d = 0; d < RLAT; ++d) acc += bf(qh[d]) * bf(krow[d]);",
                                "for (int d = 0; d < VLAT; ++d) acc += bf(qh[d]) * bf(krow[d]);"),
    "dense_scale_dropped": ("z[(int64_t)h * nk + s] = c->scale * acc;",
                            "z[(int64_t)h * nk + s] = acc;"),
    "layernorm_sample_variance": ("    var /= D;\n", "    var /= (D - 1);\n"),
    "layernorm_eps_dropped": ("const double inv = 1.0 / sqrt(var + eps);",
                              "const double inv = 1.0 / sqrt(var);"),
    "bf16_ties_away_from_zero": ("double r = nearbyint(m * 256.0);", "double r = round(m * 256.0);"),
    "sink_not_in_denominator": ("if (c->sink) l += exp(c->sink[h] - m);", ""),
    "sink_does_not_move_max": ("if (c->sink && c->sink[h] > m) m = c->sink[h];", ""),
    "e4m3_ties_away_from_zero": ("const double v = nearbyint(a / q) * q;",
                                 "const double v = round(a / q) * q;"),
    "e4m3_no_subnormal_quantum": ("if (a == 0.0 || e < -6) e = -6;", "if (a == 0.0) e = -6;"),
    "e4m3_bias_off_by_one": ("return ldexp(8.0 + m, ex - 10);", "return ldexp(8.0 + m, ex - 9);"),
    "quant_divides_once": ("const float t = (float)bf(xr[d]) * inv;",
                           "const float t = (float)bf(xr[d]) / s;"),
    "quant_scale_without_floor": ("const float s = (amax > floor_ ? amax : floor_) / 448.0f;",
                                  "const float s = amax / 448.0f;"),
    "fp8_relu_dropped": ("const double pos = dot > 0.0 ? dot : 0.0;", "const double pos = dot;"),
    "fp8_head_weight_dropped": ("score += bf(w[j]) * pos;", "score += pos;"),
    "bwd_D_dropped_in_dq": ("      const double dz = p * (dp - Dv);", "      const double dz = p * dp;"),
    "bwd_D_dropped_in_dkv": ("const double dz = p * (dp - c->D[flat * c->H + h]);", "const double dz = p * dp;"),
    "bwd_dq_scale_dropped": ("dqh[d] += c->scale * dz * row[d];", "dqh[d] += dz * row[d];"),
    "bwd_dq_rope_dims_dropped": ("for (int d = 0; d < RLAT; ++d) dqh[d] += c->scale", "for (int d = 0; d < VLAT; ++d) dqh[d] += c->scale"),
    "bwd_value_grad_dropped": ("for (int d = 0; d < VLAT; ++d) out[d] += p * dOh[d];", ""),
    "bwd_key_grad_sign_flipped": ("out[d] += c->scale * dz * qh[d];", "out[d] -= c->scale * dz * qh[d];"),
    "bwd_sink_not_in_denominator": ("    if (sk != -INFINITY) l += exp(sk - m);\n", ""),
    "fp8_key_scale_dropped": ("* (ks * dec8(k[d]));", "* dec8(k[d]);"),
    "fp8_query_scale_dropped": ("dot += (qsj * dec8(q[j * c->D_I + d]))", "dot += (dec8(q[j * c->D_I + d]))"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique/absent"
    mpath = tmp_path / "mutant.c"
    mpath.write_text(src.replace(old, new))
    lib = oracle.load(oracle.build(force=True, src=str(mpath), out=str(tmp_path / "libm.so")))
    caught = []
    for pin in ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, oracle.OracleError) as e:  # the pin noticed
            caught.append(pin.__name__)
    assert caught, f"no pin catches mutant {name}"
