"""Plausible mistakes planted in a copy of the oracle must fail some pin.

Each mutant is the oracle's C source with one textual change (a dropped
term, a wrong sign or index, a transposed operand), compiled on the CPU into
a temporary library.  The pins of ``oracle_pins`` are then run against it;
at least one must fail, otherwise the pins would not have caught that
mistake in the real oracle.  Nothing here touches a GPU.
"""
import shutil
from pathlib import Path

import pytest

import oracle as oracle_pkg
import oracle_pins

SRC = Path(oracle_pkg.SOURCE).read_text()

# (name, function the change lives in, old text, new text)
MUTANTS = [
    ("direct_exponent_off_by_one", "wkv_oracle_forward_direct",
     "exp(-(double)(t - 1 - i) * w[c] + k[IDX(b, i, c)]);\n                    num",
     "exp(-(double)(t - i) * w[c] + k[IDX(b, i, c)]);\n                    num"),
    ("direct_drops_bonus", "wkv_oracle_forward_direct",
     "double e = exp(u[c] + k[IDX(b, t, c)]);", "double e = exp(k[IDX(b, t, c)]);"),
    ("recurrent_drops_bonus", "wkv_oracle_forward_recurrent",
     "double e = exp(u[c] + kt);\n                y[", "double e = exp(kt);\n                y["),
    ("recurrent_decays_new_token", "wkv_oracle_forward_recurrent",
     "a = decay * a + ek * vt;", "a = decay * (a + ek * vt);"),
    ("adjoint_gD_sign", "wkv_oracle_backward_adjoint",
     "double gD = -g * yt / D;", "double gD = g * yt / D;"),
    ("adjoint_gw_drops_decay", "wkv_oracle_backward_adjoint",
     "sgw += -decay * (la * a[t] + lb * bb[t]);", "sgw += -(la * a[t] + lb * bb[t]);"),
    ("adjoint_lambda_index", "wkv_oracle_backward_adjoint",
     "(la * vt + lb) * ek;", "((gN + decay * la) * vt + lb) * ek;"),
    ("adjoint_gv_transposed", "wkv_oracle_backward_adjoint",
     "gv[IDX(b, t, c)] = gN * e + la * ek;", "gv[IDX(b, t, c)] = gN * ek + la * e;"),
    ("direct_grad_w_index", "wkv_oracle_backward_direct",
     "gw[c] += -g * (double)(t - 1 - i) * W", "gw[c] += -g * (double)(t - i) * W"),
    ("direct_grad_k_sign", "wkv_oracle_backward_direct",
     "gk[IDX(b, i, c)] += g * W * (vi - yt) / D;", "gk[IDX(b, i, c)] += g * W * (yt - vi) / D;"),
    ("state_pp_index", "wkv_oracle_state",
     "double ex = k[IDX(b, i, c)] - (double)(t - 1 - i) * w[c];",
     "double ex = k[IDX(b, i, c)] - (double)(t - i) * w[c];"),
    ("gated_recurrent_gate_sign", "wkv_oracle_forward_gated_recurrent",
     "out[i] = out[i] / (1.0 + exp(-r[i]));\n}\n\n/* Gradients", "out[i] = out[i] / (1.0 + exp(r[i]));\n}\n\n/* Gradients"),
    ("decode_mix_transposed", "wkv_oracle_decode_step",
     "mu_k[p] * x[o] + (1.0 - mu_k[p]) * x_prev[o]", "mu_k[p] * x_prev[o] + (1.0 - mu_k[p]) * x[o]"),
    ("decode_gate_sign", "wkv_oracle_decode_step",
     "wkv / (1.0 + exp(-r[o]))", "wkv / (1.0 + exp(r[o]))"),
    ("decode_pp_no_decay", "wkv_oracle_decode_step",
     "double pp2 = pp[o] - w[p] > k[o] ? pp[o] - w[p] : k[o];", "double pp2 = pp[o] > k[o] ? pp[o] : k[o];"),
    ("decode_drops_bonus", "wkv_oracle_decode_step",
     "double e = exp(u[p] + k[o]);", "double e = exp(k[o]);"),
    ("state_in_not_decayed", "wkv_oracle_forward_state",
     "double dp = exp(M - w[c] - m2)", "double dp = exp(M - m2)"),
    ("state_in_scale_ignored", "wkv_oracle_forward_state",
     "double sp = exp(M - q), sc", "double sp = exp(-q), sc"),
    ("shift_mix_transposed", "wkv_oracle_token_shift",
     "xk[IDX(b, t, c)] = mu_k[c] * cur + (1.0 - mu_k[c]) * prev;",
     "xk[IDX(b, t, c)] = mu_k[c] * prev + (1.0 - mu_k[c]) * cur;"),
    ("shift_grad_misses_next_token", "wkv_oracle_token_shift_backward",
     "g += (1.0 - mu_k[c]) * gxk[n] +", "g += 0.0 * gxk[n] +"),
    ("gate_sign", "wkv_oracle_forward_gated",
     "out[i] / (1.0 + exp(-r[i]))", "out[i] / (1.0 + exp(r[i]))"),
    ("gated_gy_not_gated", "wkv_oracle_backward_gated",
     "gy[i] = gout[i] * s;", "gy[i] = gout[i];"),
    ("gated_gr_drops_one_minus_s", "wkv_oracle_backward_gated",
     "gr[i] = gout[i] * y[i] * s * (1.0 - s);", "gr[i] = gout[i] * y[i] * s;"),
    ("gated_gr_uses_gated_gradient", "wkv_oracle_backward_gated",
     "gr[i] = gout[i] * y[i] * s * (1.0 - s);", "gr[i] = gy[i] * y[i] * s * (1.0 - s);"),
    ("bstate_ignores_state_in", "wkv_oracle_backward_state",
     "a[0] = given ? num_in[o] * exp(pp_in[o]) : 0.0;", "a[0] = 0.0;"),
    ("bstate_ignores_end_gradient", "wkv_oracle_backward_state",
     "double la = ga_end ? ga_end[o] : 0.0,", "double la = 0.0,"),
    ("bstate_gw_drops_decay", "wkv_oracle_backward_state",
     "sgw += -decay * (la * a[t] + lb * bb[t]);", "sgw += -(la * a[t] + lb * bb[t]);"),
    ("fold_no_decay", "wkv_oracle_state_fold",
     "double Md = M - (double)lengths[i] * w[c];", "double Md = M;"),
    ("fold_decays_segment", "wkv_oracle_state_fold",
     "A = A * dp + st[o] * ds;", "A = A * dp + st[o] * ds * exp(-(double)lengths[i] * w[c]);"),
    ("sqrelu_not_squared", "wkv_oracle_sqrelu", "a[i] = p * p;", "a[i] = p;"),
    ("sqrelu_grad_drops_two", "wkv_oracle_sqrelu_backward",
     "gk[i] = 2.0 * (k[i] > 0.0 ? k[i] : 0.0) * ga[i];", "gk[i] = (k[i] > 0.0 ? k[i] : 0.0) * ga[i];"),
    ("cmix_gate_sign", "wkv_oracle_cmix_gate", "vk[i] / (1.0 + exp(-r[i]))", "vk[i] / (1.0 + exp(r[i]))"),
    ("cmix_gr_drops_one_minus_s", "wkv_oracle_cmix_gate_backward",
     "gr[i] = gout[i] * vk[i] * s * (1.0 - s);", "gr[i] = gout[i] * vk[i] * s;"),
    ("cmix_gvk_ungated", "wkv_oracle_cmix_gate_backward", "gvk[i] = gout[i] * s;", "gvk[i] = gout[i];"),
    ("shift_grad_mu_sign", "wkv_oracle_token_shift_backward",
     "double d = x[i] - prev;", "double d = prev - x[i];"),
]


def _function_span(src, name):
    start = src.index("void " + name + "(")
    nxt = src.find("\nvoid ", start + 1)
    return start, (len(src) if nxt < 0 else nxt)


@pytest.mark.parametrize("name,func,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, func, old, new):
    a, b = _function_span(SRC, func)
    body = SRC[a:b]
    assert body.count(old) == 1, f"mutation site for {name} not unique in {func}"
    mutated = SRC[:a] + body.replace(old, new) + SRC[b:]
    src = tmp_path / f"{name}.c"
    src.write_text(mutated)
    lib = oracle_pkg.build(src, tmp_path / f"lib{name}.so")
    failed = oracle_pins.failing_pins(oracle_pkg.Oracle(lib))
    assert failed, f"mutant {name} passed every pin"
    shutil.rmtree(tmp_path, ignore_errors=True)
