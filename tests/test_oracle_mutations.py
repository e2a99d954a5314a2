"""Plant plausible mistakes in a copy of the oracle and check the pins catch each.

Every mutant is a text edit of oracle/ss_oracle.c compiled into a temporary
library on the CPU; the real oracle is untouched. A mutant that survives every
pin would mean the pins do not constrain that part of the oracle.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle
import pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "ss_oracle.c")

MUTANTS = {
    "exp_sign": ("h[n] = exp(dt * a) * h[n]", "h[n] = exp(-dt * a) * h[n]"),
    "bwd_recompute_exp_sign": ("H[(t + 1) * N + n] = exp(dt * a) *", "H[(t + 1) * N + n] = exp(-dt * a) *"),
    "drop_dt_in_input": ("bbar * Bv * uv", "Bv * uv"),
    "B_transposed": ("rd(j->B, bcrow + (long long)n * L + l", "rd(j->B, bcrow + l * N + n"),
    "C_reads_B": ("rd(j->C, bcrow", "rd(j->B, bcrow"),
    "drop_D_skip": ("yv += Dd * uv;", ";"),
    "gate_before_skip": ("yv += Dd * uv;\n            if (j->z) yv *= ss_oracle_silu(rd(j->z, urow + l, j->dtype));",
                         "if (j->z) yv *= ss_oracle_silu(rd(j->z, urow + l, j->dtype));\n            yv += Dd * uv;"),
    "softplus_branch": ("log1p(exp(x));", "log(exp(x));"),
    "softplus_sign": ("x + log1p(exp(-x))", "x + log1p(exp(x))"),
    "ignore_h0": ("h[n] = j->h0 ? j->h0[r * N + n] : 0.0;", "h[n] = 0.0;"),
    "output_before_update": (
        "h[n] = exp(dt * a) * h[n] + bbar * Bv * uv;\n                yv += Cv * h[n];",
        "yv += Cv * h[n];\n                h[n] = exp(dt * a) * h[n] + bbar * Bv * uv;"),
    "sigmoid_not_silu": ("return z / (1.0 + exp(-z));", "return 1.0 / (1.0 + exp(-z));"),
    "bias_by_batch": ("j->bias[d]", "j->bias[b % j->dim]"),
    "A_transposed": ("j->A[(long long)d * N + n]", "j->A[(long long)n * j->dim + d]"),
    "u_lagged": ("const double uv = rd(j->u, urow + l, j->dtype);",
                 "const double uv = rd(j->u, urow + (l > 0 ? l - 1 : 0), j->dtype);"),
    "z_ignored": ("if (j->z) yv *=", "if (0) yv *="),
    "D_by_n": ("(double)j->D[d]", "(double)j->D[0]"),
    # exact zero-order hold
    "zoh_ignored": ("if (!zoh || a == 0.0) return dt;", "return dt;"),
    "zoh_sign": ("return expm1(dt * a) / a;", "return expm1(-dt * a) / a;"),
    "zoh_no_division": ("return expm1(dt * a) / a;", "return -expm1(dt * a);"),
    # backward pass
    "bwd_no_decay_propagation": ("g[n] *= e;", ";"),
    "bwd_dC_prev_state": ("+= gs * H[(t + 1) * N + n];", "+= gs * H[t * N + n];"),
    "bwd_gdt_no_input_term": ("gdt += g[n] * (a * e * hp + fdt * Bv * uv);",
                              "gdt += g[n] * (a * e * hp);"),
    "bwd_dz_sigmoid_only": ("dy[urow + t] * s * sg * (1.0 + zv * (1.0 - sg))", "dy[urow + t] * s * sg"),
    "bwd_zoh_fa_dropped": ("(dt * e * hp + fa * Bv * uv)", "(dt * e * hp)"),
    "bwd_zoh_fa_limit_dropped": ("fa = 0.5 * dt * dt;", "fa = 0.0;"),
    "bwd_gx_no_sigmoid": ("const double gx = delta_softplus ? gdt / (1.0 + exp(-x)) : gdt;",
                          "const double gx = gdt;"),
    "bwd_dh_last_ignored": ("g[n] = dh_last ? dh_last[r * N + n] : 0.0;", "g[n] = 0.0;"),
    "bwd_gu_no_D": ("double gu = gs * Dd, gdt = 0.0;", "double gu = 0.0, gdt = 0.0;"),
    # causal depthwise convolution and its decode step
    "conv_kernel_reversed": ("acc += (double)wd[k] * conv_in(x, off, l - (width - 1) + k",
                             "acc += (double)wd[width - 1 - k] * conv_in(x, off, l - (width - 1) + k"),
    "conv_not_causal": ("conv_in(x, off, l - (width - 1) + k, dtype, s, width)",
                        "conv_in(x, off, l - (width - 1) / 2 + k, dtype, s, width)"),
    "conv_state_ignored": ("return s ? s[(W - 1) + j] : 0.0;", "return 0.0;"),
    "conv_state_reversed": ("return s ? s[(W - 1) + j] : 0.0;", "return s ? s[-1 - j] : 0.0;"),
    "conv_bias_dropped": ("double acc = bias ? (double)bias[d] : 0.0;\n            for (int k = 0; k < width; ++k)",
                          "double acc = 0.0;\n            for (int k = 0; k < width; ++k)"),
    "conv_final_state_shift": ("seqlen - (width - 1) + j", "seqlen - width + j"),
    "conv_update_no_shift": ("for (int k = 0; k + 1 < width - 1; ++k) s[k] = s[k + 1];", ";"),
    "conv_update_weight": ("acc += (double)wd[width - 1] * xv;", "acc += (double)wd[0] * xv;"),
    "conv_silu_dropped": ("out[off + l] = silu ? ss_oracle_silu(acc) : acc;", "out[off + l] = acc;"),
    "conv_channel_0": ("const float *wd = w + (long long)d * width;\n        const long long off",
                       "const float *wd = w;\n        const long long off"),
}


def _build(name, tmp_path):
    text = open(SRC).read()
    old, new = MUTANTS[name]
    assert text.count(old) == 1, "mutation anchor not found once: %s" % name
    src = tmp_path / ("m_%s.c" % name)
    src.write_text(text.replace(old, new))
    lib = tmp_path / ("m_%s.so" % name)
    subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-o", str(lib), str(src), "-lm",
                           "-lpthread"])
    return str(lib)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path, monkeypatch):
    oracle._load()
    lib = ctypes.CDLL(_build(name, tmp_path))
    real = oracle._lib
    for fn in ("ss_oracle_scan", "ss_oracle_state_update", "ss_oracle_softplus", "ss_oracle_silu",
               "ss_oracle_conv1d", "ss_oracle_conv1d_update", "ss_oracle_scan_bwd"):
        f = getattr(lib, fn)
        f.argtypes = getattr(real, fn).argtypes
        f.restype = getattr(real, fn).restype
    monkeypatch.setattr(oracle, "_lib", lib)
    failed = []
    for pname, pin in pins.ALL_PINS.items():
        with np.errstate(all="ignore"):
            err = pin(oracle)
        if not (err <= pins.PIN_TOL.get(pname, pins.DEFAULT_TOL)):
            failed.append(pname)
    assert failed, "mutant %s passed every pin" % name
