"""The pins must catch plausible mistakes in the oracle and in the parity checker.

Each case plants one mistake (a dropped term, a wrong sign, index or operand)
in a copy of oracle/ssm_oracle.c, compiles it on the CPU, and runs the pin
suite against it in a child process; the pins must fail.  The same is done for
the error metric every parity test uses (oracle/metrics.py) against its
hand-computed pins.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "ssm_oracle.c")

MUTANTS = {
    "abar_sign": ("const double abar = exp(dt * a);", "const double abar = exp(-dt * a);"),
    "input_dropped": ("h[n] = abar * h[n] + bbar * xv;", "h[n] = abar * h[n] + bbar;"),
    "readout_uses_B": ("y += Cv[n] * h[n];", "y += Bv[n] * h[n];"),
    "skip_dropped": ("y += (D ? D[d] : 0.0) * xv;", "y += 0.0 * xv;"),
    "gate_no_sigmoid": ("if (z) y *= silu(z[i]);", "if (z) y *= z[i];"),
    "softplus_sign": ("log1p(exp(-fabs(v)))", "log1p(exp(fabs(v)))"),
    "bias_sign": ("const double v = delta[i] + (delta_bias ? delta_bias[d] : 0.0);",
                  "const double v = delta[i] - (delta_bias ? delta_bias[d] : 0.0);"),
    "B_time_shift": (": &B[(b * seqlen + t) * dstate];", ": &B[(b * seqlen + (t > 0 ? t - 1 : 0)) * dstate];"),
    "state_in_ignored": ("h[n] = state_in ? state[(b * dim + d) * dstate + n] : 0.0;", "h[n] = 0.0;"),
    "zoh_missing_div_a": ("bbar = (a != 0.0) ? expm1(dt * a) / a * Bv[n] : dt * Bv[n];",
                          "bbar = (a != 0.0) ? expm1(dt * a) * Bv[n] : dt * Bv[n];"),
    "A_state_reversed": ("const double a = A[d * dstate + n];\n        const double abar",
                         "const double a = A[d * dstate + (dstate - 1 - n)];\n        const double abar"),
    "conv_correlates": ("x[(b * seqlen + (t - k)) * dim + d]", "x[(b * seqlen + k) * dim + d]"),
    "kernel_power_off_by_one": ("exp((double)k * dt[d] * a)", "exp((double)(k + 1) * dt[d] * a)"),
    "bilinear_numerator_sign": ("*abar = (1.0 + 0.5 * dt * a) / left;", "*abar = (1.0 - 0.5 * dt * a) / left;"),
    "euler_sign": ("*abar = 1.0 + dt * a;", "*abar = 1.0 - dt * a;"),
    "silu_sign": ("return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    "per_channel_C_row": ("const double* Cv = per_channel_bc ? &C[d * dstate]", "const double* Cv = per_channel_bc ? &C[0]"),
    "conv_taps_reversed": ("pre += w[d * width + k] * XS(t - k);", "pre += w[d * width + (width - 1 - k)] * XS(t - k);"),
    "conv_bias_dropped": ("double pre = cb ? cb[d] : 0.0;", "double pre = 0.0;"),
    "conv_history_reversed": ("past[j] = hist ? hist[(b * dim + d) * H + j] : 0.0;",
                              "past[j] = hist ? hist[(b * dim + d) * H + (H - 1 - j)] : 0.0;"),
    "conv_no_silu": ("u[(b * seqlen + t) * dim + d] = silu(pre);", "u[(b * seqlen + t) * dim + d] = pre;"),
    "conv_hist_out_shift": ("hist_out[(b * dim + d) * H + j] = XS(seqlen - H + j);",
                            "hist_out[(b * dim + d) * H + j] = XS(seqlen - H + j - 1);"),
    "bwd_lambda_uses_own_decay": ("const double lam = Ct[n] * gy + a_next[n] * lam_next[n];",
                                  "const double lam = Ct[n] * gy + a * lam_next[n];"),
    "bwd_dC_previous_state": ("dC[(b * L + t) * N + n] += gy * hcur;", "dC[(b * L + t) * N + n] += gy * hprev;"),
    "bwd_ddelta_no_sigmoid": ("const double sv = delta_softplus ? 1.0 / (1.0 + exp(-vs[t])) : 1.0;",
                              "const double sv = 1.0;"),
    "bwd_dx_no_skip": ("dx[i] = gx + gy * (D ? D[d] : 0.0);", "dx[i] = gx;"),
    "bwd_dA_no_step": ("dA[d * N + n] += lam * hprev * a * dts[t];", "dA[d * N + n] += lam * hprev * a;"),
    "bwd_dz_plain_sigmoid": ("dz[i] = dout[i] * y * sz * (1.0 + z[i] * (1.0 - sz));", "dz[i] = dout[i] * y * sz;"),
    "ssd_group_modulo": ("const int64_t b = bh / H, h = bh % H, g = h / per_group;",
                         "const int64_t b = bh / H, h = bh % H, g = h % ngroups;"),
    "ssd_decay_positive": ("const double a = exp(step * A[h]);", "const double a = exp(-step * A[h]);"),
    "ssd_input_no_step": ("hs[p * N + n] = a * hs[p * N + n] + step * Bv[n] * xv;",
                          "hs[p * N + n] = a * hs[p * N + n] + Bv[n] * xv;"),
    "ssd_readout_before_update": ("          hs[p * N + n] = a * hs[p * N + n] + step * Bv[n] * xv;\n          y += Cv[n] * hs[p * N + n];",
                                  "          y += Cv[n] * hs[p * N + n];\n          hs[p * N + n] = a * hs[p * N + n] + step * Bv[n] * xv;"),
    "ssd_softplus_always": ("const double step = dt_softplus ? oracle_softplus(s) : s;",
                            "const double step = oracle_softplus(s);"),
    "ssd_skip_dropped": ("y += (D ? D[h] : 0.0) * xv;", "y += 0.0 * xv;"),
    "ssd_state_transposed": ("hs[i] = state_in ? state[(b * H + h) * P * N + i] : 0.0;",
                             "hs[i] = state_in ? state[(b * H + h) * P * N + (i % N) * P + i / N] : 0.0;"),
    "bwd_dh0_undecayed": ("dh0[(b * dim + d) * N + n] = a_next[n] * lam_next[n];",
                          "dh0[(b * dim + d) * N + n] = lam_next[n];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    orig, mutated = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(orig) == 1, f"mutation site for {name} not found exactly once"
    mpath = tmp_path / "mutant.c"
    mpath.write_text(src.replace(orig, mutated))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-o", str(lib),
                    str(mpath), "-lm"], check=True)
    env = dict(os.environ, SSM_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pins did not catch mutant {name}:\n{r.stdout[-2000:]}"


# Planted mistakes in the parity checker (oracle/metrics.py); its hand-computed pins
# (tests/test_metrics_pins.py) must fail for each.
METRICS_SRC = os.path.join(ROOT, "oracle", "metrics.py")
METRIC_MUTANTS = {
    "mean_for_max": ("return float(np.max(np.abs(g - r) / den))", "return float(np.mean(np.abs(g - r) / den))"),
    "floor_at_max": ("fl = rms(r) if floor is None else float(floor)",
                     "fl = float(np.max(np.abs(r))) if floor is None else float(floor)"),
    "floor_at_mean_abs": ("fl = rms(r) if floor is None else float(floor)",
                          "fl = float(np.mean(np.abs(r))) if floor is None else float(floor)"),
    "rms_without_sqrt": ("return float(np.sqrt(np.mean(r * r))) if r.size else 0.0",
                         "return float(np.mean(r * r)) if r.size else 0.0"),
    "no_floor": ("den = np.maximum(np.abs(r), fl)", "den = np.abs(r)"),
    "signed_reference": ("den = np.maximum(np.abs(r), fl)", "den = np.maximum(r, fl)"),
    "signed_difference": ("return float(np.max(np.abs(g - r) / den))", "return float(np.max((g - r) / den))"),
    "finite_guard_dropped": ("    if not np.all(np.isfinite(g)):\n        return float(\"inf\")\n", ""),
    "report_unfloored_all_entries": ("\"max_rel_unfloored\": float((d[nz] / np.abs(r[nz])).max()) if nz.any() else 0.0,",
                                     "\"max_rel_unfloored\": float((d[nz] / np.abs(r[nz])).mean()) if nz.any() else 0.0,"),
}


@pytest.mark.parametrize("name", sorted(METRIC_MUTANTS))
def test_metric_pins_catch_mutant(name, tmp_path):
    orig, mutated = METRIC_MUTANTS[name]
    src = open(METRICS_SRC).read()
    assert src.count(orig) == 1, f"mutation site for {name} not found exactly once"
    mpath = tmp_path / "metrics_mutant.py"
    mpath.write_text(src.replace(orig, mutated))
    env = dict(os.environ, SSM_METRICS_PATH=str(mpath))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_metrics_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, f"metric pins did not catch mutant {name}:\n{r.stdout[-2000:]}"
