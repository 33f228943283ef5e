"""Pins for the float64 oracle: the pages' worked examples, closed forms,
the LTI convolution identity, invariants, and brute force on tiny inputs.

Each test names the page and section it checks.  None of them re-types the
oracle's loop: every expected value comes from the pages, from a different
formulation (closed-form sums, explicit products, library convolution,
numerical quadrature) or from an identity the pages state.
"""
import functools
import math

import numpy as np
import pytest

import oracle
from oracle.metrics import floored_rel_err
from selective_state_space_112_b300.workloads import (bf16_bits_to_f32, f32_to_bf16_bits,
                                                      make_workload)


def scalar_scan(u, a, b, c, step, bbar_mode, h0=None, d_skip=None):
    """Drive the oracle with one channel and one state (LTI layout)."""
    L = len(u)
    x = np.asarray(u, dtype=np.float64).reshape(1, L, 1)
    delta = np.full((1, L, 1), float(step))
    out, st = oracle.selective_scan(
        x, delta, np.array([[a]], float), np.array([[b]], float), np.array([[c]], float),
        D=None if d_skip is None else np.array([d_skip], float),
        h0=None if h0 is None else np.array([[[h0]]], float),
        delta_softplus=False, bbar_mode=bbar_mode, per_channel_bc=True)
    return out[0, :, 0], st[0, 0, 0]


# ---------------------------------------------------------------- worked examples

def test_zoh_worked_example(golden):
    """'State Space Models: Mamba and Beyond', worked example of ZOH: printed
    factors and outputs, and the analytic solution of dx/dt = -x + u."""
    g = golden("zoh_worked_example.txt")
    abar, bbar = oracle.discretize(g["A"], g["B"], g["step"], oracle.RULE_ZOH)
    assert abs(abar - g["abar"]) < g["tol"] and abs(bbar - g["bbar"]) < g["tol"]
    y, _ = scalar_scan(g["u"], g["A"], g["B"], g["C"], g["step"], bbar_mode=1)
    assert np.max(np.abs(y - np.array(g["y"]))) < g["tol"]
    # analytic trajectory: 1 - e^{-t} while u = 1 (t = 0.5, 1), then free decay
    e = math.exp
    analytic = [1 - e(-0.5), 1 - e(-1.0), (1 - e(-1.0)) * e(-0.5), (1 - e(-1.0)) * e(-1.0)]
    assert np.max(np.abs(y - np.array(analytic))) < 1e-12


def test_active_recall_answers(golden):
    """'State Space Models: Mamba and Beyond', active-recall answers 1 and 2."""
    g = golden("active_recall.txt")
    abar, bbar = oracle.discretize(g["q1_A"], g["q1_B"], g["q1_step"], oracle.RULE_ZOH)
    assert abs(abar - g["q1_abar"]) < g["tol"] and abs(bbar - g["q1_bbar"]) < g["tol"]
    abar, bbar = oracle.discretize(g["q2_A"], g["q2_B"], g["q2_step"], oracle.RULE_ZOH)
    assert abs(abar - g["q2_abar"]) < g["tol"] and abs(bbar - g["q2_bbar"]) < g["tol"]
    y, _ = scalar_scan(g["q2_u"], g["q2_A"], g["q2_B"], 1.0, g["q2_step"], bbar_mode=1)
    assert np.max(np.abs(y - np.array(g["q2_y"]))) < g["tol"]
    # both step sizes sample the same continuous trajectory at t = 1 and t = 2
    y_half, _ = scalar_scan([1, 1, 0, 0], -1.0, 1.0, 1.0, 0.5, bbar_mode=1)
    assert abs(y[0] - y_half[1]) < 1e-14 and abs(y[1] - y_half[3]) < 1e-14


def test_selection_worked_example(golden):
    """'State Space Models: Mamba and Beyond', selection example: softplus
    step and Abar = exp(step * A), pinned through the scan itself."""
    g = golden("selection_worked_example.txt")
    for v, step, abar in zip(g["pre_activation"], g["step"], g["abar"]):
        assert abs(oracle.softplus(v) - step) < g["tol"]
        # state 1, no input: one step leaves h = Abar
        x = np.zeros((1, 1, 1))
        dl = np.full((1, 1, 1), v)
        _, st = oracle.selective_scan(x, dl, np.array([[g["A"]]]), np.ones((1, 1, 1)),
                                      np.ones((1, 1, 1)), h0=np.ones((1, 1, 1)),
                                      delta_softplus=True)
        assert abs(st[0, 0, 0] - abar) < g["tol"]
        # state 0, input 1, B = 1, Bbar = step * B: one step leaves h = step
        _, st = oracle.selective_scan(np.ones((1, 1, 1)), dl, np.array([[g["A"]]]),
                                      np.ones((1, 1, 1)), np.ones((1, 1, 1)),
                                      delta_softplus=True)
        assert abs(st[0, 0, 0] - step) < g["tol"]


def test_softplus_against_library():
    """softplus(v) = log(1 + e^v) (np.logaddexp), including far tails."""
    for v in [-800.0, -40.0, -7.0, -0.5, 0.0, 1e-8, 1.0, 20.0, 40.0, 800.0]:
        ref = float(np.logaddexp(0.0, v))
        got = oracle.softplus(v)
        assert abs(got - ref) <= 1e-15 * max(abs(ref), 1e-300) + 1e-320, (v, got, ref)


# ----------------------------------------------------------- discretisation rules

def test_discretization_factors(golden):
    """'State-space models', Discretization: Euler, bilinear and ZOH factors."""
    g = golden("discretization_factors.txt")
    a = g["a"]
    assert oracle.discretize(a, 1.0, 2.5, oracle.RULE_EULER)[0] == pytest.approx(g["euler_at_2.5"], abs=1e-15)
    assert oracle.discretize(a, 1.0, 1.0, oracle.RULE_EULER)[0] == pytest.approx(g["euler_at_1"], abs=1e-15)
    zoh = oracle.discretize(a, 1.0, 2.5, oracle.RULE_ZOH)[0]
    assert 0.0 < zoh < 1.0 and zoh == pytest.approx(math.exp(-2.5), rel=1e-15)
    # bilinear stays inside the unit circle for every step when a < 0
    for dt in np.geomspace(1e-3, 1e3, 25):
        assert abs(oracle.discretize(a, 1.0, dt, oracle.RULE_BILINEAR)[0]) < 1.0
    # at step 0.1 bilinear is closer to the exact factor than Euler
    ex = math.exp(-0.1)
    bil = oracle.discretize(a, 1.0, 0.1, oracle.RULE_BILINEAR)[0]
    eul = oracle.discretize(a, 1.0, 0.1, oracle.RULE_EULER)[0]
    assert abs(bil - ex) < abs(eul - ex)
    # bilinear is the (1,1) Pade approximant of e^x: error ~ |x|^3 / 12
    x = -1e-3
    bil = oracle.discretize(-1.0, 1.0, -x, oracle.RULE_BILINEAR)[0]
    assert (bil - math.exp(x)) / x ** 3 == pytest.approx(1.0 / 12.0, rel=2e-3)
    # Euler's input factor and the simplified ZOH input factor are step * b
    assert oracle.discretize(a, 3.0, 0.25, oracle.RULE_EULER)[1] == pytest.approx(0.75, abs=1e-15)
    assert oracle.discretize(a, 3.0, 0.25, oracle.RULE_ZOH_SIMPLE)[1] == pytest.approx(0.75, abs=1e-15)
    # bilinear input factor: trapezoid-rule solution of h' = a h + b u with u = 1
    ab, bb = oracle.discretize(-2.0, 1.0, 0.3, oracle.RULE_BILINEAR)
    # trapezoid: h1 = h0 + dt/2 (a h0 + b + a h1 + b)  with h0 = 0  =>  h1 = dt b / (1 - dt a / 2)
    assert bb == pytest.approx(0.3 / (1 + 0.3), rel=1e-14)
    with pytest.raises(ValueError):
        oracle.discretize(a, 1.0, 1.0, 7)


def test_zoh_input_factor_is_integral():
    """Exact ZOH input factor = integral_0^step e^{tau a} d tau * b
    ('Structured State Space Models and Mamba', Discretization Mechanics)."""
    from scipy.integrate import quad
    for a, b, dt in [(-1.0, 1.0, 0.5), (-2.0, 0.7, 0.25), (-0.01, -1.3, 3.0), (-7.5, 2.0, 0.01)]:
        integral, _ = quad(lambda tau: math.exp(tau * a), 0.0, dt, epsabs=0.0, epsrel=1e-13, limit=200)
        _, bbar = oracle.discretize(a, b, dt, oracle.RULE_ZOH)
        assert bbar == pytest.approx(integral * b, rel=1e-12)
    # a -> 0 limit is step * b
    assert oracle.discretize(0.0, 2.0, 0.3, oracle.RULE_ZOH)[1] == pytest.approx(0.6, rel=1e-15)
    assert oracle.discretize(-1e-12, 2.0, 0.3, oracle.RULE_ZOH)[1] == pytest.approx(0.6, rel=1e-9)


def test_small_and_large_step_limits():
    """Small step: Abar -> 1 and Bbar -> 0 (token skipped); large step: Abar -> 0
    ('State Space Models: Mamba and Beyond', answer 4; llms.blog, Discretization)."""
    ab, bb = oracle.discretize(-1.0, 1.0, 1e-9, oracle.RULE_ZOH_SIMPLE)
    assert abs(ab - 1.0) < 2e-9 and abs(bb) < 2e-9
    ab, _ = oracle.discretize(-1.0, 1.0, 50.0, oracle.RULE_ZOH_SIMPLE)
    assert 0 < ab < 1e-20
    # through the scan: a tiny step keeps the state, a huge step erases it
    x = np.ones((1, 1, 1))
    _, st = oracle.selective_scan(x, np.full((1, 1, 1), 1e-9), np.array([[-1.0]]),
                                  np.ones((1, 1)), np.ones((1, 1)), h0=np.full((1, 1, 1), 3.0),
                                  delta_softplus=False, per_channel_bc=True)
    assert st[0, 0, 0] == pytest.approx(3.0, rel=1e-8)
    _, st = oracle.selective_scan(x, np.full((1, 1, 1), 60.0), np.array([[-1.0]]),
                                  np.ones((1, 1)), np.ones((1, 1)), h0=np.full((1, 1, 1), 3.0),
                                  delta_softplus=False, per_channel_bc=True, bbar_mode=1)
    assert st[0, 0, 0] == pytest.approx(1.0, rel=1e-12)   # exact ZOH: state -> input


# ------------------------------------------------------------------ closed forms

def test_scalar_closed_form():
    """h_t = sum_k a^k b x_{t-k} for constant a, b ('State-space models',
    Recurrence and convolution), with the fused scan's Bbar = step * B."""
    rng = np.random.default_rng(11)
    L = 64
    x = rng.standard_normal(L)
    A, B, step = -0.7, 1.3, 0.2
    a, b = math.exp(step * A), step * B
    y, st = scalar_scan(x, A, B, 1.0, step, bbar_mode=0)
    ref = np.array([sum(a ** k * b * x[t - k] for k in range(t + 1)) for t in range(L)])
    assert floored_rel_err(y, ref) < 1e-13
    assert st == pytest.approx(ref[-1], rel=1e-13)


def test_lti_scan_equals_causal_convolution():
    """LTI system: the recurrence equals causal convolution with
    K_k = C Abar^k Bbar plus D x ('State-space models', Recurrence and
    convolution; 'Structured State Space Models and Mamba', LTI unroll).
    Abar^k is built by repeated multiplication, the convolution by np.convolve."""
    w = make_workload("lti_small", batch=2, seqlen=512, dim=8, dstate=16, seed=1,
                      a_init="s4d_real", gate=False, lti=True, with_bias=False)
    out, _ = oracle.selective_scan(w.x, w.delta, w.A, w.B, w.C, D=w.D,
                                   delta_softplus=False, per_channel_bc=True)
    dt = w.delta[0, 0, :].astype(np.float64)
    A, B, C = (w.A.astype(np.float64), w.B.astype(np.float64), w.C.astype(np.float64))
    Abar = np.exp(dt[:, None] * A)                               # (dim, N)
    powers = np.cumprod(np.concatenate([np.ones((w.dim, w.dstate, 1)),
                                        np.repeat(Abar[:, :, None], w.seqlen - 1, axis=2)],
                                       axis=2), axis=2)          # Abar^k, k = 0..L-1
    K = np.einsum("dn,dnk,dn->dk", C, powers, dt[:, None] * B)
    ref = np.empty_like(out)
    for b in range(w.batch):
        for d in range(w.dim):
            xs = w.x[b, :, d].astype(np.float64)
            ref[b, :, d] = np.convolve(xs, K[d])[: w.seqlen] + w.D[d] * xs
    assert floored_rel_err(out, ref) < 1e-12
    # the oracle's own kernel and O(L^2) convolution agree with the same identity
    assert floored_rel_err(oracle.lti_kernel(w.A, w.B, w.C, dt, w.seqlen), K) < 1e-12
    assert floored_rel_err(oracle.causal_conv(w.x, K, w.D), ref) < 1e-12


def test_impulse_response_and_shift_invariance():
    """Feeding 1, 0, 0, ... returns the kernel K ('State-space models',
    Recurrence and convolution); the response to a later impulse is a
    translated copy (rugvailabs page, S4D section)."""
    w = make_workload("lti_imp", batch=1, seqlen=40, dim=3, dstate=4, seed=5,
                      a_init="random", gate=False, lti=True, with_bias=False)
    dt = w.delta[0, 0, :].astype(np.float64)
    K = oracle.lti_kernel(w.A, w.B, w.C, dt, w.seqlen)
    resp = {}
    for s in (0, 7):
        x = np.zeros_like(w.x)
        x[0, s, :] = 1.0
        out, _ = oracle.selective_scan(x, w.delta, w.A, w.B, w.C, D=w.D,
                                       delta_softplus=False, per_channel_bc=True)
        resp[s] = out[0]
    expect = K.T.copy()
    expect[0] += w.D
    assert floored_rel_err(resp[0], expect) < 1e-13
    assert np.all(resp[7][:7] == 0.0)
    assert floored_rel_err(resp[7][7:], resp[0][: w.seqlen - 7]) < 1e-13


# --------------------------------------------------------------- brute force

def _brute_force(w, bbar_mode):
    """h_t = (prod_{r<=t} Abar_r) h0 + sum_{s<=t} (prod_{r=s+1..t} Abar_r) Bbar_s x_s,
    each product formed explicitly ('Structured State Space Models and Mamba',
    parallel associative scan: the composition of the per-step maps)."""
    f = (lambda a: bf16_bits_to_f32(a).astype(np.float64)) if w.io == "bf16" else \
        (lambda a: np.asarray(a, dtype=np.float64))
    x, dl = f(w.x), f(w.delta)
    B = np.asarray(w.B, np.float64) if w.per_channel_bc else f(w.B)
    C = np.asarray(w.C, np.float64) if w.per_channel_bc else f(w.C)
    z = None if w.z is None else f(w.z)
    A = w.A.astype(np.float64)
    bias = np.zeros(w.dim) if w.delta_bias is None else w.delta_bias.astype(np.float64)
    Dk = np.zeros(w.dim) if w.D is None else w.D.astype(np.float64)
    out = np.zeros((w.batch, w.seqlen, w.dim))
    fin = np.zeros((w.batch, w.dim, w.dstate))
    for b in range(w.batch):
        for d in range(w.dim):
            v = dl[b, :, d] + bias[d]
            step = np.logaddexp(0.0, v) if w.delta_softplus else v
            for n in range(w.dstate):
                abar = np.exp(step * A[d, n])
                Bv = B[d, n] * np.ones(w.seqlen) if w.per_channel_bc else B[b, :, n]
                if bbar_mode == 0:
                    bbar = step * Bv
                else:
                    bbar = (abar - 1.0) / A[d, n] * Bv
                Cv = C[d, n] * np.ones(w.seqlen) if w.per_channel_bc else C[b, :, n]
                h0 = 0.0 if w.h0 is None else float(w.h0[b, d, n])
                for t in range(w.seqlen):
                    h = np.prod(abar[: t + 1]) * h0
                    for s in range(t + 1):
                        h += np.prod(abar[s + 1: t + 1]) * bbar[s] * x[b, s, d]
                    out[b, t, d] += Cv[t] * h
                    if t == w.seqlen - 1:
                        fin[b, d, n] = h
            out[b, :, d] += Dk[d] * x[b, :, d]
            if z is not None:
                out[b, :, d] *= z[b, :, d] / (1.0 + np.exp(-z[b, :, d]))
    return out, fin


@pytest.mark.parametrize("case", [
    dict(io="f32", gate=True, state_in=False, a_init="random", bbar_mode=0),
    dict(io="f32", gate=False, state_in=True, a_init="s4d_real", bbar_mode=0),
    dict(io="bf16", gate=True, state_in=True, a_init="random", bbar_mode=0),
    dict(io="f32", gate=True, state_in=True, a_init="random", bbar_mode=1),
    dict(io="f32", gate=True, state_in=False, a_init="random", bbar_mode=0, with_D=False, with_bias=False),
    dict(io="f32", gate=False, state_in=False, a_init="random", bbar_mode=1, lti=True, with_bias=False),
])
def test_brute_force_tiny(case):
    case = dict(case)
    bbar_mode = case.pop("bbar_mode")
    w = make_workload("bf", batch=2, seqlen=11, dim=3, dstate=4, seed=17, **case)
    out, fin = oracle.selective_scan(w.x, w.delta, w.A, w.B, w.C, D=w.D, z=w.z,
                                     delta_bias=w.delta_bias, h0=w.h0,
                                     delta_softplus=w.delta_softplus, bbar_mode=bbar_mode,
                                     per_channel_bc=w.per_channel_bc, io_dtype=w.io)
    ref_out, ref_fin = _brute_force(w, bbar_mode)
    assert floored_rel_err(out, ref_out) < 1e-13
    assert floored_rel_err(fin, ref_fin) < 1e-13


# ------------------------------------------------------------ scan algebra

def _combine(p, q):
    """(a1, b1) then (a2, b2) = (a1 a2, a2 b1 + b2)  ('State-space models',
    The parallel scan; llms.blog, Hardware-Aware Parallel Associative Scan)."""
    return (p[0] * q[0], q[0] * p[1] + q[1])


def test_combine_is_associative():
    rng = np.random.default_rng(3)
    for _ in range(200):
        e = [(rng.uniform(0, 1), rng.standard_normal()) for _ in range(3)]
        l = _combine(_combine(e[0], e[1]), e[2])
        r = _combine(e[0], _combine(e[1], e[2]))
        assert l[0] == pytest.approx(r[0], rel=1e-14) and l[1] == pytest.approx(r[1], rel=1e-12, abs=1e-14)


def test_tree_scan_matches_oracle_state():
    """A pairwise (tree-order) reduction of the per-step maps reaches the same
    final state as the oracle's sequential recurrence."""
    w = make_workload("tree", batch=1, seqlen=37, dim=2, dstate=3, seed=23, state_in=True)
    _, fin = oracle.selective_scan(w.x, w.delta, w.A, w.B, w.C, D=w.D, z=w.z,
                                   delta_bias=w.delta_bias, h0=w.h0)
    for d in range(w.dim):
        step = np.logaddexp(0.0, w.delta[0, :, d].astype(np.float64) + float(w.delta_bias[d]))
        for n in range(w.dstate):
            elems = [(math.exp(s * float(w.A[d, n])), s * float(w.B[0, t, n]) * float(w.x[0, t, d]))
                     for t, s in enumerate(step)]
            while len(elems) > 1:
                nxt = [_combine(elems[i], elems[i + 1]) for i in range(0, len(elems) - 1, 2)]
                if len(elems) % 2:
                    nxt.append(elems[-1])
                elems = nxt
            a_all, b_all = elems[0]
            h = a_all * float(w.h0[0, d, n]) + b_all
            assert h == pytest.approx(fin[0, d, n], rel=1e-12, abs=1e-14)


# -------------------------------------------------------------- invariants

def test_split_resume_equals_single_scan():
    """Final state is a checkpoint: scan(L1) then scan(L2) from it = scan(L1 + L2)
    (constant-size state at inference: rugvailabs page, comparison table)."""
    w = make_workload("split", batch=2, seqlen=50, dim=4, dstate=5, seed=29, io="bf16")
    kw = dict(D=w.D, delta_bias=w.delta_bias, io_dtype="bf16")
    full, fin = oracle.selective_scan(w.x, w.delta, w.A, w.B, w.C, z=w.z, **kw)
    cut = 19
    sl = lambda a, s: a[:, s]
    o1, s1 = oracle.selective_scan(sl(w.x, slice(0, cut)), sl(w.delta, slice(0, cut)), w.A,
                                   sl(w.B, slice(0, cut)), sl(w.C, slice(0, cut)),
                                   z=sl(w.z, slice(0, cut)), **kw)
    o2, s2 = oracle.selective_scan(sl(w.x, slice(cut, None)), sl(w.delta, slice(cut, None)), w.A,
                                   sl(w.B, slice(cut, None)), sl(w.C, slice(cut, None)),
                                   z=sl(w.z, slice(cut, None)), h0=s1, **kw)
    assert np.array_equal(np.concatenate([o1, o2], axis=1), full)
    assert np.array_equal(s2, fin)


def test_zero_length_and_channel_sampling():
    w = make_workload("z", batch=2, seqlen=0, dim=3, dstate=2, seed=1, state_in=True)
    out, fin = oracle.selective_scan(w.x, w.delta, w.A, w.B, w.C, D=w.D, z=w.z,
                                     delta_bias=w.delta_bias, h0=w.h0)
    assert out.shape == (2, 0, 3) and np.array_equal(fin, w.h0.astype(np.float64))
    w = make_workload("s", batch=3, seqlen=9, dim=5, dstate=2, seed=2)
    out, fin = oracle.selective_scan(w.x, w.delta, w.A, w.B, w.C, D=w.D, z=w.z,
                                     delta_bias=w.delta_bias)
    picks = [(0, 4), (2, 1), (2, 3)]
    res = oracle.selective_scan_channels(picks, w.x, w.delta, w.A, w.B, w.C, D=w.D, z=w.z,
                                         delta_bias=w.delta_bias)
    for (b, d) in picks:
        assert np.array_equal(res[(b, d)][0], out[b, :, d])
        assert np.array_equal(res[(b, d)][1], fin[b, d])


def test_workload_recipe():
    """bias = log(expm1(dt)) is the value whose softplus is dt; bf16 rounding is
    nearest-even; stored bf16 widens exactly."""
    w = make_workload("r", batch=1, seqlen=4, dim=6, dstate=2, seed=0)
    rng = np.random.Generator(np.random.PCG64(0))
    rng.standard_normal((1, 4, 6), dtype=np.float32)
    rng.standard_normal((1, 4, 6), dtype=np.float32)
    dt = rng.uniform(0.001, 0.1, size=6)
    for d in range(6):
        assert oracle.softplus(float(w.delta_bias[d])) == pytest.approx(dt[d], rel=1e-6)
    vals = np.array([1.0, 1.00390625, 1.005859375, 1.0078125 + 2 ** -9, -3.14159, 1e-30],
                    dtype=np.float32)
    bits = f32_to_bf16_bits(vals)
    back = bf16_bits_to_f32(bits)
    assert back[0] == 1.0 and back[1] == 1.0            # tie 1 + 2^-8 -> even mantissa (1.0)
    assert back[2] == 1.0078125
    assert np.all(np.abs(back - vals) <= np.abs(vals) * 2.0 ** -8)
    assert np.array_equal(oracle.widen(bits, "bf16"), back.astype(np.float64))


# ---------------------------------------------------------- block prologue (conv + silu)
# "State-space models", section "Mamba: selection", the block description: a depthwise
# causal convolution of width 4 and a silu on the branch that feeds the SSM.

def _silu(v):
    return v / (1.0 + np.exp(-v))


def test_conv_silu_matches_library_convolution():
    """pre = numpy's full linear convolution of each channel (the history prepended),
    truncated causally; u = silu(pre + bias).  hist_out = the last three inputs."""
    rng = np.random.default_rng(11)
    batch, L, dim, W = 2, 23, 5, oracle.CONV_WIDTH
    x = rng.normal(size=(batch, L, dim)).astype(np.float32)
    w = rng.normal(size=(dim, W)).astype(np.float32)
    cb = rng.normal(size=dim).astype(np.float32)
    hist = rng.normal(size=(batch, dim, W - 1)).astype(np.float32)
    u, hout = oracle.conv_silu(x, w, cb, hist)
    for b in range(batch):
        for d in range(dim):
            ext = np.concatenate([hist[b, d].astype(np.float64), x[b, :, d].astype(np.float64)])
            pre = np.convolve(ext, w[d].astype(np.float64))[W - 1:W - 1 + L] + cb[d]
            np.testing.assert_allclose(u[b, :, d], _silu(pre), rtol=1e-13, atol=1e-14)
            np.testing.assert_array_equal(hout[b, d], ext[-(W - 1):])


def test_conv_silu_impulse_response_and_causality():
    """A unit impulse at step s gives pre = w[d, t - s] for s <= t < s + 4 and 0
    elsewhere (no bias, zero history): the taps in lag order, nothing before s."""
    L, dim, W, s = 12, 3, oracle.CONV_WIDTH, 5
    w = np.array([[0.5, -1.25, 2.0, 0.75], [1.0, 0.0, 0.0, 0.0], [-0.5, 0.25, -0.125, 3.0]])
    x = np.zeros((1, L, dim))
    x[0, s, :] = 1.0
    u, _ = oracle.conv_silu(x, w)
    for d in range(dim):
        pre = np.zeros(L)
        pre[s:s + W] = w[d]
        np.testing.assert_allclose(u[0, :, d], _silu(pre), rtol=0, atol=1e-15)
        assert np.all(u[0, :s, d] == 0.0)


def test_conv_silu_identity_taps_and_silu_values():
    """Taps (1, 0, 0, 0) and no bias: u = silu(x).  silu(0) = 0, silu(v) -> v for
    large v and -> 0 for very negative v; silu(1) = 1 / (1 + 1/e)."""
    x = np.array([0.0, 1.0, 40.0, -40.0, -1.0]).reshape(1, 5, 1)
    u, _ = oracle.conv_silu(x, np.array([[1.0, 0.0, 0.0, 0.0]]))
    assert u[0, 0, 0] == 0.0
    assert abs(u[0, 1, 0] - 1.0 / (1.0 + math.exp(-1.0))) < 1e-16
    assert abs(u[0, 2, 0] - 40.0) < 1e-15
    assert 0.0 > u[0, 3, 0] > -1e-15
    assert abs(u[0, 4, 0] - (-1.0 / (1.0 + math.e))) < 1e-16


@pytest.mark.parametrize("split", [1, 2, 3, 9])
def test_conv_silu_history_continuation(split):
    """Running a sequence in two calls, the second starting from the first call's
    hist_out, equals one call over the whole sequence (also for a first part
    shorter than the history, where hist_out still holds older inputs)."""
    rng = np.random.default_rng(split)
    batch, L, dim = 2, 14, 4
    x = rng.normal(size=(batch, L, dim))
    w = rng.normal(size=(dim, oracle.CONV_WIDTH))
    cb = rng.normal(size=dim)
    h0 = rng.normal(size=(batch, dim, oracle.CONV_WIDTH - 1))
    u_all, h_all = oracle.conv_silu(x, w, cb, h0)
    u1, h1 = oracle.conv_silu(x[:, :split], w, cb, h0)
    u2, h2 = oracle.conv_silu(x[:, split:], w, cb, h1)
    np.testing.assert_array_equal(np.concatenate([u1, u2], axis=1), u_all)
    np.testing.assert_array_equal(h2, h_all)


def test_conv_scan_composes_prologue_and_scan():
    """The fused-block oracle is the prologue followed by the scan on its output:
    with taps (1, 0, 0, 0) and no bias it equals the scan of silu(x)."""
    w = make_workload("cs", batch=2, seqlen=40, dim=6, dstate=4, io="f32", seed=5)
    taps = np.tile(np.array([[1.0, 0.0, 0.0, 0.0]]), (w.dim, 1))
    out, st, hout = oracle.conv_selective_scan(
        w.x, taps, None, None, w.delta, w.A, w.B, w.C, w.D, w.z, w.delta_bias)
    ref, ref_st = oracle.selective_scan(_silu(w.x.astype(np.float64)), w.delta, w.A, w.B, w.C,
                                        w.D, w.z, w.delta_bias)
    np.testing.assert_allclose(out, ref, rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(st, ref_st, rtol=1e-14, atol=1e-14)
    np.testing.assert_array_equal(hout, w.x[:, -3:, :].transpose(0, 2, 1).astype(np.float64))


# ------------------------------------------------------------------ backward pass
# "State-space models", section "The parallel scan": the fused kernel rebuilds the
# expanded state in the backward pass.  The oracle's gradients are pinned against
# central finite differences of the forward oracle, and against torch autograd
# through a separately written float64 forward.

def _bwd_case(seed, *, gate=True, with_D=True, with_bias=True, state_in=True, softplus=True):
    w = make_workload("bwd", batch=2, seqlen=7, dim=3, dstate=4, io="f32", seed=seed, gate=gate,
                      with_D=with_D, with_bias=with_bias, state_in=state_in)
    rng = np.random.default_rng(seed + 100)
    f = lambda a: None if a is None else np.asarray(a, dtype=np.float64).copy()
    inp = dict(x=f(w.x), delta=f(w.delta), A=f(w.A), B=f(w.B), C=f(w.C), D=f(w.D), z=f(w.z),
               delta_bias=f(w.delta_bias), h0=f(w.h0))
    if not softplus:  # raw steps, small and positive
        inp["delta"] = np.abs(inp["delta"]) * 0.3
        inp["delta_bias"] = None
    dout = rng.standard_normal(w.x.shape)
    dfinal = rng.standard_normal((w.batch, w.dim, w.dstate)) if state_in else None
    return inp, dout, dfinal, softplus


def _loss(inp, dout, dfinal, softplus):
    out, st = oracle.selective_scan(inp["x"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                                    inp["z"], inp["delta_bias"], inp["h0"], delta_softplus=softplus)
    return float(np.sum(out * dout) + (np.sum(st * dfinal) if dfinal is not None else 0.0))


@pytest.mark.parametrize("variant", [dict(), dict(gate=False, with_D=False),
                                     dict(with_bias=False, state_in=False), dict(softplus=False)],
                         ids=["full", "no_gate_no_D", "no_bias_no_state", "no_softplus"])
def test_backward_matches_finite_differences(variant):
    """Every gradient the oracle returns equals the central difference of the loss
    sum(dout * out) + sum(dfinal * final_state) under the forward oracle."""
    inp, dout, dfinal, sp = _bwd_case(3, **variant)
    g = oracle.selective_scan_bwd(inp["x"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                                  inp["z"], inp["delta_bias"], inp["h0"], dout=dout, dfinal=dfinal,
                                  delta_softplus=sp)
    names = [("x", "dx"), ("delta", "ddelta"), ("A", "dA"), ("B", "dB"), ("C", "dC"), ("D", "dD"),
             ("z", "dz"), ("delta_bias", "dbias"), ("h0", "dh0")]
    for arg, gname in names:
        if inp[arg] is None:
            continue
        base = inp[arg]
        fd = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            eps = 1e-6 * max(1.0, abs(base[idx]))
            old = base[idx]
            base[idx] = old + eps
            lp = _loss(inp, dout, dfinal, sp)
            base[idx] = old - eps
            lm = _loss(inp, dout, dfinal, sp)
            base[idx] = old
            fd[idx] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(g[gname], fd, rtol=2e-6, atol=2e-7, err_msg=gname)


def test_backward_matches_autograd_of_an_independent_forward():
    """torch autograd through a float64 forward written with cumulative sums of the
    step sizes (exp(A (S_t - S_s)) weights) instead of the recurrence."""
    torch = pytest.importorskip("torch")
    inp, dout, dfinal, sp = _bwd_case(5)
    T = {k: (None if v is None else torch.tensor(v, dtype=torch.float64, requires_grad=True))
         for k, v in inp.items()}
    v = T["delta"] + T["delta_bias"]
    dt = torch.nn.functional.softplus(v)                                  # (b, L, d)
    S = torch.cumsum(dt, dim=1)                                           # S_t = sum_{s<=t} dt_s
    # h_t[n] = exp(A (S_t)) h0 + sum_{s<=t} exp(A (S_t - S_s)) dt_s B_s x_s
    Ab = T["A"][None, None]                                               # (1, 1, d, n)
    decay_all = torch.exp(Ab * S[..., None])                              # (b, L, d, n)
    L = dt.shape[1]
    mask = torch.tril(torch.ones(L, L, dtype=torch.float64))              # s <= t
    W = torch.exp(Ab[:, :, None] * (S[:, :, None, :, None] - S[:, None, :, :, None]))  # (b, t, s, d, n)
    W = W * mask[None, :, :, None, None]
    inj = dt[..., None] * T["B"][:, :, None, :] * T["x"][..., None]       # (b, s, d, n)
    h = decay_all * T["h0"][:, None] + torch.einsum("btsdn,bsdn->btdn", W, inj)
    y = torch.einsum("btdn,btn->btd", h, T["C"]) + T["D"] * T["x"]
    out = y * T["z"] * torch.sigmoid(T["z"])
    loss = (out * torch.tensor(dout)).sum() + (h[:, -1] * torch.tensor(dfinal)).sum()
    loss.backward()
    g = oracle.selective_scan_bwd(inp["x"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                                  inp["z"], inp["delta_bias"], inp["h0"], dout=dout, dfinal=dfinal)
    for arg, gname in [("x", "dx"), ("delta", "ddelta"), ("A", "dA"), ("B", "dB"), ("C", "dC"),
                       ("D", "dD"), ("z", "dz"), ("delta_bias", "dbias"), ("h0", "dh0")]:
        np.testing.assert_allclose(g[gname], T[arg].grad.numpy(), rtol=1e-11, atol=1e-12, err_msg=gname)


# ------------------------------------------------ Mamba-2 SSD (scalar decay per head)

def _ssd_case(seed, *, batch=2, L=23, H=4, P=3, G=2, N=5, state_in=True, gate=True):
    from selective_state_space_112_b300.workloads import make_ssd
    return make_ssd("pin", batch, L, H, P, N, ngroups=G, seed=seed, gate=gate, state_in=state_in)


def _ssd_inputs64(w):
    wd = lambda a: None if a is None else oracle.widen(a, "bf16")
    f = lambda a: None if a is None else np.asarray(a, dtype=np.float64)
    return (wd(w.x), wd(w.dt), f(w.A), wd(w.B), wd(w.C), f(w.D), wd(w.z), f(w.dt_bias), f(w.h0))


def _ssd(w, **kw):
    return oracle.ssd(w.x, w.dt, w.A, w.B, w.C, D=w.D, z=w.z, dt_bias=w.dt_bias, h0=w.h0, **kw)


def _masked_attention(w, zero_decay=False, softplus=True):
    """'Structured State Space Models and Mamba', section 'State Space Duality and
    Mamba-2': Y = (L o (Q K^T)) V with Q = C, K = B, V = step * x and the
    1-semiseparable L[i, j] = exp(A (S_i - S_j)) for j <= i (S = cumulative step
    sums), plus the initial state's decayed readout, D x and the gate; the final
    state is the same sum read at the last step.  One dense matrix per (b, head)."""
    x, dtr, A, B, C, D, z, bias, h0 = _ssd_inputs64(w)
    batch, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    v = dtr + (0.0 if bias is None else bias)
    step = np.logaddexp(0.0, v) if softplus else v                # softplus, (b, L, H)
    out = np.empty_like(x)
    fin = np.empty((batch, H, P, N))
    for b in range(batch):
        for h in range(H):
            g = h // (H // G)
            a = 0.0 if zero_decay else A[h]
            S = np.cumsum(step[b, :, h])
            Lm = np.tril(np.exp(a * (S[:, None] - S[None, :])))   # (L, L)
            QK = C[b, :, g] @ B[b, :, g].T                        # (L, L)
            V = step[b, :, h, None] * x[b, :, h]                  # (L, P)
            y = (Lm * QK) @ V
            st = np.zeros((P, N)) if h0 is None else h0[b, h]
            y += np.exp(a * S)[:, None] * (C[b, :, g] @ st.T)     # decayed initial state
            if D is not None:
                y += D[h] * x[b, :, h]
            if z is not None:
                y *= z[b, :, h] / (1.0 + np.exp(-z[b, :, h]))
            out[b, :, h] = y
            wlast = np.exp(a * (S[-1] - S)) * step[b, :, h]       # (L,)
            fin[b, h] = np.exp(a * S[-1]) * st + (x[b, :, h] * wlast[:, None]).T @ B[b, :, g]
    return out, fin


@pytest.mark.parametrize("seed,state_in,gate", [(31, True, True), (32, False, True), (33, True, False)])
def test_ssd_equals_masked_attention_form(seed, state_in, gate):
    """The recurrence and the pages' masked-attention form give the same outputs and
    final state (two heads per group, so the head-to-group map is exercised)."""
    w = _ssd_case(seed, state_in=state_in, gate=gate)
    out, st = _ssd(w)
    ref, ref_st = _masked_attention(w)
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(st, ref_st, rtol=1e-11, atol=1e-12)


def test_ssd_is_the_selective_scan_with_a_tied_decay():
    """'State-space models', section 'The parallel scan': Mamba-2 is the selective
    SSM with A a scalar times the identity per head.  Every channel p of head h is
    a channel of the S6 scan with A[d, n] = A[h], its head's step and D, and its
    group's B and C, so the already pinned S6 oracle must give the same numbers."""
    w = _ssd_case(34, G=2, H=4, P=3, N=5)
    out, st = _ssd(w)
    x, dtr, A, B, C, D, z, bias, h0 = _ssd_inputs64(w)
    batch, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    for g in range(G):
        heads = [h for h in range(H) if h // (H // G) == g]
        xs = x[:, :, heads].reshape(batch, L, -1)
        ds = np.repeat(dtr[:, :, heads], P, axis=2)
        A1 = np.repeat(A[heads], P)[:, None] * np.ones((1, N))
        o1, s1 = oracle.selective_scan(
            xs, ds, A1, B[:, :, g], C[:, :, g], D=np.repeat(D[heads], P),
            z=z[:, :, heads].reshape(batch, L, -1), delta_bias=np.repeat(bias[heads], P),
            h0=h0[:, heads].reshape(batch, -1, N))
        np.testing.assert_allclose(out[:, :, heads].reshape(batch, L, -1), o1, rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(st[:, heads].reshape(batch, -1, N), s1, rtol=1e-13, atol=1e-14)


def test_ssd_step_without_softplus():
    """With dt_softplus off the step is dt + dt_bias as given (small positive raw
    steps here), in the masked-attention form as well."""
    w = _ssd_case(38, state_in=True)
    raw = np.abs(np.random.default_rng(38).standard_normal(w.dt.shape)).astype(np.float32) * 0.1
    w.dt = f32_to_bf16_bits(raw)
    w.dt_bias = np.full(w.nheads, 0.01, np.float32)
    out, st = _ssd(w, dt_softplus=False)
    ref, ref_st = _masked_attention(w, softplus=False)
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(st, ref_st, rtol=1e-11, atol=1e-12)


def test_ssd_zero_decay_is_causal_linear_attention():
    """The rugvailabs.com page on state-space models and Mamba, its passage on
    Mamba-2 and state space duality: linear attention without softmax is the SSM
    with input-dependent B and C and an identity transition.  With A = 0
    the output is sum_{s <= t} (C_t . B_s) step_s x_s plus D x, gated."""
    w = _ssd_case(35, state_in=False)
    w.A = np.zeros_like(w.A)
    out, st = _ssd(w)
    ref, ref_st = _masked_attention(w, zero_decay=True)
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(st, ref_st, rtol=1e-11, atol=1e-12)


def test_ssd_split_resume_and_state_layout():
    """Two calls carrying the (b, H, P, N) state equal one call; the state of a
    single step from zero is step * B[n] * x[p] at index [b, h, p, n]."""
    w = _ssd_case(36, state_in=True, L=17)
    out, st = _ssd(w)
    from dataclasses import replace
    w1 = replace(w, x=w.x[:, :9], dt=w.dt[:, :9], B=w.B[:, :9], C=w.C[:, :9], z=w.z[:, :9])
    o1, s1 = _ssd(w1)
    w2 = replace(w, x=w.x[:, 9:], dt=w.dt[:, 9:], B=w.B[:, 9:], C=w.C[:, 9:], z=w.z[:, 9:], h0=s1)
    o2, s2 = _ssd(w2)
    np.testing.assert_allclose(np.concatenate([o1, o2], axis=1), out, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(s2, st, rtol=1e-12, atol=1e-13)
    w0 = _ssd_case(37, state_in=False, L=1, G=1, H=2, P=3, N=4)
    _, s = _ssd(w0)
    x, dtr, A, B, C, D, z, bias, h0 = _ssd_inputs64(w0)
    step = np.logaddexp(0.0, dtr[:, 0] + bias)                    # (b, H)
    for b in range(2):
        for h in range(2):
            np.testing.assert_allclose(s[b, h], step[b, h] * np.outer(x[b, 0, h], B[b, 0, 0]),
                                       rtol=1e-14)
