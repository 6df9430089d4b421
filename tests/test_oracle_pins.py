"""The fp64 oracle against its pins (CPU only), and proof that the pins bite.

``test_pin`` runs every pin against the oracle as built.  ``test_mutants``
compiles deliberately broken copies of the oracle source (each a plausible
mistake: a dropped term, a wrong sign or index, the readout before the update)
and checks that at least one pin rejects every one of them.
"""
import os
import shutil
import tempfile

import numpy as np
import pytest

import oracle
import pins

ORACLE_SRC = os.path.join(os.path.dirname(oracle.__file__), "ssm_oracle.c")


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle.load())


def test_lti_convolution_zoh():
    pins.pin_lti_equals_convolution(oracle.load(), disc=oracle.DISC_ZOH)


# (original text, mutated text) pairs; each must occur exactly once in the source
MUTANTS = [
    ("h[n] = abar * h[n] + bx;", "h[n] = abar * h[n] - bx;"),
    ("double v = y[t] + Dd * u[t];", "double v = y[t];"),
    ("double abar = exp(dts[t] * Ad[n]);", "double abar = exp(-dts[t] * Ad[n]);"),
    ("h[n] = abar * h[n] + bx;\n                    acc += Cb[n * L + t] * h[n];",
     "acc += Cb[n * L + t] * h[n];\n                    h[n] = abar * h[n] + bx;"),
    ("log1p(exp(-fabs(s)))", "log1p(exp(fabs(s)))"),
    ("if (z) v *= z[t] * sigmoid(z[t]);", "if (z) v *= sigmoid(z[t]);"),
    ("double s = delta + bias;", "double s = delta;"),
    ("double bx = input_term(dts[t], Ad[n], Bb[n * L + t], u[t], j->disc);",
     "double bx = input_term(dts[t], Ad[n], Bb[t * N + n], u[t], j->disc);"),
    ("static double sigmoid(double v) { return 1.0 / (1.0 + exp(-v)); }",
     "static double sigmoid(double v) { return 1.0 / (1.0 + exp(v)); }"),
    ("return dt * b * x; /* Euler: Bbar = Delta B */", "return dt * b; /* Euler: Bbar = Delta B */"),
    ("return expm1(dt * a_cont) / a_cont * b * x;", "return expm1(dt * a_cont) * b * x;"),
    ("h[n] = j->h0 ? j->h0[c * N + n] : 0.0;", "h[n] = 0.0;"),
    ("double hn = abar * state[c * N + n] + bx;", "double hn = state[c * N + n] + bx;"),
    ("xb[r] = la * pb + lb;", "xb[r] = pa * lb + pb;"),
    ("eb[t] = a[t] * xb[t] + b[t];", "eb[t] = xb[t] + b[t];"),
    ("acc += Cb[n * L + t] * hs[t * N + n];", "acc += Cb[n * L + t] * hs[n];"),
    # the causal convolution
    ("const int64_t src = t - (W - 1) + k;", "const int64_t src = t - W + k;"),
    ("v += w[d * W + k] * xv;", "v += w[d * W + (W - 1 - k)] * xv;"),
    ("double v = bias ? bias[d] : 0.0;\n                for", "double v = 0.0;\n                for"),
    ("x_hist[row * (W - 1) + (W - 1) + src]", "x_hist[row * (W - 1) - src - 1]"),
    ("out[row * L + t] = use_silu ? v * sigmoid(v) : v;", "out[row * L + t] = use_silu ? sigmoid(v) : v;"),
    # the backward pass
    ("lam[n] = lt * at;", "lam[n] = lt;"),
    ("dDelta += lt * (hprev * at * Ad[n] + bu * dg_dDelta);", "dDelta += lt * hprev * at * Ad[n];"),
    ("dz[c * L + t] = dyc[t] * pre[t] * sg * (1.0 + zc[t] * (1.0 - sg));", "dz[c * L + t] = dyc[t] * pre[t] * sg;"),
    ("dA[d * N + n] += lt * (hprev * at * dts[t] + bu * dg_dA);", "dA[d * N + n] += lt * (hprev * at + bu * dg_dA);"),
    ("if (dDskip) dDskip[d] += yt * uc[t];", "if (dDskip) dDskip[d] += dyc[t] * uc[t];"),
    ("dCm[b * N * L + n * L + t] += yt * hs[(t + 1) * N + n];", "dCm[b * N * L + n * L + t] += yt * hs[t * N + n];"),
    ("const double dd = delta_softplus ? dDelta * sigmoid(dl[t] + bias) : dDelta;",
     "const double dd = dDelta;"),
    ("du_acc += lt * g * Bb[n * L + t];", "du_acc += lt * Bb[n * L + t];"),
    # the backward pass with the exact-ZOH input term
    ("const double dg_dDelta = zoh ? at : 1.0;", "const double dg_dDelta = 1.0;"),
    ("const double dg_dA = zoh ? zoh_coef_dA(dts[t], Ad[n]) : 0.0;", "const double dg_dA = 0.0;"),
    ("psi = 0.5 + x / 3.0 + x * x / 8.0 + x * x * x / 30.0;", "psi = 0.5 + x / 2.0 + x * x / 8.0 + x * x * x / 30.0;"),
    ("psi = (x * exp(x) - expm1(x)) / (x * x);", "psi = (x * exp(x) - expm1(x)) / x;"),
    ("const double g = zoh ? (Ad[n] == 0.0 ? dts[t] : expm1(dts[t] * Ad[n]) / Ad[n]) : dts[t];",
     "const double g = dts[t];"),
    # the complex (S4D-Lin) scan
    ("double v = creal(acc) + Dd * ut;", "double v = cimag(acc) + Dd * ut;"),
    ("const double complex abar = cexp(dt * a);", "const double complex abar = cexp(dt * conj(a));"),
    ("const double complex abar = cexp(dt * a);", "const double complex abar = exp(dt * creal(a));"),
    ("h[n] = abar * h[n] + dt * Bm[b * N * L + n * L + t] * ut;",
     "h[n] = abar * h[n] + I * dt * Bm[b * N * L + n * L + t] * ut;"),
    ("h[n] = h0 ? h0[2 * (c * N + n)] + I * h0[2 * (c * N + n) + 1] : 0.0;",
     "h[n] = h0 ? h0[2 * (c * N + n)] : 0.0;"),
    ("h_last[2 * (c * N + n) + 1] = cimag(h[n]);", "h_last[2 * (c * N + n) + 1] = -cimag(h[n]);"),
    # the Mamba-2 SSD layer
    ("h[p * N + n] = abar * h[p * N + n] + dt * Bm[(b * L + t) * N + n] * xt;",
     "h[p * N + n] = abar * h[p * N + n] + Bm[(b * L + t) * N + n] * xt;"),
    ("const double abar = exp(dt * a[hd]);", "const double abar = exp(dt * a[0]);"),
    ("acc += Cm[(b * L + t) * N + n] * h[p * N + n];", "acc += Cm[(b * L + t) * N + n] * h[n];"),
    ("double v = acc + Dh * xt;", "double v = acc;"),
    ("h[i] = h0 ? h0[((b * H + hd) * P) * N + i] : 0.0;", "h[i] = 0.0;"),
    ("h[p * N + n] = abar * h[p * N + n] + dt * Bm[(b * L + t) * N + n] * xt;",
     "h[p * N + n] = abar * h[p * N + n] + dt * Bm[(b * N + n) * L + t] * xt;"),
]


def _run_pins(lib):
    failed = []
    for pin in pins.ALL_PINS + [lambda l: pins.pin_lti_equals_convolution(l, disc=oracle.DISC_ZOH)]:
        try:
            pin(lib)
        except (AssertionError, RuntimeError, FloatingPointError):
            failed.append(getattr(pin, "__name__", "lti_zoh"))
    return failed


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc needed to build mutants")
@pytest.mark.parametrize("orig,mut", MUTANTS, ids=[f"m{i}" for i in range(len(MUTANTS))])
def test_mutants(orig, mut):
    src = open(ORACLE_SRC).read()
    assert src.count(orig) == 1, f"mutation anchor not unique: {orig!r}"
    with tempfile.TemporaryDirectory() as td:
        path = os.path.join(td, "mut.c")
        with open(path, "w") as f:
            f.write(src.replace(orig, mut))
        so = oracle.compile_oracle(path, os.path.join(td, "libmut.so"))
        lib = oracle.load(so)
        with np.errstate(all="ignore"):
            failed = _run_pins(lib)
    assert failed, f"no pin caught mutation {mut!r}"


def test_state_update_does_not_touch_input():
    rng = np.random.default_rng(0)
    st = rng.standard_normal((1, 2, 3))
    keep = st.copy()
    oracle.state_update(st, rng.standard_normal((1, 2)), rng.standard_normal((1, 2)),
                        -np.ones((2, 3)), rng.standard_normal((1, 3)), rng.standard_normal((1, 3)))
    assert np.array_equal(st, keep)


def test_oracle_rejects_bad_args():
    lib = oracle.load()
    rc = lib.oracle_selective_scan(1, 1, 1, 1, None, None, None, None, None, None, None, None, None,
                                   1, 0, 0, None, None, 1)
    assert rc == -1


def test_oracle_empty_is_ok():
    y = oracle.selective_scan(np.zeros((0, 3, 5)), np.zeros((0, 3, 5)), -np.ones((3, 2)),
                              np.zeros((0, 2, 5)), np.zeros((0, 2, 5)))
    assert y.shape == (0, 3, 5)
