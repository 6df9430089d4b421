"""Pins that tie the fp64 oracle to facts fixed by the pages and by mathematics.

Each pin takes an oracle library handle (``oracle.load()`` or a deliberately
broken build of it) and raises AssertionError when the oracle disagrees.  None
of them re-types the oracle's own loop: each checks against a different
formula, a hand-worked value, a limit, or an invariant.

Sources (pages on the Mamba selective SSM):
  * "Mamba and state space models" (docs.ifdog.com): sections "Discretisation"
    (Abar = exp(Delta A), ZOH Bbar), "S4" (expanded outputs y[0] = CBx[0],
    y[1] = CAbarBx[0] + CBx[1], ..., i.e. the kernel K = [CB, CAbarB, ...]),
    "Hardware-aware parallel scan" (associative combine), "Mamba
    architecture" (silu gate);
  * "Mamba paper translation" (gitcode.csdn.net): section 2 (recurrent and
    convolution modes, LTI), section 3.5 (Theorem 1, gating; Delta -> inf
    resets, Delta -> 0 ignores);
  * "Mamba close reading" (alishangtian.com), section on the core innovation
    (Theorem 1 stated: N=1, A=-1 gives h_t = (1-g_t) h_{t-1} + g_t x_t).
"""
from __future__ import annotations

import math
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = (s.strip() for s in line.split("=", 1))
            vals[k] = np.array([float(x) for x in v.split()], dtype=np.float64)
    return vals


def _sigmoid(v):
    return 1.0 / (1.0 + np.exp(-v))


def _softplus(s):
    return np.logaddexp(0.0, s)


def _close(a, b, rtol=1e-12, atol=1e-13, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    err = np.max(np.abs(a - b) - rtol * np.abs(b)) if a.size else -1.0
    assert err <= atol, f"{what}: max excess error {err:.3e}"


def _rand_inputs(rng, Bsz, D, L, N, gate=True, dskip=True, h0=False):
    return dict(
        u=rng.standard_normal((Bsz, D, L)),
        delta=rng.standard_normal((Bsz, D, L)),
        z=rng.standard_normal((Bsz, D, L)) if gate else None,
        Bm=rng.standard_normal((Bsz, N, L)),
        Cm=rng.standard_normal((Bsz, N, L)),
        A=-rng.uniform(0.2, 3.0, (D, N)),
        Dskip=rng.standard_normal(D) if dskip else None,
        delta_bias=rng.uniform(-4.0, -1.0, D),
        h0=rng.standard_normal((Bsz, D, N)) if h0 else None,
    )


# --------------------------------------------------------------------------
# hand-worked examples (tests/golden)
# --------------------------------------------------------------------------

def pin_golden_recurrence(lib):
    g = _read_golden("hand_recurrence_n2_l4.txt")
    A = (g["A_over_ln2"] * math.log(2.0)).reshape(1, 2)
    Bm = np.stack([g["B0"], g["B1"]])[None]
    Cm = np.stack([g["C0"], g["C1"]])[None]
    for order in (oracle.ORDER_SEQUENTIAL, oracle.ORDER_TREE):
        y, hl = oracle.selective_scan(g["u"][None, None], g["delta"][None, None], A, Bm, Cm,
                                      Dskip=g["Dskip"], delta_softplus=False, order=order,
                                      return_last_state=True, lib=lib)
        _close(y[0, 0], g["y"], what="golden recurrence y")
        _close(hl[0, 0], g["h_last"], what="golden recurrence h_last")


def pin_golden_gated(lib):
    g = _read_golden("hand_gated_l1.txt")
    z = np.full((1, 1, 1), math.log(3.0))
    y, hl = oracle.selective_scan(g["u"].reshape(1, 1, 1), g["delta"].reshape(1, 1, 1),
                                  g["A"].reshape(1, 3), g["B"].reshape(1, 3, 1),
                                  g["C"].reshape(1, 3, 1), Dskip=g["Dskip"], z=z,
                                  delta_bias=g["bias"], delta_softplus=True,
                                  return_last_state=True, lib=lib)
    _close(y.ravel(), g["y"], what="golden gated y")
    _close(hl.ravel(), g["h_last_over_ln2"] * math.log(2.0), what="golden gated h_last")


# --------------------------------------------------------------------------
# closed forms and other formulas
# --------------------------------------------------------------------------

def pin_lti_equals_convolution(lib, disc=oracle.DISC_EULER):
    """Time-invariant case: the recurrence equals y = K * x with
    K_k = sum_n C[n] Abar[n]^k Bbar[n] (powers, not a recurrence), plus D x, gated."""
    rng = np.random.default_rng(11)
    Bsz, D, L, N = 2, 3, 40, 4
    delta_c = rng.standard_normal((Bsz, D, 1))
    Bc = rng.standard_normal((Bsz, N, 1))
    Cc = rng.standard_normal((Bsz, N, 1))
    A = -rng.uniform(0.1, 2.0, (D, N))
    bias = rng.uniform(-3.0, 0.0, D)
    Dskip = rng.standard_normal(D)
    u = rng.standard_normal((Bsz, D, L))
    z = rng.standard_normal((Bsz, D, L))
    y = oracle.selective_scan(u, np.repeat(delta_c, L, 2), A, np.repeat(Bc, L, 2),
                              np.repeat(Cc, L, 2), Dskip=Dskip, z=z, delta_bias=bias,
                              disc=disc, lib=lib)
    ks = np.arange(L)
    for b in range(Bsz):
        for d in range(D):
            dt = _softplus(delta_c[b, d, 0] + bias[d])
            abar = np.exp(dt * A[d])                               # (N,)
            if disc == oracle.DISC_ZOH:
                bbar = np.expm1(dt * A[d]) / A[d] * Bc[b, :, 0]
            else:
                bbar = dt * Bc[b, :, 0]
            K = (Cc[b, :, 0][None, :] * np.power(abar[None, :], ks[:, None]) * bbar[None, :]).sum(1)
            conv = np.array([np.dot(K[:t + 1][::-1], u[b, d, :t + 1]) for t in range(L)])
            ref = (conv + Dskip[d] * u[b, d]) * z[b, d] * _sigmoid(z[b, d])
            _close(y[b, d], ref, rtol=1e-11, atol=1e-12, what=f"LTI conv b{b} d{d}")


def pin_theorem1_gated_rnn(lib):
    """N=1, A=-1, B=1, C=1 under ZOH: h_t = (1-g_t) h_{t-1} + g_t x_t, g_t = sigmoid(s_t);
    under Euler the same holds when B_t = g_t / Delta_t."""
    rng = np.random.default_rng(5)
    L = 64
    s = rng.standard_normal(L) * 2.5
    x = rng.standard_normal(L)
    g = _sigmoid(s)
    h = np.empty(L)
    prev = 0.0
    for t in range(L):
        prev = (1.0 - g[t]) * prev + g[t] * x[t]
        h[t] = prev
    A = np.array([[-1.0]])
    ones = np.ones((1, 1, L))
    y_zoh = oracle.selective_scan(x[None, None], s[None, None], A, ones, ones,
                                  disc=oracle.DISC_ZOH, lib=lib)
    _close(y_zoh[0, 0], h, rtol=1e-12, atol=1e-13, what="theorem 1 (ZOH)")
    dt = _softplus(s)
    y_eul = oracle.selective_scan(x[None, None], s[None, None], A, (g / dt)[None, None], ones,
                                  disc=oracle.DISC_EULER, lib=lib)
    _close(y_eul[0, 0], h, rtol=1e-12, atol=1e-13, what="theorem 1 (Euler, B = g/Delta)")


def pin_unrolled_sum(lib):
    """Brute force on tiny inputs: h_t = (prod_{r<=t} a_r) h0 + sum_{s<=t} (prod_{s<r<=t} a_r) b_s."""
    rng = np.random.default_rng(3)
    Bsz, D, L, N = 2, 2, 9, 3
    for disc in (oracle.DISC_EULER, oracle.DISC_ZOH):
        p = _rand_inputs(rng, Bsz, D, L, N, h0=True)
        y, hl = oracle.selective_scan(**p, disc=disc, return_last_state=True, lib=lib)
        for b in range(Bsz):
            for d in range(D):
                dt = _softplus(p["delta"][b, d] + p["delta_bias"][d])          # (L,)
                a = np.exp(dt[:, None] * p["A"][d][None, :])                   # (L, N)
                if disc == oracle.DISC_ZOH:
                    bb = np.expm1(dt[:, None] * p["A"][d][None, :]) / p["A"][d][None, :] \
                        * p["Bm"][b].T * p["u"][b, d][:, None]
                else:
                    bb = dt[:, None] * p["Bm"][b].T * p["u"][b, d][:, None]
                hs = np.zeros((L, N))
                for t in range(L):
                    acc = np.prod(a[:t + 1], axis=0) * p["h0"][b, d]
                    for s_ in range(t + 1):
                        acc = acc + np.prod(a[s_ + 1:t + 1], axis=0) * bb[s_]
                    hs[t] = acc
                ref = (p["Cm"][b].T * hs).sum(1) + p["Dskip"][d] * p["u"][b, d]
                ref = ref * p["z"][b, d] * _sigmoid(p["z"][b, d])
                _close(y[b, d], ref, rtol=1e-11, atol=1e-12, what="unrolled sum y")
                _close(hl[b, d], hs[-1], rtol=1e-11, atol=1e-12, what="unrolled sum h_last")


def pin_single_step_closed_form(lib):
    """L = 1, h0 = 0: y = (Delta u sum_n C_n B_n + D u) * silu(z)."""
    rng = np.random.default_rng(8)
    p = _rand_inputs(rng, 3, 4, 1, 5)
    y = oracle.selective_scan(**p, lib=lib)
    dt = _softplus(p["delta"][..., 0] + p["delta_bias"][None, :])
    cb = (p["Cm"][..., 0] * p["Bm"][..., 0]).sum(1)                            # (B,)
    u0, z0 = p["u"][..., 0], p["z"][..., 0]
    ref = (dt * u0 * cb[:, None] + p["Dskip"][None, :] * u0) * z0 * _sigmoid(z0)
    _close(y[..., 0], ref, what="single step")


# --------------------------------------------------------------------------
# invariants and limits
# --------------------------------------------------------------------------

def pin_tree_order_matches_sequential(lib):
    rng = np.random.default_rng(17)
    for L in (1, 2, 3, 17, 64):
        p = _rand_inputs(rng, 2, 3, L, 4, h0=True)
        y1, h1 = oracle.selective_scan(**p, order=oracle.ORDER_SEQUENTIAL, return_last_state=True,
                                       lib=lib)
        y2, h2 = oracle.selective_scan(**p, order=oracle.ORDER_TREE, return_last_state=True, lib=lib)
        _close(y2, y1, rtol=1e-12, atol=1e-12, what=f"tree vs sequential y L={L}")
        _close(h2, h1, rtol=1e-12, atol=1e-12, what=f"tree vs sequential h L={L}")


def pin_boundary_reset(lib):
    """Delta -> inf at t*: outputs from t* on forget everything before t*."""
    rng = np.random.default_rng(23)
    Bsz, D, L, N, ts = 1, 3, 48, 4, 20
    p = _rand_inputs(rng, Bsz, D, L, N, h0=True)
    p["A"] = -np.tile(np.arange(1.0, N + 1), (D, 1))
    p["delta"][..., ts] = 60.0
    y1 = oracle.selective_scan(**p, lib=lib)
    q = dict(p)
    q["u"] = p["u"].copy()
    q["u"][..., :ts] = rng.standard_normal((Bsz, D, ts))
    q["delta"] = p["delta"].copy()
    q["delta"][..., :ts] = rng.standard_normal((Bsz, D, ts))
    q["h0"] = rng.standard_normal((Bsz, D, N))
    y2 = oracle.selective_scan(**q, lib=lib)
    _close(y2[..., ts:], y1[..., ts:], rtol=1e-12, atol=1e-12, what="reset")
    assert np.max(np.abs(y2[..., :ts] - y1[..., :ts])) > 1e-3, "prefix should differ"


def pin_ignore_window(lib):
    """Delta -> 0 over a window: the state is held and the inputs are ignored."""
    rng = np.random.default_rng(29)
    Bsz, D, L, N, t0, t1 = 2, 3, 40, 4, 10, 30
    p = _rand_inputs(rng, Bsz, D, L, N)
    p["delta"][..., t0:t1] = -60.0
    _, h_start = oracle.selective_scan(**{k: (v[..., :t0] if k in ("u", "delta", "z", "Bm", "Cm")
                                              else v) for k, v in p.items()},
                                       return_last_state=True, lib=lib)
    _, h_end = oracle.selective_scan(**{k: (v[..., :t1] if k in ("u", "delta", "z", "Bm", "Cm")
                                            else v) for k, v in p.items()},
                                     return_last_state=True, lib=lib)
    _close(h_end, h_start, rtol=1e-12, atol=1e-14, what="ignore: state held")
    y = oracle.selective_scan(**p, lib=lib)
    for t in range(t0, t1):
        ref = np.einsum("bn,bdn->bd", p["Cm"][..., t], h_start) + p["Dskip"][None] * p["u"][..., t]
        ref = ref * p["z"][..., t] * _sigmoid(p["z"][..., t])
        _close(y[..., t], ref, rtol=1e-12, atol=1e-13, what="ignore: readout of held state")


def pin_chunk_invariance(lib):
    """scan(L) == scan(L1) -> h_last -> scan(L - L1, h0 = h_last)."""
    rng = np.random.default_rng(31)
    p = _rand_inputs(rng, 2, 3, 50, 4, h0=True)
    y, hl = oracle.selective_scan(**p, return_last_state=True, lib=lib)
    for L1 in (1, 23, 49):
        head = {k: (v[..., :L1] if k in ("u", "delta", "z", "Bm", "Cm") else v) for k, v in p.items()}
        y1, h1 = oracle.selective_scan(**head, return_last_state=True, lib=lib)
        tail = {k: (v[..., L1:] if k in ("u", "delta", "z", "Bm", "Cm") else v) for k, v in p.items()}
        tail["h0"] = h1
        y2, h2 = oracle.selective_scan(**tail, return_last_state=True, lib=lib)
        _close(np.concatenate([y1, y2], -1), y, rtol=1e-13, atol=1e-14, what=f"chunk y L1={L1}")
        _close(h2, hl, rtol=1e-13, atol=1e-14, what=f"chunk h L1={L1}")


def pin_step_matches_scan(lib):
    """T decode steps from h0 equal a T-step scan from h0 (final state and every y)."""
    rng = np.random.default_rng(37)
    p = _rand_inputs(rng, 2, 3, 12, 4, h0=True)
    y, hl = oracle.selective_scan(**p, return_last_state=True, lib=lib)
    st = p["h0"]
    for t in range(12):
        st, yt = oracle.state_update(st, p["u"][..., t], p["delta"][..., t], p["A"],
                                     p["Bm"][..., t], p["Cm"][..., t], Dskip=p["Dskip"],
                                     z=p["z"][..., t], delta_bias=p["delta_bias"], lib=lib)
        _close(yt, y[..., t], rtol=1e-13, atol=1e-14, what=f"step y t={t}")
    _close(st, hl, rtol=1e-13, atol=1e-14, what="step final state")


def pin_linearity(lib):
    """Gate off: y is linear in (u, h0) for fixed delta, B, C."""
    rng = np.random.default_rng(41)
    p = _rand_inputs(rng, 2, 3, 20, 4, gate=False, h0=True)
    u2 = rng.standard_normal(p["u"].shape)
    h2 = rng.standard_normal(p["h0"].shape)
    al, be = 0.7, -1.3
    y1 = oracle.selective_scan(**p, lib=lib)
    q = dict(p, u=u2, h0=h2)
    y2 = oracle.selective_scan(**q, lib=lib)
    r = dict(p, u=al * p["u"] + be * u2, h0=al * p["h0"] + be * h2)
    y3 = oracle.selective_scan(**r, lib=lib)
    _close(y3, al * y1 + be * y2, rtol=1e-11, atol=1e-12, what="linearity")


def pin_zoh_to_euler_small_delta(lib):
    """As Delta -> 0 the exact ZOH input term tends to the Euler one, (expm1(dA)/A)/Delta -> 1."""
    rng = np.random.default_rng(43)
    p = _rand_inputs(rng, 1, 2, 10, 3, h0=True)
    p["delta"] = np.full_like(p["delta"], -30.0)      # Delta ~ e^{-30-|bias|}
    ye = oracle.selective_scan(**p, disc=oracle.DISC_EULER, lib=lib)
    yz = oracle.selective_scan(**p, disc=oracle.DISC_ZOH, lib=lib)
    _close(yz, ye, rtol=1e-10, atol=1e-14, what="zoh -> euler")


# ---------------------------------------------------------------------------
# The backward pass (gradients of the scan, for training with recomputation,
# "Mamba paper translation", gitcode.csdn.net, section 3.3.2).  Pinned to the
# forward oracle (itself pinned above) by central finite differences of the
# scalar objective sum(dy * y) + sum(dh_last * h_last), element by element.
# ---------------------------------------------------------------------------

def _fd_check_bwd(lib, gate, dskip, bias, softplus, h0, dh_last, bc_shared=False, seed=21, disc=None):
    rng = np.random.default_rng(seed)
    disc = oracle.DISC_EULER if disc is None else disc
    Bsz, D, L, N = 2, 3, 7, 4
    p = dict(u=rng.standard_normal((Bsz, D, L)), delta=rng.standard_normal((Bsz, D, L)) * 0.7,
             z=rng.standard_normal((Bsz, D, L)) if gate else None,
             Bm=rng.standard_normal((1 if bc_shared else Bsz, N, L)),
             Cm=rng.standard_normal((1 if bc_shared else Bsz, N, L)),
             A=-rng.uniform(0.3, 2.0, (D, N)), Dskip=rng.standard_normal(D) if dskip else None,
             delta_bias=rng.standard_normal(D) * 0.5 if bias else None,
             h0=rng.standard_normal((Bsz, D, N)) if h0 else None)
    if disc == oracle.DISC_ZOH:
        # one state with A = 0 and one with |A| = 1e-4: the exact-ZOH coefficient's A-derivative
        # takes its small-|Delta A| series there
        p["A"][:, 1] = 0.0
        p["A"][:, 2] = rng.choice([-1e-4, 1e-4], D)
    dy = rng.standard_normal((Bsz, D, L))
    dhl = rng.standard_normal((Bsz, D, N)) if dh_last else None

    def objective(q):
        y, hl = oracle.selective_scan(q["u"], q["delta"], q["A"], q["Bm"], q["Cm"], Dskip=q["Dskip"], z=q["z"],
                                      delta_bias=q["delta_bias"], h0=q["h0"], delta_softplus=softplus,
                                      disc=disc, return_last_state=True, nthreads=1, lib=lib)
        v = float(np.sum(dy * y))
        if dhl is not None:
            v += float(np.sum(dhl * hl))
        return v

    g = oracle.selective_scan_bwd(p["u"], p["delta"], p["A"], p["Bm"], p["Cm"], dy, Dskip=p["Dskip"], z=p["z"],
                                  delta_bias=p["delta_bias"], h0=p["h0"], delta_softplus=softplus, dh_last=dhl,
                                  disc=disc, lib=lib)
    names = {"u": "du", "delta": "ddelta", "z": "dz", "Bm": "dBm", "Cm": "dCm", "A": "dA", "Dskip": "dDskip",
             "delta_bias": "ddelta_bias", "h0": "dh0"}
    for key, gname in names.items():
        if p[key] is None:
            continue
        got = g[gname]
        fd = np.empty_like(p[key])
        for idx in np.ndindex(p[key].shape):
            eps = 1e-6 * max(1.0, abs(p[key][idx]))
            qp = dict(p); qp[key] = p[key].copy(); qp[key][idx] += eps
            qm = dict(p); qm[key] = p[key].copy(); qm[key][idx] -= eps
            fd[idx] = (objective(qp) - objective(qm)) / (2 * eps)
        scale = max(1.0, float(np.max(np.abs(fd))))
        err = float(np.max(np.abs(got - fd)))
        assert err <= 1e-6 * scale, f"{gname}: max |analytic - finite difference| = {err:.3e} (scale {scale:.2e})"
    if p["h0"] is None:
        # the gradient of a zero initial state is still defined: dh0 = a_0 lambda_0
        assert g["dh0"].shape == (Bsz, D, N)


def pin_bwd_finite_differences_full(lib):
    """Gate, D skip, bias, softplus, h0 and dh_last all on."""
    _fd_check_bwd(lib, gate=True, dskip=True, bias=True, softplus=True, h0=True, dh_last=True)


def pin_bwd_finite_differences_bare(lib):
    """No gate, no D skip, no bias, Delta = delta (no softplus), zero h0, dy only."""
    _fd_check_bwd(lib, gate=False, dskip=False, bias=False, softplus=False, h0=False, dh_last=False, seed=22)


def pin_bwd_finite_differences_shared_bc(lib):
    """B, C shared across the batch: their gradients are the sums over the batch."""
    _fd_check_bwd(lib, gate=True, dskip=True, bias=True, softplus=True, h0=False, dh_last=True, bc_shared=True,
                  seed=23)


def pin_bwd_finite_differences_zoh(lib):
    """Exact-ZOH input term, every option on; includes states with A = 0 and |A| = 1e-4."""
    _fd_check_bwd(lib, gate=True, dskip=True, bias=True, softplus=True, h0=True, dh_last=True, seed=24,
                  disc=oracle.DISC_ZOH)


def pin_bwd_finite_differences_zoh_bare(lib):
    """Exact-ZOH input term, every option off."""
    _fd_check_bwd(lib, gate=False, dskip=False, bias=False, softplus=False, h0=False, dh_last=False, seed=25,
                  disc=oracle.DISC_ZOH)


BWD_PINS = [pin_bwd_finite_differences_full, pin_bwd_finite_differences_bare, pin_bwd_finite_differences_shared_bc,
            pin_bwd_finite_differences_zoh, pin_bwd_finite_differences_zoh_bare]


# ---------------------------------------------------------------------------
# The causal depthwise convolution in front of the SSM branch ("Mamba and state
# space models", docs.ifdog.com, section "Mamba architecture", step 3a).
# ---------------------------------------------------------------------------

def pin_conv_golden(lib):
    """Hand-worked outputs of a 4-tap convolution, with and without history."""
    g = _read_golden("hand_conv_w4_l5.txt")
    x = g["x"].reshape(1, 1, -1)
    w = g["w"].reshape(1, -1)
    bias = g["bias"]
    out = oracle.causal_conv1d(x, w, bias, silu=False, lib=lib)
    _close(out.ravel(), g["out"], what="conv without history")
    out = oracle.causal_conv1d(x, w, bias, x_hist=g["hist"].reshape(1, 1, -1), silu=False, lib=lib)
    _close(out.ravel(), g["out_hist"], what="conv with history")


def pin_conv_unit_taps_shift(lib):
    """A kernel with one tap j set to 1 is a causal delay by W-1-j steps (zeros shifted in)."""
    rng = np.random.default_rng(11)
    W, L = 4, 23
    x = rng.standard_normal((2, 3, L))
    for j in range(W):
        w = np.zeros((3, W))
        w[:, j] = 1.0
        out = oracle.causal_conv1d(x, w, silu=False, lib=lib)
        lag = W - 1 - j
        want = np.zeros_like(x)
        want[..., lag:] = x[..., :L - lag]
        assert np.array_equal(out, want), f"tap {j} is not a delay of {lag}"


def pin_conv_matches_numpy_convolve(lib):
    """Against numpy's full linear convolution cut to the first L samples (kernel reversed,
    since the taps are in cross-correlation order), then SiLU v * sigmoid(v) in closed form."""
    rng = np.random.default_rng(12)
    Bsz, D, L, W = 2, 5, 37, 4
    x = rng.standard_normal((Bsz, D, L))
    w = rng.standard_normal((D, W))
    bias = rng.standard_normal(D)
    lin = np.empty_like(x)
    for b in range(Bsz):
        for d in range(D):
            lin[b, d] = np.convolve(x[b, d], w[d, ::-1])[:L] + bias[d]
    _close(oracle.causal_conv1d(x, w, bias, silu=False, lib=lib), lin, what="linear conv")
    _close(oracle.causal_conv1d(x, w, bias, silu=True, lib=lib), lin * _sigmoid(lin), what="conv + silu")


def pin_conv_silu_values(lib):
    """One tap of weight 1: out = silu(x); silu(0) = 0, silu(ln 3) = (3/4) ln 3 and
    silu(-ln 3) = -(1/4) ln 3, since sigmoid(ln 3) = 3/4."""
    ln3 = math.log(3.0)
    x = np.array([0.0, ln3, -ln3]).reshape(1, 1, 3)
    out = oracle.causal_conv1d(x, np.ones((1, 1)), silu=True, lib=lib).ravel()
    _close(out, np.array([0.0, 0.75 * ln3, -0.25 * ln3]), what="silu values")


def pin_conv_history_continuation(lib):
    """Convolving [x1, x2] in one call equals convolving x2 with the last W-1 inputs of x1 as
    its history (a sequence split at any step)."""
    rng = np.random.default_rng(13)
    W = 4
    x = rng.standard_normal((1, 3, 30))
    w = rng.standard_normal((3, W))
    bias = rng.standard_normal(3)
    whole = oracle.causal_conv1d(x, w, bias, lib=lib)
    for cut in (1, 2, 3, 17):
        head = oracle.causal_conv1d(x[..., :cut], w, bias, lib=lib)
        hist = np.zeros((1, 3, W - 1))
        k = min(cut, W - 1)
        hist[..., W - 1 - k:] = x[..., cut - k:cut]
        tail = oracle.causal_conv1d(x[..., cut:], w, bias, x_hist=hist, lib=lib)
        _close(np.concatenate([head, tail], axis=-1), whole, what=f"split at {cut}")


CONV_PINS = [
    pin_conv_golden,
    pin_conv_unit_taps_shift,
    pin_conv_matches_numpy_convolve,
    pin_conv_silu_values,
    pin_conv_history_continuation,
]


# --------------------------------------------------------------------------
# complex diagonal A (S4D-Lin, "Mamba paper translation" section 3.6): complex state,
# real input term, y = Re(C . h) + D u
# --------------------------------------------------------------------------

def _complex_inputs(rng, Bsz, D, L, N):
    x = _rand_inputs(rng, Bsz, D, L, N)
    x["A"] = -rng.uniform(0.2, 1.5, (D, N)) + 1j * rng.uniform(-4.0, 4.0, (D, N))
    x["h0"] = rng.standard_normal((Bsz, D, N)) + 1j * rng.standard_normal((Bsz, D, N))
    return x


def pin_complex_zero_imag_is_real(lib):
    """With Im A = 0 and a real h0 the complex scan is the (pinned) real scan."""
    rng = np.random.default_rng(41)
    x = _rand_inputs(rng, 2, 3, 33, 5, h0=True)
    yr, hr = oracle.selective_scan(x["u"], x["delta"], x["A"], x["Bm"], x["Cm"], Dskip=x["Dskip"], z=x["z"],
                                   delta_bias=x["delta_bias"], h0=x["h0"], return_last_state=True, lib=lib)
    yc, hc = oracle.selective_scan_complex(x["u"], x["delta"], x["A"] + 0j, x["Bm"], x["Cm"], Dskip=x["Dskip"],
                                           z=x["z"], delta_bias=x["delta_bias"], h0=x["h0"] + 0j,
                                           return_last_state=True, lib=lib)
    _close(yc, yr, rtol=1e-12, atol=1e-12, what="complex scan with real A: y")
    _close(hc.real, hr, rtol=1e-12, atol=1e-12, what="complex scan with real A: Re h_last")
    _close(hc.imag, np.zeros_like(hr), atol=0.0, what="complex scan with real A: Im h_last")


def pin_complex_lti_convolution(lib):
    """Time-invariant complex case: y = K * u + D u (gated) with
    K_k = Re(sum_n C[n] Abar[n]^k Delta B[n]), Abar = exp(Delta A) complex, as powers."""
    rng = np.random.default_rng(42)
    Bsz, D, L, N = 2, 3, 40, 4
    delta_c = rng.standard_normal((Bsz, D, 1))
    Bc = rng.standard_normal((Bsz, N, 1))
    Cc = rng.standard_normal((Bsz, N, 1))
    A = oracle.s4d_lin(D, N) * rng.uniform(0.5, 1.5, (D, N))
    bias = rng.uniform(-3.0, 0.0, D)
    Dskip = rng.standard_normal(D)
    u = rng.standard_normal((Bsz, D, L))
    z = rng.standard_normal((Bsz, D, L))
    y = oracle.selective_scan_complex(u, np.repeat(delta_c, L, 2), A, np.repeat(Bc, L, 2), np.repeat(Cc, L, 2),
                                      Dskip=Dskip, z=z, delta_bias=bias, lib=lib)
    ks = np.arange(L)
    for b in range(Bsz):
        for d in range(D):
            dt = _softplus(delta_c[b, d, 0] + bias[d])
            abar = np.exp(dt * A[d])
            K = (Cc[b, :, 0][None, :] * np.power(abar[None, :], ks[:, None]) * (dt * Bc[b, :, 0])[None, :]).sum(1).real
            conv = np.array([np.dot(K[:t + 1][::-1], u[b, d, :t + 1]) for t in range(L)])
            ref = (conv + Dskip[d] * u[b, d]) * z[b, d] * _sigmoid(z[b, d])
            _close(y[b, d], ref, rtol=1e-11, atol=1e-12, what=f"complex LTI conv b{b} d{d}")


def pin_complex_rotation_impulse(lib):
    """Re A = 0: |Abar| = 1, the state only rotates.  An impulse u_0 = 1 from h0 = 0 gives
    h_t[n] = Delta_0 B_0[n] exp(i A_im[n] (Delta_1 + ... + Delta_t)), so
    y_t = sum_n C_t[n] Delta_0 B_0[n] cos(A_im[n] S_t) + D u_t (no gate)."""
    rng = np.random.default_rng(43)
    D, L, N = 2, 25, 3
    A = 1j * rng.uniform(-3.0, 3.0, (D, N))
    u = np.zeros((1, D, L))
    u[0, :, 0] = 1.0
    delta = rng.standard_normal((1, D, L))
    bias = rng.uniform(-2.0, 0.5, D)
    Bm, Cm = rng.standard_normal((1, N, L)), rng.standard_normal((1, N, L))
    Dskip = rng.standard_normal(D)
    y, hl = oracle.selective_scan_complex(u, delta, A, Bm, Cm, Dskip=Dskip, delta_bias=bias,
                                          return_last_state=True, lib=lib)
    for d in range(D):
        dts = _softplus(delta[0, d] + bias[d])
        S = np.concatenate([[0.0], np.cumsum(dts[1:])])            # S_t = Delta_1 + ... + Delta_t
        amp = dts[0] * Bm[0, :, 0]                                   # (N,)
        ref = (Cm[0] * amp[:, None] * np.cos(A[d].imag[:, None] * S[None, :])).sum(0) + Dskip[d] * u[0, d]
        _close(y[0, d], ref, rtol=1e-11, atol=1e-12, what=f"rotation y d{d}")
        h_ref = amp * np.exp(1j * A[d].imag * S[-1])
        _close(hl[0, d].real, h_ref.real, rtol=1e-11, atol=1e-12, what=f"rotation Re h d{d}")
        _close(hl[0, d].imag, h_ref.imag, rtol=1e-11, atol=1e-12, what=f"rotation Im h d{d}")


def pin_complex_unrolled_sum(lib):
    """Brute force with numpy complex arithmetic on tiny inputs: h_t = (prod Abar) h0 +
    sum_s (prod_{r=s+1..t} Abar_r) Delta_s B_s u_s, y_t = (Re(C_t . h_t) + D u_t) silu(z_t)."""
    rng = np.random.default_rng(44)
    Bsz, D, L, N = 1, 2, 7, 3
    x = _complex_inputs(rng, Bsz, D, L, N)
    y, hl = oracle.selective_scan_complex(x["u"], x["delta"], x["A"], x["Bm"], x["Cm"], Dskip=x["Dskip"],
                                          z=x["z"], delta_bias=x["delta_bias"], h0=x["h0"],
                                          return_last_state=True, lib=lib)
    for d in range(D):
        dts = _softplus(x["delta"][0, d] + x["delta_bias"][d])
        ab = np.exp(dts[:, None] * x["A"][d][None, :])                 # (L, N)
        for t in range(L):
            h = np.prod(ab[:t + 1], axis=0) * x["h0"][0, d]
            for s_ in range(t + 1):
                h = h + np.prod(ab[s_ + 1:t + 1], axis=0) * dts[s_] * x["Bm"][0, :, s_] * x["u"][0, d, s_]
            v = np.sum(x["Cm"][0, :, t] * h).real + x["Dskip"][d] * x["u"][0, d, t]
            v *= x["z"][0, d, t] * _sigmoid(x["z"][0, d, t])
            _close(y[0, d, t], v, rtol=1e-11, atol=1e-12, what=f"complex unrolled y d{d} t{t}")
        _close(hl[0, d].real, h.real, rtol=1e-11, atol=1e-12, what=f"complex unrolled Re h d{d}")
        _close(hl[0, d].imag, h.imag, rtol=1e-11, atol=1e-12, what=f"complex unrolled Im h d{d}")


def pin_complex_conjugate_symmetry(lib):
    """Real inputs: replacing A by its conjugate conjugates the state and leaves y unchanged."""
    rng = np.random.default_rng(45)
    x = _complex_inputs(rng, 2, 3, 30, 4)
    y1, h1 = oracle.selective_scan_complex(x["u"], x["delta"], x["A"], x["Bm"], x["Cm"], Dskip=x["Dskip"],
                                           z=x["z"], delta_bias=x["delta_bias"], h0=x["h0"],
                                           return_last_state=True, lib=lib)
    y2, h2 = oracle.selective_scan_complex(x["u"], x["delta"], np.conj(x["A"]), x["Bm"], x["Cm"],
                                           Dskip=x["Dskip"], z=x["z"], delta_bias=x["delta_bias"],
                                           h0=np.conj(x["h0"]), return_last_state=True, lib=lib)
    _close(y2, y1, rtol=1e-12, atol=1e-12, what="conjugate A: y")
    _close(h2.real, h1.real, rtol=1e-12, atol=1e-12, what="conjugate A: Re h")
    _close(h2.imag, -h1.imag, rtol=1e-12, atol=1e-12, what="conjugate A: Im h")


# --------------------------------------------------------------------------
# Mamba-2 SSD (scalar A per head; "Mamba close reading", SSD section; "Mamba and state space
# models", section "Mamba-2 and structured duality"): the map is multiplication by a
# semiseparable matrix, (L o C B^T) acting on Delta x, with L the data-dependent decay mask
# --------------------------------------------------------------------------

def _ssd_inputs(rng, Bsz, H, P, L, N, gate=True, h0=False):
    return dict(
        x=rng.standard_normal((Bsz, H * P, L)),
        delta=rng.standard_normal((Bsz, H, L)),
        z=rng.standard_normal((Bsz, H * P, L)) if gate else None,
        Bm=rng.standard_normal((Bsz, L, N)),
        Cm=rng.standard_normal((Bsz, L, N)),
        a=-rng.uniform(0.2, 2.0, H),
        Dskip=rng.standard_normal(H),
        delta_bias=rng.uniform(-3.0, -0.5, H),
        h0=rng.standard_normal((Bsz, H, P, N)) if h0 else None,
    )


def pin_ssd_dual_form(lib):
    """The quadratic (dual) form computed directly: y_t = sum_{s<=t} exp(a (S_t - S_s)) (C_t . B_s) Delta_s x_s
    + exp(a S_t) C_t . h0 + D x_t, gated, with S_t = Delta_0 + ... + Delta_t."""
    rng = np.random.default_rng(51)
    Bsz, H, P, L, N = 2, 3, 2, 24, 4
    x = _ssd_inputs(rng, Bsz, H, P, L, N, h0=True)
    y, hl = oracle.ssd_scan(x["x"], x["delta"], x["a"], x["Bm"], x["Cm"], Dskip=x["Dskip"], z=x["z"],
                            delta_bias=x["delta_bias"], h0=x["h0"], return_last_state=True, lib=lib)
    for b in range(Bsz):
        G = x["Cm"][b] @ x["Bm"][b].T                                   # (L, L): C_t . B_s
        for hd in range(H):
            dts = _softplus(x["delta"][b, hd] + x["delta_bias"][hd])
            S = np.cumsum(dts)
            mask = np.tril(np.exp(x["a"][hd] * (S[:, None] - S[None, :])))
            M = mask * G                                                 # semiseparable matrix
            for p_ in range(P):
                d = hd * P + p_
                xs = x["x"][b, d]
                ys = M @ (dts * xs) + np.exp(x["a"][hd] * S) * (x["Cm"][b] @ x["h0"][b, hd, p_])
                ref = (ys + x["Dskip"][hd] * xs) * x["z"][b, d] * _sigmoid(x["z"][b, d])
                _close(y[b, d], ref, rtol=1e-11, atol=1e-12, what=f"SSD dual form b{b} h{hd} p{p_}")
            # final state: h_L = exp(a S_L) h0 + sum_s exp(a (S_L - S_s)) Delta_s x_s B_s
            w = np.exp(x["a"][hd] * (S[-1] - S)) * dts                   # (L,)
            href = np.exp(x["a"][hd] * S[-1]) * x["h0"][b, hd] + (x["x"][b, hd * P:(hd + 1) * P] * w) @ x["Bm"][b]
            _close(hl[b, hd], href, rtol=1e-11, atol=1e-12, what=f"SSD dual h_last b{b} h{hd}")


def pin_ssd_equals_s6(lib):
    """SSD is the selective scan with A[d, n] = a[head(d)] for every n, Delta shared by a head's
    channels and B / C shared by the heads (the S6 oracle is pinned on its own)."""
    rng = np.random.default_rng(52)
    Bsz, H, P, L, N = 2, 3, 4, 30, 5
    x = _ssd_inputs(rng, Bsz, H, P, L, N, h0=True)
    y, hl = oracle.ssd_scan(x["x"], x["delta"], x["a"], x["Bm"], x["Cm"], Dskip=x["Dskip"], z=x["z"],
                            delta_bias=x["delta_bias"], h0=x["h0"], return_last_state=True, lib=lib)
    A = np.repeat(x["a"], P)[:, None] * np.ones((1, N))
    ys, hs = oracle.selective_scan(x["x"], np.repeat(x["delta"], P, axis=1), A,
                                   np.transpose(x["Bm"], (0, 2, 1)), np.transpose(x["Cm"], (0, 2, 1)),
                                   Dskip=np.repeat(x["Dskip"], P), z=x["z"],
                                   delta_bias=np.repeat(x["delta_bias"], P),
                                   h0=x["h0"].reshape(Bsz, H * P, N), return_last_state=True)
    _close(y, ys, rtol=1e-12, atol=1e-12, what="SSD vs S6 y")
    _close(hl.reshape(Bsz, H * P, N), hs, rtol=1e-12, atol=1e-12, what="SSD vs S6 h_last")


def pin_ssd_semiseparable_rank(lib):
    """The impulse responses of one channel form the matrix M[t, s] (y_t for x = e_s, no gate, no D,
    Delta_s divided out); every block below the diagonal, M[k:, :k], has rank at most N."""
    rng = np.random.default_rng(53)
    L, N = 20, 3
    delta = rng.standard_normal((1, 1, L))
    Bm, Cm = rng.standard_normal((1, L, N)), rng.standard_normal((1, L, N))
    a, bias = np.array([-0.7]), np.array([-1.0])
    dts = _softplus(delta[0, 0] + bias[0])
    M = np.zeros((L, L))
    for s_ in range(L):
        xin = np.zeros((1, 1, L))
        xin[0, 0, s_] = 1.0
        M[:, s_] = oracle.ssd_scan(xin, delta, a, Bm, Cm, delta_bias=bias, lib=lib)[0, 0] / dts[s_]
    assert np.allclose(np.triu(M, 1), 0.0, atol=0.0), "SSD matrix is not causal"
    for k in range(N + 1, L - N):
        sv = np.linalg.svd(M[k:, :k], compute_uv=False)
        assert sv[N] <= 1e-10 * sv[0], f"block M[{k}:, :{k}] has rank above N: {sv[:N + 2]}"


SSD_PINS = [pin_ssd_dual_form, pin_ssd_equals_s6, pin_ssd_semiseparable_rank]


COMPLEX_PINS = [pin_complex_zero_imag_is_real, pin_complex_lti_convolution, pin_complex_rotation_impulse,
                pin_complex_unrolled_sum, pin_complex_conjugate_symmetry]


ALL_PINS = CONV_PINS + BWD_PINS + COMPLEX_PINS + SSD_PINS + [
    pin_golden_recurrence, pin_golden_gated, pin_lti_equals_convolution, pin_theorem1_gated_rnn,
    pin_unrolled_sum, pin_single_step_closed_form, pin_tree_order_matches_sequential,
    pin_boundary_reset, pin_ignore_window, pin_chunk_invariance, pin_step_matches_scan,
    pin_linearity, pin_zoh_to_euler_small_delta,
]
