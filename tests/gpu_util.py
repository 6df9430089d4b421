"""Helpers for the GPU parity tests: seeded inputs on the device, the oracle
on the same values (whole tensors or sampled channels), and the tolerances.

Tolerances (fixed by the target this library is built to):
  fp32 I/O : rel-L2 <= 1e-5 and max-abs <= 1e-4
  bf16 I/O : rel-L2 <= 5e-3 (the state and the arithmetic stay fp32)
rel-L2 = ||got - ref||_2 / ||ref||_2 over every compared element.
"""
from __future__ import annotations

import numpy as np

import oracle
from selective_state_space_126_b300 import synthetic as syn

TOL = {"f32": dict(rel_l2=1e-5, max_abs=1e-4), "bf16": dict(rel_l2=5e-3, max_abs=None)}


def torch_dtype(io):
    import torch
    return torch.float32 if io == "f32" else torch.bfloat16


def to_dev(x, io=None, device="cuda"):
    import torch
    if x is None:
        return None
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    if io is not None:
        t = t.to(torch_dtype(io))
    return t.to(device)


def rel_l2(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref.ravel())
    return float(np.linalg.norm((got - ref).ravel()) / (den if den > 0 else 1.0))


def max_abs(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.max(np.abs(got - ref))) if got.size else 0.0


def assert_close(io, got, ref, what=""):
    r = rel_l2(got, ref)
    m = max_abs(got, ref)
    tol = TOL[io]
    assert r <= tol["rel_l2"], f"{what}: rel-L2 {r:.3e} > {tol['rel_l2']:.0e} (max-abs {m:.3e})"
    if tol["max_abs"] is not None:
        assert m <= tol["max_abs"], f"{what}: max-abs {m:.3e} > {tol['max_abs']:.0e} (rel-L2 {r:.3e})"
    return r, m


def host(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


device_inputs = syn.device_inputs


def oracle_channels(cfg: syn.ScanConfig, chans, seed=0, h0=None, nthreads=0):
    """fp64 oracle on the listed (b, d) channels.  Returns y (k, L) and h_last (k, N)."""
    A, Dskip, bias = syn.layer_params(cfg.dim, cfg.dstate, cfg.dt_min, cfg.dt_max, seed)
    ys, hs = [], []
    by_b = {}
    for i, (b, d) in enumerate(chans):
        by_b.setdefault(b, []).append((i, d))
    res = [None] * len(chans)
    for b, lst in by_b.items():
        ds = [d for _, d in lst]
        u = np.stack([syn.channel_rows(cfg, syn.T_U, b, d, d + 1, seed)[0] for d in ds])[None]
        dl = np.stack([syn.channel_rows(cfg, syn.T_DELTA, b, d, d + 1, seed)[0] for d in ds])[None]
        z = np.stack([syn.channel_rows(cfg, syn.T_Z, b, d, d + 1, seed)[0] for d in ds])[None] if cfg.gate else None
        Bm = syn.bc_rows(cfg, syn.T_B, b, seed)[None]
        Cm = syn.bc_rows(cfg, syn.T_C, b, seed)[None]
        hh = None if h0 is None else np.stack([h0[b, d] for d in ds])[None]
        y, hl = oracle.selective_scan(u, dl, A[ds], Bm, Cm, Dskip=Dskip[ds] if cfg.dskip else None, z=z,
                                      delta_bias=bias[ds], h0=hh, return_last_state=True, nthreads=nthreads)
        for k, (i, _) in enumerate(lst):
            res[i] = (y[0, k], hl[0, k])
    return np.stack([r[0] for r in res]), np.stack([r[1] for r in res])


def sample_channels(cfg: syn.ScanConfig, k=48, seed=1):
    """Channels spread over batches, including tile edges and the last channel."""
    rng = np.random.default_rng(seed)
    picks = {(0, 0), (cfg.batch - 1, cfg.dim - 1), (0, min(cfg.dim - 1, 31)), (0, min(cfg.dim - 1, 32)),
             (cfg.batch - 1, min(cfg.dim - 1, 63)), (cfg.batch - 1, min(cfg.dim - 1, 64))}
    while len(picks) < min(k, cfg.batch * cfg.dim):
        picks.add((int(rng.integers(cfg.batch)), int(rng.integers(cfg.dim))))
    return sorted(picks)
