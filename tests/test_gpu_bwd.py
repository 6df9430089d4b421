"""GPU parity of ssm_scan_bwd (gradients of the scan) against the fp64 oracle's backward pass.

The oracle's backward is pinned to finite differences of the forward oracle (tests/pins.py).  Here
every gradient the library returns -- du, ddelta, dz, dA, dB, dC, dDskip, ddelta_bias, dh0 -- is
compared whole with the oracle's on the same inputs: ragged lengths (not a multiple of the 8-step
checkpoint segment), partial warps of channels, N below 16, every option on and off, B/C shared
across the batch, and the 2.8B-shaped layer at full size.
"""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_126_b300 as ssm
from selective_state_space_126_b300 import synthetic as syn
from gpu_util import host, rel_l2, to_dev

pytestmark = pytest.mark.gpu

# fp32 I/O: the arithmetic is fp32 with the SFU exponential, so the gradients carry a few 1e-7 of
# relative error per step; bf16 I/O: du, ddelta, dz are rounded to bf16 once
TOL = {"f32": 1e-5, "bf16": 5e-3}


@pytest.fixture(scope="module", autouse=True)
def _setup(ssm_lib, cuda_ok):
    yield


def make_inputs(B, D, L, N, io, seed, gate=True, dskip=True, bias=True, h0=False, dhl=False, shared_bc=False):
    rng = np.random.default_rng(seed)
    r = lambda *s: syn.round_io(rng.standard_normal(s, dtype=np.float32), io)
    A, Dv, bv = syn.layer_params(D, N, 1e-3, 1e-1, seed)
    A = A * rng.uniform(0.5, 1.5, A.shape).astype(np.float32)
    nb = 1 if shared_bc else B
    return dict(u=r(B, D, L), delta=r(B, D, L), z=r(B, D, L) if gate else None, Bm=r(nb, N, L), Cm=r(nb, N, L),
                A=A, Dskip=Dv if dskip else None, delta_bias=bv if bias else None,
                h0=rng.standard_normal((B, D, N)).astype(np.float32) if h0 else None,
                dy=r(B, D, L), dh_last=rng.standard_normal((B, D, N)).astype(np.float32) if dhl else None)


def run_and_compare(p, io, softplus=True, what="", zoh=False):
    dev = {k: to_dev(v, io if k in ("u", "delta", "z", "Bm", "Cm", "dy") else None) for k, v in p.items()}
    g = ssm.ssm_scan_bwd(dev["u"], dev["delta"], dev["A"], dev["Bm"], dev["Cm"], dev["dy"], Dskip=dev["Dskip"],
                         z=dev["z"], delta_bias=dev["delta_bias"], h0=dev["h0"], delta_softplus=softplus,
                         dh_last=dev["dh_last"], discretization=ssm.SSM_DISC_ZOH if zoh else ssm.SSM_DISC_EULER)
    torch.cuda.synchronize()
    ref = oracle.selective_scan_bwd(p["u"], p["delta"], p["A"], p["Bm"], p["Cm"], p["dy"], Dskip=p["Dskip"],
                                    z=p["z"], delta_bias=p["delta_bias"], h0=p["h0"], delta_softplus=softplus,
                                    dh_last=p["dh_last"], disc=oracle.DISC_ZOH if zoh else oracle.DISC_EULER)
    for k, v in g.items():
        r = ref[{"dB": "dBm", "dC": "dCm"}.get(k, k)]   # the oracle names them after its Bm, Cm
        got = host(v).reshape(r.shape)
        err = rel_l2(got, r)
        assert err <= TOL[io], f"{what} {k}: rel-L2 {err:.3e} > {TOL[io]:.0e}"
        if io == "f32":
            scale = max(1.0, float(np.max(np.abs(r)))) if r.size else 1.0
            m = float(np.max(np.abs(got - r))) if r.size else 0.0
            assert m <= 1e-4 * scale, f"{what} {k}: max-abs {m:.3e} > {1e-4 * scale:.2e}"
    return g, ref


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(1, 1, 1, 1), (2, 5, 7, 4), (2, 33, 40, 16), (1, 64, 256, 16), (3, 40, 100, 13)])
def test_bwd_shapes(io, shape):
    B, D, L, N = shape
    p = make_inputs(B, D, L, N, io, seed=sum(shape), h0=True, dhl=True)
    run_and_compare(p, io, what=str(shape))


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("opts", [dict(gate=False), dict(dskip=False), dict(bias=False), dict(h0=True),
                                  dict(dhl=True), dict(gate=False, dskip=False, bias=False)])
def test_bwd_options(io, opts):
    p = make_inputs(2, 48, 67, 16, io, seed=len(opts) * 7 + 1, **opts)
    run_and_compare(p, io, what=str(opts))


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_bwd_no_softplus(io):
    p = make_inputs(2, 32, 40, 16, io, seed=5)
    p["delta"] = np.abs(p["delta"]) * 0.1   # Delta = delta + bias must stay positive-ish for a stable scan
    p["delta_bias"] = np.full_like(p["delta_bias"], 0.01)
    run_and_compare(p, io, softplus=False, what="no softplus")


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_bwd_shared_bc(io):
    """B, C shared across the batch (batch stride 0): dB, dC are the sums over the batch."""
    p = make_inputs(3, 40, 50, 16, io, seed=9, shared_bc=True, dhl=True)
    g, _ = run_and_compare(p, io, what="shared B/C")
    assert tuple(g["dB"].shape) == (1, 16, 50)


def test_bwd_dh0_is_the_carried_adjoint():
    """Gradient of the initial state through one step: with L = 1 and y = C h_0, dL/dh_{-1} = Abar_0 * dL/dh_0."""
    p = make_inputs(1, 32, 1, 16, "f32", seed=3, gate=False, dskip=False, h0=True)
    g, ref = run_and_compare(p, "f32", what="L=1")
    assert np.allclose(host(g["dh0"]), ref["dh0"], rtol=1e-5, atol=1e-6)


def test_bwd_workspace_and_errors():
    p = make_inputs(2, 32, 64, 16, "bf16", seed=1)
    dev = {k: to_dev(v, "bf16" if k in ("u", "delta", "z", "Bm", "Cm", "dy") else None) for k, v in p.items()}
    fwd = ssm.make_scan_args(dev["u"], dev["delta"], dev["A"], dev["Bm"], dev["Cm"], None, dev["Dskip"], dev["z"],
                             dev["delta_bias"])
    grads = {k: torch.empty_like(dev["u"]) for k in ("du", "ddelta", "dz")}
    grads.update(dA=torch.empty(32, 16, device="cuda"), dB=torch.empty(2, 16, 64, device="cuda"),
                 dC=torch.empty(2, 16, 64, device="cuda"), dDskip=torch.empty(32, device="cuda"))
    a = ssm.make_bwd_args(fwd, dev["dy"], grads)
    lib = ssm.load_library()
    import ctypes
    n = ctypes.c_size_t(0)
    assert lib.ssm_scan_bwd_workspace_size(ctypes.byref(a), ctypes.byref(n)) == 0
    assert n.value == 2 * 32 * (64 // ssm.SSM_BWD_SEGMENT) * 16 * 4
    assert lib.ssm_scan_bwd(ctypes.byref(a), None) == ssm.SSM_ERR_WORKSPACE
    a.dz = None   # z is set, so dz is required
    assert lib.ssm_scan_bwd(ctypes.byref(a), None) == ssm.SSM_ERR_INVALID_ARG


def test_bwd_full_2p8b_layer():
    """The 2.8B-shaped layer (4 x 5120 x 2048, N = 16, bf16), every gradient against the oracle."""
    cfg = syn.M2P8
    p = make_inputs(cfg.batch, cfg.dim, cfg.seqlen, cfg.dstate, "bf16", seed=0)
    p["A"], p["Dskip"], p["delta_bias"] = syn.layer_params(cfg.dim, cfg.dstate, cfg.dt_min, cfg.dt_max, 0)
    run_and_compare(p, "bf16", what="2.8B layer")


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_bwd_checkpoint_paths_agree(io, monkeypatch):
    """The checkpoints written by the tiled forward kernel (the default for TMA-eligible layouts) and by
    the backward kernel's own forward sweep are the same states: du, ddelta, dz and dh0 match bit for
    bit; the atomically summed gradients match to fp32 reordering."""
    p = make_inputs(2, 64, 256, 16, io, seed=12, h0=True, dhl=True)
    dev = {k: to_dev(v, io if k in ("u", "delta", "z", "Bm", "Cm", "dy") else None) for k, v in p.items()}

    def run():
        g = ssm.ssm_scan_bwd(dev["u"], dev["delta"], dev["A"], dev["Bm"], dev["Cm"], dev["dy"], Dskip=dev["Dskip"],
                             z=dev["z"], delta_bias=dev["delta_bias"], h0=dev["h0"], dh_last=dev["dh_last"])
        torch.cuda.synchronize()
        return g

    tiled = run()
    monkeypatch.setenv("SSM_BWD_SWEEP", "1")
    sweep = run()
    for k in ("du", "ddelta", "dz", "dh0"):
        assert torch.equal(tiled[k], sweep[k]), k
    for k in ("dA", "dB", "dC", "dDskip", "ddelta_bias"):
        assert rel_l2(host(tiled[k]), host(sweep[k])) <= 1e-6, k


# ---- the exact zero-order-hold input term (g = (exp(Delta A) - 1) / A) ----

@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(1, 1, 1, 1), (2, 5, 7, 4), (2, 33, 40, 16), (3, 40, 100, 13)])
def test_bwd_zoh_shapes(io, shape):
    B, D, L, N = shape
    p = make_inputs(B, D, L, N, io, seed=sum(shape) + 50, h0=True, dhl=True)
    run_and_compare(p, io, what=f"zoh {shape}", zoh=True)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("opts", [dict(gate=False, dskip=False, bias=False), dict(shared_bc=True, dhl=True)])
def test_bwd_zoh_options(io, opts):
    p = make_inputs(2, 48, 67, 16, io, seed=len(opts) * 7 + 51, **opts)
    run_and_compare(p, io, what=f"zoh {opts}", zoh=True)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_bwd_zoh_small_and_zero_A(io):
    """States with A = 0 and |A| down to 1e-4, and small Delta: the coefficient and its A-derivative take
    their series branches (|Delta A| below 1/64 and 1/4) there."""
    p = make_inputs(2, 40, 60, 16, io, seed=57, h0=True, dhl=True)
    p["A"][:, 0] = 0.0
    p["A"][:, 1] = -1e-4
    p["A"][:, 2] = -3e-2
    p["delta"][0] = syn.round_io(np.full_like(p["delta"][0], -6.0), io)   # Delta ~ 2.5e-3 in batch row 0
    run_and_compare(p, io, what="zoh small A", zoh=True)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_bwd_zoh_checkpoint_paths_agree(io, monkeypatch):
    """With the exact-ZOH term too, the tiled forward kernel's checkpoints equal the backward kernel's own
    forward sweep: du, ddelta, dz and dh0 match bit for bit."""
    p = make_inputs(2, 64, 256, 16, io, seed=58, h0=True, dhl=True)
    dev = {k: to_dev(v, io if k in ("u", "delta", "z", "Bm", "Cm", "dy") else None) for k, v in p.items()}

    def run():
        g = ssm.ssm_scan_bwd(dev["u"], dev["delta"], dev["A"], dev["Bm"], dev["Cm"], dev["dy"], Dskip=dev["Dskip"],
                             z=dev["z"], delta_bias=dev["delta_bias"], h0=dev["h0"], dh_last=dev["dh_last"],
                             discretization=ssm.SSM_DISC_ZOH)
        torch.cuda.synchronize()
        return {k: v.clone() for k, v in g.items()}

    tiled = run()
    monkeypatch.setenv("SSM_BWD_SWEEP", "1")
    sweep = run()
    for k in ("du", "ddelta", "dz", "dh0"):
        assert torch.equal(tiled[k], sweep[k]), f"zoh {k} differs between the checkpoint paths"


# ---- state sizes above 16: 4 or 8 lanes per channel, checkpoints from the backward kernel's own sweep ----

@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(2, 20, 50, 32), (2, 17, 24, 24), (1, 9, 33, 64), (2, 8, 40, 48)])
@pytest.mark.parametrize("zoh", [False, True])
def test_bwd_large_dstate(io, shape, zoh):
    B, D, L, N = shape
    p = make_inputs(B, D, L, N, io, seed=sum(shape) + 70 + zoh, h0=True, dhl=True)
    run_and_compare(p, io, what=f"N={N} zoh={zoh} {shape}", zoh=zoh)


def test_bwd_large_dstate_shared_bc_and_options():
    p = make_inputs(3, 24, 41, 40, "bf16", seed=77, gate=False, dskip=False, shared_bc=True, dhl=True)
    run_and_compare(p, "bf16", what="N=40 shared B/C, no gate, no D")
