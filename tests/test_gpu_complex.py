"""GPU parity of the scan with a complex diagonal A (S4D-Lin) against the oracle's complex scan.

The oracle's complex scan (oracle/ssm_oracle.c) is pinned by the real scan at Im A = 0, the LTI
convolution with complex powers, a pure-rotation impulse, a brute-force unrolled sum and conjugate
symmetry (tests/pins.py).  Here the tiled single-pass kernel (both state-group shapes) and the
stride-general kernel take a complex A -- the S4D-Lin initialisation -1/2 + n i of "Mamba paper
translation" section 3.6, scaled per element -- with a complex h0, and y and the complex h_last are
compared with it at the library's tolerances.
"""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_126_b300 as ssm
from selective_state_space_126_b300 import synthetic as syn
from gpu_util import assert_close, host, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup(ssm_lib, cuda_ok):
    yield


def complex_inputs(B, D, L, N, io, seed, gate=True):
    rng = np.random.default_rng(seed)
    r = lambda *s: syn.round_io(rng.standard_normal(s, dtype=np.float32), io)
    _, Dv, bv = syn.layer_params(D, N, 1e-3, 1e-1, seed)
    A = (syn.s4d_lin_A(D, N) * rng.uniform(0.5, 1.5, (D, N))).astype(np.complex64)
    h0 = (rng.standard_normal((B, D, N)) + 1j * rng.standard_normal((B, D, N))).astype(np.complex64)
    return dict(u=r(B, D, L), delta=r(B, D, L), z=r(B, D, L) if gate else None, Bm=r(B, N, L), Cm=r(B, N, L),
                A=A, Dskip=Dv, delta_bias=bv, h0=h0)


def run_scan(p, io, flags=0):
    d = {k: to_dev(v, io if k in ("u", "delta", "z", "Bm", "Cm") else None)
         for k, v in p.items() if k not in ("A", "h0")}
    A = torch.from_numpy(p["A"]).cuda()
    h0 = torch.from_numpy(p["h0"]).cuda()
    y, hl = ssm.ssm_scan_fwd(d["u"], d["delta"], A, d["Bm"], d["Cm"], Dskip=d["Dskip"], z=d.get("z"),
                             delta_bias=d["delta_bias"], h0=h0, return_last_state=True, flags=flags)
    torch.cuda.synchronize()
    return y, hl


def oracle_scan(p):
    return oracle.selective_scan_complex(p["u"], p["delta"], p["A"], p["Bm"], p["Cm"], Dskip=p["Dskip"],
                                         z=p["z"], delta_bias=p["delta_bias"], h0=p["h0"], return_last_state=True)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("shape,flags,path", [
    ((1, 16, 256, 16), 0, "tiled"),                              # one CTA, 4 state groups
    ((4, 320, 512, 16), 0, "tiled"),                             # several CTAs and tiles
    ((2, 37, 96, 8), 0, "tiled"),                                # a partial warp of channels, padded states
    ((2, 37, 100, 13), 0, "generic"),                            # ragged length
    ((2, 40, 64, 24), 0, "generic"),                             # N > 16
    ((2, 64, 256, 16), ssm.SSM_SCAN_FORCE_GENERIC, "generic"),
])
def test_complex_scan(io, shape, flags, path):
    B, D, L, N = shape
    p = complex_inputs(B, D, L, N, io, seed=sum(shape) + 7)
    y, hl = run_scan(p, io, flags=flags)
    yr, hr = oracle_scan(p)
    assert_close(io, host(y), yr, f"y {shape}")
    got = hl.cpu().numpy()
    assert_close(io, np.stack([got.real, got.imag]).astype(np.float64), np.stack([hr.real, hr.imag]),
                 f"h_last {shape}")


def test_complex_path_choice():
    p = complex_inputs(2, 64, 256, 16, "bf16", seed=3)
    d = {k: to_dev(v, "bf16" if k in ("u", "delta", "z", "Bm", "Cm") else None)
         for k, v in p.items() if k not in ("A", "h0")}
    A = torch.from_numpy(p["A"]).cuda()
    y = torch.empty_like(d["u"])
    a = ssm.make_scan_args(d["u"], d["delta"], A.real.contiguous(), d["Bm"], d["Cm"], y, d["Dskip"], d["z"],
                           d["delta_bias"], A_imag=A.imag.contiguous())
    assert ssm.ssm_scan_plan_path(a) == "tiled"
    assert ssm.ssm_scan_workspace_size(a) == 0


def test_complex_full_grid_shapes(monkeypatch):
    """600 units of 32 channels (more than 4 per SM on 148 SMs) with a complex A and h0: the planner's
    four-warp CTAs in one launch, the two-warp CTAs, and the two-warp CTAs split over two launches, each
    against the oracle."""
    if torch.cuda.get_device_properties(0).multi_processor_count != 148:
        pytest.skip("the case is sized for 148 SMs")
    p = complex_inputs(4, 4790, 128, 16, "bf16", seed=11)
    d = {k: to_dev(v, "bf16" if k in ("u", "delta", "z", "Bm", "Cm") else None)
         for k, v in p.items() if k not in ("A", "h0")}
    A = torch.from_numpy(p["A"]).cuda()
    y = torch.empty_like(d["u"])
    a = ssm.make_scan_args(d["u"], d["delta"], A.real.contiguous(), d["Bm"], d["Cm"], y, d["Dskip"], d["z"],
                           d["delta_bias"], A_imag=A.imag.contiguous())
    yr, hr = oracle_scan(p)
    for env, path in ((None, "tiled"), ("k2", "tiled")):
        if env:
            monkeypatch.setenv("SSM_SCAN_KERNEL", env)
        assert ssm.ssm_scan_plan_path(a) == path
        y, hl = run_scan(p, "bf16")
        assert_close("bf16", host(y), yr, f"y {env}")
        got = hl.cpu().numpy()
        assert_close("bf16", np.stack([got.real, got.imag]).astype(np.float64), np.stack([hr.real, hr.imag]),
                     f"h_last {env}")


def test_complex_without_gate_and_state():
    p = complex_inputs(2, 64, 256, 16, "f32", seed=5, gate=False)
    d = {k: to_dev(v) for k, v in p.items() if k not in ("A", "h0") and v is not None}
    A = torch.from_numpy(p["A"]).cuda()
    y = ssm.ssm_scan_fwd(d["u"], d["delta"], A, d["Bm"], d["Cm"], Dskip=d["Dskip"], delta_bias=d["delta_bias"])
    torch.cuda.synchronize()
    yr = oracle.selective_scan_complex(p["u"], p["delta"], p["A"], p["Bm"], p["Cm"], Dskip=p["Dskip"],
                                       delta_bias=p["delta_bias"])
    assert_close("f32", host(y), yr, "y, no gate, zero h0")
