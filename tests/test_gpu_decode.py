"""GPU parity of ssm_state_update (one decode step, fp32 state in place) against the oracle."""
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


def step_inputs(B, D, N, io, seed, gate=True, dskip=True):
    rng = np.random.default_rng(seed)
    r = lambda *s: syn.round_io(rng.standard_normal(s, dtype=np.float32), io)
    A, Dv, bv = syn.layer_params(D, N, 1e-3, 1e-1, seed)
    return dict(state=rng.standard_normal((B, D, N)).astype(np.float32), u=r(B, D), delta=r(B, D),
                z=r(B, D) if gate else None, Bm=r(B, N), Cm=r(B, N), A=A, Dskip=Dv if dskip else None,
                delta_bias=bv)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(1, 1, 1), (3, 17, 5), (4, 64, 16), (2, 33, 13), (2, 8, 64), (5, 300, 32),
                                   (3, 256, 16), (7, 384, 16)])
def test_step_shapes(io, shape):
    B, D, N = shape
    p = step_inputs(B, D, N, io, seed=sum(shape))
    st = to_dev(p["state"])
    y = ssm.ssm_state_update(st, to_dev(p["u"], io), to_dev(p["delta"], io), to_dev(p["A"]),
                             to_dev(p["Bm"], io), to_dev(p["Cm"], io), Dskip=to_dev(p["Dskip"]),
                             z=to_dev(p["z"], io), delta_bias=to_dev(p["delta_bias"]))
    torch.cuda.synchronize()
    sr, yr = oracle.state_update(p["state"], p["u"], p["delta"], p["A"], p["Bm"], p["Cm"], Dskip=p["Dskip"],
                                 z=p["z"], delta_bias=p["delta_bias"])
    assert_close(io, host(y), yr, f"y {shape}")
    assert_close(io, host(st), sr, f"state {shape}")


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("kernel", ["wide", "quad", "per_item"])
def test_step_every_kernel(io, kernel, monkeypatch):
    """The three decode kernels (one thread per channel and 128 channels per CTA; four lanes per
    channel with bulk-copied rows; per-item global loads) on the same dense N = 16 inputs."""
    if kernel == "quad":
        monkeypatch.setenv("SSM_DECODE_QUAD", "1")
    if kernel == "per_item":
        monkeypatch.setenv("SSM_DECODE_PER_ITEM", "1")
    B, D, N = 37, 256, 16
    p = step_inputs(B, D, N, io, seed=11)
    st = to_dev(p["state"])
    y = ssm.ssm_state_update(st, to_dev(p["u"], io), to_dev(p["delta"], io), to_dev(p["A"]),
                             to_dev(p["Bm"], io), to_dev(p["Cm"], io), Dskip=to_dev(p["Dskip"]),
                             z=to_dev(p["z"], io), delta_bias=to_dev(p["delta_bias"]))
    torch.cuda.synchronize()
    sr, yr = oracle.state_update(p["state"], p["u"], p["delta"], p["A"], p["Bm"], p["Cm"], Dskip=p["Dskip"],
                                 z=p["z"], delta_bias=p["delta_bias"])
    assert_close(io, host(y), yr, f"y {kernel}")
    assert_close(io, host(st), sr, f"state {kernel}")


def test_step_strided_state():
    """State stored with padded rows (non-vector path) and no gate / skip."""
    p = step_inputs(3, 20, 16, "f32", seed=9, gate=False, dskip=False)
    buf = torch.zeros((3, 20, 20), device="cuda")
    buf[..., :16] = to_dev(p["state"])
    st = buf[..., :16]
    y = ssm.ssm_state_update(st, to_dev(p["u"]), to_dev(p["delta"]), to_dev(p["A"]), to_dev(p["Bm"]),
                             to_dev(p["Cm"]), delta_bias=to_dev(p["delta_bias"]))
    torch.cuda.synchronize()
    sr, yr = oracle.state_update(p["state"], p["u"], p["delta"], p["A"], p["Bm"], p["Cm"],
                                 delta_bias=p["delta_bias"])
    assert_close("f32", host(y), yr, "y")
    assert_close("f32", host(st), sr, "state")
    assert torch.count_nonzero(buf[..., 16:]) == 0      # padding untouched


def test_steps_equal_scan():
    """T decode steps reproduce a T-step scan from the same initial state (both on the GPU)."""
    B, D, L, N = 2, 48, 24, 16
    rng = np.random.default_rng(4)
    r = lambda *s: syn.round_io(rng.standard_normal(s, dtype=np.float32), "bf16")
    u, dl, z, Bm, Cm = r(B, D, L), r(B, D, L), r(B, D, L), r(B, N, L), r(B, N, L)
    A, Dv, bv = syn.layer_params(D, N, 1e-3, 1e-1, 4)
    h0 = rng.standard_normal((B, D, N)).astype(np.float32)
    y_scan, h_scan = ssm.ssm_scan_fwd(to_dev(u, "bf16"), to_dev(dl, "bf16"), to_dev(A), to_dev(Bm, "bf16"),
                                      to_dev(Cm, "bf16"), Dskip=to_dev(Dv), z=to_dev(z, "bf16"),
                                      delta_bias=to_dev(bv), h0=to_dev(h0), return_last_state=True)
    st = to_dev(h0)
    ys = []
    for t in range(L):
        ys.append(ssm.ssm_state_update(st, to_dev(u[..., t], "bf16"), to_dev(dl[..., t], "bf16"), to_dev(A),
                                       to_dev(Bm[..., t], "bf16"), to_dev(Cm[..., t], "bf16"), Dskip=to_dev(Dv),
                                       z=to_dev(z[..., t], "bf16"), delta_bias=to_dev(bv)))
    torch.cuda.synchronize()
    assert_close("bf16", np.stack([host(v) for v in ys], -1), host(y_scan), "steps vs scan y")
    assert_close("bf16", host(st), host(h_scan), "steps vs scan state")


def test_decode_workload_1000_steps_sampled():
    """The decode workload: B=256, D=5120, N=16, 1000 consecutive steps on a persistent state.
    Checks the full output of the first steps and sampled channels after all 1000."""
    cfg = syn.DECODE
    A, Dv, bv = syn.decode_params(cfg)
    h0 = syn.decode_state(cfg)
    st = to_dev(h0)
    A_d, D_d, b_d = to_dev(A), to_dev(Dv), to_dev(bv)
    rng = np.random.default_rng(2)
    chans = [(0, 0), (255, 5119)] + [(int(rng.integers(256)), int(rng.integers(5120))) for _ in range(30)]
    ref_state = np.stack([h0[b, d] for b, d in chans])[:, None, :].astype(np.float64)   # (k, 1, N)
    y_last = None
    for step in range(cfg.steps):
        p = syn.decode_step_inputs(cfg, step)
        y = ssm.ssm_state_update(st, to_dev(p["u"], "bf16"), to_dev(p["delta"], "bf16"), A_d,
                                 to_dev(p["Bm"], "bf16"), to_dev(p["Cm"], "bf16"), Dskip=D_d,
                                 z=to_dev(p["z"], "bf16"), delta_bias=b_d)
        if step < 2:   # whole-tensor check of the first steps
            torch.cuda.synchronize()
            s_full, y_full = oracle.state_update(h0 if step == 0 else s_full, p["u"], p["delta"], A, p["Bm"],
                                                 p["Cm"], Dskip=Dv, z=p["z"], delta_bias=bv)
            assert_close("bf16", host(y), y_full, f"step {step} y")
            assert_close("bf16", host(st), s_full, f"step {step} state")
        # sampled channels, one at a time through the oracle
        ys = []
        for i, (b, d) in enumerate(chans):
            ns, yv = oracle.state_update(ref_state[i:i + 1], p["u"][b:b + 1, d:d + 1], p["delta"][b:b + 1, d:d + 1],
                                         A[d:d + 1], p["Bm"][b:b + 1], p["Cm"][b:b + 1], Dskip=Dv[d:d + 1],
                                         z=p["z"][b:b + 1, d:d + 1], delta_bias=bv[d:d + 1])
            ref_state[i:i + 1] = ns
            ys.append(yv[0, 0])
        y_last = (y, np.array(ys))
    torch.cuda.synchronize()
    got_state = np.stack([host(st[b, d]) for b, d in chans])
    assert_close("bf16", got_state, ref_state[:, 0], "state after 1000 steps")
    got_y = np.array([float(y_last[0][b, d].float()) for b, d in chans])
    assert_close("bf16", got_y, y_last[1], "y at step 1000")
