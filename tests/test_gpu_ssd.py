"""GPU parity of the Mamba-2 SSD layer (ssm_ssd_fwd) against the oracle's SSD recurrence.

The oracle (oracle_ssd_scan) is pinned by the masked-attention dual form computed directly, by
equality with the selective scan under expanded parameters, and by the rank of its semiseparable
matrix (tests/pins.py).  Here the chunked tensor-core kernel (headdim 64, dstate 128, bf16: several
128-step chunks, a ragged last chunk, with and without h0 / gate) and the CUDA-core recurrence
(other shapes, fp32, strided B / C) are compared with it; the full Mamba-2-2.7B-shaped layer is
checked on sampled heads.
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


def run(inp, io, h0=None, gate=True, flags=0, want_path=None):
    d = {k: to_dev(v, io if k in ("x", "delta", "z", "Bm", "Cm") else None) for k, v in inp.items()}
    h0d = to_dev(h0) if h0 is not None else None
    y = torch.empty_like(d["x"])
    Bsz, H, L = inp["delta"].shape
    hl = torch.empty((Bsz, H, inp["x"].shape[1] // H, inp["Bm"].shape[2]), dtype=torch.float32, device="cuda")
    args = ssm.make_ssd_args(d["x"], d["delta"], d["A"], d["Bm"], d["Cm"], y, d["Dskip"], d["z"] if gate else None,
                             d["delta_bias"], h0d, hl, True, flags)
    if want_path is not None:
        assert ssm.ssm_ssd_plan_path(args) == want_path
    y2, hl2 = ssm.ssm_ssd_fwd(d["x"], d["delta"], d["A"], d["Bm"], d["Cm"], Dskip=d["Dskip"],
                              z=d["z"] if gate else None, delta_bias=d["delta_bias"], h0=h0d,
                              return_last_state=True, flags=flags, y=y, h_last=hl)
    torch.cuda.synchronize()
    assert ssm.ssm_get_device_status() == ssm.SSM_OK
    return y2, hl2


def ref(inp, h0=None, gate=True):
    return oracle.ssd_scan(inp["x"], inp["delta"], inp["A"], inp["Bm"], inp["Cm"], Dskip=inp["Dskip"],
                           z=inp["z"] if gate else None, delta_bias=inp["delta_bias"], h0=h0,
                           return_last_state=True)


@pytest.mark.parametrize("shape", [(1, 2, 64, 128, 128), (2, 3, 64, 384, 128), (2, 2, 64, 200, 128),
                                   (1, 4, 64, 1024, 128)])
@pytest.mark.parametrize("with_h0,gate", [(True, True), (False, False)])
def test_ssd_tensor_core(shape, with_h0, gate):
    B, H, P, L, N = shape
    inp = syn.ssd_inputs(B, H, P, L, N, "bf16", seed=sum(shape))
    h0 = np.random.default_rng(1).standard_normal((B, H, P, N)).astype(np.float32) if with_h0 else None
    y, hl = run(inp, "bf16", h0, gate, want_path="tensor_core")
    yr, hr = ref(inp, h0, gate)
    assert_close("bf16", host(y), yr, f"y {shape}")
    assert_close("bf16", host(hl), hr, f"h_last {shape}")


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(2, 3, 16, 77, 32), (1, 2, 64, 256, 128), (2, 2, 8, 40, 200), (1, 5, 3, 33, 5)])
def test_ssd_generic(io, shape):
    B, H, P, L, N = shape
    inp = syn.ssd_inputs(B, H, P, L, N, io, seed=sum(shape) + 3)
    h0 = np.random.default_rng(2).standard_normal((B, H, P, N)).astype(np.float32)
    y, hl = run(inp, io, h0, True, flags=ssm.SSM_SSD_FORCE_GENERIC, want_path="generic")
    yr, hr = ref(inp, h0)
    assert_close(io, host(y), yr, f"y {shape}")
    assert_close(io, host(hl), hr, f"h_last {shape}")


def test_ssd_paths_agree_and_strided_bc_is_generic():
    B, H, P, L, N = 2, 2, 64, 256, 128
    inp = syn.ssd_inputs(B, H, P, L, N, "bf16", seed=11)
    y_tc, _ = run(inp, "bf16", want_path="tensor_core")
    y_g, _ = run(inp, "bf16", flags=ssm.SSM_SSD_FORCE_GENERIC, want_path="generic")
    yr, _ = ref(inp)
    assert_close("bf16", host(y_tc), yr, "tensor core")
    assert_close("bf16", host(y_g), yr, "generic")
    # B / C given transposed in memory (time contiguous): the generic kernel takes them
    d = {k: to_dev(v, "bf16" if k in ("x", "delta", "z", "Bm", "Cm") else None) for k, v in inp.items()}
    Bt = d["Bm"].transpose(1, 2).contiguous().transpose(1, 2)
    Ct = d["Cm"].transpose(1, 2).contiguous().transpose(1, 2)
    y = torch.empty_like(d["x"])
    a = ssm.make_ssd_args(d["x"], d["delta"], d["A"], Bt, Ct, y, d["Dskip"], d["z"], d["delta_bias"])
    assert ssm.ssm_ssd_plan_path(a) == "generic"
    y2 = ssm.ssm_ssd_fwd(d["x"], d["delta"], d["A"], Bt, Ct, Dskip=d["Dskip"], z=d["z"], delta_bias=d["delta_bias"])
    torch.cuda.synchronize()
    assert_close("bf16", host(y2), yr, "strided B / C")


def test_ssd_full_mamba2_layer_sampled_heads():
    """The Mamba-2-2.7B-shaped layer (4 x 80 heads x 64, L = 2048, N = 128, bf16) on the tensor-core
    kernel; the oracle runs on sampled (batch, head) pairs of the same inputs."""
    B, H, P, L, N = 4, 80, 64, 2048, 128
    inp = syn.ssd_inputs(B, H, P, L, N, "bf16", seed=2024)
    y, hl = run(inp, "bf16", want_path="tensor_core")
    yh, hh = host(y), host(hl)
    for b, h in [(0, 0), (0, 79), (1, 13), (2, 40), (3, 79), (3, 1)]:
        sub = dict(x=inp["x"][b:b + 1, h * P:(h + 1) * P], delta=inp["delta"][b:b + 1, h:h + 1], z=inp["z"][b:b + 1, h * P:(h + 1) * P],
                   Bm=inp["Bm"][b:b + 1], Cm=inp["Cm"][b:b + 1], A=inp["A"][h:h + 1], Dskip=inp["Dskip"][h:h + 1],
                   delta_bias=inp["delta_bias"][h:h + 1])
        yr, hr = ref(sub)
        assert_close("bf16", yh[b, h * P:(h + 1) * P], yr[0], f"y (b{b}, h{h})")
        assert_close("bf16", hh[b, h], hr[0, 0], f"h_last (b{b}, h{h})")
