"""GPU parity of ssm_causal_conv1d_fwd (causal depthwise convolution + SiLU) against the oracle.

Covers both kernels (the 128-bit vector path: time stride 1, rows on 16-byte
boundaries, L a multiple of the vector, W <= 4; the generic path otherwise),
every tap count up to 16, bias and SiLU on and off, the history tensor, runs
that end inside a lane group, strided views, the full-size layer shapes, a
sequence split at arbitrary steps (bit-exact against the whole sequence), and
the convolution's output fed to the scan as u.
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


def conv_inputs(B, D, L, W, io, seed, hist=False):
    rng = np.random.default_rng(seed)
    x = syn.round_io(rng.standard_normal((B, D, L), dtype=np.float32), io)
    w, bias = syn.conv_params(D, W, seed)
    xh = syn.round_io(rng.standard_normal((B, D, W - 1), dtype=np.float32), io) if hist and W > 1 else None
    return x, w, bias, xh


def run_both(x, w, bias, xh, io, silu):
    out = ssm.ssm_causal_conv1d_fwd(to_dev(x, io), to_dev(w), bias=to_dev(bias), x_hist=to_dev(xh, io), silu=silu)
    torch.cuda.synchronize()
    ref = oracle.causal_conv1d(x, w, bias, x_hist=xh, silu=silu)
    return host(out), ref


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("W", [1, 2, 3, 4])
@pytest.mark.parametrize("silu", [True, False])
@pytest.mark.parametrize("shape", [(1, 1, 8), (2, 5, 64), (3, 7, 1032), (2, 3, 4096)])
def test_conv_vector_path(io, W, silu, shape):
    B, D, L = shape
    x, w, bias, _ = conv_inputs(B, D, L, W, io, seed=W + L)
    got, ref = run_both(x, w, bias, None, io, silu)
    assert_close(io, got, ref, f"conv {shape} W={W}")


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("shape,W", [((2, 3, 37), 4), ((1, 4, 5), 3), ((2, 6, 64), 5), ((1, 3, 100), 8),
                                     ((2, 2, 33), 16), ((1, 2, 3), 7)])
def test_conv_generic_path(io, shape, W):
    """Ragged L, or more than 4 taps (including more taps than steps)."""
    B, D, L = shape
    x, w, bias, _ = conv_inputs(B, D, L, W, io, seed=L * W)
    got, ref = run_both(x, w, bias, None, io, True)
    assert_close(io, got, ref, f"conv {shape} W={W}")


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("shape,W", [((2, 5, 64), 4), ((1, 3, 1024), 2), ((2, 4, 37), 4), ((1, 2, 16), 6)])
def test_conv_history(io, shape, W):
    B, D, L = shape
    x, w, bias, xh = conv_inputs(B, D, L, W, io, seed=7 + W, hist=True)
    got, ref = run_both(x, w, bias, xh, io, True)
    assert_close(io, got, ref, f"conv+hist {shape} W={W}")


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_conv_no_bias_and_strided_views(io):
    """No bias; x and out as channel slices of larger tensors (vector path when rows stay
    16-byte aligned, generic path when they do not)."""
    B, D, L, W = 2, 6, 256, 4
    x, w, _, _ = conv_inputs(B, D + 3, L, W, io, seed=5)
    for d0 in (0, 1):
        xd = to_dev(x, io)[:, d0:d0 + D]
        out_full = torch.empty((B, D + 2, L), dtype=xd.dtype, device="cuda")
        out = out_full[:, 1:1 + D]
        ssm.ssm_causal_conv1d_fwd(xd, to_dev(w[d0:d0 + D]), bias=None, out=out)
        torch.cuda.synchronize()
        ref = oracle.causal_conv1d(x[:, d0:d0 + D], w[d0:d0 + D], None)
        assert_close(io, host(out), ref, f"strided view d0={d0}")


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("L,cuts", [(2048, (1, 3, 8, 1000)), (101, (2, 50))])
def test_conv_split_sequence_is_exact(io, L, cuts):
    """conv(x) equals conv of the pieces, each given the last W-1 inputs before it, bit for bit
    (the same taps in the same order reach every output)."""
    B, D, W = 2, 8, 4
    x, w, bias, _ = conv_inputs(B, D, L, W, io, seed=L)
    xd, wd, bd = to_dev(x, io), to_dev(w), to_dev(bias)
    whole = ssm.ssm_causal_conv1d_fwd(xd, wd, bias=bd)
    for cut in cuts:
        head = ssm.ssm_causal_conv1d_fwd(xd[..., :cut].contiguous(), wd, bias=bd)
        hist = torch.zeros((B, D, W - 1), dtype=xd.dtype, device="cuda")
        k = min(cut, W - 1)
        hist[..., W - 1 - k:] = xd[..., cut - k:cut]
        tail = ssm.ssm_causal_conv1d_fwd(xd[..., cut:].contiguous(), wd, bias=bd, x_hist=hist)
        torch.cuda.synchronize()
        assert torch.equal(torch.cat([head, tail], dim=-1), whole), f"split at {cut}"


@pytest.mark.parametrize("shape", [(4, 5120, 2048), (8, 1536, 2048)])
def test_conv_full_layer_shapes(shape):
    """The 2.8B- and 130M-shaped layers (bf16, 4 taps, SiLU), every element against the oracle."""
    B, D, L = shape
    x, w, bias, _ = conv_inputs(B, D, L, 4, "bf16", seed=1)
    got, ref = run_both(x, w, bias, None, "bf16", True)
    assert_close("bf16", got, ref, f"conv {shape}")


def test_conv_long_sequence_sampled_rows():
    """L = 2^20 (the long-sequence workload's length), checked on sampled channels."""
    B, D, L, W = 1, 64, 1 << 20, 4
    x, w, bias, _ = conv_inputs(B, D, L, W, "bf16", seed=3)
    out = host(ssm.ssm_causal_conv1d_fwd(to_dev(x, "bf16"), to_dev(w), bias=to_dev(bias)))
    for d in (0, 17, 63):
        ref = oracle.causal_conv1d(x[:, d:d + 1], w[d:d + 1], bias[d:d + 1])
        assert_close("bf16", out[:, d:d + 1], ref, f"long row {d}")


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_conv_feeds_the_scan(io):
    """x -> conv + SiLU -> scan as u, on the GPU end to end, against the oracle chain."""
    B, D, L, N, W = 2, 64, 512, 16, 4
    cfg = syn.with_shape(syn.TINY, batch=B, dim=D, seqlen=L, dstate=N, io_dtype=io, name="conv_chain")
    p = syn.scan_inputs(cfg, seed=4)
    x, w, bias, _ = conv_inputs(B, D, L, W, io, seed=4)
    u_dev = ssm.ssm_causal_conv1d_fwd(to_dev(x, io), to_dev(w), bias=to_dev(bias))
    y = ssm.ssm_scan_fwd(u_dev, to_dev(p["delta"], io), to_dev(p["A"]), to_dev(p["Bm"], io), to_dev(p["Cm"], io),
                         Dskip=to_dev(p["Dskip"]), z=to_dev(p["z"], io), delta_bias=to_dev(p["delta_bias"]))
    torch.cuda.synchronize()
    # the oracle chain consumes the convolution output as the GPU stored it (rounded to the I/O
    # dtype), so the two scans see the same u
    u_ref = oracle.causal_conv1d(x, w, bias)
    assert_close(io, host(u_dev), u_ref, "conv stage")
    y_ref = oracle.selective_scan(host(u_dev), p["delta"], p["A"], p["Bm"], p["Cm"], Dskip=p["Dskip"], z=p["z"],
                                  delta_bias=p["delta_bias"])
    assert_close(io, host(y), y_ref, "scan of the conv output")
