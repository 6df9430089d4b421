"""ssm_scan_fwd_noalloc: the chunked scan for callers that cannot allocate device memory.

Such callers (a plugin inside an engine that owns all device memory, a host
holding only raw input/output pointers, code that must avoid the implicit
synchronisation of cudaMalloc) cannot hand the library a workspace.  This
entry point keeps the chunk records in a scratch array the library reserves
statically on each GPU, so the caller passes only inputs and outputs.

The GPU test calls it through the C ABI twice in a row, on different inputs,
with a caller chunk length and with automatic chunking, and checks each result
against the existing entry point (ssm_scan_fwd on the same chunked path with a
caller workspace): the two run the same kernels on the same plan and must agree
bit for bit.  It runs alone or after the rest
of the suite (this file is collected last).
"""
import ctypes

import numpy as np
import pytest

import selective_state_space_126_b300 as ssm
from selective_state_space_126_b300 import synthetic as syn


def _case(seed, B=2, D=96, L=4096, N=16):
    rng = np.random.default_rng(seed)
    r = lambda *s: syn.round_io(rng.standard_normal(s, dtype=np.float32), "bf16")
    A, Dv, bv = syn.layer_params(D, N, 1e-3, 1e-1, seed)
    return dict(u=r(B, D, L), delta=r(B, D, L), z=r(B, D, L), Bm=r(B, N, L), Cm=r(B, N, L), A=A, Dskip=Dv,
                delta_bias=bv, h0=rng.standard_normal((B, D, N)).astype(np.float32))


def _dev(case):
    import torch
    out = {}
    for k, v in case.items():
        t = torch.from_numpy(v)
        if k in ("u", "delta", "z", "Bm", "Cm"):
            t = t.to(torch.bfloat16)
        out[k] = t.cuda()
    return out


@pytest.mark.gpu
@pytest.mark.parametrize("chunk", [512, 0])     # a caller chunk length, and the automatic chunk sizing
def test_noalloc_matches_workspace_path_twice(ssm_lib, cuda_ok, chunk):
    import torch
    lib = ssm.load_library()
    for call, seed in enumerate((101, 202)):          # two calls in a row, different inputs
        d = _dev(_case(seed))
        # existing entry point: chunked path with a caller-owned workspace
        y_ref, h_ref = ssm.ssm_scan_fwd(d["u"], d["delta"], d["A"], d["Bm"], d["Cm"], Dskip=d["Dskip"], z=d["z"],
                                        delta_bias=d["delta_bias"], h0=d["h0"], return_last_state=True,
                                        flags=ssm.SSM_SCAN_FORCE_CHUNKED, chunk_len=chunk)
        # new entry point through the C ABI: inputs and outputs only
        y = torch.full_like(y_ref, float("nan"))
        h = torch.full_like(h_ref, float("nan"))
        args = ssm.make_scan_args(d["u"], d["delta"], d["A"], d["Bm"], d["Cm"], y, d["Dskip"], d["z"],
                                  d["delta_bias"], d["h0"], h, True, 0, chunk, None)
        rc = lib.ssm_scan_fwd_noalloc(ctypes.byref(args), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert rc == ssm.SSM_OK, lib.ssm_last_error_detail()
        torch.cuda.synchronize()
        # both run the same kernels on the same plan, so the results agree bit for bit
        for got, ref, what in ((y, y_ref, "y"), (h, h_ref, "h_last")):
            assert torch.isfinite(got.float()).all(), f"call {call}: {what} not fully written"
            assert torch.equal(got, ref), \
                f"call {call}: {what} differs, max |diff| {(got.float() - ref.float()).abs().max().item():.3e}"
    assert ssm.ssm_get_device_status() == ssm.SSM_OK


def test_noalloc_long_workload_fits_the_scratch(ssm_lib):
    """Host-side: the 1 x 1536-channel, 2^20-step bf16 scan with automatic chunking needs no more
    chunk records than the static scratch holds (the plan depends on the SM count: 148 on B300,
    also the library's value when no GPU is present)."""
    import torch
    if torch.cuda.is_available() and torch.cuda.get_device_properties(0).multi_processor_count != 148:
        pytest.skip("the chunk plan is sized for 148 SMs")
    lib = ssm.load_library()
    a = ssm.ScanArgs()
    B, D, L, N = 1, 1536, 1 << 20, 16
    a.batch, a.dim, a.seqlen, a.dstate = B, D, L, N
    a.io_dtype, a.delta_softplus = ssm.SSM_BF16, 1
    base = 0x20_0000_0000
    for i, f in enumerate(("u", "delta", "z", "Bm", "Cm", "A", "y")):
        setattr(a, f, base + i * 0x10_0000_0000)
    for f in ("stride_u", "stride_delta", "stride_z", "stride_y"):
        getattr(a, f)[:] = [D * L, L, 1]
    a.stride_B[:] = [N * L, L, 1]
    a.stride_C[:] = [N * L, L, 1]
    a.stride_A[:] = [N, 1]
    a.flags, a.chunk_len = ssm.SSM_SCAN_FORCE_CHUNKED, 0
    need = ssm.ssm_scan_workspace_size(a)
    assert 0 < need <= ssm.SSM_NOALLOC_SCRATCH_BYTES, need
    # a tuning flag other than the chunked one is refused before anything else
    a.flags = ssm.SSM_SCAN_FORCE_TILED
    assert lib.ssm_scan_fwd_noalloc(ctypes.byref(a), None) == ssm.SSM_ERR_INVALID_ARG


def test_noalloc_rejects_problems_beyond_the_scratch(ssm_lib):
    """Host-side: a problem whose records exceed the static scratch is refused before any CUDA call."""
    lib = ssm.load_library()
    a = ssm.ScanArgs()
    B, D, L, N = 8, 5120, 1 << 16, 16
    a.batch, a.dim, a.seqlen, a.dstate = B, D, L, N
    a.io_dtype, a.delta_softplus = ssm.SSM_BF16, 1
    base = 0x20_0000_0000
    for i, f in enumerate(("u", "delta", "Bm", "Cm", "A", "y")):
        setattr(a, f, base + i * 0x10_0000_0000)
    for f in ("stride_u", "stride_delta", "stride_y"):
        getattr(a, f)[:] = [D * L, L, 1]
    a.stride_B[:] = [N * L, L, 1]
    a.stride_C[:] = [N * L, L, 1]
    a.stride_A[:] = [N, 1]
    a.chunk_len = 1024
    rc = lib.ssm_scan_fwd_noalloc(ctypes.byref(a), None)
    assert rc == ssm.SSM_ERR_WORKSPACE
    assert b"static scratch" in lib.ssm_last_error_detail()
    # too short for the chunked path at all
    a.seqlen = 16
    for f in ("stride_u", "stride_delta", "stride_y"):
        getattr(a, f)[:] = [D * 16, 16, 1]
    a.stride_B[:] = [N * 16, 16, 1]
    a.stride_C[:] = [N * 16, 16, 1]
    assert lib.ssm_scan_fwd_noalloc(ctypes.byref(a), None) == ssm.SSM_ERR_UNSUPPORTED
