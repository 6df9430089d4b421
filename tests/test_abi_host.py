"""C-ABI checks that need no GPU: the library loads, exports every symbol that
include/ssm.h declares, its structs match the binding, host-side validation
rejects bad arguments with the documented codes, and path planning picks the
kernels it should.  No call here reaches a kernel: every argument set is
either invalid (rejected before any CUDA call) or goes to host-only entry
points (workspace size, plan)."""
import ctypes
import os
import re

import pytest

import selective_state_space_126_b300 as ssm

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "ssm.h")

# fake, distinct, 1 KiB-aligned device addresses; never dereferenced by these tests
FAKE = {k: 0x10_0000_0000 + i * 0x1_0000_0000 for i, k in enumerate(
    ["u", "delta", "z", "Bm", "Cm", "A", "Dskip", "bias", "h0", "h_last", "y", "state", "ws"])}


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ssm_[a-z0-9_]+)\s*\(", text)))


def scan_args(B=2, D=64, L=256, N=16, io=ssm.SSM_BF16, **over):
    a = ssm.ScanArgs()
    a.batch, a.dim, a.seqlen, a.dstate = B, D, L, N
    a.io_dtype = io
    a.delta_softplus = 1
    a.u, a.delta, a.z, a.Bm, a.Cm = FAKE["u"], FAKE["delta"], FAKE["z"], FAKE["Bm"], FAKE["Cm"]
    a.A, a.Dskip, a.delta_bias, a.y = FAKE["A"], FAKE["Dskip"], FAKE["bias"], FAKE["y"]
    for f in ("stride_u", "stride_delta", "stride_z", "stride_y"):
        getattr(a, f)[:] = [D * L, L, 1]
    a.stride_B[:] = [N * L, L, 1]
    a.stride_C[:] = [N * L, L, 1]
    a.stride_A[:] = [N, 1]
    for k, v in over.items():
        if isinstance(v, list):
            getattr(a, k)[:] = v
        else:
            setattr(a, k, v)
    return a


def call_scan(a):
    lib = ssm.load_library()
    return lib.ssm_scan_fwd(ctypes.byref(a), None)


@pytest.fixture(scope="module")
def lib(ssm_lib):
    return ssm.load_library()


def test_every_header_symbol_is_exported(lib):
    names = header_functions()
    assert names, "no declarations parsed"
    assert sorted(ssm.EXPORTED_SYMBOLS) == names
    for n in names:
        assert hasattr(lib, n), n


def test_struct_sizes_match(lib):
    assert lib.ssm_abi_sizeof(0) == ctypes.sizeof(ssm.ScanArgs)
    assert lib.ssm_abi_sizeof(1) == ctypes.sizeof(ssm.StepArgs)
    assert lib.ssm_abi_sizeof(2) == ctypes.sizeof(ssm.ConvArgs)
    assert lib.ssm_abi_sizeof(7) == 0
    assert ssm.ssm_version() >> 16 == 1


def test_status_strings(lib):
    for code, name in enumerate(["SSM_OK", "SSM_ERR_INVALID_ARG", "SSM_ERR_UNSUPPORTED", "SSM_ERR_CUDA",
                                 "SSM_ERR_TIMEOUT", "SSM_ERR_WORKSPACE"]):
        assert ssm.ssm_status_string(code) == name
    assert ssm.ssm_status_string(99) == "SSM_ERR_UNKNOWN"


@pytest.mark.parametrize("over,code", [
    (dict(dstate=0), ssm.SSM_ERR_UNSUPPORTED),
    (dict(dstate=65), ssm.SSM_ERR_UNSUPPORTED),
    (dict(batch=-1), ssm.SSM_ERR_INVALID_ARG),
    (dict(seqlen=-5), ssm.SSM_ERR_INVALID_ARG),
    (dict(io_dtype=7), ssm.SSM_ERR_INVALID_ARG),
    (dict(u=None), ssm.SSM_ERR_INVALID_ARG),
    (dict(delta=None), ssm.SSM_ERR_INVALID_ARG),
    (dict(Bm=None), ssm.SSM_ERR_INVALID_ARG),
    (dict(Cm=None), ssm.SSM_ERR_INVALID_ARG),
    (dict(A=None), ssm.SSM_ERR_INVALID_ARG),
    (dict(y=None), ssm.SSM_ERR_INVALID_ARG),
    (dict(stride_u=[64 * 256, 256, 2]), ssm.SSM_ERR_UNSUPPORTED),      # time stride must be 1
    (dict(stride_B=[16 * 256, -256, 1]), ssm.SSM_ERR_INVALID_ARG),     # negative stride
    (dict(y=FAKE["u"] + 1024), ssm.SSM_ERR_INVALID_ARG),               # y overlaps u
    (dict(stride_y=[256, 256, 1]), ssm.SSM_ERR_INVALID_ARG),           # y maps two (b,d,t) to one address
    (dict(u=FAKE["u"] + 1), ssm.SSM_ERR_INVALID_ARG),                  # misaligned bf16 pointer
    (dict(h_last=FAKE["Bm"]), ssm.SSM_ERR_INVALID_ARG),                # h_last overlaps B
])
def test_scan_validation(lib, over, code):
    rc = call_scan(scan_args(**over))
    assert rc == code, (rc, ssm.ssm_status_string(rc), lib.ssm_last_error_detail())
    assert lib.ssm_last_error_detail()


def test_null_args(lib):
    assert lib.ssm_scan_fwd(None, None) == ssm.SSM_ERR_INVALID_ARG
    assert lib.ssm_state_update(None, None) == ssm.SSM_ERR_INVALID_ARG
    n = ctypes.c_size_t(5)
    assert lib.ssm_scan_workspace_size(None, ctypes.byref(n)) == ssm.SSM_ERR_INVALID_ARG
    assert lib.ssm_scan_workspace_size(ctypes.byref(scan_args()), None) == ssm.SSM_ERR_INVALID_ARG


def test_empty_problem_is_a_noop(lib):
    # batch 0 or dim 0: nothing to read or write, no CUDA call
    assert call_scan(scan_args(batch=0)) == ssm.SSM_OK
    assert call_scan(scan_args(dim=0, u=None, y=None)) == ssm.SSM_OK


def step_args(B=4, D=32, N=16, **over):
    a = ssm.StepArgs()
    a.batch, a.dim, a.dstate = B, D, N
    a.io_dtype = ssm.SSM_BF16
    a.delta_softplus = 1
    a.state, a.u, a.delta, a.z = FAKE["state"], FAKE["u"], FAKE["delta"], FAKE["z"]
    a.Bm, a.Cm, a.A, a.y = FAKE["Bm"], FAKE["Cm"], FAKE["A"], FAKE["y"]
    a.stride_state[:] = [D * N, N, 1]
    for f in ("stride_u", "stride_delta", "stride_z", "stride_y"):
        getattr(a, f)[:] = [D, 1]
    a.stride_B[:] = [N, 1]
    a.stride_C[:] = [N, 1]
    a.stride_A[:] = [N, 1]
    for k, v in over.items():
        if isinstance(v, list):
            getattr(a, k)[:] = v
        else:
            setattr(a, k, v)
    return a


@pytest.mark.parametrize("over,code", [
    (dict(dstate=0), ssm.SSM_ERR_UNSUPPORTED),
    (dict(state=None), ssm.SSM_ERR_INVALID_ARG),
    (dict(y=FAKE["state"]), ssm.SSM_ERR_INVALID_ARG),          # y overlaps the state
    (dict(stride_state=[16, 16, 1]), ssm.SSM_ERR_INVALID_ARG),  # state rows alias
    (dict(u=FAKE["state"] + 64), ssm.SSM_ERR_INVALID_ARG),      # input inside the state
    (dict(stride_u=[-1, 1]), ssm.SSM_ERR_INVALID_ARG),
])
def test_step_validation(lib, over, code):
    rc = lib.ssm_state_update(ctypes.byref(step_args(**over)), None)
    assert rc == code, (rc, lib.ssm_last_error_detail())


def test_step_empty_is_noop(lib):
    assert lib.ssm_state_update(ctypes.byref(step_args(batch=0)), None) == ssm.SSM_OK


@pytest.mark.parametrize("kw,path", [
    (dict(L=255), "generic"),                       # ragged rows: not 16-byte vectors
    (dict(L=256), "tiled"),
    (dict(L=260, io=ssm.SSM_F32), "tiled"),          # fp32 rows of 4-element vectors
    (dict(L=258, io=ssm.SSM_F32), "generic"),
    (dict(L=256, flags=ssm.SSM_SCAN_FORCE_GENERIC), "generic"),
    (dict(L=4096, flags=ssm.SSM_SCAN_FORCE_CHUNKED, chunk_len=1024), "chunked"),
    (dict(B=1, D=1536, L=1 << 20), "chunked"),       # long sequence, few channels
    (dict(B=4, D=5120, L=2048), "split"),            # 640 CTAs: 592 (4 per SM) + 48 four-warp CTAs
    (dict(B=4, D=5120, L=2048, io=ssm.SSM_F32), "tiled"),   # the split is a bf16 form
    (dict(B=4, D=5120, L=2048, disc=ssm.SSM_DISC_ZOH), "tiled"),   # ZOH keeps one launch (measured faster)
    (dict(B=4, D=5920, L=2048), "split"),            # 740 CTAs: 148 four-warp CTAs, one per SM
    (dict(B=4, D=5952, L=2048), "tiled"),            # 744 CTAs: more than 5 per SM, two waves anyway
    (dict(B=4, D=4736, L=2048), "tiled"),            # 592 CTAs: 4 per SM already
    (dict(B=4, D=5120, L=2048, cplx=True), "tiled"),  # complex A: four-warp CTAs, one launch
    (dict(B=1, D=5120, L=2048), "chunked"),          # 160 CTAs: about one per SM
    (dict(B=4, D=1536, L=2048), "tiled"),            # 192 CTAs: the single pass measured faster
    (dict(B=1, D=5120, L=1024), "tiled"),            # too short to chunk
    (dict(B=4, D=1536, L=8192), "chunked"),          # long and under two CTAs per SM
    (dict(L=255, flags=ssm.SSM_SCAN_FORCE_WARPSCAN), "warpscan"),   # any layout: plain strided loads
    (dict(B=1, D=5120, L=2048, flags=ssm.SSM_SCAN_FORCE_WARPSCAN), "warpscan"),
])
def test_plan(lib, kw, path):
    # the planner's cut-offs are in CTAs per SM; these expected paths hold for 148 SMs (B300, and
    # the value the library assumes when no GPU is present)
    import torch
    if torch.cuda.is_available() and torch.cuda.get_device_properties(0).multi_processor_count != 148:
        pytest.skip("expected paths are for 148 SMs")
    kw = dict(kw)
    flags = kw.pop("flags", 0)
    chunk_len = kw.pop("chunk_len", 0)
    B, D, L = kw.get("B", 2), kw.get("D", 64), kw["L"]
    a = scan_args(B=B, D=D, L=L, io=kw.get("io", ssm.SSM_BF16), flags=flags, chunk_len=chunk_len,
                  discretization=kw.get("disc", ssm.SSM_DISC_EULER))
    if kw.get("cplx"):
        a.A_imag = FAKE["ws"]
    if path == "split":
        import os
        os.environ["SSM_SCAN_KERNEL"] = "k2"        # the single launch on request
        try:
            assert ssm.ssm_scan_plan_path(a) == "tiled"
        finally:
            del os.environ["SSM_SCAN_KERNEL"]
    assert ssm.ssm_scan_plan_path(a) == path
    ws = ssm.ssm_scan_workspace_size(a)
    assert (ws > 0) == (path == "chunked")


@pytest.mark.parametrize("kw,code", [
    (dict(N=17), ssm.SSM_ERR_UNSUPPORTED),                                   # more than 16 states
    (dict(discretization=ssm.SSM_DISC_ZOH), ssm.SSM_ERR_UNSUPPORTED),        # Euler input term only
    (dict(A_imag=FAKE["ws"]), ssm.SSM_ERR_UNSUPPORTED),                      # real A only
    (dict(extra=ssm.SSM_SCAN_FORCE_TILED), ssm.SSM_ERR_INVALID_ARG),         # one forced path at a time
    (dict(extra=ssm.SSM_SCAN_FORCE_CHUNKED), ssm.SSM_ERR_INVALID_ARG),
])
def test_warpscan_limits(lib, kw, code):
    kw = dict(kw)
    extra = kw.pop("extra", 0)
    a = scan_args(flags=ssm.SSM_SCAN_FORCE_WARPSCAN | extra, **kw)
    assert call_scan(a) == code, lib.ssm_last_error_detail()


def test_force_tiled_on_ragged_is_unsupported(lib):
    a = scan_args(L=255, flags=ssm.SSM_SCAN_FORCE_TILED)
    assert call_scan(a) == ssm.SSM_ERR_UNSUPPORTED


def test_chunked_without_workspace_is_rejected(lib):
    a = scan_args(L=4096, flags=ssm.SSM_SCAN_FORCE_CHUNKED, chunk_len=1024)
    assert call_scan(a) == ssm.SSM_ERR_WORKSPACE
    a.workspace = FAKE["ws"]
    a.workspace_bytes = 16
    assert call_scan(a) == ssm.SSM_ERR_WORKSPACE


def test_workspace_size_formula(lib):
    # records: (N padded + 1) floats per (batch, channel, chunk)
    a = scan_args(B=2, D=64, L=4096, flags=ssm.SSM_SCAN_FORCE_CHUNKED, chunk_len=1000)
    ws = ssm.ssm_scan_workspace_size(a)
    chunk = 1024                       # rounded up to the 32-step tile
    nchunks = -(-4096 // chunk)
    assert ws == 2 * 64 * nchunks * (16 + 1) * 4


def conv_args(B=2, D=64, L=256, W=4, io=ssm.SSM_BF16, **over):
    a = ssm.ConvArgs()
    a.batch, a.dim, a.seqlen, a.width = B, D, L, W
    a.io_dtype = io
    a.silu = 1
    a.x, a.weight, a.bias, a.out = FAKE["u"], FAKE["A"], FAKE["bias"], FAKE["y"]
    a.stride_x[:] = [D * L, L, 1]
    a.stride_out[:] = [D * L, L, 1]
    a.stride_weight[:] = [W, 1]
    for k, v in over.items():
        if isinstance(v, list):
            getattr(a, k)[:] = v
        else:
            setattr(a, k, v)
    return a


def call_conv(a):
    return ssm.load_library().ssm_causal_conv1d_fwd(ctypes.byref(a), None)


@pytest.mark.parametrize("over,code", [
    (dict(x=None), ssm.SSM_ERR_INVALID_ARG),
    (dict(weight=None), ssm.SSM_ERR_INVALID_ARG),
    (dict(out=None), ssm.SSM_ERR_INVALID_ARG),
    (dict(width=0), ssm.SSM_ERR_UNSUPPORTED),
    (dict(width=17), ssm.SSM_ERR_UNSUPPORTED),
    (dict(io_dtype=7), ssm.SSM_ERR_INVALID_ARG),
    (dict(seqlen=-1), ssm.SSM_ERR_INVALID_ARG),
    (dict(stride_x=[64 * 256, 256, 2]), ssm.SSM_ERR_UNSUPPORTED),
    (dict(stride_out=[64 * 256, 256, 2]), ssm.SSM_ERR_UNSUPPORTED),
    (dict(stride_out=[0, 256, 1]), ssm.SSM_ERR_INVALID_ARG),          # two batch rows on one output row
    (dict(stride_weight=[-4, 1]), ssm.SSM_ERR_INVALID_ARG),
    (dict(out=FAKE["u"] + 512), ssm.SSM_ERR_INVALID_ARG),              # out overlaps x
    (dict(out=FAKE["A"]), ssm.SSM_ERR_INVALID_ARG),                    # out overlaps the weights
    (dict(x=FAKE["u"] + 1), ssm.SSM_ERR_INVALID_ARG),                  # not element-aligned
])
def test_conv_validation(lib, over, code):
    assert call_conv(conv_args(**over)) == code


@pytest.mark.parametrize("over", [dict(batch=0), dict(dim=0), dict(seqlen=0),
                                  dict(seqlen=0, x=None, weight=None, out=None)])
def test_conv_empty_is_a_no_op(lib, over):
    assert call_conv(conv_args(**over)) == ssm.SSM_OK


def bwd_args(B=2, D=64, L=256, N=16, **over):
    a = ssm.BwdArgs()
    a.fwd = scan_args(B, D, L, N)
    a.fwd.y = None
    a.dy = FAKE["y"]
    a.stride_dy[:] = [D * L, L, 1]
    base = 0x40_0000_0000
    for i, k in enumerate(("du", "ddelta", "dz", "dA", "dB", "dC", "dDskip", "ddelta_bias", "dh0")):
        setattr(a, k, base + i * 0x1_0000_0000)
    for k in ("stride_du", "stride_ddelta", "stride_dz"):
        getattr(a, k)[:] = [D * L, L, 1]
    a.stride_dB[:] = [N * L, L, 1]
    a.stride_dC[:] = [N * L, L, 1]
    a.stride_dh0[:] = [D * N, N, 1]
    for k, v in over.items():
        if isinstance(v, list):
            getattr(a, k)[:] = v
        else:
            setattr(a, k, v)
    return a


def bwd_ws(a):
    n = ctypes.c_size_t(0)
    rc = ssm.load_library().ssm_scan_bwd_workspace_size(ctypes.byref(a), ctypes.byref(n))
    return rc, n.value


def test_bwd_workspace_size(lib):
    rc, n = bwd_ws(bwd_args(B=2, D=64, L=250, N=16))
    assert rc == ssm.SSM_OK and n == 2 * 64 * 32 * 16 * 4   # ceil(250 / 8) = 32 checkpoints per channel


@pytest.mark.parametrize("over,code", [
    (dict(dA=None), ssm.SSM_ERR_INVALID_ARG),
    (dict(du=None), ssm.SSM_ERR_INVALID_ARG),
    (dict(dz=None), ssm.SSM_ERR_INVALID_ARG),          # z is set
    (dict(dDskip=None), ssm.SSM_ERR_INVALID_ARG),      # Dskip is set
    (dict(dy=None), ssm.SSM_ERR_INVALID_ARG),
    (dict(stride_du=[64 * 256, 256, 2]), ssm.SSM_ERR_UNSUPPORTED),
    (dict(stride_dB=[0, 256, 1]), ssm.SSM_ERR_INVALID_ARG),   # two batch rows of dB on one row
    (dict(ddelta=0x40_0000_0000), ssm.SSM_ERR_INVALID_ARG),   # ddelta on du
    (dict(du=FAKE["u"]), ssm.SSM_ERR_INVALID_ARG),            # a gradient on an input
    (dict(dy=FAKE["u"] + 2), ssm.SSM_ERR_INVALID_ARG),        # dy overlaps u (read-only, but y's checks apply)
])
def test_bwd_validation(lib, over, code):
    assert bwd_ws(bwd_args(**over))[0] == code


def test_bwd_state_sizes(lib):
    # dstate up to 64: the checkpoint record is 16, 32 or 64 floats (8 states per lane, 2 / 4 / 8 lanes);
    # beyond 64 the call is refused
    def args(N):
        a = bwd_args(B=2, D=64, L=256, N=N)
        a.stride_dB[:] = [N * 256, 256, 1]
        a.stride_dC[:] = [N * 256, 256, 1]
        a.stride_dh0[:] = [64 * N, N, 1]
        a.fwd.stride_B[:] = [N * 256, 256, 1]
        a.fwd.stride_C[:] = [N * 256, 256, 1]
        a.fwd.stride_A[:] = [N, 1]
        return a
    for N, rec in ((5, 16), (16, 16), (17, 32), (32, 32), (33, 64), (64, 64)):
        rc, n = bwd_ws(args(N))
        assert rc == ssm.SSM_OK and n == 2 * 64 * 32 * rec * 4, (N, rc, n)
    assert bwd_ws(args(65))[0] == ssm.SSM_ERR_UNSUPPORTED


def test_discretization_validation(lib):
    assert call_scan(scan_args(discretization=2)) == ssm.SSM_ERR_INVALID_ARG
    assert call_scan(scan_args(discretization=-1)) == ssm.SSM_ERR_INVALID_ARG
    n = ctypes.c_size_t(0)
    assert lib.ssm_scan_workspace_size(ctypes.byref(scan_args(discretization=ssm.SSM_DISC_ZOH)), ctypes.byref(n)) == 0


def test_bwd_takes_zoh_and_rejects_complex_a(lib):
    # the exact-ZOH input term is differentiated: same workspace (the checkpoints) as Euler
    a = bwd_args()
    a.fwd.discretization = ssm.SSM_DISC_ZOH
    rc, n = bwd_ws(a)
    assert rc == ssm.SSM_OK and n == bwd_ws(bwd_args())[1] > 0
    a.fwd.discretization = 2
    assert bwd_ws(a)[0] == ssm.SSM_ERR_INVALID_ARG
    c = bwd_args()
    c.fwd.A_imag = FAKE["ws"]
    assert bwd_ws(c)[0] == ssm.SSM_ERR_UNSUPPORTED


def test_step_discretization_validation(lib):
    a = ssm.StepArgs()
    a.batch, a.dim, a.dstate, a.io_dtype = 2, 8, 16, ssm.SSM_BF16
    a.discretization = 3
    assert lib.ssm_state_update(ctypes.byref(a), None) == ssm.SSM_ERR_INVALID_ARG


def test_complex_validation(lib):
    # complex A: chunked and ZOH are refused, the plan is single pass or generic, no workspace
    a = scan_args(B=1, D=1536, L=1 << 20, A_imag=FAKE["ws"])
    assert ssm.ssm_scan_plan_path(a) == "tiled"
    assert ssm.ssm_scan_workspace_size(a) == 0
    a = scan_args(L=4096, flags=ssm.SSM_SCAN_FORCE_CHUNKED, chunk_len=1024, A_imag=FAKE["ws"])
    assert call_scan(a) == ssm.SSM_ERR_UNSUPPORTED
    a = scan_args(discretization=ssm.SSM_DISC_ZOH, A_imag=FAKE["ws"])
    assert call_scan(a) == ssm.SSM_ERR_UNSUPPORTED
    a = scan_args(N=24, A_imag=FAKE["ws"])
    assert ssm.ssm_scan_plan_path(a) == "generic"
    a = scan_args(A_imag=FAKE["ws"] + 2)
    assert call_scan(a) == ssm.SSM_ERR_INVALID_ARG
    # a complex h_last is (B, D, N, 2): (re, im) pairs that must not overlap
    B, D, N = 2, 64, 16
    a = scan_args(A_imag=FAKE["ws"], h_last=FAKE["h_last"], stride_h_last=[D * N, N, 1])
    assert call_scan(a) == ssm.SSM_ERR_INVALID_ARG
    # the backward pass and the no-allocation entry point take a real A
    assert lib.ssm_scan_fwd_noalloc(ctypes.byref(scan_args(L=4096, A_imag=FAKE["ws"])), None) == \
        ssm.SSM_ERR_UNSUPPORTED


def ssd_args(B=2, H=3, P=64, L=256, N=128, io=ssm.SSM_BF16, **over):
    a = ssm.SsdArgs()
    a.batch, a.nheads, a.headdim, a.seqlen, a.dstate = B, H, P, L, N
    a.io_dtype = io
    a.delta_softplus = 1
    a.x, a.delta, a.z, a.Bm, a.Cm = FAKE["u"], FAKE["delta"], FAKE["z"], FAKE["Bm"], FAKE["Cm"]
    a.A, a.Dskip, a.delta_bias, a.y = FAKE["A"], FAKE["Dskip"], FAKE["bias"], FAKE["y"]
    D = H * P
    for f in ("stride_x", "stride_z", "stride_y"):
        getattr(a, f)[:] = [D * L, L, 1]
    a.stride_delta[:] = [H * L, L, 1]
    a.stride_B[:] = [L * N, N, 1]
    a.stride_C[:] = [L * N, N, 1]
    for k, v in over.items():
        if isinstance(v, list):
            getattr(a, k)[:] = v
        else:
            setattr(a, k, v)
    return a


@pytest.mark.parametrize("over,code", [
    (dict(x=None), ssm.SSM_ERR_INVALID_ARG),
    (dict(A=None), ssm.SSM_ERR_INVALID_ARG),
    (dict(Bm=None), ssm.SSM_ERR_INVALID_ARG),
    (dict(dstate=0), ssm.SSM_ERR_UNSUPPORTED),
    (dict(dstate=257), ssm.SSM_ERR_UNSUPPORTED),
    (dict(io_dtype=5), ssm.SSM_ERR_INVALID_ARG),
    (dict(seqlen=-1), ssm.SSM_ERR_INVALID_ARG),
    (dict(flags=2), ssm.SSM_ERR_INVALID_ARG),
    (dict(stride_x=[3 * 64 * 256, 256, 2]), ssm.SSM_ERR_UNSUPPORTED),
    (dict(stride_y=[0, 256, 1]), ssm.SSM_ERR_INVALID_ARG),            # two batch rows on one output row
    (dict(y=FAKE["u"] + 1024), ssm.SSM_ERR_INVALID_ARG),               # y overlaps x
    (dict(h_last=FAKE["A"], stride_h_last=[3 * 64 * 128, 64 * 128, 128, 1]), ssm.SSM_ERR_INVALID_ARG),
    (dict(x=FAKE["u"] + 1), ssm.SSM_ERR_INVALID_ARG),                  # misaligned
])
def test_ssd_validation(lib, over, code):
    assert lib.ssm_ssd_fwd(ctypes.byref(ssd_args(**over)), None) == code


def test_ssd_plan(lib):
    assert ssm.ssm_ssd_plan_path(ssd_args()) == "tensor_core"
    assert ssm.ssm_ssd_plan_path(ssd_args(flags=ssm.SSM_SSD_FORCE_GENERIC)) == "generic"
    assert ssm.ssm_ssd_plan_path(ssd_args(P=32)) == "generic"                  # headdim other than 64
    assert ssm.ssm_ssd_plan_path(ssd_args(N=64, stride_B=[256 * 64, 64, 1], stride_C=[256 * 64, 64, 1])) == "generic"
    assert ssm.ssm_ssd_plan_path(ssd_args(io=ssm.SSM_F32)) == "generic"
    assert ssm.ssm_ssd_plan_path(ssd_args(L=252)) == "generic"                 # rows not 16-byte aligned
    assert ssm.ssm_ssd_plan_path(ssd_args(stride_B=[128 * 256, 1, 256])) == "generic"   # state not contiguous
    assert lib.ssm_ssd_fwd(ctypes.byref(ssd_args(B=0)), None) == ssm.SSM_OK
