#!/usr/bin/env python3
"""Benchmark of the selective-scan hot path on B300.

Default workload: the Mamba-2.8B-shaped layer scan, bf16 I/O with fp32 state,
batch 4, D = 5120, L = 2048, N = 16 (671,088,640 state updates per step).  A
step is one full ``ssm_scan_fwd`` over that batch: softplus discretisation,
exp(Delta A), the recurrence, the C contraction, the D skip and the silu gate,
in one kernel launch.

Metric: state-updates/s = B*D*L*N / time, and the achieved HBM GB/s of the
scan kernel against the measured B300 copy bandwidth.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--small] [--no-e2e] [--no-cpu-baseline]

Under torchrun (N > 1) every rank runs an independent replica of the
workload on its own GPU (channels are independent: no data-path collective);
the step time is the max over ranks and the value counts all ranks' updates.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "selective-scan state-updates/s (B·D·L·N/s); achieved HBM GB/s vs B300 peak"
UNIT = "state-updates/s"
SCAN_SOURCES = ["selective_state_space_126_b300/csrc/scan_tiled.cu",
                "selective_state_space_126_b300/csrc/scan_common.cuh",
                "selective_state_space_126_b300/csrc/async_copy.cuh",
                "selective_state_space_126_b300/csrc/device_math.cuh"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "scan_tiled_traffic.txt")   # JSON text written from an ncu capture


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="mamba2.8b_bf16_b4_d5120_l2048_n16")
    ap.add_argument("--small", action="store_true", help="batch 2 of the workload (profiling captures)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-rows", action="store_true", help="skip the other workloads' timing rows")
    ap.add_argument("--only-rows", action="store_true",
                    help="time only the other workloads' rows (one line of JSON; for profiling their kernels)")
    ap.add_argument("--rows", default="all",
                    help="comma-separated subset of rows: m130, ti, long, decode, conv, bwd, bwdzoh, zoh, cplx, ssd")
    ap.add_argument("--decode-steps", type=int, default=1000, help="decode steps of the decode row")
    return ap.parse_args()


def dist_info():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def workload(args):
    from selective_state_space_126_b300 import synthetic as syn
    cfg = syn.SCAN_CONFIGS[args.workload]
    if args.small:
        cfg = syn.with_shape(cfg, batch=2, name=cfg.name + "_batch2")
    return cfg


def algorithmic_bytes(cfg) -> int:
    """Bytes the scan must move once: read u, delta, z; write y (B*D*L each); read B, C
    (B*N*L each, once per batch row); read A (D*N) and D, delta_bias (D) in fp32."""
    es = 4 if cfg.io_dtype == "f32" else 2
    bd_l = cfg.batch * cfg.dim * cfg.seqlen
    seq = (3 if cfg.gate else 2) * bd_l + bd_l
    bc = 2 * (1 if cfg.shared_bc else cfg.batch) * cfg.dstate * cfg.seqlen
    params = cfg.dim * cfg.dstate * 4 + 2 * cfg.dim * 4
    return (seq + bc) * es + params


def bench_config(cfg, world) -> dict:
    """The workload description both arms print (the reference arm runs a bounded sample of it)."""
    algo = algorithmic_bytes(cfg)
    return {"workload": cfg.name, "batch": cfg.batch, "dim": cfg.dim, "seqlen": cfg.seqlen, "dstate": cfg.dstate,
            "io_dtype": cfg.io_dtype, "l2": f"inputs larger than L2 ({algo / 1e6:.0f} MB moved per step vs 126 MB L2)",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "timing": "per-step CUDA events; L2 flushed between steps by a 256 MB read outside the events"}


def source_sha() -> str:
    h = hashlib.sha256()
    for f in SCAN_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest of every rank's x (the job's step time is its slowest rank's); x itself at N = 1."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(updates_per_rank: int, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank's state updates over the job's (slowest rank's) step time."""
    return updates_per_rank * world / (ms_per_step * 1e-3)


def ssm_launches(lib, ssm, args) -> int:
    """Kernel launches one ssm_scan_fwd makes for these arguments."""
    return {"tiled": 1, "split": 2, "chunked": 3, "generic": 1, "warpscan": 1}[ssm.ssm_scan_plan_path(args)]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6400.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.15)

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()

    def summary(self, t0, t1):
        rows = [s for t, s in self.samples if t0 - 0.03 <= t <= t1 + 0.03] or [s for _, s in self.samples]
        window = "timed" if any(t0 - 0.03 <= t <= t1 + 0.03 for t, _ in self.samples) else "around-timed"
        mhz, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            f = [x.strip() for x in r.split(",")]
            if len(f) < 7:
                continue
            try:
                mhz.append(float(f[0]))
                maxes.append(float(f[1]))
            except ValueError:
                continue
            for name, v in zip(names, f[3:7]):
                if v.lower() == "active":
                    reasons.add(name)
        if not mhz:
            return None
        return {"sm_mhz": float(np.median(mhz)), "sm_max_mhz": max(maxes), "reasons": sorted(reasons),
                "samples": len(mhz), "window": window}


def oracle_row(cfg, b, threads, max_chans=None):
    """One bounded sample of the workload on the host: batch row b (every channel when the row has at
    most 2^24 elements, else the first channels up to that size, and at most max_chans), full L, through
    the fp64 oracle as it stands.  Returns (state updates, seconds of oracle time, channels)."""
    import oracle
    from selective_state_space_126_b300 import synthetic as syn
    L, N = cfg.seqlen, cfg.dstate
    A, Dskip, bias = syn.layer_params(cfg.dim, N, cfg.dt_min, cfg.dt_max)
    chans = cfg.dim if cfg.seqlen * cfg.dim <= (1 << 24) else max(threads, (1 << 24) // cfg.seqlen)
    if max_chans is not None:
        chans = max(1, min(chans, max_chans))
    u = syn.channel_rows(cfg, syn.T_U, b, 0, chans)[None]
    dl = syn.channel_rows(cfg, syn.T_DELTA, b, 0, chans)[None]
    z = syn.channel_rows(cfg, syn.T_Z, b, 0, chans)[None] if cfg.gate else None
    Bm = syn.bc_rows(cfg, syn.T_B, b)[None]
    Cm = syn.bc_rows(cfg, syn.T_C, b)[None]
    t0 = time.perf_counter()
    oracle.selective_scan(u, dl, A[:chans], Bm, Cm, Dskip=Dskip[:chans] if cfg.dskip else None, z=z,
                          delta_bias=bias[:chans], nthreads=threads)
    return chans * L * N, time.perf_counter() - t0, chans


def cpu_baseline(cfg, target_s=10.0):
    """The fp64 oracle, as it stands, on a bounded sample of the workload: whole batch rows
    (see oracle_row), taken in order and repeated until about ``target_s`` of CPU time."""
    import oracle
    threads = oracle.default_threads()
    try:
        cores = len(os.sched_getaffinity(0))
    except AttributeError:
        cores = os.cpu_count() or 1
    elapsed, updates, rows, chans = 0.0, 0, 0, 0
    while elapsed < target_s and rows < 64:
        n, dt, chans = oracle_row(cfg, rows % cfg.batch, threads)
        elapsed += dt
        updates += n
        rows += 1
    return {"value": updates / elapsed, "unit": UNIT, "cores": threads, "host_cores_visible": cores,
            "kind": "oracle",
            "sample": f"{rows} batch rows of the workload (channels 0..{chans - 1} of {cfg.dim} each, "
                      f"full L={cfg.seqlen}, N={cfg.dstate}), {updates} state updates in {elapsed:.1f} s "
                      f"of oracle time"}


def random_device_inputs(cfg, seed, device):
    """Inputs with the workload's shapes and value distributions drawn on the GPU (seeded); used for
    the timing-only rows, where the host-side per-row recipe would take minutes to generate."""
    import torch
    from selective_state_space_126_b300 import synthetic as syn
    g = torch.Generator(device=device)
    g.manual_seed(1000 + seed)
    dt = torch.float32 if cfg.io_dtype == "f32" else torch.bfloat16
    B, D, L, N = cfg.batch, cfg.dim, cfg.seqlen, cfg.dstate

    def randn(*shape):
        return torch.randn(*shape, generator=g, device=device, dtype=torch.float32).to(dt)

    out = {"u": randn(B, D, L), "z": randn(B, D, L) if cfg.gate else None}
    nb = 1 if cfg.shared_bc else B
    if cfg.time_invariant:
        out["delta"] = randn(B, D, 1).expand(B, D, L).contiguous()
        out["Bm"] = randn(nb, N, 1).expand(nb, N, L).contiguous()
        out["Cm"] = randn(nb, N, 1).expand(nb, N, L).contiguous()
    else:
        out["delta"] = randn(B, D, L)
        out["Bm"], out["Cm"] = randn(nb, N, L), randn(nb, N, L)
    if cfg.shared_bc:
        out["Bm"], out["Cm"] = out["Bm"][0], out["Cm"][0]
    A, Dskip, bias = syn.layer_params(D, N, cfg.dt_min, cfg.dt_max, seed)
    out["A"] = torch.from_numpy(A).to(device)
    out["Dskip"] = torch.from_numpy(Dskip).to(device) if cfg.dskip else None
    out["delta_bias"] = torch.from_numpy(bias).to(device)
    return out


def sfu_ops_per_update(cfg):
    """SFU operations the bf16 scan kernel issues per state update: one ex2 for Abar per update, and per
    (batch, channel, step) one ex2 in softplus and, with the gate, one ex2 and one rcp in silu."""
    per_bdl_ex2 = 1 + (1 if cfg.gate else 0)
    per_bdl_rcp = 1 if cfg.gate else 0
    return 1.0 + per_bdl_ex2 / cfg.dstate, per_bdl_rcp / cfg.dstate


def probe_sfu_rate(lib, op, sms, stream, dev):
    """SFU operations per second on this GPU, measured with the library's probe kernel (8 independent
    chains per thread, 8 blocks of 256 threads per SM), best of 5 launches after a warm-up."""
    import torch
    blocks, iters = 8 * sms, 2048
    sink = torch.empty(blocks * 256, dtype=torch.float32, device=dev)
    sh = ctypes.c_void_p(stream.cuda_stream)
    run = lambda: lib.ssm_probe_sfu(op, blocks, iters, ctypes.c_void_p(sink.data_ptr()), sh)
    if run() != 0:
        raise RuntimeError("ssm_probe_sfu failed")
    best = None
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        best = ms if best is None else min(best, ms)
    return blocks * 256 * iters * 8 / (best * 1e-3)


def sfu_roofline(lib, cfg, launch_ms, sms, mhz, stream, dev):
    """The scan's second roofline: SFU work per launch in ex2-equivalents (an rcp counts as the ratio of
    the measured ex2 and rcp rates) over the launch time, against the measured ex2 rate."""
    ex2_rate = probe_sfu_rate(lib, 0, sms, stream, dev)
    rcp_rate = probe_sfu_rate(lib, 1, sms, stream, dev)
    ex2_pu, rcp_pu = sfu_ops_per_update(cfg)
    equiv = ex2_pu + rcp_pu * ex2_rate / rcp_rate
    achieved = cfg.updates * equiv / (launch_ms * 1e-3)
    return {"bound": "alu", "achieved": achieved / 1e12, "peak": ex2_rate / 1e12, "unit": "Tex2-equiv/s",
            "frac": achieved / ex2_rate, "ex2_per_update": ex2_pu, "rcp_per_update": rcp_pu,
            "ex2_equiv_per_update": equiv,
            "peak_basis": (f"measured by ssm_probe_sfu on this GPU: ex2 {ex2_rate / 1e12:.2f} T/s "
                           f"({ex2_rate / (sms * mhz * 1e6):.1f}/clk/SM at the median {mhz:.0f} MHz), "
                           f"rcp {rcp_rate / 1e12:.2f} T/s")}


def time_launches(run, n, stream, flush=None):
    """Mean device time of ``run`` over n launches (CUDA events on the launching stream), with an
    optional L2 flush between launches outside the timed events."""
    import torch
    ms = []
    for _ in range(n):
        if flush is not None:
            flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run()
        e1.record(stream)
        ms.append((e0, e1))
    torch.cuda.synchronize()
    return float(np.mean([a.elapsed_time(b) for a, b in ms]))


def decode_bytes(cfg) -> int:
    """Bytes one decode step must move: the fp32 state read and written; u, delta, z read and y
    written (B*D each, I/O dtype); B, C (B*N each); A (D*N) and D, delta_bias (D) in fp32."""
    es = 4 if cfg.io_dtype == "f32" else 2
    bd = cfg.batch * cfg.dim
    return (2 * bd * cfg.dstate * 4 + ((3 if cfg.gate else 2) + 1) * bd * es + 2 * cfg.batch * cfg.dstate * es
            + cfg.dim * cfg.dstate * 4 + 2 * cfg.dim * 4)


ROW_KEYS = {"cplx": "mamba2.8b_s4dlin_complex_bf16_b4_d5120_l2048_n16",
            "m130": "mamba130m_bf16_b8_d1536_l2048_n16", "ti": "mamba2.8b_ti_bf16_b1_d5120_l2048_n16",
            "long": "long_bf16_b1_d1536_l1048576_n16", "decode": "decode_bf16_b256_d5120_n16_x1000",
            "conv": "conv1d_silu_bf16_b4_d5120_l2048_w4", "bwd": "scan_bwd_mamba2.8b_bf16_b4_d5120_l2048_n16",
            "ssd": "ssd_mamba2_2.7b_bf16_b4_h80_p64_l2048_n128",
            "bwdzoh": "scan_bwd_zoh_mamba2.8b_bf16_b4_d5120_l2048_n16",
            "zoh": "mamba2.8b_zoh_bf16_b4_d5120_l2048_n16"}


def other_rows(lib, ssm, peak, stream, dev, which="all", decode_steps=1000):
    """The remaining rows of the hot path, each timed on its own full-size workload: the other
    scan shapes (single pass, time-invariant, the 2^20-step chunked scan) and 1000 decode steps."""
    import torch
    from selective_state_space_126_b300 import synthetic as syn
    sh = ctypes.c_void_p(stream.cuda_stream)
    # Reading 2x the L2 evicts the previous launch's lines and leaves only clean ones behind (a
    # write-based flush would leave dirty lines whose write-back lands in the timed launch).
    flush_buf = torch.ones(64 << 20, dtype=torch.float32, device=dev)
    flush_sink = torch.empty((), dtype=torch.float32, device=dev)

    def flush():
        torch.sum(flush_buf, dim=0, out=flush_sink)

    sel = set(ROW_KEYS) if which == "all" else set(which.split(","))
    rows = {}
    # (the "zoh" row: the 2.8B-shaped scan with the exact zero-order-hold input term)
    # (the "cplx" row: the 2.8B-shaped scan with a complex A, the S4D-Lin initialisation)
    for key, n in (("m130", 200), ("ti", 200), ("long", 5), ("zoh", 200), ("cplx", 100)):
        if key not in sel:
            continue
        name = ROW_KEYS[key]
        cfg = syn.M2P8 if key in ("zoh", "cplx") else syn.SCAN_CONFIGS[name]
        disc = ssm.SSM_DISC_ZOH if key == "zoh" else ssm.SSM_DISC_EULER
        inp = random_device_inputs(cfg, 0, dev)
        A_imag = None
        if key == "cplx":
            Ac = torch.from_numpy(syn.s4d_lin_A(cfg.dim, cfg.dstate)).to(dev)
            inp["A"], A_imag = Ac.real.contiguous(), Ac.imag.contiguous()
        y = torch.empty_like(inp["u"])
        a = ssm.make_scan_args(inp["u"], inp["delta"], inp["A"], inp["Bm"], inp["Cm"], y, inp["Dskip"], inp["z"],
                               inp["delta_bias"], discretization=disc, A_imag=A_imag)
        wsb = ssm.ssm_scan_workspace_size(a)
        ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=dev)
        a.workspace, a.workspace_bytes = ws.data_ptr(), wsb
        path = ssm.ssm_scan_plan_path(a)
        argp = ctypes.byref(a)

        def run():
            rc = lib.ssm_scan_fwd(argp, sh)
            if rc != 0:
                raise RuntimeError(ssm.status_name(rc))

        for _ in range(3):
            run()
        algo = algorithmic_bytes(cfg)
        ms = time_launches(run, n, stream, flush if algo < (256 << 20) else None)
        gbs = algo / (ms * 1e-3) / 1e9
        rows[name] = {"ms": ms, "value": cfg.updates / (ms * 1e-3), "unit": UNIT, "path": path,
                      "launches": {"tiled": 1, "split": 2, "chunked": 3, "generic": 1}[path],
                      "hbm_gbs_algorithmic": gbs, "frac": gbs / peak, "algorithmic_bytes": algo,
                      "l2": "flushed between launches" if algo < (256 << 20) else "inputs larger than L2"}
        del inp, y, ws
        torch.cuda.empty_cache()

    if "conv" in sel:
        # the causal depthwise convolution + SiLU in front of the scan, on the 2.8B-shaped layer
        name = ROW_KEYS["conv"]
        Bsz, D, L, W = 4, 5120, 2048, 4
        g = torch.Generator(device=dev)
        g.manual_seed(3000)
        x = torch.randn(Bsz, D, L, generator=g, device=dev).to(torch.bfloat16)
        bound = 1.0 / W ** 0.5
        wt = (torch.rand(D, W, generator=g, device=dev) * 2 - 1) * bound
        cb = (torch.rand(D, generator=g, device=dev) * 2 - 1) * bound
        xo = torch.empty_like(x)
        ca = ssm.make_conv_args(x, wt, xo, cb, None, True)

        def crun():
            rc = lib.ssm_causal_conv1d_fwd(ctypes.byref(ca), sh)
            if rc != 0:
                raise RuntimeError(ssm.status_name(rc))

        for _ in range(3):
            crun()
        ms = time_launches(crun, 200, stream, flush)
        byt = 2 * x.numel() * x.element_size() + wt.numel() * 4 + cb.numel() * 4
        gbs = byt / (ms * 1e-3) / 1e9
        rows[name] = {"ms": ms, "value": x.numel() / (ms * 1e-3), "unit": "outputs/s", "launches": 1,
                      "hbm_gbs_algorithmic": gbs, "frac": gbs / peak, "algorithmic_bytes": byt,
                      "l2": "flushed between launches"}
        del x, xo, wt, cb
        torch.cuda.empty_cache()

    for bkey, bdisc in (("bwd", ssm.SSM_DISC_EULER), ("bwdzoh", ssm.SSM_DISC_ZOH)):
        if bkey not in sel:
            continue
        # the backward pass (all gradients, states recomputed) on the 2.8B-shaped layer
        name = ROW_KEYS[bkey]
        cfg = syn.M2P8
        inp = random_device_inputs(cfg, 0, dev)
        dy = torch.randn(inp["u"].shape, generator=torch.Generator(device=dev).manual_seed(4000), device=dev).to(
            inp["u"].dtype)
        Bsz, D, L, N = cfg.batch, cfg.dim, cfg.seqlen, cfg.dstate
        grads = {k: torch.empty_like(inp["u"]) for k in ("du", "ddelta", "dz")}
        grads.update(dA=torch.empty(D, N, device=dev), dB=torch.empty(Bsz, N, L, device=dev),
                     dC=torch.empty(Bsz, N, L, device=dev), dDskip=torch.empty(D, device=dev),
                     ddelta_bias=torch.empty(D, device=dev), dh0=torch.empty(Bsz, D, N, device=dev))
        fa = ssm.make_scan_args(inp["u"], inp["delta"], inp["A"], inp["Bm"], inp["Cm"], None, inp["Dskip"], inp["z"],
                                inp["delta_bias"], discretization=bdisc)
        ba = ssm.make_bwd_args(fa, dy, grads)
        need = ctypes.c_size_t(0)
        if lib.ssm_scan_bwd_workspace_size(ctypes.byref(ba), ctypes.byref(need)) != 0:
            raise RuntimeError("ssm_scan_bwd_workspace_size failed")
        bws = torch.empty(max(need.value, 16), dtype=torch.uint8, device=dev)
        ba.fwd.workspace, ba.fwd.workspace_bytes = bws.data_ptr(), need.value

        def brun():
            rc = lib.ssm_scan_bwd(ctypes.byref(ba), sh)
            if rc != 0:
                raise RuntimeError(ssm.status_name(rc) + " " + lib.ssm_last_error_detail().decode())

        for _ in range(3):
            brun()
        ms = time_launches(brun, 20, stream, None)
        # read u, delta, z, dy and write du, ddelta, dz once; B, C read and dB, dC written (fp32) once
        es = inp["u"].element_size()
        byt = 7 * Bsz * D * L * es + 2 * Bsz * N * L * es + 2 * Bsz * N * L * 4 + (D * N + 2 * D) * 4
        gbs = byt / (ms * 1e-3) / 1e9
        # checkpoint pass (two launches when it takes the split single pass), zeroing, backward kernel
        ckpt_launches = 2 if ssm.ssm_scan_plan_path(ssm.make_scan_args(
            inp["u"], inp["delta"], inp["A"], inp["Bm"], inp["Cm"], dy, inp["Dskip"], inp["z"], inp["delta_bias"],
            discretization=bdisc, flags=ssm.SSM_SCAN_FORCE_TILED)) == "split" else 1
        rows[name] = {"ms": ms, "value": cfg.updates / (ms * 1e-3), "unit": UNIT, "launches": 2 + ckpt_launches,
                      "hbm_gbs_algorithmic": gbs, "frac": gbs / peak, "algorithmic_bytes": byt,
                      "workspace_bytes": need.value, "l2": "inputs larger than L2"}
        del inp, dy, grads, bws
        torch.cuda.empty_cache()

    if "ssd" in sel:
        # the Mamba-2 SSD layer (scalar A per head): 4 x 80 heads x 64 channels, L = 2048, N = 128, bf16
        name = ROW_KEYS["ssd"]
        Bsz, H, P, L, N = 4, 80, 64, 2048, 128
        g = torch.Generator(device=dev)
        g.manual_seed(5000)
        rnd = lambda *shape: torch.randn(*shape, generator=g, device=dev).to(torch.bfloat16)
        x, z, dl = rnd(Bsz, H * P, L), rnd(Bsz, H * P, L), rnd(Bsz, H, L)
        Bm, Cm = rnd(Bsz, L, N), rnd(Bsz, L, N)
        small = syn.ssd_inputs(1, H, 1, 8, N, "bf16", seed=5000)     # per-head A, Dskip, delta_bias
        Ah, Dh, bh = (torch.from_numpy(small[k]).to(dev) for k in ("A", "Dskip", "delta_bias"))
        ys = torch.empty_like(x)
        sa = ssm.make_ssd_args(x, dl, Ah, Bm, Cm, ys, Dh, z, bh)
        path = ssm.ssm_ssd_plan_path(sa)

        def srun():
            rc = lib.ssm_ssd_fwd(ctypes.byref(sa), sh)
            if rc != 0:
                raise RuntimeError(ssm.status_name(rc) + " " + lib.ssm_last_error_detail().decode())

        for _ in range(3):
            srun()
        ms = time_launches(srun, 50, stream, None)
        es = 2
        byt = (3 * Bsz * H * P * L + Bsz * H * L + 2 * Bsz * L * N) * es + 3 * H * 4
        chunks = (L + 127) // 128
        flops = Bsz * H * chunks * 2 * (128 * 128 * N + 3 * 128 * P * 128)   # C B^T, state, inter- and intra-chunk
        gbs = byt / (ms * 1e-3) / 1e9
        tfl = flops / (ms * 1e-3) / 1e12
        rows[name] = {"ms": ms, "value": Bsz * H * P * N * L / (ms * 1e-3), "unit": UNIT, "path": path,
                      "launches": 1, "hbm_gbs_algorithmic": gbs, "frac": gbs / peak, "algorithmic_bytes": byt,
                      "tensor_tflops": tfl, "tensor_flops_per_launch": flops, "l2": "inputs larger than L2"}
        del x, z, dl, Bm, Cm, ys
        torch.cuda.empty_cache()

    if "decode" not in sel:
        del flush_buf, flush_sink
        return rows
    # decode: consecutive steps (1000 by default) against one persistent fp32 state
    dc = syn.with_decode_steps(syn.DECODE, decode_steps) if decode_steps != syn.DECODE.steps else syn.DECODE
    g = torch.Generator(device=dev)
    g.manual_seed(2000)
    Bsz, D, N, steps = dc.batch, dc.dim, dc.dstate, dc.steps
    bf = torch.bfloat16 if dc.io_dtype == "bf16" else torch.float32
    state = torch.randn(Bsz, D, N, generator=g, device=dev)
    toks = {k: torch.randn(steps, Bsz, D, generator=g, device=dev).to(bf) for k in ("u", "delta", "z")}
    bcs = {k: torch.randn(steps, Bsz, N, generator=g, device=dev).to(bf) for k in ("Bm", "Cm")}
    A, Dskip, bias = syn.decode_params(dc)
    A, Dskip, bias = (torch.from_numpy(x).to(dev) for x in (A, Dskip, bias))
    yd = torch.empty(Bsz, D, dtype=bf, device=dev)
    sargs = [ssm.make_step_args(state, toks["u"][i], toks["delta"][i], A, bcs["Bm"][i], bcs["Cm"][i], yd, Dskip,
                                toks["z"][i], bias) for i in range(steps)]
    it = iter(range(10 ** 9))

    def dstep():
        i = next(it) % steps
        rc = lib.ssm_state_update(ctypes.byref(sargs[i]), sh)
        if rc != 0:
            raise RuntimeError(ssm.status_name(rc))

    for _ in range(3):
        dstep()
    ms = time_launches(dstep, steps, stream, flush)
    byt = decode_bytes(dc)
    gbs = byt / (ms * 1e-3) / 1e9
    rows[dc.name] = {"ms_per_step": ms, "value": dc.updates_per_step / (ms * 1e-3), "unit": UNIT,
                     "steps": steps, "hbm_gbs_algorithmic": gbs, "frac": gbs / peak, "algorithmic_bytes": byt,
                     "l2": "flushed between steps (the 84 MB state would otherwise stay in the 126 MB L2)"}
    del flush_buf, flush_sink, state, toks, bcs
    torch.cuda.empty_cache()
    return rows


def run_reference(args, rank, world):
    """--impl reference: the fp64 oracle timed on the host cores (rank 0 only).  Each step is one
    bounded sample of the workload, the same sample the cpu_baseline leg takes: one whole batch row
    (every channel, full L), rows taken in order."""
    if rank != 0:
        return
    import oracle
    cfg = workload(args)
    threads = oracle.default_threads()
    # whole rows unless the run would then exceed about a minute of oracle time (at ~6e8 updates/s)
    cap = max(256, int(3.6e10 / max(1, args.steps + args.warmup) / (cfg.seqlen * cfg.dstate)))
    for i in range(args.warmup):
        oracle_row(cfg, i % cfg.batch, threads, cap)
    updates, elapsed, chans = 0, 0.0, 0
    for i in range(args.steps):
        n, dt, chans = oracle_row(cfg, i % cfg.batch, threads, cap)
        updates += n
        elapsed += dt
    value = updates / elapsed
    sample = (f"each step: one batch row of the workload (channels 0..{chans - 1} of {cfg.dim}, full "
              f"L={cfg.seqlen}, N={cfg.dstate}), rows in order; the cpu_baseline leg takes the same whole rows")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": elapsed / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": bench_config(cfg, world),
        "cpu_baseline": {"kind": "oracle", "cores": threads, "sample": sample, "value": value, "unit": UNIT},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    args = parse()
    rank, world, local = dist_info()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    import torch
    import selective_state_space_126_b300 as ssm
    from selective_state_space_126_b300 import build
    from selective_state_space_126_b300.synthetic import device_inputs

    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    if build.is_stale():
        if rank == 0:
            build.build_library(quiet=True)
        if world > 1:
            torch.distributed.barrier()
    lib = ssm.load_library()
    cfg = workload(args)
    dev = torch.device("cuda", torch.cuda.current_device())
    if args.only_rows:
        if rank == 0:
            peak, _ = measured_peaks()
            print(json.dumps({"rows": other_rows(lib, ssm, peak, torch.cuda.current_stream(), dev, args.rows,
                                                 args.decode_steps)}), flush=True)
        return

    # ---- inputs resident in HBM (each rank its own replica, seeded by rank) ----
    inp = device_inputs(cfg, seed=rank)
    y = torch.empty_like(inp["u"])
    a = ssm.make_scan_args(inp["u"], inp["delta"], inp["A"], inp["Bm"], inp["Cm"], y, inp["Dskip"], inp["z"],
                           inp["delta_bias"])
    path = ssm.ssm_scan_plan_path(a)
    ws_bytes = ssm.ssm_scan_workspace_size(a)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    a.workspace, a.workspace_bytes = ws.data_ptr(), ws_bytes
    launches_per_step = ssm_launches(lib, ssm, a)
    stream = torch.cuda.current_stream()
    sh = ctypes.c_void_p(stream.cuda_stream)
    argp = ctypes.byref(a)

    def step():
        rc = lib.ssm_scan_fwd(argp, sh)
        if rc != 0:
            raise RuntimeError(ssm.status_name(rc) + " " + lib.ssm_last_error_detail().decode())

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()

    # L2 flush between steps, outside the step events: a read of twice the L2 leaves only clean lines
    # behind, so no write-back of the previous step's y lands in the next timed step
    flush_buf = torch.ones(64 << 20, dtype=torch.float32, device=dev)
    flush_sink = torch.empty((), dtype=torch.float32, device=dev)

    def flush():
        torch.sum(flush_buf, dim=0, out=flush_sink)

    sampler = ClockSampler(int(os.environ.get("CUDA_VISIBLE_DEVICES", "0").split(",")[0])
                           if os.environ.get("CUDA_VISIBLE_DEVICES", "").isdigit() else local)
    sampler.start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    w0 = time.time()
    start.record(stream)
    for i in range(args.steps):
        flush()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    stop.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    w1 = time.time()
    sampler.stop()
    region_ms = start.elapsed_time(stop)
    launch_ms = float(np.mean([s.elapsed_time(e) for s, e in ev]))
    # a step is the scan between its events; the flushes between steps are not part of it
    ms_per_step = max_over_ranks(launch_ms, world, dev)
    del flush_buf, flush_sink
    updates_per_step = cfg.updates * world
    value = job_value(cfg.updates, world, ms_per_step)

    # ---- end to end through the C ABI from pinned host buffers ----
    # Batch rows are independent scans, so the step is pipelined over chunks of rows on three streams:
    # the host-to-device copies of chunk i+1 overlap the scan of chunk i and the read-back of chunk i-1,
    # and both copy directions run at once.  Every byte of input and of y crosses the link every step.
    e2e = None
    if not args.no_e2e:
        seq_names = ["u", "delta", "z"] + (["Bm", "Cm"] if inp["Bm"].dim() == 3 else [])
        par_names = ["A", "Dskip", "delta_bias"] + ([] if inp["Bm"].dim() == 3 else ["Bm", "Cm"])
        hbuf = {k: inp[k].cpu().pin_memory() for k in seq_names + par_names if inp[k] is not None}
        y_resident = y.float().cpu()
        hy = torch.empty(y.shape, dtype=y.dtype).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in hbuf.values())
        d2h = hy.numel() * hy.element_size()
        nchunk = min(cfg.batch, 4)
        bounds = [(i * cfg.batch // nchunk, (i + 1) * cfg.batch // nchunk) for i in range(nchunk)]
        s_in, s_run, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
        # the small per-channel parameters are double-buffered across steps, so that copying the next
        # step's never waits for this step's last scan
        par = [{k: inp[k] if inp[k] is None else torch.empty_like(inp[k]) for k in par_names} for _ in range(2)]
        chunk_args, chunk_ws = [[], []], []
        for b0, b1 in bounds:
            wsb = 0
            for q in range(2):
                src = dict(inp, **par[q])
                rows = lambda k: src[k][b0:b1] if src[k] is not None else None
                bc = (lambda k: src[k][b0:b1]) if src["Bm"].dim() == 3 else (lambda k: src[k])
                ca = ssm.make_scan_args(rows("u"), rows("delta"), src["A"], bc("Bm"), bc("Cm"), y[b0:b1],
                                        src["Dskip"], rows("z"), src["delta_bias"])
                if q == 0:
                    wsb = ssm.ssm_scan_workspace_size(ca)
                    chunk_ws.append(torch.empty(max(wsb, 16), dtype=torch.uint8, device=dev))
                ca.workspace, ca.workspace_bytes = chunk_ws[-1].data_ptr(), wsb
                chunk_args[q].append(ca)
        ev_in = [torch.cuda.Event() for _ in bounds]
        ev_run = [torch.cuda.Event() for _ in bounds]
        ev_out = [torch.cuda.Event() for _ in bounds]
        ev_par = [torch.cuda.Event() for _ in range(2)]
        ev_par_used = [torch.cuda.Event() for _ in range(2)]
        h_run = ctypes.c_void_p(s_run.cuda_stream)
        n_e2e = [0]

        def e2e_step(first):
            q = n_e2e[0] % 2
            n_e2e[0] += 1
            with torch.cuda.stream(s_in):
                if n_e2e[0] > 2:
                    s_in.wait_event(ev_par_used[q])     # the scans of two steps ago are done with this buffer
                for k in par_names:
                    if inp[k] is not None:
                        par[q][k].copy_(hbuf[k], non_blocking=True)
                ev_par[q].record(s_in)
            for i, (b0, b1) in enumerate(bounds):
                with torch.cuda.stream(s_in):
                    if not first:
                        s_in.wait_event(ev_run[i])      # the previous step's scan of these rows has read them
                    for k in seq_names:
                        if inp[k] is not None:
                            inp[k][b0:b1].copy_(hbuf[k][b0:b1], non_blocking=True)
                    ev_in[i].record(s_in)
                s_run.wait_event(ev_in[i])
                s_run.wait_event(ev_par[q])
                if not first:
                    s_run.wait_event(ev_out[i])     # the previous step's read-back of these rows is done
                rc = lib.ssm_scan_fwd(ctypes.byref(chunk_args[q][i]), h_run)
                if rc != 0:
                    raise RuntimeError(ssm.status_name(rc) + " " + lib.ssm_last_error_detail().decode())
                ev_run[i].record(s_run)
                s_out.wait_event(ev_run[i])
                with torch.cuda.stream(s_out):
                    hy[b0:b1].copy_(y[b0:b1], non_blocking=True)
                    ev_out[i].record(s_out)
            ev_par_used[q].record(s_run)

        for w in range(3):
            e2e_step(w == 0)
        torch.cuda.synchronize()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for st in (s_in, s_run, s_out):
            st.wait_event(s0)
        for _ in range(args.e2e_steps):
            e2e_step(False)
        for e in ev_out:
            stream.wait_event(e)
        s1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = s0.elapsed_time(s1) / args.e2e_steps
        e2e_ms = max_over_ranks(e2e_ms, world, dev)
        # the pipelined, host-to-host result must be the device-resident one
        e2e_diff = float((hy.float() - y_resident).abs().max())
        if not e2e_diff <= 1e-2 * max(1.0, float(y_resident.abs().max())):
            raise RuntimeError(f"pipelined end-to-end y differs from the resident run by {e2e_diff}")
        e2e = {"value": updates_per_step / (e2e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "steps": args.e2e_steps,
               "host_memory": "pinned", "pipeline": f"{nchunk} chunks of batch rows on 3 streams",
               "max_abs_diff_vs_resident": e2e_diff,
               "gpu_launches_per_step": sum(ssm_launches(lib, ssm, ca) for ca in chunk_args[0])}

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    # ---- roofline of the scan kernel ----
    peak, peak_kind = measured_peaks()
    algo = algorithmic_bytes(cfg)
    # the split single pass's two launches run side by side: their union is the scan kernel's time
    kernel_ms = launch_ms / launches_per_step if path not in ("tiled", "split") else launch_ms
    achieved = algo / (launch_ms * 1e-3) / 1e9
    traffic = None
    if os.path.exists(TRAFFIC_FILE):
        with open(TRAFFIC_FILE) as f:
            tr = json.load(f)
        if tr.get("kernel_source_sha") == source_sha() and tr.get("workload") == cfg.name:
            traffic = tr.get("dram_bytes_per_launch")
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    clocks = sampler.summary(w0, w1)
    mhz = (clocks or {}).get("sm_mhz") or 1900.0
    sfu = sfu_roofline(lib, cfg, launch_ms, sms, mhz, stream, dev)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_per_step, "timed_region_ms": region_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": bench_config(cfg, world), "path": path,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic, "peak_kind": peak_kind, "algorithmic_bytes_per_launch": algo,
                     "kernel_ms": kernel_ms},
        "sfu_roofline": sfu,
        "gpu_launches": args.steps * launches_per_step,
        "clocks": clocks,
        "e2e": e2e,
    }
    if not args.no_rows:
        line["rows"] = other_rows(lib, ssm, peak, stream, dev, args.rows, args.decode_steps)
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg)
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
