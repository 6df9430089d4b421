"""Seeded synthetic inputs for the selective scan and the decode step.

This module holds the input recipe only -- none of the scan's arithmetic --
so that the CUDA path and the fp64 oracle can consume identical values.

Recipe (the distributions of the Mamba layer workloads):
  * u, delta, z, B, C, D ~ N(0, 1) drawn as float32;
  * Delta0[d] log-uniform in [dt_min, dt_max] per channel, and
    delta_bias = softplus^-1(Delta0) (the Delta-bias initialisation of the
    Mamba paper, "gitcode.csdn.net", section 3.6 "Parameterization of Delta");
  * A[d, n] = -(n + 1) (S4D-Real initialisation, same page, section 3.6
    "Initialization");
  * tensors whose I/O dtype is bf16 are rounded once, round-to-nearest-even,
    and both sides consume exactly those values;
  * the causal convolution in front of the scan: input x ~ N(0, 1) (a stream
    of its own), taps and bias ~ U(-1/sqrt(W), 1/sqrt(W)), the default
    initialisation of a framework's depthwise Conv1d (fan-in W).

Every row of every tensor has its own PCG64 stream, keyed by
(seed, tensor id, batch index, row index[, step]).  Any channel can therefore
be regenerated alone, which is how the oracle checks sampled channels of
workloads too large to hold on the host.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np

# tensor ids of the per-row streams
T_U, T_DELTA, T_Z, T_B, T_C, T_D, T_DT0, T_STATE, T_X, T_CONVW, T_CONVB = range(11)


@dataclass(frozen=True)
class ScanConfig:
    name: str
    batch: int
    dim: int
    seqlen: int
    dstate: int
    io_dtype: str            # "f32" or "bf16"
    dt_min: float = 1e-3
    dt_max: float = 1e-1
    gate: bool = True
    dskip: bool = True
    time_invariant: bool = False   # delta, B, C constant over t
    shared_bc: bool = False        # B, C shared across the batch (batch stride 0)

    @property
    def updates(self) -> int:
        return self.batch * self.dim * self.seqlen * self.dstate


@dataclass(frozen=True)
class DecodeConfig:
    name: str
    batch: int
    dim: int
    dstate: int
    steps: int
    io_dtype: str = "bf16"
    dt_min: float = 1e-3
    dt_max: float = 1e-1
    gate: bool = True
    dskip: bool = True

    @property
    def updates_per_step(self) -> int:
        return self.batch * self.dim * self.dstate


# The five workloads: a tiny fp32 case, two Mamba layer shapes, a long
# sequence, and the decode step.
TINY = ScanConfig("tiny_fp32_b1_d16_l256_n16", 1, 16, 256, 16, "f32")
M130 = ScanConfig("mamba130m_bf16_b8_d1536_l2048_n16", 8, 1536, 2048, 16, "bf16")
M2P8 = ScanConfig("mamba2.8b_bf16_b4_d5120_l2048_n16", 4, 5120, 2048, 16, "bf16")
M2P8_TI = ScanConfig("mamba2.8b_ti_bf16_b1_d5120_l2048_n16", 1, 5120, 2048, 16, "bf16",
                     time_invariant=True, shared_bc=True)
LONG = ScanConfig("long_bf16_b1_d1536_l1048576_n16", 1, 1536, 1 << 20, 16, "bf16",
                  dt_min=1e-4, dt_max=1e-2)
DECODE = DecodeConfig("decode_bf16_b256_d5120_n16_x1000", 256, 5120, 16, 1000)

SCAN_CONFIGS = {c.name: c for c in (TINY, M130, M2P8, M2P8_TI, LONG)}


def with_decode_steps(cfg: DecodeConfig, steps: int) -> DecodeConfig:
    """A copy of the decode workload with another number of steps (same shapes and distributions)."""
    return replace(cfg, steps=steps, name=f"{cfg.name}_steps{steps}")


def with_shape(cfg: ScanConfig, **kw) -> ScanConfig:
    """A copy of ``cfg`` with some fields replaced (same distributions)."""
    return replace(cfg, **kw)


def _rng(seed: int, *key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, *key])))


def round_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round-to-nearest-even."""
    bits = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (bits >> 16) & np.uint32(1)
    return ((bits + np.uint32(0x7FFF) + lsb) >> 16).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def round_io(x: np.ndarray, io_dtype: str) -> np.ndarray:
    """Round float32 values to the I/O dtype and return them as exact float32."""
    x = np.asarray(x, dtype=np.float32)
    if io_dtype == "bf16":
        return bf16_bits_to_f32(round_to_bf16_bits(x))
    if io_dtype == "f32":
        return x
    raise ValueError(io_dtype)


def _normal_row(seed: int, tensor: int, b: int, row: int, n: int) -> np.ndarray:
    return _rng(seed, tensor, b, row).standard_normal(n, dtype=np.float32)


def channel_rows(cfg: ScanConfig, tensor: int, b: int, d0: int, d1: int, seed: int = 0) -> np.ndarray:
    """Rows d0..d1-1 of u / delta / z for batch b: float32 (d1-d0, L), rounded to the I/O dtype."""
    L = cfg.seqlen
    out = np.empty((d1 - d0, L), dtype=np.float32)
    for i, d in enumerate(range(d0, d1)):
        if tensor == T_DELTA and cfg.time_invariant:
            out[i, :] = _normal_row(seed, tensor, b, d, 1)[0]
        else:
            out[i, :] = _normal_row(seed, tensor, b, d, L)
    return round_io(out, cfg.io_dtype)


def bc_rows(cfg: ScanConfig, tensor: int, b: int, seed: int = 0) -> np.ndarray:
    """B or C for batch b: float32 (N, L), rounded to the I/O dtype."""
    N, L = cfg.dstate, cfg.seqlen
    bb = 0 if cfg.shared_bc else b
    out = np.empty((N, L), dtype=np.float32)
    for n in range(N):
        if cfg.time_invariant:
            out[n, :] = _normal_row(seed, tensor, bb, n, 1)[0]
        else:
            out[n, :] = _normal_row(seed, tensor, bb, n, L)
    return round_io(out, cfg.io_dtype)


def softplus_inverse(x: np.ndarray) -> np.ndarray:
    """softplus^-1(x) = log(exp(x) - 1) = x + log(-expm1(-x)), stable for small x."""
    x = np.asarray(x, dtype=np.float64)
    return x + np.log(-np.expm1(-x))


def layer_params(dim: int, dstate: int, dt_min: float, dt_max: float, seed: int = 0):
    """A (D, N), Dskip (D,), delta_bias (D,) as float32."""
    A = -np.tile(np.arange(1, dstate + 1, dtype=np.float32), (dim, 1))
    Dskip = _rng(seed, T_D).standard_normal(dim, dtype=np.float32)
    lo, hi = np.log(dt_min), np.log(dt_max)
    dt0 = np.exp(_rng(seed, T_DT0).uniform(lo, hi, dim))
    delta_bias = softplus_inverse(dt0).astype(np.float32)
    return A, Dskip, delta_bias


def s4d_lin_A(dim: int, dstate: int):
    """The S4D-Lin initialisation of a complex diagonal A ("Mamba paper translation", section 3.6):
    A[d, n] = -1/2 + n i, as complex64 (D, N)."""
    return np.tile((-0.5 + 1j * np.arange(dstate)).astype(np.complex64), (dim, 1))


def ssd_inputs(batch: int, nheads: int, headdim: int, seqlen: int, dstate: int, io_dtype: str = "bf16",
               seed: int = 0, dt_min: float = 1e-3, dt_max: float = 1e-1) -> dict:
    """Inputs of the Mamba-2 SSD layer as float32 arrays (values exact in the I/O dtype).

    x, z (B, H*P, L), delta (B, H, L), Bm, Cm (B, L, N) ~ N(0, 1); per head A = -U(1, 16) (the
    scalar times the identity), Dskip ~ N(0, 1), delta_bias = softplus^-1(Delta0) with Delta0
    log-uniform in [dt_min, dt_max]."""
    rng = np.random.default_rng([seed, 7001])
    r = lambda *shape: round_io(rng.standard_normal(shape, dtype=np.float32), io_dtype)
    D = nheads * headdim
    x, z = r(batch, D, seqlen), r(batch, D, seqlen)
    delta = r(batch, nheads, seqlen)
    Bm, Cm = r(batch, seqlen, dstate), r(batch, seqlen, dstate)
    A = (-rng.uniform(1.0, 16.0, nheads)).astype(np.float32)
    Dskip = rng.standard_normal(nheads, dtype=np.float32)
    dt0 = np.exp(rng.uniform(np.log(dt_min), np.log(dt_max), nheads))
    bias = softplus_inverse(dt0).astype(np.float32)
    return dict(x=x, delta=delta, z=z, Bm=Bm, Cm=Cm, A=A, Dskip=Dskip, delta_bias=bias)


def conv_params(dim: int, width: int, seed: int = 0):
    """Conv taps (D, W) and bias (D,) as float32, uniform in +-1/sqrt(W)."""
    bound = 1.0 / np.sqrt(width)
    w = _rng(seed, T_CONVW).uniform(-bound, bound, (dim, width)).astype(np.float32)
    bias = _rng(seed, T_CONVB).uniform(-bound, bound, dim).astype(np.float32)
    return w, bias


def scan_inputs(cfg: ScanConfig, seed: int = 0, batches=None) -> dict:
    """All scan inputs of ``cfg`` as float32 arrays (values exact in the I/O dtype).

    Keys: u, delta, z (B, D, L); Bm, Cm (B or 1, N, L); A (D, N); Dskip,
    delta_bias (D,).  ``batches`` restricts the batch indices generated.
    """
    bs = list(range(cfg.batch)) if batches is None else list(batches)
    D = cfg.dim
    u = np.stack([channel_rows(cfg, T_U, b, 0, D, seed) for b in bs])
    delta = np.stack([channel_rows(cfg, T_DELTA, b, 0, D, seed) for b in bs])
    z = np.stack([channel_rows(cfg, T_Z, b, 0, D, seed) for b in bs]) if cfg.gate else None
    bc_b = [0] if cfg.shared_bc else bs
    Bm = np.stack([bc_rows(cfg, T_B, b, seed) for b in bc_b])
    Cm = np.stack([bc_rows(cfg, T_C, b, seed) for b in bc_b])
    A, Dskip, delta_bias = layer_params(D, cfg.dstate, cfg.dt_min, cfg.dt_max, seed)
    return dict(u=u, delta=delta, z=z, Bm=Bm, Cm=Cm, A=A,
                Dskip=Dskip if cfg.dskip else None, delta_bias=delta_bias)


def decode_params(cfg: DecodeConfig, seed: int = 0):
    return layer_params(cfg.dim, cfg.dstate, cfg.dt_min, cfg.dt_max, seed)


def decode_state(cfg: DecodeConfig, seed: int = 0, batches=None) -> np.ndarray:
    """Initial persistent state h ~ N(0,1), float32 (B, D, N)."""
    bs = list(range(cfg.batch)) if batches is None else list(batches)
    return np.stack([_rng(seed, T_STATE, b).standard_normal((cfg.dim, cfg.dstate), dtype=np.float32)
                     for b in bs])


def decode_step_inputs(cfg: DecodeConfig, step: int, seed: int = 0) -> dict:
    """One token per sequence: u, delta, z (B, D) and Bm, Cm (B, N), rounded to the I/O dtype."""
    B, D, N = cfg.batch, cfg.dim, cfg.dstate

    def draw(tensor, shape):
        return round_io(_rng(seed, tensor, 1_000_000 + step).standard_normal(shape, dtype=np.float32),
                        cfg.io_dtype)

    return dict(u=draw(T_U, (B, D)), delta=draw(T_DELTA, (B, D)),
                z=draw(T_Z, (B, D)) if cfg.gate else None,
                Bm=draw(T_B, (B, N)), Cm=draw(T_C, (B, N)))


def device_inputs(cfg: ScanConfig, seed=0, block=128, workers=8, device="cuda"):
    """All inputs of ``cfg`` on the GPU (torch tensors), generated block by block on the host."""
    import concurrent.futures as cf

    import torch
    B, D, L, N = cfg.batch, cfg.dim, cfg.seqlen, cfg.dstate
    dt = torch.float32 if cfg.io_dtype == "f32" else torch.bfloat16
    out = {}
    tensors = [("u", T_U), ("delta", T_DELTA)] + ([("z", T_Z)] if cfg.gate else [])
    for name, _ in tensors:
        out[name] = torch.empty((B, D, L), dtype=dt, device=device)
    jobs = [(name, tid, b, d0, min(D, d0 + block)) for name, tid in tensors for b in range(B)
            for d0 in range(0, D, block)]

    def gen(job):
        name, tid, b, d0, d1 = job
        return job, channel_rows(cfg, tid, b, d0, d1, seed)

    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        for (name, tid, b, d0, d1), rows in ex.map(gen, jobs):
            out[name][b, d0:d1].copy_(torch.from_numpy(rows).to(dt))
    if not cfg.gate:
        out["z"] = None
    bb = [0] if cfg.shared_bc else list(range(B))
    up = lambda x, t=torch.float32: torch.from_numpy(np.ascontiguousarray(x)).to(t).to(device)
    out["Bm"] = up(np.stack([bc_rows(cfg, T_B, b, seed) for b in bb]), dt)
    out["Cm"] = up(np.stack([bc_rows(cfg, T_C, b, seed) for b in bb]), dt)
    A, Dskip, bias = layer_params(D, N, cfg.dt_min, cfg.dt_max, seed)
    out["A"] = up(A)
    out["Dskip"] = up(Dskip) if cfg.dskip else None
    out["delta_bias"] = up(bias)
    return out
