// scan_warp.cu -- the selective scan as a time-parallel associative scan across
// the lanes of a warp ("Mamba and state space models", docs.ifdog.com, section
// "Hardware-aware parallel scan": the recurrence h_t = Abar_t h_{t-1} + Bbar_t x_t
// is a composition of affine maps, combined associatively as
// (a2, b2) o (a1, b1) = (a2 a1, a2 b1 + b2); "Mamba paper translation",
// gitcode.csdn.net, section 3.3.2, parallel scan).
//
// One warp per (batch, channel); a tile is 32 consecutive steps, one per lane.
// Each lane forms (Abar_t[n], Delta_t B_t[n] u_t) of its step for every state,
// five shuffle rounds (offsets 1, 2, 4, 8, 16) turn them into the inclusive
// compositions over the tile, and the state entering the tile (the carry, the
// same in every lane) is applied to all 32 steps at once: h_t = a h_in + b.
// Lane 31's state is the next tile's carry.  Steps past the end of the
// sequence take the identity map (1, 0), so the carry after the last tile is
// h_last.  Euler input term, real A, dstate <= 16, any strides.
//
// It is selected only on request (SSM_SCAN_FORCE_WARPSCAN): against the
// thread-sequential scans it does about six times the arithmetic per state
// update (the five combine rounds and their shuffles) to put 32 times as many
// threads on each channel.
#include "device_math.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int kWarpScanThreads = 128;

template <typename IO, bool PRECISE>
__global__ void __launch_bounds__(kWarpScanThreads) scan_warp_kernel(const ScanProblem p) {
  const int lane = threadIdx.x & 31;
  const int64_t c = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (c >= p.B * p.D) return;   // a whole warp leaves together
  const int64_t b = c / p.D, d = c % p.D;
  const int N = (int)p.N;
  const IO* u = static_cast<const IO*>(p.u) + b * p.su[0] + d * p.su[1];
  const IO* dl = static_cast<const IO*>(p.delta) + b * p.sd[0] + d * p.sd[1];
  const IO* z = p.z ? static_cast<const IO*>(p.z) + b * p.sz[0] + d * p.sz[1] : nullptr;
  const IO* Bm = static_cast<const IO*>(p.Bm) + b * p.sB[0];
  const IO* Cm = static_cast<const IO*>(p.Cm) + b * p.sC[0];
  IO* y = static_cast<IO*>(p.y) + b * p.sy[0] + d * p.sy[1];

  float A2[16], carry[16];
#pragma unroll
  for (int n = 0; n < 16; ++n) {
    A2[n] = 0.f;
    carry[n] = 0.f;
    if (n < N) {
      A2[n] = p.A[d * p.sA[0] + n * p.sA[1]] * kLog2e;
      if (p.h0) carry[n] = p.h0[b * p.sh0[0] + d * p.sh0[1] + n * p.sh0[2]];
    }
  }
  const float bias = p.bias ? p.bias[d] : 0.f;
  const float Dd = p.Dskip ? p.Dskip[d] : 0.f;

  for (int64_t t0 = 0; t0 < p.L; t0 += 32) {
    const int64_t t = t0 + lane;
    const bool in = t < p.L;
    float uv = 0.f, dt = 0.f;
    if (in) {
      uv = to_f32(u[t]);
      dt = delta_of<PRECISE>(to_f32(dl[t]), bias, p.softplus);
    }
    const float du = dt * uv;
    // this step's affine map per state; the identity past the end and for padded states
    float a[16], bx[16];
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      a[n] = 1.f;
      bx[n] = 0.f;
      if (in && n < N) {
        a[n] = ex2_approx(dt * A2[n]);
        bx[n] = du * to_f32(Bm[n * p.sB[1] + t]);
      }
    }
    // inclusive scan over the lanes: lane t ends with the composition of steps t0 .. t
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
#pragma unroll
      for (int n = 0; n < 16; ++n) {
        const float ap = __shfl_up_sync(0xffffffffu, a[n], off);
        const float bp = __shfl_up_sync(0xffffffffu, bx[n], off);
        if (lane >= off) {
          bx[n] = fmaf(a[n], bp, bx[n]);   // the later map applied to the earlier one's offset
          a[n] *= ap;
        }
      }
    }
    // the states of all 32 steps from the tile's incoming state, the C contraction, and the carry
    float acc = 0.f;
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      const float hn = fmaf(a[n], carry[n], bx[n]);
      if (in && n < N) acc = fmaf(to_f32(Cm[n * p.sC[1] + t]), hn, acc);
      carry[n] = __shfl_sync(0xffffffffu, hn, 31);
    }
    if (in) {
      float out = fmaf(Dd, uv, acc);
      if (z) out *= silu<PRECISE>(to_f32(z[t]));
      y[t] = from_f32<IO>(out);
    }
  }
  if (p.h_last && lane == 0) {
#pragma unroll
    for (int n = 0; n < 16; ++n)
      if (n < N) p.h_last[b * p.shl[0] + d * p.shl[1] + n * p.shl[2]] = carry[n];
  }
}

}  // namespace

cudaError_t launch_scan_warp(const ScanProblem& p, cudaStream_t s) {
  const int64_t warps = p.B * p.D;
  const dim3 grid((unsigned)((warps * 32 + kWarpScanThreads - 1) / kWarpScanThreads));
  if (p.io == SSM_F32) scan_warp_kernel<float, true><<<grid, kWarpScanThreads, 0, s>>>(p);
  else scan_warp_kernel<__nv_bfloat16, false><<<grid, kWarpScanThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace ssm
