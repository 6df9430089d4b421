// scan_generic.cu -- stride-general selective scan, one thread per (batch, channel).
//
// Used for the shapes the tiled kernel does not take: unaligned or ragged
// rows (seqlen not a multiple of the 16-byte vector), strided layouts, empty
// sequences.  It runs the recurrence of the Mamba paper ("gitcode.csdn.net",
// section 2, recurrent mode; Delta = softplus(delta + bias), Abar = exp(Delta A),
// Bbar x = Delta B u, or the exact zero-order hold) with the state in registers, the silu gate of the Mamba
// block ("docs.ifdog.com", section "Mamba architecture") and the D skip term;
// a second kernel takes a complex A.
#include "device_math.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

template <typename IO, int NB, bool PRECISE>
__global__ void __launch_bounds__(128) scan_generic_kernel(const ScanProblem p) {
  const int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= p.B * p.D) return;
  const int64_t b = c / p.D, d = c % p.D;
  const int N = (int)p.N;
  const IO* u = static_cast<const IO*>(p.u) + b * p.su[0] + d * p.su[1];
  const IO* dl = static_cast<const IO*>(p.delta) + b * p.sd[0] + d * p.sd[1];
  const IO* z = p.z ? static_cast<const IO*>(p.z) + b * p.sz[0] + d * p.sz[1] : nullptr;
  const IO* Bm = static_cast<const IO*>(p.Bm) + b * p.sB[0];
  const IO* Cm = static_cast<const IO*>(p.Cm) + b * p.sC[0];
  IO* y = static_cast<IO*>(p.y) + b * p.sy[0] + d * p.sy[1];

  float A2[NB], h[NB], Ai[NB];
#pragma unroll
  for (int n = 0; n < NB; ++n) {
    const float a = n < N ? p.A[d * p.sA[0] + n * p.sA[1]] : 0.f;
    A2[n] = a * kLog2e;
    Ai[n] = 1.f / a;   // ZOH: 1 / A (infinite at A = 0, where zoh_coef takes its series)
    h[n] = (n < N && p.h0) ? p.h0[b * p.sh0[0] + d * p.sh0[1] + n * p.sh0[2]] : 0.f;
  }
  const float bias = p.bias ? p.bias[d] : 0.f;
  const float Dd = p.Dskip ? p.Dskip[d] : 0.f;

  for (int64_t t = 0; t < p.L; ++t) {
    const float uv = to_f32(u[t]);
    const float dt = delta_of<PRECISE>(to_f32(dl[t]), bias, p.softplus);
    const float du = dt * uv;
    float acc = 0.f;
#pragma unroll
    for (int n = 0; n < NB; ++n) {
      if (n < N) {
        const float a = ex2_approx(dt * A2[n]);
        const float bx = p.zoh ? zoh_coef<PRECISE>(dt, dt * A2[n] * kLn2, a, Ai[n]) * uv : du;
        h[n] = fmaf(a, h[n], bx * to_f32(Bm[n * p.sB[1] + t]));
        acc = fmaf(to_f32(Cm[n * p.sC[1] + t]), h[n], acc);
      }
    }
    float out = fmaf(Dd, uv, acc);
    if (z) out *= silu<PRECISE>(to_f32(z[t]));
    y[t] = from_f32<IO>(out);
  }
  if (p.h_last) {
#pragma unroll
    for (int n = 0; n < NB; ++n)
      if (n < N) p.h_last[b * p.shl[0] + d * p.shl[1] + n * p.shl[2]] = h[n];
  }
}

// Complex A ("gitcode", section 3.6): complex state, Abar = exp(Delta A) complex, the real input
// term Delta B u, y = Re(sum_n C h) + D u (then the gate).  h0 / h_last hold (re, im) pairs.
template <typename IO, int NB, bool PRECISE>
__global__ void __launch_bounds__(128) scan_generic_complex_kernel(const ScanProblem p) {
  const int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= p.B * p.D) return;
  const int64_t b = c / p.D, d = c % p.D;
  const int N = (int)p.N;
  const IO* u = static_cast<const IO*>(p.u) + b * p.su[0] + d * p.su[1];
  const IO* dl = static_cast<const IO*>(p.delta) + b * p.sd[0] + d * p.sd[1];
  const IO* z = p.z ? static_cast<const IO*>(p.z) + b * p.sz[0] + d * p.sz[1] : nullptr;
  const IO* Bm = static_cast<const IO*>(p.Bm) + b * p.sB[0];
  const IO* Cm = static_cast<const IO*>(p.Cm) + b * p.sC[0];
  IO* y = static_cast<IO*>(p.y) + b * p.sy[0] + d * p.sy[1];

  float A2[NB], Am[NB], hr[NB], hm[NB];
#pragma unroll
  for (int n = 0; n < NB; ++n) {
    A2[n] = n < N ? p.A[d * p.sA[0] + n * p.sA[1]] * kLog2e : 0.f;
    Am[n] = n < N ? p.Aim[d * p.sA[0] + n * p.sA[1]] : 0.f;
    const int64_t o = b * p.sh0[0] + d * p.sh0[1] + n * p.sh0[2];
    hr[n] = (n < N && p.h0) ? p.h0[o] : 0.f;
    hm[n] = (n < N && p.h0) ? p.h0[o + 1] : 0.f;
  }
  const float bias = p.bias ? p.bias[d] : 0.f;
  const float Dd = p.Dskip ? p.Dskip[d] : 0.f;

  for (int64_t t = 0; t < p.L; ++t) {
    const float uv = to_f32(u[t]);
    const float dt = delta_of<PRECISE>(to_f32(dl[t]), bias, p.softplus);
    const float du = dt * uv;
    float acc = 0.f;
#pragma unroll
    for (int n = 0; n < NB; ++n) {
      if (n < N) {
        const float mag = ex2_approx(dt * A2[n]);
        const float2 cs = cos_sin<PRECISE>(dt * Am[n]);
        const float ar = mag * cs.x, ai = mag * cs.y;
        const float r = fmaf(ar, hr[n], fmaf(-ai, hm[n], du * to_f32(Bm[n * p.sB[1] + t])));
        hm[n] = fmaf(ar, hm[n], ai * hr[n]);
        hr[n] = r;
        acc = fmaf(to_f32(Cm[n * p.sC[1] + t]), hr[n], acc);
      }
    }
    float out = fmaf(Dd, uv, acc);
    if (z) out *= silu<PRECISE>(to_f32(z[t]));
    y[t] = from_f32<IO>(out);
  }
  if (p.h_last) {
#pragma unroll
    for (int n = 0; n < NB; ++n)
      if (n < N) {
        const int64_t o = b * p.shl[0] + d * p.shl[1] + n * p.shl[2];
        p.h_last[o] = hr[n];
        p.h_last[o + 1] = hm[n];
      }
  }
}

template <typename IO, bool PRECISE>
cudaError_t launch_complex(const ScanProblem& p, cudaStream_t s) {
  const int64_t channels = p.B * p.D;
  const dim3 block(128);
  const dim3 grid((unsigned)((channels + 127) / 128));
  if (p.N <= 8) scan_generic_complex_kernel<IO, 8, PRECISE><<<grid, block, 0, s>>>(p);
  else if (p.N <= 16) scan_generic_complex_kernel<IO, 16, PRECISE><<<grid, block, 0, s>>>(p);
  else if (p.N <= 32) scan_generic_complex_kernel<IO, 32, PRECISE><<<grid, block, 0, s>>>(p);
  else scan_generic_complex_kernel<IO, 64, PRECISE><<<grid, block, 0, s>>>(p);
  return cudaGetLastError();
}

template <typename IO, bool PRECISE>
cudaError_t launch_typed(const ScanProblem& p, cudaStream_t s) {
  if (p.cplx) return launch_complex<IO, PRECISE>(p, s);
  const int64_t channels = p.B * p.D;
  const dim3 block(128);
  const dim3 grid((unsigned)((channels + 127) / 128));
  if (p.N <= 4) scan_generic_kernel<IO, 4, PRECISE><<<grid, block, 0, s>>>(p);
  else if (p.N <= 8) scan_generic_kernel<IO, 8, PRECISE><<<grid, block, 0, s>>>(p);
  else if (p.N <= 16) scan_generic_kernel<IO, 16, PRECISE><<<grid, block, 0, s>>>(p);
  else if (p.N <= 32) scan_generic_kernel<IO, 32, PRECISE><<<grid, block, 0, s>>>(p);
  else scan_generic_kernel<IO, 64, PRECISE><<<grid, block, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_scan_generic(const ScanProblem& p, cudaStream_t s) {
  if (p.B * p.D == 0) return cudaSuccess;
  if (p.io == SSM_F32) return launch_typed<float, true>(p, s);
  return launch_typed<__nv_bfloat16, false>(p, s);
}

}  // namespace ssm
