// state_update.cu -- one recurrent (decode) step against a persistent fp32 state.
//
// Constant time and memory per generated token ("gitcode.csdn.net", section 1,
// and section 2: the recurrent mode used for autoregressive inference):
//   h[b,d,n] <- exp(Delta A[d,n]) h[b,d,n] + Delta B[b,n] u[b,d]
//   y[b,d]    = (sum_n C[b,n] h[b,d,n] + D[d] u[b,d]) * silu(z[b,d])
// The step is bound by the state read and write (64 + 64 bytes per channel at
// N = 16).  Q adjacent lanes share one channel, each owning four consecutive
// states, so a warp reads and writes the state as contiguous 512-byte runs;
// the output is reduced over the Q lanes with shuffles.
#include "device_math.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

template <typename IO, int Q, bool PRECISE>
__global__ void __launch_bounds__(256) state_update_kernel(const StepProblem p, const bool vec_state) {
  const int64_t gtid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int q = (int)(gtid % Q);
  const int64_t c = gtid / Q;
  const bool active = c < p.B * p.D;
  const int64_t b = active ? c / p.D : 0, d = active ? c % p.D : 0;
  const int N = (int)p.N;

  float acc = 0.f;
  float uv = 0.f, zv = 0.f;
  if (active) {
    uv = to_f32(static_cast<const IO*>(p.u)[b * p.su[0] + d * p.su[1]]);
    const float dv = to_f32(static_cast<const IO*>(p.delta)[b * p.sd[0] + d * p.sd[1]]);
    if (p.z) zv = to_f32(static_cast<const IO*>(p.z)[b * p.sz[0] + d * p.sz[1]]);
    const float dt = delta_of<PRECISE>(dv, p.bias ? p.bias[d] : 0.f, p.softplus);
    const float du = dt * uv;
    const IO* Bm = static_cast<const IO*>(p.Bm) + b * p.sB[0];
    const IO* Cm = static_cast<const IO*>(p.Cm) + b * p.sC[0];
    float* st = p.state + b * p.sst[0] + d * p.sst[1];
    const int n0 = q * 4;
    float h[4];
    if (vec_state && n0 < N) {
      const float4 v = *reinterpret_cast<const float4*>(st + n0);
      h[0] = v.x; h[1] = v.y; h[2] = v.z; h[3] = v.w;
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) h[i] = (n0 + i < N) ? st[(n0 + i) * p.sst[2]] : 0.f;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int n = n0 + i;
      if (n < N) {
        const float a = ex2_approx(dt * (p.A[d * p.sA[0] + n * p.sA[1]] * kLog2e));
        h[i] = fmaf(a, h[i], du * to_f32(Bm[n * p.sB[1]]));
        acc = fmaf(to_f32(Cm[n * p.sC[1]]), h[i], acc);
      }
    }
    if (vec_state && n0 < N) {
      *reinterpret_cast<float4*>(st + n0) = make_float4(h[0], h[1], h[2], h[3]);
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (n0 + i < N) st[(n0 + i) * p.sst[2]] = h[i];
    }
  }
#pragma unroll
  for (int off = 1; off < Q; off <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (active && q == 0) {
    float out = fmaf(p.Dskip ? p.Dskip[d] : 0.f, uv, acc);
    if (p.z) out *= silu<PRECISE>(zv);
    static_cast<IO*>(p.y)[b * p.sy[0] + d * p.sy[1]] = from_f32<IO>(out);
  }
}

template <typename IO, bool PRECISE>
cudaError_t launch_typed(const StepProblem& p, cudaStream_t s) {
  // vectorised state access: contiguous states, 16-byte aligned rows, whole quads
  const bool vec = p.sst[2] == 1 && (p.N % 4 == 0) && (p.sst[0] % 4 == 0) && (p.sst[1] % 4 == 0) &&
                   (reinterpret_cast<uintptr_t>(p.state) % 16 == 0);
  const int quads = (int)((p.N + 3) / 4);
  int Q = 1;
  while (Q < quads) Q <<= 1;
  const int64_t threads = p.B * p.D * Q;
  const dim3 block(256);
  const dim3 grid((unsigned)((threads + 255) / 256));
  switch (Q) {
    case 1: state_update_kernel<IO, 1, PRECISE><<<grid, block, 0, s>>>(p, vec); break;
    case 2: state_update_kernel<IO, 2, PRECISE><<<grid, block, 0, s>>>(p, vec); break;
    case 4: state_update_kernel<IO, 4, PRECISE><<<grid, block, 0, s>>>(p, vec); break;
    case 8: state_update_kernel<IO, 8, PRECISE><<<grid, block, 0, s>>>(p, vec); break;
    default: state_update_kernel<IO, 16, PRECISE><<<grid, block, 0, s>>>(p, vec); break;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_state_update(const StepProblem& p, cudaStream_t s) {
  if (p.B * p.D == 0) return cudaSuccess;
  if (p.io == SSM_F32) return launch_typed<float, true>(p, s);
  return launch_typed<__nv_bfloat16, false>(p, s);
}

}  // namespace ssm
