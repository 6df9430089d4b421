// scan_bwd.cu -- gradients of the selective scan, for training.
//
// What it computes: the reverse-mode derivative of the forward recurrence
// (see scan_tiled.cu) through the chain rule,
//   Delta_t = softplus(s_t), s_t = delta_t + bias      dDelta/ds = sigmoid(s_t)
//   Abar_t[n] = exp(Delta_t A[n]),  h_t = Abar_t h_{t-1} + Delta_t B_t u_t
//   p_t = sum_n C_t[n] h_t[n] + D u_t,  y_t = p_t silu(z_t)
// with the adjoint lambda_t[n] = dL/dh_t[n] = (dy_t silu(z_t)) C_t[n]
// + Abar_{t+1}[n] lambda_{t+1}[n], run backwards in time.  As in section 3.3.2
// of the Mamba paper ("Mamba paper translation", gitcode.csdn.net) the forward
// states are recomputed, not stored: a forward sweep keeps one checkpoint of
// the state every SEG steps, and the reverse sweep recomputes each SEG-step
// segment from its checkpoint before running the adjoint through it.
//
// Design: one warp per CTA covers 32 channels of one batch row, one channel per
// lane, all (up to 16) states of a channel in that lane's registers.
//   * B_t and C_t of a segment are staged in shared memory by the lanes and
//     read as warp-wide broadcasts;
//   * the recomputed states of a segment go to shared memory, laid out
//     [step][4 states][lane] as 16-byte pieces so that every access is
//     conflict-free;
//   * dB_t[n] and dC_t[n] are sums over the channels: per step each lane
//     writes its 32 contributions to a row of a shared 32 x 32 block, every
//     lane then sums one column, and one atomic add per (t, n) per warp goes
//     to global memory;
//   * dA, dD and the Delta-bias gradient accumulate in registers over the
//     whole sequence and are added atomically at the end (several batch rows
//     share a channel).
#include <algorithm>

#include "device_math.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int SEG = SSM_BWD_SEGMENT;   // steps per checkpoint
constexpr int NPL = 16;                // states per lane
constexpr float kLn2 = 0.69314718055994531f;

template <bool PRECISE>
__device__ __forceinline__ float sigmoid_f(float v) {
  if (PRECISE) return 1.f / (1.f + expf(-v));
  return rcp_approx(1.f + ex2_approx(-v * kLog2e));
}

template <typename IO>
__device__ __forceinline__ float ld(const void* base, int64_t off) {
  return to_f32(static_cast<const IO*>(base)[off]);
}

template <typename IO>
__device__ __forceinline__ void st(void* base, int64_t off, float v) {
  static_cast<IO*>(base)[off] = from_f32<IO>(v);
}

// Zeroes the summed gradients (dA, dB, dC, dD, the Delta-bias gradient).
__global__ void __launch_bounds__(256) bwd_zero_kernel(const BwdProblem p) {
  const ScanProblem& f = p.f;
  const int64_t nA = f.D * f.N, nBC = p.bc_rows * f.N * f.L;
  const int64_t nD = f.D;
  const int64_t total = nA + 2 * nBC + 2 * nD;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    int64_t k = i;
    if (k < nA) { p.dA[k] = 0.f; continue; }
    k -= nA;
    if (k < 2 * nBC) {
      float* g = k < nBC ? p.dB : p.dC;
      const int64_t* sg = k < nBC ? p.sdB : p.sdC;
      const int64_t j = k < nBC ? k : k - nBC;
      const int64_t t = j % f.L, n = (j / f.L) % f.N, b = j / (f.L * f.N);
      g[b * sg[0] + n * sg[1] + t * sg[2]] = 0.f;
      continue;
    }
    k -= 2 * nBC;
    if (k < nD) { if (p.dD) p.dD[k] = 0.f; continue; }
    k -= nD;
    if (p.dbias) p.dbias[k] = 0.f;
  }
}

template <typename IO, bool PRECISE>
__global__ void __launch_bounds__(32) scan_bwd_kernel(const BwdProblem p) {
  __shared__ float4 hist[(SEG + 1) * 4 * 32];   // [row][state quad][lane]; row 0 = state before the segment
  __shared__ float bcs[SEG][32];                // [t][B_t[0..15] | C_t[0..15]]
  __shared__ __align__(16) float red[32][36];   // per-step transpose block for the channel sums (16-byte rows)
  const ScanProblem& f = p.f;
  const int lane = threadIdx.x;
  const int64_t b = blockIdx.y;
  const int64_t d = (int64_t)blockIdx.x * 32 + lane;
  const bool valid = d < f.D;
  const int N = (int)f.N;
  const int64_t L = f.L;
  const int64_t c = b * f.D + (valid ? d : 0);

  float A2[NPL], h[NPL];
#pragma unroll
  for (int n = 0; n < NPL; ++n) {
    A2[n] = (valid && n < N) ? f.A[d * f.sA[0] + n * f.sA[1]] * kLog2e : 0.f;
    h[n] = (valid && n < N && f.h0) ? f.h0[b * f.sh0[0] + d * f.sh0[1] + n * f.sh0[2]] : 0.f;
  }
  const float bias = (valid && f.bias) ? f.bias[d] : 0.f;
  const float Dd = (valid && f.Dskip) ? f.Dskip[d] : 0.f;
  const int64_t ou = b * f.su[0] + d * f.su[1], odl = b * f.sd[0] + d * f.sd[1], oz = b * f.sz[0] + d * f.sz[1];
  const int64_t ody = b * p.sdy[0] + d * p.sdy[1];
  float4* ck = reinterpret_cast<float4*>(p.ckpt + c * p.nseg * NPL);

  // B_t and C_t of segment `seg` into shared memory (lane j: row j % 16 of B for j < 16, of C otherwise)
  auto stage_bc = [&](int64_t seg) {
    __syncwarp();
    const int n = lane & 15;
    const void* base = lane < 16 ? f.Bm : f.Cm;
    const int64_t* sb = lane < 16 ? f.sB : f.sC;
    const int64_t t0 = seg * SEG;
#pragma unroll
    for (int t = 0; t < SEG; ++t)
      bcs[t][lane] = (n < N && t0 + t < L) ? ld<IO>(base, b * sb[0] + n * sb[1] + t0 + t) : 0.f;
    __syncwarp();
  };

  // ---- forward sweep: a checkpoint of the state before every segment (unless the
  // tiled forward kernel has written them already) ----
  for (int64_t seg = 0; p.sweep && seg < p.nseg; ++seg) {
    stage_bc(seg);
    if (valid) {
#pragma unroll
      for (int q = 0; q < 4; ++q) ck[seg * 4 + q] = make_float4(h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]);
    }
    const int64_t t0 = seg * SEG;
#pragma unroll
    for (int t = 0; t < SEG; ++t) {
      if (t0 + t >= L) break;
      const float dt = valid ? delta_of<PRECISE>(ld<IO>(f.delta, odl + t0 + t), bias, f.softplus) : 0.f;
      const float du = valid ? dt * ld<IO>(f.u, ou + t0 + t) : 0.f;
#pragma unroll
      for (int n = 0; n < NPL; ++n) h[n] = fmaf(ex2_approx(dt * A2[n]), h[n], du * bcs[t][n]);
    }
  }

  // ---- reverse sweep ----
  float lam[NPL], dA[NPL];
#pragma unroll
  for (int n = 0; n < NPL; ++n) {
    lam[n] = (valid && n < N && p.dhl) ? p.dhl[b * p.sdhl[0] + d * p.sdhl[1] + n * p.sdhl[2]] : 0.f;
    dA[n] = 0.f;
  }
  float dD = 0.f, dbias = 0.f;
  for (int64_t seg = p.nseg - 1; seg >= 0; --seg) {
    stage_bc(seg);
    const int64_t t0 = seg * SEG;
    const int steps = L - t0 < SEG ? (int)(L - t0) : SEG;
    // recompute the segment's states from its checkpoint
    if (valid) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 v = ck[seg * 4 + q];
        h[4 * q] = v.x; h[4 * q + 1] = v.y; h[4 * q + 2] = v.z; h[4 * q + 3] = v.w;
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) hist[q * 32 + lane] = make_float4(h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]);
    float dts[SEG], us[SEG], yts[SEG], ss[SEG];
#pragma unroll
    for (int t = 0; t < SEG; ++t) {
      dts[t] = 0.f; us[t] = 0.f; yts[t] = 0.f; ss[t] = 0.f;
      if (t >= steps) continue;
      const int64_t tg = t0 + t;
      float uv = 0.f, s = 0.f, dyv = 0.f, zv = 0.f;
      if (valid) {
        uv = ld<IO>(f.u, ou + tg);
        s = ld<IO>(f.delta, odl + tg) + bias;
        dyv = ld<IO>(p.dy, ody + tg);
        if (f.z) zv = ld<IO>(f.z, oz + tg);
      }
      const float dt = valid ? (f.softplus ? softplus<PRECISE>(s) : s) : 0.f;
      const float du = dt * uv;
      float acc = 0.f;
#pragma unroll
      for (int n = 0; n < NPL; ++n) {
        h[n] = fmaf(ex2_approx(dt * A2[n]), h[n], du * bcs[t][n]);
        acc = fmaf(bcs[t][16 + n], h[n], acc);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q)
        hist[((t + 1) * 4 + q) * 32 + lane] = make_float4(h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]);
      float yt = dyv;
      if (f.z) {
        const float pre = fmaf(Dd, uv, acc);
        const float sg = sigmoid_f<PRECISE>(zv);
        yt = dyv * zv * sg;
        if (valid) st<IO>(p.dz, b * p.sdz[0] + d * p.sdz[1] + tg, dyv * pre * sg * fmaf(zv, 1.f - sg, 1.f));
      }
      dts[t] = dt; us[t] = uv; yts[t] = yt; ss[t] = s;
    }
    __syncwarp();
    // the adjoint through the segment, last step first
#pragma unroll
    for (int t = SEG - 1; t >= 0; --t) {
      if (t >= steps) continue;
      const int64_t tg = t0 + t;
      const float dt = dts[t], uv = us[t], yt = yts[t], du = dt * uv;
      float sq = 0.f, sb = 0.f;
      float vb[NPL], vc[NPL];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 hp4 = hist[(t * 4 + q) * 32 + lane];
        const float4 ht4 = hist[((t + 1) * 4 + q) * 32 + lane];
        const float hp[4] = {hp4.x, hp4.y, hp4.z, hp4.w};
        const float ht[4] = {ht4.x, ht4.y, ht4.z, ht4.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int n = 4 * q + i;
          const float l = fmaf(yt, bcs[t][16 + n], lam[n]);   // lambda_t[n]
          const float a = ex2_approx(dt * A2[n]);
          const float qv = l * hp[i] * a;
          dA[n] = fmaf(qv, dt, dA[n]);
          sq = fmaf(qv, A2[n], sq);
          sb = fmaf(l, bcs[t][n], sb);
          vb[n] = l * du;
          vc[n] = yt * ht[i];
          lam[n] = l * a;
        }
      }
      if (valid) {
        const float dDelta = fmaf(sq, kLn2, sb * uv);
        st<IO>(p.du, b * p.sdu[0] + d * p.sdu[1] + tg, fmaf(sb, dt, yt * Dd));
        const float dd = f.softplus ? dDelta * sigmoid_f<PRECISE>(ss[t]) : dDelta;
        st<IO>(p.ddelta, b * p.sdd[0] + d * p.sdd[1] + tg, dd);
        dbias += dd;
        dD = fmaf(yt, uv, dD);
      }
      // channel sums of dB_t[n], dC_t[n]: transpose through shared memory
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        *reinterpret_cast<float4*>(&red[lane][4 * q]) = make_float4(vb[4 * q], vb[4 * q + 1], vb[4 * q + 2], vb[4 * q + 3]);
        *reinterpret_cast<float4*>(&red[lane][16 + 4 * q]) =
            make_float4(vc[4 * q], vc[4 * q + 1], vc[4 * q + 2], vc[4 * q + 3]);
      }
      __syncwarp();
      float sum = 0.f;
#pragma unroll
      for (int r = 0; r < 32; ++r) sum += red[r][lane];
      __syncwarp();
      const int n = lane & 15;
      if (n < N) {
        if (lane < 16) atomicAdd(p.dB + b * p.sdB[0] + n * p.sdB[1] + tg * p.sdB[2], sum);
        else atomicAdd(p.dC + b * p.sdC[0] + n * p.sdC[1] + tg * p.sdC[2], sum);
      }
    }
  }
  if (!valid) return;
  // ---- the summed parameter gradients and dh0 ----
#pragma unroll
  for (int n = 0; n < NPL; ++n) {
    if (n >= N) break;
    atomicAdd(p.dA + d * N + n, dA[n]);
    if (p.dh0) p.dh0[b * p.sdh0[0] + d * p.sdh0[1] + n * p.sdh0[2]] = lam[n];
  }
  if (p.dD) atomicAdd(p.dD + d, dD);
  if (p.dbias) atomicAdd(p.dbias + d, dbias);
}

template <typename IO, bool PRECISE>
cudaError_t launch_typed(const BwdProblem& p, int sms, cudaStream_t s) {
  const int64_t zero_total = p.f.D * p.f.N + 2 * p.bc_rows * p.f.N * p.f.L + 2 * p.f.D;
  const int zb = (int)std::min<int64_t>((zero_total + 255) / 256, (int64_t)sms * 8);
  bwd_zero_kernel<<<zb, 256, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)((p.f.D + 31) / 32), (unsigned)p.f.B);
  scan_bwd_kernel<IO, PRECISE><<<grid, 32, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_scan_bwd(const BwdProblem& p, int sms, cudaStream_t s) {
  if (p.f.io == SSM_F32) return launch_typed<float, true>(p, sms, s);
  return launch_typed<__nv_bfloat16, false>(p, sms, s);
}

}  // namespace ssm
