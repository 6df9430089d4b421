// scan_bwd.cu -- gradients of the selective scan, for training.
//
// What it computes: the reverse-mode derivative of the forward recurrence
// (see scan_tiled.cu) through the chain rule,
//   Delta_t = softplus(s_t), s_t = delta_t + bias      dDelta/ds = sigmoid(s_t)
//   Abar_t[n] = exp(Delta_t A[n]),  h_t = Abar_t h_{t-1} + g_t B_t u_t
// with the input coefficient g = Delta (Euler) or the exact zero-order hold
// g = (Abar - 1) / A ("Mamba and state space models", docs.ifdog.com, section
// "Discretisation"), whose partial derivatives are dg/dDelta = Abar and
// dg/dA = Delta^2 psi(Delta A), psi(x) = (x e^x - (e^x - 1)) / x^2,
//   p_t = sum_n C_t[n] h_t[n] + D u_t,  y_t = p_t silu(z_t)
// with the adjoint lambda_t[n] = dL/dh_t[n] = (dy_t silu(z_t)) C_t[n]
// + Abar_{t+1}[n] lambda_{t+1}[n], run backwards in time.  As in section 3.3.2
// of the Mamba paper ("Mamba paper translation", gitcode.csdn.net) the forward
// states are recomputed, not stored: one checkpoint of the state every SEG
// steps comes from the tiled forward kernel's checkpoint mode (or, for layouts
// it cannot take, from a forward sweep in this kernel), and the reverse sweep
// recomputes each SEG-step segment from its checkpoint before running the
// adjoint through it.
//
// Design: one warp per CTA covers 16 channels of one batch row, two lanes per
// channel (8 states each, as f32x2 pairs), so that twice as many warps share
// the work; the sums over a channel's states take one shuffle between its two
// lanes.
//   * A segment's inputs of a channel arrive as one 128-bit load per tensor
//     when the rows allow it (L1-cached: a 128-byte line holds eight
//     consecutive segments of a row);
//   * B_t and C_t of a segment are staged in shared memory, one 128-bit load
//     per row, and read as warp-wide broadcasts;
//   * the recomputed states of a segment go to shared memory, laid out
//     [step][half of the lane's states][lane] as 16-byte pieces;
//   * dB_t[n] and dC_t[n] are sums over the channels: per step each lane
//     writes its 16 contributions to its channel's row of a shared 16 x 36
//     block and every lane sums one column; a segment's 8 sums per lane leave
//     as two float4 atomic adds;
//   * du, ddelta, dz of a segment leave as one 16-byte store per row;
//   * dA, dD and the Delta-bias gradient accumulate in registers over the
//     whole sequence and are added atomically at the end (several batch rows
//     share a channel).
#include <algorithm>

#include "device_math.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int SEG = SSM_BWD_SEGMENT;   // steps per checkpoint

// The A-derivative of the exact-ZOH coefficient g = (e^x - 1) / A (x = Delta A, a = e^x) for a pair of
// states: dg/dA = (Delta a - g) / A.  That difference cancels for small |x|, so below |x| = 1/4 it is
// Delta^2 psi(x), psi(x) = sum_{k>=1} k x^(k-1) / (k+1)! = 1/2 + x/3 + x^2/8 + x^3/30 + x^4/144
// + x^5/840 + x^6/5760 + ... (the next term is below 3e-9 relative there); above it the difference
// keeps all but a few bits.  Both forms are evaluated on packed f32x2 operations and selected per
// state, so the lanes of a warp do not diverge.
__device__ __forceinline__ float2 zoh_dg_dA2(float dt, float2 x, float2 a, float2 g, float2 inv_a) {
  const float2 d2 = make_float2(dt, dt);
  float2 psi = __ffma2_rn(x, make_float2(1.7361111111111111e-04f, 1.7361111111111111e-04f),   // 1/5760
                          make_float2(1.1904761904761905e-03f, 1.1904761904761905e-03f));      // 1/840
  psi = __ffma2_rn(psi, x, make_float2(6.9444444444444444e-03f, 6.9444444444444444e-03f));     // 1/144
  psi = __ffma2_rn(psi, x, make_float2(3.3333333333333333e-02f, 3.3333333333333333e-02f));     // 1/30
  psi = __ffma2_rn(psi, x, make_float2(0.125f, 0.125f));                                       // 1/8
  psi = __ffma2_rn(psi, x, make_float2(3.3333333333333333e-01f, 3.3333333333333333e-01f));     // 1/3
  psi = __ffma2_rn(psi, x, make_float2(0.5f, 0.5f));
  const float2 small = __fmul2_rn(__fmul2_rn(d2, d2), psi);
  const float2 large = __fmul2_rn(__ffma2_rn(d2, a, make_float2(-g.x, -g.y)), inv_a);
  return make_float2(fabsf(x.x) < 0.25f ? small.x : large.x, fabsf(x.y) < 0.25f ? small.y : large.y);
}

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

// 128-bit read-only load of segment data.  It is L1-cached (a 128-byte line
// holds eight segments of a row, read one after another, and the two lanes of
// a channel read the same piece) and asks L2 for 256 bytes on a miss.
__device__ __forceinline__ uint4 ld_seg16(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

// SEG steps of one row starting at `ptr` (time stride 1) as fp32: one or two
// 128-bit loads when the row is 16-byte aligned and the segment is whole,
// element loads otherwise.
template <typename IO>
__device__ __forceinline__ void load_seg(const void* base, int64_t off, bool vec, int steps, float (&out)[SEG]) {
  const IO* ptr = static_cast<const IO*>(base) + off;
  if (vec) {
    if (sizeof(IO) == 2) {
      float f[8];
      unpack16(ld_seg16(ptr), f);
#pragma unroll
      for (int t = 0; t < SEG; ++t) out[t] = f[t];
    } else {
      float f0[4], f1[4];
      unpack16(ld_seg16(ptr), f0);
      unpack16(ld_seg16(ptr + 4), f1);
#pragma unroll
      for (int t = 0; t < 4; ++t) { out[t] = f0[t]; out[t + 4] = f1[t]; }
    }
  } else {
#pragma unroll
    for (int t = 0; t < SEG; ++t) out[t] = t < steps ? to_f32(ptr[t]) : 0.f;
  }
}

// The inverse of load_seg: SEG values to a 16-byte aligned row piece.
template <typename IO>
__device__ __forceinline__ void store_seg(void* base, int64_t off, const float (&v)[SEG]) {
  IO* ptr = static_cast<IO*>(base) + off;
  if (sizeof(IO) == 2) {
    float f[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) f[t] = v[t];
    stg_v4(ptr, pack16(f));
  } else {
    float f0[4] = {v[0], v[1], v[2], v[3]}, f1[4] = {v[4], v[5], v[6], v[7]};
    stg_v4(ptr, pack16(f0));
    stg_v4(ptr + 4, pack16(f1));
  }
}

__device__ __forceinline__ float2 f2(float v) { return make_float2(v, v); }

// One warp per CTA: 32 / LPC channels of one batch row, LPC lanes per channel
// (lanes c, c + 32 / LPC, ...), each lane holding 8 of the channel's states as
// four f32x2 pairs (LPC = 2, 4, 8 for N up to 16, 32, 64).  Sums over the
// states (the C contraction, dDelta, du) take log2(LPC) shuffles between the
// lanes of a channel.
template <typename IO, bool PRECISE, bool ZOH, int LPC>
__global__ void __launch_bounds__(32) scan_bwd_kernel(const BwdProblem p) {
  constexpr int CHW = 32 / LPC;                      // channels per warp
  constexpr int NP = 8 * LPC;                        // states per channel, padded
  constexpr int NCOL = 2 * NP / 32;                  // dB / dC columns each lane sums
  __shared__ float4 hist[(SEG + 1) * 2 * 32];        // [row][half of the lane's 8 states][lane]
  __shared__ __align__(16) float bcs[SEG][2 * NP];   // [t][B_t[0..NP) | C_t[0..NP)]
  __shared__ __align__(16) float red[CHW][2 * NP + 4];   // [channel][dB_t[0..NP) | dC_t[0..NP)]
  const ScanProblem& f = p.f;
  const int lane = threadIdx.x;
  const int ch = lane % CHW, g = lane / CHW;         // channel within the warp, group of 8 of its states
  const int64_t b = blockIdx.y;
  const int64_t d = (int64_t)blockIdx.x * CHW + ch;
  const bool valid = d < f.D;
  const bool lead = g == 0;                          // writes the channel's per-step outputs
  const int N = (int)f.N;
  const int64_t L = f.L;
  const int64_t c = b * f.D + (valid ? d : 0);

  float2 A2[4], h[4], Ai[4];   // Ai: 1 / A, for the exact-ZOH coefficient
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    float av[2], hv[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int n = g * 8 + 2 * q + e;
      av[e] = (valid && n < N) ? f.A[d * f.sA[0] + n * f.sA[1]] * kLog2e : 0.f;
      hv[e] = (valid && n < N && f.h0) ? f.h0[b * f.sh0[0] + d * f.sh0[1] + n * f.sh0[2]] : 0.f;
    }
    A2[q] = make_float2(av[0], av[1]);
    // infinite at A = 0, where the coefficient takes its series
    Ai[q] = ZOH ? make_float2(kLog2e / av[0], kLog2e / av[1]) : make_float2(0.f, 0.f);
    h[q] = make_float2(hv[0], hv[1]);
  }
  const float bias = (valid && f.bias) ? f.bias[d] : 0.f;
  const float Dd = (valid && f.Dskip) ? f.Dskip[d] : 0.f;
  const int64_t ou = b * f.su[0] + d * f.su[1], odl = b * f.sd[0] + d * f.sd[1], oz = b * f.sz[0] + d * f.sz[1];
  const int64_t ody = b * p.sdy[0] + d * p.sdy[1];
  // this lane's 8 floats of each NP-float checkpoint record
  float4* ck = reinterpret_cast<float4*>(p.ckpt + c * p.nseg * NP + g * 8);
  constexpr int CKQ = NP / 4;                        // float4 pieces per checkpoint record
  // the sum of a per-lane value over the LPC lanes of this lane's channel
  auto channel_sum = [](float v) {
#pragma unroll
    for (int o = CHW; o < 32; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
  };

  // rows j < NP of the staging block are B's, the others C's; lane l stages rows l, l + 32, ...
  auto stage_bc = [&](int64_t seg) {
    __syncwarp();
    const int64_t t0 = seg * SEG;
    const int steps = L - t0 < SEG ? (int)(L - t0) : SEG;
#pragma unroll
    for (int k = 0; k < NCOL; ++k) {
      const int row = lane + 32 * k;
      const int n = row % NP;
      const void* base = row < NP ? f.Bm : f.Cm;
      const int64_t* sb = row < NP ? f.sB : f.sC;
      float v[SEG];
      if (n < N) {
        load_seg<IO>(base, b * sb[0] + n * sb[1] + t0, p.vecbc && steps == SEG, steps, v);
      } else {
#pragma unroll
        for (int t = 0; t < SEG; ++t) v[t] = 0.f;
      }
#pragma unroll
      for (int t = 0; t < SEG; ++t) bcs[t][row] = v[t];
    }
    __syncwarp();
  };
  auto bpair = [&](int t, int q) { return *reinterpret_cast<const float2*>(&bcs[t][g * 8 + 2 * q]); };
  auto cpair = [&](int t, int q) { return *reinterpret_cast<const float2*>(&bcs[t][NP + g * 8 + 2 * q]); };
  auto abar = [&](float dt, int q) {
    const float2 x = __fmul2_rn(f2(dt), A2[q]);
    return make_float2(ex2_approx(x.x), ex2_approx(x.y));
  };
  // Delta A (natural base) of a pair of states
  auto dtA = [&](float dt, int q) { return __fmul2_rn(__fmul2_rn(f2(dt), A2[q]), f2(kLn2)); };
  // the exact-ZOH input coefficient g of a pair of states, as the forward kernels compute it
  auto zoh_g = [&](float dt, int q, float2 a) {
    const float2 x = dtA(dt, q);
    if (PRECISE) return make_float2(zoh_coef<true>(dt, x.x, a.x, Ai[q].x), zoh_coef<true>(dt, x.y, a.y, Ai[q].y));
    return zoh_coef2_fast(f2(dt), x, a, Ai[q]);
  };
  // the input term of a pair of states: Delta u B (Euler) or g u B (exact ZOH)
  auto input = [&](float dt, float uv, int q, float2 a, float2 bq) {
    if constexpr (ZOH) return __fmul2_rn(__fmul2_rn(zoh_g(dt, q, a), f2(uv)), bq);
    return __fmul2_rn(f2(dt * uv), bq);
  };

  // ---- forward sweep: the checkpoints, unless the tiled forward kernel wrote them ----
  for (int64_t seg = 0; p.sweep && seg < p.nseg; ++seg) {
    stage_bc(seg);
    if (valid) {
      ck[seg * CKQ] = make_float4(h[0].x, h[0].y, h[1].x, h[1].y);
      ck[seg * CKQ + 1] = make_float4(h[2].x, h[2].y, h[3].x, h[3].y);
    }
    const int64_t t0 = seg * SEG;
#pragma unroll
    for (int t = 0; t < SEG; ++t) {
      if (t0 + t >= L) break;
      const float dt = valid ? delta_of<PRECISE>(ld<IO>(f.delta, odl + t0 + t), bias, f.softplus) : 0.f;
      const float uv = valid ? ld<IO>(f.u, ou + t0 + t) : 0.f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 a = abar(dt, q);
        h[q] = __ffma2_rn(a, h[q], input(dt, uv, q, a, bpair(t, q)));
      }
    }
  }

  // ---- reverse sweep ----
  float2 lam[4], dA[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    float lv[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int n = g * 8 + 2 * q + e;
      lv[e] = (valid && n < N && p.dhl) ? p.dhl[b * p.sdhl[0] + d * p.sdhl[1] + n * p.sdhl[2]] : 0.f;
    }
    lam[q] = make_float2(lv[0], lv[1]);
    dA[q] = make_float2(0.f, 0.f);
  }
  float dD = 0.f, dbias = 0.f;
  for (int64_t seg = p.nseg - 1; seg >= 0; --seg) {
    stage_bc(seg);
    const int64_t t0 = seg * SEG;
    const int steps = L - t0 < SEG ? (int)(L - t0) : SEG;
    if (valid) {
      const float4 v0 = ck[seg * CKQ], v1 = ck[seg * CKQ + 1];
      h[0] = make_float2(v0.x, v0.y); h[1] = make_float2(v0.z, v0.w);
      h[2] = make_float2(v1.x, v1.y); h[3] = make_float2(v1.z, v1.w);
    }
    hist[lane] = make_float4(h[0].x, h[0].y, h[1].x, h[1].y);
    hist[32 + lane] = make_float4(h[2].x, h[2].y, h[3].x, h[3].y);
    // the segment's inputs of this channel
    float us[SEG], ss[SEG], zs[SEG], dys[SEG];
    const bool vec = valid && p.vec && steps == SEG;
    if (valid) {
      load_seg<IO>(f.u, ou + t0, vec, steps, us);
      load_seg<IO>(f.delta, odl + t0, vec, steps, ss);
      load_seg<IO>(p.dy, ody + t0, vec, steps, dys);
      if (f.z) load_seg<IO>(f.z, oz + t0, vec, steps, zs);
    }
    float dts[SEG], yts[SEG];
    float dzo[SEG], duo[SEG], ddo[SEG], sums[NCOL][SEG];   // the segment's outputs, written once it is done
    // recompute the segment's states from its checkpoint
#pragma unroll
    for (int t = 0; t < SEG; ++t) {
      dts[t] = 0.f; yts[t] = 0.f;
      if (t >= steps) continue;
      const float uv = valid ? us[t] : 0.f;
      const float s = valid ? ss[t] + bias : 0.f;
      ss[t] = s;
      const float dt = valid ? (f.softplus ? softplus<PRECISE>(s) : s) : 0.f;
      float2 acc = make_float2(0.f, 0.f);
      if constexpr (ZOH) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 a = abar(dt, q);
          h[q] = __ffma2_rn(a, h[q], input(dt, uv, q, a, bpair(t, q)));
          acc = __ffma2_rn(cpair(t, q), h[q], acc);
        }
      } else {
        const float du = dt * uv;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          h[q] = __ffma2_rn(abar(dt, q), h[q], __fmul2_rn(f2(du), bpair(t, q)));
          acc = __ffma2_rn(cpair(t, q), h[q], acc);
        }
      }
      hist[((t + 1) * 2) * 32 + lane] = make_float4(h[0].x, h[0].y, h[1].x, h[1].y);
      hist[((t + 1) * 2 + 1) * 32 + lane] = make_float4(h[2].x, h[2].y, h[3].x, h[3].y);
      const float part = channel_sum(acc.x + acc.y);   // over all the channel's states
      const float dyv = valid ? dys[t] : 0.f;
      float yt = dyv;
      if (f.z) {
        const float zv = valid ? zs[t] : 0.f;
        const float sg = sigmoid_f<PRECISE>(zv);
        yt = dyv * zv * sg;
        if (valid && lead)
          dzo[t] = dyv * fmaf(Dd, uv, part) * sg * fmaf(zv, 1.f - sg, 1.f);
      }
      dts[t] = dt; yts[t] = yt;
    }
    __syncwarp();
    // the adjoint through the segment, last step first; h_t of a step is h_{t-1} of the one after
    // it, so each step reads one state from shared memory
    float4 ht0 = make_float4(h[0].x, h[0].y, h[1].x, h[1].y), ht1 = make_float4(h[2].x, h[2].y, h[3].x, h[3].y);
#pragma unroll
    for (int t = SEG - 1; t >= 0; --t) {
      if (t >= steps) continue;   // (the first step taken is steps-1, whose h_t is the recompute's last h)
      const int64_t tg = t0 + t;
      const float dt = dts[t], yt = yts[t];
      const float uv = valid ? us[t] : 0.f;
      const float du = dt * uv;
      const float4 hp0 = hist[(t * 2) * 32 + lane], hp1 = hist[(t * 2 + 1) * 32 + lane];
      const float2 hp[4] = {make_float2(hp0.x, hp0.y), make_float2(hp0.z, hp0.w), make_float2(hp1.x, hp1.y),
                            make_float2(hp1.z, hp1.w)};
      const float2 ht[4] = {make_float2(ht0.x, ht0.y), make_float2(ht0.z, ht0.w), make_float2(ht1.x, ht1.y),
                            make_float2(ht1.z, ht1.w)};
      float2 vb[4], vc[4];
      float sqs, sbs, sgs = 0.f;
      if constexpr (ZOH) {
        // sq: sum_n lambda h_{t-1} Abar A log2(e); sb: sum_n Abar lambda B (dg/dDelta = Abar);
        // sg: sum_n lambda g B
        float2 sq = make_float2(0.f, 0.f), sb = make_float2(0.f, 0.f), sg = make_float2(0.f, 0.f);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 l = __ffma2_rn(f2(yt), cpair(t, q), lam[q]);   // lambda_t
          const float2 a = abar(dt, q);
          const float2 qv = __fmul2_rn(__fmul2_rn(l, hp[q]), a);
          const float2 ln = __fmul2_rn(l, a);                         // lambda carried to step t - 1
          const float2 x = dtA(dt, q);
          const float2 g = zoh_g(dt, q, a);
          const float2 w = zoh_dg_dA2(dt, x, a, g, Ai[q]);
          const float2 lb = __fmul2_rn(l, bpair(t, q));
          dA[q] = __ffma2_rn(qv, f2(dt), __ffma2_rn(__fmul2_rn(lb, f2(uv)), w, dA[q]));
          sq = __ffma2_rn(qv, A2[q], sq);
          sb = __ffma2_rn(ln, bpair(t, q), sb);
          sg = __ffma2_rn(lb, g, sg);
          vb[q] = __fmul2_rn(__fmul2_rn(l, g), f2(uv));
          vc[q] = __fmul2_rn(f2(yt), ht[q]);
          lam[q] = ln;
        }
        sqs = sq.x + sq.y;
        sbs = sb.x + sb.y;
        sgs = channel_sum(sg.x + sg.y);
      } else {
        float2 sq = make_float2(0.f, 0.f), sb = make_float2(0.f, 0.f);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 l = __ffma2_rn(f2(yt), cpair(t, q), lam[q]);   // lambda_t
          const float2 a = abar(dt, q);
          const float2 qv = __fmul2_rn(__fmul2_rn(l, hp[q]), a);
          dA[q] = __ffma2_rn(qv, f2(dt), dA[q]);
          sq = __ffma2_rn(qv, A2[q], sq);
          sb = __ffma2_rn(l, bpair(t, q), sb);
          vb[q] = __fmul2_rn(l, f2(du));
          vc[q] = __fmul2_rn(f2(yt), ht[q]);
          lam[q] = __fmul2_rn(l, a);
        }
        sqs = sq.x + sq.y;
        sbs = sb.x + sb.y;
      }
      ht0 = hp0;
      ht1 = hp1;
      sqs = channel_sum(sqs);
      sbs = channel_sum(sbs);
      if (valid && lead) {
        const float dDelta = fmaf(sqs, kLn2, sbs * uv);
        duo[t] = ZOH ? sgs + yt * Dd : fmaf(sbs, dt, yt * Dd);
        const float dd = f.softplus ? dDelta * sigmoid_f<PRECISE>(ss[t]) : dDelta;
        ddo[t] = dd;
        dbias += dd;
        dD = fmaf(yt, uv, dD);
      }
      // channel sums of dB_t[n] and dC_t[n]: transpose through shared memory
      *reinterpret_cast<float4*>(&red[ch][g * 8]) = make_float4(vb[0].x, vb[0].y, vb[1].x, vb[1].y);
      *reinterpret_cast<float4*>(&red[ch][g * 8 + 4]) = make_float4(vb[2].x, vb[2].y, vb[3].x, vb[3].y);
      *reinterpret_cast<float4*>(&red[ch][NP + g * 8]) = make_float4(vc[0].x, vc[0].y, vc[1].x, vc[1].y);
      *reinterpret_cast<float4*>(&red[ch][NP + g * 8 + 4]) = make_float4(vc[2].x, vc[2].y, vc[3].x, vc[3].y);
      __syncwarp();
#pragma unroll
      for (int k = 0; k < NCOL; ++k) {   // lane l sums columns l, l + 32, ...
        float sum = 0.f;
#pragma unroll
        for (int r = 0; r < CHW; ++r) sum += red[r][lane + 32 * k];
        sums[k][t] = sum;
      }
      __syncwarp();
      (void)tg;
    }
    // the segment's outputs: per-step values of this channel (lead lane) and the channel sums of
    // dB / dC (column j: row j of dB for j < NP, row j - NP of dC otherwise), as 16-byte pieces when
    // the rows allow it
    if (valid && lead) {
      const int64_t odu = b * p.sdu[0] + d * p.sdu[1] + t0, odd = b * p.sdd[0] + d * p.sdd[1] + t0;
      const int64_t odz = b * p.sdz[0] + d * p.sdz[1] + t0;
      if (p.vecout && steps == SEG) {
        store_seg<IO>(p.du, odu, duo);
        store_seg<IO>(p.ddelta, odd, ddo);
        if (f.z) store_seg<IO>(p.dz, odz, dzo);
      } else {
#pragma unroll
        for (int t = 0; t < SEG; ++t) {
          if (t >= steps) break;
          st<IO>(p.du, odu + t, duo[t]);
          st<IO>(p.ddelta, odd + t, ddo[t]);
          if (f.z) st<IO>(p.dz, odz + t, dzo[t]);
        }
      }
    }
#pragma unroll
    for (int k = 0; k < NCOL; ++k) {
      const int col = lane + 32 * k;
      const int n = col % NP;
      if (n < N) {
        float* dst = col < NP ? p.dB + b * p.sdB[0] + n * p.sdB[1] : p.dC + b * p.sdC[0] + n * p.sdC[1];
        const int64_t st2 = col < NP ? p.sdB[2] : p.sdC[2];
        if (p.vecdbc && steps == SEG) {
          atomicAdd(reinterpret_cast<float4*>(dst + t0), make_float4(sums[k][0], sums[k][1], sums[k][2], sums[k][3]));
          atomicAdd(reinterpret_cast<float4*>(dst + t0 + 4), make_float4(sums[k][4], sums[k][5], sums[k][6], sums[k][7]));
        } else {
#pragma unroll
          for (int t = 0; t < SEG; ++t) {
            if (t >= steps) break;
            atomicAdd(dst + (t0 + t) * st2, sums[k][t]);
          }
        }
      }
    }
  }
  if (!valid) return;
  // ---- the summed parameter gradients and dh0 ----
#pragma unroll
  for (int q = 0; q < 4; ++q) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int n = g * 8 + 2 * q + e;
      if (n >= N) continue;
      atomicAdd(p.dA + d * N + n, e ? dA[q].y : dA[q].x);
      if (p.dh0) p.dh0[b * p.sdh0[0] + d * p.sdh0[1] + n * p.sdh0[2]] = e ? lam[q].y : lam[q].x;
    }
  }
  if (lead) {
    if (p.dD) atomicAdd(p.dD + d, dD);
    if (p.dbias) atomicAdd(p.dbias + d, dbias);
  }
}

template <typename IO, bool PRECISE>
cudaError_t launch_typed(const BwdProblem& p, int sms, cudaStream_t s) {
  const int64_t zero_total = p.f.D * p.f.N + 2 * p.bc_rows * p.f.N * p.f.L + 2 * p.f.D;
  const int zb = (int)std::min<int64_t>((zero_total + 255) / 256, (int64_t)sms * 8);
  bwd_zero_kernel<<<zb, 256, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // lanes per channel by the state size: 2 (N <= 16, 16 channels per warp), 4 (N <= 32), 8 (N <= 64)
  const int lpc = bwd_lanes_per_channel(p.f.N);
  const int chw = 32 / lpc;
  const dim3 grid((unsigned)((p.f.D + chw - 1) / chw), (unsigned)p.f.B);
#define SSM_BWD_LAUNCH(L)                                                   \
  if (lpc == L) {                                                           \
    if (p.f.zoh) scan_bwd_kernel<IO, PRECISE, true, L><<<grid, 32, 0, s>>>(p); \
    else scan_bwd_kernel<IO, PRECISE, false, L><<<grid, 32, 0, s>>>(p);        \
  }
  SSM_BWD_LAUNCH(2)
  SSM_BWD_LAUNCH(4)
  SSM_BWD_LAUNCH(8)
#undef SSM_BWD_LAUNCH
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_scan_bwd(const BwdProblem& p, int sms, cudaStream_t s) {
  if (p.f.io == SSM_F32) return launch_typed<float, true>(p, sms, s);
  return launch_typed<__nv_bfloat16, false>(p, sms, s);
}

}  // namespace ssm
