// conv1d.cu -- the causal depthwise convolution along time, with an optional
// SiLU, that produces the input of the SSM branch ("Mamba and state space
// models", docs.ifdog.com, section "Mamba architecture", step 3a: every
// channel is convolved on its own with a kernel of d_conv taps, so each step
// sees itself and the d_conv - 1 steps before it; step 3b: the result feeds the
// projections that make Delta, B and C, and the scan as u):
//
//   out[b,d,t] = act(bias[d] + sum_{k<W} w[d,k] x[b,d,t-(W-1)+k]),
//
// with the W-1 inputs before t = 0 taken from a history tensor or zero.
//
// The operation reads each input once and writes each output once (4 bytes
// per element in bf16), so it is bound by HBM.  Because its output also feeds
// the projections ahead of the scan, it is a kernel of its own: folding it into
// the scan's u load would not remove the write of its output.
//
//   * Vector path (time stride 1, rows on 16-byte boundaries, L a multiple of
//     the 16-byte vector, W <= 4): a run is 32 x kRunU consecutive 16-byte
//     vectors of one row, lane l holding vectors l, 32 + l, ...; all kRunU
//     128-bit loads are issued before any is used, so each thread keeps 128
//     bytes in flight.  Each warp takes a contiguous block of runs.  The W-1 inputs in front of a lane's vector come from
//     the lane before it by shuffle (lane 0 takes them from lane 31 of the
//     previous group, and at the start of a run from memory, the history or
//     zero).  The taps are padded to 4 with leading zeros, so every output
//     pair takes one unrolled sequence of packed f32x2 fused multiply-adds in
//     tap order.  Outputs leave as 128-bit stores.  The grid is persistent
//     (the blocks resident at once on every SM).
//   * Generic path: one thread per output element, any non-negative strides,
//     W <= 16, the same tap order.
#include <algorithm>

#include "device_math.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int kConvVecMaxW = 4;    // taps of the vector path
#ifndef SSM_CONV_RUN_U
#define SSM_CONV_RUN_U 8
#endif
#ifndef SSM_CONV_BLOCKS_PER_SM
#define SSM_CONV_BLOCKS_PER_SM 16
#endif
constexpr int kRunU = SSM_CONV_RUN_U;   // 16-byte vectors per lane per run
constexpr int kConvThreads = 128;  // vector-path block
constexpr int kConvBlocksPerSM = SSM_CONV_BLOCKS_PER_SM;

// Raw bits of one element (for assembling the history into vector form).
__device__ __forceinline__ uint32_t raw_of(float v) { return __float_as_uint(v); }
__device__ __forceinline__ uint32_t raw_of(__nv_bfloat16 v) { return (uint32_t)__bfloat16_as_ushort(v); }

// Shuffles the words of `q` that hold its last three elements from lane
// `src` (relative: up by `delta` when UP, else absolute lane `delta`).
template <typename IO, bool UP>
__device__ __forceinline__ uint4 shfl_tail3(const uint4& q, int delta) {
  uint4 r = q;
  if (UP) {
    if (sizeof(IO) == 4) r.y = __shfl_up_sync(0xffffffffu, q.y, delta);
    r.z = __shfl_up_sync(0xffffffffu, q.z, delta);
    r.w = __shfl_up_sync(0xffffffffu, q.w, delta);
  } else {
    if (sizeof(IO) == 4) r.y = __shfl_sync(0xffffffffu, q.y, delta);
    r.z = __shfl_sync(0xffffffffu, q.z, delta);
    r.w = __shfl_sync(0xffffffffu, q.w, delta);
  }
  return r;
}

// Element pair (x[m], x[m+1]) of the window around a vector: m in -3..VEC-2,
// where x[0..VEC-1] is the vector `cur` and x[-4..-1] the tail of `prev`.
// For bf16 an even m is one 32-bit word split in two; an odd m takes the high
// half of one word and the low half of the next.
template <typename IO>
__device__ __forceinline__ float2 win_pair(const uint4& prev, const uint4& cur, int m);
template <>
__device__ __forceinline__ float2 win_pair<__nv_bfloat16>(const uint4& prev, const uint4& cur, int m) {
  // word k of the 6-word window: prev.z, prev.w (elements -4..-1), cur.x .. cur.w
  auto word = [&](int k) { return k == 0 ? prev.z : k == 1 ? prev.w : k == 2 ? cur.x : k == 3 ? cur.y : k == 4 ? cur.z : cur.w; };
  const int e = m + 4;   // element index in the window, 0..11
  if ((e & 1) == 0) {
    const uint32_t w = word(e >> 1);
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  }
  return make_float2(__uint_as_float(word(e >> 1) & 0xffff0000u), __uint_as_float(word((e >> 1) + 1) << 16));
}
template <>
__device__ __forceinline__ float2 win_pair<float>(const uint4& prev, const uint4& cur, int m) {
  auto word = [&](int k) { return k == 0 ? prev.y : k == 1 ? prev.z : k == 2 ? prev.w : k == 3 ? cur.x : k == 4 ? cur.y : k == 5 ? cur.z : cur.w; };
  const int e = m + 3;   // element index in the window (prev.y = x[-3]), 0..6
  return make_float2(__uint_as_float(word(e)), __uint_as_float(word(e + 1)));
}

// A warp takes a contiguous block of runs (so the row, and with it the
// channel's taps, changes only every runs_per_row runs and no division is
// needed per run); in each run lane l holds vectors v0 + l, v0 + 32 + l, ...
// of the row, all loaded before any is used.  Output pairs (i, i+1) are
// computed on packed f32x2 FMAs, taps in order, which rounds exactly like the
// scalar form: bias, then w[0] x[t-3] + ... + w[3] x[t], one fused step each.
template <typename IO, bool PRECISE, bool SILU>
__global__ void __launch_bounds__(kConvThreads) conv1d_vec_kernel(const ConvProblem p, int64_t runs_per_row,
                                                                 int64_t nruns, int64_t runs_per_warp) {
  constexpr int VEC = Vec16<IO>::kN;
  const int lane = threadIdx.x & 31;
  const int64_t nvec = p.L / VEC;
  int64_t run = (((int64_t)blockIdx.x * kConvThreads + threadIdx.x) >> 5) * runs_per_warp;
  const int64_t end = min(run + runs_per_warp, nruns);
  if (run >= end) return;
  const int64_t row0 = run / runs_per_row;
  int64_t seg = run - row0 * runs_per_row;
  int64_t b = row0 / p.D, d = row0 - b * p.D;
  float2 w2[kConvVecMaxW];
  float2 bias2;
  auto load_taps = [&]() {
#pragma unroll
    for (int k = 0; k < kConvVecMaxW; ++k) {   // padded to 4 with leading zeros; tap 3 on the current step
      const int kk = k - (kConvVecMaxW - p.W);
      const float wv = kk >= 0 ? p.w[d * p.sw[0] + kk * p.sw[1]] : 0.f;
      w2[k] = make_float2(wv, wv);
    }
    const float bv = p.bias ? p.bias[d] : 0.f;
    bias2 = make_float2(bv, bv);
  };
  load_taps();
  for (; run < end; ++run) {
    const IO* xrow = static_cast<const IO*>(p.x) + b * p.sx[0] + d * p.sx[1];
    IO* orow = static_cast<IO*>(p.out) + b * p.so[0] + d * p.so[1];
    const int64_t v0 = seg * 32 * kRunU;
    uint4 cur[kRunU];
#pragma unroll
    for (int j = 0; j < kRunU; ++j) {
      const int64_t vi = v0 + j * 32 + lane;
      cur[j] = vi < nvec ? ldg_nc_v4(xrow + vi * VEC) : make_uint4(0, 0, 0, 0);
    }
    // the 16 bytes in front of the run, for lane 0: memory, else the history, else zero
    uint4 front = make_uint4(0, 0, 0, 0);
    if (lane == 0) {
      if (v0 > 0) {
        front = ldg_nc_v4(xrow + (v0 - 1) * VEC);
      } else if (p.x_hist) {
        const IO* h = static_cast<const IO*>(p.x_hist) + b * p.sxh[0] + d * p.sxh[1];
        uint32_t words[4] = {0, 0, 0, 0};
#pragma unroll
        for (int slot = VEC - 3; slot < VEC; ++slot) {   // vector slot VEC-(W-1)+i holds history element i
          const int i = slot - (VEC - (p.W - 1));
          if (i < 0) continue;
          const uint32_t raw = raw_of(h[i * p.sxh[2]]);
          if (sizeof(IO) == 4) words[slot] = raw;
          else words[slot >> 1] |= (slot & 1) ? (raw << 16) : raw;
        }
        front = make_uint4(words[0], words[1], words[2], words[3]);
      }
    }
#pragma unroll
    for (int j = 0; j < kRunU; ++j) {
      // the vector before this lane's: lane-1's, or for lane 0 lane 31's of the previous group
      const uint4 up = shfl_tail3<IO, true>(cur[j], 1);
      const uint4 wrap = j == 0 ? front : shfl_tail3<IO, false>(cur[j - 1], 31);
      const uint4 prev = lane == 0 ? wrap : up;
      float o[VEC];
#pragma unroll
      for (int i = 0; i < VEC; i += 2) {
        float2 v = bias2;
#pragma unroll
        for (int k = 0; k < kConvVecMaxW; ++k) v = __ffma2_rn(w2[k], win_pair<IO>(prev, cur[j], i + k - 3), v);
        if (SILU) v = silu2<PRECISE>(v);
        o[i] = v.x;
        o[i + 1] = v.y;
      }
      const int64_t vi = v0 + j * 32 + lane;
      if (vi < nvec) stg_v4(orow + vi * VEC, pack16(o));
    }
    if (++seg == runs_per_row) {   // next row: next channel (and batch row)
      seg = 0;
      if (++d == p.D) {
        d = 0;
        ++b;
      }
      if (run + 1 < end) load_taps();
    }
  }
}

template <typename IO, bool PRECISE>
__global__ void __launch_bounds__(256) conv1d_generic_kernel(const ConvProblem p) {
  const int64_t total = p.B * p.D * p.L;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
    const int64_t t = i % p.L;
    const int64_t row = i / p.L;
    const int64_t b = row / p.D, d = row - b * p.D;
    const IO* x = static_cast<const IO*>(p.x) + b * p.sx[0] + d * p.sx[1];
    const IO* h = p.x_hist ? static_cast<const IO*>(p.x_hist) + b * p.sxh[0] + d * p.sxh[1] : nullptr;
    float v = p.bias ? p.bias[d] : 0.f;
    for (int k = 0; k < p.W; ++k) {
      const int64_t src = t - (p.W - 1) + k;
      float xv = 0.f;
      if (src >= 0) xv = to_f32(x[src * p.sx[2]]);
      else if (h) xv = to_f32(h[(p.W - 1 + src) * p.sxh[2]]);
      v = fmaf(p.w[d * p.sw[0] + k * p.sw[1]], xv, v);
    }
    if (p.silu) v = silu<PRECISE>(v);
    static_cast<IO*>(p.out)[b * p.so[0] + d * p.so[1] + t * p.so[2]] = from_f32<IO>(v);
  }
}

bool vec_eligible(const ConvProblem& p) {
  const int es = p.io == SSM_F32 ? 4 : 2;
  const int vec = 16 / es;
  if (p.W > kConvVecMaxW || p.L % vec != 0) return false;
  if (p.sx[2] != 1 || p.so[2] != 1) return false;
  if (reinterpret_cast<uintptr_t>(p.x) % 16 || reinterpret_cast<uintptr_t>(p.out) % 16) return false;
  if (p.D > 1 && ((p.sx[1] * es) % 16 || (p.so[1] * es) % 16)) return false;
  if (p.B > 1 && ((p.sx[0] * es) % 16 || (p.so[0] * es) % 16)) return false;
  return true;
}

template <typename IO, bool PRECISE>
cudaError_t launch_typed(const ConvProblem& p, int sms, cudaStream_t s) {
  if (vec_eligible(p)) {
    const int64_t nvec = p.L / Vec16<IO>::kN;
    const int64_t runs_per_row = (nvec + 32 * kRunU - 1) / (32 * kRunU);
    const int64_t nruns = p.B * p.D * runs_per_row;
    // a persistent grid: exactly the blocks that are resident at once (the runs are dealt
    // to warps statically, so a block that had to wait for a slot would double the tail)
    auto kern = p.silu ? conv1d_vec_kernel<IO, PRECISE, true> : conv1d_vec_kernel<IO, PRECISE, false>;
    static int occupancy[2] = {0, 0};   // per SiLU form; a racing duplicate query is harmless
    int per_sm = occupancy[p.silu ? 1 : 0];
    if (per_sm == 0) {
      cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kConvThreads, 0);
      if (e != cudaSuccess) return e;
      per_sm = std::max(1, std::min(per_sm, kConvBlocksPerSM));
      occupancy[p.silu ? 1 : 0] = per_sm;
    }
    const int64_t warps_max = (int64_t)sms * per_sm * (kConvThreads / 32);
    const int64_t runs_per_warp = (nruns + warps_max - 1) / warps_max;
    const int64_t warps = (nruns + runs_per_warp - 1) / runs_per_warp;
    const int blocks = (int)((warps + kConvThreads / 32 - 1) / (kConvThreads / 32));
    kern<<<blocks, kConvThreads, 0, s>>>(p, runs_per_row, nruns, runs_per_warp);
  } else {
    const int64_t total = p.B * p.D * p.L;
    const int blocks = (int)std::min<int64_t>((total + 255) / 256, (int64_t)sms * 16);
    conv1d_generic_kernel<IO, PRECISE><<<blocks, 256, 0, s>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_causal_conv1d(const ConvProblem& p, int sms, cudaStream_t s) {
  if (p.io == SSM_F32) return launch_typed<float, true>(p, sms, s);
  return launch_typed<__nv_bfloat16, false>(p, sms, s);
}

}  // namespace ssm
