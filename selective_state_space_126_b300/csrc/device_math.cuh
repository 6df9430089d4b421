// device_math.cuh -- small device helpers shared by the scan and decode kernels.
//
// Precision policy:
//  * the state recurrence, the C contraction and every intermediate are fp32;
//  * exp(Delta * A) uses the SFU base-2 exponential (ex2.approx.ftz) on
//    Delta * A * log2(e), relative error a few ulp;
//  * softplus has two forms.  For bf16 I/O:
//    max(s,0) + log1p(e) with e = 2^(-|s| log2 e) from the SFU and
//    log1p(e) = e * q(e) evaluated as a polynomial on the FMA pipe (q fitted
//    on [0, 1] by fit_log1p.py, relative error 2.3e-7), so Delta keeps its
//    relative accuracy however small it is.  For fp32 I/O the library
//    log1pf/expf form is used;
//  * silu(z) = z / (1 + 2^(-z log2 e)) with the SFU reciprocal;
//  * the exact-ZOH input coefficient (exp(Delta A) - 1) / A: see zoh_coef.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

namespace ssm {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// log1p(e) for e in [0, 1] as e * (1 + e * r(e)); r is the degree-7
// polynomial printed by fit_log1p.py (relative error 2.3e-7 in fp32).
__device__ __forceinline__ float log1p_unit(float e) {
  float r = 6.479088217e-03f;
  r = fmaf(r, e, -3.448650241e-02f);
  r = fmaf(r, e, 8.630371094e-02f);
  r = fmaf(r, e, -1.434402466e-01f);
  r = fmaf(r, e, 1.942283958e-01f);
  r = fmaf(r, e, -2.492260784e-01f);
  r = fmaf(r, e, 3.332882226e-01f);
  r = fmaf(r, e, -4.999993443e-01f);
  return e * fmaf(e, r, 1.f);
}

// Two-lane form of log1p_unit on packed f32x2 FMAs.
__device__ __forceinline__ float2 log1p_unit2(float2 e) {
  float2 r = make_float2(6.479088217e-03f, 6.479088217e-03f);
  r = __ffma2_rn(r, e, make_float2(-3.448650241e-02f, -3.448650241e-02f));
  r = __ffma2_rn(r, e, make_float2(8.630371094e-02f, 8.630371094e-02f));
  r = __ffma2_rn(r, e, make_float2(-1.434402466e-01f, -1.434402466e-01f));
  r = __ffma2_rn(r, e, make_float2(1.942283958e-01f, 1.942283958e-01f));
  r = __ffma2_rn(r, e, make_float2(-2.492260784e-01f, -2.492260784e-01f));
  r = __ffma2_rn(r, e, make_float2(3.332882226e-01f, 3.332882226e-01f));
  r = __ffma2_rn(r, e, make_float2(-4.999993443e-01f, -4.999993443e-01f));
  return __fmul2_rn(e, __ffma2_rn(e, r, make_float2(1.f, 1.f)));
}

// softplus(s) = log(1 + e^s) = max(s, 0) + log1p(e^{-|s|})
template <bool PRECISE>
__device__ __forceinline__ float softplus(float s) {
  if (PRECISE) {
    return fmaxf(s, 0.f) + log1pf(expf(-fabsf(s)));
  } else {
    return fmaxf(s, 0.f) + log1p_unit(ex2_approx(-fabsf(s) * kLog2e));
  }
}

template <bool PRECISE>
__device__ __forceinline__ float silu(float z) {
  if (PRECISE) {
    return z / (1.f + expf(-z));
  } else {
    return z * rcp_approx(1.f + ex2_approx(-z * kLog2e));
  }
}

// silu(z) = z sigmoid(z) = z (1 + tanh(z / 2)) / 2 with the SFU tanh: one SFU operation instead
// of an ex2 and a half-rate reciprocal.  The tanh approximation's relative error (about 2^-11) is
// below the rounding of a bf16 output.
__device__ __forceinline__ float silu_tanh(float z) {
  float th;
  asm("tanh.approx.f32 %0, %1;" : "=f"(th) : "f"(0.5f * z));
  return z * fmaf(0.5f, th, 0.5f);
}

// Two-lane forms of the fast softplus and silu above, with the FMA-pipe work
// on packed f32x2 instructions (same arithmetic, half the issue slots).
__device__ __forceinline__ float2 softplus2_fast(float2 s) {
  const float2 x = __fmul2_rn(make_float2(fabsf(s.x), fabsf(s.y)), make_float2(-kLog2e, -kLog2e));
  return __fadd2_rn(make_float2(fmaxf(s.x, 0.f), fmaxf(s.y, 0.f)),
                    log1p_unit2(make_float2(ex2_approx(x.x), ex2_approx(x.y))));
}

__device__ __forceinline__ float2 silu2_fast(float2 z) {
  const float2 x = __fmul2_rn(z, make_float2(-kLog2e, -kLog2e));
  const float2 den = __fadd2_rn(make_float2(ex2_approx(x.x), ex2_approx(x.y)), make_float2(1.f, 1.f));
  return __fmul2_rn(z, make_float2(rcp_approx(den.x), rcp_approx(den.y)));
}

// Exact zero-order-hold input coefficient of one state ("Mamba and state space
// models", docs.ifdog.com, section "Discretisation": Bbar = (Delta A)^-1
// (exp(Delta A) - 1) Delta B, so Bbar x = g B u with g = (exp(Delta A) - 1) / A
// = Delta phi(Delta A), phi(x) = (e^x - 1) / x).  Given x = Delta A, a = e^x
// and inv_a = 1 / A (infinite at A = 0, where the series branch is taken):
//  * fp32 I/O: |x| < 1/2 : g = Delta (1 + x/2! + ... + x^7/8!), the Taylor
//    series of phi (truncation below 1.1e-8); |x| >= 1/2 : g = expm1f(x) / A;
//  * bf16 I/O: |x| < 1/64 : g = Delta (1 + x/2 + x^2/6) (truncation below
//    1.6e-7); |x| >= 1/64 : g = (a - 1) / A with a from the SFU, whose error
//    relative to |a - 1| >= 0.0155 stays below 2e-5 -- far inside the bf16
//    rounding of the output, and a third of the series' work.
__device__ __forceinline__ float phi_series(float x) {
  float r = 2.4801587301587302e-05f;                 // 1/8!
  r = fmaf(r, x, 1.9841269841269841e-04f);          // 1/7!
  r = fmaf(r, x, 1.3888888888888889e-03f);          // 1/6!
  r = fmaf(r, x, 8.3333333333333333e-03f);          // 1/5!
  r = fmaf(r, x, 4.1666666666666667e-02f);          // 1/4!
  r = fmaf(r, x, 1.6666666666666667e-01f);          // 1/3!
  r = fmaf(r, x, 0.5f);                             // 1/2!
  return fmaf(r, x, 1.f);
}

constexpr float kZohFastCut = 0.015625f;   // 1/64

template <bool PRECISE>
__device__ __forceinline__ float zoh_coef(float dt, float x, float a, float inv_a) {
  if (PRECISE) return fabsf(x) < 0.5f ? dt * phi_series(x) : expm1f(x) * inv_a;
  const float small = dt * fmaf(fmaf(x, 1.6666666666666667e-01f, 0.5f), x, 1.f);
  return fabsf(x) < kZohFastCut ? small : (a - 1.f) * inv_a;
}

// Two-lane form of the bf16-I/O zoh_coef on packed f32x2 FMAs.
__device__ __forceinline__ float2 zoh_coef2_fast(float2 dt, float2 x, float2 a, float2 inv_a) {
  const float2 r = __ffma2_rn(x, make_float2(1.6666666666666667e-01f, 1.6666666666666667e-01f), make_float2(0.5f, 0.5f));
  const float2 small = __fmul2_rn(dt, __ffma2_rn(r, x, make_float2(1.f, 1.f)));
  const float2 large = __fmul2_rn(__fadd2_rn(a, make_float2(-1.f, -1.f)), inv_a);
  return make_float2(fabsf(x.x) < kZohFastCut ? small.x : large.x, fabsf(x.y) < kZohFastCut ? small.y : large.y);
}

// cos and sin of theta, for the rotation part exp(i theta) of a complex Abar.
// PRECISE: the library sincosf.  Fast form: Cody-Waite reduction (Cody and
// Waite, "Software Manual for the Elementary Functions", 1980) of theta to
// [-pi, pi] with 2 pi split as 6.28125 (exact in 8 bits, so k * 6.28125 is
// exact for |k| < 2^16) plus the remainder 2 pi - 6.28125, then the SFU
// sin / cos on the reduced argument.
constexpr float kTwoPiHi = 6.28125f;
constexpr float kTwoPiLo = 1.9353071795864769e-3f;
constexpr float kInvTwoPi = 0.15915494309189535f;

__device__ __forceinline__ float sin_approx(float x) {
  float y;
  asm("sin.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float cos_approx(float x) {
  float y;
  asm("cos.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <bool PRECISE>
__device__ __forceinline__ float2 cos_sin(float th) {
  if (PRECISE) {
    float s, c;
    sincosf(th, &s, &c);
    return make_float2(c, s);
  }
  const float k = rintf(th * kInvTwoPi);
  const float r = fmaf(-k, kTwoPiLo, fmaf(-k, kTwoPiHi, th));
  return make_float2(cos_approx(r), sin_approx(r));
}

// Delta for one element: softplus(delta + bias) or the plain sum.
template <bool PRECISE>
__device__ __forceinline__ float delta_of(float delta, float bias, bool use_softplus) {
  const float s = delta + bias;
  return use_softplus ? softplus<PRECISE>(s) : s;
}

// Delta for two elements of one channel.
template <bool PRECISE>
__device__ __forceinline__ float2 delta_of2(float2 delta, float bias, bool use_softplus) {
  const float2 s = __fadd2_rn(delta, make_float2(bias, bias));
  if (!use_softplus) return s;
  if (PRECISE) return make_float2(softplus<true>(s.x), softplus<true>(s.y));
  return softplus2_fast(s);
}

// silu of two elements.
template <bool PRECISE>
__device__ __forceinline__ float2 silu2(float2 z) {
  if (PRECISE) return make_float2(silu<true>(z.x), silu<true>(z.y));
  return silu2_fast(z);
}

// ---------------------------------------------------------------------------
// I/O element types
// ---------------------------------------------------------------------------
__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T>
__device__ __forceinline__ T from_f32(float v);
template <>
__device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// 16-byte vectors: 8 bf16 or 4 fp32 values.
template <typename T>
struct Vec16;
template <>
struct Vec16<float> {
  static constexpr int kN = 4;
};
template <>
struct Vec16<__nv_bfloat16> {
  static constexpr int kN = 8;
};

__device__ __forceinline__ void unpack16(const uint4& q, float (&f)[4]) {
  f[0] = __uint_as_float(q.x);
  f[1] = __uint_as_float(q.y);
  f[2] = __uint_as_float(q.z);
  f[3] = __uint_as_float(q.w);
}

__device__ __forceinline__ void unpack16(const uint4& q, float (&f)[8]) {
  f[0] = __uint_as_float(q.x << 16);
  f[1] = __uint_as_float(q.x & 0xffff0000u);
  f[2] = __uint_as_float(q.y << 16);
  f[3] = __uint_as_float(q.y & 0xffff0000u);
  f[4] = __uint_as_float(q.z << 16);
  f[5] = __uint_as_float(q.z & 0xffff0000u);
  f[6] = __uint_as_float(q.w << 16);
  f[7] = __uint_as_float(q.w & 0xffff0000u);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint4 pack16(const float (&f)[4]) {
  return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
}

__device__ __forceinline__ uint4 pack16(const float (&f)[8]) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ void stg_v4(void* p, const uint4& v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// ---------------------------------------------------------------------------
// device status word (bounded waits record SSM_ERR_TIMEOUT here)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void record_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

}  // namespace ssm
