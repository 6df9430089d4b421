// state_update.cu -- one recurrent (decode) step against a persistent fp32 state.
//
// Constant time and memory per generated token ("gitcode.csdn.net", section 1,
// and section 2: the recurrent mode used for autoregressive inference):
//   h[b,d,n] <- exp(Delta A[d,n]) h[b,d,n] + Delta B[b,n] u[b,d]
//   y[b,d]    = (sum_n C[b,n] h[b,d,n] + D[d] u[b,d]) * silu(z[b,d])
// with Delta = softplus(delta[b,d] + bias[d]).
//
// The step is bound by the state read and write (64 + 64 bytes per channel at
// N = 16).  Q = N/4 adjacent lanes share one channel, each owning four
// consecutive states, so a warp writes the state as contiguous 512-byte runs
// and the output is reduced over the Q lanes with shuffles.
//
// Fast path (dense layouts, N in {8, 16, 32, 64} for bf16, {4, ..., 64} for
// fp32, D a multiple of the CTA's 128 / Q channels): each CTA owns one range
// of channels, keeps their A, bias and D in registers, and walks a strided
// set of batch rows.  A ring of 8 shared-memory slots, filled by 1-D bulk
// async copies (cp.async.bulk, one mbarrier per slot), keeps 8 rows' state
// tiles (2 KB each) and their u, delta, z, B, C in flight per CTA without
// holding them in registers, which is what it takes to cover the memory
// latency at full HBM bandwidth.  Other layouts use a per-item kernel that
// loads from global memory directly.
#include <algorithm>
#include <cstdlib>

#include "async_copy.cuh"
#include "device_math.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int ITEMS = 1;   // (channel, quad) items per thread of the per-item kernel
#ifndef SSM_DECODE_SLOTS
#define SSM_DECODE_SLOTS 16
#endif
constexpr int kRowSlots = SSM_DECODE_SLOTS;   // bulk-copy ring depth of the fast path (batch rows in flight per CTA)
#ifndef SSM_DECODE_GROUP
#define SSM_DECODE_GROUP 8
#endif
constexpr int kRowGroup = SSM_DECODE_GROUP;   // batch rows per barrier of the fast path
static_assert(kRowSlots % kRowGroup == 0 && kRowSlots >= 2 * kRowGroup, "ring of whole groups");

__device__ __forceinline__ void load4(const __nv_bfloat16* p, int64_t stride, int n0, int N, bool vec, float (&v)[4]) {
  if (vec) {
    const uint2 r = *reinterpret_cast<const uint2*>(p + n0);
    v[0] = __uint_as_float(r.x << 16);
    v[1] = __uint_as_float(r.x & 0xffff0000u);
    v[2] = __uint_as_float(r.y << 16);
    v[3] = __uint_as_float(r.y & 0xffff0000u);
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = (n0 + i < N) ? __bfloat162float(p[(n0 + i) * stride]) : 0.f;
  }
}

__device__ __forceinline__ void load4(const float* p, int64_t stride, int n0, int N, bool vec, float (&v)[4]) {
  if (vec) {
    const float4 r = *reinterpret_cast<const float4*>(p + n0);
    v[0] = r.x; v[1] = r.y; v[2] = r.z; v[3] = r.w;
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = (n0 + i < N) ? p[(n0 + i) * stride] : 0.f;
  }
}

// vec_state: state rows contiguous, 16-byte aligned, N % 4 == 0.
// vec_bc:    B and C rows contiguous with 8-byte (bf16) / 16-byte (fp32) aligned rows, N % 4 == 0.
// vec_a:     A rows contiguous, 16-byte aligned, N % 4 == 0.
template <typename IO, int Q, bool PRECISE>
__global__ void __launch_bounds__(256) state_update_kernel(const StepProblem p, const bool vec_state, const bool vec_bc,
                                                           const bool vec_a) {
  const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
  const int64_t gtid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t total = p.B * p.D * Q;
  const int N = (int)p.N;
  const int q = (int)(gtid % Q);   // nthreads is a multiple of Q, so every item of a thread has the same quad
  const int n0 = q * 4;

  float h[ITEMS][4], Bv[ITEMS][4], Cv[ITEMS][4], Av[ITEMS][4];
  float uv[ITEMS], dv[ITEMS], zv[ITEMS], bias[ITEMS], Dd[ITEMS];
  bool active[ITEMS];
  float* st[ITEMS];
  int64_t bb[ITEMS], dd[ITEMS];

  // ---- every load of every item first ----
#pragma unroll
  for (int it = 0; it < ITEMS; ++it) {
    const int64_t g = gtid + it * nthreads;
    active[it] = g < total;
    const int64_t c = active[it] ? g / Q : 0;
    const int64_t b = c / p.D, d = c % p.D;
    bb[it] = b;
    dd[it] = d;
    st[it] = p.state + b * p.sst[0] + d * p.sst[1];
    if (active[it] && n0 < N) {
      if (vec_state) {
        const float4 v = *reinterpret_cast<const float4*>(st[it] + n0);
        h[it][0] = v.x; h[it][1] = v.y; h[it][2] = v.z; h[it][3] = v.w;
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) h[it][i] = (n0 + i < N) ? st[it][(n0 + i) * p.sst[2]] : 0.f;
      }
      load4(static_cast<const IO*>(p.Bm) + b * p.sB[0], p.sB[1], n0, N, vec_bc, Bv[it]);
      load4(static_cast<const IO*>(p.Cm) + b * p.sC[0], p.sC[1], n0, N, vec_bc, Cv[it]);
      load4(p.A + d * p.sA[0], p.sA[1], n0, N, vec_a, Av[it]);
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) h[it][i] = Bv[it][i] = Cv[it][i] = Av[it][i] = 0.f;
    }
    if (active[it]) {
      uv[it] = to_f32(static_cast<const IO*>(p.u)[b * p.su[0] + d * p.su[1]]);
      dv[it] = to_f32(static_cast<const IO*>(p.delta)[b * p.sd[0] + d * p.sd[1]]);
      zv[it] = p.z ? to_f32(static_cast<const IO*>(p.z)[b * p.sz[0] + d * p.sz[1]]) : 0.f;
      bias[it] = p.bias ? p.bias[d] : 0.f;
      Dd[it] = p.Dskip ? p.Dskip[d] : 0.f;
    } else {
      uv[it] = dv[it] = zv[it] = bias[it] = Dd[it] = 0.f;
    }
  }

  // ---- the step ----
#pragma unroll
  for (int it = 0; it < ITEMS; ++it) {
    const float dt = delta_of<PRECISE>(dv[it], bias[it], p.softplus);
    const float du = dt * uv[it];
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float a = ex2_approx(dt * (Av[it][i] * kLog2e));
      const float bx = p.zoh ? zoh_coef<PRECISE>(dt, dt * Av[it][i], a, 1.f / Av[it][i]) * uv[it] : du;
      h[it][i] = fmaf(a, h[it][i], bx * Bv[it][i]);
      acc = fmaf(Cv[it][i], h[it][i], acc);
    }
#pragma unroll
    for (int off = 1; off < Q; off <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (active[it] && n0 < N) {
      if (vec_state) {
        *reinterpret_cast<float4*>(st[it] + n0) = make_float4(h[it][0], h[it][1], h[it][2], h[it][3]);
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (n0 + i < N) st[it][(n0 + i) * p.sst[2]] = h[it][i];
      }
    }
    if (active[it] && q == 0) {
      float out = fmaf(Dd[it], uv[it], acc);
      if (p.z) out *= silu<PRECISE>(zv[it]);
      static_cast<IO*>(p.y)[bb[it] * p.sy[0] + dd[it] * p.sy[1]] = from_f32<IO>(out);
    }
  }
}

// Shared-memory slot of the fast path: one batch row of one channel range.
template <typename IO, int Q>
struct RowSlot {
  static constexpr int CH = 128 / Q;                       // channels per CTA
  static constexpr int N = 4 * Q;
  static constexpr int kState = 0;                         // float [CH][N]: 2 KB
  static constexpr int kU = CH * N * 4;                    // IO [CH] each for u, delta, z
  static constexpr int kSeq = (CH * (int)sizeof(IO) + 15) / 16 * 16;
  static constexpr int kDelta = kU + kSeq, kZ = kU + 2 * kSeq;
  static constexpr int kB = kU + 3 * kSeq;                 // IO [N] each for B, C
  static constexpr int kBC = (N * (int)sizeof(IO) + 15) / 16 * 16;
  static constexpr int kC = kB + kBC;
  static constexpr int kBytes = kC + kBC;
  static_assert(CH * (int)sizeof(IO) % 16 == 0 && N * (int)sizeof(IO) % 16 == 0, "bulk copy sizes");
};

template <typename IO, int Q, bool PRECISE>
__global__ void __launch_bounds__(128) state_update_bulk_kernel(const StepProblem p, int row_groups, int* status) {
  using R = RowSlot<IO, Q>;
  constexpr int CH = R::CH;
  __shared__ __align__(128) unsigned char slots[kRowSlots][R::kBytes];
  __shared__ __align__(8) uint64_t bars[kRowSlots];

  const int tid = threadIdx.x;
  const int c = tid / Q, q = tid % Q, n0 = 4 * q;
  const int64_t d0 = (int64_t)blockIdx.x * CH;
  const int64_t d = d0 + c;
  const int g = blockIdx.y;
  const int rows = (int)((p.B - g + row_groups - 1) / row_groups);   // rows g, g + G, g + 2G, ...

  float A4[4];
  {
    const float4 a = *reinterpret_cast<const float4*>(p.A + d * p.sA[0] + n0);
    A4[0] = a.x * kLog2e; A4[1] = a.y * kLog2e; A4[2] = a.z * kLog2e; A4[3] = a.w * kLog2e;
  }
  const float bias = p.bias ? p.bias[d] : 0.f;
  const float Dd = p.Dskip ? p.Dskip[d] : 0.f;
  const bool has_z = p.z != nullptr;

  const uint32_t bar0 = smem_u32(&bars[0]);
  if (tid == 0) {
    for (int s = 0; s < kRowSlots; ++s) mbar_init(bar0 + 8 * s, 1);
    mbar_init_fence();
  }
  __syncthreads();
  const uint32_t tile_bytes = (uint32_t)(CH * R::N * 4 + (2 + (has_z ? 1 : 0)) * CH * (int)sizeof(IO) +
                                         2 * R::N * (int)sizeof(IO));
  auto issue = [&](int k) {
    const int64_t b = g + (int64_t)k * row_groups;
    const int s = k % kRowSlots;
    const uint32_t dst = smem_u32(&slots[s][0]), bar = bar0 + 8 * s;
    mbar_expect_tx(bar, tile_bytes);
    bulk_load(dst + R::kState, p.state + b * p.sst[0] + d0 * R::N, CH * R::N * 4, bar);
    bulk_load(dst + R::kU, static_cast<const IO*>(p.u) + b * p.su[0] + d0, CH * sizeof(IO), bar);
    bulk_load(dst + R::kDelta, static_cast<const IO*>(p.delta) + b * p.sd[0] + d0, CH * sizeof(IO), bar);
    if (has_z) bulk_load(dst + R::kZ, static_cast<const IO*>(p.z) + b * p.sz[0] + d0, CH * sizeof(IO), bar);
    bulk_load(dst + R::kB, static_cast<const IO*>(p.Bm) + b * p.sB[0], R::N * sizeof(IO), bar);
    bulk_load(dst + R::kC, static_cast<const IO*>(p.Cm) + b * p.sC[0], R::N * sizeof(IO), bar);
  };
  if (tid == 0)
    for (int k = 0; k < kRowSlots && k < rows; ++k) issue(k);

  // Rows go in groups of kRowGroup per barrier: every thread waits for the
  // group's slots, updates its quad of each row, then (after one barrier)
  // thread 0 refills the group's slots with rows kRowSlots further on.
  for (int k0 = 0; k0 < rows; k0 += kRowGroup) {
    bool ok = true;
#pragma unroll
    for (int r = 0; r < kRowGroup; ++r) {
      const int k = k0 + r;
      if (k < rows) ok = ok && mbar_wait(bar0 + 8 * (k % kRowSlots), (uint32_t)(k / kRowSlots) & 1u);
    }
    if (__syncthreads_or(!ok)) {
      // a copy never completed: record it, let the others in flight land (bounded), leave
      if (tid == 0) {
        record_status(status, SSM_ERR_TIMEOUT);
        const int issued = k0 >= kRowGroup ? k0 - kRowGroup + kRowSlots : kRowSlots;   // rows [0, issued) went out
        for (int j = k0; j < issued && j < rows; ++j)
          (void)mbar_wait(bar0 + 8 * (j % kRowSlots), (uint32_t)(j / kRowSlots) & 1u);
      }
      return;
    }
    // every thread is done with the previous group: its slots take the rows kRowSlots further on
    if (tid == 0 && k0 >= kRowGroup)
      for (int k = k0 - kRowGroup; k < k0; ++k)
        if (k + kRowSlots < rows) issue(k + kRowSlots);
#pragma unroll
    for (int r = 0; r < kRowGroup; ++r) {
      const int k = k0 + r;
      if (k >= rows) break;
      const unsigned char* sl = slots[k % kRowSlots];
      const int64_t b = g + (int64_t)k * row_groups;
      const float4 hv = *reinterpret_cast<const float4*>(sl + R::kState + (c * R::N + n0) * 4);
      const float uv = to_f32(reinterpret_cast<const IO*>(sl + R::kU)[c]);
      const float dv = to_f32(reinterpret_cast<const IO*>(sl + R::kDelta)[c]);
      const float zv = has_z ? to_f32(reinterpret_cast<const IO*>(sl + R::kZ)[c]) : 0.f;
      const IO* Bs = reinterpret_cast<const IO*>(sl + R::kB);
      const IO* Cs = reinterpret_cast<const IO*>(sl + R::kC);
      const float dt = delta_of<PRECISE>(dv, bias, p.softplus);
      const float du = dt * uv;
      float h[4] = {hv.x, hv.y, hv.z, hv.w};
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float a = ex2_approx(dt * A4[i]);
        h[i] = fmaf(a, h[i], du * to_f32(Bs[n0 + i]));
        acc = fmaf(to_f32(Cs[n0 + i]), h[i], acc);
      }
#pragma unroll
      for (int off = 1; off < Q; off <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      *reinterpret_cast<float4*>(p.state + b * p.sst[0] + d * R::N + n0) = make_float4(h[0], h[1], h[2], h[3]);
      if (q == 0) {
        float out = fmaf(Dd, uv, acc);
        if (has_z) out *= silu<PRECISE>(zv);
        static_cast<IO*>(p.y)[b * p.sy[0] + d] = from_f32<IO>(out);
      }
    }
  }
}

// Wide fast path for N = 16: one thread per channel with all 16 states, 128
// channels per CTA, so that a batch row is one 8 KB state copy plus three
// 256-byte copies of u, delta, z and two 32-byte copies of B, C.  The new
// state is written back into the slot and leaves, with the row of y, as two
// bulk stores (8 KB and 256 bytes), so that HBM sees whole contiguous rows in
// both directions.  Thread c
// visits its four 16-byte state pieces in an order rotated by (c / 2) % 4,
// which spreads a quarter-warp's shared-memory reads over all bank groups; A,
// B and C are read in the same rotated order, so no piece is ever moved back.
template <typename IO>
struct WideSlot {
  static constexpr int CH = 128;
  static constexpr int kState = 0;                                      // float [128][16]: 8 KB
  static constexpr int kU = CH * 16 * 4;                                // IO [128] each for u, delta, z
  static constexpr int kSeq = CH * (int)sizeof(IO);
  static constexpr int kDelta = kU + kSeq, kZ = kU + 2 * kSeq;
  static constexpr int kB = kU + 3 * kSeq;                              // IO [16] each for B, C
  static constexpr int kBC = 16 * (int)sizeof(IO);
  static constexpr int kC = kB + kBC;
  static constexpr int kBytes = (kC + kBC + 127) / 128 * 128;
};
constexpr int kWideSlots = 4;

__device__ __forceinline__ void load_piece(const __nv_bfloat16* p, float (&v)[4]) {
  const uint2 r = *reinterpret_cast<const uint2*>(p);
  v[0] = __uint_as_float(r.x << 16);
  v[1] = __uint_as_float(r.x & 0xffff0000u);
  v[2] = __uint_as_float(r.y << 16);
  v[3] = __uint_as_float(r.y & 0xffff0000u);
}
__device__ __forceinline__ void load_piece(const float* p, float (&v)[4]) {
  const float4 r = *reinterpret_cast<const float4*>(p);
  v[0] = r.x; v[1] = r.y; v[2] = r.z; v[3] = r.w;
}

template <typename IO, bool PRECISE>
__global__ void __launch_bounds__(128) state_update_wide_kernel(const StepProblem p, int row_groups, int* status) {
  using W = WideSlot<IO>;
  __shared__ __align__(128) unsigned char slots[kWideSlots][W::kBytes];
  __shared__ __align__(8) uint64_t bars[kWideSlots];

  const int c = threadIdx.x;
  const int rot = (c >> 1) & 3;
  const int64_t d0 = (int64_t)blockIdx.x * W::CH;
  const int64_t d = d0 + c;
  const int g = blockIdx.y;
  const int rows = (int)((p.B - g + row_groups - 1) / row_groups);   // rows g, g + G, g + 2G, ...

  float2 A2[8];   // A * log2(e), pieces in rotated order
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float4 a = *reinterpret_cast<const float4*>(p.A + d * p.sA[0] + 4 * ((j + rot) & 3));
    A2[2 * j] = make_float2(a.x * kLog2e, a.y * kLog2e);
    A2[2 * j + 1] = make_float2(a.z * kLog2e, a.w * kLog2e);
  }
  const float bias = p.bias ? p.bias[d] : 0.f;
  const float Dd = p.Dskip ? p.Dskip[d] : 0.f;
  const bool has_z = p.z != nullptr;

  const uint32_t bar0 = smem_u32(&bars[0]);
  if (c == 0) {
    for (int s = 0; s < kWideSlots; ++s) mbar_init(bar0 + 8 * s, 1);
    mbar_init_fence();
  }
  __syncthreads();
  const uint32_t tile_bytes = (uint32_t)(W::CH * 16 * 4 + (2 + (has_z ? 1 : 0)) * W::kSeq + 2 * W::kBC);
  auto issue = [&](int k) {
    const int64_t b = g + (int64_t)k * row_groups;
    const int s = k % kWideSlots;
    const uint32_t dst = smem_u32(&slots[s][0]), bar = bar0 + 8 * s;
    mbar_expect_tx(bar, tile_bytes);
    bulk_load(dst + W::kState, p.state + b * p.sst[0] + d0 * 16, W::CH * 16 * 4, bar);
    bulk_load(dst + W::kU, static_cast<const IO*>(p.u) + b * p.su[0] + d0, W::kSeq, bar);
    bulk_load(dst + W::kDelta, static_cast<const IO*>(p.delta) + b * p.sd[0] + d0, W::kSeq, bar);
    if (has_z) bulk_load(dst + W::kZ, static_cast<const IO*>(p.z) + b * p.sz[0] + d0, W::kSeq, bar);
    bulk_load(dst + W::kB, static_cast<const IO*>(p.Bm) + b * p.sB[0], W::kBC, bar);
    bulk_load(dst + W::kC, static_cast<const IO*>(p.Cm) + b * p.sC[0], W::kBC, bar);
  };
  if (c == 0)
    for (int k = 0; k < kWideSlots && k < rows; ++k) issue(k);

  for (int k = 0; k < rows; ++k) {
    const int s = k % kWideSlots;
    const bool ok = mbar_wait(bar0 + 8 * s, (uint32_t)(k / kWideSlots) & 1u);
    if (__syncthreads_or(!ok)) {
      // a copy never completed: record it, let the others in flight land (bounded), leave
      if (c == 0) {
        record_status(status, SSM_ERR_TIMEOUT);
        const int issued = k >= 1 ? k - 1 + kWideSlots : kWideSlots;   // rows [0, issued) went out
        for (int j = k; j < issued && j < rows; ++j)
          (void)mbar_wait(bar0 + 8 * (j % kWideSlots), (uint32_t)(j / kWideSlots) & 1u);
        bulk_wait<0>();
      }
      return;
    }
    // every thread is done with row k-1 and its store has read the slot: the slot takes row k-1+kWideSlots
    if (c == 0 && k >= 1 && k - 1 + kWideSlots < rows) {
      bulk_wait_read<0>();
      issue(k - 1 + kWideSlots);
    }
    unsigned char* sl = slots[s];
    const int64_t b = g + (int64_t)k * row_groups;
    const float uv = to_f32(reinterpret_cast<const IO*>(sl + W::kU)[c]);
    const float dv = to_f32(reinterpret_cast<const IO*>(sl + W::kDelta)[c]);
    const float zv = has_z ? to_f32(reinterpret_cast<const IO*>(sl + W::kZ)[c]) : 0.f;
    const float dt = delta_of<PRECISE>(dv, bias, p.softplus);
    const float2 dt2 = make_float2(dt, dt), du2 = make_float2(dt * uv, dt * uv);
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int piece = (j + rot) & 3;
      float4* hp = reinterpret_cast<float4*>(sl + W::kState + (c * 16 + 4 * piece) * 4);
      const float4 hv = *hp;
      float Bv[4], Cv[4];
      load_piece(reinterpret_cast<const IO*>(sl + W::kB) + 4 * piece, Bv);
      load_piece(reinterpret_cast<const IO*>(sl + W::kC) + 4 * piece, Cv);
      const float2 x0 = __fmul2_rn(dt2, A2[2 * j]), x1 = __fmul2_rn(dt2, A2[2 * j + 1]);
      const float2 a0 = make_float2(ex2_approx(x0.x), ex2_approx(x0.y));
      const float2 a1 = make_float2(ex2_approx(x1.x), ex2_approx(x1.y));
      const float2 h0 = __ffma2_rn(a0, make_float2(hv.x, hv.y), __fmul2_rn(du2, make_float2(Bv[0], Bv[1])));
      const float2 h1 = __ffma2_rn(a1, make_float2(hv.z, hv.w), __fmul2_rn(du2, make_float2(Bv[2], Bv[3])));
      acc = __ffma2_rn(make_float2(Cv[0], Cv[1]), h0, acc);
      acc = __ffma2_rn(make_float2(Cv[2], Cv[3]), h1, acc);
      *hp = make_float4(h0.x, h0.y, h1.x, h1.y);   // the new state goes back into the slot
    }
    float out = fmaf(Dd, uv, acc.x + acc.y);
    if (has_z) out *= silu<PRECISE>(zv);
    reinterpret_cast<IO*>(sl + W::kU)[c] = from_f32<IO>(out);   // y over this thread's own u
    // the slot's state tile and y row leave as two bulk stores once every thread has written them
    fence_async_smem();
    __syncthreads();
    if (c == 0) {
      bulk_store(p.state + b * p.sst[0] + d0 * 16, smem_u32(sl + W::kState), W::CH * 16 * 4);
      bulk_store(static_cast<IO*>(p.y) + b * p.sy[0] + d0, smem_u32(sl + W::kU), W::kSeq);
      bulk_commit();
    }
  }
  if (c == 0) bulk_wait<0>();   // the slots outlive their stores
}

// Whether the fast path takes these arguments (dense rows, 16-byte aligned bulk copies).
template <typename IO>
bool bulk_eligible(const StepProblem& p, int* Qout) {
  const int es = sizeof(IO);
  int Q = 0;
  switch (p.N) {
    case 4: Q = es == 4 ? 1 : 0; break;
    case 8: Q = 2; break;
    case 16: Q = 4; break;
    case 32: Q = 8; break;
    case 64: Q = 16; break;
    default: Q = 0;
  }
  if (!Q) return false;
  const int CH = 128 / Q;
  auto a16 = [](const void* ptr) { return reinterpret_cast<uintptr_t>(ptr) % 16 == 0; };
  if (p.D % CH != 0) return false;
  if (p.sst[2] != 1 || p.sst[1] != p.N || (p.sst[0] * 4) % 16 != 0 || !a16(p.state)) return false;
  const int64_t* seq[] = {p.su, p.sd, p.sz, p.sy};
  const void* sp[] = {p.u, p.delta, p.z, p.y};
  for (int i = 0; i < 4; ++i) {
    if (!sp[i]) continue;
    if (seq[i][1] != 1 || (seq[i][0] * es) % 16 != 0 || !a16(sp[i])) return false;
  }
  if (p.sB[1] != 1 || p.sC[1] != 1 || (p.sB[0] * es) % 16 != 0 || (p.sC[0] * es) % 16 != 0 || !a16(p.Bm) ||
      !a16(p.Cm))
    return false;
  if (p.sA[1] != 1 || (p.sA[0] * 4) % 16 != 0 || !a16(p.A)) return false;
  if (p.B > 65535LL * 1024) return false;
  *Qout = Q;
  return true;
}

template <typename IO, int Q, bool PRECISE>
cudaError_t launch_bulk(const StepProblem& p, cudaStream_t s) {
  constexpr int CH = 128 / Q;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t ranges = p.D / CH;
  // about 5 resident CTAs per SM; every CTA walks B / G batch rows
  int64_t G = (5 * (int64_t)sms + ranges - 1) / ranges;
  G = std::max<int64_t>(1, std::min<int64_t>(G, std::min<int64_t>(p.B, 65535)));
  state_update_bulk_kernel<IO, Q, PRECISE><<<dim3((unsigned)ranges, (unsigned)G), 128, 0, s>>>(p, (int)G,
                                                                                           device_status_ptr());
  return cudaGetLastError();
}

template <typename IO, bool PRECISE>
cudaError_t launch_wide(const StepProblem& p, cudaStream_t s) {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t ranges = p.D / WideSlot<IO>::CH;
  // about 5 resident CTAs per SM; every CTA walks B / G batch rows
  int64_t G = (5 * (int64_t)sms + ranges - 1) / ranges;
  G = std::max<int64_t>(1, std::min<int64_t>(G, std::min<int64_t>(p.B, 65535)));
  state_update_wide_kernel<IO, PRECISE><<<dim3((unsigned)ranges, (unsigned)G), 128, 0, s>>>(p, (int)G,
                                                                                          device_status_ptr());
  return cudaGetLastError();
}

template <typename IO, bool PRECISE>
cudaError_t launch_typed(const StepProblem& p, cudaStream_t s) {
  int Qb = 0;
  // the exact-ZOH input term is implemented in the per-item kernel only
  const bool bulk = !p.zoh && bulk_eligible<IO>(p, &Qb) && getenv("SSM_DECODE_PER_ITEM") == nullptr;
  if (bulk && p.N == 16 && p.D % WideSlot<IO>::CH == 0 && getenv("SSM_DECODE_QUAD") == nullptr)
    return launch_wide<IO, PRECISE>(p, s);
  if (bulk) {
    switch (Qb) {
      case 1:
        if constexpr (sizeof(IO) == 4) return launch_bulk<IO, 1, PRECISE>(p, s);
        break;   // not eligible for bf16 (B and C rows of 8 bytes)
      case 2: return launch_bulk<IO, 2, PRECISE>(p, s);
      case 4: return launch_bulk<IO, 4, PRECISE>(p, s);
      case 8: return launch_bulk<IO, 8, PRECISE>(p, s);
      default: return launch_bulk<IO, 16, PRECISE>(p, s);
    }
  }
  const int es = sizeof(IO);
  const bool quads = p.N % 4 == 0;
  const bool vec_state = quads && p.sst[2] == 1 && (p.sst[0] % 4 == 0) && (p.sst[1] % 4 == 0) &&
                         (reinterpret_cast<uintptr_t>(p.state) % 16 == 0);
  const int bc_align = 4 * es;   // bytes of four B (or C) values
  const bool vec_bc = quads && p.sB[1] == 1 && p.sC[1] == 1 && (p.sB[0] * es) % bc_align == 0 &&
                      (p.sC[0] * es) % bc_align == 0 && reinterpret_cast<uintptr_t>(p.Bm) % bc_align == 0 &&
                      reinterpret_cast<uintptr_t>(p.Cm) % bc_align == 0;
  const bool vec_a = quads && p.sA[1] == 1 && (p.sA[0] % 4 == 0) && (reinterpret_cast<uintptr_t>(p.A) % 16 == 0);
  const int nq = (int)((p.N + 3) / 4);
  int Q = 1;
  while (Q < nq) Q <<= 1;
  const int64_t items = p.B * p.D * Q;
  const int64_t threads = (items + ITEMS - 1) / ITEMS;
  const dim3 block(256);
  const dim3 grid((unsigned)((threads + 255) / 256));   // 256 threads: a multiple of every Q
  switch (Q) {
    case 1: state_update_kernel<IO, 1, PRECISE><<<grid, block, 0, s>>>(p, vec_state, vec_bc, vec_a); break;
    case 2: state_update_kernel<IO, 2, PRECISE><<<grid, block, 0, s>>>(p, vec_state, vec_bc, vec_a); break;
    case 4: state_update_kernel<IO, 4, PRECISE><<<grid, block, 0, s>>>(p, vec_state, vec_bc, vec_a); break;
    case 8: state_update_kernel<IO, 8, PRECISE><<<grid, block, 0, s>>>(p, vec_state, vec_bc, vec_a); break;
    default: state_update_kernel<IO, 16, PRECISE><<<grid, block, 0, s>>>(p, vec_state, vec_bc, vec_a); break;
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
