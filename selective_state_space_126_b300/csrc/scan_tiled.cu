// scan_tiled.cu -- the fused selective scan for sm_103a.
//
// What it computes: the selective SSM of the Mamba paper, per batch b,
// channel d and state n ("gitcode.csdn.net", section 2 for the recurrence and
// the diagonal A, section 3.2 for Delta/B/C as functions of the input and
// tau_Delta = softplus; "docs.ifdog.com", section "Discretisation" for
// Abar = exp(Delta A) and the numpy listing for Bbar x = Delta B u; section
// "Mamba architecture" for the silu gate).  Section 3.3.2 of the paper fuses
// discretisation, recurrence and the C product so that the (B, L, D, N)
// state never reaches HBM; this kernel keeps that property with a design of
// its own for this GPU:
//
//   * one CTA = 32*K threads = one batch row and CH = 32 channels; K threads
//     share a channel, each owning NS = NP/K states in registers.  Warp g holds
//     state group g of all 32 channels, so every read of B_t / C_t from shared
//     memory is a warp-uniform broadcast.  Small CTAs keep the work per SM even
//     (640 CTAs for 4 x 5120 channels on 148 SMs) and let the load, scan and
//     store phases of neighbouring CTAs overlap;
//   * the time axis is walked in tiles of T = 32 steps.  Per tile:
//       A. u / delta (and z) arrive through coalesced 16-byte loads issued one
//          tile ahead; Delta = softplus(delta + bias) and Delta*u are computed
//          once per (channel, t) and staged in shared memory.  The B and C
//          tiles (N x T, shared by every channel of the batch row) arrive by
//          TMA (cp.async.bulk.tensor, double-buffered on an mbarrier) and are
//          widened to fp32 in a [t][B|C][n] layout;
//       B. the scan: per step one SFU ex2 per state, Abar*h + (Delta u) B on
//          packed f32x2 FMAs, and the C contraction into a partial y;
//       C. the K partial outputs are summed, D*u added, multiplied by silu(z)
//          and written back with coalesced 16-byte stores.
//   * h stays in registers across tiles (never written to HBM, except the
//     optional final state and the chunk records below).
//
// Long sequences with too few channels to fill the GPU use three passes
// (the chunk-carry path): (1) MODE_RECORD scans every chunk from a zero
// state and records its end state and the chunk's sum of Delta; (2) a small
// carry kernel composes the chunks in order, h_in[c+1] = exp(A sum Delta_c)
// h_in[c] + h_end[c] (the associative combine of "docs.ifdog.com", section
// "Hardware-aware parallel scan", applied to whole chunks); (3) MODE_OUTPUT
// rescans each chunk from its true initial state and emits y.
#include <cstdio>

#include "device_math.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int CH = 32;   // channels per CTA, one per lane

// Minimum resident CTAs of 128 threads per SM the register allocation is sized for.
#ifndef SSM_TILED_MIN_BLOCKS
#define SSM_TILED_MIN_BLOCKS 3
#endif
constexpr int T = kTileT;
constexpr int MODE_OUTPUT = 0;
constexpr int MODE_RECORD = 1;
constexpr uint32_t kWaitLimit = 1u << 20;

struct TiledParams {
  int64_t B, D, L;
  int N;
  int nchunks;
  int64_t chunk_len;
  const void* u;
  const void* delta;
  const void* z;
  void* y;
  int64_t su0, su1, sd0, sd1, sz0, sz1, sy0, sy1;
  const float* A;
  int64_t sA0, sA1;
  const float* Dskip;
  const float* bias;
  const float* h0;
  int64_t sh00, sh01, sh02;
  float* h_last;
  int64_t shl0, shl1, shl2;
  float* rec_h;     // [B][D][nchunks][NP]: chunk end state (record pass) / chunk initial state (output pass)
  float* rec_s;     // [B][D][nchunks]: sum of Delta over the chunk
  int softplus;
  int bc_rank3;     // B/C tensor maps carry a batch dimension
  int* status;
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// Bounded wait on an mbarrier phase: false if the limit ran out.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t phase) {
  for (uint32_t i = 0; i < kWaitLimit; ++i) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(phase)
        : "memory");
    if (done) return true;
  }
  return false;
}

__device__ __forceinline__ void tma_load(uint32_t dst, const CUtensorMap* map, int x, int y, int z, bool rank3,
                                         uint32_t bar) {
  if (rank3) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
            dst),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
  } else {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"(map), "r"(x), "r"(y), "r"(bar)
        : "memory");
  }
}

// Shared-memory layout of one CTA (byte offsets from a 1024-aligned base).
template <typename IO, int K, int NS>
struct Smem {
  static constexpr int NP = K * NS;
  static constexpr int kRawStage = 2 * NP * T * (int)sizeof(IO);   // B and C tiles, N <= NP rows
  static constexpr int kRaw = 0;
  static constexpr int kBC = kRaw + 2 * kRawStage;                  // float [T][2][NP]
  static constexpr int kDT = kBC + T * 2 * NP * 4;                  // float2 [CH][T+2]
  static constexpr int kDTRow = T + 2;
  static constexpr int kPart = kDT + CH * kDTRow * 8;               // float [K][CH][T+4]
  static constexpr int kPartRow = T + 4;
  static constexpr int kBar = kPart + K * CH * kPartRow * 4;        // 2 x uint64
  static constexpr int kBytes = kBar + 16;
  static constexpr int kAlloc = kBytes + 1024;                      // slack for the 1024-byte alignment
};

template <typename IO, int K, int NS, int MODE, bool PRECISE>
__global__ void __launch_bounds__(32 * K, SSM_TILED_MIN_BLOCKS * 4 / K)
    scan_tiled_kernel(const __grid_constant__ TiledParams p, const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmC) {
  using S = Smem<IO, K, NS>;
  constexpr int kThreads = 32 * K;
  constexpr int NP = S::NP;
  constexpr int VEC = Vec16<IO>::kN;     // elements per 16-byte vector
  constexpr int VPR = T / VEC;           // vectors per channel row per tile
  constexpr int NV = CH * VPR / kThreads;
  static_assert(CH * VPR % kThreads == 0, "vector mapping");
  static_assert(NS % 4 == 0, "states per thread");

  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  float* bc_s = reinterpret_cast<float*>(smem + S::kBC);
  float2* dt_s = reinterpret_cast<float2*>(smem + S::kDT);
  float* part_s = reinterpret_cast<float*>(smem + S::kPart);
  const uint32_t raw_base = smem_u32(smem + S::kRaw);
  const uint32_t bar_base = smem_u32(smem + S::kBar);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int g = warp;                            // state group of this warp
  const int c = lane;                            // channel within the CTA
  const int64_t b = blockIdx.z;
  const int chunk = blockIdx.y;
  const int64_t d0 = (int64_t)blockIdx.x * CH;
  const int64_t d = d0 + c;
  const bool valid = d < p.D;
  const int N = p.N;

  const int64_t t_begin = (int64_t)chunk * p.chunk_len;
  const int64_t t_end = min(p.L, t_begin + p.chunk_len);
  const int ntiles = (int)((t_end - t_begin + T - 1) / T);

  // ---- per-thread state: A * log2(e) and h for this thread's NS states ----
  float2 A2[NS / 2], h[NS / 2];
#pragma unroll
  for (int i = 0; i < NS; ++i) {
    const int n = g * NS + i;
    float a = 0.f, hv = 0.f;
    if (valid && n < N) {
      a = p.A[d * p.sA0 + n * p.sA1] * kLog2e;
      if (MODE == MODE_OUTPUT) {
        if (chunk == 0) {
          if (p.h0) hv = p.h0[b * p.sh00 + d * p.sh01 + n * p.sh02];
        } else {
          hv = p.rec_h[((b * p.D + d) * p.nchunks + chunk) * NP + n];
        }
      }
    }
    if (i & 1) { A2[i / 2].y = a; h[i / 2].y = hv; }
    else { A2[i / 2].x = a; h[i / 2].x = hv; }
  }

  // ---- per-vector constants for the load / store stages ----
  int vc[NV], vt[NV];
  bool vvalid[NV];
  float vbias[NV], vD[NV];
  const IO* u_ptr[NV];
  const IO* d_ptr[NV];
  const IO* z_ptr[NV];
  IO* y_ptr[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int v = tid + i * kThreads;
    vc[i] = v / VPR;
    vt[i] = (v % VPR) * VEC;
    const int64_t dv = d0 + vc[i];
    vvalid[i] = dv < p.D;
    const int64_t dvc = vvalid[i] ? dv : 0;
    vbias[i] = p.bias ? p.bias[dvc] : 0.f;
    vD[i] = p.Dskip ? p.Dskip[dvc] : 0.f;
    u_ptr[i] = static_cast<const IO*>(p.u) + b * p.su0 + dvc * p.su1 + vt[i];
    d_ptr[i] = static_cast<const IO*>(p.delta) + b * p.sd0 + dvc * p.sd1 + vt[i];
    z_ptr[i] = p.z ? static_cast<const IO*>(p.z) + b * p.sz0 + dvc * p.sz1 + vt[i] : nullptr;
    y_ptr[i] = static_cast<IO*>(p.y) + b * p.sy0 + dvc * p.sy1 + vt[i];
  }

  // ---- one-time set-up: zero the B/C tile (padded states stay zero), barriers ----
  for (int i = tid; i < T * 2 * NP; i += kThreads) bc_s[i] = 0.f;
  if (tid == 0) {
    mbar_init(bar_base, 1);
    mbar_init(bar_base + 8, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  const uint32_t tile_bytes = 2u * (uint32_t)N * T * (uint32_t)sizeof(IO);
  const int bc_z = p.bc_rank3 ? (int)b : 0;
  auto issue_bc = [&](int tile, int stage) {
    const int x = (int)(t_begin + (int64_t)tile * T);
    const uint32_t bar = bar_base + 8 * stage;
    const uint32_t dst = raw_base + stage * S::kRawStage;
    mbar_expect_tx(bar, tile_bytes);
    tma_load(dst, &tmB, x, 0, bc_z, p.bc_rank3, bar);
    tma_load(dst + NP * T * (uint32_t)sizeof(IO), &tmC, x, 0, bc_z, p.bc_rank3, bar);
  };
  if (tid == 0 && ntiles > 0) issue_bc(0, 0);

  // ---- register prefetch of the first tile's u / delta / z ----
  uint4 pu[NV], pd[NV], pz[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const bool in = vvalid[i] && (t_begin + vt[i] < t_end);
    pu[i] = in ? ldg_nc_v4(u_ptr[i] + t_begin) : make_uint4(0, 0, 0, 0);
    pd[i] = in ? ldg_nc_v4(d_ptr[i] + t_begin) : make_uint4(0, 0, 0, 0);
    pz[i] = (in && p.z) ? ldg_nc_v4(z_ptr[i] + t_begin) : make_uint4(0, 0, 0, 0);
  }

  float dsum = 0.f;
  for (int k = 0; k < ntiles; ++k) {
    const int64_t t0 = t_begin + (int64_t)k * T;
    const int stage = k & 1;
    const uint32_t phase = (uint32_t)(k >> 1) & 1u;
    if (tid == 0 && k + 1 < ntiles) issue_bc(k + 1, stage ^ 1);

    // ---- stage A: Delta and Delta*u for this tile -> shared memory ----
    float cu[NV][VEC], cz[NV][VEC];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      float dv[VEC];
      unpack16(pu[i], cu[i]);
      unpack16(pd[i], dv);
      if (MODE == MODE_OUTPUT) unpack16(pz[i], cz[i]);
      float2 out[VEC];
#pragma unroll
      for (int j = 0; j < VEC; ++j) {
        const bool in = vvalid[i] && (t0 + vt[i] + j < t_end);
        const float dt = in ? delta_of<PRECISE>(dv[j], vbias[i], p.softplus) : 0.f;
        out[j] = make_float2(dt, dt * cu[i][j]);
      }
      float4* dst = reinterpret_cast<float4*>(dt_s + vc[i] * S::kDTRow + vt[i]);
#pragma unroll
      for (int j = 0; j < VEC / 2; ++j) dst[j] = make_float4(out[2 * j].x, out[2 * j].y, out[2 * j + 1].x, out[2 * j + 1].y);
    }
    // prefetch the next tile
    if (k + 1 < ntiles) {
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int64_t tn = t0 + T;
        const bool in = vvalid[i] && (tn + vt[i] < t_end);
        pu[i] = in ? ldg_nc_v4(u_ptr[i] + tn) : make_uint4(0, 0, 0, 0);
        pd[i] = in ? ldg_nc_v4(d_ptr[i] + tn) : make_uint4(0, 0, 0, 0);
        if (MODE == MODE_OUTPUT) pz[i] = (in && p.z) ? ldg_nc_v4(z_ptr[i] + tn) : make_uint4(0, 0, 0, 0);
      }
    }

    // ---- stage A': B / C tile (TMA) -> fp32 [t][B|C][n] ----
    const bool ok = mbar_wait(bar_base + 8 * stage, phase);
    if (ok) {
      const unsigned char* raw = smem + S::kRaw + stage * S::kRawStage;
      const int per_tensor = N * VPR;                     // 16-byte vectors per tile
      for (int v = tid; v < 2 * per_tensor; v += kThreads) {
        const int tensor = v >= per_tensor ? 1 : 0;        // 0: B, 1: C (C starts at row NP)
        const int rem = v - tensor * per_tensor;
        const int n = rem / VPR;
        const int tv = (rem % VPR) * VEC;
        float f[VEC];
        unpack16(*reinterpret_cast<const uint4*>(raw + (size_t)tensor * NP * T * sizeof(IO) + (size_t)rem * 16), f);
#pragma unroll
        for (int j = 0; j < VEC; ++j) bc_s[(tv + j) * 2 * NP + tensor * NP + n] = f[j];
      }
    } else {
      record_status(p.status, SSM_ERR_TIMEOUT);
    }
    if (__syncthreads_or(!ok)) {
      // a TMA copy never completed: give the other stage a bounded wait, then leave
      if (tid == 0 && k + 1 < ntiles) (void)mbar_wait(bar_base + 8 * (stage ^ 1), (uint32_t)((k + 1) >> 1) & 1u);
      return;
    }

    // ---- stage B: the recurrence over T steps ----
    {
      const float* dtrow = reinterpret_cast<const float*>(dt_s + c * S::kDTRow);
      float* prow = part_s + (g * CH + c) * S::kPartRow;
#pragma unroll 2
      for (int t = 0; t < T; t += 4) {
        float yv[4];
#pragma unroll
        for (int j = 0; j < 4; j += 2) {
          const float4 dd = *reinterpret_cast<const float4*>(dtrow + 2 * (t + j));
#pragma unroll
          for (int s = 0; s < 2; ++s) {
            const float dt = s ? dd.z : dd.x;
            const float du = s ? dd.w : dd.y;
            const float* Bt = bc_s + (t + j + s) * 2 * NP + g * NS;
            const float2 dt2 = make_float2(dt, dt);
            const float2 du2 = make_float2(du, du);
            float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
            for (int q = 0; q < NS; q += 4) {
              const float4 bq = *reinterpret_cast<const float4*>(Bt + q);
              const float2 x0 = __fmul2_rn(dt2, A2[q / 2]);
              const float2 x1 = __fmul2_rn(dt2, A2[q / 2 + 1]);
              const float2 a0 = make_float2(ex2_approx(x0.x), ex2_approx(x0.y));
              const float2 a1 = make_float2(ex2_approx(x1.x), ex2_approx(x1.y));
              h[q / 2] = __ffma2_rn(a0, h[q / 2], __fmul2_rn(du2, make_float2(bq.x, bq.y)));
              h[q / 2 + 1] = __ffma2_rn(a1, h[q / 2 + 1], __fmul2_rn(du2, make_float2(bq.z, bq.w)));
              if (MODE == MODE_OUTPUT) {
                const float4 cq = *reinterpret_cast<const float4*>(Bt + NP + q);
                acc0 = __ffma2_rn(make_float2(cq.x, cq.y), h[q / 2], acc0);
                acc1 = __ffma2_rn(make_float2(cq.z, cq.w), h[q / 2 + 1], acc1);
              }
            }
            yv[j + s] = (acc0.x + acc1.x) + (acc0.y + acc1.y);
            if (MODE == MODE_RECORD) dsum += dt;
          }
        }
        if (MODE == MODE_OUTPUT) *reinterpret_cast<float4*>(prow + t) = make_float4(yv[0], yv[1], yv[2], yv[3]);
      }
    }
    __syncthreads();

    // ---- stage C: sum the K partials, D skip, gate, store ----
    if (MODE == MODE_OUTPUT) {
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        if (!(vvalid[i] && (t0 + vt[i] < t_end))) continue;
        float yv[VEC];
#pragma unroll
        for (int j = 0; j < VEC; j += 4) {
          float4 s4 = *reinterpret_cast<const float4*>(part_s + vc[i] * S::kPartRow + vt[i] + j);
#pragma unroll
          for (int gg = 1; gg < K; ++gg) {
            const float4 o = *reinterpret_cast<const float4*>(part_s + (gg * CH + vc[i]) * S::kPartRow + vt[i] + j);
            s4.x += o.x; s4.y += o.y; s4.z += o.z; s4.w += o.w;
          }
          yv[j] = s4.x; yv[j + 1] = s4.y; yv[j + 2] = s4.z; yv[j + 3] = s4.w;
        }
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
          float o = fmaf(vD[i], cu[i][j], yv[j]);
          if (p.z) o *= silu<PRECISE>(cz[i][j]);
          yv[j] = o;
        }
        stg_v4(y_ptr[i] + t0, pack16(yv));
      }
    }
  }

  // ---- epilogue: final state or chunk record ----
  if (MODE == MODE_OUTPUT) {
    if (p.h_last && valid && chunk == p.nchunks - 1) {
#pragma unroll
      for (int i = 0; i < NS; ++i) {
        const int n = g * NS + i;
        if (n < N) p.h_last[b * p.shl0 + d * p.shl1 + n * p.shl2] = (i & 1) ? h[i / 2].y : h[i / 2].x;
      }
    }
  } else {
    if (valid) {
      const int64_t r = (b * p.D + d) * p.nchunks + chunk;
#pragma unroll
      for (int i = 0; i < NS; ++i) {
        const int n = g * NS + i;
        if (n < NP) p.rec_h[r * NP + n] = (i & 1) ? h[i / 2].y : h[i / 2].x;
      }
      if (g == 0) p.rec_s[r] = dsum;
    }
  }
}

// Chunk carry: turns the per-chunk end states (from zero) into each chunk's
// true initial state, in chunk order.  One thread per (b, d, n).
__global__ void __launch_bounds__(256) chunk_carry_kernel(const TiledParams p, int NP) {
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t total = p.B * p.D * NP;
  if (gid >= total) return;
  const int n = (int)(gid % NP);
  const int64_t c = gid / NP;
  const int64_t b = c / p.D, d = c % p.D;
  if (n >= p.N) return;
  const float a2 = p.A[d * p.sA0 + n * p.sA1] * kLog2e;
  float hcur = p.h0 ? p.h0[b * p.sh00 + d * p.sh01 + n * p.sh02] : 0.f;
  for (int k = 0; k < p.nchunks; ++k) {
    const int64_t r = c * p.nchunks + k;
    const float hend = p.rec_h[r * NP + n];
    p.rec_h[r * NP + n] = hcur;
    hcur = fmaf(ex2_approx(a2 * p.rec_s[r]), hcur, hend);
  }
}

template <typename IO, int K, int NS, int MODE, bool PRECISE>
cudaError_t launch_one(const TiledParams& tp, const CUtensorMap& mB, const CUtensorMap& mC, dim3 grid,
                       cudaStream_t s) {
  using S = Smem<IO, K, NS>;
  auto kern = scan_tiled_kernel<IO, K, NS, MODE, PRECISE>;
  static unsigned long long attr_set = 0;   // one bit per device; a racing duplicate set is harmless
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(__atomic_load_n(&attr_set, __ATOMIC_ACQUIRE) & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kAlloc);
    if (e != cudaSuccess) return e;
    __atomic_fetch_or(&attr_set, bit, __ATOMIC_RELEASE);
  }
  kern<<<grid, 32 * K, S::kAlloc, s>>>(tp, mB, mC);
  return cudaGetLastError();
}

template <typename IO, int K, int NS, bool PRECISE>
cudaError_t launch_shape(const ScanProblem& p, const ScanPlan& plan, TiledParams& tp, const CUtensorMap& mB,
                         const CUtensorMap& mC, cudaStream_t s) {
  constexpr int NP = K * NS;
  const dim3 grid((unsigned)((p.D + CH - 1) / CH), (unsigned)plan.nchunks, (unsigned)p.B);
  cudaError_t e;
  if (plan.nchunks > 1) {
    e = launch_one<IO, K, NS, MODE_RECORD, PRECISE>(tp, mB, mC, grid, s);
    if (e != cudaSuccess) return e;
    const int64_t total = p.B * p.D * NP;
    chunk_carry_kernel<<<(unsigned)((total + 255) / 256), 256, 0, s>>>(tp, NP);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return launch_one<IO, K, NS, MODE_OUTPUT, PRECISE>(tp, mB, mC, grid, s);
}

bool encode_bc_map(CUtensorMap* map, const void* base, const int64_t* strides, const ScanProblem& p) {
  EncodeTiledFn enc = get_encode_tiled();
  if (!enc) return false;
  const int es = p.io == SSM_F32 ? 4 : 2;
  const CUtensorMapDataType dt = p.io == SSM_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const bool rank3 = strides[0] != 0 && p.B > 1;
  cuuint64_t dims[3] = {(cuuint64_t)p.L, (cuuint64_t)p.N, (cuuint64_t)p.B};
  cuuint64_t gstr[2] = {(cuuint64_t)(strides[1] * es), (cuuint64_t)(strides[0] * es)};
  cuuint32_t box[3] = {(cuuint32_t)T, (cuuint32_t)p.N, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, dt, rank3 ? 3 : 2, const_cast<void*>(base), dims, gstr, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <typename IO, bool PRECISE>
cudaError_t launch_typed(const ScanProblem& p, const ScanPlan& plan, TiledParams& tp, const CUtensorMap& mB,
                         const CUtensorMap& mC, cudaStream_t s) {
  const int K = plan.shape.K, NS = plan.shape.NS;
  if (K == 1 && NS == 16) return launch_shape<IO, 1, 16, PRECISE>(p, plan, tp, mB, mC, s);
  if (K == 2 && NS == 8) return launch_shape<IO, 2, 8, PRECISE>(p, plan, tp, mB, mC, s);
  if (K == 4 && NS == 4) return launch_shape<IO, 4, 4, PRECISE>(p, plan, tp, mB, mC, s);
  if (K == 4 && NS == 8) return launch_shape<IO, 4, 8, PRECISE>(p, plan, tp, mB, mC, s);
  if (K == 4 && NS == 16) return launch_shape<IO, 4, 16, PRECISE>(p, plan, tp, mB, mC, s);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_scan_tiled(const ScanProblem& p, const ScanPlan& plan, void* workspace, cudaStream_t s) {
  TiledParams tp{};
  tp.B = p.B; tp.D = p.D; tp.L = p.L; tp.N = (int)p.N;
  tp.nchunks = (int)plan.nchunks;
  tp.chunk_len = plan.nchunks > 1 ? plan.chunk_len : p.L;
  tp.u = p.u; tp.delta = p.delta; tp.z = p.z; tp.y = p.y;
  tp.su0 = p.su[0]; tp.su1 = p.su[1];
  tp.sd0 = p.sd[0]; tp.sd1 = p.sd[1];
  tp.sz0 = p.sz[0]; tp.sz1 = p.sz[1];
  tp.sy0 = p.sy[0]; tp.sy1 = p.sy[1];
  tp.A = p.A; tp.sA0 = p.sA[0]; tp.sA1 = p.sA[1];
  tp.Dskip = p.Dskip; tp.bias = p.bias;
  tp.h0 = p.h0; tp.sh00 = p.sh0[0]; tp.sh01 = p.sh0[1]; tp.sh02 = p.sh0[2];
  tp.h_last = p.h_last; tp.shl0 = p.shl[0]; tp.shl1 = p.shl[1]; tp.shl2 = p.shl[2];
  tp.softplus = p.softplus ? 1 : 0;
  tp.status = device_status_ptr();
  const int NP = plan.shape.K * plan.shape.NS;
  if (plan.nchunks > 1) {
    float* ws = static_cast<float*>(workspace);
    tp.rec_h = ws;
    tp.rec_s = ws + p.B * p.D * plan.nchunks * NP;
  }
  CUtensorMap mB, mC;
  if (!encode_bc_map(&mB, p.Bm, p.sB, p) || !encode_bc_map(&mC, p.Cm, p.sC, p)) return cudaErrorInvalidValue;
  tp.bc_rank3 = (p.sB[0] != 0 && p.B > 1) ? 1 : 0;
  if ((p.sC[0] != 0 && p.B > 1) != (tp.bc_rank3 == 1)) return cudaErrorInvalidValue;  // planned away
  if (p.io == SSM_F32) return launch_typed<float, true>(p, plan, tp, mB, mC, s);
  return launch_typed<__nv_bfloat16, false>(p, plan, tp, mB, mC, s);
}

size_t tiled_smem_bytes(ssm_dtype_t io, int K, int NS) {
#define SSM_SMEM_CASE(k, ns)                                                         \
  if (K == k && NS == ns)                                                            \
    return io == SSM_F32 ? (size_t)Smem<float, k, ns>::kAlloc : (size_t)Smem<__nv_bfloat16, k, ns>::kAlloc;
  SSM_SMEM_CASE(1, 16)
  SSM_SMEM_CASE(2, 8)
  SSM_SMEM_CASE(4, 4)
  SSM_SMEM_CASE(4, 8)
  SSM_SMEM_CASE(4, 16)
#undef SSM_SMEM_CASE
  return 0;
}

}  // namespace ssm
