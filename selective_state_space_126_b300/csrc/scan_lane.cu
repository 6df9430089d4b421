// scan_lane.cu -- the fused selective scan for N <= 16: one warp per CTA,
// one channel per lane, every state of the channel in that lane's registers.
//
// What it computes: per batch b, channel d and state n, the selective SSM of
// the Mamba paper ("gitcode.csdn.net", section 2 for the recurrence and the
// diagonal A, section 3.2 for the input-dependent Delta, B, C and
// tau_Delta = softplus, section 3.6 for the Delta bias; "docs.ifdog.com",
// section "Discretisation" for Abar = exp(Delta A) and the numpy listing for
// Bbar x = Delta B u, section "Mamba architecture" for the silu gate):
//   Delta_t = softplus(delta_t + bias),  h_t = exp(Delta_t A) h_{t-1} + Delta_t B_t u_t,
//   y_t = (C_t . h_t + D u_t) * silu(z_t).
// As in section 3.3.2 of the paper the state lives only on chip.
//
// Design for this GPU.  The recurrence is bound by how fast operands reach
// the lanes' registers, the SFU (one ex2 per state update) and the FMA pipe.
// A lane that owns a whole channel needs no data from other lanes except
// B_t and C_t, which every lane reads with the same address (a broadcast,
// the cheapest shared-memory read).  So:
//   * each CTA is one warp: 32 channels of one batch row (or of one chunk of
//     the sequence on the chunked path);
//   * u, delta, z come by TMA as (32 steps x 32 channels) boxes with the
//     64-byte swizzle, so that lane c can read 8 consecutive steps of its own
//     row with one conflict-free 16-byte load; B and C come as (32 steps x N)
//     boxes; three ring slots keep two tiles in flight ahead of the compute;
//   * per tile the warp widens B and C to fp32 in a [t][B | C] layout; per
//     step each lane computes Delta and Delta*u of its channel, 16 ex2 and
//     16 fused updates on packed f32x2 FMAs, the C contraction, D u and the
//     gate, all in registers;
//   * y goes through a swizzled staging box and leaves by a TMA store.
// No CTA-wide barrier is needed: the warp synchronises with __syncwarp and
// with the TMA mbarriers (whose waits are bounded).
//
// The chunked path (long sequences with few channels) uses the same kernel
// in MODE_RECORD (end state and sum of Delta of every chunk, from a zero
// state), a carry kernel that composes the chunks in order, and MODE_OUTPUT
// from each chunk's true initial state.
#include <cstring>

#include "async_copy.cuh"
#include "device_math.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int LT = 32;      // time steps per tile
constexpr int LS = 3;       // TMA ring slots
constexpr int NPL = 16;     // states per lane (N <= 16; missing states are zero)
constexpr int MODE_OUTPUT = 0;
constexpr int MODE_RECORD = 1;

// 16-byte chunks of a tile row unrolled together (1 = one chunk of steps at a time).
#ifndef SSM_LANE_UNROLL
#define SSM_LANE_UNROLL 1
#endif
constexpr int kLaneUnroll = SSM_LANE_UNROLL;

struct LaneParams {
  int64_t B, D, L;
  int N;
  int nchunks;
  int64_t chunk_len;
  const float* A;
  int64_t sA0, sA1;
  const float* Dskip;
  const float* bias;
  const float* h0;
  int64_t sh00, sh01, sh02;
  float* h_last;
  int64_t shl0, shl1, shl2;
  float* rec_h;     // [B][D][nchunks][16]: chunk end state (record pass) / chunk initial state (output pass)
  float* rec_s;     // [B][D][nchunks]: sum of Delta over the chunk
  int softplus;
  int has_z;
  int seq_rank3;    // u / delta / z maps carry a batch dimension
  int bc_rank3;     // B / C maps carry a batch dimension
  int y_rank3;      // the y map carries a batch dimension
  int* status;
};

struct LaneMaps {
  CUtensorMap u, delta, z, B, C, y;
};

// Shared memory of one CTA (offsets from a 1024-byte aligned base; every TMA
// box starts on a 1024-byte boundary, as the swizzled layouts need).
template <typename IO>
struct LaneSmem {
  static constexpr int ROWB = LT * (int)sizeof(IO);   // bytes per box row: 64 (bf16) or 128 (fp32)
  static constexpr int SEQ = 32 * ROWB;               // (32 channels x 32 steps)
  static constexpr int BC = NPL * ROWB;               // (16 states x 32 steps)
  static constexpr int kU = 0, kDelta = SEQ, kZ = 2 * SEQ, kB = 3 * SEQ, kC = 3 * SEQ + BC;
  static constexpr int kSlot = (3 * SEQ + 2 * BC + 1023) / 1024 * 1024;
  static constexpr int kRing = 0;
  static constexpr int kY = kRing + LS * kSlot;       // two y staging boxes
  static constexpr int kBCT = kY + 2 * SEQ;           // float [LT][32]: B_t[n] at n, C_t[n] at 16 + n
  static constexpr int kBar = kBCT + LT * 32 * 4;
  static constexpr int kBytes = kBar + 8 * LS;
  static constexpr int kAlloc = kBytes + 1024;
  static_assert(SEQ % 1024 == 0 && BC % 1024 == 0, "box alignment");
};

// Byte offset of 16-byte chunk `chunk` of row `row` in a box written by TMA
// with the 64-byte (rows of 64 bytes) or 128-byte (rows of 128 bytes)
// swizzle: the chunk index is XOR-ed with address bits 7.. of the row start.
template <int ROWB>
__device__ __forceinline__ int swz(int row, int chunk) {
  if (ROWB == 64) return row * 64 + ((chunk ^ ((row >> 1) & 3)) << 4);
  return row * 128 + ((chunk ^ (row & 7)) << 4);
}

template <typename IO, int MODE, bool PRECISE>
__global__ void __launch_bounds__(32) scan_lane_kernel(const __grid_constant__ LaneParams p,
                                                       const __grid_constant__ LaneMaps tm) {
  using S = LaneSmem<IO>;
  constexpr int ROWB = S::ROWB;
  constexpr int VEC = 16 / (int)sizeof(IO);   // steps per 16-byte chunk
  constexpr int NCH = LT / VEC;               // chunks per row

  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  float* bct = reinterpret_cast<float*>(smem + S::kBCT);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + S::kBar;

  const int lane = threadIdx.x;
  const int64_t b = blockIdx.z;
  const int chunk = blockIdx.y;
  const int64_t d0 = (int64_t)blockIdx.x * 32;
  const int64_t d = d0 + lane;
  const bool valid = d < p.D;
  const int N = p.N;
  const int64_t t_begin = (int64_t)chunk * p.chunk_len;
  const int64_t t_end = min(p.L, t_begin + p.chunk_len);
  const int ntiles = (int)((t_end - t_begin + LT - 1) / LT);

  // ---- the lane's channel: A * log2(e), initial state, bias, skip ----
  float2 A2[NPL / 2], h[NPL / 2];
#pragma unroll
  for (int n = 0; n < NPL; ++n) {
    float a = 0.f, hv = 0.f;
    if (valid && n < N) {
      a = p.A[d * p.sA0 + n * p.sA1] * kLog2e;
      if (MODE == MODE_OUTPUT) {
        if (chunk == 0) {
          if (p.h0) hv = p.h0[b * p.sh00 + d * p.sh01 + n * p.sh02];
        } else {
          hv = p.rec_h[((b * p.D + d) * p.nchunks + chunk) * NPL + n];
        }
      }
    }
    if (n & 1) { A2[n / 2].y = a; h[n / 2].y = hv; }
    else { A2[n / 2].x = a; h[n / 2].x = hv; }
  }
  const float bias = (valid && p.bias) ? p.bias[d] : 0.f;
  const float Dd = (valid && p.Dskip) ? p.Dskip[d] : 0.f;

  for (int i = lane; i < LT * 32; i += 32) bct[i] = 0.f;   // states >= N stay zero
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < LS; ++s) mbar_init(bar0 + 8 * s, 1);
    mbar_init_fence();
  }
  __syncwarp();

  const bool load_z = MODE == MODE_OUTPUT && p.has_z;
  const uint32_t tile_bytes = (uint32_t)((2 + (load_z ? 1 : 0)) * S::SEQ) +
                              (uint32_t)((MODE == MODE_OUTPUT ? 2 : 1) * N * ROWB);
  const int seq_z = p.seq_rank3 ? (int)b : 0;
  const int bc_z = p.bc_rank3 ? (int)b : 0;
  auto issue = [&](int tile) {
    const int x = (int)(t_begin + (int64_t)tile * LT);
    const int slot = tile % LS;
    const uint32_t bar = bar0 + 8 * slot;
    const uint32_t dst = sbase + S::kRing + slot * S::kSlot;
    mbar_expect_tx(bar, tile_bytes);
    tma_load(dst + S::kU, &tm.u, x, (int)d0, seq_z, p.seq_rank3, bar);
    tma_load(dst + S::kDelta, &tm.delta, x, (int)d0, seq_z, p.seq_rank3, bar);
    if (load_z) tma_load(dst + S::kZ, &tm.z, x, (int)d0, seq_z, p.seq_rank3, bar);
    tma_load(dst + S::kB, &tm.B, x, 0, bc_z, p.bc_rank3, bar);
    if (MODE == MODE_OUTPUT) tma_load(dst + S::kC, &tm.C, x, 0, bc_z, p.bc_rank3, bar);
  };
  if (lane == 0)
    for (int i = 0; i < LS && i < ntiles; ++i) issue(i);

  float dsum = 0.f;
  for (int k = 0; k < ntiles; ++k) {
    const int64_t t0 = t_begin + (int64_t)k * LT;
    const int slot = k % LS;
    const unsigned char* ring = smem + S::kRing + slot * S::kSlot;
    const bool ok = mbar_wait(bar0 + 8 * slot, (uint32_t)(k / LS) & 1u);
    if (__any_sync(0xffffffffu, !ok)) {
      // A copy never completed: record it, let the other copies in flight
      // land (bounded), and leave.
      if (lane == 0) {
        record_status(p.status, SSM_ERR_TIMEOUT);
        for (int j = k + 1; j < k + LS && j < ntiles; ++j) (void)mbar_wait(bar0 + 8 * (j % LS), (uint32_t)(j / LS) & 1u);
        if (MODE == MODE_OUTPUT) bulk_wait<0>();
      }
      return;
    }

    // ---- B and C of the tile, widened to fp32 as [t][B | C] ----
    {
      const int tensor = lane >> 4, n = lane & 15;   // lanes 0-15: B rows, 16-31: C rows
      if (n < N && (MODE == MODE_OUTPUT || tensor == 0)) {
        const unsigned char* src = ring + S::kB + tensor * S::BC;
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
          float f[VEC];
          unpack16(*reinterpret_cast<const uint4*>(src + swz<ROWB>(n, j)), f);
#pragma unroll
          for (int e = 0; e < VEC; ++e) bct[(j * VEC + e) * 32 + lane] = f[e];
        }
      }
    }
    // the staging box of this tile was last read by the store of tile k-2
    if (MODE == MODE_OUTPUT && k >= 2 && lane == 0) bulk_wait_read<1>();
    __syncwarp();

    unsigned char* ybox = smem + S::kY + (k & 1) * S::SEQ;
#pragma unroll kLaneUnroll
    for (int j = 0; j < NCH; ++j) {
      const int off = swz<ROWB>(lane, j);
      float uv[VEC], dv[VEC], zv[VEC], yo[VEC];
      unpack16(*reinterpret_cast<const uint4*>(ring + S::kU + off), uv);
      unpack16(*reinterpret_cast<const uint4*>(ring + S::kDelta + off), dv);
      if (load_z) unpack16(*reinterpret_cast<const uint4*>(ring + S::kZ + off), zv);
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        const int t = j * VEC + e;
        const float dt = (t0 + t < t_end) ? delta_of<PRECISE>(dv[e], bias, p.softplus) : 0.f;
        const float du = dt * uv[e];
        const float2 dt2 = make_float2(dt, dt), du2 = make_float2(du, du);
        const float* bt = bct + t * 32;
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int q = 0; q < NPL / 4; ++q) {
          const float4 bq = *reinterpret_cast<const float4*>(bt + 4 * q);
          const float2 x0 = __fmul2_rn(dt2, A2[2 * q]);
          const float2 x1 = __fmul2_rn(dt2, A2[2 * q + 1]);
          const float2 a0 = make_float2(ex2_approx(x0.x), ex2_approx(x0.y));
          const float2 a1 = make_float2(ex2_approx(x1.x), ex2_approx(x1.y));
          h[2 * q] = __ffma2_rn(a0, h[2 * q], __fmul2_rn(du2, make_float2(bq.x, bq.y)));
          h[2 * q + 1] = __ffma2_rn(a1, h[2 * q + 1], __fmul2_rn(du2, make_float2(bq.z, bq.w)));
          if (MODE == MODE_OUTPUT) {
            const float4 cq = *reinterpret_cast<const float4*>(bt + 16 + 4 * q);
            acc = __ffma2_rn(make_float2(cq.x, cq.y), h[2 * q], acc);
            acc = __ffma2_rn(make_float2(cq.z, cq.w), h[2 * q + 1], acc);
          }
        }
        if (MODE == MODE_RECORD) {
          dsum += dt;
        } else {
          float o = fmaf(Dd, uv[e], acc.x + acc.y);
          if (load_z) o *= silu<PRECISE>(zv[e]);
          yo[e] = o;
        }
      }
      if (MODE == MODE_OUTPUT) *reinterpret_cast<uint4*>(ybox + off) = pack16(yo);
    }
    __syncwarp();   // every lane is done with the ring slot (and has written its y)

    if (lane == 0 && k + LS < ntiles) issue(k + LS);
    if (MODE == MODE_OUTPUT) {
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store(&tm.y, smem_u32(ybox), (int)t0, (int)d0, p.y_rank3 ? (int)b : 0, p.y_rank3);
        bulk_commit();
      }
    }
  }
  if (MODE == MODE_OUTPUT && lane == 0) bulk_wait<0>();   // the staging boxes outlive their stores

  // ---- final state or chunk record ----
  if (MODE == MODE_OUTPUT) {
    if (p.h_last && valid && chunk == p.nchunks - 1) {
#pragma unroll
      for (int n = 0; n < NPL; ++n)
        if (n < N) p.h_last[b * p.shl0 + d * p.shl1 + n * p.shl2] = (n & 1) ? h[n / 2].y : h[n / 2].x;
    }
  } else if (valid) {
    const int64_t r = (b * p.D + d) * p.nchunks + chunk;
    float4* dst = reinterpret_cast<float4*>(p.rec_h + r * NPL);
#pragma unroll
    for (int q = 0; q < NPL / 4; ++q) dst[q] = make_float4(h[2 * q].x, h[2 * q].y, h[2 * q + 1].x, h[2 * q + 1].y);
    p.rec_s[r] = dsum;
  }
}

// Chunk carry: each chunk's end state (from zero) becomes the next chunk's
// true initial state, h_in[c+1] = exp(A sum Delta_c) h_in[c] + h_end[c], in
// chunk order.  One thread per (b, d, n).
__global__ void __launch_bounds__(256) lane_carry_kernel(const LaneParams p) {
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (gid >= p.B * p.D * NPL) return;
  const int n = (int)(gid % NPL);
  const int64_t c = gid / NPL;
  const int64_t b = c / p.D, d = c % p.D;
  if (n >= p.N) return;
  const float a2 = p.A[d * p.sA0 + n * p.sA1] * kLog2e;
  float hcur = p.h0 ? p.h0[b * p.sh00 + d * p.sh01 + n * p.sh02] : 0.f;
  for (int k = 0; k < p.nchunks; ++k) {
    const int64_t r = c * p.nchunks + k;
    const float hend = p.rec_h[r * NPL + n];
    p.rec_h[r * NPL + n] = hcur;
    hcur = fmaf(ex2_approx(a2 * p.rec_s[r]), hcur, hend);
  }
}

template <typename IO, int MODE, bool PRECISE>
cudaError_t launch_lane(const LaneParams& lp, const LaneMaps& tm, dim3 grid, cudaStream_t s) {
  auto kern = scan_lane_kernel<IO, MODE, PRECISE>;
  static unsigned long long attr_set = 0;   // one bit per device; a racing duplicate set is harmless
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(__atomic_load_n(&attr_set, __ATOMIC_ACQUIRE) & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, LaneSmem<IO>::kAlloc);
    if (e != cudaSuccess) return e;
    __atomic_fetch_or(&attr_set, bit, __ATOMIC_RELEASE);
  }
  kern<<<grid, 32, LaneSmem<IO>::kAlloc, s>>>(lp, tm);
  return cudaGetLastError();
}

template <typename IO, bool PRECISE>
cudaError_t launch_typed(const ScanProblem& p, const ScanPlan& plan, const LaneParams& lp, const LaneMaps& tm,
                         cudaStream_t s) {
  const dim3 grid((unsigned)((p.D + 31) / 32), (unsigned)plan.nchunks, (unsigned)p.B);
  cudaError_t e;
  if (plan.nchunks > 1) {
    e = launch_lane<IO, MODE_RECORD, PRECISE>(lp, tm, grid, s);
    if (e != cudaSuccess) return e;
    const int64_t total = p.B * p.D * NPL;
    lane_carry_kernel<<<(unsigned)((total + 255) / 256), 256, 0, s>>>(lp);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return launch_lane<IO, MODE_OUTPUT, PRECISE>(lp, tm, grid, s);
}

// Tensor map of a (batch, rows, L) tensor, time stride 1: box (32 steps x
// box_rows), swizzled so that a row's 16-byte chunks spread over the banks.
bool encode_map(CUtensorMap* map, const void* base, const int64_t* strides, int64_t rows, uint32_t box_rows,
                const ScanProblem& p, bool rank3) {
  EncodeTiledFn enc = get_encode_tiled();
  if (!enc) return false;
  const int es = p.io == SSM_F32 ? 4 : 2;
  const CUtensorMapDataType dt = p.io == SSM_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int64_t row_stride = rows > 1 ? strides[1] : (p.L + 7) / 8 * 8;   // unused over one row
  cuuint64_t dims[3] = {(cuuint64_t)p.L, (cuuint64_t)rows, (cuuint64_t)p.B};
  cuuint64_t gstr[2] = {(cuuint64_t)(row_stride * es), (cuuint64_t)(strides[0] * es)};
  cuuint32_t box[3] = {(cuuint32_t)LT, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapSwizzle swz = es == 2 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
  CUresult r = enc(map, dt, rank3 ? 3 : 2, const_cast<void*>(base), dims, gstr, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_scan_lane(const ScanProblem& p, const ScanPlan& plan, void* workspace, cudaStream_t s) {
  if (p.N > NPL) return cudaErrorInvalidValue;
  LaneParams lp{};
  lp.B = p.B; lp.D = p.D; lp.L = p.L; lp.N = (int)p.N;
  lp.nchunks = (int)plan.nchunks;
  lp.chunk_len = plan.nchunks > 1 ? plan.chunk_len : p.L;
  lp.A = p.A; lp.sA0 = p.sA[0]; lp.sA1 = p.sA[1];
  lp.Dskip = p.Dskip; lp.bias = p.bias;
  lp.h0 = p.h0; lp.sh00 = p.sh0[0]; lp.sh01 = p.sh0[1]; lp.sh02 = p.sh0[2];
  lp.h_last = p.h_last; lp.shl0 = p.shl[0]; lp.shl1 = p.shl[1]; lp.shl2 = p.shl[2];
  lp.softplus = p.softplus ? 1 : 0;
  lp.has_z = p.z ? 1 : 0;
  lp.status = device_status_ptr();
  if (plan.nchunks > 1) {
    float* ws = static_cast<float*>(workspace);
    lp.rec_h = ws;
    lp.rec_s = ws + p.B * p.D * plan.nchunks * NPL;
  }
  // the planner only takes this path when u, delta, z share one batch layout
  // kind (batched or broadcast) and B, C share another; y (an output) is
  // batched whenever B > 1
  lp.seq_rank3 = (p.su[0] != 0 && p.B > 1) ? 1 : 0;
  lp.bc_rank3 = (p.sB[0] != 0 && p.B > 1) ? 1 : 0;
  lp.y_rank3 = p.B > 1 ? 1 : 0;
  const bool r3 = lp.seq_rank3 == 1, b3 = lp.bc_rank3 == 1, y3 = lp.y_rank3 == 1;
  LaneMaps tm;
  std::memset(&tm, 0, sizeof(tm));
  if (!encode_map(&tm.u, p.u, p.su, p.D, 32, p, r3) || !encode_map(&tm.delta, p.delta, p.sd, p.D, 32, p, r3) ||
      (p.z && !encode_map(&tm.z, p.z, p.sz, p.D, 32, p, r3)) || !encode_map(&tm.y, p.y, p.sy, p.D, 32, p, y3) ||
      !encode_map(&tm.B, p.Bm, p.sB, p.N, (uint32_t)p.N, p, b3) ||
      !encode_map(&tm.C, p.Cm, p.sC, p.N, (uint32_t)p.N, p, b3))
    return cudaErrorInvalidValue;
  if (p.io == SSM_F32) return launch_typed<float, true>(p, plan, lp, tm, s);
  return launch_typed<__nv_bfloat16, false>(p, plan, lp, tm, s);
}

}  // namespace ssm
