// ssd.cu -- the Mamba-2 state-space-dual (SSD) layer on the fifth-generation tensor cores.
//
// What it computes ("Mamba close reading", alishangtian.com, section on SSD and
// Mamba-2: A is a scalar times the identity per head, heads as in multi-head
// attention, states 8x larger; "Mamba and state space models", docs.ifdog.com,
// section "Mamba-2 and structured duality"): per batch b, head h, head channel
// p (channel d = h P + p), state n and step t,
//     Delta_t  = softplus(delta[b,h,t] + bias[h]),   abar_t = exp(Delta_t a[h])
//     h_t[p,n] = abar_t h_{t-1}[p,n] + Delta_t B[b,t,n] x[b,d,t]
//     y[b,d,t] = (sum_n C[b,t,n] h_t[p,n] + D[h] x[b,d,t]) * silu(z[b,d,t]).
// The pages' duality: the map x -> y is multiplication by a semiseparable
// matrix, M = L o (C B^T) with the decay mask L[t,s] = exp(a (S_t - S_s)),
// S_t = Delta_0 + ... + Delta_t, for s <= t.  Cut the sequence into chunks of
// Q = 128 steps; within a chunk the masked product is dense, across chunks
// the state (N x P per head) carries the rest:
//     G        = C_c B_c^T                                  (Q x Q)
//     Y_diag   = (L_c o G) diag(Delta) X_c                  (Q x P)
//     Y_off    = diag(exp(a S_t)) C_c H_in                   (Q x P)
//     H_chunk  = B_c^T diag(exp(a (S_end - S_s)) Delta_s) X_c  (N x P)
//     H_out    = exp(a S_end) H_in + H_chunk.
// The four products are dense contractions and run as tcgen05.mma (bf16
// operands in shared memory, fp32 accumulators in tensor memory); the decay
// mask, the scalings, the state recurrence across chunks (fp32, in registers)
// and the output (D skip, gate) run on the CUDA cores.
//
// ssd_chunk_kernel: one CTA of 512 threads per (batch, head) walks its chunks
// in order, for P = 64 and N = 128 with bf16 I/O.  Threads i, i + 128, i + 256
// and i + 384 own time row i of the chunk (tensor-memory lane i of G, Y_diag,
// Y_off; each one quarter of the columns) and state row i (lane i of H_chunk,
// and a quarter each of the fp32 state H[i][0..63] in registers).  The phases
// between the MMAs are thread work with little parallelism inside a thread, so
// four warps per scheduler (rather than two) hide their latencies.  Per chunk:
//   1. TMA: C_c and B_c ((L, N) rows of 128 B, 128B swizzle, two 64-column
//      boxes each) and X_c ((P, L) rows, two 64-step boxes) -- each already
//      the K-major operand layout of the MMAs below -- and the gate's z_c,
//      on three barriers: the next chunk's B is loaded as soon as this one's
//      is consumed (after G), its C and X once every MMA of this chunk is
//      complete (they are read only by the MMAs), its z after the output;
//   2. Delta, the inclusive prefix sum S (warp shuffles and one shared step),
//      the weights w_s = exp(a (S_end - S_s)) Delta_s and the column terms
//      a S_s log2(e) - log2(Delta_s) of the scores; threads write the incoming
//      state H_in^T (K = n) in bf16;
//   3. MMA: G = C B^T, issued as soon as C and B are in, runs while the
//      threads write B~^T = w_s B^T (K = s) with 8 x 8 transposing loads and
//      stores (ldmatrix.trans / stmatrix); then H_chunk = B~^T X and
//      Y_off = C H_in are queued behind it (one commit each);
//   4. threads read G (tcgen05.ld), apply the causal decay mask and the step
//      factor, exp(a (S_t - S_s)) Delta_s, on the SFU and write the bf16
//      scores (K = s); blocks above the diagonal are written as zeros, and D
//      is added on the diagonal so that Y_diag carries the skip term D x_t;
//   5. MMA: Y_diag = scores X;
//   6. threads update H = exp(a S_end) H + H_chunk and emit
//      y = (Y_diag + exp(a S_t) Y_off) silu(z), coalesced along t.
// Other shapes and fp32 I/O take ssd_generic_kernel (one warp per channel, the
// recurrence itself).
#include <cstdio>
#include <cstring>

#include "device_math.cuh"
#include "scan_common.cuh"
#include "ssm_internal.h"
#include "tcgen05.cuh"

namespace ssm {
namespace {

constexpr int kQ = 128;          // chunk length
constexpr int kP = 64;           // head dimension of the tensor-core kernel
constexpr int kN = 128;          // state size of the tensor-core kernel
constexpr int kSsdThreads = 512;
constexpr int kCQ = kSsdThreads / kQ;  // threads per chunk row (column quarters)
constexpr int kPQ = kP / kCQ;          // head channels per thread (state update, output)
constexpr int kSQ = kQ / kCQ;          // steps per thread (weighted B^T, scores)
static_assert(kSQ % 32 == 0 && kPQ % 16 == 0, "thread split");
// The thread that issues the TMA loads and the MMAs: lane 0 of the warp for rows 0..31 and the last
// quarter of the steps, whose block of the causal score matrix is all zero, so that the time it
// spends issuing MMAs does not hold back the score phase.
constexpr int kIssuer = (kCQ - 1) * kQ;

struct SsdSmem {
  static constexpr int kC = 0;                 // C chunk: 2 x [128 t][64 n] bf16, swizzled
  static constexpr int kB = kC + 32768;        // B chunk: 2 x [128 s][64 n]
  static constexpr int kX = kB + 32768;        // X chunk: 2 x [64 p][64 s]
  static constexpr int kSP = kX + 16384;       // masked scores: 2 x [128 t][64 s]
  static constexpr int kBT = kSP + 32768;      // weighted B^T: 2 x [128 n][64 s]
  static constexpr int kSI = kBT + 32768;      // incoming state H_in^T: 2 x [64 p][64 n]
  static constexpr int kZ = kSI + 16384;       // z chunk: 2 x [64 p][64 t] (the gate)
  static constexpr int kDelta = kZ + 16384;    // float [128]
  static constexpr int kCum = kDelta + 512;    // float [128]
  static constexpr int kW = kCum + 512;        // float [128]
  static constexpr int kAS = kW + 512;         // float [128]: -a S_s log2(e), plus log2(Delta_s) under softplus
  static constexpr int kWarp = kAS + 512;      // float [4] warp totals of the prefix sum
  static constexpr int kBar = kWarp + 16;      // 6 mbarriers: TMA (C, X), TMA (B), G, (H_chunk, Y_off), Y_diag, TMA (z)
  static constexpr int kTaddr = kBar + 48;
  static constexpr int kBytes = kTaddr + 16;
  static constexpr int kAlloc = kBytes + 1024;
};

// tensor-memory columns of the accumulators (lanes = rows)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColG = 0, kColYd = 128, kColYo = 192, kColH = 256;

// Four 8 x 8 bf16 matrices from shared memory, transposed on the way (lane l gives the address of
// row l % 8 of matrix l / 8); register m of lane l holds elements (2 (l % 4), l / 4) and
// (2 (l % 4) + 1, l / 4) of matrix m, the first in the low half.
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&v)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
               : "r"(addr));
}

// Four 8 x 8 bf16 matrices to shared memory (lane l gives the address of row l % 8 of matrix l / 8);
// register m of lane l holds elements (l / 4, 2 (l % 4)) and (l / 4, 2 (l % 4) + 1) of matrix m.
__device__ __forceinline__ void stsm_x4(uint32_t addr, const uint32_t (&v)[4]) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v[0]), "r"(v[1]),
               "r"(v[2]), "r"(v[3])
               : "memory");
}

// (lo, hi) bf16 pair times (w.x, w.y) in fp32, rounded back to a bf16 pair.
__device__ __forceinline__ uint32_t scale_bf16x2(uint32_t v, float2 w) {
  const float lo = __uint_as_float(v << 16) * w.x, hi = __uint_as_float(v & 0xffff0000u) * w.y;
  const __nv_bfloat162 r = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&r);
}

struct SsdMaps {
  CUtensorMap x, z, B, C;
};

__global__ void __launch_bounds__(kSsdThreads, 1)
    ssd_chunk_kernel(const __grid_constant__ SsdProblem p, const __grid_constant__ SsdMaps tm) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  using S = SsdSmem;
  float* sDelta = reinterpret_cast<float*>(smem + S::kDelta);
  float* sCum = reinterpret_cast<float*>(smem + S::kCum);
  float* sW = reinterpret_cast<float*>(smem + S::kW);
  float* sAS = reinterpret_cast<float*>(smem + S::kAS);
  float* sWarp = reinterpret_cast<float*>(smem + S::kWarp);
  const uint32_t bar_tma = smem_u32(smem + S::kBar), bar_tmab = bar_tma + 8, bar_g = bar_tma + 16,
                 bar_ho = bar_tma + 24, bar_d = bar_tma + 32, bar_tmaz = bar_tma + 40;
  uint32_t* taddr_s = reinterpret_cast<uint32_t*>(smem + S::kTaddr);

  // thread = (row r, quarter cq): row r is time step r of the chunk and state index r; the quarter
  // picks steps [kSQ cq, kSQ cq + kSQ) of the score row and head channels [kPQ cq, kPQ cq + kPQ);
  // warp w reaches tensor-memory lanes 32 (w % 4) .. + 31, which are its rows
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = tid & (kQ - 1), cq = tid / kQ;
  const int64_t bh = blockIdx.x;
  const int64_t b = bh / p.H, h = bh % p.H;
  const int nchunks = (int)((p.L + kQ - 1) / kQ);
  const float a2 = p.a[h] * kLog2e;
  const float bias = p.bias ? p.bias[h] : 0.f;
  const float Dh = p.Dskip ? p.Dskip[h] : 0.f;

  if (tid == 0) {
    for (int i = 0; i < 6; ++i) mbar_init(bar_tma + 8 * i, 1);
    mbar_init_fence();
  }
  if (warp == 0) tmem_alloc(smem_u32(taddr_s), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *taddr_s;
  const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;   // this warp's 32 tensor-memory lanes: rows r

  // state H[r][kPQ cq .. kPQ cq + kPQ - 1] (state row n = r, head channels p), fp32 in registers
  float H[kPQ];
#pragma unroll
  for (int j = 0; j < kPQ; ++j)
    H[j] = p.h0 ? p.h0[b * p.sh0[0] + h * p.sh0[1] + (kPQ * cq + j) * p.sh0[2] + r * p.sh0[3]] : 0.f;

  // the issuing thread tracks the copies (chunk index, or -1) and MMA groups in flight for a bounded
  // drain on failure
  const bool issuer = tid == kIssuer;
  int cx_pend = -1, z_pend = -1, b_pend = -1;
  bool g_out = false, ho_out = false, d_out = false;
  // C and X of chunk c: read only by the MMAs, so the next chunk's can land as soon as Y_diag (the
  // last MMA to read them) is complete
  auto issue_cx = [&](int c) {
    const int t0 = c * kQ;
    mbar_expect_tx(bar_tma, 2 * 16384 + 2 * 8192);
    for (int j = 0; j < 2; ++j) {
      tma_load(smem_u32(smem + S::kC + j * 16384), &tm.C, 64 * j, t0, (int)b, true, bar_tma);
      tma_load(smem_u32(smem + S::kX + j * 8192), &tm.x, t0 + 64 * j, (int)(h * kP), (int)b, true, bar_tma);
    }
    cx_pend = c;
  };
  // z of chunk c: read by the threads in the output phase, so the next chunk's lands after it
  auto issue_z = [&](int c) {
    if (!p.z) return;
    mbar_expect_tx(bar_tmaz, 2 * 8192);
    for (int j = 0; j < 2; ++j)
      tma_load(smem_u32(smem + S::kZ + j * 8192), &tm.z, c * kQ + 64 * j, (int)(h * kP), (int)b, true, bar_tmaz);
    z_pend = c;
  };
  auto issue_b = [&](int c) {     // B of chunk c (its buffer frees up earlier than the others)
    mbar_expect_tx(bar_tmab, 2 * 16384);
    for (int j = 0; j < 2; ++j)
      tma_load(smem_u32(smem + S::kB + j * 16384), &tm.B, 64 * j, c * kQ, (int)b, true, bar_tmab);
    b_pend = c;
  };
  if (issuer && nchunks > 0) {
    issue_b(0);
    issue_cx(0);
    issue_z(0);
  }

  const uint32_t id128 = umma_idesc_bf16(128, 128), id64 = umma_idesc_bf16(128, 64);
  // raw delta of step t (this row's step of a chunk; bf16 bits, this kernel's I/O type), loaded one
  // chunk ahead and widened only where it is used, so that no instruction of the issuing chunk waits
  // for the load
  auto load_delta = [&](int64_t t) -> unsigned short {
    if (cq != 0 || t >= p.L) return 0;
    return __ldg(static_cast<const unsigned short*>(p.delta) + b * p.sd[0] + h * p.sd[1] + t);
  };
  unsigned short dnext = nchunks > 0 ? load_delta(r) : 0;
  bool failed = false;
  int c = 0;
  for (; c < nchunks; ++c) {
    const uint32_t par = (uint32_t)c & 1u;
    const int64_t t0 = (int64_t)c * kQ;
    const int valid = (int)(p.L - t0 < kQ ? p.L - t0 : kQ);   // steps of this chunk inside the sequence

    // ---- 2. Delta, prefix sum S (rows, half 0), weights; the incoming state as an operand ----
    float dt = 0.f;
    if (cq == 0 && r < valid) dt = delta_of<false>(__uint_as_float((uint32_t)dnext << 16), bias, p.softplus);
    dnext = load_delta(t0 + kQ + r);   // the next chunk's, in flight during this one
    float cum = dt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float v = __shfl_up_sync(0xffffffffu, cum, o);
      if (lane >= o) cum += v;
    }
    if (cq == 0 && lane == 31) sWarp[warp] = cum;
    // H_in^T as the bf16 operand: row p, K = n (this thread's n = r, its 32 head channels)
#pragma unroll
    for (int j = 0; j < kPQ; ++j)
      *reinterpret_cast<__nv_bfloat16*>(smem + S::kSI + (r >> 6) * 8192 + sw128_offset(kPQ * cq + j, r & 63)) =
          __float2bfloat16_rn(H[j]);
    __syncthreads();
    if (cq == 0) {
      for (int w = 0; w < warp; ++w) cum += sWarp[w];
      sDelta[r] = dt;
      sCum[r] = cum;
    }
    __syncthreads();
    cum = sCum[r];
    const float cum_end = sCum[kQ - 1];
    if (cq == 0) {
      sW[r] = ex2_approx(a2 * (cum_end - cum)) * sDelta[r];
      // the score's column factor Delta_s enters the exponent when it is positive (softplus)
      sAS[r] = p.softplus ? __log2f(sDelta[r]) - a2 * cum : -a2 * cum;
    }
    const float et = ex2_approx(a2 * cum);   // exp(a S_t) of row t = r

    // ---- 1. B of this chunk; B~^T[n][s] = w_s B[s][n] (thread: n = r, steps [kSQ cq, kSQ cq + kSQ)) ----
    const bool ok_b = mbar_wait(bar_tmab, par);
    if (!ok_b) record_status(p.status, SSM_ERR_TIMEOUT);
    if (issuer && ok_b) b_pend = -1;
    __syncthreads();   // sW visible
    // ---- 3. G = C B^T needs only the two TMA tiles: it runs while the threads build B~^T ----
    const uint32_t sC = smem_u32(smem + S::kC);
    if (issuer && ok_b && mbar_wait(bar_tma, par)) {
      tc_fence_after();
      const uint32_t sB = smem_u32(smem + S::kB);
      for (int k = 0; k < 8; ++k) {
        const uint32_t o16 = (k >> 2) * 16384 + (k & 3) * 32;
        umma_bf16(tmem + kColG, umma_desc_sw128(sC + o16), umma_desc_sw128(sB + o16), id128, k > 0);
      }
      umma_commit(bar_g);
      g_out = true;
    }
    // warp w transposes steps [32 (w % 4), +32) x states [32 (w / 4), +32) in 8 x 8 blocks: lane l
    // addresses row l % 8 of block l / 8 (one 16-byte row piece each), and after the transposing
    // load holds, for each of the four step blocks m, the pair of steps 32 (w % 4) + 8 m + 2 (l % 4)
    // + {0, 1} of state n0 + l / 4; the weights of those steps are the same for every state block
    if (__all_sync(0xffffffffu, ok_b)) {
      const int s0 = 32 * (warp & 3), nb0 = 32 * (warp >> 2), mi = lane >> 3, ri = lane & 7;
      float2 wv[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) wv[m] = *reinterpret_cast<const float2*>(sW + s0 + 8 * m + 2 * (lane & 3));
#pragma unroll
      for (int nb = 0; nb < 4; ++nb) {
        const int n0 = nb0 + 8 * nb;
        uint32_t v[4];
        ldsm_x4_trans(smem_u32(smem + S::kB + (n0 >> 6) * 16384 + sw128_offset(s0 + 8 * mi + ri, n0 & 63)), v);
#pragma unroll
        for (int m = 0; m < 4; ++m) v[m] = scale_bf16x2(v[m], wv[m]);
        const int n = n0 + ri, sb = s0 + 8 * mi;
        stsm_x4(smem_u32(smem + S::kBT + (sb >> 6) * 16384 + n * 128 + ((((sb & 63) >> 3) ^ (n & 7)) << 4)), v);
      }
    }
    // ---- C, X and z of this chunk ----
    const bool ok_t = ok_b && mbar_wait(bar_tma, par);
    if (!ok_t) record_status(p.status, SSM_ERR_TIMEOUT);
    if (issuer && ok_t) cx_pend = -1;
    fence_async_smem();
    tc_fence_before();
    if (__syncthreads_or(!ok_t)) { failed = true; break; }

    // ---- 4. causal decay mask on G -> bf16 scores (thread: row t = r, steps [kSQ cq, kSQ cq + kSQ)) ----
    const bool ok_g = mbar_wait(bar_g, par);
    if (!ok_g) record_status(p.status, SSM_ERR_TIMEOUT);
    tc_fence_after();
    if (__syncthreads_or(!ok_g)) { failed = true; break; }
    // H_chunk = B~^T X and Y_off = C H_in (operands written by the threads) run on the tensor cores
    // while the threads build the scores; B is consumed (B~^T built, G complete), so the next
    // chunk's B can land meanwhile
    if (issuer) {
      g_out = false;
      tc_fence_after();
      const uint32_t sX = smem_u32(smem + S::kX), sBT = smem_u32(smem + S::kBT), sSI = smem_u32(smem + S::kSI);
      for (int k = 0; k < 8; ++k) {
        const uint32_t o16 = (k >> 2) * 16384 + (k & 3) * 32, o8 = (k >> 2) * 8192 + (k & 3) * 32;
        umma_bf16(tmem + kColH, umma_desc_sw128(sBT + o16), umma_desc_sw128(sX + o8), id64, k > 0);
      }
      for (int k = 0; k < 8; ++k) {
        const uint32_t o16 = (k >> 2) * 16384 + (k & 3) * 32, o8 = (k >> 2) * 8192 + (k & 3) * 32;
        umma_bf16(tmem + kColYo, umma_desc_sw128(sC + o16), umma_desc_sw128(sSI + o8), id64, k > 0);
      }
      umma_commit(bar_ho);
      ho_out = true;
      if (c + 1 < nchunks) issue_b(c + 1);
    }
#pragma unroll 1
    for (int s0 = kSQ * cq; s0 < kSQ * cq + kSQ; s0 += 32) {
      if (s0 > 32 * (warp & 3) + 31) {   // above the diagonal for every row of this warp: zeros
#pragma unroll
        for (int j = 0; j < 32; j += 8) {
          const int sblk = (s0 + j) >> 6, piece = ((s0 + j) & 63) >> 3;
          *reinterpret_cast<uint4*>(smem + S::kSP + sblk * 16384 + r * 128 + ((piece ^ (r & 7)) << 4)) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        continue;
      }
      float g[32];
      tmem_ld32(tmem + lane_off + kColG + (uint32_t)s0, g);
      // scores[t][s] = exp(a (S_t - S_s)) Delta_s G[t][s] for s <= t, two columns per packed operation;
      // only the diagonal block has entries above the diagonal to clear
      const float2 ac2 = make_float2(a2 * cum, a2 * cum);
      const bool diag = s0 == (r & ~31);
#pragma unroll
      for (int j = 0; j < 32; j += 8) {
        float f[8];
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          const int s = s0 + j + e;
          const float2 x = __fadd2_rn(ac2, *reinterpret_cast<const float2*>(sAS + s));
          float2 v = __fmul2_rn(make_float2(g[j + e], g[j + e + 1]), make_float2(ex2_approx(x.x), ex2_approx(x.y)));
          if (!p.softplus) v = __fmul2_rn(v, *reinterpret_cast<const float2*>(sDelta + s));
          f[e] = v.x;
          f[e + 1] = v.y;
        }
        if (diag) {
#pragma unroll
          for (int e = 0; e < 8; ++e)
            if (s0 + j + e > r) f[e] = 0.f;
        }
        const int sblk = (s0 + j) >> 6, piece = ((s0 + j) & 63) >> 3;
        *reinterpret_cast<uint4*>(smem + S::kSP + sblk * 16384 + r * 128 + ((piece ^ (r & 7)) << 4)) = pack16(f);
      }
      if (diag) {   // D x_t enters Y_diag through scores[t][t]
        __nv_bfloat16* dg =
            reinterpret_cast<__nv_bfloat16*>(smem + S::kSP + (r >> 6) * 16384 + sw128_offset(r, r & 63));
        *dg = __float2bfloat16_rn(__bfloat162float(*dg) + Dh);
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- 5. Y_diag = scores X ----
    if (issuer) {
      tc_fence_after();
      const uint32_t sSP = smem_u32(smem + S::kSP), sX = smem_u32(smem + S::kX);
      for (int k = 0; k < 8; ++k) {
        const uint32_t o16 = (k >> 2) * 16384 + (k & 3) * 32, o8 = (k >> 2) * 8192 + (k & 3) * 32;
        umma_bf16(tmem + kColYd, umma_desc_sw128(sSP + o16), umma_desc_sw128(sX + o8), id64, k > 0);
      }
      umma_commit(bar_d);
      d_out = true;
    }

    // ---- 6. state update (thread: n = r, channels [kPQ cq, +kPQ)), then the output (t = r, same channels) ----
    const bool ok_ho = mbar_wait(bar_ho, par);
    if (!ok_ho) record_status(p.status, SSM_ERR_TIMEOUT);
    tc_fence_after();
    if (ok_ho) {
      const float decay = ex2_approx(a2 * cum_end);
      float hc[kPQ];
      tmem_ld(tmem + lane_off + kColH + (uint32_t)(kPQ * cq), hc);
#pragma unroll
      for (int j = 0; j < kPQ; ++j) H[j] = fmaf(decay, H[j], hc[j]);
    }
    const bool ok_d = mbar_wait(bar_d, par);
    if (!ok_d) record_status(p.status, SSM_ERR_TIMEOUT);
    tc_fence_after();
    // every MMA of this chunk is complete: C and X of the next chunk can land now
    if (issuer && ok_ho && ok_d && c + 1 < nchunks) issue_cx(c + 1);
    const bool ok_z = !p.z || mbar_wait(bar_tmaz, par);
    if (!ok_z) record_status(p.status, SSM_ERR_TIMEOUT);
    if (issuer && p.z && ok_z) z_pend = -1;
    if (ok_ho && ok_d && ok_z) {
      const int64_t t = t0 + r;
      float yd[kPQ], yo[kPQ];
      tmem_ld(tmem + lane_off + kColYd + (uint32_t)(kPQ * cq), yd);
      tmem_ld(tmem + lane_off + kColYo + (uint32_t)(kPQ * cq), yo);
      if (r < valid) {
#pragma unroll
        for (int j = 0; j < kPQ; ++j) {
          const int q = kPQ * cq + j;
          const int64_t d = h * kP + q;
          const int zx = (r >> 6) * 8192 + sw128_offset(q, r & 63);
          float v = fmaf(et, yo[j], yd[j]);
          if (p.z) v *= silu_tanh(__bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(smem + S::kZ + zx)));
          static_cast<__nv_bfloat16*>(p.y)[b * p.sy[0] + d * p.sy[1] + t] = __float2bfloat16_rn(v);
        }
      }
    }
    tc_fence_before();
    if (__syncthreads_or(!(ok_ho && ok_d && ok_z))) { failed = true; break; }
    ho_out = d_out = false;
    if (issuer && c + 1 < nchunks) issue_z(c + 1);
  }

  if (failed) {
    // let every copy and MMA this CTA started finish (bounded waits) before its tensor memory is freed
    if (issuer) {
      if (b_pend >= 0) mbar_wait(bar_tmab, (uint32_t)b_pend & 1u);
      if (cx_pend >= 0) mbar_wait(bar_tma, (uint32_t)cx_pend & 1u);
      if (z_pend >= 0) mbar_wait(bar_tmaz, (uint32_t)z_pend & 1u);
      const uint32_t par = (uint32_t)c & 1u;
      if (g_out) mbar_wait(bar_g, par);
      if (ho_out) mbar_wait(bar_ho, par);
      if (d_out) mbar_wait(bar_d, par);
    }
  } else if (p.h_last) {
#pragma unroll
    for (int j = 0; j < kPQ; ++j)
      p.h_last[b * p.shl[0] + h * p.shl[1] + (kPQ * cq + j) * p.shl[2] + r * p.shl[3]] = H[j];
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// The recurrence itself, one warp per (batch, channel): lane l keeps states n = l, l + 32, ...;
// the C contraction is a warp sum.  Any head size, state size up to 256, any strides, fp32 or bf16.
template <typename IO, int NPL, bool PRECISE>
__global__ void __launch_bounds__(128) ssd_generic_kernel(const SsdProblem p) {
  const int64_t wid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t D = p.H * p.P;
  if (wid >= p.B * D) return;
  const int64_t b = wid / D, d = wid % D, h = d / p.P, q = d % p.P;
  const int N = (int)p.N;
  const float a2 = p.a[h] * kLog2e;
  const float bias = p.bias ? p.bias[h] : 0.f;
  const float Dh = p.Dskip ? p.Dskip[h] : 0.f;
  const IO* x = static_cast<const IO*>(p.x) + b * p.sx[0] + d * p.sx[1];
  const IO* z = p.z ? static_cast<const IO*>(p.z) + b * p.sz[0] + d * p.sz[1] : nullptr;
  const IO* dl = static_cast<const IO*>(p.delta) + b * p.sd[0] + h * p.sd[1];
  const IO* Bm = static_cast<const IO*>(p.Bm) + b * p.sB[0];
  const IO* Cm = static_cast<const IO*>(p.Cm) + b * p.sC[0];
  IO* y = static_cast<IO*>(p.y) + b * p.sy[0] + d * p.sy[1];
  float hs[NPL];
#pragma unroll
  for (int j = 0; j < NPL; ++j) {
    const int n = lane + 32 * j;
    hs[j] = (n < N && p.h0) ? p.h0[b * p.sh0[0] + h * p.sh0[1] + q * p.sh0[2] + n * p.sh0[3]] : 0.f;
  }
  for (int64_t t = 0; t < p.L; ++t) {
    const float dt = delta_of<PRECISE>(to_f32(dl[t]), bias, p.softplus);
    const float ab = ex2_approx(dt * a2);
    const float xv = to_f32(x[t]);
    const float dx = dt * xv;
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < NPL; ++j) {
      const int n = lane + 32 * j;
      if (n < N) {
        hs[j] = fmaf(ab, hs[j], dx * to_f32(Bm[t * p.sB[1] + n * p.sB[2]]));
        acc = fmaf(to_f32(Cm[t * p.sC[1] + n * p.sC[2]]), hs[j], acc);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) {
      float v = acc + Dh * xv;
      if (z) v *= silu<PRECISE>(to_f32(z[t]));
      y[t] = from_f32<IO>(v);
    }
  }
  if (p.h_last) {
#pragma unroll
    for (int j = 0; j < NPL; ++j) {
      const int n = lane + 32 * j;
      if (n < N) p.h_last[b * p.shl[0] + h * p.shl[1] + q * p.shl[2] + n * p.shl[3]] = hs[j];
    }
  }
}

template <typename IO, bool PRECISE>
cudaError_t launch_generic(const SsdProblem& p, cudaStream_t s) {
  const int64_t warps = p.B * p.H * p.P;
  const dim3 grid((unsigned)((warps * 32 + 127) / 128));
  if (p.N <= 32) ssd_generic_kernel<IO, 1, PRECISE><<<grid, 128, 0, s>>>(p);
  else if (p.N <= 64) ssd_generic_kernel<IO, 2, PRECISE><<<grid, 128, 0, s>>>(p);
  else if (p.N <= 128) ssd_generic_kernel<IO, 4, PRECISE><<<grid, 128, 0, s>>>(p);
  else ssd_generic_kernel<IO, 8, PRECISE><<<grid, 128, 0, s>>>(p);
  return cudaGetLastError();
}

// Tensor map of a rank-3 bf16 tensor with dims (inner, mid, outer) and byte strides (mid, outer),
// box (64, box_mid, 1), 128-byte swizzle.
bool encode_ssd_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t mid, uint64_t outer,
                    uint64_t stride_mid_bytes, uint64_t stride_outer_bytes, uint32_t box_mid) {
  EncodeTiledFn enc = get_encode_tiled();
  if (!enc) return false;
  cuuint64_t dims[3] = {inner, mid, outer};
  cuuint64_t gstr[2] = {stride_mid_bytes, stride_outer_bytes};
  cuuint32_t box[3] = {64, box_mid, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, gstr, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool ssd_tensor_core_eligible(const SsdProblem& p) {
  if (p.io != SSM_BF16 || p.P != kP || p.N != kN || p.L <= 0) return false;
  if (p.L % 8 != 0 || p.L > (int64_t)INT32_MAX - kQ || p.B > 65535) return false;
  const int64_t D = p.H * p.P;
  // x: (B, D, L) with time stride 1, rows of L, 16-byte aligned; B / C: (B, L, N) dense rows of N
  auto aligned16 = [](const void* q) { return reinterpret_cast<uintptr_t>(q) % 16 == 0; };
  if (!aligned16(p.x) || !aligned16(p.Bm) || !aligned16(p.Cm)) return false;
  if (p.sx[1] != p.L || (p.B > 1 && p.sx[0] != D * p.L)) return false;
  if (p.z && (!aligned16(p.z) || p.sz[1] != p.L || (p.B > 1 && p.sz[0] != D * p.L))) return false;
  if (p.sB[2] != 1 || p.sB[1] != kN || (p.B > 1 && p.sB[0] != p.L * kN)) return false;
  if (p.sC[2] != 1 || p.sC[1] != kN || (p.B > 1 && p.sC[0] != p.L * kN)) return false;
  return true;
}

size_t ssd_smem_bytes() { return SsdSmem::kAlloc; }

cudaError_t launch_ssd(const SsdProblem& p, bool tensor_cores, cudaStream_t s) {
  if (p.B * p.H * p.P == 0) return cudaSuccess;
  if (!tensor_cores) {
    if (p.io == SSM_F32) return launch_generic<float, true>(p, s);
    return launch_generic<__nv_bfloat16, false>(p, s);
  }
  SsdMaps tm;
  std::memset(&tm, 0, sizeof(tm));
  const int64_t D = p.H * p.P;
  if (!encode_ssd_map(&tm.x, p.x, (uint64_t)p.L, (uint64_t)D, (uint64_t)p.B, (uint64_t)p.L * 2,
                      (uint64_t)(D * p.L * 2), 64) ||
      (p.z && !encode_ssd_map(&tm.z, p.z, (uint64_t)p.L, (uint64_t)D, (uint64_t)p.B, (uint64_t)p.L * 2,
                              (uint64_t)(D * p.L * 2), 64)) ||
      !encode_ssd_map(&tm.B, p.Bm, kN, (uint64_t)p.L, (uint64_t)p.B, kN * 2, (uint64_t)(p.L * kN * 2), kQ) ||
      !encode_ssd_map(&tm.C, p.Cm, kN, (uint64_t)p.L, (uint64_t)p.B, kN * 2, (uint64_t)(p.L * kN * 2), kQ))
    return cudaErrorInvalidValue;
  static unsigned long long attr_set = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(__atomic_load_n(&attr_set, __ATOMIC_ACQUIRE) & bit)) {
    e = cudaFuncSetAttribute(ssd_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SsdSmem::kAlloc);
    if (e != cudaSuccess) return e;
    __atomic_fetch_or(&attr_set, bit, __ATOMIC_RELEASE);
  }
  ssd_chunk_kernel<<<(unsigned)(p.B * p.H), kSsdThreads, SsdSmem::kAlloc, s>>>(p, tm);
  return cudaGetLastError();
}

}  // namespace ssm
