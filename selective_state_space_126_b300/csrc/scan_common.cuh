// scan_common.cuh -- pieces shared by the scan kernels: kernel parameters,
// tensor maps of the sequence tensors, swizzled shared-memory addressing, and
// the chunk-carry kernel of the long-sequence path.
#pragma once

#include <cstring>

#include "async_copy.cuh"
#include "device_math.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int MODE_OUTPUT = 0;   // scan and emit y (and h_last)
constexpr int MODE_RECORD = 1;   // chunked path, first pass: scan from zero, record end state and sum of Delta
constexpr int MODE_CKPT = 2;     // backward pass, first step: scan from h0, keep the state every SSM_BWD_SEGMENT steps

struct ScanKernelParams {
  int64_t B, D, L;
  int N;
  int nchunks;
  int64_t chunk_len;
  const float* A;
  const float* Aim;  // imaginary part of a complex A (same strides), or null
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
  int has_z;
  int seq_rank3;    // u / delta / z tensor maps carry a batch dimension (else shared across the batch)
  int bc_rank3;     // B / C tensor maps carry a batch dimension
  int y_rank3;      // the y tensor map carries a batch dimension
  int* status;
  float* ckpt;      // MODE_CKPT: [B][D][nseg][16], the state before every segment
  int64_t nseg;
  // split single pass (see ssm_api.cu): with nblk > 0, CTA j runs unit u = unit0 + j, batch row
  // u / nblk and channels 32 (u % nblk) ..; else the grid gives (channel block, chunk, batch)
  int64_t unit0, nblk;
  int pdl;          // 1: let the next launch start at once; 2: before exiting, wait for the launch before
};

struct ScanMaps {
  CUtensorMap u, delta, z, B, C, y;
};

// Byte offset of 16-byte piece `chunk` of row `row` in a box that TMA wrote
// with the swizzle matching its row length (32, 64 or 128 bytes): the piece
// index is XOR-ed with the address bits just above the 128-byte line.
template <int ROWB>
__device__ __forceinline__ int swz(int row, int chunk) {
  if (ROWB == 32) return row * 32 + ((chunk ^ ((row >> 2) & 1)) << 4);
  if (ROWB == 64) return row * 64 + ((chunk ^ ((row >> 1) & 3)) << 4);
  return row * 128 + ((chunk ^ (row & 7)) << 4);
}

// Chunk carry: turns the per-chunk end states (from zero) into each chunk's
// true initial state, in chunk order: h_in[c+1] = exp(A sum Delta_c) h_in[c]
// + h_end[c] (the associative combine of "docs.ifdog.com", section
// "Hardware-aware parallel scan", applied to whole chunks).  One thread per
// (b, d, n).
__global__ void __launch_bounds__(256) chunk_carry_kernel(const ScanKernelParams p, int NP) {
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

// Tensor map of a (batch, rows, L) tensor with time stride 1: box (box_t
// steps x box_rows), swizzled by its row length (see swz).  Rank 3 (t, row, b)
// when the batch stride is used, else rank 2 (t, row).
inline bool encode_map(CUtensorMap* map, const void* base, const int64_t* strides, int64_t rows, uint32_t box_t,
                       uint32_t box_rows, const ScanProblem& p, bool rank3) {
  EncodeTiledFn enc = get_encode_tiled();
  if (!enc) return false;
  const int es = p.io == SSM_F32 ? 4 : 2;
  const CUtensorMapDataType dt = p.io == SSM_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int64_t row_stride = rows > 1 ? strides[1] : (p.L + 7) / 8 * 8;   // unused over one row
  cuuint64_t dims[3] = {(cuuint64_t)p.L, (cuuint64_t)rows, (cuuint64_t)p.B};
  cuuint64_t gstr[2] = {(cuuint64_t)(row_stride * es), (cuuint64_t)(strides[0] * es)};
  cuuint32_t box[3] = {box_t, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const uint32_t rowb = box_t * es;
  const CUtensorMapSwizzle swz = rowb == 32   ? CU_TENSOR_MAP_SWIZZLE_32B
                                 : rowb == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                              : CU_TENSOR_MAP_SWIZZLE_128B;
  CUresult r = enc(map, dt, rank3 ? 3 : 2, const_cast<void*>(base), dims, gstr, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Parameters and tensor maps of one scan call (boxes of box_t steps x 32
// channels for u, delta, z, y and box_t x N for B, C).
inline bool make_scan_kernel_args(const ScanProblem& p, const ScanPlan& plan, void* workspace, int NP, uint32_t box_t,
                                  ScanKernelParams* kp, ScanMaps* tm) {
  std::memset(kp, 0, sizeof(*kp));
  kp->B = p.B; kp->D = p.D; kp->L = p.L; kp->N = (int)p.N;
  kp->nchunks = (int)plan.nchunks;
  kp->chunk_len = plan.nchunks > 1 ? plan.chunk_len : p.L;
  kp->A = p.A; kp->Aim = p.Aim; kp->sA0 = p.sA[0]; kp->sA1 = p.sA[1];
  kp->Dskip = p.Dskip; kp->bias = p.bias;
  kp->h0 = p.h0; kp->sh00 = p.sh0[0]; kp->sh01 = p.sh0[1]; kp->sh02 = p.sh0[2];
  kp->h_last = p.h_last; kp->shl0 = p.shl[0]; kp->shl1 = p.shl[1]; kp->shl2 = p.shl[2];
  kp->softplus = p.softplus ? 1 : 0;
  kp->has_z = p.z ? 1 : 0;
  kp->status = device_status_ptr();
  if (plan.nchunks > 1) {
    float* ws = static_cast<float*>(workspace);
    kp->rec_h = ws;
    kp->rec_s = ws + p.B * p.D * plan.nchunks * NP;
  }
  // the planner only takes the tiled paths when u, delta, z share one batch
  // layout kind (batched or broadcast) and B, C share another; y, an output,
  // is batched whenever B > 1
  kp->seq_rank3 = (p.su[0] != 0 && p.B > 1) ? 1 : 0;
  kp->bc_rank3 = (p.sB[0] != 0 && p.B > 1) ? 1 : 0;
  kp->y_rank3 = p.B > 1 ? 1 : 0;
  std::memset(tm, 0, sizeof(*tm));
  const bool r3 = kp->seq_rank3 == 1, b3 = kp->bc_rank3 == 1, y3 = kp->y_rank3 == 1;
  return encode_map(&tm->u, p.u, p.su, p.D, box_t, 32, p, r3) &&
         encode_map(&tm->delta, p.delta, p.sd, p.D, box_t, 32, p, r3) &&
         (!p.z || encode_map(&tm->z, p.z, p.sz, p.D, box_t, 32, p, r3)) &&
         encode_map(&tm->y, p.y, p.sy, p.D, box_t, 32, p, y3) &&
         encode_map(&tm->B, p.Bm, p.sB, p.N, box_t, (uint32_t)p.N, p, b3) &&
         encode_map(&tm->C, p.Cm, p.sC, p.N, box_t, (uint32_t)p.N, p, b3);
}

}  // namespace
}  // namespace ssm
