// ssm_internal.h -- host-side structures shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "../../include/ssm.h"

namespace ssm {

// Validated scan problem, strides in elements.
struct ScanProblem {
  int64_t B, D, L, N;
  ssm_dtype_t io;
  bool softplus;
  bool zoh;               // exact zero-order-hold input term (else Euler)
  bool cplx;              // complex A (A + i Aim): complex state, y = Re(C h) + D u
  const void *u, *delta, *z, *Bm, *Cm;
  const float *A, *Aim, *Dskip, *bias, *h0;
  float* h_last;
  void* y;
  int64_t su[3], sd[3], sz[3], sy[3], sB[3], sC[3], sA[2], sh0[3], shl[3];
};

struct StepProblem {
  int64_t B, D, N;
  ssm_dtype_t io;
  bool softplus;
  bool zoh;
  float* state;
  const void *u, *delta, *z, *Bm, *Cm;
  const float *A, *Dskip, *bias;
  void* y;
  int64_t sst[3], su[2], sd[2], sz[2], sy[2], sB[2], sC[2], sA[2];
};

// Validated backward problem: the forward inputs, the upstream gradients and
// the gradient outputs (strides in elements).
struct BwdProblem {
  ScanProblem f;
  const void* dy;
  const float* dhl;
  void *du, *ddelta, *dz;
  float *dA, *dB, *dC, *dD, *dbias, *dh0;
  int64_t sdy[3], sdu[3], sdd[3], sdz[3], sdB[3], sdC[3], sdhl[3], sdh0[3];
  int64_t bc_rows;     // rows of dB / dC: 1 when B / C are shared across the batch
  int64_t nseg;        // checkpoints per channel
  float* ckpt;         // [B][D][nseg][8 * bwd_lanes_per_channel(N)] fp32
  int sweep;           // 1: the backward kernel writes the checkpoints itself; 0: they are already there
  int vec;             // u, delta, z, dy rows start on 16-byte boundaries (128-bit segment loads)
  int vecbc;           // the same for the rows of B and C
  int vecout;          // du, ddelta, dz rows start on 16-byte boundaries (128-bit segment stores)
  int vecdbc;          // dB, dC rows start on 16-byte boundaries with time stride 1 (float4 atomic adds)
};

struct ConvProblem {
  int64_t B, D, L;
  int W;
  ssm_dtype_t io;
  bool silu;
  const void* x;
  const float *w, *bias;
  const void* x_hist;
  void* out;
  int64_t sx[3], so[3], sw[2], sxh[3];
};

// Validated Mamba-2 SSD problem, strides in elements.
struct SsdProblem {
  int64_t B, H, P, L, N;
  ssm_dtype_t io;
  bool softplus;
  const void *x, *delta, *z, *Bm, *Cm;
  const float *a, *Dskip, *bias, *h0;
  float* h_last;
  void* y;
  int64_t sx[3], sz[3], sy[3], sd[3], sB[3], sC[3], sh0[4], shl[4];
  int* status;
};

enum ScanPath { kPathGeneric = 0, kPathTiled = 1, kPathChunked = 2, kPathWarpScan = 3 };

// Tiled-kernel shape: K threads share one channel's states, NS states per thread.
struct TiledShape {
  int K;        // threads per channel (1, 2 or 4)
  int NS;       // states per thread
  int CH;       // channels per CTA (32)
};

struct ScanPlan {
  ScanPath path;
  TiledShape shape;
  int64_t chunk_len;      // chunked path: timesteps per chunk (multiple of the tile)
  int64_t nchunks;
  size_t workspace_bytes;
  int split_home, split_extra;   // split single pass: units of the two-warp launch / of the four-warp one
};

// device status word of the current device (bounded-wait timeouts)
int* device_status_ptr();

// launchers (return a cudaError_t from the launch)
cudaError_t launch_scan_generic(const ScanProblem& p, cudaStream_t s);
cudaError_t launch_scan_warp(const ScanProblem& p, cudaStream_t s);
cudaError_t launch_scan_tiled(const ScanProblem& p, const ScanPlan& plan, void* workspace, cudaStream_t s);
cudaError_t launch_state_update(const StepProblem& p, cudaStream_t s);
cudaError_t launch_causal_conv1d(const ConvProblem& p, int sms, cudaStream_t s);
cudaError_t launch_scan_bwd(const BwdProblem& p, int sms, cudaStream_t s);
// lanes of the backward kernel per channel (8 states each) and so the checkpoint record length / 8
inline int bwd_lanes_per_channel(int64_t N) { return N <= 16 ? 2 : N <= 32 ? 4 : 8; }
cudaError_t launch_ssd(const SsdProblem& p, bool tensor_cores, cudaStream_t s);
bool ssd_tensor_core_eligible(const SsdProblem& p);
cudaError_t launch_scan_ckpt(const ScanProblem& p, const ScanPlan& plan, float* ckpt, int64_t nseg, cudaStream_t s);

// tile length of the tiled kernel (timesteps)
#ifndef SSM_TILE_T
#define SSM_TILE_T 32
#endif
constexpr int kTileT = SSM_TILE_T;

// tensor-map encoder from the driver (resolved once through the runtime)
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn get_encode_tiled();

}  // namespace ssm
