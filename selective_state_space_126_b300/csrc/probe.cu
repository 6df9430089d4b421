// probe.cu -- SFU throughput probe for the scan's second roofline.
//
// The scan evaluates one base-2 exponential per state update on the special
// function unit (plus, per (batch, channel, step), the exponentials and the
// reciprocal of softplus and silu), so its compute ceiling is the SFU rate of
// the GPU it runs on.  This kernel measures that rate: every thread keeps
// eight independent chains of one SFU operation each, so that the unit, not
// the latency of one chain, bounds it.  The host times the launch with
// events; nothing here is part of the method.
#include "ssm_internal.h"
#include "device_math.cuh"

namespace ssm {
namespace {

constexpr int kProbeThreads = 256;
constexpr int kChains = 8;

template <int OP>
__global__ void __launch_bounds__(kProbeThreads) sfu_probe_kernel(int iters, float* sink) {
  float x[kChains];
#pragma unroll
  for (int j = 0; j < kChains; ++j) x[j] = OP == 0 ? -0.03125f * (float)(j + 1) : 1.0f + 0.0625f * (float)j;
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < kChains; ++j) {
      // ex2: x in [-1, 0] maps to 2^x - 1 in [-0.5, 0]; rcp: x in [1, 2] maps to 1/x + 0.5 in [1, 1.5]
      x[j] = OP == 0 ? ex2_approx(x[j]) - 1.0f : rcp_approx(x[j]) + 0.5f;
    }
  }
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < kChains; ++j) s += x[j];
  sink[(size_t)blockIdx.x * kProbeThreads + threadIdx.x] = s;
}

}  // namespace
}  // namespace ssm

extern "C" ssm_status_t ssm_probe_sfu(int op, int blocks, int iters, float* sink, void* stream) {
  if ((op != 0 && op != 1) || blocks <= 0 || iters <= 0 || !sink) return SSM_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (op == 0) ssm::sfu_probe_kernel<0><<<blocks, ssm::kProbeThreads, 0, s>>>(iters, sink);
  else ssm::sfu_probe_kernel<1><<<blocks, ssm::kProbeThreads, 0, s>>>(iters, sink);
  if (cudaGetLastError() != cudaSuccess) return SSM_ERR_CUDA;
  return SSM_OK;
}
