// ssm_api.cu -- the C ABI: argument validation, path planning, dispatch.
//
// Every check here runs on the host before anything is enqueued, so a bad
// argument never reaches a kernel.  The library allocates nothing: the
// chunked path's records live in the caller's workspace.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "ssm_internal.h"

namespace ssm {

size_t tiled_smem_bytes(ssm_dtype_t io, int K, int NS);

namespace {

thread_local char g_detail[256] = {0};

ssm_status_t fail(ssm_status_t st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_detail, sizeof(g_detail), fmt, ap);
  va_end(ap);
  return st;
}

ssm_status_t ok() {
  g_detail[0] = 0;
  return SSM_OK;
}

int elem_size(ssm_dtype_t t) { return t == SSM_F32 ? 4 : 2; }

// Address range [lo, hi) touched by a strided tensor (bytes), extents all > 0.
void tensor_range(const void* base, int rank, const int64_t* ext, const int64_t* str, int es, uintptr_t* lo,
                  uintptr_t* hi) {
  int64_t last = 0;
  for (int i = 0; i < rank; ++i) last += (ext[i] - 1) * str[i];
  *lo = reinterpret_cast<uintptr_t>(base);
  *hi = *lo + (uintptr_t)(last + 1) * es;
}

// Sufficient condition for a strided mapping to be one-to-one: sorted by
// stride, each stride is at least the span of the dimensions below it.
bool injective(int rank, const int64_t* ext, const int64_t* str) {
  int idx[4];
  int m = 0;
  for (int i = 0; i < rank; ++i)
    if (ext[i] > 1) idx[m++] = i;
  for (int i = 1; i < m; ++i)   // insertion sort by stride (m <= 3)
    for (int j = i; j > 0 && str[idx[j]] < str[idx[j - 1]]; --j) {
      const int tmp = idx[j];
      idx[j] = idx[j - 1];
      idx[j - 1] = tmp;
    }
  int64_t span = 1;
  for (int k = 0; k < m; ++k) {
    if (str[idx[k]] < span) return false;
    span = str[idx[k]] * ext[idx[k]];
  }
  return true;
}

bool overlaps(uintptr_t a0, uintptr_t a1, uintptr_t b0, uintptr_t b1) { return a0 < b1 && b0 < a1; }

bool aligned(const void* p, int bytes) { return reinterpret_cast<uintptr_t>(p) % bytes == 0; }

int device_sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) return 148;
  return sms;
}

ssm_status_t validate_scan(const ssm_scan_args_t* a, ScanProblem* p) {
  if (!a) return fail(SSM_ERR_INVALID_ARG, "args is NULL");
  if (a->io_dtype != SSM_F32 && a->io_dtype != SSM_BF16) return fail(SSM_ERR_INVALID_ARG, "io_dtype %d", (int)a->io_dtype);
  if (a->batch < 0 || a->dim < 0 || a->seqlen < 0) return fail(SSM_ERR_INVALID_ARG, "negative size");
  if (a->dstate < 1 || a->dstate > 64) return fail(SSM_ERR_UNSUPPORTED, "dstate %lld outside [1, 64]", (long long)a->dstate);
  if (a->batch > 65535) return fail(SSM_ERR_UNSUPPORTED, "batch %lld > 65535", (long long)a->batch);
  std::memset(p, 0, sizeof(*p));
  p->B = a->batch; p->D = a->dim; p->L = a->seqlen; p->N = a->dstate;
  p->io = a->io_dtype;
  p->softplus = a->delta_softplus != 0;
  if (a->discretization != SSM_DISC_EULER && a->discretization != SSM_DISC_ZOH)
    return fail(SSM_ERR_INVALID_ARG, "discretization %d", (int)a->discretization);
  p->zoh = a->discretization == SSM_DISC_ZOH;
  p->u = a->u; p->delta = a->delta; p->z = a->z; p->Bm = a->Bm; p->Cm = a->Cm;
  p->A = a->A; p->Dskip = a->Dskip; p->bias = a->delta_bias; p->h0 = a->h0; p->h_last = a->h_last; p->y = a->y;
  p->Aim = a->A_imag;
  p->cplx = a->A_imag != nullptr;
  if (p->cplx && p->zoh) return fail(SSM_ERR_UNSUPPORTED, "complex A takes the Euler input term");
  std::memcpy(p->su, a->stride_u, sizeof(p->su));
  std::memcpy(p->sd, a->stride_delta, sizeof(p->sd));
  std::memcpy(p->sz, a->stride_z, sizeof(p->sz));
  std::memcpy(p->sy, a->stride_y, sizeof(p->sy));
  std::memcpy(p->sB, a->stride_B, sizeof(p->sB));
  std::memcpy(p->sC, a->stride_C, sizeof(p->sC));
  std::memcpy(p->sA, a->stride_A, sizeof(p->sA));
  std::memcpy(p->sh0, a->stride_h0, sizeof(p->sh0));
  std::memcpy(p->shl, a->stride_h_last, sizeof(p->shl));
  if (p->B == 0 || p->D == 0) return ok();   // nothing to compute or write

  if (!p->A) return fail(SSM_ERR_INVALID_ARG, "A is NULL");
  if (p->sA[0] < 0 || p->sA[1] < 0) return fail(SSM_ERR_INVALID_ARG, "negative A stride");
  const int es = elem_size(p->io);
  struct Seq {
    const char* name;
    const void* ptr;
    const int64_t* s;
    int64_t ext1;
    bool required;
  } seqs[] = {{"u", p->u, p->su, p->D, true},         {"delta", p->delta, p->sd, p->D, true},
              {"z", p->z, p->sz, p->D, false},        {"y", p->y, p->sy, p->D, true},
              {"Bm", p->Bm, p->sB, p->N, true},       {"Cm", p->Cm, p->sC, p->N, true}};
  for (const Seq& q : seqs) {
    if (!q.ptr) {
      // an empty sequence reads and writes none of these tensors
      if (q.required && p->L > 0) return fail(SSM_ERR_INVALID_ARG, "%s is NULL", q.name);
      continue;
    }
    if (q.s[0] < 0 || q.s[1] < 0) return fail(SSM_ERR_INVALID_ARG, "%s has a negative stride", q.name);
    if (q.s[2] != 1 && p->L > 1) return fail(SSM_ERR_UNSUPPORTED, "%s time stride must be 1", q.name);
    if (!aligned(q.ptr, es)) return fail(SSM_ERR_INVALID_ARG, "%s is not %d-byte aligned", q.name, es);
  }
  if (!aligned(p->A, 4)) return fail(SSM_ERR_INVALID_ARG, "A misaligned");
  if (p->cplx && !aligned(p->Aim, 4)) return fail(SSM_ERR_INVALID_ARG, "A_imag misaligned");
  for (int i = 0; i < 3; ++i)
    if ((p->h0 && p->sh0[i] < 0) || (p->h_last && p->shl[i] < 0))
      return fail(SSM_ERR_INVALID_ARG, "negative state stride");

  // outputs: one-to-one and disjoint from every input and from each other
  int64_t ey[3] = {p->B, p->D, p->L};
  int64_t sy[3] = {p->sy[0], p->sy[1], 1};
  // a complex state is (B, D, N, 2): the imaginary part one float after the real part
  const int hrank = p->cplx ? 4 : 3;
  int64_t eh[4] = {p->B, p->D, p->N, 2};
  int64_t shl[4] = {p->shl[0], p->shl[1], p->shl[2], 1};
  if (p->L > 0 && !injective(3, ey, sy)) return fail(SSM_ERR_INVALID_ARG, "y strides overlap");
  if (p->h_last && !injective(hrank, eh, shl)) return fail(SSM_ERR_INVALID_ARG, "h_last strides overlap");
  uintptr_t y0 = 0, y1 = 0, hl0 = 0, hl1 = 0;
  if (p->L > 0) tensor_range(p->y, 3, ey, sy, es, &y0, &y1);
  if (p->h_last) tensor_range(p->h_last, hrank, eh, shl, 4, &hl0, &hl1);
  struct In {
    const void* ptr;
    int rank;
    int64_t ext[4];
    int64_t str[4];
    int es;
  } ins[] = {
      {p->u, 3, {p->B, p->D, p->L, 1}, {p->su[0], p->su[1], 1, 0}, es},
      {p->delta, 3, {p->B, p->D, p->L, 1}, {p->sd[0], p->sd[1], 1, 0}, es},
      {p->z, 3, {p->B, p->D, p->L, 1}, {p->sz[0], p->sz[1], 1, 0}, es},
      {p->Bm, 3, {p->B, p->N, p->L, 1}, {p->sB[0], p->sB[1], 1, 0}, es},
      {p->Cm, 3, {p->B, p->N, p->L, 1}, {p->sC[0], p->sC[1], 1, 0}, es},
      {p->A, 2, {p->D, p->N, 1, 1}, {p->sA[0], p->sA[1], 0, 0}, 4},
      {p->Aim, 2, {p->D, p->N, 1, 1}, {p->sA[0], p->sA[1], 0, 0}, 4},
      {p->Dskip, 1, {p->D, 1, 1, 1}, {1, 0, 0, 0}, 4},
      {p->bias, 1, {p->D, 1, 1, 1}, {1, 0, 0, 0}, 4},
      {p->h0, hrank, {p->B, p->D, p->N, 2}, {p->sh0[0], p->sh0[1], p->sh0[2], 1}, 4},
  };
  for (const In& in : ins) {
    if (!in.ptr) continue;
    if (in.ext[2] == 0) continue;   // empty sequence: nothing is read
    uintptr_t i0, i1;
    tensor_range(in.ptr, in.rank, in.ext, in.str, in.es, &i0, &i1);
    if (p->L > 0 && overlaps(y0, y1, i0, i1)) return fail(SSM_ERR_INVALID_ARG, "y overlaps an input");
    if (p->h_last && overlaps(hl0, hl1, i0, i1)) return fail(SSM_ERR_INVALID_ARG, "h_last overlaps an input");
  }
  if (p->L > 0 && p->h_last && overlaps(y0, y1, hl0, hl1)) return fail(SSM_ERR_INVALID_ARG, "y overlaps h_last");
  return ok();
}

// Tiled path eligibility: every sequence tensor is read through TMA boxes of
// 32 steps (16-byte aligned base and row strides), y is written with 16-byte
// stores, and the batch dimension of each tensor is either nested outside its
// rows or broadcast (stride 0).
bool tiled_eligible(const ScanProblem& p) {
  const int es = elem_size(p.io);
  const int vec = 16 / es;
  if (p.L <= 0 || p.L % vec != 0) return false;
  if (p.L > (int64_t)INT32_MAX - 64 || p.D > (int64_t)INT32_MAX - 64) return false;
  // rows: D for u / delta / z, N for B / C
  auto tma_ok = [&](const void* ptr, const int64_t* s, int64_t rows) {
    if (!aligned(ptr, 16) || s[0] % vec != 0 || s[1] % vec != 0) return false;
    if (rows > 1 && s[1] < p.L) return false;                       // rows may not overlap
    if (p.B > 1 && s[0] != 0 && rows > 1 && s[0] < s[1] * rows) return false;
    if (p.B > 1 && s[0] != 0 && rows == 1 && s[0] < p.L) return false;
    return true;
  };
  if (!tma_ok(p.u, p.su, p.D) || !tma_ok(p.delta, p.sd, p.D) || !tma_ok(p.y, p.sy, p.D)) return false;
  if (p.z && !tma_ok(p.z, p.sz, p.D)) return false;
  if (!tma_ok(p.Bm, p.sB, p.N) || !tma_ok(p.Cm, p.sC, p.N)) return false;
  // u, delta, z share one batch layout kind (batched or broadcast); so do B and C
  auto batched = [&](const int64_t* s) { return s[0] != 0 && p.B > 1; };
  if (batched(p.sd) != batched(p.su) || (p.z && batched(p.sz) != batched(p.su))) return false;
  return batched(p.sB) == batched(p.sC);
}

// Tiled kernel shape.  N > 16 needs 4 threads per channel.  For N <= 16 two
// threads per channel (8 states each) is the better balance of per-thread
// parallelism against shared-memory traffic, except when the whole grid fits
// on the GPU at 4 CTAs of 128 threads per SM: then 4 threads per channel give
// twice the warps.  SSM_SCAN_KERNEL (k1, k2, k4) overrides the choice for
// tuning.
TiledShape pick_shape(const ScanProblem& p, int64_t ctas, int sms) {
  if (p.N > 32) return TiledShape{4, 16, 32};
  if (p.N > 16) return TiledShape{4, 8, 32};
  const char* env = getenv("SSM_SCAN_KERNEL");
  if (env) {
    if (!strcmp(env, "k1")) return TiledShape{1, 16, 32};
    if (!strcmp(env, "k2")) return TiledShape{2, 8, 32};
    if (!strcmp(env, "k4")) return TiledShape{4, 4, 32};
  }
  if (ctas <= 4 * (int64_t)sms) return TiledShape{4, 4, 32};
  // the exact-ZOH and complex-A variants do several times the arithmetic per state, in longer dependent
  // chains, and gain more from warps than from states per thread: on B300 (4 x 5120 x 2048, bf16) the
  // ZOH scan took 407 us with 4 threads per channel against 503 us with 2, the complex scan 709 us
  // against 970 us (753 us split over two launches)
  if (p.zoh || p.cplx) return TiledShape{4, 4, 32};
  return TiledShape{2, 8, 32};
}

// Split single pass.  An SM's four schedulers each issue for their own warps,
// and a one-wave grid of the two-warp (K = 2) CTAs takes as long as the
// schedulers holding the most warps: on B300, 592 CTAs of a 4 x D x 2048 scan
// (4 per SM, 2 warps per scheduler) took 193 us for D = 4736, while 640 and
// 740 CTAs (4 x 5120 and 4 x 5920 channels: 3 warps on some schedulers) both
// took 253 us.  So when the grid has more than 4 and at most 5 CTAs per SM,
// the first 4 per SM ("home" units of a batch row and 32 channels) run as one
// launch and the rest ("extra" units, at most one per SM) as a second launch
// of the four-warp CTA (4 states per thread), which starts while the first
// runs (programmatic dependent launch) and fits beside its 4 CTAs: each extra
// unit adds one quarter-unit warp to a scheduler instead of a third half-unit
// one.  Taken for the Euler term with a real A (252.8 -> 223.5 us on
// 4 x 5120 x 2048); the exact-ZOH and complex-A variants run the four-warp
// CTA instead (pick_shape).  SSM_SCAN_KERNEL=k2 keeps the single launch.
void plan_split(const ScanProblem& p, int sms, ScanPlan* plan) {
  const char* env = getenv("SSM_SCAN_KERNEL");
  if (env) return;
  if (p.io != SSM_BF16 || p.zoh || p.cplx || p.N > 16 || plan->shape.K != 2 || plan->shape.NS != 8) return;
  const int64_t units = p.B * ((p.D + 31) / 32), home = 4 * (int64_t)sms;
  if (units <= home || units > home + sms) return;
  plan->split_home = (int)home;
  plan->split_extra = (int)(units - home);
}

ssm_status_t plan_scan(const ssm_scan_args_t* a, const ScanProblem& p, ScanPlan* plan) {
  std::memset(plan, 0, sizeof(*plan));
  plan->nchunks = 1;
  plan->chunk_len = p.L;
  const bool eligible = tiled_eligible(p);
  const int flags = a->flags;
  if (flags & SSM_SCAN_FORCE_GENERIC) {
    plan->path = kPathGeneric;
    return ok();
  }
  if (flags & SSM_SCAN_FORCE_WARPSCAN) {
    if (flags & (SSM_SCAN_FORCE_TILED | SSM_SCAN_FORCE_CHUNKED))
      return fail(SSM_ERR_INVALID_ARG, "SSM_SCAN_FORCE_WARPSCAN excludes the other paths");
    if (p.zoh || p.cplx || p.N > 16)
      return fail(SSM_ERR_UNSUPPORTED, "the warp-shuffle scan takes the Euler term, a real A and dstate <= 16");
    plan->path = kPathWarpScan;
    return ok();
  }
  if (!eligible) {
    if (flags & (SSM_SCAN_FORCE_TILED | SSM_SCAN_FORCE_CHUNKED))
      return fail(SSM_ERR_UNSUPPORTED, "layout not eligible for the tiled kernels (alignment / strides / seqlen)");
    plan->path = kPathGeneric;
    return ok();
  }
  if (p.cplx) {
    // complex A: the single-pass tiled kernel for N <= 16, else the stride-general one; no chunked path
    if (flags & SSM_SCAN_FORCE_CHUNKED) return fail(SSM_ERR_UNSUPPORTED, "complex A has no chunked path");
    if (p.N > 16) {
      if (flags & SSM_SCAN_FORCE_TILED) return fail(SSM_ERR_UNSUPPORTED, "complex A on the tiled kernel takes dstate <= 16");
      plan->path = kPathGeneric;
      return ok();
    }
    plan->path = kPathTiled;
    plan->shape = pick_shape(p, p.B * ((p.D + 31) / 32), device_sm_count());
    if (plan->shape.K == 1) plan->shape = TiledShape{2, 8, 32};   // the complex variant exists for K = 2 and 4
    return ok();
  }
  const int sms = device_sm_count();
  const int64_t ctas = p.B * ((p.D + 31) / 32);
  bool chunk_wanted = false;
  if (flags & SSM_SCAN_FORCE_CHUNKED) chunk_wanted = true;
  else if (!(flags & SSM_SCAN_FORCE_TILED)) {
    // Long sequences on fewer than two CTAs per SM; from 2048 steps, grids of about one CTA per SM
    // or fewer.  On B300 (148 SMs, L = 2048, D = 1536 or 5120): 96 CTAs 103 -> 91 us and 160 CTAs
    // 129 -> 118 us chunked, but 192 CTAs 128 -> 155 us and 240 CTAs 129 -> 171 us.
    chunk_wanted = (ctas < 2 * (int64_t)sms && p.L >= 8 * 1024) || (ctas <= sms + sms / 8 && p.L >= 2048);
  }
  // the chunked path launches many more CTAs than the single pass
  plan->shape = pick_shape(p, chunk_wanted ? 8 * (int64_t)sms : ctas, sms);
  const int NP = plan->shape.K * plan->shape.NS;
  int64_t chunk_len = 0;
  if (chunk_wanted) {
    if (a->chunk_len > 0) {
      chunk_len = (a->chunk_len + kTileT - 1) / kTileT * kTileT;
    } else {
      // enough chunks for ~8 CTAs per SM, chunks of at least 256 steps (on B300 a 1 x 5120 x 2048
      // scan, 160 CTAs, takes 118 us in 8 chunks against 129 us in one pass).  With long chunks (4096
      // steps and more) every CTA runs long, and the SMs that get the most CTAs set the time, so the
      // count is rounded down to at most 8 CTAs per SM: the 1 x 1536 x 2^20 scan (48 CTAs per chunk)
      // took 12.87 ms in 24 chunks (1152 CTAs) against 13.92 ms in 25 (1200 CTAs, 9 on some SMs).
      int64_t want = (8 * (int64_t)sms + ctas - 1) / ctas;
      if (p.L / want >= 4096) want = std::max<int64_t>(1, (8 * (int64_t)sms) / ctas);
      want = std::max<int64_t>(2, std::min<int64_t>(want, p.L / 256));
      chunk_len = (p.L + want - 1) / want;
      chunk_len = (chunk_len + kTileT - 1) / kTileT * kTileT;
    }
    const int64_t nchunks = (p.L + chunk_len - 1) / chunk_len;
    if (nchunks > 65535) return fail(SSM_ERR_UNSUPPORTED, "too many chunks (%lld)", (long long)nchunks);
    if (nchunks >= 2) {
      plan->path = kPathChunked;
      plan->nchunks = nchunks;
      plan->chunk_len = chunk_len;
      plan->workspace_bytes = (size_t)(p.B * p.D * nchunks * (NP + 1)) * sizeof(float);
      return ok();
    }
  }
  plan->path = kPathTiled;
  plan_split(p, sms, plan);
  return ok();
}

ssm_status_t cuda_fail(cudaError_t e) {
  cudaGetLastError();   // clear the sticky-free error state
  return fail(SSM_ERR_CUDA, "%s", cudaGetErrorString(e));
}

std::mutex g_enc_mu;
EncodeTiledFn g_enc = nullptr;

}  // namespace

EncodeTiledFn get_encode_tiled() {
  std::lock_guard<std::mutex> lk(g_enc_mu);
  if (!g_enc) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_enc = reinterpret_cast<EncodeTiledFn>(fn);
  }
  return g_enc;
}

// Device status words, one per device (set only by bounded waits that gave up).
__device__ int g_device_status;

int* device_status_ptr() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return static_cast<int*>(p);
}

}  // namespace ssm

using namespace ssm;

extern "C" {

int ssm_version(void) { return (1 << 16) | 3; }

size_t ssm_abi_sizeof(int which) {
  if (which == 0) return sizeof(ssm_scan_args_t);
  if (which == 1) return sizeof(ssm_step_args_t);
  if (which == 2) return sizeof(ssm_conv_args_t);
  if (which == 3) return sizeof(ssm_scan_bwd_args_t);
  if (which == 4) return sizeof(ssm_ssd_args_t);
  return 0;
}

const char* ssm_status_string(ssm_status_t s) {
  switch (s) {
    case SSM_OK: return "SSM_OK";
    case SSM_ERR_INVALID_ARG: return "SSM_ERR_INVALID_ARG";
    case SSM_ERR_UNSUPPORTED: return "SSM_ERR_UNSUPPORTED";
    case SSM_ERR_CUDA: return "SSM_ERR_CUDA";
    case SSM_ERR_TIMEOUT: return "SSM_ERR_TIMEOUT";
    case SSM_ERR_WORKSPACE: return "SSM_ERR_WORKSPACE";
  }
  return "SSM_ERR_UNKNOWN";
}

const char* ssm_last_error_detail(void) { return g_detail; }

ssm_status_t ssm_scan_workspace_size(const ssm_scan_args_t* args, size_t* bytes) {
  if (!bytes) return fail(SSM_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = 0;
  ScanProblem p;
  ssm_status_t st = validate_scan(args, &p);
  if (st != SSM_OK) return st;
  if (p.B == 0 || p.D == 0) return ok();
  ScanPlan plan;
  st = plan_scan(args, p, &plan);
  if (st != SSM_OK) return st;
  *bytes = plan.workspace_bytes;
  return ok();
}

int ssm_scan_plan_path(const ssm_scan_args_t* args) {
  ScanProblem p;
  if (validate_scan(args, &p) != SSM_OK) return -1;
  if (p.B == 0 || p.D == 0) return 0;
  ScanPlan plan;
  if (plan_scan(args, p, &plan) != SSM_OK) return -1;
  if (plan.path == kPathTiled && plan.split_home > 0) return 4;   // the single pass in two launches
  return (int)plan.path;
}

ssm_status_t ssm_scan_fwd(const ssm_scan_args_t* args, void* stream) {
  ScanProblem p;
  ssm_status_t st = validate_scan(args, &p);
  if (st != SSM_OK) return st;
  if (p.B == 0 || p.D == 0) return ok();
  ScanPlan plan;
  st = plan_scan(args, p, &plan);
  if (st != SSM_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (plan.path == kPathGeneric) {
    e = launch_scan_generic(p, s);
  } else if (plan.path == kPathWarpScan) {
    e = launch_scan_warp(p, s);
  } else {
    if (plan.workspace_bytes > 0) {
      if (!args->workspace) return fail(SSM_ERR_WORKSPACE, "workspace of %zu bytes required", plan.workspace_bytes);
      if (args->workspace_bytes < plan.workspace_bytes)
        return fail(SSM_ERR_WORKSPACE, "workspace %zu < %zu bytes", args->workspace_bytes, plan.workspace_bytes);
      if (!aligned(args->workspace, 16)) return fail(SSM_ERR_WORKSPACE, "workspace not 16-byte aligned");
    }
    e = launch_scan_tiled(p, plan, args->workspace, s);
  }
  if (e != cudaSuccess) return cuda_fail(e);
  return ok();
}

ssm_status_t ssm_state_update(const ssm_step_args_t* a, void* stream) {
  if (!a) return fail(SSM_ERR_INVALID_ARG, "args is NULL");
  if (a->io_dtype != SSM_F32 && a->io_dtype != SSM_BF16) return fail(SSM_ERR_INVALID_ARG, "io_dtype");
  if (a->batch < 0 || a->dim < 0) return fail(SSM_ERR_INVALID_ARG, "negative size");
  if (a->dstate < 1 || a->dstate > 64) return fail(SSM_ERR_UNSUPPORTED, "dstate outside [1, 64]");
  StepProblem p;
  std::memset(&p, 0, sizeof(p));
  if (a->discretization != SSM_DISC_EULER && a->discretization != SSM_DISC_ZOH)
    return fail(SSM_ERR_INVALID_ARG, "discretization %d", (int)a->discretization);
  p.B = a->batch; p.D = a->dim; p.N = a->dstate; p.io = a->io_dtype; p.softplus = a->delta_softplus != 0;
  p.zoh = a->discretization == SSM_DISC_ZOH;
  p.state = a->state; p.u = a->u; p.delta = a->delta; p.z = a->z; p.Bm = a->Bm; p.Cm = a->Cm;
  p.A = a->A; p.Dskip = a->Dskip; p.bias = a->delta_bias; p.y = a->y;
  std::memcpy(p.sst, a->stride_state, sizeof(p.sst));
  std::memcpy(p.su, a->stride_u, sizeof(p.su));
  std::memcpy(p.sd, a->stride_delta, sizeof(p.sd));
  std::memcpy(p.sz, a->stride_z, sizeof(p.sz));
  std::memcpy(p.sy, a->stride_y, sizeof(p.sy));
  std::memcpy(p.sB, a->stride_B, sizeof(p.sB));
  std::memcpy(p.sC, a->stride_C, sizeof(p.sC));
  std::memcpy(p.sA, a->stride_A, sizeof(p.sA));
  if (p.B == 0 || p.D == 0) return ok();
  if (!p.state || !p.u || !p.delta || !p.Bm || !p.Cm || !p.A || !p.y)
    return fail(SSM_ERR_INVALID_ARG, "required pointer is NULL");
  const int es = elem_size(p.io);
  const int64_t* strides[] = {p.su, p.sd, p.sz, p.sy, p.sB, p.sC, p.sA};
  for (const int64_t* s : strides)
    if (s[0] < 0 || s[1] < 0) return fail(SSM_ERR_INVALID_ARG, "negative stride");
  for (int i = 0; i < 3; ++i)
    if (p.sst[i] < 0) return fail(SSM_ERR_INVALID_ARG, "negative state stride");
  const void* eptrs[] = {p.u, p.delta, p.z, p.Bm, p.Cm, p.y};
  for (const void* q : eptrs)
    if (q && !aligned(q, es)) return fail(SSM_ERR_INVALID_ARG, "misaligned pointer");
  if (!aligned(p.state, 4) || !aligned(p.A, 4)) return fail(SSM_ERR_INVALID_ARG, "misaligned fp32 pointer");
  int64_t est[3] = {p.B, p.D, p.N};
  int64_t ey[2] = {p.B, p.D};
  if (!injective(3, est, p.sst)) return fail(SSM_ERR_INVALID_ARG, "state strides overlap");
  if (!injective(2, ey, p.sy)) return fail(SSM_ERR_INVALID_ARG, "y strides overlap");
  uintptr_t s0, s1, y0, y1;
  tensor_range(p.state, 3, est, p.sst, 4, &s0, &s1);
  tensor_range(p.y, 2, ey, p.sy, es, &y0, &y1);
  if (overlaps(s0, s1, y0, y1)) return fail(SSM_ERR_INVALID_ARG, "y overlaps state");
  struct In {
    const void* ptr;
    int rank;
    int64_t ext[2];
    const int64_t* str;
    int es;
  } ins[] = {{p.u, 2, {p.B, p.D}, p.su, es},  {p.delta, 2, {p.B, p.D}, p.sd, es}, {p.z, 2, {p.B, p.D}, p.sz, es},
             {p.Bm, 2, {p.B, p.N}, p.sB, es}, {p.Cm, 2, {p.B, p.N}, p.sC, es},    {p.A, 2, {p.D, p.N}, p.sA, 4}};
  for (const In& in : ins) {
    if (!in.ptr) continue;
    uintptr_t i0, i1;
    tensor_range(in.ptr, in.rank, in.ext, in.str, in.es, &i0, &i1);
    if (overlaps(s0, s1, i0, i1) || overlaps(y0, y1, i0, i1))
      return fail(SSM_ERR_INVALID_ARG, "an output overlaps an input");
  }
  const void* vecs[] = {p.Dskip, p.bias};
  for (const void* v : vecs) {
    if (!v) continue;
    uintptr_t i0 = reinterpret_cast<uintptr_t>(v), i1 = i0 + (uintptr_t)p.D * 4;
    if (overlaps(s0, s1, i0, i1) || overlaps(y0, y1, i0, i1))
      return fail(SSM_ERR_INVALID_ARG, "an output overlaps an input");
  }
  cudaError_t e = launch_state_update(p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return ok();
}

}  // extern "C"

namespace ssm {
namespace {

// Validates the backward arguments: the forward inputs (with dy standing in
// for y as a read-only sequence tensor) and every gradient output.
ssm_status_t validate_bwd(const ssm_scan_bwd_args_t* a, BwdProblem* p) {
  if (!a) return fail(SSM_ERR_INVALID_ARG, "args is NULL");
  ssm_scan_args_t fa = a->fwd;
  fa.y = const_cast<void*>(a->dy);
  std::memcpy(fa.stride_y, a->stride_dy, sizeof(fa.stride_y));
  fa.h_last = nullptr;
  std::memset(p, 0, sizeof(*p));
  ssm_status_t st = validate_scan(&fa, &p->f);
  if (st != SSM_OK) return st;
  const ScanProblem& f = p->f;
  if (f.N > 64) return fail(SSM_ERR_UNSUPPORTED, "the backward pass takes dstate <= 64");
  if (f.cplx) return fail(SSM_ERR_UNSUPPORTED, "the backward pass takes a real A");
  p->dy = a->dy; p->dhl = a->dh_last;
  p->du = a->du; p->ddelta = a->ddelta; p->dz = a->dz;
  p->dA = a->dA; p->dB = a->dB; p->dC = a->dC; p->dD = a->dDskip; p->dbias = a->ddelta_bias; p->dh0 = a->dh0;
  std::memcpy(p->sdy, a->stride_dy, sizeof(p->sdy));
  std::memcpy(p->sdu, a->stride_du, sizeof(p->sdu));
  std::memcpy(p->sdd, a->stride_ddelta, sizeof(p->sdd));
  std::memcpy(p->sdz, a->stride_dz, sizeof(p->sdz));
  std::memcpy(p->sdB, a->stride_dB, sizeof(p->sdB));
  std::memcpy(p->sdC, a->stride_dC, sizeof(p->sdC));
  std::memcpy(p->sdhl, a->stride_dh_last, sizeof(p->sdhl));
  std::memcpy(p->sdh0, a->stride_dh0, sizeof(p->sdh0));
  p->nseg = (f.L + SSM_BWD_SEGMENT - 1) / SSM_BWD_SEGMENT;
  const bool shared_b = f.sB[0] == 0 && f.B > 1, shared_c = f.sC[0] == 0 && f.B > 1;
  if (shared_b != shared_c) return fail(SSM_ERR_UNSUPPORTED, "B and C must be both shared or both per batch row");
  p->bc_rows = shared_b ? 1 : f.B;
  if (f.B == 0 || f.D == 0) return ok();
  if (!p->dA) return fail(SSM_ERR_INVALID_ARG, "dA is NULL");
  if (f.L > 0 && (!p->dy || !p->du || !p->ddelta || !p->dB || !p->dC))
    return fail(SSM_ERR_INVALID_ARG, "dy, du, ddelta, dB or dC is NULL");
  if ((f.z != nullptr) != (p->dz != nullptr) && f.L > 0) return fail(SSM_ERR_INVALID_ARG, "dz must be given exactly when z is");
  if ((f.Dskip != nullptr) != (p->dD != nullptr)) return fail(SSM_ERR_INVALID_ARG, "dDskip must be given exactly when Dskip is");
  if (shared_b && (p->sdB[0] != 0 || p->sdC[0] != 0))
    return fail(SSM_ERR_INVALID_ARG, "B/C are shared across the batch: dB/dC need batch stride 0");
  const int es = elem_size(f.io);
  struct Out {
    const char* name;
    const void* ptr;
    int rank;
    int64_t ext[3];
    const int64_t* str;
    int es;
  };
  const int64_t sA[2] = {f.N, 1}, s1[1] = {1};
  int64_t sdB[3] = {p->sdB[0], p->sdB[1], p->sdB[2]}, sdC[3] = {p->sdC[0], p->sdC[1], p->sdC[2]};
  const Out outs[] = {{"du", p->du, 3, {f.B, f.D, f.L}, p->sdu, es},
                      {"ddelta", p->ddelta, 3, {f.B, f.D, f.L}, p->sdd, es},
                      {"dz", p->dz, 3, {f.B, f.D, f.L}, p->sdz, es},
                      {"dB", p->dB, 3, {p->bc_rows, f.N, f.L}, sdB, 4},
                      {"dC", p->dC, 3, {p->bc_rows, f.N, f.L}, sdC, 4},
                      {"dA", p->dA, 2, {f.D, f.N, 1}, sA, 4},
                      {"dDskip", p->dD, 1, {f.D, 1, 1}, s1, 4},
                      {"ddelta_bias", p->dbias, 1, {f.D, 1, 1}, s1, 4},
                      {"dh0", p->dh0, 3, {f.B, f.D, f.N}, p->sdh0, 4}};
  uintptr_t lo[9], hi[9];
  int m = 0;
  for (const Out& o : outs) {
    if (!o.ptr || o.ext[o.rank - 1] == 0) continue;
    for (int i = 0; i < o.rank; ++i)
      if (o.str[i] < 0) return fail(SSM_ERR_INVALID_ARG, "%s has a negative stride", o.name);
    const bool seq = o.ptr == p->du || o.ptr == p->ddelta || o.ptr == p->dz;   // written along t with stride 1
    if (seq && o.str[2] != 1 && f.L > 1) return fail(SSM_ERR_UNSUPPORTED, "%s time stride must be 1", o.name);
    if (!aligned(o.ptr, o.es)) return fail(SSM_ERR_INVALID_ARG, "%s misaligned", o.name);
    if (o.rank == 3 && !injective(3, o.ext, o.str)) return fail(SSM_ERR_INVALID_ARG, "%s strides overlap", o.name);
    tensor_range(o.ptr, o.rank, o.ext, o.str, o.es, &lo[m], &hi[m]);
    ++m;
  }
  for (int i = 0; i < m; ++i)
    for (int j = i + 1; j < m; ++j)
      if (overlaps(lo[i], hi[i], lo[j], hi[j])) return fail(SSM_ERR_INVALID_ARG, "two gradient outputs overlap");
  // no gradient output may overlap an input
  struct In {
    const void* ptr;
    int rank;
    int64_t ext[3];
    int64_t str[3];
    int es;
  } ins[] = {
      {f.u, 3, {f.B, f.D, f.L}, {f.su[0], f.su[1], 1}, es},
      {f.delta, 3, {f.B, f.D, f.L}, {f.sd[0], f.sd[1], 1}, es},
      {f.z, 3, {f.B, f.D, f.L}, {f.sz[0], f.sz[1], 1}, es},
      {p->dy, 3, {f.B, f.D, f.L}, {p->sdy[0], p->sdy[1], 1}, es},
      {f.Bm, 3, {f.B, f.N, f.L}, {f.sB[0], f.sB[1], 1}, es},
      {f.Cm, 3, {f.B, f.N, f.L}, {f.sC[0], f.sC[1], 1}, es},
      {f.A, 2, {f.D, f.N, 1}, {f.sA[0], f.sA[1], 0}, 4},
      {f.Dskip, 1, {f.D, 1, 1}, {1, 0, 0}, 4},
      {f.bias, 1, {f.D, 1, 1}, {1, 0, 0}, 4},
      {f.h0, 3, {f.B, f.D, f.N}, {f.sh0[0], f.sh0[1], f.sh0[2]}, 4},
      {p->dhl, 3, {f.B, f.D, f.N}, {p->sdhl[0], p->sdhl[1], p->sdhl[2]}, 4},
  };
  for (const In& in : ins) {
    if (!in.ptr || in.ext[in.rank - 1] == 0) continue;
    for (int i = 0; i < in.rank; ++i)
      if (in.str[i] < 0) return fail(SSM_ERR_INVALID_ARG, "negative input stride");
    uintptr_t i0, i1;
    tensor_range(in.ptr, in.rank, in.ext, in.str, in.es, &i0, &i1);
    for (int k = 0; k < m; ++k)
      if (overlaps(lo[k], hi[k], i0, i1)) return fail(SSM_ERR_INVALID_ARG, "a gradient output overlaps an input");
  }
  return ok();
}

size_t bwd_workspace_bytes(const BwdProblem& p) {
  return (size_t)(p.f.B * p.f.D * p.nseg) * (size_t)(8 * bwd_lanes_per_channel(p.f.N)) * sizeof(float);
}

}  // namespace
}  // namespace ssm

extern "C" {

ssm_status_t ssm_scan_bwd_workspace_size(const ssm_scan_bwd_args_t* args, size_t* bytes) {
  if (!bytes) return fail(SSM_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = 0;
  BwdProblem p;
  ssm_status_t st = validate_bwd(args, &p);
  if (st != SSM_OK) return st;
  *bytes = bwd_workspace_bytes(p);
  return ok();
}

ssm_status_t ssm_scan_bwd(const ssm_scan_bwd_args_t* args, void* stream) {
  BwdProblem p;
  ssm_status_t st = validate_bwd(args, &p);
  if (st != SSM_OK) return st;
  if (p.f.B == 0 || p.f.D == 0) return ok();
  const size_t need = bwd_workspace_bytes(p);
  if (need > 0) {
    if (!args->fwd.workspace) return fail(SSM_ERR_WORKSPACE, "workspace of %zu bytes required", need);
    if (args->fwd.workspace_bytes < need)
      return fail(SSM_ERR_WORKSPACE, "workspace %zu < %zu bytes", args->fwd.workspace_bytes, need);
    if (!aligned(args->fwd.workspace, 16)) return fail(SSM_ERR_WORKSPACE, "workspace not 16-byte aligned");
  }
  p.ckpt = static_cast<float*>(args->fwd.workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  {
    const int es = elem_size(p.f.io);
    auto rows16 = [&](const void* ptr, const int64_t* st) {
      if (!ptr) return true;
      if (!aligned(ptr, 16)) return false;
      if (p.f.D > 1 && (st[1] * es) % 16) return false;
      if (p.f.B > 1 && (st[0] * es) % 16) return false;
      return true;
    };
    p.vec = rows16(p.f.u, p.f.su) && rows16(p.f.delta, p.f.sd) && rows16(p.f.z, p.f.sz) && rows16(p.dy, p.sdy) ? 1 : 0;
    auto bc16 = [&](const void* ptr, const int64_t* st) {   // rows n of B / C: batch stride 0 allowed
      if (!aligned(ptr, 16)) return false;
      if (p.f.N > 1 && (st[1] * es) % 16) return false;
      if (p.f.B > 1 && (st[0] * es) % 16) return false;
      return true;
    };
    p.vecbc = bc16(p.f.Bm, p.f.sB) && bc16(p.f.Cm, p.f.sC) ? 1 : 0;
    p.vecout = rows16(p.du, p.sdu) && rows16(p.ddelta, p.sdd) && rows16(p.dz, p.sdz) ? 1 : 0;
    auto g16 = [&](const float* ptr, const int64_t* st) {   // fp32 rows (b, n) of dB / dC
      if (!aligned(ptr, 16) || st[2] != 1) return false;
      if (p.f.N > 1 && (st[1] * 4) % 16) return false;
      if (p.bc_rows > 1 && (st[0] * 4) % 16) return false;
      return true;
    };
    p.vecdbc = g16(p.dB, p.sdB) && g16(p.dC, p.sdC) ? 1 : 0;
  }
  // the checkpoints come from the tiled forward kernel when the layout allows it (one pass, from h0)
  p.sweep = 1;
  if (p.f.L > 0 && tiled_eligible(p.f) && !getenv("SSM_BWD_SWEEP")) {
    ssm_scan_args_t fa = args->fwd;
    fa.y = const_cast<void*>(args->dy);
    std::memcpy(fa.stride_y, args->stride_dy, sizeof(fa.stride_y));
    fa.h_last = nullptr;
    fa.flags = SSM_SCAN_FORCE_TILED;
    ScanPlan plan;
    if (plan_scan(&fa, p.f, &plan) == SSM_OK && plan.path == kPathTiled && plan.shape.K * plan.shape.NS == 16) {
      cudaError_t e = launch_scan_ckpt(p.f, plan, p.ckpt, p.nseg, s);
      if (e != cudaSuccess) return cuda_fail(e);
      p.sweep = 0;
    }
  }
  cudaError_t e = launch_scan_bwd(p, device_sm_count(), s);
  if (e != cudaSuccess) return cuda_fail(e);
  return ok();
}

ssm_status_t ssm_causal_conv1d_fwd(const ssm_conv_args_t* a, void* stream) {
  if (!a) return fail(SSM_ERR_INVALID_ARG, "args is NULL");
  if (a->io_dtype != SSM_F32 && a->io_dtype != SSM_BF16) return fail(SSM_ERR_INVALID_ARG, "io_dtype");
  if (a->batch < 0 || a->dim < 0 || a->seqlen < 0) return fail(SSM_ERR_INVALID_ARG, "negative size");
  if (a->width < 1 || a->width > 16) return fail(SSM_ERR_UNSUPPORTED, "width outside [1, 16]");
  ConvProblem p;
  std::memset(&p, 0, sizeof(p));
  p.B = a->batch; p.D = a->dim; p.L = a->seqlen; p.W = a->width; p.io = a->io_dtype; p.silu = a->silu != 0;
  p.x = a->x; p.w = a->weight; p.bias = a->bias; p.x_hist = a->x_hist; p.out = a->out;
  std::memcpy(p.sx, a->stride_x, sizeof(p.sx));
  std::memcpy(p.so, a->stride_out, sizeof(p.so));
  std::memcpy(p.sw, a->stride_weight, sizeof(p.sw));
  std::memcpy(p.sxh, a->stride_x_hist, sizeof(p.sxh));
  if (p.B == 0 || p.D == 0 || p.L == 0) return ok();
  if (!p.x || !p.w || !p.out) return fail(SSM_ERR_INVALID_ARG, "required pointer is NULL");
  for (int i = 0; i < 3; ++i)
    if (p.sx[i] < 0 || p.so[i] < 0 || p.sxh[i] < 0) return fail(SSM_ERR_INVALID_ARG, "negative stride");
  if (p.sw[0] < 0 || p.sw[1] < 0) return fail(SSM_ERR_INVALID_ARG, "negative stride");
  if (p.sx[2] != 1 || p.so[2] != 1) return fail(SSM_ERR_UNSUPPORTED, "time stride must be 1");
  const int es = elem_size(p.io);
  if (!aligned(p.x, es) || !aligned(p.out, es) || (p.x_hist && !aligned(p.x_hist, es)))
    return fail(SSM_ERR_INVALID_ARG, "misaligned pointer");
  if (!aligned(p.w, 4) || (p.bias && !aligned(p.bias, 4))) return fail(SSM_ERR_INVALID_ARG, "misaligned fp32 pointer");
  int64_t eo[3] = {p.B, p.D, p.L};
  if (!injective(3, eo, p.so)) return fail(SSM_ERR_INVALID_ARG, "out strides overlap");
  uintptr_t o0, o1;
  tensor_range(p.out, 3, eo, p.so, es, &o0, &o1);
  struct In {
    const void* ptr;
    int rank;
    int64_t ext[3];
    const int64_t* str;
    int es;
  } ins[] = {{p.x, 3, {p.B, p.D, p.L}, p.sx, es},
             {p.w, 2, {p.D, p.W, 1}, p.sw, 4},
             {p.x_hist, 3, {p.B, p.D, p.W - 1}, p.sxh, es}};
  for (const In& in : ins) {
    if (!in.ptr || in.ext[in.rank - 1] == 0) continue;
    uintptr_t i0, i1;
    tensor_range(in.ptr, in.rank, in.ext, in.str, in.es, &i0, &i1);
    if (overlaps(o0, o1, i0, i1)) return fail(SSM_ERR_INVALID_ARG, "out overlaps an input");
  }
  if (p.bias) {
    uintptr_t i0 = reinterpret_cast<uintptr_t>(p.bias), i1 = i0 + (uintptr_t)p.D * 4;
    if (overlaps(o0, o1, i0, i1)) return fail(SSM_ERR_INVALID_ARG, "out overlaps an input");
  }
  cudaError_t e = launch_causal_conv1d(p, device_sm_count(), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return ok();
}

// ---------------------------------------------------------------------------
// ssm_ssd_fwd: the Mamba-2 SSD layer
// ---------------------------------------------------------------------------
}  // extern "C"

namespace ssm {
namespace {

ssm_status_t validate_ssd(const ssm_ssd_args_t* a, SsdProblem* p) {
  if (!a) return fail(SSM_ERR_INVALID_ARG, "args is NULL");
  if (a->io_dtype != SSM_F32 && a->io_dtype != SSM_BF16) return fail(SSM_ERR_INVALID_ARG, "io_dtype %d", (int)a->io_dtype);
  if (a->batch < 0 || a->nheads < 0 || a->headdim < 0 || a->seqlen < 0) return fail(SSM_ERR_INVALID_ARG, "negative size");
  if (a->dstate < 1 || a->dstate > 256) return fail(SSM_ERR_UNSUPPORTED, "dstate %lld outside [1, 256]", (long long)a->dstate);
  if (a->flags & ~SSM_SSD_FORCE_GENERIC) return fail(SSM_ERR_INVALID_ARG, "flags 0x%x", (unsigned)a->flags);
  std::memset(p, 0, sizeof(*p));
  p->B = a->batch; p->H = a->nheads; p->P = a->headdim; p->L = a->seqlen; p->N = a->dstate;
  p->io = a->io_dtype;
  p->softplus = a->delta_softplus != 0;
  p->x = a->x; p->delta = a->delta; p->z = a->z; p->Bm = a->Bm; p->Cm = a->Cm;
  p->a = a->A; p->Dskip = a->Dskip; p->bias = a->delta_bias; p->h0 = a->h0; p->h_last = a->h_last; p->y = a->y;
  std::memcpy(p->sx, a->stride_x, sizeof(p->sx));
  std::memcpy(p->sz, a->stride_z, sizeof(p->sz));
  std::memcpy(p->sy, a->stride_y, sizeof(p->sy));
  std::memcpy(p->sd, a->stride_delta, sizeof(p->sd));
  std::memcpy(p->sB, a->stride_B, sizeof(p->sB));
  std::memcpy(p->sC, a->stride_C, sizeof(p->sC));
  std::memcpy(p->sh0, a->stride_h0, sizeof(p->sh0));
  std::memcpy(p->shl, a->stride_h_last, sizeof(p->shl));
  if (p->B == 0 || p->H == 0 || p->P == 0) return ok();
  if (!p->a) return fail(SSM_ERR_INVALID_ARG, "A is NULL");
  const int es = elem_size(p->io);
  const int64_t D = p->H * p->P;
  struct Seq {
    const char* name;
    const void* ptr;
    const int64_t* s;
    bool required;
  } seqs[] = {{"x", p->x, p->sx, true}, {"delta", p->delta, p->sd, true}, {"z", p->z, p->sz, false},
              {"y", p->y, p->sy, true}};
  for (const Seq& q : seqs) {
    if (!q.ptr) {
      if (q.required && p->L > 0) return fail(SSM_ERR_INVALID_ARG, "%s is NULL", q.name);
      continue;
    }
    if (q.s[0] < 0 || q.s[1] < 0) return fail(SSM_ERR_INVALID_ARG, "%s has a negative stride", q.name);
    if (q.s[2] != 1 && p->L > 1) return fail(SSM_ERR_UNSUPPORTED, "%s time stride must be 1", q.name);
    if (!aligned(q.ptr, es)) return fail(SSM_ERR_INVALID_ARG, "%s is not %d-byte aligned", q.name, es);
  }
  for (const void* q : {p->Bm, p->Cm}) {
    if (!q && p->L > 0) return fail(SSM_ERR_INVALID_ARG, "Bm or Cm is NULL");
    if (q && !aligned(q, es)) return fail(SSM_ERR_INVALID_ARG, "Bm or Cm misaligned");
  }
  for (int i = 0; i < 3; ++i)
    if (p->sB[i] < 0 || p->sC[i] < 0) return fail(SSM_ERR_INVALID_ARG, "negative B / C stride");
  for (int i = 0; i < 4; ++i)
    if ((p->h0 && p->sh0[i] < 0) || (p->h_last && p->shl[i] < 0)) return fail(SSM_ERR_INVALID_ARG, "negative state stride");
  for (const float* q : {p->a, p->Dskip, p->bias, p->h0, static_cast<const float*>(p->h_last)})
    if (q && !aligned(q, 4)) return fail(SSM_ERR_INVALID_ARG, "misaligned fp32 pointer");
  // outputs one-to-one and disjoint from every input and from each other
  int64_t ey[3] = {p->B, D, p->L};
  int64_t sy[3] = {p->sy[0], p->sy[1], 1};
  int64_t eh[4] = {p->B, p->H, p->P, p->N};
  if (p->L > 0 && !injective(3, ey, sy)) return fail(SSM_ERR_INVALID_ARG, "y strides overlap");
  if (p->h_last && !injective(4, eh, p->shl)) return fail(SSM_ERR_INVALID_ARG, "h_last strides overlap");
  uintptr_t y0 = 0, y1 = 0, hl0 = 0, hl1 = 0;
  if (p->L > 0) tensor_range(p->y, 3, ey, sy, es, &y0, &y1);
  if (p->h_last) tensor_range(p->h_last, 4, eh, p->shl, 4, &hl0, &hl1);
  struct In {
    const void* ptr;
    int rank;
    int64_t ext[4];
    int64_t str[4];
    int es;
  } ins[] = {
      {p->x, 3, {p->B, D, p->L, 1}, {p->sx[0], p->sx[1], 1, 0}, es},
      {p->delta, 3, {p->B, p->H, p->L, 1}, {p->sd[0], p->sd[1], 1, 0}, es},
      {p->z, 3, {p->B, D, p->L, 1}, {p->sz[0], p->sz[1], 1, 0}, es},
      {p->Bm, 3, {p->B, p->L, p->N, 1}, {p->sB[0], p->sB[1], p->sB[2], 0}, es},
      {p->Cm, 3, {p->B, p->L, p->N, 1}, {p->sC[0], p->sC[1], p->sC[2], 0}, es},
      {p->a, 1, {p->H, 1, 1, 1}, {1, 0, 0, 0}, 4},
      {p->Dskip, 1, {p->H, 1, 1, 1}, {1, 0, 0, 0}, 4},
      {p->bias, 1, {p->H, 1, 1, 1}, {1, 0, 0, 0}, 4},
      {p->h0, 4, {p->B, p->H, p->P, p->N}, {p->sh0[0], p->sh0[1], p->sh0[2], p->sh0[3]}, 4},
  };
  for (const In& in : ins) {
    if (!in.ptr) continue;
    if (in.rank == 3 && p->L == 0 && in.ptr != p->h0) continue;   // empty sequence: nothing is read
    uintptr_t i0, i1;
    tensor_range(in.ptr, in.rank, in.ext, in.str, in.es, &i0, &i1);
    if (p->L > 0 && overlaps(y0, y1, i0, i1)) return fail(SSM_ERR_INVALID_ARG, "y overlaps an input");
    if (p->h_last && overlaps(hl0, hl1, i0, i1)) return fail(SSM_ERR_INVALID_ARG, "h_last overlaps an input");
  }
  if (p->L > 0 && p->h_last && overlaps(y0, y1, hl0, hl1)) return fail(SSM_ERR_INVALID_ARG, "y overlaps h_last");
  if (p->B * p->H > 2147483647LL) return fail(SSM_ERR_UNSUPPORTED, "too many (batch, head) pairs");
  return ok();
}

}  // namespace
}  // namespace ssm

extern "C" {

int ssm_ssd_plan_path(const ssm_ssd_args_t* args) {
  SsdProblem p;
  if (validate_ssd(args, &p) != SSM_OK) return -1;
  if (p.B == 0 || p.H == 0 || p.P == 0 || p.L == 0) return 0;
  return (!(args->flags & SSM_SSD_FORCE_GENERIC) && ssd_tensor_core_eligible(p)) ? 1 : 0;
}

ssm_status_t ssm_ssd_fwd(const ssm_ssd_args_t* args, void* stream) {
  SsdProblem p;
  ssm_status_t st = validate_ssd(args, &p);
  if (st != SSM_OK) return st;
  if (p.B == 0 || p.H == 0 || p.P == 0) return ok();
  const bool tc = !(args->flags & SSM_SSD_FORCE_GENERIC) && ssd_tensor_core_eligible(p);
  if (p.L == 0 && !p.h_last) return ok();
  p.status = device_status_ptr();
  cudaError_t e = launch_ssd(p, tc, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return ok();
}

// ---------------------------------------------------------------------------
// ssm_scan_fwd_noalloc: the chunked scan with its records in a static device
// array instead of a caller workspace (for callers that cannot allocate).
// ---------------------------------------------------------------------------
}  // extern "C"

namespace ssm {
namespace {

// One per device that loads the library, held until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SSM_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array in the current device's context.  It is
// looked up on every call (a host-side query, no allocation), so that a
// context rebuilt after cudaDeviceReset, where the array may sit elsewhere,
// never receives a stale address.  Returns nullptr (and fills *err) if the
// lookup fails.
void* noalloc_scratch(cudaError_t* err) {
  void* p = nullptr;
  *err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  return *err == cudaSuccess ? p : nullptr;
}

}  // namespace
}  // namespace ssm

extern "C" {

ssm_status_t ssm_scan_fwd_noalloc(const ssm_scan_args_t* args, void* stream) {
  ScanProblem p;
  ssm_status_t st = validate_scan(args, &p);
  if (st != SSM_OK) return st;
  if (p.B == 0 || p.D == 0) return ok();
  if (args->flags & ~SSM_SCAN_FORCE_CHUNKED)
    return fail(SSM_ERR_INVALID_ARG, "flags 0x%x: this entry point runs only the chunked path", (unsigned)args->flags);
  ssm_scan_args_t a = *args;
  a.flags = SSM_SCAN_FORCE_CHUNKED;
  a.workspace = nullptr;
  a.workspace_bytes = 0;
  ScanPlan plan;
  st = plan_scan(&a, p, &plan);
  if (st != SSM_OK) return st;
  if (plan.path != kPathChunked)
    return fail(SSM_ERR_UNSUPPORTED, "sequence too short for the chunked path (%lld steps)", (long long)p.L);
  if (plan.workspace_bytes > SSM_NOALLOC_SCRATCH_BYTES)
    return fail(SSM_ERR_WORKSPACE, "needs %zu bytes of chunk records; the static scratch holds %zu",
                plan.workspace_bytes, (size_t)SSM_NOALLOC_SCRATCH_BYTES);
  cudaError_t e = cudaSuccess;
  void* scratch = noalloc_scratch(&e);
  if (!scratch) return cuda_fail(e);
  e = launch_scan_tiled(p, plan, scratch, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return ok();
}

ssm_status_t ssm_get_device_status(void* stream, int clear, int* code) {
  if (!code) return fail(SSM_ERR_INVALID_ARG, "code is NULL");
  *code = SSM_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int host = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&host, g_device_status, sizeof(int), 0, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess && clear && host != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbolAsync(g_device_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  }
  if (e != cudaSuccess) return cuda_fail(e);
  *code = host;
  return ok();
}

}  // extern "C"
