// kda_api.cu -- the C ABI of libkda (declared in include/kda.h): argument
// validation, workspace sizing, the device-side chunk plan and kernel dispatch.
//
// All checks happen on the host before anything is enqueued, so a call that
// returns an error has launched nothing.  Nothing here synchronizes except
// kda_get_device_error().
#include <cmath>
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdlib.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "../../include/kda.h"
#include "kda_internal.cuh"

namespace kda {

// Device error flag: bounded waits and the plan's sequence checks write a code
// here; kda_get_device_error() reads and clears it.
__device__ int g_device_error;

int* device_error_flag() {
  static int* ptrs[64] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<int*>(p);
  }
  return ptrs[dev];
}

// ---------------------------------------------------------------- profiling
namespace {
struct ProfRecord {
  const char* name;
  cudaEvent_t start, stop;
};
struct ProfState {
  std::mutex mu;
  bool on = false;
  ProfRecord* recs = nullptr;
  int n = 0, cap = 0;
  // aggregated results after kda_profile_collect()
  const char* names[64];
  int launches[64];
  double total_ms[64];
  int n_names = 0;
};
ProfState& prof() {
  static ProfState p;
  return p;
}
}  // namespace

ProfScope::ProfScope(const char* name, cudaStream_t s) : slot(-1), stream(s) {
  ProfState& P = prof();
  std::lock_guard<std::mutex> lock(P.mu);
  if (!P.on) return;
  if (P.n == P.cap) {
    const int ncap = P.cap ? 2 * P.cap : 1024;
    ProfRecord* r = static_cast<ProfRecord*>(realloc(P.recs, sizeof(ProfRecord) * ncap));
    if (!r) return;
    P.recs = r;
    P.cap = ncap;
  }
  ProfRecord& rec = P.recs[P.n];
  if (cudaEventCreate(&rec.start) != cudaSuccess) return;
  if (cudaEventCreate(&rec.stop) != cudaSuccess) {
    cudaEventDestroy(rec.start);
    return;
  }
  rec.name = name;
  cudaEventRecord(rec.start, s);
  slot = P.n++;
}

ProfScope::~ProfScope() {
  if (slot < 0) return;
  ProfState& P = prof();
  std::lock_guard<std::mutex> lock(P.mu);
  cudaEventRecord(P.recs[slot].stop, stream);
}

static size_t plan_head_bytes(int n_seqs) {
  const size_t b = 2 * sizeof(int32_t) * (size_t)(n_seqs + 1);
  return (b + 255) & ~size_t(255);
}

size_t plan_bytes(int64_t n_tokens, int n_seqs) {
  const size_t tab = sizeof(int2) * (size_t)chunks_upper_bound(n_tokens, n_seqs);
  return plan_head_bytes(n_seqs) + ((tab + 255) & ~size_t(255));
}

Plan plan_in(void* ws, int64_t n_tokens, int n_seqs) {
  (void)n_tokens;
  Plan plan;
  plan.cu = static_cast<const int32_t*>(ws);
  plan.chunk_off = plan.cu + (n_seqs + 1);
  plan.tab = reinterpret_cast<const int2*>(static_cast<const char*>(ws) + plan_head_bytes(n_seqs));
  plan.n_seqs = n_seqs;
  return plan;
}

// One CTA: writes cu[N+1] (copied from cu_seqlens, or n*T_per_seq), the
// exclusive prefix sum of ceil(len/64) into chunk_off[N+1], and for every chunk
// its first token and token count into tab.  Invalid sequence
// offsets (decreasing, outside [0, NT], cu[0] != 0 or cu[N] != NT) are clamped so
// that no later kernel can index outside the inputs, and flag an error.
__global__ void __launch_bounds__(1024) plan_kernel(const int32_t* __restrict__ cu_in, int n_seqs,
                                                    int64_t T_per_seq, int64_t n_tokens,
                                                    int32_t* __restrict__ cu_out,
                                                    int32_t* __restrict__ chunk_off,
                                                    int2* __restrict__ tab, int* err_flag) {
  __shared__ int32_t warp_sums[32];
  __shared__ int32_t carry;
  const int tid = threadIdx.x;
  if (tid == 0) {
    carry = 0;
  }
  __syncthreads();
  bool bad = false;
  for (int base = 0; base <= n_seqs; base += blockDim.x) {
    const int n = base + tid;
    int32_t cu_n = 0, nchunks = 0;
    if (n <= n_seqs) {
      int64_t x = cu_in ? (int64_t)cu_in[n] : (int64_t)n * T_per_seq;
      if (n == 0 && x != 0) bad = true;
      if (n == n_seqs && x != n_tokens) bad = true;
      if (x < 0) { x = 0; bad = true; }
      if (x > n_tokens) { x = n_tokens; bad = true; }
      cu_n = (int32_t)x;
      cu_out[n] = cu_n;
    }
    __syncthreads();
    if (n < n_seqs) {
      int64_t nx = cu_in ? (int64_t)cu_in[n + 1] : (int64_t)(n + 1) * T_per_seq;
      if (nx > n_tokens) nx = n_tokens;
      if (nx < cu_n) { nx = cu_n; bad = true; }
      nchunks = (int32_t)((nx - cu_n + kChunk - 1) / kChunk);
    }
    // block-wide exclusive scan of nchunks
    int32_t v = nchunks;
    const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += y;
    }
    if (lane == 31) warp_sums[warp] = v;
    __syncthreads();
    if (warp == 0) {
      int32_t w = lane < (int)(blockDim.x >> 5) ? warp_sums[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      warp_sums[lane] = w;
    }
    __syncthreads();
    const int32_t incl = v + (warp > 0 ? warp_sums[warp - 1] : 0);
    if (n <= n_seqs) chunk_off[n] = carry + incl - nchunks;
    __syncthreads();
    if (tid == blockDim.x - 1) carry += incl;
    __syncthreads();
  }
  __syncthreads();
  const int total = chunk_off[n_seqs];
  for (int j = tid; j < total; j += blockDim.x) {
    int lo = 0, hi = n_seqs - 1;  // the last sequence whose chunks start at or before j
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (chunk_off[mid] <= j) lo = mid; else hi = mid - 1;
    }
    const int64_t t0 = (int64_t)cu_out[lo] + (int64_t)(j - chunk_off[lo]) * kChunk;
    const int64_t end = cu_out[lo + 1];
    tab[j] = make_int2((int)t0, (int)(end - t0 < kChunk ? end - t0 : kChunk));
  }
  if (bad && err_flag) atomicExch(err_flag, kDevErrBadSeqlens);
}

cudaError_t launch_plan(const int32_t* cu_seqlens_or_null, int n_seqs, int64_t T_per_seq,
                        int64_t n_tokens, void* ws, int* err_flag, cudaStream_t s) {
  const Plan plan = plan_in(ws, n_tokens, n_seqs);
  ProfScope prof_scope("kda_plan", s);
  plan_kernel<<<1, 1024, 0, s>>>(cu_seqlens_or_null, n_seqs, T_per_seq, n_tokens,
                                 const_cast<int32_t*>(plan.cu),
                                 const_cast<int32_t*>(plan.chunk_off),
                                 const_cast<int2*>(plan.tab), err_flag);
  return cudaGetLastError();
}

}  // namespace kda

// ============================================================================ C ABI
namespace {

thread_local char t_err[512] = "no error";

kda_status_t fail(kda_status_t st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_err, sizeof(t_err), fmt, ap);
  va_end(ap);
  return st;
}

kda_status_t cuda_fail(cudaError_t e, const char* what) {
  return fail(KDA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// KDA_CHECKS=1 (any value but "0" or empty) in the environment turns the input
// precondition pass on for every chunk call; read once per process.
bool checks_from_env() {
  static const bool on = [] {
    const char* v = getenv("KDA_CHECKS");
    return v && v[0] && strcmp(v, "0") != 0;
  }();
  return on;
}

// Byte offset, in the workspace of the fp32-core path, of the scalar gates spread
// over the channels (after the plan and that path's own scratch, 256-aligned).
size_t simt_scalar_gate_offset(int64_t n_tokens, int n_seqs, int H) {
  const size_t b = kda::plan_bytes(n_tokens, n_seqs) + kda::simt_workspace_bytes(n_tokens, n_seqs, H);
  return (b + 255) & ~(size_t)255;
}

kda_status_t check_device() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3)
    return fail(KDA_ERR_NO_DEVICE, "device %d is sm_%d%d; libkda is built for sm_103a only", dev,
                major, minor);
  return KDA_OK;
}

}  // namespace

namespace kda {
// Lets other translation units of the library set the message that
// kda_last_error_string() returns on this thread.
void set_error_message(const char* msg) { fail(KDA_OK, "%s", msg); }
}  // namespace kda

extern "C" {

const char* kda_version(void) { return "0.1.0"; }

int kda_profile_enable(int on) {
  kda::ProfState& P = kda::prof();
  std::lock_guard<std::mutex> lock(P.mu);
  for (int i = 0; i < P.n; ++i) {
    cudaEventDestroy(P.recs[i].start);
    cudaEventDestroy(P.recs[i].stop);
  }
  P.n = 0;
  P.n_names = 0;
  P.on = on != 0;
  return 0;
}

int kda_profile_collect(void) {
  kda::ProfState& P = kda::prof();
  std::lock_guard<std::mutex> lock(P.mu);
  P.n_names = 0;
  for (int i = 0; i < P.n; ++i) {
    if (cudaEventSynchronize(P.recs[i].stop) != cudaSuccess) return -1;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, P.recs[i].start, P.recs[i].stop) != cudaSuccess) return -1;
    int j = 0;
    while (j < P.n_names && strcmp(P.names[j], P.recs[i].name) != 0) ++j;
    if (j == P.n_names) {
      if (P.n_names == 64) continue;
      P.names[j] = P.recs[i].name;
      P.launches[j] = 0;
      P.total_ms[j] = 0.0;
      ++P.n_names;
    }
    P.launches[j] += 1;
    P.total_ms[j] += ms;
  }
  return P.n_names;
}

int kda_profile_get(int i, const char** name, int* launches, double* total_ms) {
  kda::ProfState& P = kda::prof();
  std::lock_guard<std::mutex> lock(P.mu);
  if (i < 0 || i >= P.n_names || !name || !launches || !total_ms) return -1;
  *name = P.names[i];
  *launches = P.launches[i];
  *total_ms = P.total_ms[i];
  return 0;
}

const char* kda_last_error_string(void) { return t_err; }

kda_status_t kda_get_device_error(kda_stream_t stream) {
  int* flag = kda::device_error_flag();
  if (!flag) return fail(KDA_ERR_CUDA, "device error flag unavailable");
  int host = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(&host, flag, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "reading device error flag");
  if (host == 0) return KDA_OK;
  const int zero = 0;
  e = cudaMemcpyAsync(flag, &zero, sizeof(int), cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "clearing device error flag");
  if (host == kda::kDevErrTimeout)
    return fail(KDA_ERR_DEVICE_TIMEOUT, "a bounded device-side wait gave up");
  if (host == kda::kDevErrCkptCapacity)
    return fail(KDA_ERR_INVALID_ARG,
                "more state checkpoints than ckpt_capacity (the excess was not written)");
  if (host == kda::kDevErrBadSeqlens)
    return fail(KDA_ERR_INVALID_ARG,
                "cu_seqlens was not nondecreasing from 0 to n_tokens (clamped on the device)");
  if (host == kda::kDevErrPrecondition)
    return fail(KDA_ERR_INVALID_ARG,
                "input check: a log-decay g outside [-5, 0] (outside (-inf, 0] with "
                "KDA_CHUNK_UNBOUNDED_GATE) or a beta outside [0, 1], or a NaN");
  return fail(KDA_ERR_CUDA, "device error code %d", host);
}

kda_status_t kda_selftest_wait_timeout(uint32_t timeout_us, int* warps_gave_up,
                                       kda_stream_t stream) {
  if (timeout_us < 1 || timeout_us > 1000000u)
    return fail(KDA_ERR_INVALID_ARG, "kda_selftest_wait_timeout: timeout_us=%u (1..1000000)",
                timeout_us);
  if (!warps_gave_up) return fail(KDA_ERR_INVALID_ARG, "kda_selftest_wait_timeout: null output");
  kda_status_t st = check_device();
  if (st != KDA_OK) return st;
  int* flag = kda::device_error_flag();
  if (!flag) return fail(KDA_ERR_CUDA, "device error flag unavailable");
  const cudaError_t e = kda::launch_wait_selftest((uint64_t)timeout_us * 1000u, flag,
                                                  warps_gave_up,
                                                  reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kda_selftest_wait_timeout");
  return KDA_OK;
}

kda_status_t kda_gate(const void* z, int z_dtype, const float* A, float g_min, float* g,
                      int64_t n_tokens, int H, int dk, float* gcum, const int32_t* cu_seqlens,
                      int n_seqs, kda_stream_t stream) {
  if (z_dtype != KDA_F32 && z_dtype != KDA_BF16)
    return fail(KDA_ERR_UNSUPPORTED_DTYPE, "kda_gate: z_dtype %d", z_dtype);
  if (dk != kda::kD) return fail(KDA_ERR_UNSUPPORTED_SHAPE, "kda_gate: dk=%d (need 128)", dk);
  if (H < 1) return fail(KDA_ERR_UNSUPPORTED_SHAPE, "kda_gate: H=%d", H);
  if (n_tokens < 0 || n_tokens > INT32_MAX)
    return fail(KDA_ERR_INVALID_ARG, "kda_gate: n_tokens=%lld", (long long)n_tokens);
  if (!(g_min < 0.f)) return fail(KDA_ERR_INVALID_ARG, "kda_gate: g_min must be < 0");
  if (n_tokens == 0) return KDA_OK;
  if (!z || !A || !g) return fail(KDA_ERR_INVALID_ARG, "kda_gate: null z, A or g");
  if (!aligned16(z) || !aligned16(g) || (gcum && !aligned16(gcum)))
    return fail(KDA_ERR_MISALIGNED, "kda_gate: z, g, gcum must be 16-byte aligned");
  if (gcum && cu_seqlens && n_seqs < 1)
    return fail(KDA_ERR_INVALID_ARG, "kda_gate: n_seqs=%d with cu_seqlens", n_seqs);
  kda_status_t st = check_device();
  if (st != KDA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (gcum)
    e = kda::launch_gate_cumsum(z, z_dtype == KDA_BF16, A, g_min, g, gcum, n_tokens, H,
                                cu_seqlens, cu_seqlens ? n_seqs : 1, s);
  else
    e = kda::launch_gate(z, z_dtype == KDA_BF16, A, g_min, g, n_tokens, H, s);
  if (e != cudaSuccess) return cuda_fail(e, "kda_gate launch");
  return KDA_OK;
}

kda_status_t kda_gate_softplus(const void* z, int z_dtype, const float* A, float* g,
                               int64_t n_tokens, int H, int dk, kda_stream_t stream) {
  if (z_dtype != KDA_F32 && z_dtype != KDA_BF16)
    return fail(KDA_ERR_UNSUPPORTED_DTYPE, "kda_gate_softplus: z_dtype %d", z_dtype);
  if (dk != kda::kD) return fail(KDA_ERR_UNSUPPORTED_SHAPE, "kda_gate_softplus: dk=%d", dk);
  if (H < 1) return fail(KDA_ERR_UNSUPPORTED_SHAPE, "kda_gate_softplus: H=%d", H);
  if (n_tokens < 0 || n_tokens > INT32_MAX)
    return fail(KDA_ERR_INVALID_ARG, "kda_gate_softplus: n_tokens=%lld", (long long)n_tokens);
  if (n_tokens == 0) return KDA_OK;
  if (!z || !A || !g) return fail(KDA_ERR_INVALID_ARG, "kda_gate_softplus: null z, A or g");
  if (!aligned16(z) || !aligned16(g))
    return fail(KDA_ERR_MISALIGNED, "kda_gate_softplus: z, g must be 16-byte aligned");
  kda_status_t st = check_device();
  if (st != KDA_OK) return st;
  cudaError_t e = kda::launch_gate_softplus(z, z_dtype == KDA_BF16, A, g, n_tokens, H,
                                            reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kda_gate_softplus launch");
  return KDA_OK;
}

kda_status_t kda_output_gate(const void* o, int dtype, const void* gate, const float* weight,
                             float eps, void* y, int64_t n_tokens, int H, int dv,
                             kda_stream_t stream) {
  const char* fn = "kda_output_gate";
  if (dtype != KDA_F32 && dtype != KDA_BF16)
    return fail(KDA_ERR_UNSUPPORTED_DTYPE, "%s: dtype %d", fn, dtype);
  if (dv != kda::kD) return fail(KDA_ERR_UNSUPPORTED_SHAPE, "%s: dv=%d (need 128)", fn, dv);
  if (H < 1) return fail(KDA_ERR_UNSUPPORTED_SHAPE, "%s: H=%d", fn, H);
  if (n_tokens < 0 || n_tokens > INT32_MAX)
    return fail(KDA_ERR_INVALID_ARG, "%s: n_tokens=%lld", fn, (long long)n_tokens);
  if (!(eps >= 0.f && std::isfinite(eps)))
    return fail(KDA_ERR_INVALID_ARG, "%s: eps=%g (need finite, >= 0)", fn, (double)eps);
  if (n_tokens == 0) return KDA_OK;
  if (!o || !gate || !y) return fail(KDA_ERR_INVALID_ARG, "%s: null o, gate or y", fn);
  if (!aligned16(o) || !aligned16(gate) || !aligned16(y) || (weight && !aligned16(weight)))
    return fail(KDA_ERR_MISALIGNED, "%s: pointers must be 16-byte aligned", fn);
  kda_status_t st = check_device();
  if (st != KDA_OK) return st;
  cudaError_t e = kda::launch_output_gate(o, dtype == KDA_BF16, gate, weight, eps, y, n_tokens,
                                          H, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kda_output_gate launch");
  return KDA_OK;
}

size_t kda_chunk_fwd_workspace_size_ex(int64_t n_tokens, int n_seqs, int H, int dtype,
                                       unsigned flags) {
  if (n_tokens < 0 || n_seqs < 1 || H < 1) return 0;
  if (dtype == KDA_BF16 && !(flags & (KDA_CHUNK_FP32_CORES | KDA_CHUNK_UNBOUNDED_GATE))) {
    const int segc = kda::chain_segment_chunks(n_tokens, n_seqs, H, (int)(flags >> 16),
                                               (flags & KDA_CHUNK_SEQUENTIAL) != 0);
    return kda::plan_bytes(n_tokens, n_seqs) +
           kda::tc_workspace_bytes(n_tokens, n_seqs, H, segc, (flags & KDA_CHUNK_PRECISE) != 0);
  }
  if (dtype == KDA_F32 || dtype == KDA_BF16) {
    if (!(flags & KDA_CHUNK_SCALAR_GATE))
      return kda::plan_bytes(n_tokens, n_seqs) + kda::simt_workspace_bytes(n_tokens, n_seqs, H);
    return simt_scalar_gate_offset(n_tokens, n_seqs, H) +
           (size_t)n_tokens * H * kda::kD * sizeof(float);  // the spread gates
  }
  return 0;
}

size_t kda_chunk_fwd_workspace_size(int64_t n_tokens, int n_seqs, int H, int dtype) {
  return kda_chunk_fwd_workspace_size_ex(n_tokens, n_seqs, H, dtype, 0u);
}

}  // extern "C"

namespace {

// Shared body of the chunk entry points.  Exactly one of g and z is non-null; with
// z the gate is evaluated inside the tensor-core prepare kernel (bf16 only).
kda_status_t chunk_fwd_impl(const char* fn, const void* q, const void* k, const void* v,
                            int dtype, const float* g, const void* z, const float* A,
                            float g_min, const void* beta, const float* h0,
                            const int32_t* cu_seqlens, int n_seqs, int B, int64_t T, int H,
                            int dk, int dv, void* o, float* hT, void* workspace,
                            size_t ws_bytes, kda_stream_t stream, unsigned flags,
                            kda::CkptArgs ck = kda::CkptArgs{nullptr, 0, 0},
                            kda::FuseArgs fz = kda::FuseArgs{-1.f, nullptr, nullptr, 0.f}) {
  if (dtype != KDA_F32 && dtype != KDA_BF16)
    return fail(KDA_ERR_UNSUPPORTED_DTYPE, "%s: dtype %d", fn, dtype);
  if (dk != kda::kD || dv != kda::kD)
    return fail(KDA_ERR_UNSUPPORTED_SHAPE, "%s: dk=%d dv=%d (need 128)", fn, dk, dv);
  if (H < 1) return fail(KDA_ERR_UNSUPPORTED_SHAPE, "%s: H=%d", fn, H);
  int N;
  int64_t NT, T_per_seq = 0;
  if (cu_seqlens) {
    if (B != 1) return fail(KDA_ERR_INVALID_ARG, "%s: B must be 1 with cu_seqlens", fn);
    if (n_seqs < 1) return fail(KDA_ERR_INVALID_ARG, "%s: n_seqs=%d", fn, n_seqs);
    N = n_seqs;
    NT = T;
  } else {
    if (B < 1) return fail(KDA_ERR_INVALID_ARG, "%s: B=%d", fn, B);
    N = B;
    NT = (int64_t)B * T;
    T_per_seq = T;
  }
  if (T < 0 || NT > INT32_MAX - 2 * kda::kChunk)
    return fail(KDA_ERR_INVALID_ARG, "%s: token count out of range", fn);
  if ((NT > 0 && (!q || !k || !v || !(g || (z && A)) || !beta || !o)) || (N > 0 && !workspace))
    return fail(KDA_ERR_INVALID_ARG, "%s: null required pointer", fn);
  const void* ptrs[] = {q, k, v, g, z, beta, h0, o, hT};
  for (const void* p : ptrs)
    if (p && !aligned16(p))
      return fail(KDA_ERR_MISALIGNED, "%s: pointers must be 16-byte aligned", fn);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(KDA_ERR_MISALIGNED, "%s: workspace must be 256-byte aligned", fn);
  const size_t need = kda_chunk_fwd_workspace_size_ex(NT, N, H, dtype, flags);
  if (ws_bytes < need)
    return fail(KDA_ERR_WORKSPACE_TOO_SMALL, "%s: workspace %zu < %zu bytes", fn,
                ws_bytes, need);
  if (flags & ~(unsigned)(KDA_CHUNK_FP32_CORES | KDA_CHUNK_SEQUENTIAL |
                          KDA_CHUNK_UNBOUNDED_GATE | KDA_CHUNK_SCALAR_GATE |
                          KDA_CHUNK_CHECK_INPUTS | KDA_CHUNK_PRECISE | 0xffff0000u))
    return fail(KDA_ERR_INVALID_ARG, "%s: unknown flags 0x%x", fn, flags);
  if ((flags & KDA_CHUNK_UNBOUNDED_GATE) && z)
    return fail(KDA_ERR_INVALID_ARG, "%s: the unbounded-gate mode takes g, not z", fn);
  if ((flags & KDA_CHUNK_SCALAR_GATE) && z)
    return fail(KDA_ERR_INVALID_ARG, "%s: the scalar-gate mode takes g, not z", fn);
  const bool scalar_g = (flags & KDA_CHUNK_SCALAR_GATE) != 0;
  kda_status_t st = check_device();
  if (st != KDA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int* err = kda::device_error_flag();
  cudaError_t e;
  if (((flags & KDA_CHUNK_CHECK_INPUTS) || checks_from_env()) && NT > 0) {
    // the precondition pass: g in [-5, 0] (any finite g <= 0 in the unbounded mode)
    // and beta in [0, 1]; a gate formed from z is in range by construction
    const float g_lo = (flags & KDA_CHUNK_UNBOUNDED_GATE) ? -3.402823466e38f : -5.f;
    const int64_t n_g = g ? NT * H * (scalar_g ? 1 : kda::kD) : 0;
    e = kda::launch_check_inputs(g, n_g, g_lo, beta, dtype == KDA_BF16, NT * H, err, s);
    if (e != cudaSuccess) return cuda_fail(e, "input check launch");
  }
  e = kda::launch_plan(cu_seqlens, N, T_per_seq, NT, workspace, err, s);
  if (e != cudaSuccess) return cuda_fail(e, "chunk plan launch");
  if (dtype == KDA_BF16 && !(flags & (KDA_CHUNK_FP32_CORES | KDA_CHUNK_UNBOUNDED_GATE))) {
    e = kda::launch_chunk_tc(q, k, v, g, z, A, g_min, beta, h0, o, hT, NT, N, H,
                             kda::chain_segment_chunks(NT, N, H, (int)(flags >> 16),
                                                       (flags & KDA_CHUNK_SEQUENTIAL) != 0),
                             ck, fz, scalar_g, (flags & KDA_CHUNK_PRECISE) != 0, workspace,
                             err, s);

  } else {
    const float* gf = g;
    if (scalar_g) {  // this path reads per-channel decays: spread the scalar ones first
      float* gx = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                           simt_scalar_gate_offset(NT, N, H));
      e = kda::launch_expand_scalar_gate(g, gx, NT, H, s);
      if (e != cudaSuccess) return cuda_fail(e, "scalar gate launch");
      gf = gx;
    }
    e = kda::launch_chunk_simt(q, k, v, dtype == KDA_BF16, gf, beta, h0, o, hT, NT, N, H,
                               workspace, s, (flags & KDA_CHUNK_UNBOUNDED_GATE) ? 1 : 0);
  }
  if (e != cudaSuccess) return cuda_fail(e, "chunk launch");
  return KDA_OK;
}

}  // namespace

extern "C" {

kda_status_t kda_chunk_fwd_ex(const void* q, const void* k, const void* v, int dtype,
                              const float* g, const void* beta, const float* h0,
                              const int32_t* cu_seqlens, int n_seqs, int B, int64_t T, int H,
                              int dk, int dv, void* o, float* hT, void* workspace,
                              size_t ws_bytes, kda_stream_t stream, unsigned flags) {
  return chunk_fwd_impl("kda_chunk_fwd", q, k, v, dtype, g, nullptr, nullptr, 0.f, beta, h0,
                        cu_seqlens, n_seqs, B, T, H, dk, dv, o, hT, workspace, ws_bytes, stream,
                        flags);
}

kda_status_t kda_chunk_fwd_gated(const void* q, const void* k, const void* v, int dtype,
                                 const void* z, const float* A, float g_min, const void* beta,
                                 const float* h0, const int32_t* cu_seqlens, int n_seqs, int B,
                                 int64_t T, int H, int dk, int dv, void* o, float* hT,
                                 void* workspace, size_t ws_bytes, kda_stream_t stream) {
  if (dtype != KDA_BF16)
    return fail(KDA_ERR_UNSUPPORTED_DTYPE,
                "kda_chunk_fwd_gated: dtype %d (bf16 only; for fp32 call kda_gate first)", dtype);
  if (!(g_min >= -5.f && g_min < 0.f))
    return fail(KDA_ERR_INVALID_ARG, "kda_chunk_fwd_gated: g_min=%g outside [-5, 0)",
                (double)g_min);
  return chunk_fwd_impl("kda_chunk_fwd_gated", q, k, v, dtype, nullptr, z, A, g_min, beta, h0,
                        cu_seqlens, n_seqs, B, T, H, dk, dv, o, hT, workspace, ws_bytes, stream,
                        0u);
}

kda_status_t kda_chunk_fwd_checkpointed(const void* q, const void* k, const void* v, int dtype,
                                        const float* g, const void* beta, const float* h0,
                                        const int32_t* cu_seqlens, int n_seqs, int B, int64_t T,
                                        int H, int dk, int dv, void* o, float* hT, float* ckpt,
                                        int ckpt_tokens, int64_t ckpt_capacity, void* workspace,
                                        size_t ws_bytes, kda_stream_t stream, unsigned flags) {
  const char* fn = "kda_chunk_fwd_checkpointed";
  if (dtype != KDA_BF16 || (flags & (KDA_CHUNK_FP32_CORES | KDA_CHUNK_UNBOUNDED_GATE)))
    return fail(KDA_ERR_UNSUPPORTED_DTYPE, "%s: bf16 on the tensor-core path only", fn);
  if (ckpt_tokens < kda::kChunk || ckpt_tokens % kda::kChunk != 0)
    return fail(KDA_ERR_INVALID_ARG, "%s: ckpt_tokens=%d (a positive multiple of %d)", fn,
                ckpt_tokens, kda::kChunk);
  if (ckpt_capacity < 0 || (ckpt_capacity > 0 && !ckpt))
    return fail(KDA_ERR_INVALID_ARG, "%s: ckpt_capacity=%lld with ckpt=%p", fn,
                (long long)ckpt_capacity, (void*)ckpt);
  if (ckpt && (reinterpret_cast<uintptr_t>(ckpt) & 31u) != 0)
    return fail(KDA_ERR_MISALIGNED, "%s: ckpt must be 32-byte aligned", fn);
  return chunk_fwd_impl(fn, q, k, v, dtype, g, nullptr, nullptr, 0.f, beta, h0, cu_seqlens,
                        n_seqs, B, T, H, dk, dv, o, hT, workspace, ws_bytes, stream, flags,
                        kda::CkptArgs{ckpt_capacity > 0 ? ckpt : nullptr,
                                      ckpt_tokens / kda::kChunk, ckpt_capacity});
}

kda_status_t kda_chunk_fwd_fused(const void* q, const void* k, const void* v, int dtype,
                                 const float* g, const void* z, const float* A, float g_min,
                                 const void* beta, const float* h0, const int32_t* cu_seqlens,
                                 int n_seqs, int B, int64_t T, int H, int dk, int dv,
                                 float qk_l2_eps, const void* out_gate,
                                 const float* out_norm_weight, float out_norm_eps, void* o,
                                 float* hT, void* workspace, size_t ws_bytes, kda_stream_t stream,
                                 unsigned flags) {
  const char* fn = "kda_chunk_fwd_fused";
  if (dtype != KDA_BF16 || (flags & (KDA_CHUNK_FP32_CORES | KDA_CHUNK_UNBOUNDED_GATE)))
    return fail(KDA_ERR_UNSUPPORTED_DTYPE, "%s: bf16 on the tensor-core path only", fn);
  if ((g != nullptr) == (z != nullptr))
    return fail(KDA_ERR_INVALID_ARG, "%s: give exactly one of g and z", fn);
  if (z && !(g_min >= -5.f && g_min < 0.f))
    return fail(KDA_ERR_INVALID_ARG, "%s: g_min=%g outside [-5, 0)", fn, (double)g_min);
  if (!(qk_l2_eps < 0.f || std::isfinite(qk_l2_eps)))
    return fail(KDA_ERR_INVALID_ARG, "%s: qk_l2_eps is not finite", fn);
  if (out_gate && !(out_norm_eps >= 0.f && std::isfinite(out_norm_eps)))
    return fail(KDA_ERR_INVALID_ARG, "%s: out_norm_eps=%g (need finite, >= 0)", fn,
                (double)out_norm_eps);
  if ((out_gate && !aligned16(out_gate)) || (out_norm_weight && !aligned16(out_norm_weight)))
    return fail(KDA_ERR_MISALIGNED, "%s: out_gate, out_norm_weight must be 16-byte aligned", fn);
  if (out_norm_weight && !out_gate)
    return fail(KDA_ERR_INVALID_ARG, "%s: out_norm_weight without out_gate", fn);
  return chunk_fwd_impl(fn, q, k, v, dtype, g, z, A, g_min, beta, h0, cu_seqlens, n_seqs, B, T, H,
                        dk, dv, o, hT, workspace, ws_bytes, stream, flags,
                        kda::CkptArgs{nullptr, 0, 0},
                        kda::FuseArgs{qk_l2_eps < 0.f ? -1.f : qk_l2_eps, out_gate,
                                      out_norm_weight, out_norm_eps});
}

kda_status_t kda_chunk_fwd(const void* q, const void* k, const void* v, int dtype,
                           const float* g, const void* beta, const float* h0,
                           const int32_t* cu_seqlens, int n_seqs, int B, int64_t T, int H,
                           int dk, int dv, void* o, float* hT, void* workspace, size_t ws_bytes,
                           kda_stream_t stream) {
  return kda_chunk_fwd_ex(q, k, v, dtype, g, beta, h0, cu_seqlens, n_seqs, B, T, H, dk, dv, o, hT,
                          workspace, ws_bytes, stream, 0u);
}

kda_status_t kda_recurrent_step(const void* q, const void* k, const void* v, int dtype,
                                const float* g, const void* beta, float* S, void* o, int N, int H,
                                int dk, int dv, kda_stream_t stream) {
  if (dtype != KDA_F32 && dtype != KDA_BF16)
    return fail(KDA_ERR_UNSUPPORTED_DTYPE, "kda_recurrent_step: dtype %d", dtype);
  if (dk != kda::kD || dv != kda::kD)
    return fail(KDA_ERR_UNSUPPORTED_SHAPE, "kda_recurrent_step: dk=%d dv=%d (need 128)", dk, dv);
  if (H < 1 || N < 0) return fail(KDA_ERR_UNSUPPORTED_SHAPE, "kda_recurrent_step: N=%d H=%d", N, H);
  if ((int64_t)N * H > INT32_MAX)
    return fail(KDA_ERR_INVALID_ARG, "kda_recurrent_step: N*H too large");
  if (N == 0) return KDA_OK;
  if (!q || !k || !v || !g || !beta || !S || !o)
    return fail(KDA_ERR_INVALID_ARG, "kda_recurrent_step: null pointer");
  const void* ptrs[] = {q, k, v, g, S, o};
  for (const void* p : ptrs)
    if (!aligned16(p))
      return fail(KDA_ERR_MISALIGNED, "kda_recurrent_step: pointers must be 16-byte aligned");
  kda_status_t st = check_device();
  if (st != KDA_OK) return st;
  cudaError_t e = kda::launch_decode(q, k, v, dtype == KDA_BF16, g, beta, S, o, N, H,
                                     reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kda_recurrent_step launch");
  return KDA_OK;
}

kda_status_t kda_recurrent_multi_step(const void* q, const void* k, const void* v, int dtype,
                                      const float* g, const void* beta, float* S, void* o,
                                      const int32_t* n_advance, int N, int T, int H, int dk,
                                      int dv, kda_stream_t stream) {
  if (dtype != KDA_F32 && dtype != KDA_BF16)
    return fail(KDA_ERR_UNSUPPORTED_DTYPE, "kda_recurrent_multi_step: dtype %d", dtype);
  if (dk != kda::kD || dv != kda::kD)
    return fail(KDA_ERR_UNSUPPORTED_SHAPE, "kda_recurrent_multi_step: dk=%d dv=%d (need 128)",
                dk, dv);
  if (H < 1 || N < 0 || T < 1 || T > KDA_MULTI_STEP_MAX_T)
    return fail(KDA_ERR_UNSUPPORTED_SHAPE, "kda_recurrent_multi_step: N=%d T=%d H=%d", N, T, H);
  if ((int64_t)N * H > INT32_MAX)
    return fail(KDA_ERR_INVALID_ARG, "kda_recurrent_multi_step: N*H too large");
  if (N == 0) return KDA_OK;
  if (!q || !k || !v || !g || !beta || !S)
    return fail(KDA_ERR_INVALID_ARG, "kda_recurrent_multi_step: null pointer");
  const void* ptrs[] = {q, k, v, g, S, o};
  for (const void* p : ptrs)
    if (p && !aligned16(p))
      return fail(KDA_ERR_MISALIGNED, "kda_recurrent_multi_step: pointers must be 16-byte aligned");
  kda_status_t st = check_device();
  if (st != KDA_OK) return st;
  cudaError_t e = kda::launch_decode_multi(q, k, v, dtype == KDA_BF16, g, beta, S, o, n_advance,
                                           N, T, H, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kda_recurrent_multi_step launch");
  return KDA_OK;
}

}  // extern "C"
