// kda_checks.cu -- device-side checks that stand in for a sanitizer.
//
// 1. The input-precondition pass of the chunked prefill (KDA_CHUNK_CHECK_INPUTS,
//    or KDA_CHECKS=1 in the environment): the tensor-core path is exact only
//    while every log-decay lies in [g_min, 0] with g_min = -5, because then the
//    cumulative log-decay of a 16-token tile stays in (-80, 0] and its inverse
//    decay below e^80, inside the bf16/fp32 range ("Kimi K3 technical report
//    review" (devpress/CSDN), section 3.2; "Kimi K3 architecture" (orkas.ai),
//    section "A lower bound removes a GPU code path").  The write strength beta
//    is a sigmoid output, so it lies in [0, 1].  The pass reads g and beta once
//    and raises the device error flag (kDevErrPrecondition) if any value is out
//    of range or not a number; it changes nothing else.
//
// 2. A self-test of the bounded waits: a kernel whose threads wait on mbarriers
//    that nothing ever signals, with a short limit.  The waits must give up,
//    record kDevErrTimeout, stop the other waiting threads through the CTA's
//    abort word, drain a bulk copy that is really in flight, and return -- the
//    same wait and drain code the prefill kernels use.
#include "kda_internal.cuh"
#include "kda_sm100.cuh"

namespace kda {
namespace {

using namespace sm100;

// One grid-stride pass; each warp votes and one lane writes the flag.
template <typename TB>
__global__ void __launch_bounds__(256) check_inputs_kernel(const float* __restrict__ g,
                                                           int64_t n_g, float g_lo,
                                                           const TB* __restrict__ beta,
                                                           int64_t n_beta, int* err) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  bool bad = false;
  if (g) {
    const int64_t n4 = n_g >> 2;  // whole float4 groups (g is 16-byte aligned)
    const float4* g4 = reinterpret_cast<const float4*>(g);
    for (int64_t i = tid; i < n4; i += stride) {
      const float4 x = __ldcs(g4 + i);
      // a NaN fails both comparisons, so it counts as out of range
      bad |= !(x.x >= g_lo && x.x <= 0.f) | !(x.y >= g_lo && x.y <= 0.f) |
             !(x.z >= g_lo && x.z <= 0.f) | !(x.w >= g_lo && x.w <= 0.f);
    }
    for (int64_t i = 4 * n4 + tid; i < n_g; i += stride) bad |= !(g[i] >= g_lo && g[i] <= 0.f);
  }
  for (int64_t i = tid; i < n_beta; i += stride) {
    const float b = to_f32(beta[i]);
    bad |= !(b >= 0.f && b <= 1.f);
  }
  if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0 && err)
    atomicExch(err, kDevErrPrecondition);
}

// Source of the self-test's bulk copy and the per-warp outcomes it writes.
__device__ __align__(128) uint4 g_selftest_src[256];
__device__ int g_selftest_out[4];

// Wait self-test, one CTA of 128 threads.  Thread 0 puts a 4 KB bulk copy in
// flight on barrier `copy` (it completes normally); warps 0-3 then wait on
// barrier `never`, which nothing signals, through wait_or_abort with the short
// limit: the first to run out records the timeout and raises the abort word, the
// others see it and return.  Thread 0 finally drains the copy with mbar_wait (as
// the prefill kernels drain their copies after an abort).  Each warp writes 1 to
// g_selftest_out[warp] if its wait ended without the barrier completing.
__global__ void __launch_bounds__(128) wait_selftest_kernel(uint64_t timeout_ns, int* err) {
  __shared__ __align__(128) uint4 buf[256];
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ int abort_word;
  const int t = threadIdx.x;
  const uint32_t bar_copy = smem_addr(&bars[0]), bar_never = smem_addr(&bars[1]);
  if (t == 0) {
    mbar_init(bar_copy, 1);
    mbar_init(bar_never, 1);
    abort_word = 0;
    mbar_fence_init();
  }
  __syncthreads();
  if (t == 0) {
    mbar_arrive_expect_tx(bar_copy, sizeof(buf));
    bulk_g2s(smem_addr(buf), g_selftest_src, sizeof(buf), bar_copy);
  }
  const bool ok = wait_or_abort(bar_never, 0, err, &abort_word, timeout_ns);
  if ((t & 31) == 0) g_selftest_out[t >> 5] = ok ? 0 : 1;
  if (t == 0) mbar_wait(bar_copy, 0, err, timeout_ns);  // the copy must land before exit
  __syncthreads();
}

}  // namespace

cudaError_t launch_check_inputs(const float* g, int64_t n_g, float g_lo, const void* beta,
                                int beta_bf16, int64_t n_beta, int* err, cudaStream_t s) {
  if (n_g <= 0 && n_beta <= 0) return cudaSuccess;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t work = (n_g > n_beta ? (n_g + 3) / 4 : n_beta);
  int64_t blocks = (work + 255) / 256;
  if (blocks > 8 * (int64_t)sms) blocks = 8 * (int64_t)sms;
  if (blocks < 1) blocks = 1;
  ProfScope prof_scope("kda_check_inputs", s);
  if (beta_bf16)
    check_inputs_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, s>>>(
        g, n_g, g_lo, static_cast<const __nv_bfloat16*>(beta), n_beta, err);
  else
    check_inputs_kernel<float><<<(unsigned)blocks, 256, 0, s>>>(
        g, n_g, g_lo, static_cast<const float*>(beta), n_beta, err);
  return cudaGetLastError();
}

cudaError_t launch_wait_selftest(uint64_t timeout_ns, int* err, int* warps_gave_up,
                                 cudaStream_t s) {
  const int minus1[4] = {-1, -1, -1, -1};
  cudaError_t e = cudaMemcpyToSymbolAsync(g_selftest_out, minus1, sizeof(minus1), 0,
                                          cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return e;
  {
    ProfScope prof_scope("kda_wait_selftest", s);
    wait_selftest_kernel<<<1, 128, 0, s>>>(timeout_ns, err);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  int out[4];
  e = cudaMemcpyFromSymbolAsync(out, g_selftest_out, sizeof(out), 0, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return e;
  int n = 0;
  for (int w = 0; w < 4; ++w) n += out[w] == 1 ? 1 : 0;
  *warps_gave_up = n;
  return cudaSuccess;
}

}  // namespace kda
