// kda_gate.cu -- K1: the bounded log-decay of KDA,
//     g = g_min * Sigmoid(exp(A_h) * z)        ("Kimi K3 technical report review"
//                                               (devpress/CSDN), section 3.2, Eq. 5)
// and, optionally, its running sum inside each 64-token chunk of each sequence
// (the log of the in-chunk cumulative decay Gamma of the chunkwise form,
// "Kimi K3 notes" (s1mplewind blog), section "Chunkwise form").
//
// The unbounded gate it replaces, g = -exp(A_h) * Softplus(z) (Kimi Linear, the same
// review, section 3.2), is formed by the same kernel for the range-robust mode.
//
// Memory-bound elementwise work: 8-element groups, four per thread in flight
// (16-byte bf16 or 32-byte fp32 loads, 32-byte stores), grid-stride over a grid
// sized to the SM count.
#include "kda_internal.cuh"

namespace kda {
namespace {

__device__ __forceinline__ float bounded_decay(float z, float scale, float g_min) {
  // g_min * Sigmoid(x) = g_min / (1 + exp(-x)); exp(-x) -> inf gives 0 (the fast
  // quotient multiplies by the reciprocal, which is 0), -> 0 gives g_min.
  return __fdividef(g_min, 1.0f + __expf(-scale * z));
}

// -scale * Softplus(z), Softplus(x) = log(1 + e^x) (= x to fp32 precision above 20)
__device__ __forceinline__ float softplus_decay(float z, float scale) {
  return -scale * (z > 20.f ? z : log1pf(expf(z)));
}

template <typename Tz, bool kSoftplus = false>
__global__ void __launch_bounds__(256) gate_kernel(const Tz* __restrict__ z,
                                                   const float* __restrict__ A, float g_min,
                                                   float* __restrict__ g, int64_t n_groups,
                                                   int H) {
  // group = 8 consecutive channels of one (token, head), kD / 8 = 16 groups per
  // (t, h).  Each thread takes four groups one grid stride apart (every access of a
  // warp is one contiguous span) and issues their loads before any store.  The grid
  // stride is a whole number of (token, head) rows, so the head index of the next
  // group steps by a constant: one division per thread.
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t g0 = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (g0 >= n_groups) return;
  int h = (int)((g0 >> 4) % H);
  const int hstep = (int)((stride >> 4) % H);
  for (int64_t grp = g0; grp < n_groups; grp += 4 * stride) {
    float x[4][8];
    int hj[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      hj[j] = h;
      h += hstep;
      if (h >= H) h -= H;
      if (grp + j * stride < n_groups) load8(z + (grp + j * stride) * 8, x[j]);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (grp + j * stride >= n_groups) break;
      const float scale = expf(__ldg(A + hj[j]));
      float y[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        y[i] = kSoftplus ? softplus_decay(x[j][i], scale) : bounded_decay(x[j][i], scale, g_min);
      float4* out = reinterpret_cast<float4*>(g + (grp + j * stride) * 8);
      out[0] = make_float4(y[0], y[1], y[2], y[3]);
      out[1] = make_float4(y[4], y[5], y[6], y[7]);
    }
  }
}

// One CTA per (64-token window, head); thread c walks the window's tokens for
// channel c, resetting the running sum at every chunk start (cu[n] + 64 m).  A
// window that begins inside a chunk first re-accumulates that chunk's earlier
// tokens.  Stores are coalesced across the 128 channel threads.
template <typename Tz>
__global__ void __launch_bounds__(128) gate_cumsum_kernel(const Tz* __restrict__ z,
                                                          const float* __restrict__ A,
                                                          float g_min, float* __restrict__ g,
                                                          float* __restrict__ gcum,
                                                          int64_t n_tokens, int H,
                                                          const int32_t* __restrict__ cu,
                                                          int n_seqs) {
  const int c = threadIdx.x;
  const int h = blockIdx.y;
  const int64_t t0 = (int64_t)blockIdx.x * kChunk;
  const int64_t t1 = min(t0 + kChunk, n_tokens);
  const float scale = expf(__ldg(A + h));
  auto seq_start = [&](int n) -> int64_t {
    if (!cu) return 0;
    int64_t x = cu[n];
    return x < 0 ? 0 : (x > n_tokens ? n_tokens : x);
  };
  auto seq_end = [&](int n) -> int64_t { return cu ? seq_start(n + 1) : n_tokens; };
  // sequence containing t0: the last n with start(n) <= t0
  int n = 0;
  if (cu) {
    int lo = 0, hi = n_seqs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (seq_start(mid) <= t0) lo = mid; else hi = mid - 1;
    }
    n = lo;
  }
  int64_t cs = seq_start(n);
  cs += ((t0 - cs) / kChunk) * kChunk;  // start of the chunk holding t0
  float acc = 0.f;
  for (int64_t t = cs; t < t0; ++t)
    acc += bounded_decay(to_f32(z[(t * H + h) * kD + c]), scale, g_min);
  for (int64_t t = t0; t < t1; ++t) {
    while (n + 1 < n_seqs && seq_end(n) <= t) {
      ++n;
      if (seq_start(n) == t) acc = 0.f;  // a new sequence starts a new chunk
    }
    if (((t - seq_start(n)) % kChunk) == 0) acc = 0.f;
    const int64_t i = (t * H + h) * kD + c;
    const float gv = bounded_decay(to_f32(z[i]), scale, g_min);
    acc += gv;
    g[i] = gv;
    gcum[i] = acc;
  }
}

int grid_for(int64_t work, int threads) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t need = (work + threads - 1) / threads;
  const int64_t cap = (int64_t)sms * 8;
  return (int)(need < cap ? (need < 1 ? 1 : need) : cap);
}

}  // namespace

cudaError_t launch_gate(const void* z, int z_bf16, const float* A, float g_min, float* g,
                        int64_t n_tokens, int H, cudaStream_t s) {
  const int64_t n_groups = n_tokens * H * (kD / 8);
  const int grid = grid_for(n_groups, 256);
  ProfScope prof_scope("kda_gate", s);
  if (z_bf16)
    gate_kernel<<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(z), A, g_min, g, n_groups, H);
  else
    gate_kernel<<<grid, 256, 0, s>>>(static_cast<const float*>(z), A, g_min, g, n_groups, H);
  return cudaGetLastError();
}

namespace {

// Output gate, a half warp per (token, head): lane l of the half holds channels
// 8l .. 8l + 7 of o and of the gate logits (16-byte accesses for bf16); the sum of
// squares meets by a half-warp all-reduce, and each warp keeps four token-heads
// in flight.
//   y = Sigmoid(x) * w * o / sqrt(mean(o^2) + eps)
// ("Kimi K3 technical report review", section 3.3, Eq. 6, without W_o and W_g)
template <typename T>
__global__ void __launch_bounds__(256) out_gate_kernel(const T* __restrict__ o,
                                                       const T* __restrict__ x,
                                                       const float* __restrict__ w, float eps,
                                                       T* y, int64_t n_rows) {
  const int hl = threadIdx.x & 15, half = (threadIdx.x >> 4) & 1;
  const int64_t warp_g = blockIdx.x * (int64_t)(blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  float wv[8] = {1.f, 1.f, 1.f, 1.f, 1.f, 1.f, 1.f, 1.f};
  if (w) load8(w + 8 * hl, wv);
  // warp g takes rows 2g + half + 2 nwarps (2i + k): every row once; the loop and
  // the shuffles are uniform over the warp, validity only gates loads and stores
  for (int64_t base = 2 * warp_g; base < n_rows; base += 4 * nwarps) {
    float ov[2][8], xv[2][8];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int64_t row = base + k * 2 * nwarps + half;
      if (row < n_rows) {
        load8(o + row * kD + 8 * hl, ov[k]);
        load8(x + row * kD + 8 * hl, xv[k]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) ov[k][i] = xv[k][i] = 0.f;
      }
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      float ss = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) ss = fmaf(ov[k][i], ov[k][i], ss);
#pragma unroll
      for (int m = 8; m >= 1; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
      const float r = rsqrtf(ss * (1.f / kD) + eps);
      const int64_t row = base + k * 2 * nwarps + half;
      if (row < n_rows) {
        float yv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          yv[i] = __fdividef(ov[k][i] * r * wv[i], 1.f + __expf(-xv[k][i]));
        store8(y + row * kD + 8 * hl, yv);
      }
    }
  }
}

}  // namespace

namespace {

// Scalar gate (one log-decay per token and head, as Gated DeltaNet's gate) spread
// over the kD channels for the fp32 chunk path: thread = 4 channels of one
// (token, head), 16-byte stores.
__global__ void __launch_bounds__(256) expand_scalar_gate_kernel(const float* __restrict__ gs,
                                                                 float* __restrict__ g,
                                                                 int64_t n_quads) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n_quads;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float x = __ldg(gs + i / (kD / 4));  // kD / 4 quads per (token, head)
    reinterpret_cast<float4*>(g)[i] = make_float4(x, x, x, x);
  }
}

}  // namespace

cudaError_t launch_expand_scalar_gate(const float* gs, float* g, int64_t n_tokens, int H,
                                      cudaStream_t s) {
  const int64_t n_quads = n_tokens * H * (kD / 4);
  if (n_quads == 0) return cudaSuccess;
  ProfScope prof_scope("kda_expand_scalar_gate", s);
  expand_scalar_gate_kernel<<<grid_for(n_quads, 256), 256, 0, s>>>(gs, g, n_quads);
  return cudaGetLastError();
}

cudaError_t launch_output_gate(const void* o, int bf16, const void* x, const float* w, float eps,
                               void* y, int64_t n_tokens, int H, cudaStream_t s) {
  const int64_t rows = n_tokens * H;
  if (rows == 0) return cudaSuccess;
  const int grid = grid_for(rows * 8, 256);
  ProfScope prof_scope("kda_output_gate", s);
  if (bf16)
    out_gate_kernel<<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(o),
                                         static_cast<const __nv_bfloat16*>(x), w, eps,
                                         static_cast<__nv_bfloat16*>(y), rows);
  else
    out_gate_kernel<<<grid, 256, 0, s>>>(static_cast<const float*>(o),
                                         static_cast<const float*>(x), w, eps,
                                         static_cast<float*>(y), rows);
  return cudaGetLastError();
}

cudaError_t launch_gate_softplus(const void* z, int z_bf16, const float* A, float* g,
                                 int64_t n_tokens, int H, cudaStream_t s) {
  const int64_t n_groups = n_tokens * H * (kD / 8);
  const int grid = grid_for(n_groups, 256);
  ProfScope prof_scope("kda_gate_softplus", s);
  if (z_bf16)
    gate_kernel<__nv_bfloat16, true><<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(z), A,
                                                          0.f, g, n_groups, H);
  else
    gate_kernel<float, true><<<grid, 256, 0, s>>>(static_cast<const float*>(z), A, 0.f, g,
                                                  n_groups, H);
  return cudaGetLastError();
}

cudaError_t launch_gate_cumsum(const void* z, int z_bf16, const float* A, float g_min, float* g,
                               float* gcum, int64_t n_tokens, int H, const int32_t* cu,
                               int n_seqs, cudaStream_t s) {
  const dim3 grid((unsigned)((n_tokens + kChunk - 1) / kChunk), (unsigned)H);
  ProfScope prof_scope("kda_gate_cumsum", s);
  if (z_bf16)
    gate_cumsum_kernel<<<grid, kD, 0, s>>>(static_cast<const __nv_bfloat16*>(z), A, g_min, g, gcum,
                                           n_tokens, H, cu, n_seqs);
  else
    gate_cumsum_kernel<<<grid, kD, 0, s>>>(static_cast<const float*>(z), A, g_min, g, gcum,
                                           n_tokens, H, cu, n_seqs);
  return cudaGetLastError();
}

}  // namespace kda
