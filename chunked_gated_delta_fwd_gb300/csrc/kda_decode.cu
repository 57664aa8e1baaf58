// kda_decode.cu -- K5: one decode token of KDA for N x H independent states,
// updated in place, in the delta form
//     S <- D S + beta k (v^T - k^T D S),   D = Diag(exp(g)),   o = S^T q
// ("Kimi K3: architecture, training and inference systems" (weigao.cc),
//  section 3.1 for the form, sections 11.2 / 13.2 for the in-place decode step).
//
// The state is stored transposed, S^T [dv][dk] fp32, so row j (one value column
// of S) is 128 contiguous floats = 512 bytes.  Per row j:
//     s_bar = alpha (.) s_j,   p = k . s_bar,   r = q . s_bar
//     s_j  <- s_bar + beta (v_j - p) k
//     o_j   = q . s_j = r + beta (v_j - p) (q . k)
// One CTA per (sequence, head), four warps, each warp streams 32 rows; lane l
// holds channels 4l..4l+3, so a row is one coalesced 128-bit load and one
// 128-bit store per lane.  The per-row dot products p and r of a warp's 8 rows
// in flight are reduce-scattered across the lanes (each halving step swaps half
// of the partial sums with a partner lane, 9 shuffles for 8 rows); p is then
// gathered back to every lane, r stays with the lane that writes o_j.  The
// kernel is HBM-bound: 2 x 64 KiB of state per head and step.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kDecodeThreads = 128;
constexpr int kRowsPerIter = 8;  // rows in flight per warp

template <typename T>
__global__ void __launch_bounds__(kDecodeThreads) decode_kernel(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
    const float* __restrict__ g, const T* __restrict__ beta, float* __restrict__ S,
    T* __restrict__ o) {
  const int unit = blockIdx.x;  // n * H + h
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int64_t vec = (int64_t)unit * kD;

  float qv[4], kv[4], alpha[4];
  load4(q + vec + 4 * lane, qv);
  load4(k + vec + 4 * lane, kv);
  {
    const float4 gg = *reinterpret_cast<const float4*>(g + vec + 4 * lane);
    alpha[0] = expf(gg.x);
    alpha[1] = expf(gg.y);
    alpha[2] = expf(gg.z);
    alpha[3] = expf(gg.w);
  }
  const float b = to_f32(beta[unit]);
  float qk = qv[0] * kv[0] + qv[1] * kv[1] + qv[2] * kv[2] + qv[3] * kv[3];
#pragma unroll
  for (int o_ = 16; o_ > 0; o_ >>= 1) qk += __shfl_xor_sync(0xffffffffu, qk, o_);
  const int row0 = warp * 32;
  const float v_mine = to_f32(v[vec + row0 + lane]);
  float o_mine = 0.f;

  float4* Srow = reinterpret_cast<float4*>(S + (int64_t)unit * kD * kD) + row0 * (kD / 4) + lane;

#pragma unroll 1
  for (int r0 = 0; r0 < 32; r0 += kRowsPerIter) {
    float4 s[kRowsPerIter];
#pragma unroll
    for (int i = 0; i < kRowsPerIter; ++i) s[i] = __ldcs(Srow + (r0 + i) * (kD / 4));
    float p[kRowsPerIter], r[kRowsPerIter];
#pragma unroll
    for (int i = 0; i < kRowsPerIter; ++i) {
      s[i].x *= alpha[0];
      s[i].y *= alpha[1];
      s[i].z *= alpha[2];
      s[i].w *= alpha[3];
      p[i] = kv[0] * s[i].x + kv[1] * s[i].y + kv[2] * s[i].z + kv[3] * s[i].w;
      r[i] = qv[0] * s[i].x + qv[1] * s[i].y + qv[2] * s[i].z + qv[3] * s[i].w;
    }
    // reduce-scatter of the 8 rows' k.s and q.s (see decode_multi_kernel): lane l
    // ends with row R(l) = 4 b4 + 2 b3 + b2; k.s is gathered back to every lane
    {
      const bool u4 = (lane & 16) != 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        p[i] = (u4 ? p[4 + i] : p[i]) + __shfl_xor_sync(0xffffffffu, u4 ? p[i] : p[4 + i], 16);
        r[i] = (u4 ? r[4 + i] : r[i]) + __shfl_xor_sync(0xffffffffu, u4 ? r[i] : r[4 + i], 16);
      }
      const bool u3 = (lane & 8) != 0;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        p[i] = (u3 ? p[2 + i] : p[i]) + __shfl_xor_sync(0xffffffffu, u3 ? p[i] : p[2 + i], 8);
        r[i] = (u3 ? r[2 + i] : r[i]) + __shfl_xor_sync(0xffffffffu, u3 ? r[i] : r[2 + i], 8);
      }
      const bool u2 = (lane & 4) != 0;
      p[0] = (u2 ? p[1] : p[0]) + __shfl_xor_sync(0xffffffffu, u2 ? p[0] : p[1], 4);
      r[0] = (u2 ? r[1] : r[0]) + __shfl_xor_sync(0xffffffffu, u2 ? r[0] : r[1], 4);
      p[0] += __shfl_xor_sync(0xffffffffu, p[0], 2);
      r[0] += __shfl_xor_sync(0xffffffffu, r[0], 2);
      p[0] += __shfl_xor_sync(0xffffffffu, p[0], 1);
      r[0] += __shfl_xor_sync(0xffffffffu, r[0], 1);
    }
    const int Rl = 4 * ((lane >> 4) & 1) + 2 * ((lane >> 3) & 1) + ((lane >> 2) & 1);
    const float pR = p[0], rR = r[0];
#pragma unroll
    for (int i = 0; i < kRowsPerIter; ++i) {
      const float pi = __shfl_sync(0xffffffffu, pR, 16 * (i >> 2) + 8 * ((i >> 1) & 1) + 4 * (i & 1));
      const float vj = __shfl_sync(0xffffffffu, v_mine, r0 + i);
      const float u = b * (vj - pi);
      s[i].x = fmaf(u, kv[0], s[i].x);
      s[i].y = fmaf(u, kv[1], s[i].y);
      s[i].z = fmaf(u, kv[2], s[i].z);
      s[i].w = fmaf(u, kv[3], s[i].w);
      __stcs(Srow + (r0 + i) * (kD / 4), s[i]);
    }
    // o of row r0 + R(l) = (u q.k + q.s) on the lanes that hold it
    const float vR = __shfl_sync(0xffffffffu, v_mine, r0 + Rl);
    const float oR = fmaf(b * (vR - pR), qk, rR);
    const float oj = __shfl_sync(0xffffffffu, oR,
                                 16 * (((lane - r0) & 7) >> 2) + 8 * ((((lane - r0) & 7) >> 1) & 1) +
                                     4 * ((lane - r0) & 1));
    if (lane >= r0 && lane < r0 + kRowsPerIter) o_mine = oj;
  }
  o[vec + row0 + lane] = from_f32<T>(o_mine);
}

// ---------------------------------------------------------------- several tokens
// T tokens per (sequence, head) in one pass over the state: rows of S^T are
// independent across tokens (row j only needs token t's k, q, alpha, beta and
// v_j), so a warp keeps 8 rows in registers while it walks all T tokens, whose
// vectors sit in shared memory.  The outputs of all T tokens are written; the
// state written back is the state after the first n_adv tokens (n_adv = T when
// no counts are given, 0 leaves the state as it was): a speculative-decode
// verify pass (outputs for every draft token) and the commit of the accepted
// prefix ("Kimi K3: architecture, training and inference systems", section
// 13.2, speculative replay) in one kernel.
constexpr int kMultiMaxT = 16;

template <typename T>
__global__ void __launch_bounds__(kDecodeThreads) decode_multi_kernel(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
    const float* __restrict__ g, const T* __restrict__ beta, float* __restrict__ S,
    T* __restrict__ o, const int32_t* __restrict__ n_advance, int H, int Tn) {
  // per token: q, k, alpha (4 x 128 floats with v), beta and q.k
  __shared__ __align__(16) float tq[kMultiMaxT][kD], tk[kMultiMaxT][kD], ta[kMultiMaxT][kD],
      tv[kMultiMaxT][kD];
  __shared__ float tb[kMultiMaxT], tqk[kMultiMaxT];
  const int unit = blockIdx.x;  // n * H + h
  const int n = unit / H, h = unit - n * H;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, tid = threadIdx.x;
  int adv = n_advance ? n_advance[n] : Tn;
  adv = adv < 0 ? 0 : (adv > Tn ? Tn : adv);
  for (int t = warp; t < Tn; t += kDecodeThreads / 32) {
    const int64_t vec = (((int64_t)n * Tn + t) * H + h) * kD;
    float qv[4], kv[4], vv[4];
    load4(q + vec + 4 * lane, qv);
    load4(k + vec + 4 * lane, kv);
    load4(v + vec + 4 * lane, vv);
    const float4 gg = *reinterpret_cast<const float4*>(g + vec + 4 * lane);
    *reinterpret_cast<float4*>(&tq[t][4 * lane]) = make_float4(qv[0], qv[1], qv[2], qv[3]);
    *reinterpret_cast<float4*>(&tk[t][4 * lane]) = make_float4(kv[0], kv[1], kv[2], kv[3]);
    *reinterpret_cast<float4*>(&tv[t][4 * lane]) = make_float4(vv[0], vv[1], vv[2], vv[3]);
    *reinterpret_cast<float4*>(&ta[t][4 * lane]) =
        make_float4(expf(gg.x), expf(gg.y), expf(gg.z), expf(gg.w));
    float qk = qv[0] * kv[0] + qv[1] * kv[1] + qv[2] * kv[2] + qv[3] * kv[3];
#pragma unroll
    for (int o_ = 16; o_ > 0; o_ >>= 1) qk += __shfl_xor_sync(0xffffffffu, qk, o_);
    if (lane == 0) {
      tqk[t] = qk;
      tb[t] = to_f32(beta[((int64_t)n * Tn + t) * H + h]);
    }
  }
  __syncthreads();
  (void)tid;
  const int row0 = warp * 32;
  float4* Srow = reinterpret_cast<float4*>(S + (int64_t)unit * kD * kD) + row0 * (kD / 4) + lane;
  // The next block of rows is loaded while the T tokens walk the current one, so
  // that the state stream stays in flight during the token loop.
  float4 s[kRowsPerIter], sn[kRowsPerIter];
#pragma unroll
  for (int i = 0; i < kRowsPerIter; ++i) s[i] = __ldcs(Srow + i * (kD / 4));
#pragma unroll 1
  for (int r0 = 0; r0 < 32; r0 += kRowsPerIter) {
    if (r0 + kRowsPerIter < 32) {
#pragma unroll
      for (int i = 0; i < kRowsPerIter; ++i) sn[i] = __ldcs(Srow + (r0 + kRowsPerIter + i) * (kD / 4));
    }
#pragma unroll 1
    for (int t = 0; t < Tn; ++t) {
      const float4 al = *reinterpret_cast<const float4*>(&ta[t][4 * lane]);
      const float4 kk = *reinterpret_cast<const float4*>(&tk[t][4 * lane]);
      const float4 qq = *reinterpret_cast<const float4*>(&tq[t][4 * lane]);
      float p[kRowsPerIter], r[kRowsPerIter];
#pragma unroll
      for (int i = 0; i < kRowsPerIter; ++i) {
        s[i].x *= al.x;
        s[i].y *= al.y;
        s[i].z *= al.z;
        s[i].w *= al.w;
        p[i] = kk.x * s[i].x + kk.y * s[i].y + kk.z * s[i].z + kk.w * s[i].w;
        r[i] = qq.x * s[i].x + qq.y * s[i].y + qq.z * s[i].z + qq.w * s[i].w;
      }
      // Halving reduce-scatter of the 8 rows' partial sums over the warp (9 shuffles
      // each instead of 40): lane l ends with the full k.s and q.s of row
      // R(l) = 4 b4 + 2 b3 + b2 (b = bits of l).  Every lane then gathers all 8 k.s
      // (the erase needs them); q.s stays with the lanes that store o.
      {
        const bool u4 = (lane & 16) != 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          p[i] = (u4 ? p[4 + i] : p[i]) + __shfl_xor_sync(0xffffffffu, u4 ? p[i] : p[4 + i], 16);
          r[i] = (u4 ? r[4 + i] : r[i]) + __shfl_xor_sync(0xffffffffu, u4 ? r[i] : r[4 + i], 16);
        }
        const bool u3 = (lane & 8) != 0;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          p[i] = (u3 ? p[2 + i] : p[i]) + __shfl_xor_sync(0xffffffffu, u3 ? p[i] : p[2 + i], 8);
          r[i] = (u3 ? r[2 + i] : r[i]) + __shfl_xor_sync(0xffffffffu, u3 ? r[i] : r[2 + i], 8);
        }
        const bool u2 = (lane & 4) != 0;
        p[0] = (u2 ? p[1] : p[0]) + __shfl_xor_sync(0xffffffffu, u2 ? p[0] : p[1], 4);
        r[0] = (u2 ? r[1] : r[0]) + __shfl_xor_sync(0xffffffffu, u2 ? r[0] : r[1], 4);
        p[0] += __shfl_xor_sync(0xffffffffu, p[0], 2);
        r[0] += __shfl_xor_sync(0xffffffffu, r[0], 2);
        p[0] += __shfl_xor_sync(0xffffffffu, p[0], 1);
        r[0] += __shfl_xor_sync(0xffffffffu, r[0], 1);
      }
      const int Rl = 4 * ((lane >> 4) & 1) + 2 * ((lane >> 3) & 1) + ((lane >> 2) & 1);
      const float pR = p[0], rR = r[0];  // row Rl of this block
      float pa[kRowsPerIter];
#pragma unroll
      for (int i = 0; i < kRowsPerIter; ++i)  // row i sits on lane 16 (i>>2) + 8 ((i>>1)&1) + 4 (i&1)
        pa[i] = __shfl_sync(0xffffffffu, pR, 16 * (i >> 2) + 8 * ((i >> 1) & 1) + 4 * (i & 1));
      const float b = tb[t], qk = tqk[t];
#pragma unroll
      for (int i = 0; i < kRowsPerIter; ++i) {
        const float u = b * (tv[t][row0 + r0 + i] - pa[i]);
        s[i].x = fmaf(u, kk.x, s[i].x);
        s[i].y = fmaf(u, kk.y, s[i].y);
        s[i].z = fmaf(u, kk.z, s[i].z);
        s[i].w = fmaf(u, kk.w, s[i].w);
      }
      if (o && (lane & 3) == 0) {
        const float uR = b * (tv[t][row0 + r0 + Rl] - pR);
        o[(((int64_t)n * Tn + t) * H + h) * kD + row0 + r0 + Rl] = from_f32<T>(fmaf(uR, qk, rR));
      }
      if (t + 1 == adv) {
#pragma unroll
        for (int i = 0; i < kRowsPerIter; ++i) __stcs(Srow + (r0 + i) * (kD / 4), s[i]);
      }
    }
#pragma unroll
    for (int i = 0; i < kRowsPerIter; ++i) s[i] = sn[i];
  }
}

}  // namespace

cudaError_t launch_decode_multi(const void* q, const void* k, const void* v, int bf16,
                                const float* g, const void* beta, float* S, void* o,
                                const int32_t* n_advance, int N, int T, int H, cudaStream_t s) {
  const unsigned grid = (unsigned)((int64_t)N * H);
  ProfScope prof_scope("kda_decode_multi", s);
  if (bf16) {
    using E = __nv_bfloat16;
    decode_multi_kernel<E><<<grid, kDecodeThreads, 0, s>>>(
        static_cast<const E*>(q), static_cast<const E*>(k), static_cast<const E*>(v), g,
        static_cast<const E*>(beta), S, static_cast<E*>(o), n_advance, H, T);
  } else {
    decode_multi_kernel<float><<<grid, kDecodeThreads, 0, s>>>(
        static_cast<const float*>(q), static_cast<const float*>(k), static_cast<const float*>(v),
        g, static_cast<const float*>(beta), S, static_cast<float*>(o), n_advance, H, T);
  }
  return cudaGetLastError();
}

cudaError_t launch_decode(const void* q, const void* k, const void* v, int bf16, const float* g,
                          const void* beta, float* S, void* o, int N, int H, cudaStream_t s) {
  const unsigned grid = (unsigned)((int64_t)N * H);
  ProfScope prof_scope("kda_decode", s);
  if (bf16) {
    using T = __nv_bfloat16;
    decode_kernel<T><<<grid, kDecodeThreads, 0, s>>>(
        static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v), g,
        static_cast<const T*>(beta), S, static_cast<T*>(o));
  } else {
    decode_kernel<float><<<grid, kDecodeThreads, 0, s>>>(
        static_cast<const float*>(q), static_cast<const float*>(k), static_cast<const float*>(v),
        g, static_cast<const float*>(beta), S, static_cast<float*>(o));
  }
  return cudaGetLastError();
}

}  // namespace kda
