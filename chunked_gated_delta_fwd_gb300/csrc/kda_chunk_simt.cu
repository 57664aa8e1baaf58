// kda_chunk_simt.cu -- the chunkwise KDA forward on fp32 CUDA cores.
//
// This is the path for fp32 inputs (where bf16 tensor-core operands could not
// meet fp32 accuracy) and an fp32 cross-check of the tensor-core path for bf16
// inputs.  It evaluates the WY/UT chunkwise form ("Kimi K3 notes" (s1mplewind
// blog), section "Chunkwise form") for 64-token chunks:
//
//   G   = running sum of g inside the chunk (per channel), Gamma = exp(G)
//   A   = StrictTril(Diag(beta) (Gamma*K) (K/Gamma)^T),  T = (I + A)^{-1}
//   W   = T Diag(beta) (Gamma*K),   U = T Diag(beta) V
//   Vt  = U - W S,   O = (Gamma*Q) S + Tril((Gamma*Q)(K/Gamma)^T) Vt
//   S  <- Diag(gamma_C) S + ((gamma_C/Gamma)*K)^T Vt
//
// K/Gamma overflows over a whole chunk (the cumulative log-decay reaches -320),
// so the two 64x64 products are formed block by block over 16-token tiles with
// a reference per tile, the scheme the bounded decay makes safe ("Kimi K3
// technical report review" (devpress/CSDN), section 3.2): with R_a the log-decay
// at the end of the tile before tile a, for row r in tile a and column i in tile
// b <= a,
//   exp(G_r - G_i) = exp(G_r - R_a) * exp(R_a - R_b) * exp(R_b - G_i)
// where the first two factors are <= 1 and the last is < e^80 (16 tokens with
// g >= -5).
//
// Range-robust mode (any g <= 0, e.g. the unbounded softplus gate of Kimi Linear,
// "Kimi K3 technical report review", section 3.2): tiles below the diagonal take
// the reference at the END of the key tile,
//   exp(G_r - G_i) = exp(L_r) * exp(sum of the tile totals between) * exp(M_i),
// with L_r the sum of g over tile a up to r and M_i the sum over tile b after i:
// every factor <= 1.  The diagonal tiles are formed pair by pair,
// sum_c k_rc k_ic exp(g_{i+1,c} + ... + g_{r,c}) -- the position-pair path the
// bound removes.  Every exponent is a sum of non-positive terms, never the
// difference of two running sums, so decays stay exact to fp32 rounding even
// where a single g is -10^4.
//
// Two kernels: `simt_prep` (one CTA per (chunk, head), fully parallel) writes
// W, U, Gamma*Q, (gamma_C/Gamma)*K, the masked 64x64 A_qk and gamma_C to the
// workspace; `simt_chain` (one CTA per (sequence, head, 32-column slice of S))
// walks the chunks of a sequence in order, keeping its slice of S in shared
// memory.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int C = kChunk;        // 64
constexpr int D = kD;            // 128
constexpr int LD = D + 4;        // padded row stride (floats) of 64x128 smem tiles
constexpr int LC = C + 1;        // padded row stride of 64x64 smem tiles
constexpr int kPrepThreads = 256;

// Per (chunk, head) unit of the fp32 workspace.
constexpr int64_t kOffW = 0;
constexpr int64_t kOffU = kOffW + C * D;
constexpr int64_t kOffQg = kOffU + C * D;
constexpr int64_t kOffKt = kOffQg + C * D;
constexpr int64_t kOffAqk = kOffKt + C * D;
constexpr int64_t kOffGam = kOffAqk + C * C;
constexpr int64_t kUnitFloats = kOffGam + D;

struct PrepSmem {
  float Kb[C][LD];  // k -> k*exp(G - R_a) -> beta*Gamma*K
  float Qb[C][LD];  // q -> q*exp(G - R_a) -> Gamma*Q
  float KN[C][LD];  // k*exp(R_b - G) -> (gamma_C/Gamma)*K
  float Vs[C][LD];  // v -> beta*v
  union {
    float G[C][LD];  // g -> running sum G
    struct {
      float L[C][LC];  // A_kk (strict lower, beta applied), then T = (I + A_kk)^{-1}
      float Aq[C][LC];  // A_qk (lower incl. diagonal)
    } m;
  } u;
  float R[4][D];       // tile references R_0 = 0, R_a = G[16a - 1]
  float E[4][4][D];    // exp(R_a - R_b) for a > b
  float X[C][LD];      // range-robust mode: the raw g
  float Tt[4][D];      // range-robust mode: sum of g over tile a
  float GC[D];         // G at the chunk's last token
  float beta[C];
};

__device__ __forceinline__ int find_seq(const int32_t* chunk_off, int n_seqs, int chunk) {
  // last n with chunk_off[n] <= chunk
  int lo = 0, hi = n_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(chunk_off + mid) <= chunk) lo = mid; else hi = mid - 1;
  }
  return lo;
}

template <typename T>
__global__ void __launch_bounds__(kPrepThreads, 1) simt_prep(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
    const float* __restrict__ g, const T* __restrict__ beta, Plan plan, int H,
    float* __restrict__ out, int robust) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  PrepSmem& sm = *reinterpret_cast<PrepSmem*>(smem_raw);
  const int chunk = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  const int total = __ldg(plan.chunk_off + plan.n_seqs);
  if (chunk >= total) return;
  const int n = find_seq(plan.chunk_off, plan.n_seqs, chunk);
  const int j = chunk - __ldg(plan.chunk_off + n);
  const int64_t t0 = (int64_t)__ldg(plan.cu + n) + (int64_t)j * C;
  const int len = (int)min((int64_t)C, (int64_t)__ldg(plan.cu + n + 1) - t0);

  // ---- 1. load the chunk (rows >= len are zero; g = 0 keeps G flat there)
  for (int e = tid; e < C * (D / 4); e += kPrepThreads) {
    const int r = e / (D / 4), c4 = (e % (D / 4)) * 4;
    float kk[4] = {0, 0, 0, 0}, qq[4] = {0, 0, 0, 0}, vv[4] = {0, 0, 0, 0}, gg[4] = {0, 0, 0, 0};
    if (r < len) {
      const int64_t off = ((t0 + r) * H + h) * D + c4;
      load4(k + off, kk);
      load4(q + off, qq);
      load4(v + off, vv);
      load4(g + off, gg);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      sm.Kb[r][c4 + i] = kk[i];
      sm.Qb[r][c4 + i] = qq[i];
      sm.Vs[r][c4 + i] = vv[i];
      sm.u.G[r][c4 + i] = gg[i];
    }
  }
  if (tid < C) sm.beta[tid] = tid < len ? to_f32(beta[(t0 + tid) * H + h]) : 0.f;
  __syncthreads();

  // ---- 2. running sum of g per channel, tile references
  if (tid < D && !robust) {
    const int c = tid;
    float acc = 0.f;
    sm.R[0][c] = 0.f;
    for (int r = 0; r < C; ++r) {
      acc += sm.u.G[r][c];
      sm.u.G[r][c] = acc;
      if ((r & (kTile - 1)) == kTile - 1 && r + 1 < C) sm.R[(r + 1) / kTile][c] = acc;
    }
    sm.GC[c] = acc;
  } else if (tid < D) {
    // range-robust: raw g kept in X; G <- L (sum over the tile up to r), KN <- M (sum
    // over the tile after r), tile totals, R_a = totals before tile a
    const int c = tid;
    float pre = 0.f;
    for (int a = 0; a < 4; ++a) {
      sm.R[a][c] = pre;
      float l = 0.f;
      for (int e = 0; e < kTile; ++e) {
        const int r = a * kTile + e;
        const float gv = sm.u.G[r][c];
        sm.X[r][c] = gv;
        l += gv;
        sm.u.G[r][c] = l;
      }
      float m = 0.f;
      for (int e = kTile - 1; e >= 0; --e) {
        const int r = a * kTile + e;
        sm.KN[r][c] = m;
        m += sm.X[r][c];
      }
      sm.Tt[a][c] = l;
      pre += l;
    }
    sm.GC[c] = pre;
  }
  __syncthreads();

  // ---- 2b. range-robust mode: the diagonal tiles pair by pair from the raw rows
  //          (thread -> row ri, key ii of every diagonal tile)
  float dk_[4] = {0.f, 0.f, 0.f, 0.f}, dq_[4] = {0.f, 0.f, 0.f, 0.f};
  if (robust) {
    const int ri = tid / 16, ii = tid % 16;
    if (ii <= ri) {
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const int r = a * kTile + ri, i = a * kTile + ii;
        float ak = 0.f, aq = 0.f;
#pragma unroll 4
        for (int c = 0; c < D; ++c) {
          float sg = 0.f;  // g over tokens i+1 .. r of this channel
          for (int jj = i + 1; jj <= r; ++jj) sg += sm.X[jj][c];
          const float t = sm.Kb[i][c] * expf(sg);
          ak = fmaf(sm.Kb[r][c], t, ak);
          aq = fmaf(sm.Qb[r][c], t, aq);
        }
        dk_[a] = ak;
        dq_[a] = aq;
      }
    }
  }
  if (robust) __syncthreads();  // the raw rows are read before step 3 rescales them
  // sum of the tile totals over tiles lo..hi (range-robust mode)
  auto tiles_sum = [&](int lo, int hi, int c) {
    float s = 0.f;
    for (int t2 = lo; t2 <= hi; ++t2) s += sm.Tt[t2][c];
    return s;
  };

  // ---- 3. tile-referenced factors
  for (int e = tid; e < C * D; e += kPrepThreads) {
    const int r = e / D, c = e % D, a = r / kTile;
    // G_r - R_a: in (-80, 0] (bounded), L_r (robust)
    const float d = robust ? sm.u.G[r][c] : sm.u.G[r][c] - sm.R[a][c];
    const float f = expf(d);
    const float kk = sm.Kb[r][c];
    sm.Kb[r][c] = kk * f;
    sm.Qb[r][c] *= f;
    sm.KN[r][c] = kk * expf(robust ? sm.KN[r][c] : -d);  // < e^80 (bounded), <= 1 (robust)
  }
  for (int e = tid; e < 16 * D; e += kPrepThreads) {
    const int ab = e / D, c = e % D, a = ab / 4, b = ab % 4;
    sm.E[a][b][c] = a <= b ? 1.f
                           : expf(robust ? tiles_sum(b + 1, a - 1, c) : sm.R[a][c] - sm.R[b][c]);
  }
  __syncthreads();

  // ---- 4. the 64x64 products block by block: A_kk (strict, beta) and A_qk (incl. diag)
  {
    const int ri = tid / 16, ii = tid % 16;
    for (int a = 0; a < 4; ++a) {
      for (int b = 0; b < 4; ++b) {
        const int r = a * kTile + ri, i = b * kTile + ii;
        float ak = 0.f, aq = 0.f;
        if (robust && b == a) {
          ak = dk_[a];
          aq = dq_[a];
        } else if (b <= a) {
#pragma unroll 8
          for (int c = 0; c < D; ++c) {
            const float t = sm.E[a][b][c] * sm.KN[i][c];
            ak = fmaf(sm.Kb[r][c], t, ak);
            aq = fmaf(sm.Qb[r][c], t, aq);
          }
        }
        sm.u.m.L[r][i] = (i < r) ? sm.beta[r] * ak : 0.f;
        sm.u.m.Aq[r][i] = (i <= r) ? aq : 0.f;
      }
    }
  }
  __syncthreads();

  // ---- 5. T = (I + A_kk)^{-1} by forward substitution, one column per thread
  //         (threads 0..63); the other threads finish the scaled operands.
  if (tid < C) {
    const int jc = tid;
    float x[C];
#pragma unroll
    for (int r = 0; r < C; ++r) {
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < r; ++i) acc = fmaf(sm.u.m.L[r][i], x[i], acc);
      x[r] = (r < jc) ? 0.f : (r == jc ? 1.f : -acc);
    }
    asm volatile("bar.sync 1, 64;" ::: "memory");  // all columns read L before T overwrites it
#pragma unroll
    for (int r = 0; r < C; ++r) sm.u.m.L[r][jc] = x[r];
  } else {
    for (int e = tid - C; e < C * D; e += kPrepThreads - C) {
      const int r = e / D, c = e % D, a = r / kTile;
      const float ea = expf(sm.R[a][c]);                     // exp(R_a), <= 1
      // exp(G_C - reference of the key tile), <= 1
      const float ec = expf(robust ? tiles_sum(a + 1, 3, c) : sm.GC[c] - sm.R[a][c]);
      sm.Kb[r][c] *= ea * sm.beta[r];                        // beta * Gamma * K
      sm.Qb[r][c] *= ea;                                     // Gamma * Q
      sm.KN[r][c] *= ec;                                     // (gamma_C / Gamma) * K
      sm.Vs[r][c] *= sm.beta[r];                             // beta * V
    }
  }
  __syncthreads();

  // ---- 6. W = T (beta Gamma K), U = T (beta V); write the unit
  float* unit = out + ((int64_t)chunk * H + h) * kUnitFloats;
  {
    const int c = tid % D, par = tid / D;  // rows of parity par
    for (int r = par; r < C; r += 2) {
      float w = 0.f, uu = 0.f;
      for (int i = 0; i <= r; ++i) {
        const float t = sm.u.m.L[r][i];
        w = fmaf(t, sm.Kb[i][c], w);
        uu = fmaf(t, sm.Vs[i][c], uu);
      }
      unit[kOffW + r * D + c] = w;
      unit[kOffU + r * D + c] = uu;
      unit[kOffQg + r * D + c] = sm.Qb[r][c];
      unit[kOffKt + r * D + c] = sm.KN[r][c];
    }
  }
  for (int e = tid; e < C * C; e += kPrepThreads) unit[kOffAqk + e] = sm.u.m.Aq[e / C][e % C];
  if (tid < D) unit[kOffGam + tid] = expf(sm.GC[tid]);
}

// ---------------------------------------------------------------------- chain
constexpr int kSlice = 32;  // columns of S (values) per CTA
constexpr int kChainThreads = 256;

struct ChainSmem {
  float S[D][kSlice];     // slice of the state, S[c][j] (dk x slice)
  float W[C][LD];
  float Qg[C][LD];
  float Kt[C][LD];
  float Aq[C][LC];
  float U[C][kSlice + 1];
  float Vt[C][kSlice + 1];
  float gam[D];
};

template <typename T>
__global__ void __launch_bounds__(kChainThreads, 1) simt_chain(
    const float* __restrict__ ws, const float* __restrict__ h0, Plan plan, int H,
    T* __restrict__ o, float* __restrict__ hT) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  ChainSmem& sm = *reinterpret_cast<ChainSmem*>(smem_raw);
  const int n = blockIdx.x, h = blockIdx.y, j0 = blockIdx.z * kSlice, tid = threadIdx.x;
  const int64_t state = ((int64_t)n * H + h) * D * D;  // [dv][dk]
  // S[c][j] = stored[j0 + j][c]
  for (int e = tid; e < D * kSlice; e += kChainThreads) {
    const int jj = e / D, c = e % D;
    sm.S[c][jj] = h0 ? h0[state + (int64_t)(j0 + jj) * D + c] : 0.f;
  }
  const int c0 = __ldg(plan.chunk_off + n), c1 = __ldg(plan.chunk_off + n + 1);
  const int64_t tstart = __ldg(plan.cu + n);
  const int64_t tend = max(tstart, (int64_t)__ldg(plan.cu + n + 1));
  const int lane = tid & 31, grp = tid >> 5;  // lane = value column, grp = row group
  __syncthreads();
  for (int chunk = c0; chunk < c1; ++chunk) {
    const float* unit = ws + ((int64_t)chunk * H + h) * kUnitFloats;
    for (int e = tid; e < C * (D / 4); e += kChainThreads) {
      const int r = e / (D / 4), c4 = (e % (D / 4)) * 4;
      const float4 w = *reinterpret_cast<const float4*>(unit + kOffW + r * D + c4);
      const float4 qg = *reinterpret_cast<const float4*>(unit + kOffQg + r * D + c4);
      const float4 kt = *reinterpret_cast<const float4*>(unit + kOffKt + r * D + c4);
      sm.W[r][c4] = w.x; sm.W[r][c4 + 1] = w.y; sm.W[r][c4 + 2] = w.z; sm.W[r][c4 + 3] = w.w;
      sm.Qg[r][c4] = qg.x; sm.Qg[r][c4 + 1] = qg.y; sm.Qg[r][c4 + 2] = qg.z; sm.Qg[r][c4 + 3] = qg.w;
      sm.Kt[r][c4] = kt.x; sm.Kt[r][c4 + 1] = kt.y; sm.Kt[r][c4 + 2] = kt.z; sm.Kt[r][c4 + 3] = kt.w;
    }
    for (int e = tid; e < C * C; e += kChainThreads) sm.Aq[e / C][e % C] = unit[kOffAqk + e];
    for (int e = tid; e < C * kSlice; e += kChainThreads) {
      const int r = e / kSlice, jj = e % kSlice;
      sm.U[r][jj] = unit[kOffU + r * D + j0 + jj];
    }
    if (tid < D) sm.gam[tid] = unit[kOffGam + tid];
    __syncthreads();
    // Vt = U - W S   (rows grp, grp+8, ..., column lane)
    for (int r = grp; r < C; r += 8) {
      float acc = 0.f;
#pragma unroll 8
      for (int c = 0; c < D; ++c) acc = fmaf(sm.W[r][c], sm.S[c][lane], acc);
      sm.Vt[r][lane] = sm.U[r][lane] - acc;
    }
    __syncthreads();
    // O = Qg S + Aq Vt
    const int64_t tc = tstart + (int64_t)(chunk - c0) * C;
    for (int r = grp; r < C; r += 8) {
      float acc = 0.f;
#pragma unroll 8
      for (int c = 0; c < D; ++c) acc = fmaf(sm.Qg[r][c], sm.S[c][lane], acc);
      for (int i = 0; i <= r; ++i) acc = fmaf(sm.Aq[r][i], sm.Vt[i][lane], acc);
      if (tc + r < tend) o[((tc + r) * H + h) * D + j0 + lane] = from_f32<T>(acc);
    }
    __syncthreads();
    // S = Diag(gamma_C) S + Kt^T Vt   (rows c = grp, grp+8, ...)
    for (int c = grp; c < D; c += 8) {
      float acc = sm.gam[c] * sm.S[c][lane];
#pragma unroll 8
      for (int i = 0; i < C; ++i) acc = fmaf(sm.Kt[i][c], sm.Vt[i][lane], acc);
      sm.S[c][lane] = acc;
    }
    __syncthreads();
  }
  if (hT) {
    for (int e = tid; e < D * kSlice; e += kChainThreads) {
      const int jj = e / D, c = e % D;
      hT[state + (int64_t)(j0 + jj) * D + c] = sm.S[c][jj];
    }
  }
}

}  // namespace

size_t simt_workspace_bytes(int64_t n_tokens, int n_seqs, int H) {
  return (size_t)chunks_upper_bound(n_tokens, n_seqs) * H * kUnitFloats * sizeof(float);
}

cudaError_t launch_chunk_simt(const void* q, const void* k, const void* v, int bf16,
                              const float* g, const void* beta, const float* h0, void* o,
                              float* hT, int64_t n_tokens, int n_seqs, int H, void* ws,
                              cudaStream_t s, int robust) {
  const Plan plan = plan_in(ws, n_tokens, n_seqs);
  float* body = reinterpret_cast<float*>(static_cast<char*>(ws) + plan_bytes(n_tokens, n_seqs));
  const int64_t chunks = chunks_upper_bound(n_tokens, n_seqs);
  const size_t prep_smem = sizeof(PrepSmem), chain_smem = sizeof(ChainSmem);
  cudaError_t e;
  if (chunks > 0) {
    const dim3 grid((unsigned)chunks, (unsigned)H);
    ProfScope prof_scope("kda_simt_prep", s);
    if (bf16) {
      using T = __nv_bfloat16;
      e = cudaFuncSetAttribute(simt_prep<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)prep_smem);
      if (e != cudaSuccess) return e;
      simt_prep<T><<<grid, kPrepThreads, prep_smem, s>>>(
          static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v), g,
          static_cast<const T*>(beta), plan, H, body, robust);
    } else {
      e = cudaFuncSetAttribute(simt_prep<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)prep_smem);
      if (e != cudaSuccess) return e;
      simt_prep<float><<<grid, kPrepThreads, prep_smem, s>>>(
          static_cast<const float*>(q), static_cast<const float*>(k),
          static_cast<const float*>(v), g, static_cast<const float*>(beta), plan, H, body,
          robust);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const dim3 cgrid((unsigned)n_seqs, (unsigned)H, (unsigned)(D / kSlice));
  ProfScope prof_scope("kda_simt_chain", s);
  if (bf16) {
    using T = __nv_bfloat16;
    e = cudaFuncSetAttribute(simt_chain<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)chain_smem);
    if (e != cudaSuccess) return e;
    simt_chain<T><<<cgrid, kChainThreads, chain_smem, s>>>(body, h0, plan, H,
                                                           static_cast<T*>(o), hT);
  } else {
    e = cudaFuncSetAttribute(simt_chain<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)chain_smem);
    if (e != cudaSuccess) return e;
    simt_chain<float><<<cgrid, kChainThreads, chain_smem, s>>>(body, h0, plan, H,
                                                               static_cast<float*>(o), hT);
  }
  return cudaGetLastError();
}

}  // namespace kda
