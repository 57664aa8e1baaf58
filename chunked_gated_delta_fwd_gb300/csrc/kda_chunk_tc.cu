// kda_chunk_tc.cu -- the chunkwise KDA forward for bf16 inputs on the sm_103a
// tensor cores (tcgen05.mma, fp32 accumulation in TMEM, fp32 state).
//
// Form evaluated ("Kimi K3 notes" (s1mplewind blog), section "Chunkwise form";
// "Hybrid KDA-MLA: Kimi K3 attention explained", section "KDA kernel"), per
// 64-token chunk with G the in-chunk running sum of g and Gamma = exp(G):
//   A_kk = StrictTril(Diag(beta)(Gamma*K)(K/Gamma)^T), A_qk = Tril((Gamma*Q)(K/Gamma)^T)
//   T = (I + A_kk)^{-1},  W = T Diag(beta)(Gamma*K),  U = T Diag(beta) V
//   Vt = U - W S,   O = (Gamma*Q) S + A_qk Vt,   S <- Diag(gamma_C) S + Kt^T Vt
// with Kt = (gamma_C/Gamma)*K.  S stays fp32 in tensor memory for a whole sequence.
//
// The two 64x64 products are dense tensor-core MMAs over 16-token tiles
// ("Kimi K3 technical report review" (devpress/CSDN), section 3.2: with g >= -5
// the cumulative log-decay of a 16-token tile is in (-80, 0), so the inverse
// decay inside a tile stays below e^80, inside the bf16 range).  With R_a the
// running log-decay just before tile a, the key operand for row tile a is
//   KC(a)_i = k_i * exp(R_a - G_i)     (i up to the end of tile a, zero beyond)
// whose entries are <= 1 outside tile a and < e^80 inside it, and the row operand
// is k_r * exp(G_r - R_a) <= 1 (resp. q_r * exp(G_r - R_a)); their product over
// the channels is sum_c k_rc k_ic exp(G_rc - G_ic).
//
// Kernel 1, tc_prep: one persistent CTA per SM walks (chunk, head) units and
// writes, per unit, MMA-ready bf16 tiles to the workspace:
//   WQ [128 rows][128]: rows 0..63 = W, rows 64..127 = Gamma*Q   (B of MMA1)
//   UT [128 rows][64] : U^T (dv rows, token columns)             (read by threads)
//   AK [192 rows][64] : rows 0..63 = A_qk, rows 64..191 = Kt^T   (B of MMA2)
// and gamma_C (fp32 [128]) separately.
// Kernel 2, tc_chain: one CTA per (sequence, head) walks its chunks in order.
// TMEM holds S^T (lanes = dv, columns = dk) and two buffers for
//   MMA1: D1 = S^T [W; Gamma*Q]^T        -> (W S)^T | (Gamma*Q S)^T
//   MMA2: D1[:,64:] += Vt^T A_qk^T ;  S^T += Vt^T Kt  (after S^T *= gamma_C)
// where Vt^T = U^T - (W S)^T is formed by the epilogue warps.  Tiles stream in
// with 1-D bulk async copies through a two-stage ring.
#include "kda_internal.cuh"
#include "kda_sm100.cuh"

namespace kda {
namespace {

using namespace sm100;

constexpr int C = kChunk;  // 64
constexpr int D = kD;      // 128

// ---- workspace unit (bytes)
constexpr uint32_t kWQ = 0;                   // 128 rows x 128 cols bf16, SW128 K-major
constexpr uint32_t kUT = 32768;               // 128 rows x 64 cols
constexpr uint32_t kAK = 49152;               // 192 rows x 64 cols
constexpr uint32_t kUnitBytes = 73728;
constexpr uint32_t kGamBytes = D * 4;

// ============================================================== prep kernel
constexpr int kPrepThreads = 128;
// shared memory (offsets from a 1024-aligned base)
constexpr uint32_t kP_Bop = 0;         // [Kb t0; Qb t0; Kb t1; Qb t1; ...] 128 rows x 128 (32 KB)
constexpr uint32_t kP_T = 0;           //   reused: T (64 x 64 bf16, 8 KB) after the products
constexpr uint32_t kP_L = 8192;        //   reused: L (64 x 65 fp32) after the products
constexpr uint32_t kP_KC01 = 32768;    // [KC(0); KC(1)] 128 rows x 128 (32 KB)
constexpr uint32_t kP_KC23 = 65536;    // [KC(2); KC(3)]
constexpr uint32_t kP_BKg = 98304;     // (beta Gamma K)^T 128 rows x 64 (16 KB)
constexpr uint32_t kP_BV = 114688;     // (beta V)^T 128 rows x 64
constexpr uint32_t kP_beta = 131072;   // 64 fp32
constexpr uint32_t kP_bars = 131328;   // 2 mbarriers + TMEM base
constexpr uint32_t kP_Smem = kP_bars + 64 + 1024;  // + alignment slack
constexpr int kLdL = 65;

__device__ __forceinline__ void st_bf16(uint8_t* base, uint32_t off, float x) {
  *reinterpret_cast<__nv_bfloat16*>(base + off) = __float2bfloat16_rn(x);
}

__global__ void __launch_bounds__(kPrepThreads, 1)
    tc_prep(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
            const __nv_bfloat16* __restrict__ v, const float* __restrict__ g,
            const __nv_bfloat16* __restrict__ beta, Plan plan, int H, int64_t units_ub,
            uint8_t* __restrict__ tiles, float* __restrict__ gam_out, int* err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_addr(sm);
  float* beta_s = reinterpret_cast<float*>(sm + kP_beta);
  float* Ls = reinterpret_cast<float*>(sm + kP_L);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kP_bars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kP_bars + 16);
  const uint32_t bar_p = smem_addr(&bars[0]), bar_w = smem_addr(&bars[1]);
  const int t = threadIdx.x, warp = t >> 5;

  // the KC tiles keep zero rows beyond their tile for the whole kernel
  for (uint32_t o = t * 16; o < 65536; o += kPrepThreads * 16)
    *reinterpret_cast<uint4*>(sm + kP_KC01 + o) = make_uint4(0, 0, 0, 0);
  if (t == 0) {
    mbar_init(bar_p, 1);
    mbar_init(bar_w, 1);
    mbar_fence_init();
  }
  if (warp == 0) tmem_alloc(smem_addr(tmem_slot), 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
  const int total = __ldg(plan.chunk_off + plan.n_seqs);
  uint32_t iter = 0;

  for (int64_t u = blockIdx.x; u < units_ub; u += gridDim.x) {
    const int chunk = (int)(u / H), h = (int)(u % H);
    if (chunk >= total) break;  // units are chunk-major: the rest are past the end
    int n = 0;
    {
      int lo = 0, hi = plan.n_seqs - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(plan.chunk_off + mid) <= chunk) lo = mid; else hi = mid - 1;
      }
      n = lo;
    }
    const int64_t t0 = (int64_t)__ldg(plan.cu + n) + (int64_t)(chunk - __ldg(plan.chunk_off + n)) * C;
    const int len = (int)min((int64_t)C, (int64_t)__ldg(plan.cu + n + 1) - t0);
    uint8_t* unit = tiles + (size_t)u * kUnitBytes;
    const int c = t;  // channel owned by this thread in the elementwise passes

    // ---- pass 1: running log-decay of channel c, tile references
    float G[C];
    {
      float acc = 0.f;
#pragma unroll
      for (int r = 0; r < C; ++r) {
        const float gv = (r < len) ? __ldg(g + ((t0 + r) * H + h) * D + c) : 0.f;
        acc += gv;
        G[r] = acc;
      }
    }
    if (t < C) beta_s[t] = (t < len) ? __bfloat162float(beta[(t0 + t) * H + h]) : 0.f;
    const float R[4] = {0.f, G[15], G[31], G[47]};
    const float GC = G[63];
    __syncthreads();

    // ---- pass 2: operands
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      float E[4];  // exp(R_a' - R_a) for a' >= a
#pragma unroll
      for (int ap = 0; ap < 4; ++ap) E[ap] = (ap > a) ? __expf(R[ap] - R[a]) : 1.f;
      const float eRa = __expf(R[a]);           // exp(R_a) <= 1
      const float eCa = __expf(GC - R[a]);      // exp(G_C - R_a) <= 1
      float kr[16], qr[16], vr[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int r = a * 16 + j;
        const int64_t off = ((t0 + r) * H + h) * D + c;
        const bool in = r < len;
        kr[j] = in ? __bfloat162float(k[off]) : 0.f;
        qr[j] = in ? __bfloat162float(q[off]) : 0.f;
        vr[j] = in ? __bfloat162float(v[off]) : 0.f;
      }
      uint32_t pk_kg[8], pk_v[8], pk_kt[8];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int r = a * 16 + j;
        const float d = G[r] - R[a];  // (-80, 0]
        const float f = __expf(d), fi = __expf(-d);
        const float kb = kr[j] * f, qb = qr[j] * f, kn = kr[j] * fi;
        st_bf16(sm, kP_Bop + sw128_offset(128, 32 * a + j, c), kb);
        st_bf16(sm, kP_Bop + sw128_offset(128, 32 * a + 16 + j, c), qb);
#pragma unroll
        for (int ap = a; ap < 4; ++ap)
          st_bf16(sm, (ap < 2 ? kP_KC01 : kP_KC23) + sw128_offset(128, 64 * (ap & 1) + r, c),
                  kn * E[ap]);
        const float kg = kb * eRa * beta_s[r];
        const float vb = vr[j] * beta_s[r];
        const float kt = kn * eCa;
        if (j & 1) {
          pk_kg[j >> 1] = pack_bf16(__uint_as_float(pk_kg[j >> 1]), kg);
          pk_v[j >> 1] = pack_bf16(__uint_as_float(pk_v[j >> 1]), vb);
          pk_kt[j >> 1] = pack_bf16(__uint_as_float(pk_kt[j >> 1]), kt);
        } else {
          pk_kg[j >> 1] = __float_as_uint(kg);
          pk_v[j >> 1] = __float_as_uint(vb);
          pk_kt[j >> 1] = __float_as_uint(kt);
        }
        // Gamma*Q -> WQ rows 64.., column c
        *reinterpret_cast<__nv_bfloat16*>(unit + kWQ + sw128_offset(128, 64 + r, c)) =
            __float2bfloat16_rn(qb * eRa);
      }
#pragma unroll
      for (int hc = 0; hc < 2; ++hc) {
        const int ch = 2 * a + hc;  // token chunk of 8
        const uint4 wk = make_uint4(pk_kg[4 * hc], pk_kg[4 * hc + 1], pk_kg[4 * hc + 2], pk_kg[4 * hc + 3]);
        const uint4 wv = make_uint4(pk_v[4 * hc], pk_v[4 * hc + 1], pk_v[4 * hc + 2], pk_v[4 * hc + 3]);
        const uint4 wt = make_uint4(pk_kt[4 * hc], pk_kt[4 * hc + 1], pk_kt[4 * hc + 2], pk_kt[4 * hc + 3]);
        *reinterpret_cast<uint4*>(sm + kP_BKg + sw128_chunk(128, c, ch)) = wk;
        *reinterpret_cast<uint4*>(sm + kP_BV + sw128_chunk(128, c, ch)) = wv;
        *reinterpret_cast<uint4*>(unit + kAK + sw128_chunk(192, 64 + c, ch)) = wt;
      }
    }
    gam_out[(size_t)u * D + c] = __expf(GC);

    // ---- block products: D[:, 0:64] = [KC0; KC1] x Bop[0:64]^T, D[:, 64:128] = [KC2; KC3] x Bop[64:128]^T
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (t == 0) {
      tc_fence_after();
      const uint32_t id = idesc_bf16(128, 64);
      mma_tile(tmem + 0, sbase + kP_KC01, 128, sbase + kP_Bop, 128, D, id, false);
      mma_tile(tmem + 64, sbase + kP_KC23, 128, sbase + kP_Bop + 64 * 128, 128, D, id, false);
      mma_commit(bar_p);
    }
    bool ok = mbar_wait(bar_p, iter & 1, err);
    if (!__syncthreads_and(ok)) break;
    tc_fence_after();
    {
      const int half = t >> 6, i = t & 63;
      float pv[2][32];
      tmem_ld32(lane_addr + 32 * half, pv[0]);
      tmem_ld32(lane_addr + 64 + 32 * half, pv[1]);
      tmem_wait_ld();
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        const int a = half + 2 * s;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int r = 16 * a + j;
          Ls[r * kLdL + i] = (i < r) ? beta_s[r] * pv[s][j] : 0.f;
          *reinterpret_cast<__nv_bfloat16*>(unit + kAK + sw128_offset(192, r, i)) =
              __float2bfloat16_rn((i <= r) ? pv[s][16 + j] : 0.f);
        }
      }
    }
    __syncthreads();

    // ---- T = (I + L)^{-1}: forward substitution, one column per thread (warps 0-1)
    if (t < C) {
      const int jc = t;
      float x[C];
#pragma unroll
      for (int r = 0; r < C; ++r) {
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < r; ++i) acc = fmaf(Ls[r * kLdL + i], x[i], acc);
        x[r] = (r < jc) ? 0.f : (r == jc ? 1.f : -acc);
      }
#pragma unroll
      for (int r = 0; r < C; ++r) st_bf16(sm, kP_T + sw128_offset(64, r, jc), x[r]);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (t == 0) {
      tc_fence_after();
      const uint32_t id = idesc_bf16(128, 64);
      mma_tile(tmem + 128, sbase + kP_BKg, 128, sbase + kP_T, 64, C, id, false);  // W^T
      mma_tile(tmem + 192, sbase + kP_BV, 128, sbase + kP_T, 64, C, id, false);   // U^T
      mma_commit(bar_w);
    }
    ok = mbar_wait(bar_w, iter & 1, err);
    if (!__syncthreads_and(ok)) break;
    tc_fence_after();
    {
      float w0[32], w1[32];
      tmem_ld32(lane_addr + 128, w0);
      tmem_ld32(lane_addr + 160, w1);
      tmem_wait_ld();
#pragma unroll
      for (int r = 0; r < 32; ++r) {
        *reinterpret_cast<__nv_bfloat16*>(unit + kWQ + sw128_offset(128, r, c)) = __float2bfloat16_rn(w0[r]);
        *reinterpret_cast<__nv_bfloat16*>(unit + kWQ + sw128_offset(128, 32 + r, c)) = __float2bfloat16_rn(w1[r]);
      }
      tmem_ld32(lane_addr + 192, w0);
      tmem_ld32(lane_addr + 224, w1);
      tmem_wait_ld();
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        const float* src = ch < 4 ? &w0[8 * ch] : &w1[8 * (ch - 4)];
        const uint4 wv = make_uint4(pack_bf16(src[0], src[1]), pack_bf16(src[2], src[3]),
                                    pack_bf16(src[4], src[5]), pack_bf16(src[6], src[7]));
        *reinterpret_cast<uint4*>(unit + kUT + sw128_chunk(128, c, ch)) = wv;
      }
    }
    tc_fence_before();
    __syncthreads();
    ++iter;
  }
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

// ============================================================= chain kernel
constexpr int kStages = 2;
constexpr uint32_t kStageBytes = 75776;                 // unit (72 KB) + gamma (512 B), 1024-aligned
constexpr uint32_t kC_Sbf = kStages * kStageBytes;      // S^T bf16, 128 x 128 (32 KB)
constexpr uint32_t kC_Vt = kC_Sbf + 32768;              // Vt^T bf16, 128 x 64 (16 KB)
constexpr uint32_t kC_bars = kC_Vt + 16384;
constexpr uint32_t kC_Smem = kC_bars + 128 + 1024;
constexpr int kChainThreads = 160;  // warps 0-3: epilogue (TMEM lanes), warp 4: copies + MMA

__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, int* err,
                                              volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > kWaitTimeoutNs) {
        if (err) atomicExch(err, kDevErrTimeout);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

__global__ void __launch_bounds__(kChainThreads, 1)
    tc_chain(const uint8_t* __restrict__ tiles, const float* __restrict__ gam,
             const float* __restrict__ h0, Plan plan, int H, __nv_bfloat16* __restrict__ o,
             float* __restrict__ hT, int* err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_addr(sm);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kC_bars);
  // bars: 0,1 = full[stage], 2 = S ready (bf16 copy written, S scaled), 3 = MMA1 done,
  //       4 = Vt ready, 5 = MMA2 done
  const uint32_t bar_full0 = smem_addr(&bars[0]);
  const uint32_t bar_s = smem_addr(&bars[2]), bar_m1 = smem_addr(&bars[3]);
  const uint32_t bar_vt = smem_addr(&bars[4]), bar_m2 = smem_addr(&bars[5]);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kC_bars + 64);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kC_bars + 72);
  const int t = threadIdx.x, warp = t >> 5;
  const int n = blockIdx.x, h = blockIdx.y;

  if (t == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(bar_full0 + 8 * s, 1);
    mbar_init(bar_s, 128);
    mbar_init(bar_m1, 1);
    mbar_init(bar_vt, 128);
    mbar_init(bar_m2, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 0) tmem_alloc(smem_addr(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int c0 = __ldg(plan.chunk_off + n), c1 = __ldg(plan.chunk_off + n + 1);
  const int nch = c1 - c0;
  const int64_t tstart = __ldg(plan.cu + n);
  const int64_t tend = max(tstart, (int64_t)__ldg(plan.cu + n + 1));
  const int64_t state = ((int64_t)n * H + h) * D * D;

  if (warp == 4) {
    // ------------------------------------------------ copies + MMA issue (one thread)
    if ((t & 31) == 0) {
      auto issue = [&](int jj) {
        const int s = jj % kStages;
        const int64_t u = (int64_t)(c0 + jj) * H + h;
        const uint32_t bar = bar_full0 + 8 * s;
        mbar_arrive_expect_tx(bar, kUnitBytes + kGamBytes);
        bulk_g2s(sbase + s * kStageBytes, tiles + (size_t)u * kUnitBytes, kUnitBytes, bar);
        bulk_g2s(sbase + s * kStageBytes + kUnitBytes, gam + (size_t)u * D, kGamBytes, bar);
      };
      int issued = 0, consumed = 0;
      for (; issued < min(kStages, nch); ++issued) issue(issued);
      const uint32_t id1 = idesc_bf16(128, 128), id2a = idesc_bf16(128, 64);
      int j = 0;
      bool mma_pending = false;
      for (; j < nch; ++j) {
        const int s = j % kStages;
        const uint32_t st = sbase + s * kStageBytes;
        if (!wait_or_abort(bar_s, j & 1, err, abort_flag)) break;
        if (!wait_or_abort(bar_full0 + 8 * s, (j / kStages) & 1, err, abort_flag)) break;
        consumed = j + 1;
        tc_fence_after();
        const uint32_t d1 = tmem + 128 + 128 * (j & 1);
        mma_tile(d1, sbase + kC_Sbf, 128, st + kWQ, 128, D, id1, false);
        mma_commit(bar_m1);
        if (!wait_or_abort(bar_vt, j & 1, err, abort_flag)) { mma_pending = true; break; }
        tc_fence_after();
        mma_tile(d1 + 64, sbase + kC_Vt, 128, st + kAK, 192, C, id2a, true);
        mma_tile(tmem + 0, sbase + kC_Vt, 128, st + kAK + 64 * 128, 192, C, id1, true);
        mma_commit(bar_m2);
        if (j + kStages < nch) {
          if (!wait_or_abort(bar_m2, j & 1, err, abort_flag)) { mma_pending = true; break; }
          issue(issued++);
        }
      }
      if (*abort_flag) {
        // drain: copies and MMAs already issued must land before the CTA exits
        for (int jj = consumed; jj < issued; ++jj)
          mbar_wait(bar_full0 + 8 * (jj % kStages), (jj / kStages) & 1, nullptr);
        if (mma_pending) mbar_wait(bar_m2, j & 1, nullptr);
      }
    }
  } else {
    // ------------------------------------------------ epilogue warps: TMEM lane = dv = t
    const uint32_t lane = tmem + ((uint32_t)(warp * 32) << 16);
    {
      float sv[32];
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        if (h0) {
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float4 x = *reinterpret_cast<const float4*>(h0 + state + (int64_t)t * D + 32 * qq + i);
            sv[i] = x.x; sv[i + 1] = x.y; sv[i + 2] = x.z; sv[i + 3] = x.w;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) sv[i] = 0.f;
        }
        tmem_st32(lane + 32 * qq, sv);
      }
      tmem_wait_st();
    }
    auto store_o = [&](int jj) {
      float ov[2][32];
      const uint32_t d1 = lane + 128 + 128 * (jj & 1) + 64;
      tmem_ld32(d1, ov[0]);
      tmem_ld32(d1 + 32, ov[1]);
      tmem_wait_ld();
      const int64_t tc = tstart + (int64_t)jj * C;
#pragma unroll
      for (int r = 0; r < C; ++r)
        if (tc + r < tend) o[((tc + r) * H + h) * D + t] = __float2bfloat16_rn(ov[r >> 5][r & 31]);
    };
    bool alive = true;
    for (int j = 0; j < nch && alive; ++j) {
      const int s = j % kStages;
      uint8_t* st = sm + s * kStageBytes;
      const float* gam_s = reinterpret_cast<const float*>(st + kUnitBytes);
      // E0: S^T row -> bf16 operand copy, then S^T *= gamma_C (column-wise)
      if (j > 0 && !wait_or_abort(bar_m2, (j - 1) & 1, err, abort_flag)) { alive = false; break; }
      if (!wait_or_abort(bar_full0 + 8 * s, (j / kStages) & 1, err, abort_flag)) { alive = false; break; }
      tc_fence_after();
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        float sv[32];
        tmem_ld32(lane + 32 * qq, sv);
        tmem_wait_ld();
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          const uint4 w = make_uint4(pack_bf16(sv[8 * ch], sv[8 * ch + 1]),
                                     pack_bf16(sv[8 * ch + 2], sv[8 * ch + 3]),
                                     pack_bf16(sv[8 * ch + 4], sv[8 * ch + 5]),
                                     pack_bf16(sv[8 * ch + 6], sv[8 * ch + 7]));
          *reinterpret_cast<uint4*>(sm + kC_Sbf + sw128_chunk(128, t, 4 * qq + ch)) = w;
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) sv[i] *= gam_s[32 * qq + i];
        tmem_st32(lane + 32 * qq, sv);
      }
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar_s);
      // E2 of the previous chunk (its D1 buffer is not touched by MMA1 of this chunk)
      if (j > 0) store_o(j - 1);
      // E1: Vt^T = U^T - (W S)^T
      if (!wait_or_abort(bar_m1, j & 1, err, abort_flag)) { alive = false; break; }
      tc_fence_after();
      {
        float wsv[2][32];
        const uint32_t d1 = lane + 128 + 128 * (j & 1);
        tmem_ld32(d1, wsv[0]);
        tmem_ld32(d1 + 32, wsv[1]);
        tmem_wait_ld();
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          const uint4 uu = *reinterpret_cast<const uint4*>(st + kUT + sw128_chunk(128, t, ch));
          const float* wsrc = &wsv[ch >> 2][8 * (ch & 3)];
          const uint32_t uw[4] = {uu.x, uu.y, uu.z, uu.w};
          uint32_t out[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            out[e] = pack_bf16(bf16_lo(uw[e]) - wsrc[2 * e], bf16_hi(uw[e]) - wsrc[2 * e + 1]);
          *reinterpret_cast<uint4*>(sm + kC_Vt + sw128_chunk(128, t, ch)) =
              make_uint4(out[0], out[1], out[2], out[3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar_vt);
    }
    if (alive && nch > 0 && wait_or_abort(bar_m2, (nch - 1) & 1, err, abort_flag)) {
      tc_fence_after();
      store_o(nch - 1);
    }
    if (hT && !*abort_flag) {
      tc_fence_after();
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        float sv[32];
        tmem_ld32(lane + 32 * qq, sv);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; i += 4)
          *reinterpret_cast<float4*>(hT + state + (int64_t)t * D + 32 * qq + i) =
              make_float4(sv[i], sv[i + 1], sv[i + 2], sv[i + 3]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

int sm_count() {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms;
}

}  // namespace

size_t tc_workspace_bytes(int64_t n_tokens, int n_seqs, int H) {
  const size_t units = (size_t)chunks_upper_bound(n_tokens, n_seqs) * H;
  return units * (kUnitBytes + kGamBytes) + 1024;
}

cudaError_t launch_chunk_tc(const void* q, const void* k, const void* v, const float* g,
                            const void* beta, const float* h0, void* o, float* hT,
                            int64_t n_tokens, int n_seqs, int H, void* ws, int* err,
                            cudaStream_t s) {
  Plan plan;
  plan.cu = static_cast<const int32_t*>(ws);
  plan.chunk_off = plan.cu + (n_seqs + 1);
  plan.n_seqs = n_seqs;
  const int64_t units = chunks_upper_bound(n_tokens, n_seqs) * H;
  uintptr_t body = reinterpret_cast<uintptr_t>(ws) + plan_bytes(n_seqs);
  body = (body + 1023) & ~uintptr_t(1023);
  uint8_t* tiles = reinterpret_cast<uint8_t*>(body);
  float* gam = reinterpret_cast<float*>(tiles + (size_t)units * kUnitBytes);
  cudaError_t e;
  using T = __nv_bfloat16;
  if (units > 0) {
    e = cudaFuncSetAttribute(tc_prep, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kP_Smem);
    if (e != cudaSuccess) return e;
    const int grid = (int)(units < sm_count() ? units : sm_count());
    ProfScope prof_scope("kda_tc_prep", s);
    tc_prep<<<grid, kPrepThreads, kP_Smem, s>>>(
        static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v), g,
        static_cast<const T*>(beta), plan, H, units, tiles, gam, err);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  e = cudaFuncSetAttribute(tc_chain, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kC_Smem);
  if (e != cudaSuccess) return e;
  const dim3 cgrid((unsigned)n_seqs, (unsigned)H);
  ProfScope prof_scope("kda_tc_chain", s);
  tc_chain<<<cgrid, kChainThreads, kC_Smem, s>>>(tiles, gam, h0, plan, H, static_cast<T*>(o), hT,
                                                  err);
  return cudaGetLastError();
}

}  // namespace kda
