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
// Kernel 1, tc_prep: persistent 256-thread CTAs, two per SM, walk (chunk, head)
// units, each CTA one unit at a time; the SM's two CTAs overlap each other's
// phases.  A unit's k, q and z (or g) arrive by 3-D tensor copies issued during the
// previous unit; each thread sums the decays of 16 tokens x 2 channels in
// registers and builds their operands; one thread issues the MMAs (the four tile
// products in one N=160 chain, then W^T and U^T); the (I + A_kk)^{-1} inverse runs
// in fp32 on the CUDA cores.  The unit leaves as MMA-ready bf16 tiles written with
// bulk copies from shared memory:
//   W, Gamma*Q: MN-major, 64 token columns x 128 channels each (one operand with
//               a 16 KB atom stride)
//   UT: K-major, U^T (128 value rows x 64 tokens)
//   AQ: K-major, A_qk (64 x 64);  KT: K-major, Kt^T (128 channel rows x 64 tokens)
// plus gamma_C (fp32 [128]).
// Kernel 2, tc_chain: one CTA per (sequence, head) walks its chunks in order.
// TMEM holds S^T (lanes = dv, columns = dk, fp32 for the whole sequence), its bf16
// copy (the A operand of MMA1), two D1 buffers and two Vt^T buffers:
//   MMA1: D1 = S^T [W; Gamma*Q]^T      -> (W S)^T | (Gamma*Q S)^T
//   MMA2: S^T += Vt^T Kt (after S^T *= gamma_C);  D1[:, 64:] += Vt^T A_qk^T
// where Vt^T = U^T - (W S)^T is formed by eight epilogue warps, two of whose
// threads issue the serial MMAs ((W S)^T, the state update) after named barriers;
// an output warp issues the (Gamma*Q S)^T half and the O product, four store warps
// write o, and a copy warp streams the tiles through a three-stage ring of bulk
// copies.
#include "kda_internal.cuh"
#include "kda_sm100.cuh"

#include <cuda.h>

#include <string.h>

#include <mutex>

namespace kda {
namespace {

using namespace sm100;

constexpr int C = kChunk;  // 64
constexpr int D = kD;      // 128

// ---- workspace unit (bytes)
constexpr uint32_t kW = 0;         // MN-major X=64 (tokens), K=128: 16 KB
constexpr uint32_t kQ = 16384;     // same layout; [W | Q] read as one X=128 operand
constexpr uint32_t kUT = 32768;    // K-major 128 rows x 64: 16 KB
constexpr uint32_t kAQ = 49152;    // K-major A_qk, 64 rows r x 64 columns i: 8 KB
constexpr uint32_t kKT = 57344;    // K-major 128 rows x 64: 16 KB
constexpr uint32_t kUnitBytes = 73728;
constexpr uint32_t kGamBytes = D * 4;
// The precise-state mode keeps Kt^T in fp32 (K-major SW128 with 32 fp32 per
// 128-byte row: two column blocks of 128 rows x 32 tokens), 16 KB more per unit.
template <bool kP>
__host__ __device__ constexpr uint32_t unit_bytes() { return kP ? kUnitBytes + 16384 : kUnitBytes; }
// Byte offset of tokens 4 xc .. 4 xc + 3 of row (channel) c in the fp32 Kt^T tile.
__host__ __device__ __forceinline__ uint32_t kt32_chunk(int c, int xc) {
  return (uint32_t)((xc >> 3) * 16384 + c * 128 + (((xc & 7) ^ (c & 7)) << 4));
}

// ============================================================== prep kernel
// The key operand, MN-major X=192 (tokens), K=128: [KC(0) | KC(1) | KC(2) | KC(3)] at
// X = 0, 16, 48, 96 (16, 32, 48, 64 rows), X = 160..191 unused.
constexpr int kKCX = 192;
// The inverse's scratch: L, T fp32 [64][68] (16-byte rows: float4 loads along k) and
// the block products, fp32 [3][16][16].
constexpr int kLdL = 68, kLdT = 68;
constexpr int kInvThreads = 256;  // the inverse runs on warps 0-7
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ uint4 pack8(const float* x) {
  return make_uint4(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]), pack_bf16(x[4], x[5]),
                    pack_bf16(x[6], x[7]));
}
__device__ __forceinline__ uint4 pack8(const float2* x) {
  return make_uint4(pack_bf16(x[0].x, x[0].y), pack_bf16(x[1].x, x[1].y), pack_bf16(x[2].x, x[2].y),
                    pack_bf16(x[3].x, x[3].y));
}
// Products and sums on two fp32 lanes at once (one packed f32x2 instruction, each
// lane rounded like the scalar operation): s2 broadcasts a scalar into both lanes.
__device__ __forceinline__ float2 s2(float a) { return make_float2(a, a); }
__device__ __forceinline__ float2 lo2(float4 v) { return make_float2(v.x, v.y); }
__device__ __forceinline__ float2 hi2(float4 v) { return make_float2(v.z, v.w); }

// One 16-byte chunk of M = T Diag(beta) as the bf16 B operand of the W/U products
// (MN-major, X = row r, K = column j): rows 8 o8 .. 8 o8 + 7 of column j, zero above
// the diagonal.  A warp reads 32 consecutive columns of one row: no bank conflicts.
// With beta in M, W = M (Gamma K) and U = M V take Gamma K and V as they are (beta
// is zero on the rows past a sequence's end).
__device__ __forceinline__ void store_m_chunk(const float* __restrict__ Tb,
                                              const float* __restrict__ beta_s,
                                              uint8_t* __restrict__ mt, int o8, int j) {
  const float bj = beta_s[j];
  float x[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const int r = 8 * o8 + e;
    x[e] = (r >= j) ? Tb[r * kLdT + j] * bj : 0.f;
  }
  *reinterpret_cast<uint4*>(mt + mn_chunk(64, o8, j)) = pack8(x);
}

// T = (I + L)^{-1} of a unit's strictly lower, beta-scaled L (fp32 [64][kLdL] in Lb)
// into Tb (fp32 [64][kLdT], zeros above the diagonal of each stored block), with
// block products in Ps, and M = T Diag(beta) into the bf16 tile mt: three quarters
// of it once level 1 is done, the lower-left 32x32 block by the warp pair that forms
// it.  Called by threads 0..255 (warps 0-7) together; uses named barriers 2-9.
// before_level2() runs on every thread between level 1 and level 2.
template <typename Hook>
__device__ __forceinline__ void invert_unit_lower(const float* __restrict__ Lb,
                                                  float* __restrict__ Tb,
                                                  float* __restrict__ Ps,
                                                  const float* __restrict__ beta_s,
                                                  uint8_t* __restrict__ mt, int t,
                                                  Hook&& before_level2) {
  const int warp = t >> 5;
  if (t < 128) {
    // ---- T = (I + L)^{-1} in fp32.  Warp wq owns diagonal 16x16 block wq: its 8x8
    //      halves by forward substitution, then [A 0; C B]^{-1} lower-left
    //      = -B^{-1} C A^{-1}, warp-synchronous.  Level 1: warp 2b forms
    //      P = L_{2b+1,2b} D_{2b} from its own block and hands it to warp 2b+1
    //      (named barrier 3 + b), which forms T_{2b+1,2b} = -D_{2b+1} P.  Level 2 below,
    //      on warps 4-7 from the end of level 0 and on warps 0-7 after level 1.
    //      Stored blocks carry zeros above their diagonals; blocks above the
    //      diagonal are never stored nor read.
    const int wq = warp, o = 16 * wq, wl = t & 31;  // warp, its block, lane in warp
    if (wl < 16) {  // A^{-1} (lanes 0-7), B^{-1} (lanes 8-15): one column per lane
      const int ob = o + 8 * (wl >> 3), cc = wl & 7;
      float x[8];
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        float lr[8];
        *reinterpret_cast<float4*>(lr) = *reinterpret_cast<const float4*>(Lb + (ob + m) * kLdL + ob);
        *reinterpret_cast<float4*>(lr + 4) =
            *reinterpret_cast<const float4*>(Lb + (ob + m) * kLdL + ob + 4);
        float acc = 0.f;
#pragma unroll
        for (int i2 = 0; i2 < m; ++i2) acc = fmaf(lr[i2], x[i2], acc);
        x[m] = (m < cc) ? 0.f : (m == cc ? 1.f : -acc);
      }
#pragma unroll
      for (int m = 0; m < 8; ++m) Tb[(ob + m) * kLdT + ob + cc] = x[m];
      if (wl < 8) {  // the zero upper-right 8x8 of the 16x16 block
#pragma unroll
        for (int m = 0; m < 8; ++m) Tb[(ob + m) * kLdT + ob + 8 + cc] = 0.f;
      }
    }
    __syncwarp();
    const int di = wl >> 2, dj = 2 * (wl & 3);  // 8x8: row di, columns dj, dj + 1
    {  // P = C A^{-1}
      float lr[8];
      *reinterpret_cast<float4*>(lr) = *reinterpret_cast<const float4*>(Lb + (o + 8 + di) * kLdL + o);
      *reinterpret_cast<float4*>(lr + 4) =
          *reinterpret_cast<const float4*>(Lb + (o + 8 + di) * kLdL + o + 4);
      float a0 = 0.f, a1 = 0.f;
#pragma unroll
      for (int k = 0; k < 8; ++k) {  // A^{-1} has stored zeros above the diagonal
        a0 = fmaf(lr[k], Tb[(o + k) * kLdT + o + dj], a0);
        a1 = fmaf(lr[k], Tb[(o + k) * kLdT + o + dj + 1], a1);
      }
      Ps[wq * 64 + di * 8 + dj] = a0;
      Ps[wq * 64 + di * 8 + dj + 1] = a1;
    }
    __syncwarp();
    {  // lower-left 8x8 = -B^{-1} P
      float wr[8];
      *reinterpret_cast<float4*>(wr) = *reinterpret_cast<const float4*>(Tb + (o + 8 + di) * kLdT + o + 8);
      *reinterpret_cast<float4*>(wr + 4) =
          *reinterpret_cast<const float4*>(Tb + (o + 8 + di) * kLdT + o + 12);
      float a0 = 0.f, a1 = 0.f;
#pragma unroll
      for (int k = 0; k < 8; ++k) {  // B^{-1} has stored zeros above the diagonal
        a0 = fmaf(wr[k], Ps[wq * 64 + k * 8 + dj], a0);
        a1 = fmaf(wr[k], Ps[wq * 64 + k * 8 + dj + 1], a1);
      }
      Tb[(o + 8 + di) * kLdT + o + dj] = -a0;
      Tb[(o + 8 + di) * kLdT + o + dj + 1] = -a1;
    }
    __syncwarp();
    if (wq < 2) named_arrive(5, 192);  // D_0, D_1 are stored: warps 4-7 may read them
    // level 1 (2 rows x 4 columns per wl: rows rp and rp + 8)
    const int blk = wq >> 1, a = 2 * blk, R = a + 1, rp = (wl >> 2) & 7, cq = wl & 3;
    float* P1 = Ps + 256 + blk * 256;
    if ((wq & 1) == 0) {  // P = L_{a+1,a} D_a
      float2 acc[2][2] = {};
#pragma unroll 1  // kept rolled: less code for the instruction cache
      for (int k4 = 0; k4 < 16; k4 += 4) {
        float lv[2][4];
#pragma unroll
        for (int r = 0; r < 2; ++r)
          *reinterpret_cast<float4*>(lv[r]) =
              *reinterpret_cast<const float4*>(Lb + (16 * R + rp + 8 * r) * kLdL + 16 * a + k4);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const float4 tv =
              *reinterpret_cast<const float4*>(Tb + (16 * a + k4 + kk) * kLdT + 16 * a + 4 * cq);
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            acc[r][0] = __ffma2_rn(s2(lv[r][kk]), lo2(tv), acc[r][0]);
            acc[r][1] = __ffma2_rn(s2(lv[r][kk]), hi2(tv), acc[r][1]);
          }
        }
      }
#pragma unroll
      for (int r = 0; r < 2; ++r)
        *reinterpret_cast<float4*>(P1 + (rp + 8 * r) * 16 + 4 * cq) =
            make_float4(acc[r][0].x, acc[r][0].y, acc[r][1].x, acc[r][1].y);
      named_arrive(3 + blk, 64);
    } else {  // T_{a+1,a} = -D_{a+1} P
      named_sync(3 + blk, 64);
      float2 acc[2][2] = {};
#pragma unroll 1  // kept rolled: less code for the instruction cache
      for (int k4 = 0; k4 < 16; k4 += 4) {
        float wv[2][4];
#pragma unroll
        for (int r = 0; r < 2; ++r)
          *reinterpret_cast<float4*>(wv[r]) =
              *reinterpret_cast<const float4*>(Tb + (16 * R + rp + 8 * r) * kLdT + 16 * R + k4);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const float4 pv = *reinterpret_cast<const float4*>(P1 + (k4 + kk) * 16 + 4 * cq);
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            acc[r][0] = __ffma2_rn(s2(wv[r][kk]), lo2(pv), acc[r][0]);
            acc[r][1] = __ffma2_rn(s2(wv[r][kk]), hi2(pv), acc[r][1]);
          }
        }
      }
#pragma unroll
      for (int r = 0; r < 2; ++r)
        *reinterpret_cast<float4*>(Tb + (16 * R + rp + 8 * r) * kLdT + 16 * a + 4 * cq) =
            make_float4(-acc[r][0].x, -acc[r][0].y, -acc[r][1].x, -acc[r][1].y);
    }
  } else if (t < kInvThreads) {
    // Warps 4-7, while warps 0-3 run level 1: the terms of level 2's
    // M = L[32:64, 0:32] T[0:32, 0:32] that need only D_0 and D_1, i.e.
    // M[:, 0:16] = L[32:64, 0:16] D_0 and M[:, 16:32] = L[32:64, 16:32] D_1
    // (T[0:16, 16:32] is zero), into the unused upper-right block of Tb (rows
    // 0..31, columns 32..63).  2 rows x 4 columns per thread.
    named_sync(5, 192);
    const int tt = t - 128, rp = tt >> 3, cq = tt & 7, kb = cq >= 4 ? 16 : 0;
    float2 acc[2][2] = {};
#pragma unroll 1  // kept rolled: less code for the instruction cache
    for (int k4 = 0; k4 < 16; k4 += 4) {
      float lv[2][4];
#pragma unroll
      for (int r = 0; r < 2; ++r)
        *reinterpret_cast<float4*>(lv[r]) =
            *reinterpret_cast<const float4*>(Lb + (32 + 2 * rp + r) * kLdL + kb + k4);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const float4 tv = *reinterpret_cast<const float4*>(Tb + (kb + k4 + kk) * kLdT + 4 * cq);
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          acc[r][0] = __ffma2_rn(s2(lv[r][kk]), lo2(tv), acc[r][0]);
          acc[r][1] = __ffma2_rn(s2(lv[r][kk]), hi2(tv), acc[r][1]);
        }
      }
    }
#pragma unroll
    for (int r = 0; r < 2; ++r)
      *reinterpret_cast<float4*>(Tb + 32 + (2 * rp + r) * kLdT + 4 * cq) =
          make_float4(acc[r][0].x, acc[r][0].y, acc[r][1].x, acc[r][1].y);
  }
  before_level2();
  if (t < kInvThreads) {
    // level 2 on warps 0-7 (barrier 2, 256 threads): M[:, 0:16] += L[32:64, 16:32]
    // T_{1,0} (one row x 2 columns per thread), then T[32:64, 0:32] = -T22 M.
    named_sync(2, kInvThreads);
    // rows 0..31 and T[32:64, 32:64] are final: their chunks of M
    store_m_chunk(Tb, beta_s, mt, t >> 6, t & 63);
    if ((t & 63) >= 32) store_m_chunk(Tb, beta_s, mt, 4 + (t >> 6), t & 63);
    float* Mb = Tb + 32;
    {
      const int r = t >> 3, cp = t & 7;
      float2 a01 = make_float2(0.f, 0.f);
#pragma unroll
      for (int k4 = 16; k4 < 32; k4 += 4) {
        const float4 l4 = *reinterpret_cast<const float4*>(Lb + (32 + r) * kLdL + k4);
        const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const float2 tv = *reinterpret_cast<const float2*>(Tb + (k4 + kk) * kLdT + 2 * cp);
          a01 = __ffma2_rn(s2(lv[kk]), tv, a01);
        }
      }
      float2* mp = reinterpret_cast<float2*>(Mb + r * kLdT + 2 * cp);
      *mp = __fadd2_rn(*mp, a01);
    }
    const int rp = t >> 4, cq = t & 15;
    named_sync(2, kInvThreads);
    {  // T[32:64, 0:32] = -T[32:64, 32:64] M; T[32:48, 48:64] is zero
      const int kn = rp < 8 ? 16 : 32;  // warp-uniform: warps 0-3 hold rows 32..47
      float2 acc[2] = {};
#pragma unroll 1  // kept rolled: less code for the instruction cache
      for (int k4 = 0; k4 < 32; k4 += 4) {
        if (k4 < kn) {
          float wv[2][4];
#pragma unroll
          for (int r = 0; r < 2; ++r)
            *reinterpret_cast<float4*>(wv[r]) =
                *reinterpret_cast<const float4*>(Tb + (32 + 2 * rp + r) * kLdT + 32 + k4);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const float2 mv = *reinterpret_cast<const float2*>(Mb + (k4 + kk) * kLdT + 2 * cq);
#pragma unroll
            for (int r = 0; r < 2; ++r) acc[r] = __ffma2_rn(s2(wv[r][kk]), mv, acc[r]);
          }
        }
      }
#pragma unroll
      for (int r = 0; r < 2; ++r)
        *reinterpret_cast<float2*>(Tb + (32 + 2 * rp + r) * kLdT + 2 * cq) =
            make_float2(-acc[r].x, -acc[r].y);
    }
    // rows 32 + 8 o .. + 7 of T[32:64, 0:32] come from threads 64 o .. 64 o + 63
    named_sync(6 + (t >> 6), 64);
    if ((t & 63) < 32) store_m_chunk(Tb, beta_s, mt, 4 + (t >> 6), t & 31);
  }
}

// tc_prep: two 256-thread CTAs share an SM (111 KB of shared memory, 256 TMEM
// columns and at most 128 registers a thread each).  A CTA takes its units one
// after the other; the two CTAs of an SM overlap each other's phases (one's
// latency-bound inverse under the other's issue-bound operand pass, its products
// under the other's copies).
//
// Thread t -> channel pair (cp, cp + 1), cp = 2 (t & 63), and 16-token tile
// ta = t >> 6, for the whole operand side: the thread reads its 16 rows of k, q
// and g (or z) from the staged copy into registers, sums the decays in registers
// and builds the operands of its 16 rows x 2 channels.  Only the per-tile totals of
// g cross threads.  Every shared-memory block serves several phases of a unit:
//   row operand (32 KB): K/Q rows for the products; then Gamma*Q and Kt^T on
//     their way out (parked in TMEM meanwhile); then V (tensor copy, once the
//     Gamma*Q copy has read its space), T Diag(beta) and the next unit's z rows
//     0-31 (copied in between the inverse's levels, once the Kt^T copy has read
//     its space); then the next unit's g (fp32), or U^T on its way out (gate fused)
//   key operand (48 KB): KC for the products; then the inverse's scratch; then the
//     next unit's k and q (copied in once T is read), or U^T on its way out (g read)
//   (Gamma K)^T (16 KB): the W product's A operand; then W on its way out
//   A_qk (8 KB) on its way out; then the next unit's z rows 32-63
constexpr int kP2Threads = 256;
constexpr uint32_t kQ_Bop = 0;              // MN-major X=128 (K/Q rows), K=128
constexpr uint32_t kQ_V = kQ_Bop;           //   V: two 64-channel SW128 boxes
constexpr uint32_t kQ_T = kQ_Bop + 16384;   //   bf16 T Diag(beta), MN-major 64x64
constexpr uint32_t kQ_Zlo = kQ_Bop + 24576;  //   the next unit's z rows 0-31 (bf16)
constexpr uint32_t kQ_Gin = kQ_Bop;         //   the next unit's g, fp32 [64][128]
constexpr uint32_t kQ_KC = 32768;           // MN-major X=192, K=128
constexpr uint32_t kQ_Tb = kQ_KC;           //   the inverse's scratch: T, the block
constexpr uint32_t kQ_Ps = kQ_Tb + 17408;   //   products, and L at the end (dead one
constexpr uint32_t kQ_Lb = kQ_KC + 49152 - 17408;  //   phase before T)
constexpr uint32_t kQ_Kin = kQ_KC;          //   the next unit's k, q (bf16 [64][128])
constexpr uint32_t kQ_Qin = kQ_KC + 16384;
constexpr uint32_t kQ_Ug = kQ_KC + 32768;   //   U^T on its way out (g read)
constexpr uint32_t kQ_BKg = 81920;          // K-major (Gamma K)^T 128 x 64
constexpr uint32_t kQ_AQ = 98304;           // K-major A_qk 64 x 64
constexpr uint32_t kQ_Zhi = kQ_AQ;          //   the next unit's z rows 32-63 (bf16)
constexpr uint32_t kQ_Tot = kQ_AQ + 8192;   // per-tile sums of g, fp32 [4][128]
constexpr uint32_t kQ_beta = kQ_Tot + 2048;  // fp32 [64]
constexpr uint32_t kQ_Gsc = kQ_beta + 256;   // scalar gates, fp32 [64]
constexpr uint32_t kQ_Red = kQ_Gsc + 256;    // row sums of squares, fp32 [8 warps][32]
constexpr uint32_t kQ_bars = kQ_Red + 1024;  // five mbarriers + the TMEM base
constexpr uint32_t kQ_Smem = kQ_bars + 64 + 1024;  // + slack for the 1024-byte alignment
static_assert(kQ_Ps + 3072 <= kQ_Lb && kQ_Lb + 17408 == kQ_BKg, "the inverse scratch fits the KC space");
static_assert(kQ_Qin + 16384 <= kQ_Lb + 1024 && kQ_T + 8192 <= kQ_Zlo, "k, q land in T's space, z past T");
static_assert(2 * (kQ_Smem + 1024) <= 233472, "two CTAs per SM");
template <bool kZ>
__host__ __device__ constexpr uint32_t q_ustage() { return kZ ? kQ_Bop : kQ_Ug; }

// kZ: tm_g maps z (bf16) instead of g, and g = g_min * Sigmoid(exp(A_h) z) is formed
// while the decays are summed ("Kimi K3 technical report review", section 3.2).
// kP: the precise-state mode, Kt^T written in fp32 (straight to the workspace).
// tm_g maps g (fp32) otherwise; g_sc: one gate per token and head (fp32 [NT][H])
// instead, or null.  kN: q and k are L2-normalised per token and head here (with
// qk_eps), a template argument so that the other instances carry none of its code.
template <bool kZ, bool kP, bool kN>
__global__ void __launch_bounds__(kP2Threads, 2)
    tc_prep(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
             const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
             const __nv_bfloat16* __restrict__ beta, const float* __restrict__ A, float g_min,
             Plan plan, int H, int64_t units_ub, uint8_t* __restrict__ tiles,
             float* __restrict__ gam_out, float qk_eps, const float* __restrict__ g_sc_arg,
             int* err) {
  // scalar gates exist only without the fused gate: a constant null otherwise, so
  // that the gated instances carry none of their code
  const float* __restrict__ const g_sc = kZ ? nullptr : g_sc_arg;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_addr(sm);
  float* Tot = reinterpret_cast<float*>(sm + kQ_Tot);
  float* beta_s = reinterpret_cast<float*>(sm + kQ_beta);
  float* gsc_s = reinterpret_cast<float*>(sm + kQ_Gsc);
  float* red = reinterpret_cast<float*>(sm + kQ_Red);
  float* Lb = reinterpret_cast<float*>(sm + kQ_Lb);
  float* Tb = reinterpret_cast<float*>(sm + kQ_Tb);
  float* Ps = reinterpret_cast<float*>(sm + kQ_Ps);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kQ_bars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kQ_bars + 48);
  const uint32_t bar_p = smem_addr(&bars[0]), bar_v = smem_addr(&bars[1]);
  const uint32_t bar_w = smem_addr(&bars[2]), bar_kq = smem_addr(&bars[3]);
  const uint32_t bar_g = smem_addr(&bars[4]);  // the next unit's z or g
  const int t = threadIdx.x, warp = t >> 5, lane32 = t & 31;
  const bool g_fp32 = !kZ && g_sc == nullptr;  // g arrives by its own copy

  if (t == 0) {
    mbar_init(bar_p, 1);
    mbar_init(bar_v, 1);
    mbar_init(bar_w, 1);
    mbar_init(bar_kq, 1);
    mbar_init(bar_g, 1);
    mbar_fence_init();
  }
  if (warp == 0) tmem_alloc(smem_addr(tmem_slot), 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int total = __ldg(plan.chunk_off + plan.n_seqs);
  const float gmin2 = g_min * kLog2e;
  constexpr bool qk_norm = kN;

  const int pr = t & 63, ta = t >> 6, cp = 2 * pr, sw = (pr >> 2) & 1;
  const uint32_t lane_addr = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
  // Gamma*Q and Kt^T of the thread's 16 rows x 2 channels wait in TMEM columns
  // 160..223 (idle during the products) until the products have freed the row
  // operand, which then stages them for one bulk copy: TMEM lane 64 (ta & 1) + pr
  // (the thread's own warp's lane quarter), 32 columns per pair of tiles,
  // Gamma*Q in the first 16 and Kt^T in the next 16, 4 per (channel visit, half)
  const uint32_t t_park = lane_addr + 160u + 32u * (uint32_t)(ta >> 1);
  constexpr int kCopier = 224;  // warp 7 lane 0: copies out Gamma*Q, Kt^T and A_qk, then V in

  // (chunk, head) of the current and the next two units, stepped by the grid
  // without dividing; table entries are loaded two units ahead, beta and the
  // scalar gates one unit ahead
  const int grid_q = (int)(gridDim.x / H), grid_r = (int)(gridDim.x % H);
  const int64_t chunks_ub = units_ub / H;
  auto step = [&](int64_t& ch, int& hh) {
    ch += grid_q;
    hh += grid_r;
    if (hh >= H) {
      hh -= H;
      ++ch;
    }
  };
  int64_t cur_chunk = blockIdx.x / H, nx_chunk = cur_chunk;
  int cur_h = (int)(blockIdx.x % H), nx_h = cur_h;
  step(nx_chunk, nx_h);
  int2 cur_e = cur_chunk < chunks_ub ? __ldg(plan.tab + cur_chunk) : make_int2(0, 0);
  float cur_a = (kZ && cur_chunk < chunks_ub) ? __ldg(A + cur_h) : 0.f;
  int2 nx_e = nx_chunk < chunks_ub ? __ldg(plan.tab + nx_chunk) : make_int2(0, 0);
  float nx_a = (kZ && nx_chunk < chunks_ub) ? __ldg(A + nx_h) : 0.f;
  // outstanding asynchronous work of the issuing thread (thread 0; kCopier for V
  // and z): the phase it completes, or -1; drained before the CTA exits
  int pend_p = -1, pend_v = -1, pend_w = -1, pend_kq = -1, pend_g = -1;
  auto issue_kq = [&](int hh, int tt0, int ph) {  // k, q into the key-operand space
    mbar_arrive_expect_tx(bar_kq, 32768u);
    tma_load_3d(sbase + kQ_Kin, &tm_k, 0, hh, tt0, bar_kq);
    tma_load_3d(sbase + kQ_Qin, &tm_q, 0, hh, tt0, bar_kq);
    pend_kq = ph;
  };
  // z (bf16, two 32-token boxes) or g (fp32) into the row-operand space
  auto issue_g = [&](int hh, int tt0, int ph) {
    mbar_arrive_expect_tx(bar_g, kZ ? 16384u : 32768u);
    if (kZ) {
      tma_load_3d(sbase + kQ_Zlo, &tm_g, 0, hh, tt0, bar_g);
      tma_load_3d(sbase + kQ_Zhi, &tm_g, 0, hh, tt0 + 32, bar_g);
    } else {
      tma_load_3d(sbase + kQ_Gin, &tm_g, 0, hh, tt0, bar_g);
    }
    pend_g = ph;
  };
  // threads 0..63: beta (bf16 bits) and the scalar gate of token t of this and the
  // next unit
  uint32_t b_cur = 0u, b_nx = 0u;
  float gs_nx = 0.f;
  {
    const bool valid = cur_chunk < chunks_ub && cur_chunk < total;
    if (t == 0 && valid) {
      issue_kq(cur_h, cur_e.x, 0);
      if (kZ || g_fp32) issue_g(cur_h, cur_e.x, 0);
    }
    if (t < 64) {
      const bool in = valid && t < cur_e.y;
      if (in) b_cur = __ldg(reinterpret_cast<const unsigned short*>(beta) + ((size_t)cur_e.x + t) * H + cur_h);
      if (g_sc) gsc_s[t] = in ? __ldg(g_sc + ((size_t)cur_e.x + t) * H + cur_h) : 0.f;
    }
    __syncthreads();
  }
  bool ok = true;
  uint32_t it = 0;
  for (int64_t u = blockIdx.x; u < units_ub; u += gridDim.x, ++it) {
    const int h = cur_h;
    if (cur_chunk >= total) break;
    const int64_t t0 = cur_e.x;
    const int len = cur_e.y;
    const float ea = kZ ? expf(cur_a) * kLog2e : 0.f;
    uint8_t* unit = tiles + (size_t)u * unit_bytes<kP>();
    // the unit after next: its entry is loaded now and used a unit from now
    int64_t n2_chunk = nx_chunk;
    int n2_h = nx_h;
    step(n2_chunk, n2_h);
    // (predicated loads, no select on their results: nothing waits for them here)
    int2 n2_e = make_int2(0, 0);
    float n2_a = 0.f;
    if (n2_chunk < chunks_ub) {
      n2_e = __ldg(plan.tab + n2_chunk);
      if (kZ) n2_a = __ldg(A + n2_h);
    }
    const bool nx_valid = nx_chunk < chunks_ub && nx_chunk < total;
    if (t < 64) {
      beta_s[t] = bf16_lo(b_cur);
      b_nx = 0u;
      gs_nx = 0.f;
      if (nx_valid && t < nx_e.y) {
        b_nx = __ldg(reinterpret_cast<const unsigned short*>(beta) + ((size_t)nx_e.x + t) * H + nx_h);
        if (g_sc) gs_nx = __ldg(g_sc + ((size_t)nx_e.x + t) * H + nx_h);
      }
    }

    // ---- this unit's rows, copied in during the previous unit: 16 rows x 2 channels;
    //      z / g first (pass 1 reads them), k and q meanwhile
    bool okin = (!kZ && !g_fp32) || mbar_wait(bar_g, it & 1, err);
    uint32_t kw[16], qw[16];
    float Gl[2][16];
    {
      float s0 = 0.f, s1 = 0.f;
      // ---- pass 1: the gate (kZ) and the running log-decay over the thread's tile,
      //      base 2, tile-relative: Gl[c][e] = G_r - R_a for row r = 16 ta + e
#pragma unroll
      for (int e = 0; e < 16; e += 2) {
        const int r = 16 * ta + e;
        float gv[4];  // rows r, r + 1 x channels cp, cp + 1
        if constexpr (kZ) {
          // g = g_min / d with d = 1 + exp(-exp(A_h) z); the four quotients share one
          // reciprocal, the exponent clamped at 30 (see the key-operand layout above)
          const uint8_t* zrow = sm + (ta < 2 ? kQ_Zlo : kQ_Zhi) + (r & 31) * 256 + cp * 2;
          const uint32_t z0 = *reinterpret_cast<const uint32_t*>(zrow);
          const uint32_t z1 = *reinterpret_cast<const uint32_t*>(zrow + 256);
          const float d0 = 1.f + exp2_approx(fminf(-ea * bf16_lo(z0), 30.f));
          const float d1 = 1.f + exp2_approx(fminf(-ea * bf16_hi(z0), 30.f));
          const float d2 = 1.f + exp2_approx(fminf(-ea * bf16_lo(z1), 30.f));
          const float d3 = 1.f + exp2_approx(fminf(-ea * bf16_hi(z1), 30.f));
          const float d01 = d0 * d1, d23 = d2 * d3;
          const float rall = rcp_approx(d01 * d23);
          const float q01 = gmin2 * d23 * rall, q23 = gmin2 * d01 * rall;
          gv[0] = d1 * q01;
          gv[1] = d0 * q01;
          gv[2] = d3 * q23;
          gv[3] = d2 * q23;
        } else if (g_sc) {
          gv[0] = gv[1] = gsc_s[r] * kLog2e;
          gv[2] = gv[3] = gsc_s[r + 1] * kLog2e;
        } else {
          const float2 a = *reinterpret_cast<const float2*>(sm + kQ_Gin + r * 512 + cp * 4);
          const float2 b = *reinterpret_cast<const float2*>(sm + kQ_Gin + (r + 1) * 512 + cp * 4);
          gv[0] = a.x * kLog2e;
          gv[1] = a.y * kLog2e;
          gv[2] = b.x * kLog2e;
          gv[3] = b.y * kLog2e;
        }
        if (r >= len) gv[0] = gv[1] = 0.f;  // rows past the sequence end
        if (r + 1 >= len) gv[2] = gv[3] = 0.f;
        s0 += gv[0];
        s1 += gv[1];
        Gl[0][e] = s0;
        Gl[1][e] = s1;
        s0 += gv[2];
        s1 += gv[3];
        Gl[0][e + 1] = s0;
        Gl[1][e + 1] = s1;
      }
      *reinterpret_cast<float2*>(Tot + ta * D + cp) = make_float2(s0, s1);
    }
    okin = mbar_wait(bar_kq, it & 1, err) && okin;
    if (okin) pend_kq = pend_g = -1;  // (the issuing threads' records)
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const int r = 16 * ta + e;
      const bool in = r < len;
      kw[e] = in ? *reinterpret_cast<const uint32_t*>(sm + kQ_Kin + r * 256 + cp * 2) : 0u;
      qw[e] = in ? *reinterpret_cast<const uint32_t*>(sm + kQ_Qin + r * 256 + cp * 2) : 0u;
    }
    if (qk_norm) {
      // |k_r|^2 and |q_r|^2 over this warp's 64 channels, each by a reduce-scatter
      // over 16 lanes and one exchange: lane i ends with row i & 15 summed over the
      // warp (k for lanes 0-15, q for lanes 16-31)
      float sk = 0.f, sq = 0.f;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        float v[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const uint32_t x = which ? qw[e] : kw[e];
          v[e] = fmaf(bf16_lo(x), bf16_lo(x), bf16_hi(x) * bf16_hi(x));
        }
#pragma unroll
        for (int w = 8; w >= 1; w >>= 1) {
          const bool up = (lane32 & w) != 0;
#pragma unroll
          for (int i = 0; i < w; ++i) {
            const float send = up ? v[i] : v[i + w];
            const float keep = up ? v[i + w] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
          }
        }
        v[0] += __shfl_xor_sync(0xffffffffu, v[0], 16);
        if (which) sq = v[0]; else sk = v[0];
      }
      red[warp * 32 + lane32] = lane32 < 16 ? sk : sq;
    }
    // the previous unit's outgoing copies have read their staging space (the blocks
    // the operand pass below rewrites)
    if (lane32 == 0) bulk_wait_read_all();
    // the previous unit's W/U wait, this unit's copies, every thread's tile totals
    if (!__syncthreads_and(ok && okin)) break;
    if (qk_norm) {
      // normalised rows, rounded to bf16 like normalised inputs.  Lane i forms
      // 1 / sqrt(|x|^2 + eps) of row i & 15 of the tile (k rows for lanes 0-15, q
      // rows for 16-31) from the two warps' halves of the channels; every thread
      // takes its rows' factors from those lanes.
      const float rn = rsqrtf(red[64 * ta + lane32] + red[64 * ta + 32 + lane32] + qk_eps);
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float rk = __shfl_sync(0xffffffffu, rn, e);
        const float rq = __shfl_sync(0xffffffffu, rn, 16 + e);
        const bool in = 16 * ta + e < len;
        kw[e] = in ? pack_bf16(bf16_lo(kw[e]) * rk, bf16_hi(kw[e]) * rk) : 0u;
        qw[e] = in ? pack_bf16(bf16_lo(qw[e]) * rq, bf16_hi(qw[e]) * rq) : 0u;
      }
    }

    // ---- operands of the thread's 16 rows, one channel at a time (the order sw
    //      makes each warp's 16-byte stores cover all eight swizzle positions)
    if (sw) {
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        kw[e] = __byte_perm(kw[e], 0u, 0x1032);
        qw[e] = __byte_perm(qw[e], 0u, 0x1032);
        const float tmp = Gl[0][e];
        Gl[0][e] = Gl[1][e];
        Gl[1][e] = tmp;
      }
    }
#pragma unroll
    for (int o2 = 0; o2 < 2; ++o2) {
      const int c = cp + (o2 ^ sw);
      float R[4], GC = 0.f;  // R_b = sum of the tile sums before tile b; G_C = all
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        R[b] = GC;
        GC += Tot[b * D + c];
      }
      const float Ra = ta == 0 ? R[0] : (ta == 1 ? R[1] : (ta == 2 ? R[2] : R[3]));
      const float eRa = exp2_approx(Ra);       // exp(R_a) <= 1
      const float eCa = exp2_approx(GC - Ra);  // exp(G_C - R_a) <= 1
#pragma unroll
      for (int hq = 0; hq < 2; ++hq) {
        // rows 8 hq + 2 i, 8 hq + 2 i + 1 of the tile in lanes x, y
        float2 f[4], fi[4], kv[4], x[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float d0 = Gl[o2][8 * hq + 2 * i], d1 = Gl[o2][8 * hq + 2 * i + 1];  // G_r - R_a, in (-80, 0]
          f[i] = make_float2(exp2_approx(d0), exp2_approx(d1));
          fi[i] = make_float2(exp2_approx(-d0), exp2_approx(-d1));
          const uint32_t k0 = kw[8 * hq + 2 * i], k1 = kw[8 * hq + 2 * i + 1];
          kv[i] = o2 ? make_float2(bf16_hi(k0), bf16_hi(k1)) : make_float2(bf16_lo(k0), bf16_lo(k1));
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) x[i] = __fmul2_rn(kv[i], f[i]);  // k exp(G_r - R_a)
        *reinterpret_cast<uint4*>(sm + kQ_Bop + mn_chunk(128, 4 * ta + hq, c)) = pack8(x);
#pragma unroll
        for (int i = 0; i < 4; ++i) x[i] = __fmul2_rn(x[i], s2(eRa));  // Gamma k (beta is folded into T)
        *reinterpret_cast<uint4*>(sm + kQ_BKg + sw128_chunk(128, c, 2 * ta + hq)) = pack8(x);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t q0 = qw[8 * hq + 2 * i], q1 = qw[8 * hq + 2 * i + 1];
          x[i] = __fmul2_rn(o2 ? make_float2(bf16_hi(q0), bf16_hi(q1)) : make_float2(bf16_lo(q0), bf16_lo(q1)),
                            f[i]);
        }
        *reinterpret_cast<uint4*>(sm + kQ_Bop + mn_chunk(128, 4 * ta + 2 + hq, c)) = pack8(x);
#pragma unroll
        for (int i = 0; i < 4; ++i) x[i] = __fmul2_rn(x[i], s2(eRa));  // Gamma q
        tmem_st4(t_park + 4 * (2 * o2 + hq), pack8(x));
#pragma unroll
        for (int i = 0; i < 4; ++i) kv[i] = __fmul2_rn(kv[i], fi[i]);  // k exp(R_a - G_r)
#pragma unroll
        for (int i = 0; i < 4; ++i) x[i] = __fmul2_rn(kv[i], s2(eCa));  // (gamma_C / Gamma) k
        if (kP) {  // fp32, tokens 8 hq .. +3 and +4 .. +7 of the tile
          *reinterpret_cast<float4*>(unit + kKT + kt32_chunk(c, 4 * ta + 2 * hq)) =
              make_float4(x[0].x, x[0].y, x[1].x, x[1].y);
          *reinterpret_cast<float4*>(unit + kKT + kt32_chunk(c, 4 * ta + 2 * hq + 1)) =
              make_float4(x[2].x, x[2].y, x[3].x, x[3].y);
        } else {
          tmem_st4(t_park + 16 + 4 * (2 * o2 + hq), pack8(x));
        }
#pragma unroll
        for (int ap = 0; ap < 4; ++ap) {
          if (ap < ta) continue;
          const float E = (ap > ta) ? exp2_approx(R[ap] - Ra) : 1.f;  // exp(R_ap - R_a) <= 1
#pragma unroll
          for (int i = 0; i < 4; ++i) x[i] = __fmul2_rn(kv[i], s2(E));
          *reinterpret_cast<uint4*>(sm + kQ_KC + mn_chunk(kKCX, ap * (ap + 1) + 2 * ta + hq, c)) =
              pack8(x);
        }
      }
      if (ta == 0) gam_out[(size_t)u * D + c] = exp2_approx(GC);
    }
    tmem_wait_st();

    // ---- block products in one N=160 MMA chain (see the key-operand layout above)
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (t == 0) {
      tc_fence_after();
      const uint32_t id = idesc_bf16_mn(128, 160, 1, 1);
      const uint64_t da = mnmajor_desc(sbase + kQ_Bop, 2048, 0);
      const uint64_t db = mnmajor_desc(sbase + kQ_KC, mn_sbo(kKCX), 0);
#pragma unroll
      for (int s = 0; s < D / 16; ++s)
        mma_bf16(tmem + 0, desc_advance(da, s * 2 * 2048), desc_advance(db, s * 2 * mn_sbo(kKCX)),
                 id, s > 0);
      mma_commit(bar_p);
      pend_p = (int)(it & 1);
    }
    if (t == 32 && nx_valid) {
      // the next unit's k, q and z / g into L2 (its v is copied in late enough in
      // its unit not to need it: prefetching it as well measured slower)
      tma_prefetch_l2_3d(&tm_k, 0, nx_h, nx_e.x);
      tma_prefetch_l2_3d(&tm_q, 0, nx_h, nx_e.x);
      if (!g_sc) tma_prefetch_l2_3d(&tm_g, 0, nx_h, nx_e.x);
      if (kZ) tma_prefetch_l2_3d(&tm_g, 0, nx_h, nx_e.x + 32);
    }
    const bool okp = mbar_wait(bar_p, it & 1, err);
    if (t == 0 && okp) pend_p = -1;
    tc_fence_after();
    {  // the parked Gamma*Q and Kt^T -> the row operand's space (dead now), MMA-ready
      float pk[32];
      tmem_ld32(t_park, pk);
      tmem_wait_ld();
#pragma unroll
      for (int o2 = 0; o2 < 2; ++o2) {
        const int c = cp + (o2 ^ sw);
#pragma unroll
        for (int hq = 0; hq < 2; ++hq) {
          const int j = 4 * (2 * o2 + hq);
          *reinterpret_cast<uint4*>(sm + kQ_Bop + mn_chunk(64, 2 * ta + hq, c)) =
              make_uint4(__float_as_uint(pk[j]), __float_as_uint(pk[j + 1]),
                         __float_as_uint(pk[j + 2]), __float_as_uint(pk[j + 3]));
          if (!kP)
            *reinterpret_cast<uint4*>(sm + kQ_Bop + 16384 + sw128_chunk(128, c, 2 * ta + hq)) =
                make_uint4(__float_as_uint(pk[16 + j]), __float_as_uint(pk[17 + j]),
                           __float_as_uint(pk[18 + j]), __float_as_uint(pk[19 + j]));
        }
      }
    }
    {
      // read-out: warp -> tile tw (its TMEM lane quarter) and key pieces pc of 16
      // keys; lane -> row r = 16 tw + (lane & 15), a K row or (lane & 16) a Q row
      const int tw = warp & 3, r = 16 * tw + (t & 15);
      const bool qrow = (t & 16) != 0;
#pragma unroll
      for (int pp = 0; pp < 2; ++pp) {
        const int pc = 2 * (warp >> 2) + pp;
        float pv[16];
        if (pc <= tw) {
          tmem_ld16(lane_addr + 8 * tw * (tw + 1) + 16 * pc, pv);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) pv[jj] = 0.f;
        }
        if (!qrow) {
          if (pc <= tw) {
            const float br = beta_s[r];
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) pv[jj] = (16 * pc + jj < r) ? br * pv[jj] : 0.f;
#pragma unroll
            for (int q = 0; q < 4; ++q)
              *reinterpret_cast<float4*>(Lb + r * kLdL + 16 * pc + 4 * q) =
                  make_float4(pv[4 * q], pv[4 * q + 1], pv[4 * q + 2], pv[4 * q + 3]);
          }
        } else {
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) pv[jj] = (16 * pc + jj <= r) ? pv[jj] : 0.f;
          *reinterpret_cast<uint4*>(sm + kQ_AQ + sw128_chunk(64, r, 2 * pc)) = pack8(pv);
          *reinterpret_cast<uint4*>(sm + kQ_AQ + sw128_chunk(64, r, 2 * pc + 1)) = pack8(pv + 8);
        }
      }
    }
    fence_proxy_async_smem();  // Gamma*Q, Kt^T and A_qk leave by bulk copies
    tc_fence_before();
    if (!__syncthreads_and(okp)) {
      ok = false;
      break;
    }
    if (t == kCopier) {
      bulk_s2g(unit + kQ, sbase + kQ_Bop, 16384);
      bulk_commit();  // Gamma*Q: its space is V's
      if (!kP) bulk_s2g(unit + kKT, sbase + kQ_Bop + 16384, 16384);
      bulk_s2g(unit + kAQ, sbase + kQ_AQ, 8192);
      bulk_commit();  // Kt^T and A_qk: their space is the next unit's z
      // V lands in the row operand's space once the Gamma*Q copy has read it (while
      // warps 0-3 run the first level of the inverse)
      bulk_wait_read_all_but_last();
      mbar_arrive_expect_tx(bar_v, 16384);
      tma_load_3d(sbase + kQ_V, &tm_v, 0, h, (int)t0, bar_v);
      tma_load_3d(sbase + kQ_V + 8192, &tm_v, 64, h, (int)t0, bar_v);
      pend_v = (int)(it & 1);
    }
    invert_unit_lower(Lb, Tb, Ps, beta_s, sm + kQ_T, t, [&] {
      if (kZ && t == kCopier) {
        // Kt^T and A_qk have left by now: the next unit's z lands in the row
        // operand's tail and the A_qk block
        bulk_wait_read_all();
        if (nx_valid) issue_g(nx_h, nx_e.x, (int)((it + 1) & 1));
      }
    });
    if (g_sc && t < 64) gsc_s[t] = gs_nx;  // the next unit's pass 1 reads them
    fence_proxy_async_smem();
    tc_fence_before();
    bool okv = true;
    if (t == kCopier) {
      okv = mbar_wait(bar_v, it & 1, err);
      if (okv) pend_v = -1;
    }
    if (!__syncthreads_and(okv)) {
      ok = false;
      break;
    }
    if (t == 0) {
      tc_fence_after();
      const uint32_t id = idesc_bf16_mn(128, 64, 0, 1);
      const uint32_t idv = idesc_bf16_mn(128, 64, 1, 1);  // A = V^T read MN-major
      const uint64_t dk = kmajor_desc(sbase + kQ_BKg, 128, 0);
      const uint64_t dv = mnmajor_desc_lbo(sbase + kQ_V, 8192, 1024, 0);
      const uint64_t dt = mnmajor_desc(sbase + kQ_T, 1024, 0);
#pragma unroll
      for (int s = 0; s < C / 16; ++s)  // W^T = (Gamma K)^T M^T
        mma_bf16(tmem + 0, desc_advance(dk, s * 32), desc_advance(dt, s * 2048), id, s > 0);
#pragma unroll
      for (int s = 0; s < C / 16; ++s)  // U^T = V^T M^T
        mma_bf16(tmem + 64, desc_advance(dv, s * 2048), desc_advance(dt, s * 2048), idv, s > 0);
      mma_commit(bar_w);
      pend_w = (int)(it & 1);
      // T is read: the next unit's k and q land in its space
      if (nx_valid) issue_kq(nx_h, nx_e.x, (int)((it + 1) & 1));
    }
    ok = mbar_wait(bar_w, it & 1, err);
    if (t == 0 && ok) {
      pend_w = -1;
      // the W/U products have read V and T: the next unit's g lands in their space
      if (g_fp32 && nx_valid) issue_g(nx_h, nx_e.x, (int)((it + 1) & 1));
    }
    tc_fence_after();
    {  // W (MN-major, warps 0-3) and U^T (K-major, warps 4-7), row = TMEM lane: each
       // warp's 32 rows are 4 KB of the tile, staged and sent by one bulk copy
      const int row = 32 * (warp & 3) + lane32;
      const uint32_t stage = warp < 4 ? kQ_BKg : q_ustage<kZ>();
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        float w[32];
        tmem_ld32(lane_addr + 64 * (warp >> 2) + 32 * part, w);
        tmem_wait_ld();
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          const int xc = 4 * part + ch;
          const uint32_t off = warp < 4 ? mn_chunk(64, xc, row) : sw128_chunk(128, row, xc);
          *reinterpret_cast<uint4*>(sm + stage + off) = pack8(&w[8 * ch]);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane32 == 0) {
        const uint32_t piece = 4096u * (uint32_t)(warp & 3);
        bulk_s2g(unit + (warp < 4 ? kW : kUT) + piece, sbase + stage + piece, 4096);
        bulk_commit();
      }
    }
    tc_fence_before();
    cur_chunk = nx_chunk;
    cur_h = nx_h;
    cur_e = nx_e;
    cur_a = nx_a;
    nx_chunk = n2_chunk;
    nx_h = n2_h;
    nx_e = n2_e;
    nx_a = n2_a;
    b_cur = b_nx;
  }
  // after an abort: let the copies and products in flight finish before the TMEM
  // and the shared memory go away (each issuing thread waits for its own)
  if (pend_p >= 0) mbar_wait(bar_p, (uint32_t)pend_p, err);
  if (pend_v >= 0) mbar_wait(bar_v, (uint32_t)pend_v, err);
  if (pend_w >= 0) mbar_wait(bar_w, (uint32_t)pend_w, err);
  if (pend_kq >= 0) mbar_wait(bar_kq, (uint32_t)pend_kq, err);
  if (pend_g >= 0) mbar_wait(bar_g, (uint32_t)pend_g, err);
  if (lane32 == 0) bulk_wait_all();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// ============================================================= chain kernel
// Stages of the tile ring: a unit (72 KB; 88 KB with fp32 Kt^T) + gamma (512 B),
// 1024-aligned; three of them, two in the precise-state mode.
template <bool kP> __host__ __device__ constexpr int stages() { return kP ? 2 : 3; }
template <bool kP> __host__ __device__ constexpr uint32_t stage_bytes() {
  return (unit_bytes<kP>() + kGamBytes + 1023) & ~1023u;
}
template <bool kP> __host__ __device__ constexpr uint32_t chain_bars() {
  return stages<kP>() * stage_bytes<kP>();
}
// After the stages: 256 bytes of barriers and flags, then the output gate's
// per-token partial sums (fp32 [4 store warps][64]) and 1/rms (fp32 [64]).
constexpr uint32_t kC_GateScratch = 4 * 64 * 4 + 64 * 4;
template <bool kP> __host__ __device__ constexpr uint32_t chain_smem() {
  return chain_bars<kP>() + 256 + kC_GateScratch + 1024;
}
static_assert(chain_smem<false>() <= 232448 && chain_smem<true>() <= 232448, "chain smem");
// TMEM columns.  Default: S^T fp32 [0,128); two D1 buffers [128,256), [256,384)
// (each (W S)^T | (Gamma Q S)^T then O); the bf16 A operands of MMA1 (S^T, packed
// pairs, [384,448)) and MMA2 (Vt^T, two buffers of 32 columns at [448,512)).
// Precise-state mode: S^T [0,128); (W S)^T [128,192) (read by the epilogue before
// the next MMA1 is issued, so one buffer); two O buffers [192,256), [256,320); the
// bf16 S^T copy [320,384); Vt^T in fp32, the tf32 A operand of MMA2, [384,448);
// the bf16 Vt^T buffers of the O product [448,512).
template <bool kP> __device__ __forceinline__ uint32_t t_ws(int j) {
  return kP ? 128u : 128u + 128u * (uint32_t)(j & 1);
}
template <bool kP> __device__ __forceinline__ uint32_t t_o(int j) {
  return kP ? 192u + 64u * (uint32_t)(j & 1) : 192u + 128u * (uint32_t)(j & 1);
}
template <bool kP> __host__ __device__ constexpr uint32_t t_sb() { return kP ? 320u : 384u; }
constexpr uint32_t kT_VF = 384, kT_VT = 448;
constexpr int kEpi = 256;    // epilogue warps 0-7: (TMEM lane, column half)
// Store warps from warp 8 on, TMEM lane = value row: four warps over all 64 tokens
// of a chunk; with the output gate (kG) eight, warps 8-11 on tokens 0-31 and 12-15
// on tokens 32-63 (two on each SM sub-partition, for the gate's extra work).  Then
// the copy warp and the output-MMA warp.
template <bool kG> __host__ __device__ constexpr int store_threads() { return kG ? 256 : 128; }
template <bool kG> __host__ __device__ constexpr int copy_warp() {
  return (kEpi + store_threads<kG>()) / 32;
}
template <bool kG> __host__ __device__ constexpr int chain_threads() {
  return kEpi + store_threads<kG>() + 64;
}

// Sequence-segment parallel chain (the KCP algebra applied inside one GPU: "Kimi
// K3 technical report review", section 8.1 Eq. 17).  A long sequence is cut into P
// segments; with A_c = Diag(gamma_C) - Kt^T W the linear part of one chunk step,
// a segment maps its incoming state to S_end = S~ + M S_in, where S~ is the
// segment run from a zero state and M the product of its A_c.
//   mode 1 (grid z = 0): segment 0 runs from h0 with outputs (its end state is
//          exact); segments k >= 1 run from zero without outputs (S~);
//   mode 1 (grid z = 1): segments 1 .. P-2 run from the identity with U = 0 (M^T);
//   scan:  S_in(1) = S_end(0), S_in(k+1) = S~(k) + M(k) S_in(k)  (seg_scan_kernel);
//   mode 2: segments k >= 1 run from S_in(k) with outputs; the last writes hT.
// mode 0 is the plain chain, one CTA per (sequence, head).  States are S^T.
// The head-wise RMSNorm x Sigmoid output gate applied by the store warps before o
// is written ("Kimi K3 technical report review", section 3.3, Eq. 6):
//   y = Sigmoid(x) * w * o / sqrt(mean over the dv channels of o^2 + eps),
// x the gate logits [NT][H][128] bf16 (read one 64-token tile per chunk by a tensor
// copy, tm_x), w fp32 [128] (null: ones).  Used by the kG instances of tc_chain.
struct GateArgs {
  const float* w;
  float eps;
};

struct SegArgs {
  int mode;
  const int4* tab;  // per segment: (sequence, first chunk, chunks, k | P << 16); x < 0: unused
  float* s_end;     // [segments][H][128][128]
  float* m_t;
  float* s_in;
};

// kP: the precise-state mode (Kt^T fp32 in the tiles, Vt^T fp32 in TMEM, the state
// update as kind::tf32 MMAs).  kG: the output gate is applied before o is written.
// kC: state checkpoints may be requested (ck.ckpt); a template argument so that the
// other instances carry none of their code.
template <bool kP, bool kG, bool kC>
__global__ void __launch_bounds__(chain_threads<kG>(), 1)
    tc_chain(const uint8_t* __restrict__ tiles, const float* __restrict__ gam,
             const float* __restrict__ h0, Plan plan, int H, __nv_bfloat16* __restrict__ o,
             float* __restrict__ hT, SegArgs sg, CkptArgs ck, const int* __restrict__ ck_off,
             int* err, const __grid_constant__ CUtensorMap tm_x, GateArgs ga) {
  // ---- this CTA's job: chunk range, initial and final state, outputs or not
  const int h = blockIdx.y;
  int n, c0, nch;
  int64_t tstart;
  const float* init = nullptr;  // initial S^T (null: zero, unless `ident`)
  bool ident = false, use_u = true, write_o = true;
  float* fin = nullptr;         // final S^T goes here (null: nowhere)
  if (sg.mode == 0) {
    n = blockIdx.x;
    c0 = __ldg(plan.chunk_off + n);
    nch = __ldg(plan.chunk_off + n + 1) - c0;
    tstart = __ldg(plan.cu + n);
    const int64_t sn = ((int64_t)n * H + h) * D * D;
    init = h0 ? h0 + sn : nullptr;
    fin = hT ? hT + sn : nullptr;
  } else {
    const int4 e = sg.tab[blockIdx.x];
    if (e.x < 0) return;  // beyond the last segment (uniform over the CTA)
    n = e.x;
    c0 = e.y;
    nch = e.z;
    const int k = e.w & 0xffff, P = e.w >> 16;
    tstart = nch > 0 ? (int64_t)__ldg(plan.tab + c0).x : (int64_t)__ldg(plan.cu + n);
    const int64_t sn = ((int64_t)n * H + h) * D * D;
    const int64_t ss = ((int64_t)blockIdx.x * H + h) * D * D;
    if (sg.mode == 1 && blockIdx.z == 0) {
      init = (k == 0 && h0) ? h0 + sn : nullptr;
      write_o = k == 0;
      fin = P == 1 ? (hT ? hT + sn : nullptr) : sg.s_end + ss;
    } else if (sg.mode == 1) {
      if (k == 0 || k == P - 1) return;
      ident = true;
      use_u = false;
      write_o = false;
      fin = sg.m_t + ss;
    } else {
      if (k == 0) return;
      init = sg.s_in + ss;
      fin = (k == P - 1 && hT) ? hT + sn : nullptr;
    }
  }
  const int64_t tend = max(tstart, (int64_t)__ldg(plan.cu + n + 1));
  const bool gate_on = kG && write_o;  // uniform over the CTA
  // state checkpoints of this job: the true state after every ck.every chunks of
  // the sequence (chunk-local index jl counts from the sequence start)
  const bool ckpt_on = kC && ck.ckpt != nullptr && write_o;
  const int jl0 = c0 - __ldg(plan.chunk_off + n);
  const int64_t slen = (int64_t)__ldg(plan.cu + n + 1) - __ldg(plan.cu + n);
  auto ckpt_row = [&](int jl_end) -> float* {  // the state after local chunk jl_end - 1
    if (!ckpt_on || jl_end <= 0 || jl_end % ck.every != 0 || (int64_t)jl_end * C > slen)
      return nullptr;
    const int64_t idx = (int64_t)__ldg(ck_off + n) + jl_end / ck.every - 1;
    if (idx >= __ldg(ck_off + n + 1) || idx >= ck.cap) return nullptr;
    return ck.ckpt + (idx * H + h) * D * D;
  };

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_addr(sm);
  constexpr int kStages = stages<kP>();
  constexpr int kStore = store_threads<kG>(), kCopyWarp = copy_warp<kG>();
  constexpr int kOutWarp = kCopyWarp + 1;
  constexpr uint32_t kStageBytes = stage_bytes<kP>(), kC_bars = chain_bars<kP>();
  constexpr uint32_t kUnitB = unit_bytes<kP>(), kT_SB = t_sb<kP>();
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kC_bars);
  // bars: 0..2 = full[stage], 3..5 = empty[stage] (every MMA of its chunk done),
  //       6 = MMA1 done, 7 = S update done, 8,9 = O of D1 buffer b final,
  //       10,11 = D1 buffer b read out, 12..14 = drain of MMA-issuing thread 0, the
  //       output warp, thread 64 (abort path), 15 = the (Gamma Q S)^T half of MMA1
  //       done (it reads the bf16 S^T copy), 16 = (W S)^T issued, 17 = S update issued,
  //       18..20 = gate-logit tile of stage s landed (output gate only)
  const uint32_t bar_full0 = smem_addr(&bars[0]), bar_empty0 = smem_addr(&bars[3]);
  const uint32_t bar_x0 = smem_addr(&bars[18]);
  const uint32_t bar_m1 = smem_addr(&bars[6]), bar_m2 = smem_addr(&bars[7]);
  const uint32_t bar_o0 = smem_addr(&bars[8]), bar_f0 = smem_addr(&bars[10]);
  const uint32_t bar_dr = smem_addr(&bars[12]), bar_q = smem_addr(&bars[15]);
  const uint32_t bar_wi = smem_addr(&bars[16]), bar_2i = smem_addr(&bars[17]);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kC_bars + 192);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kC_bars + 200);
  const int t = threadIdx.x, warp = t >> 5;

  if (t == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_full0 + 8 * s, 1);
      // one commit from each MMA-issuing thread, and with the output gate one arrival
      // from the store warps once they have read the gate logits kept in the stage
      mbar_init(bar_empty0 + 8 * s, gate_on ? 4 : 3);
      mbar_init(bar_x0 + 8 * s, 1);
    }
    mbar_init(bar_m1, 1);
    mbar_init(bar_m2, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_o0 + 8 * b, 1);
      mbar_init(bar_f0 + 8 * b, kStore);
    }
    for (int i = 0; i < 3; ++i) mbar_init(bar_dr + 8 * i, 1);
    mbar_init(bar_q, 1);
    mbar_init(bar_wi, 1);
    mbar_init(bar_2i, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 0) tmem_alloc(smem_addr(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kCopyWarp) {
    // ------------------------------------------------------ tile copies (one thread)
    // A stage is refilled once every MMA of the chunk it held has completed (its
    // empty barrier, committed after the chunk's last MMA): the refill for chunk
    // jj + kStages is what lets that stage's barriers advance again, so no wait
    // here can fall two phases behind.
    if ((t & 31) == 0) {
      auto issue = [&](int jj) {
        const int s = jj % kStages;
        const int64_t u = (int64_t)(c0 + jj) * H + h;
        const uint32_t bar = bar_full0 + 8 * s;
        mbar_arrive_expect_tx(bar, kUnitB + kGamBytes);
        bulk_g2s(sbase + s * kStageBytes, tiles + (size_t)u * kUnitB, kUnitB, bar);
        bulk_g2s(sbase + s * kStageBytes + kUnitB, gam + (size_t)u * D, kGamBytes, bar);
        // the chunk's gate logits into L2, for the copy the output warp makes later
        if (gate_on) tma_prefetch_l2_3d(&tm_x, 0, h, (int)(tstart + (int64_t)jj * C));
      };
      int issued = 0;
      for (; issued < min(kStages, nch); ++issued) issue(issued);
      for (int jj = 0; issued < nch; ++jj) {
        if (!wait_or_abort(bar_empty0 + 8 * (jj % kStages), (jj / kStages) & 1, err, abort_flag))
          break;
        issue(issued++);
      }
      if (*abort_flag) {
        // copies already issued must land before the CTA exits
        for (int jj = max(0, issued - kStages); jj < issued; ++jj)
          mbar_wait(bar_full0 + 8 * (jj % kStages), (jj / kStages) & 1, err);
      }
    }
  } else if (warp == kOutWarp) {
    // ------------------------------------------- output MMAs (one thread, off the
    // serial path): (Gamma Q S)^T once the (W S)^T half is in the tensor pipe and the
    // D1 buffer's outputs have been read (chunk j - 2); O^T += Vt^T A_qk^T once the
    // state update is in the pipe.  No epilogue warp stalls on these issues.
    if ((t & 31) == 0) {
      const uint32_t id1 = idesc_bf16_mn(128, 64, 0, 1);
      const uint32_t id2a = idesc_bf16_mn(128, 64, 0, 0);
      bool any_mma = false;
      int x_issued = 0;  // gate-logit tile copies issued
      for (int j = 0; j < nch; ++j) {
        const int s = j % kStages;
        const uint32_t sts = sbase + s * kStageBytes;
        const uint32_t dq = tmem + t_o<kP>(j);  // (Gamma Q S)^T, then O of chunk j
        if (!wait_or_abort(bar_wi, j & 1, err, abort_flag)) break;
        if (j >= 2 && !wait_or_abort(bar_f0 + 8 * (j & 1), ((j - 2) >> 1) & 1, err, abort_flag))
          break;
        tc_fence_after();
        const uint64_t bq = mnmajor_desc(sts + kQ, 1024, 0);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          mma_bf16_ta(dq, tmem + kT_SB + 8 * ks, desc_advance(bq, ks * 2048), id1, ks > 0);
        mma_commit(bar_q);
        any_mma = true;
        if (!wait_or_abort(bar_2i, j & 1, err, abort_flag)) break;
        tc_fence_after();
        const uint32_t vt = tmem + kT_VT + 32 * (j & 1);
        const uint64_t ba = kmajor_desc(sts + kAQ, 64, 0);
#pragma unroll
        for (int ks = 0; ks < C / 16; ++ks)
          mma_bf16_ta(dq, vt + 8 * ks, desc_advance(ba, ks * 32), id2a, 1u);
        mma_commit(bar_o0 + 8 * (j & 1));  // o of chunk j final
        mma_commit(bar_empty0 + 8 * s);
        if (gate_on) {
          // W is dead once the (W S)^T half of MMA1 has read it, which the epilogue
          // waited for before the state update was issued: the chunk's gate logits
          // (64 tokens x 128 bf16, 16 KB) take its place in the stage
          mbar_arrive_expect_tx(bar_x0 + 8 * s, 16384);
          tma_load_3d(sts + kW, &tm_x, 0, h, (int)(tstart + (int64_t)j * C), bar_x0 + 8 * s);
          ++x_issued;
        }
      }
      if (*abort_flag && any_mma) {  // drain MMAs in flight
        mma_commit(bar_dr + 8);
        mbar_wait(bar_dr + 8, 0, err);
      }
      if (*abort_flag) {  // gate-logit copies in flight must land before the CTA exits
        for (int jx = max(0, x_issued - kStages); jx < x_issued; ++jx)
          mbar_wait(bar_x0 + 8 * (jx % kStages), (jx / kStages) & 1, err);
      }
    }
  } else if (warp < kEpi / 32) {
    // ------------------------- epilogue warps: TMEM lane = dv, ch = column half
    const int lane = t & 127, ch = t >> 7;
    const uint32_t lrow = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    {
      float sv[32];
#pragma unroll
      for (int qq = 0; qq < 2; ++qq) {
        const int col = 64 * ch + 32 * qq;
        if (init) {
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float4 x = *reinterpret_cast<const float4*>(init + (int64_t)lane * D + col + i);
            sv[i] = x.x; sv[i + 1] = x.y; sv[i + 2] = x.z; sv[i + 3] = x.w;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) sv[i] = (ident && lane == col + i) ? 1.f : 0.f;
        }
        tmem_st32(lrow + col, sv);
      }
      tmem_wait_st();
    }
    // Threads 0 and 64 issue the serial MMAs as soon as the epilogue warps meet at
    // a named barrier (measured faster than handing them to a separate MMA warp);
    // the output MMAs, which only o needs, go to the output warp, so that no
    // epilogue warp stalls on them (an issuing thread stalls while the tensor pipe
    // drains).  Barriers that end a wait reduce the threads' results with
    // bar.red.and, so an expired wait stops every epilogue thread at the same point.
    const uint32_t id1 = idesc_bf16_mn(128, 64, 0, 1);    // S^T x W^T
    const uint32_t id2b = idesc_bf16_mn(128, 128, 0, 0);  // Vt^T x Kt^T (K-major B)
    bool any_mma = false;
    bool alive = true;
    for (int j = 0; j < nch && alive; ++j) {
      const int s = j % kStages;
      uint8_t* st = sm + s * kStageBytes;
      const uint32_t sts = sbase + s * kStageBytes;
      const float* gam_s = reinterpret_cast<const float*>(st + kUnitB);
      // E0: S^T row -> bf16 operand copy (MMA1 may start), then S^T *= gamma_C
      // S^T updated, and the bf16 copy of the previous chunk read by both MMA1 halves
      bool ok = j == 0 || (wait_or_abort(bar_m2, (j - 1) & 1, err, abort_flag) &&
                           wait_or_abort(bar_q, (j - 1) & 1, err, abort_flag));
      ok = ok && wait_or_abort(bar_full0 + 8 * s, (j / kStages) & 1, err, abort_flag);
      if (!named_sync_and(1, kEpi, ok)) { alive = false; break; }
      tc_fence_after();
      // With the gate, the kernel runs more threads and fewer registers each, so the
      // state is handled 32 columns at a time and read again for the scaling below;
      // without it the thread keeps its 64 columns in registers.
      float sv[kG ? 1 : 2][32];
      {
        float* cp = j > 0 ? ckpt_row(jl0 + j) : nullptr;
        if constexpr (!kG) {  // both halves in flight at once: one load round trip
          tmem_ld32(lrow + 64 * ch, sv[0]);
          tmem_ld32(lrow + 64 * ch + 32, sv[kG ? 0 : 1]);
          tmem_wait_ld();
        }
#pragma unroll
        for (int qq = 0; qq < 2; ++qq) {  // this thread's 64 columns of S^T, 32 at a time
          float* v = sv[kG ? 0 : qq];
          if constexpr (kG) {
            tmem_ld32(lrow + 64 * ch + 32 * qq, *reinterpret_cast<float(*)[32]>(v));
            tmem_wait_ld();
          }
          if (cp) {
#pragma unroll
            for (int i = 0; i < 32; i += 8)
              st_global_v8(cp + (int64_t)lane * D + 64 * ch + 32 * qq + i, &v[i]);
          }
          uint32_t pk[16];  // bf16 pairs
#pragma unroll
          for (int e = 0; e < 16; ++e) pk[e] = pack_bf16(v[2 * e], v[2 * e + 1]);
          tmem_st16(lrow + kT_SB + 32 * ch + 16 * qq, pk);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      named_sync(1, kEpi);
      // MMA1 in two N = 64 halves: thread 0 the (W S)^T half that the Vt pass waits
      // for, the output warp the (Gamma Q S)^T half, which only the output needs.
      // A = bf16 S^T from TMEM; the descriptor of K step ks is the step-0
      // descriptor with its start advanced.
      const uint32_t d1 = tmem + t_ws<kP>(j);
      if (t == 0) {
        tc_fence_after();
        const uint64_t bw = mnmajor_desc(sts + kW, 1024, 0);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          mma_bf16_ta(d1, tmem + kT_SB + 8 * ks, desc_advance(bw, ks * 2048), id1, ks > 0);
        mma_commit(bar_m1);
        mma_commit(bar_empty0 + 8 * s);
        tc_fence_before();
        mbar_arrive(bar_wi);  // the output warp may issue the (Gamma Q S)^T half
        any_mma = true;
      }
      // S^T *= gamma_C (with the gate read again from TMEM while MMA1 runs: MMA1
      // reads the bf16 copy); the scaled state is ordered before MMA2 by the barrier
      // after E1
#pragma unroll
      for (int qq = 0; qq < 2; ++qq) {
        float* v = sv[kG ? 0 : qq];
        if (kG) {
          tmem_ld32(lrow + 64 * ch + 32 * qq, *reinterpret_cast<float(*)[32]>(v));
          tmem_wait_ld();
        }
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          const float4 gm = *reinterpret_cast<const float4*>(gam_s + 64 * ch + 32 * qq + i);
          const float2 v01 = __fmul2_rn(make_float2(v[i], v[i + 1]), lo2(gm));
          const float2 v23 = __fmul2_rn(make_float2(v[i + 2], v[i + 3]), hi2(gm));
          v[i] = v01.x; v[i + 1] = v01.y; v[i + 2] = v23.x; v[i + 3] = v23.y;
        }
        tmem_st32(lrow + 64 * ch + 32 * qq, *reinterpret_cast<float(*)[32]>(v));
      }
      tmem_wait_st();
      // E1: Vt^T = U^T - (W S)^T on this thread's 32 tokens
      ok = wait_or_abort(bar_m1, j & 1, err, abort_flag);
      if (ok) {
        tc_fence_after();
        float wsv[32];
        tmem_ld32(lrow + t_ws<kP>(j) + 32 * ch, wsv);
        tmem_wait_ld();
        uint32_t pk[16];  // bf16 pairs of this thread's 32 tokens of Vt^T
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint4 uu = use_u ? *reinterpret_cast<const uint4*>(st + kUT + sw128_chunk(128, lane, 4 * ch + e))
                                 : make_uint4(0, 0, 0, 0);
          const uint32_t uw[4] = {uu.x, uu.y, uu.z, uu.w};
#pragma unroll
          for (int p = 0; p < 4; ++p) {  // u - ws as one fused (-1) ws + u per pair
            const float2 d = __ffma2_rn(make_float2(wsv[8 * e + 2 * p], wsv[8 * e + 2 * p + 1]), s2(-1.f),
                                        make_float2(bf16_lo(uw[p]), bf16_hi(uw[p])));
            wsv[8 * e + 2 * p] = d.x;
            wsv[8 * e + 2 * p + 1] = d.y;
            pk[4 * e + p] = pack_bf16(d.x, d.y);
          }
        }
        tmem_st16(lrow + kT_VT + 32 * (j & 1) + 16 * ch, pk);
        if (kP) tmem_st32(lrow + kT_VF + 32 * ch, wsv);  // Vt^T in fp32 for the tf32 update
        tmem_wait_st();
      }
      tc_fence_before();
      if (!named_sync_and(1, kEpi, ok)) { alive = false; break; }
      const uint32_t vt = tmem + kT_VT + 32 * (j & 1);
      if (t == 64) {  // S^T += Vt^T Kt
        tc_fence_after();
        if (kP) {  // kind::tf32, fp32 Vt^T from TMEM, fp32 Kt^T (two 32-token blocks)
          constexpr uint32_t id2t = idesc_tf32_mn(128, 128, 0, 0);
#pragma unroll
          for (int ks = 0; ks < C / 8; ++ks)
            mma_tf32_ta(tmem + 0, tmem + kT_VF + 8 * ks, kmajor_desc(sts + kKT, 128, ks), id2t, 1u);
        } else {
          const uint64_t bk = kmajor_desc(sts + kKT, 128, 0);
#pragma unroll
          for (int ks = 0; ks < C / 16; ++ks)
            mma_bf16_ta(tmem + 0, vt + 8 * ks, desc_advance(bk, ks * 32), id2b, 1u);
        }
        mma_commit(bar_m2);
        mma_commit(bar_empty0 + 8 * s);
        tc_fence_before();
        mbar_arrive(bar_2i);  // the output warp may issue O
        any_mma = true;
      }
    }
    if ((t == 0 || t == 64) && *abort_flag && any_mma) {  // drain MMAs in flight
      mma_commit(bar_dr + 8 * (t >> 5));
      mbar_wait(bar_dr + 8 * (t >> 5), 0, err);
    }
    if (alive && nch > 0 && wait_or_abort(bar_m2, (nch - 1) & 1, err, abort_flag))
      tc_fence_after();
    float* cp_end = (alive && nch > 0) ? ckpt_row(jl0 + nch) : nullptr;
    if ((fin || cp_end) && !*abort_flag) {
      tc_fence_after();
#pragma unroll
      for (int qq = 0; qq < 2; ++qq) {
        const int col = 64 * ch + 32 * qq;
        float sv[32];
        tmem_ld32(lrow + col, sv);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; i += 4)
          if (fin)
            *reinterpret_cast<float4*>(fin + (int64_t)lane * D + col + i) =
                make_float4(sv[i], sv[i + 1], sv[i + 2], sv[i + 3]);
        if (cp_end) {
#pragma unroll
          for (int i = 0; i < 32; i += 8) st_global_v8(cp_end + (int64_t)lane * D + col + i, &sv[i]);
        }
      }
    }
  } else {
    // ------------------------- store warps: o rows of each chunk, off the serial path
    // Without the gate: thread = value row dv; it reads the 64 outputs of its row
    // from the chunk's D1 buffer and writes them (2-byte stores, 64 contiguous bytes
    // per warp), then frees the buffer for MMA1 two chunks later.
    if constexpr (!kG) {
      const int dv = t - kEpi;
      const uint32_t lrow = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
      for (int j = 0; j < nch; ++j) {
        const int b = j & 1;
        // warp-uniform outcome: the TMEM loads below are whole-warp instructions
        if (!__all_sync(0xffffffffu, wait_or_abort(bar_o0 + 8 * b, (j >> 1) & 1, err, abort_flag)))
          break;
        tc_fence_after();
        float ov[2][32];
        const uint32_t d1 = lrow + t_o<kP>(j);
        tmem_ld32(d1, ov[0]);
        tmem_ld32(d1 + 32, ov[1]);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(bar_f0 + 8 * b);
        const int64_t tc = tstart + (int64_t)j * C;
        __nv_bfloat16* orow = o + (tc * H + h) * D + dv;
#pragma unroll
        for (int r = 0; r < C; ++r)
          if (write_o && tc + r < tend) orow[(int64_t)r * H * D] = __float2bfloat16_rn(ov[r >> 5][r & 31]);
      }
    } else {
    // With the gate: eight warps, thread = value row and one 32-token half of the
    // chunk.  A thread reads its 32 outputs and frees the D1 buffer at once; the
    // warps form each token's sum of o^2 over the 128 value rows (a halving
    // reduce-scatter inside the warp leaves lane l the warp's sum for token l of its
    // half; the four warps of a half meet in shared memory); each thread takes its
    // column of the gate logits that the output warp copied into the stage into
    // registers and the stage goes back to the copy warp; the outputs are scaled by
    // Sigmoid(x) w / rms and stored.  Segment runs without outputs (gate_on false)
    // only read the buffers out and free them.
    const int st = t - kEpi, sw = (st >> 5) & 3, th = st >> 7, sl = st & 31;
    const int dv = 32 * sw + sl, t0h = 32 * th;  // value row, first token of the half
    const uint32_t lrow = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    float* gpart = reinterpret_cast<float*>(sm + kC_bars + 256);  // [4 row quarters][64 tokens]
    float* grr = gpart + 4 * 64;                                    // [64]: 1 / rms
    const float gw = (gate_on && ga.w) ? __ldg(ga.w + dv) : 1.f;
    for (int j = 0; j < nch; ++j) {
      const int b = j & 1, s = j % kStages;
      // warp-uniform outcome: the TMEM load below is a whole-warp instruction
      const bool ok_o = __all_sync(0xffffffffu, wait_or_abort(bar_o0 + 8 * b, (j >> 1) & 1, err,
                                                              abort_flag));
      float ov[32];
      if (ok_o) {
        tc_fence_after();
        tmem_ld32(lrow + t_o<kP>(j) + t0h, ov);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(bar_f0 + 8 * b);  // D1 buffer b read out
      }
      if (!gate_on) {
        if (!ok_o) break;
        continue;
      }
      if (ok_o) {
        float a[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) a[i] = ov[i] * ov[i];
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) {  // 32 sums over the lanes -> one per lane
          const bool up = (sl & m) != 0;
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (i < m) a[i] = (up ? a[i + m] : a[i]) + __shfl_xor_sync(0xffffffffu, up ? a[i] : a[i + m], m);
        }
        gpart[sw * 64 + t0h + sl] = a[0];  // token t0h + sl
      }
      const bool ok_x = ok_o && wait_or_abort(bar_x0 + 8 * s, (j / kStages) & 1, err, abort_flag);
      if (!named_sync_and(2, kStore, ok_x)) break;
      uint32_t xp[16];  // this thread's column of its 32 logits, bf16 pairs (tokens 2i, 2i+1)
      {
        const uint8_t* xs = sm + s * kStageBytes + kW + t0h * 256 + dv * 2;  // [64][128] bf16
#pragma unroll
        for (int i = 0; i < 16; ++i)
          xp[i] = (uint32_t)*reinterpret_cast<const uint16_t*>(xs + (2 * i) * 256) |
                  ((uint32_t)*reinterpret_cast<const uint16_t*>(xs + (2 * i + 1) * 256) << 16);
      }
      if (st < C)
        grr[st] = rsqrtf((gpart[st] + gpart[64 + st] + gpart[128 + st] + gpart[192 + st]) *
                             (1.f / D) + ga.eps);
      named_sync(2, kStore);  // logits read, 1 / rms formed
      if (st == 0) mbar_arrive(bar_empty0 + 8 * s);  // the stage may be refilled
      const int64_t tc = tstart + (int64_t)j * C + t0h;
      __nv_bfloat16* orow = o + (tc * H + h) * D + dv;
#pragma unroll
      for (int g8 = 0; g8 < 32; g8 += 8) {
        float rg[8];
        *reinterpret_cast<float4*>(rg) = *reinterpret_cast<const float4*>(grr + t0h + g8);
        *reinterpret_cast<float4*>(rg + 4) = *reinterpret_cast<const float4*>(grr + t0h + g8 + 4);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = g8 + i;
          const float x = (r & 1) ? bf16_hi(xp[r >> 1]) : bf16_lo(xp[r >> 1]);
          const float sig = fmaf(0.5f, tanh_approx(0.5f * x), 0.5f);  // Sigmoid(x)
          const float y = ov[r] * (rg[i] * gw) * sig;
          if (tc + r < tend) orow[(int64_t)r * H * D] = __float2bfloat16_rn(y);
        }
      }
      // (grr and gpart are rewritten only after the next chunk's first barrier,
      // which every thread reaches after its last read of them here)
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

// One CTA: cuts every sequence into segments of at most L chunks, writes the
// segment table (sequence, first chunk, chunks, k | P << 16) and marks entries
// beyond the last segment unused.  An empty sequence is one segment of no chunks.
__global__ void __launch_bounds__(1024) seg_plan_kernel(Plan plan, int L, int4* __restrict__ tab,
                                                        int segs_ub) {
  __shared__ int32_t warp_sums[32];
  __shared__ int32_t carry;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < plan.n_seqs; base += blockDim.x) {
    const int n = base + tid;
    int c0 = 0, nch = 0, P = 0;
    if (n < plan.n_seqs) {
      c0 = plan.chunk_off[n];
      nch = plan.chunk_off[n + 1] - c0;
      P = nch > 0 ? (nch + L - 1) / L : 1;
    }
    int32_t v = P;  // block-wide inclusive scan of P
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
    const int32_t first = carry + v - P + (warp > 0 ? warp_sums[warp - 1] : 0);
    for (int k = 0; k < P && first + k < segs_ub; ++k)
      tab[first + k] = make_int4(n, c0 + k * L, min(L, nch - k * L) > 0 ? min(L, nch - k * L) : 0,
                                 k | (P << 16));
    __syncthreads();
    if (tid == blockDim.x - 1) carry = first + P;
    __syncthreads();
  }
  for (int i = carry + tid; i < segs_ub; i += blockDim.x) tab[i] = make_int4(-1, 0, 0, 0);
}

// Checkpoint offsets: off[n] = number of state checkpoints of the sequences before n,
// where sequence n has floor(len_n / (every * C)) of them (one per `every` whole
// chunks, counted from its first token).  A total above `cap` flags
// kDevErrCkptCapacity; the chain then writes only the checkpoints with index < cap.
__global__ void __launch_bounds__(1024) ckpt_plan_kernel(Plan plan, int every, int64_t cap,
                                                         int* __restrict__ off, int* err) {
  __shared__ int64_t warp_sums[32];
  __shared__ int64_t carry;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) carry = 0;
  __syncthreads();
  const int64_t span = (int64_t)every * C;
  for (int base = 0; base < plan.n_seqs; base += blockDim.x) {
    const int n = base + tid;
    int64_t cnt = 0;
    if (n < plan.n_seqs) cnt = max((int64_t)0, (int64_t)(plan.cu[n + 1] - plan.cu[n])) / span;
    int64_t v = cnt;  // block-wide inclusive scan of the counts
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += y;
    }
    if (lane == 31) warp_sums[warp] = v;
    __syncthreads();
    if (warp == 0) {
      int64_t w = lane < (int)(blockDim.x >> 5) ? warp_sums[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      warp_sums[lane] = w;
    }
    __syncthreads();
    const int64_t first = carry + v - cnt + (warp > 0 ? warp_sums[warp - 1] : 0);
    if (n < plan.n_seqs) off[n] = (int)min(first, (int64_t)INT32_MAX);
    __syncthreads();
    if (tid == blockDim.x - 1) carry = first + cnt;
    __syncthreads();
  }
  if (tid == 0) {
    off[plan.n_seqs] = (int)min(carry, (int64_t)INT32_MAX);
    if (carry > cap && err) atomicExch(err, kDevErrCkptCapacity);
  }
}

// Incoming states of the segments of one (sequence, head), in order:
//   S_in(1) = S_end(0),   S_in(k+1)^T = S~(k)^T + S_in(k)^T M(k)^T,
// in fp32 on the CUDA cores; each thread forms an 8 x 8 block of the 128 x 128 product.
constexpr int kScanLd = 129;  // padded rows of the running state in shared memory
constexpr uint32_t kScanSmem = (128 * kScanLd + 128 * 128) * 4;

__global__ void __launch_bounds__(256, 1)
    seg_scan_kernel(const int4* __restrict__ tab, int segs_ub, int H,
                    const float* __restrict__ s_end, const float* __restrict__ m_t,
                    float* __restrict__ s_in) {
  extern __shared__ __align__(16) float scan_sm[];
  float* X = scan_sm;                 // [128][kScanLd]
  float* Mt = scan_sm + 128 * kScanLd;  // [128][128]
  const int h = blockIdx.y, tid = threadIdx.x;
  // the first segment of sequence blockIdx.x (the table is in sequence order)
  const int n = blockIdx.x;
  int first = -1;
  for (int i = 0; i < segs_ub; ++i) {
    const int4 e = tab[i];
    if (e.x == n) { first = i; break; }
    if (e.x < 0 || e.x > n) break;
  }
  if (first < 0) return;
  const int P = tab[first].w >> 16;
  if (P <= 1) return;
  const auto head = [&](int seg) { return ((int64_t)seg * H + h) * D * D; };
  // S_in(1) = S_end(0)
  for (int i = tid; i < D * D; i += 256) {
    const float x = s_end[head(first) + i];
    X[(i >> 7) * kScanLd + (i & 127)] = x;
    s_in[head(first + 1) + i] = x;
  }
  const int v0 = (tid >> 4) * 8, d0 = (tid & 15) * 8;
  for (int k = 1; k + 1 < P; ++k) {
    for (int i = tid; i < D * D / 4; i += 256)
      reinterpret_cast<float4*>(Mt)[i] = reinterpret_cast<const float4*>(m_t + head(first + k))[i];
    __syncthreads();
    float acc[8][8];
#pragma unroll
    for (int a = 0; a < 8; ++a)
#pragma unroll
      for (int b = 0; b < 8; ++b) acc[a][b] = 0.f;
    for (int e = 0; e < D; ++e) {
      const float4 m0 = *reinterpret_cast<const float4*>(Mt + e * D + d0);
      const float4 m1 = *reinterpret_cast<const float4*>(Mt + e * D + d0 + 4);
      const float mv[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
#pragma unroll
      for (int a = 0; a < 8; ++a) {
        const float xv = X[(v0 + a) * kScanLd + e];
#pragma unroll
        for (int b = 0; b < 8; ++b) acc[a][b] = fmaf(xv, mv[b], acc[a][b]);
      }
    }
    __syncthreads();  // every read of X done
    const float* se = s_end + head(first + k);
    float* out = s_in + head(first + k + 1);
#pragma unroll
    for (int a = 0; a < 8; ++a)
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        const int idx = (v0 + a) * D + d0 + b;
        const float y = se[idx] + acc[a][b];
        X[(v0 + a) * kScanLd + d0 + b] = y;
        out[idx] = y;
      }
    __syncthreads();
  }
}

// cuTensorMapEncodeTiled, resolved once through the runtime's driver entry points
// (the library does not link libcuda directly).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &qr) == cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Tensor map over a token-major [NT][H][128] tensor: boxes of 64 tokens of one head,
// `box_c` channels wide, with the given shared-memory swizzle.
cudaError_t encode_rows(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int esz,
                        int H, int64_t n_tokens, int box_c = D,
                        CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_NONE, int box_t = C) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)n_tokens};
  const cuuint64_t strides[2] = {(cuuint64_t)D * esz, (cuuint64_t)H * D * esz};
  const cuuint32_t box[3] = {(cuuint32_t)box_c, 1u, (cuuint32_t)box_t};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUresult r = fn(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

int sm_count() {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms;
}

}  // namespace

namespace {

// The tensor-core workspace after the plan: tiles, gamma_C, and with segments
// the segment table and the three state arrays.
struct TcLayout {
  uint8_t* tiles;
  float* gam;
  int4* segtab;
  int* ck_off;  // [n_seqs + 1] checkpoint offsets
  float *s_end, *m_t, *s_in;
  int segs_ub;
  size_t bytes;  // from the start of the workspace
};

TcLayout tc_layout(void* ws, int64_t n_tokens, int n_seqs, int H, int seg_chunks,
                   bool precise) {
  TcLayout l{};
  const int64_t chunks = chunks_upper_bound(n_tokens, n_seqs);
  const size_t units = (size_t)chunks * H;
  size_t off = (plan_bytes(n_tokens, n_seqs) + 1023) & ~size_t(1023);
  uint8_t* base = static_cast<uint8_t*>(ws);
  l.tiles = base + off;
  off += units * (precise ? unit_bytes<true>() : unit_bytes<false>());
  l.gam = reinterpret_cast<float*>(base + off);
  off += units * kGamBytes;
  off = (off + 255) & ~size_t(255);
  l.ck_off = reinterpret_cast<int*>(base + off);
  off += ((size_t)n_seqs + 1) * sizeof(int);
  if (seg_chunks > 0) {
    l.segs_ub = (int)(chunks / seg_chunks + n_seqs);
    off = (off + 255) & ~size_t(255);
    l.segtab = reinterpret_cast<int4*>(base + off);
    off += (size_t)l.segs_ub * sizeof(int4);
    off = (off + 255) & ~size_t(255);
    const size_t st = (size_t)l.segs_ub * H * D * D * sizeof(float);
    l.s_end = reinterpret_cast<float*>(base + off);
    l.m_t = reinterpret_cast<float*>(base + off + st);
    l.s_in = reinterpret_cast<float*>(base + off + 2 * st);
    off += 3 * st;
  }
  l.bytes = off + 1024;  // slack for the 1024-byte alignment of an unaligned base
  return l;
}

}  // namespace

int chain_segment_chunks(int64_t n_tokens, int n_seqs, int H, int forced, bool sequential) {
  if (sequential || n_seqs < 1 || H < 1) return 0;
  if (forced > 0) return forced;
  const int64_t sms = sm_count();
  const int64_t chains = (int64_t)n_seqs * H;
  if (2 * chains > sms) return 0;  // enough chains to fill the GPU
  const int64_t per_seq = chunks_upper_bound(n_tokens, n_seqs) / n_seqs;
  if (per_seq < 256) return 0;     // short chains: the serial chain is short
  // P segments of L chunks: the first launch runs chains x (2P - 2) CTAs (the runs
  // from zero and the transition products), the rerun chains x (P - 1); each CTA
  // walks L chunks.  Pick the P with the fewest waves x L.
  auto waves = [&](int64_t ctas) { return (ctas + sms - 1) / sms; };
  int64_t best_p = 1, best_cost = per_seq;
  for (int64_t P = 2; P <= 64; ++P) {
    const int64_t L = (per_seq + P - 1) / P;
    if (L < 64) break;
    const int64_t cost = (waves(chains * (2 * P - 2)) + waves(chains * (P - 1))) * L;
    if (cost < best_cost) {
      best_cost = cost;
      best_p = P;
    }
  }
  if (best_p == 1) return 0;
  return (int)((per_seq + best_p - 1) / best_p);
}

size_t tc_workspace_bytes(int64_t n_tokens, int n_seqs, int H, int seg_chunks, bool precise) {
  return tc_layout(nullptr, n_tokens, n_seqs, H, seg_chunks, precise).bytes -
         plan_bytes(n_tokens, n_seqs);
}

cudaError_t launch_chunk_tc(const void* q, const void* k, const void* v, const float* g,
                            const void* z, const float* A, float g_min, const void* beta,
                            const float* h0, void* o, float* hT, int64_t n_tokens, int n_seqs,
                            int H, int seg_chunks, CkptArgs ck, FuseArgs fz, bool scalar_g,
                            bool precise, void* ws, int* err, cudaStream_t s) {
  const Plan plan = plan_in(ws, n_tokens, n_seqs);
  const int64_t units = chunks_upper_bound(n_tokens, n_seqs) * H;
  const TcLayout lay = tc_layout(ws, n_tokens, n_seqs, H, seg_chunks, precise);
  uint8_t* tiles = lay.tiles;
  float* gam = lay.gam;
  cudaError_t e;
  using T = __nv_bfloat16;
  const bool fused = z != nullptr;
  if (units > 0 && n_tokens > 0) {  // with no tokens there are no chunks to prepare
    // instances: <gate fused, precise, q/k normalised>
    using PrepFn = decltype(&tc_prep<false, false, false>);
    static const PrepFn kPrep[2][2][2] = {
        {{tc_prep<false, false, false>, tc_prep<false, false, true>},
         {tc_prep<false, true, false>, tc_prep<false, true, true>}},
        {{tc_prep<true, false, false>, tc_prep<true, false, true>},
         {tc_prep<true, true, false>, tc_prep<true, true, true>}}};
    const PrepFn kern = kPrep[fused ? 1 : 0][precise ? 1 : 0][fz.qk_eps >= 0.f ? 1 : 0];
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kQ_Smem);
    if (e == cudaSuccess)  // room for two CTAs per SM
      e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                               (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    const int ctas = 2 * sm_count();
    const int grid = (int)(units < ctas ? units : ctas);
    CUtensorMap tm[4];
    e = encode_rows(&tm[0], k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, n_tokens);
    if (e == cudaSuccess) e = encode_rows(&tm[1], q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, n_tokens);
    if (e == cudaSuccess)
      e = encode_rows(&tm[2], v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, n_tokens, 64,
                      CU_TENSOR_MAP_SWIZZLE_128B);
    if (e == cudaSuccess) {
      if (fused)  // z in two boxes of 32 tokens
        e = encode_rows(&tm[3], z, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, n_tokens, D,
                        CU_TENSOR_MAP_SWIZZLE_NONE, C / 2);
      else if (scalar_g)
        tm[3] = tm[0];  // not used: scalar gates are plain loads, not prefetched
      else
        e = encode_rows(&tm[3], g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, H, n_tokens);
    }
    if (e != cudaSuccess) return e;
    ProfScope prof_scope(fused ? "kda_tc_prep_gated" : "kda_tc_prep", s);
    kern<<<grid, kP2Threads, kQ_Smem, s>>>(tm[0], tm[1], tm[2], tm[3],
                                           static_cast<const T*>(beta), A, g_min, plan, H,
                                           units, tiles, gam, fz.qk_eps,
                                           (scalar_g && !fused) ? g : nullptr, err);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (ck.every > 0) {  // checkpoints requested (a null ck.ckpt only checks the count)
    ProfScope prof_scope("kda_ckpt_plan", s);
    ckpt_plan_kernel<<<1, 1024, 0, s>>>(plan, ck.every, ck.cap, lay.ck_off, err);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // the output gate, applied by the chain's store warps (a tensor map over the logits)
  CUtensorMap tm_x;
  memset(&tm_x, 0, sizeof(tm_x));
  const GateArgs ga{fz.w, fz.eps};
  if (fz.gz) {
    e = encode_rows(&tm_x, fz.gz, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, n_tokens);
    if (e != cudaSuccess) return e;
  }
  // instances: <precise, output gate, checkpoints>
  using ChainFn = decltype(&tc_chain<false, false, false>);
  static const ChainFn kChain[2][2][2] = {
      {{tc_chain<false, false, false>, tc_chain<false, false, true>},
       {tc_chain<false, true, false>, tc_chain<false, true, true>}},
      {{tc_chain<true, false, false>, tc_chain<true, false, true>},
       {tc_chain<true, true, false>, tc_chain<true, true, true>}}};
  const ChainFn chain = kChain[precise ? 1 : 0][fz.gz ? 1 : 0][ck.ckpt ? 1 : 0];
  const int chain_thr = fz.gz ? chain_threads<true>() : chain_threads<false>();
  const uint32_t chain_sm = precise ? chain_smem<true>() : chain_smem<false>();
  e = cudaFuncSetAttribute(chain, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)chain_sm);
  if (e != cudaSuccess) return e;
  if (seg_chunks <= 0) {
    const dim3 cgrid((unsigned)n_seqs, (unsigned)H);
    ProfScope prof_scope("kda_tc_chain", s);
    chain<<<cgrid, chain_thr, chain_sm, s>>>(tiles, gam, h0, plan, H, static_cast<T*>(o),
                                                    hT, SegArgs{0, nullptr, nullptr, nullptr, nullptr},
                                                    ck, lay.ck_off, err, tm_x, ga);
    return cudaGetLastError();
  }
  // sequence-segment parallel chain: segments, end states and transitions, scan, rerun
  SegArgs sg{1, lay.segtab, lay.s_end, lay.m_t, lay.s_in};
  {
    ProfScope prof_scope("kda_seg_plan", s);
    seg_plan_kernel<<<1, 1024, 0, s>>>(plan, seg_chunks, lay.segtab, lay.segs_ub);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  {
    ProfScope prof_scope("kda_tc_chain_seg", s);
    chain<<<dim3((unsigned)lay.segs_ub, (unsigned)H, 2), chain_thr, chain_sm, s>>>(
        tiles, gam, h0, plan, H, static_cast<T*>(o), hT, sg, ck, lay.ck_off, err, tm_x, ga);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  e = cudaFuncSetAttribute(seg_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kScanSmem);
  if (e != cudaSuccess) return e;
  {
    ProfScope prof_scope("kda_seg_scan", s);
    seg_scan_kernel<<<dim3((unsigned)n_seqs, (unsigned)H), 256, kScanSmem, s>>>(
        lay.segtab, lay.segs_ub, H, lay.s_end, lay.m_t, lay.s_in);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  sg.mode = 2;
  ProfScope prof_scope("kda_tc_chain_seg", s);
  chain<<<dim3((unsigned)lay.segs_ub, (unsigned)H, 1), chain_thr, chain_sm, s>>>(
      tiles, gam, h0, plan, H, static_cast<T*>(o), hT, sg, ck, lay.ck_off, err, tm_x, ga);
  return cudaGetLastError();
}

}  // namespace kda
