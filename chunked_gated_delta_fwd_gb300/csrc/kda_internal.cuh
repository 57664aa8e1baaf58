// kda_internal.cuh -- declarations shared by the translation units of libkda.
//
// Every kernel launcher here is called only from kda_api.cu after the public
// arguments have been validated; launchers return the cudaError_t of the launch.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kda {

constexpr int kD = 128;      // dk = dv = 128 (the published K3 head size)
constexpr int kChunk = 64;   // tokens per chunk of the chunkwise form
constexpr int kTile = 16;    // tokens per decay-reference tile inside a chunk

// Device error codes written to the flag returned by device_error_flag().
constexpr int kDevErrNone = 0;
constexpr int kDevErrTimeout = 7;
constexpr int kDevErrBadSeqlens = 1;
constexpr int kDevErrCkptCapacity = 2;
constexpr int kDevErrPrecondition = 3;  // an input outside its stated range (checks pass)

// Address of this device's error flag (int on the device), or nullptr.
int* device_error_flag();

// ---- per-kernel event timing (enabled by kda_profile_enable) ---------------
// Launchers hold a ProfScope across each kernel launch; when profiling is off
// it does nothing.  Events are recorded on the launching stream.
struct ProfScope {
  ProfScope(const char* name, cudaStream_t s);
  ~ProfScope();
  int slot;
  cudaStream_t stream;
};

// ---- element access helpers (inputs are fp32 or bf16, math is fp32) --------
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Loads 8 consecutive elements (16-byte aligned for bf16, 32-byte for fp32) as fp32.
__device__ __forceinline__ void load8(const float* p, float* out) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4);
  out[0] = a.x; out[1] = a.y; out[2] = a.z; out[3] = a.w;
  out[4] = b.x; out[5] = b.y; out[6] = b.z; out[7] = b.w;
}
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float* out) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    out[2 * i] = __uint_as_float(w[i] << 16);
    out[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
__device__ __forceinline__ void load4(const float* p, float* out) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  out[0] = a.x; out[1] = a.y; out[2] = a.z; out[3] = a.w;
}
__device__ __forceinline__ void load4(const __nv_bfloat16* p, float* out) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  out[0] = __uint_as_float(u.x << 16);
  out[1] = __uint_as_float(u.x & 0xffff0000u);
  out[2] = __uint_as_float(u.y << 16);
  out[3] = __uint_as_float(u.y & 0xffff0000u);
}
// Stores 8 consecutive elements from fp32 (32-byte aligned for fp32, 16-byte for bf16).
__device__ __forceinline__ void store8(float* p, const float* v) {
  reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}
__device__ __forceinline__ void store8(__nv_bfloat16* p, const float* v) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    w[i] = *reinterpret_cast<const uint32_t*>(&b);
  }
  *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}
// Stores 4 consecutive elements from fp32 (16-byte aligned for fp32, 8-byte for bf16).
__device__ __forceinline__ void store4(float* p, const float* v) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
}
__device__ __forceinline__ void store4(__nv_bfloat16* p, const float* v) {
  const __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]), b = __floats2bfloat162_rn(v[2], v[3]);
  *reinterpret_cast<uint2*>(p) =
      make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
}

// ---- chunk plan -------------------------------------------------------------
// The workspace starts with the plan: cu[N+1] (int32 token offsets) followed by
// chunk_off[N+1] (int32, first global chunk of each sequence; chunk_off[N] is
// the total number of chunks).  Built on the device by launch_plan().
struct Plan {
  const int32_t* cu;
  const int32_t* chunk_off;
  const int2* tab;  // per chunk: (first token, token count)
  int n_seqs;
};
size_t plan_bytes(int64_t n_tokens, int n_seqs);
// The plan arrays as laid out at the start of the workspace.
Plan plan_in(void* ws, int64_t n_tokens, int n_seqs);
cudaError_t launch_plan(const int32_t* cu_seqlens_or_null, int n_seqs, int64_t T_per_seq,
                        int64_t n_tokens, void* ws, int* err_flag, cudaStream_t s);
// Upper bound of the number of 64-token chunks of n_seqs sequences totalling n_tokens.
inline int64_t chunks_upper_bound(int64_t n_tokens, int n_seqs) {
  return n_tokens / kChunk + n_seqs;
}

// ---- kernels ----------------------------------------------------------------
cudaError_t launch_gate(const void* z, int z_bf16, const float* A, float g_min, float* g,
                        int64_t n_tokens, int H, cudaStream_t s);
cudaError_t launch_gate_softplus(const void* z, int z_bf16, const float* A, float* g,
                                 int64_t n_tokens, int H, cudaStream_t s);
// y = Sigmoid(x) * w * o / sqrt(mean(o^2) + eps) per (token, head); y may alias o.
cudaError_t launch_output_gate(const void* o, int bf16, const void* x, const float* w, float eps,
                               void* y, int64_t n_tokens, int H, cudaStream_t s);
cudaError_t launch_gate_cumsum(const void* z, int z_bf16, const float* A, float g_min, float* g,
                               float* gcum, int64_t n_tokens, int H, const int32_t* cu,
                               int n_seqs, cudaStream_t s);
// T (<= 16) tokens per (sequence, head); the state is advanced by n_advance[n]
// tokens (all T when n_advance is null); o may be null.
cudaError_t launch_decode_multi(const void* q, const void* k, const void* v, int bf16,
                                const float* g, const void* beta, float* S, void* o,
                                const int32_t* n_advance, int N, int T, int H, cudaStream_t s);
cudaError_t launch_decode(const void* q, const void* k, const void* v, int bf16, const float* g,
                          const void* beta, float* S, void* o, int N, int H, cudaStream_t s);

// fp32 CUDA-core chunk path (any input dtype, fp32 arithmetic throughout).
size_t simt_workspace_bytes(int64_t n_tokens, int n_seqs, int H);
cudaError_t launch_chunk_simt(const void* q, const void* k, const void* v, int bf16,
                              const float* g, const void* beta, const float* h0, void* o,
                              float* hT, int64_t n_tokens, int n_seqs, int H, void* ws,
                              cudaStream_t s, int robust = 0);

// bf16 tensor-core (tcgen05) chunk path.
// Chunks per chain segment for the sequence-segment parallel chain (0: the chain of
// each (sequence, head) runs in one CTA).  `forced` > 0 overrides the choice.
int chain_segment_chunks(int64_t n_tokens, int n_seqs, int H, int forced, bool sequential);
// precise: the precise-state mode (Kt fp32 in the workspace, tf32 state update).
size_t tc_workspace_bytes(int64_t n_tokens, int n_seqs, int H, int seg_chunks, bool precise);
// With z non-null the gate is fused: g is formed from z (bf16), A and g_min and g
// is ignored.  With scalar_g, g is [n_tokens][H]: one log-decay per token and head.
// State checkpoints: the state after every `every` chunks of each sequence (ckpt:
// fp32 [cap][H][dv][dk], in sequence order); null ckpt writes none.
struct CkptArgs {
  float* ckpt;
  int every;
  int64_t cap;
};
// Fused prologue / epilogue of the tensor-core chunk path: q, k L2-normalised in the
// prepare kernel (qk_eps < 0: off) and the output RMSNorm x Sigmoid gate applied by
// the chain's store warps before o is written (gz: bf16 logits [NT][H][128], null:
// off; w null: unit weight).
struct FuseArgs {
  float qk_eps;
  const void* gz;
  const float* w;
  float eps;
};
cudaError_t launch_chunk_tc(const void* q, const void* k, const void* v, const float* g,
                            const void* z, const float* A, float g_min, const void* beta,
                            const float* h0, void* o, float* hT, int64_t n_tokens, int n_seqs,
                            int H, int seg_chunks, CkptArgs ck, FuseArgs fz, bool scalar_g,
                            bool precise, void* ws, int* err_flag, cudaStream_t s);
// Input-precondition pass: raises kDevErrPrecondition in *err if any of the n_g
// log-decays g is outside [g_lo, 0] or any of the n_beta write strengths outside
// [0, 1] (NaN counts as outside).  g or beta may be null (nothing to check).
cudaError_t launch_check_inputs(const float* g, int64_t n_g, float g_lo, const void* beta,
                                int beta_bf16, int64_t n_beta, int* err, cudaStream_t s);
// Bounded-wait self-test: a kernel whose waits nothing signals gives up after
// timeout_ns (recording kDevErrTimeout in *err); synchronizes s and returns in
// *warps_gave_up how many of its four waiting warps saw their wait end unsatisfied.
cudaError_t launch_wait_selftest(uint64_t timeout_ns, int* err, int* warps_gave_up,
                                 cudaStream_t s);
// g[t][h][c] = gs[t][h] for every channel c: scalar gates spread for the fp32 path.
cudaError_t launch_expand_scalar_gate(const float* gs, float* g, int64_t n_tokens, int H,
                                      cudaStream_t s);

}  // namespace kda
