/*
 * kda.h -- C ABI of the GB300 Kimi Delta Attention (KDA) forward library.
 *
 * KDA, per head, with state S in R^{dk x dv}:
 *     S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = S_t^T q_t
 *     alpha_t = exp(g_t),  g_t = g_min * Sigmoid(exp(A_h) * z_t),  g_min = -5
 * ("Kimi K3 technical report review" (devpress/CSDN), section 3.1 Eq. 1 and
 *  section 3.2 Eq. 5; "Kimi K3: architecture, training and inference systems"
 *  (weigao.cc), section 3.1).
 *
 * Conventions shared by every call
 *  - Pointers are DEVICE pointers unless a name says otherwise; the caller owns
 *    every buffer and the stream.  The library allocates no device memory, keeps
 *    no pointer after a call returns, and enqueues all work on `stream`
 *    (asynchronous: results are ready when the stream reaches them).
 *  - Token-major layouts.  A batch of N sequences is packed along the token
 *    axis: q, k: [NT][H][dk], v, o: [NT][H][dv], g: [NT][H][dk], beta: [NT][H].
 *    Sequence n owns tokens cu_seqlens[n] .. cu_seqlens[n+1]-1.
 *  - The state is stored TRANSPOSED, fp32: S^T as [N][H][dv][dk] (dk contiguous),
 *    the [B, H, V, K] layout of the FlashKDA state ("Kimi K3: architecture,
 *    training and inference systems", section 13.1).  hT of kda_chunk_fwd and S of
 *    kda_recurrent_step use the same layout, so a prefill's hT is a decode's S.
 *  - dk = dv = 128 is required (the published K3 head size); anything else
 *    returns KDA_ERR_UNSUPPORTED_SHAPE.
 *  - Every pointer must be 16-byte aligned and every tensor contiguous;
 *    otherwise KDA_ERR_MISALIGNED.  Arguments are checked before any launch: a
 *    call that returns an error has enqueued nothing.
 *  - Errors: a non-zero kda_status_t; kda_last_error_string() (per thread)
 *    describes the last error.  Device-side waits are bounded: a kernel whose
 *    wait runs out of iterations records KDA_ERR_DEVICE_TIMEOUT in a device flag
 *    and exits; kda_get_device_error() reads and clears it.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* kda_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
  KDA_OK = 0,
  KDA_ERR_INVALID_ARG = 1,       /* null pointer where one is required, bad count or bound */
  KDA_ERR_UNSUPPORTED_SHAPE = 2, /* dk or dv other than 128, H < 1 */
  KDA_ERR_UNSUPPORTED_DTYPE = 3, /* dtype code not in kda_dtype_t */
  KDA_ERR_MISALIGNED = 4,        /* pointer not 16-byte aligned */
  KDA_ERR_WORKSPACE_TOO_SMALL = 5,
  KDA_ERR_CUDA = 6,            /* a CUDA runtime call or launch failed */
  KDA_ERR_DEVICE_TIMEOUT = 7,  /* a bounded device-side wait gave up */
  KDA_ERR_NO_DEVICE = 8        /* no usable sm_103 device for this call */
} kda_status_t;

typedef enum { KDA_F32 = 0, KDA_BF16 = 1 } kda_dtype_t;

/*
 * kda_gate -- bounded log-decay, elementwise:
 *     g[t][h][c] = g_min * Sigmoid(exp(A[h]) * z[t][h][c])
 * ("Kimi K3 technical report review", section 3.2, Eq. 5; g lies in [g_min, 0]).
 *
 *   z        [n_tokens][H][dk], dtype z_dtype (KDA_F32 or KDA_BF16)
 *   A        [H] fp32, one log-scale per head
 *   g_min    lower bound of the decay (the K3 report fixes -5); must be < 0
 *   g        [n_tokens][H][dk] fp32, written
 *   gcum     optional (NULL to skip) [n_tokens][H][dk] fp32: the inclusive running
 *            sum of g inside each 64-token chunk of each sequence, restarting at
 *            every chunk start (token cu[n] + 64 m) -- the log of the in-chunk
 *            cumulative decay Gamma of the chunkwise form ("Kimi K3 notes"
 *            (s1mplewind blog), section "Chunkwise form").
 *   cu_seqlens optional device int32 [n_seqs+1] giving the sequence starts for
 *            gcum; NULL means one sequence of n_tokens tokens.  Ignored if gcum is NULL.
 * n_tokens == 0 is a no-op.
 */
kda_status_t kda_gate(const void* z, int z_dtype, const float* A, float g_min, float* g,
                      int64_t n_tokens, int H, int dk, float* gcum, const int32_t* cu_seqlens,
                      int n_seqs, kda_stream_t stream);

/*
 * kda_gate_softplus -- the unbounded log-decay that the bounded gate replaced
 * (Kimi Linear; "Kimi K3 technical report review", section 3.2), elementwise:
 *     g[t][h][c] = -exp(A[h]) * Softplus(z[t][h][c]),  Softplus(x) = log(1 + e^x)
 * g lies in (-inf, 0); a prefill on it needs KDA_CHUNK_UNBOUNDED_GATE.  Arguments,
 * layouts and errors as kda_gate (no g_min, no running sum).
 */
kda_status_t kda_gate_softplus(const void* z, int z_dtype, const float* A, float* g,
                               int64_t n_tokens, int H, int dk, kda_stream_t stream);

/*
 * kda_chunk_fwd_workspace_size -- bytes of device workspace kda_chunk_fwd needs
 * for n_tokens tokens in n_seqs sequences and H heads with inputs of `dtype`.
 * Returns 0 for invalid arguments.
 */
size_t kda_chunk_fwd_workspace_size(int64_t n_tokens, int n_seqs, int H, int dtype);
/* The same for kda_chunk_fwd_ex with `flags` (kda_chunk_fwd_workspace_size is flags = 0). */
size_t kda_chunk_fwd_workspace_size_ex(int64_t n_tokens, int n_seqs, int H, int dtype,
                                       unsigned flags);

/*
 * kda_chunk_fwd -- prefill: the KDA forward over whole sequences, evaluated in
 * 64-token chunks with the WY/UT chunkwise form ("Kimi K3 notes", section
 * "Chunkwise form"; "Hybrid KDA-MLA: Kimi K3 attention explained", section
 * "KDA kernel"), variable-length sequences included.
 *
 *   q, k     [NT][H][dk], dtype; q and k are expected L2-normalised per token and head
 *   v        [NT][H][dv], dtype
 *   dtype    KDA_BF16 (tensor-core path, fp32 accumulation and fp32 state) or
 *            KDA_F32 (fp32 CUDA-core path)
 *   g        [NT][H][dk] fp32 log-decays.  PRECONDITION: g_min_bound <= g <= 0 with
 *            g_min_bound = -5 (the output range of kda_gate with g_min = -5); the
 *            16-token tile range argument of the K3 report relies on it.  Values
 *            outside give unspecified (possibly non-finite) output; they are
 *            detected only by the optional input check (KDA_CHUNK_CHECK_INPUTS of
 *            kda_chunk_fwd_ex, or KDA_CHECKS=1 in the environment).
 *   beta     [NT][H], dtype, write strengths (expected in [0, 1])
 *   h0       optional [N][H][dv][dk] fp32 initial states (NULL = zero state)
 *   cu_seqlens optional device int32 [N+1], nondecreasing, cu[0] = 0, cu[N] = NT;
 *            NULL means B sequences of T tokens each (N = B, NT = B*T).
 *   n_seqs   N when cu_seqlens is given (ignored otherwise)
 *   B, T     batch and length when cu_seqlens is NULL; with cu_seqlens, B must be 1
 *            and T = NT
 *   o        [NT][H][dv], dtype, written (must not alias an input)
 *   hT       optional [N][H][dv][dk] fp32 final states (NULL to skip).  hT may alias
 *            h0: each (sequence, head) state is read before it is written.
 *   workspace, ws_bytes  device scratch of at least
 *            kda_chunk_fwd_workspace_size(NT, N, H, dtype) bytes, 256-byte aligned;
 *            its contents on entry do not matter and are garbage on return.
 * A sequence of length 0 gets hT = h0 (or zeros).  NT == 0 writes only hT.
 */
kda_status_t kda_chunk_fwd(const void* q, const void* k, const void* v, int dtype,
                           const float* g, const void* beta, const float* h0,
                           const int32_t* cu_seqlens, int n_seqs, int B, int64_t T, int H,
                           int dk, int dv, void* o, float* hT, void* workspace, size_t ws_bytes,
                           kda_stream_t stream);

/* Flags of kda_chunk_fwd_ex. */
enum {
  KDA_CHUNK_FP32_CORES = 1u,     /* evaluate on fp32 CUDA cores even for bf16 inputs */
  KDA_CHUNK_SEQUENTIAL = 2u,     /* never split a sequence's chain into segments */
  KDA_CHUNK_UNBOUNDED_GATE = 4u, /* any g <= 0 (range-robust fp32-core evaluation) */
  KDA_CHUNK_SCALAR_GATE = 8u,    /* g is [NT][H]: one log-decay per token and head */
  KDA_CHUNK_CHECK_INPUTS = 16u,  /* check the g and beta preconditions on the device */
  KDA_CHUNK_PRECISE = 32u        /* tensor-core path: the state update at tf32 precision */
};
/* Split every sequence's chain into segments of n chunks (n in 1..65535). */
#define KDA_CHUNK_SEGMENT_CHUNKS(n) (((unsigned)(n) & 0xffffu) << 16)

/*
 * kda_chunk_fwd_ex -- kda_chunk_fwd with option flags (0 = kda_chunk_fwd).
 * KDA_CHUNK_FP32_CORES selects the fp32 CUDA-core evaluation of the same chunkwise
 * form for bf16 inputs (the path KDA_F32 inputs always take).
 *
 * KDA_CHUNK_UNBOUNDED_GATE lifts the g >= -5 precondition: any finite g <= 0 (the
 * unbounded gate -exp(A) Softplus(z) of Kimi Linear, kda_gate_softplus).  The
 * 16-token tile references are then taken so that every rescaling factor is <= 1
 * and the diagonal 16x16 tiles are formed pair by pair, exp(G_r - G_i) per
 * channel -- the position-pair path that the bound makes unnecessary ("Kimi K3
 * technical report review", section 3.2).  It runs on the fp32 CUDA cores for
 * either dtype (workspace as for KDA_CHUNK_FP32_CORES).
 *
 * Sequence segments (bf16 tensor-core path): the state update of one (sequence,
 * head) is serial over its chunks.  When there are too few (sequence, head)
 * chains to occupy the GPU (2 N H <= number of SMs) and sequences average at
 * least 256 chunks, the library cuts each sequence into segments that run in
 * parallel and joins them with the context-parallel algebra of the K3 report
 * ("Kimi K3 technical report review", section 8.1, Eq. 17): each segment's end
 * state is S~ + M S_in with S~ its run from a zero state and M the product of its
 * chunk transitions; the incoming states follow by an ordered scan and the
 * segments are rerun from them.  The result equals the serial chain up to
 * rounding.  KDA_CHUNK_SEQUENTIAL turns this off; KDA_CHUNK_SEGMENT_CHUNKS(n)
 * forces segments of n chunks.
 *
 * KDA_CHUNK_SCALAR_GATE: g is [NT][H] fp32, one log-decay per token and head
 * applied to every key channel -- the scalar gate of Gated DeltaNet, which KDA
 * refines to one decay per channel ("Kimi K3 notes", section "Kimi Delta
 * Attention", its comparison with Gated DeltaNet).  The same precondition (-5 <= g <= 0 unless
 * KDA_CHUNK_UNBOUNDED_GATE) holds.  The tensor-core path reads the scalars
 * directly (4 bytes per token and head instead of 512); the fp32-core path
 * first spreads them over the channels in the workspace.  Not combinable with a
 * gate formed from z.
 *
 * KDA_CHUNK_PRECISE (bf16 tensor-core path): the chunk's state update
 * S <- Diag(gamma_C) S + Kt^T Vt takes Kt = (gamma_C / Gamma) K and the pseudo-values
 * Vt = U - W S at tf32 precision (kind::tf32 MMAs, Kt kept in fp32 in the
 * workspace) instead of bf16.  With nearly parallel keys and beta near 1 the
 * update cancels large terms, and the bf16 rounding of Kt and Vt is what moves the
 * final state most: on keys with k_i . k_j ~ 0.99, beta = 1 and slow decay the
 * final state is at relative L2 ~1.2e-2 by default and ~6e-3 with this flag.  It
 * costs 16 KB more workspace per (chunk, head), a two-stage tile ring in the chain
 * and twice the tensor-pipe time of the update.  Workspace:
 * kda_chunk_fwd_workspace_size_ex with the flag.
 *
 * KDA_CHUNK_CHECK_INPUTS (also turned on for every chunk call by the environment
 * variable KDA_CHECKS=1, read once per process): before the prefill, one pass
 * over g and beta checks the preconditions the method relies on -- every
 * log-decay in [-5, 0] (the bounded gate, "Kimi K3 technical report review",
 * section 3.2; in the unbounded mode only g <= 0 and finite) and every beta in
 * [0, 1] (a sigmoid output) -- and raises the device error flag if one fails or
 * is NaN; kda_get_device_error then returns KDA_ERR_INVALID_ARG.  The prefill
 * still runs (its output is then unspecified).  With a gate formed from z only
 * beta is checked.  The pass reads g and beta once (about 60 us for the
 * B=1, T=8192, H=96 workload) and is off by default.
 *
 * The workspace requirement depends on the flags:
 * kda_chunk_fwd_workspace_size_ex(NT, N, H, dtype, flags).  Unknown flag bits
 * return KDA_ERR_INVALID_ARG.
 */
kda_status_t kda_chunk_fwd_ex(const void* q, const void* k, const void* v, int dtype,
                              const float* g, const void* beta, const float* h0,
                              const int32_t* cu_seqlens, int n_seqs, int B, int64_t T, int H,
                              int dk, int dv, void* o, float* hT, void* workspace,
                              size_t ws_bytes, kda_stream_t stream, unsigned flags);

/*
 * kda_chunk_fwd_fused -- the bf16 tensor-core prefill with its prologue and
 * epilogue fused: the gate from z (as kda_chunk_fwd_gated), q and k
 * L2-normalised per token and head inside the prepare kernel (the FlashKDA
 * prepare kernel normalises before the gate prefix sums: "Kimi K3 notes",
 * section "FlashKDA", kernel K1), and the head-wise RMSNorm x Sigmoid output gate
 * ("Kimi K3 technical report review", section 3.3, Eq. 6; "Kimi K3:
 * architecture, training and inference systems", section 3.3) applied to o.
 *   g or z, A, g_min  exactly one of g (as kda_chunk_fwd) and z (as
 *              kda_chunk_fwd_gated; A and g_min then as there).
 *   qk_l2_eps  >= 0: q_t <- q_t / sqrt(|q_t|^2 + qk_l2_eps), the same for k, per
 *              token and head, before anything else uses them (the normalised
 *              rows are rounded to bf16, as normalised inputs would be);
 *              < 0: q and k are used as given (expected normalised).
 *   out_gate   optional [NT][H][dv] of `dtype`, 16-byte aligned: gate logits x.
 *              When given, o_t = Sigmoid(x_t) * w * o~_t / sqrt(mean(o~_t^2) +
 *              out_norm_eps) with the mean over the dv channels of one head and
 *              o~ the KDA output; NULL: o = o~.  The chain kernel applies it before
 *              it writes o: each 64-token tile of logits is copied into the chain's
 *              tile ring, the per-token RMS is reduced across the warps that hold
 *              o~ in fp32, and y is written once (o~ never goes to memory).
 *   out_norm_weight  optional fp32 [dv] RMSNorm weight w shared by the heads
 *              (NULL: ones); only with out_gate.
 *   out_norm_eps  finite, >= 0 (used only with out_gate).
 * flags: KDA_CHUNK_SEQUENTIAL and KDA_CHUNK_SEGMENT_CHUNKS(n) as for
 * kda_chunk_fwd_ex; the workspace is kda_chunk_fwd_workspace_size_ex(NT, N, H,
 * KDA_BF16, flags).  Every other argument and result as kda_chunk_fwd.
 * Errors: dtype other than KDA_BF16 or KDA_CHUNK_FP32_CORES ->
 * KDA_ERR_UNSUPPORTED_DTYPE; both or neither of g and z, g_min outside [-5, 0),
 * a non-finite epsilon or out_norm_weight without out_gate -> KDA_ERR_INVALID_ARG;
 * otherwise as kda_chunk_fwd_ex.
 */
kda_status_t kda_chunk_fwd_fused(const void* q, const void* k, const void* v, int dtype,
                                 const float* g, const void* z, const float* A, float g_min,
                                 const void* beta, const float* h0, const int32_t* cu_seqlens,
                                 int n_seqs, int B, int64_t T, int H, int dk, int dv,
                                 float qk_l2_eps, const void* out_gate,
                                 const float* out_norm_weight, float out_norm_eps, void* o,
                                 float* hT, void* workspace, size_t ws_bytes, kda_stream_t stream,
                                 unsigned flags);

/*
 * kda_output_gate -- the head-wise RMSNorm x Sigmoid output gate on KDA outputs
 * ("Kimi K3 technical report review", section 3.3, Eq. 6, without the W_o and W_g
 * projections), per token t and head h over the dv channels c:
 *     y[t][h][c] = Sigmoid(gate[t][h][c]) * weight[c] * o[t][h][c]
 *                  / sqrt(mean_c(o[t][h][c]^2) + eps)
 *   o, gate, y  [n_tokens][H][dv] of `dtype` (KDA_F32 or KDA_BF16), 16-byte aligned;
 *               y may alias o (in place).
 *   weight      optional fp32 [dv] (NULL: ones), shared by the heads.
 *   eps         finite, >= 0.
 * dv must be 128.  n_tokens == 0 is a no-op.  Errors as kda_gate.
 */
kda_status_t kda_output_gate(const void* o, int dtype, const void* gate, const float* weight,
                             float eps, void* y, int64_t n_tokens, int H, int dv,
                             kda_stream_t stream);

/*
 * kda_chunk_fwd_checkpointed -- kda_chunk_fwd_ex that also writes the state at
 * fixed token boundaries of every sequence, the KDA state checkpoints a prefix
 * cache keeps at hash endpoints (e.g. every 512 tokens; "Kimi K3: architecture,
 * training and inference systems", section 12.2).
 *   ckpt         fp32 [ckpt_capacity][H][dv][dk], device, 32-byte aligned,
 *                caller-owned; may be null only when ckpt_capacity is 0.
 *   ckpt_tokens  checkpoint interval in tokens, a positive multiple of 64.
 *   ckpt_capacity number of checkpoint slots in ckpt.
 * Sequence n (of length len_n, in the order of cu_seqlens or of the batch) has
 * c_n = floor(len_n / ckpt_tokens) checkpoints; its i-th (i = 1..c_n) is the state
 * S^T after its first i * ckpt_tokens tokens, in the layout of hT, and is stored
 * at index c_0 + ... + c_{n-1} + i - 1.  A checkpoint at the sequence end equals
 * that sequence's hT.  Every other argument, the workspace size
 * (kda_chunk_fwd_workspace_size_ex with the same flags) and the results are those
 * of kda_chunk_fwd_ex.  The count is formed on the device from cu_seqlens: when
 * it exceeds ckpt_capacity only the first ckpt_capacity checkpoints are written
 * and kda_get_device_error reports KDA_ERR_INVALID_ARG.
 * Errors: dtype other than KDA_BF16 or KDA_CHUNK_FP32_CORES set ->
 * KDA_ERR_UNSUPPORTED_DTYPE (checkpoints are written by the tensor-core chain
 * only); ckpt_tokens not a positive multiple of 64, negative capacity or null
 * ckpt with a positive capacity -> KDA_ERR_INVALID_ARG; misaligned ckpt ->
 * KDA_ERR_MISALIGNED; otherwise as kda_chunk_fwd_ex.
 */
kda_status_t kda_chunk_fwd_checkpointed(const void* q, const void* k, const void* v, int dtype,
                                        const float* g, const void* beta, const float* h0,
                                        const int32_t* cu_seqlens, int n_seqs, int B, int64_t T,
                                        int H, int dk, int dv, void* o, float* hT, float* ckpt,
                                        int ckpt_tokens, int64_t ckpt_capacity, void* workspace,
                                        size_t ws_bytes, kda_stream_t stream, unsigned flags);

/*
 * kda_chunk_fwd_gated -- kda_chunk_fwd with the bounded gate evaluated inside the
 * chunk kernels instead of read as g.  The gate is that of kda_gate ("Kimi K3
 * technical report review", section 3.2: g = g_min * Sigmoid(exp(A_h) z)); it is
 * formed from z while each chunk's decays are summed and is never written to
 * memory, as the FlashKDA prepare kernel forms its gate prefix sums in place
 * ("Kimi K3 notes", section "FlashKDA", kernel K1).  Only the bf16 tensor-core
 * path has this form.
 *   z      [NT, H, dk] of `dtype`, device, same layout and alignment as k.
 *   A      fp32 [H], device (per-head log scale of the gate).
 *   g_min  lower bound of the gate, in [-5, 0): the 16-token tile range argument
 *          needs g >= -5.
 * Every other argument, the workspace size (kda_chunk_fwd_workspace_size with
 * KDA_BF16) and the results are those of kda_chunk_fwd with g = kda_gate(z, A).
 * Errors: dtype other than KDA_BF16 -> KDA_ERR_UNSUPPORTED_DTYPE (for fp32 inputs
 * call kda_gate, then kda_chunk_fwd); g_min outside [-5, 0) -> KDA_ERR_INVALID_ARG;
 * otherwise as kda_chunk_fwd.
 */
kda_status_t kda_chunk_fwd_gated(const void* q, const void* k, const void* v, int dtype,
                                 const void* z, const float* A, float g_min, const void* beta,
                                 const float* h0, const int32_t* cu_seqlens, int n_seqs, int B,
                                 int64_t T, int H, int dk, int dv, void* o, float* hT,
                                 void* workspace, size_t ws_bytes, kda_stream_t stream);

/*
 * kda_chunk_fwd_noalloc -- kda_chunk_fwd without a caller-supplied workspace.
 * The KDA pages have no counterpart for this entry point: it exists for callers
 * that must not allocate device memory where they run the prefill (a serving
 * engine that reserved all device memory up front, a plugin host that offers no
 * allocator, a latency-critical loop that cannot pay an allocation's implicit
 * synchronization).  Arguments, layouts and results are those of kda_chunk_fwd.
 *
 * The scratch comes from one fixed array of KDA_NOALLOC_SCRATCH_BYTES in device
 * memory, declared by the library; every GPU that loads the library holds it
 * until the process exits.  The call allocates nothing.  A problem whose
 * workspace (kda_chunk_fwd_workspace_size) exceeds the capacity is rejected with
 * KDA_ERR_WORKSPACE_TOO_SMALL before anything is enqueued.  The first call on a
 * device resolves the array's device address (cudaGetSymbolAddress, with that
 * device current); make that first call before any stream capture.  All calls
 * share the array and it keeps the last call's contents (nothing in it needs to
 * start at zero); calls whose work overlaps on the GPU, e.g. on two streams
 * without ordering between them, race on it.
 */
#define KDA_NOALLOC_SCRATCH_BYTES ((size_t)128 << 20) /* 128 MiB */
kda_status_t kda_chunk_fwd_noalloc(const void* q, const void* k, const void* v, int dtype,
                                   const float* g, const void* beta, const float* h0,
                                   const int32_t* cu_seqlens, int n_seqs, int B, int64_t T,
                                   int H, int dk, int dv, void* o, float* hT,
                                   kda_stream_t stream);
/* Capacity in bytes of the array behind kda_chunk_fwd_noalloc. */
size_t kda_chunk_fwd_noalloc_capacity(void);

/*
 * kda_recurrent_step -- decode: one token per sequence, state updated in place
 * (the recurrent form used for cached single-token decode, "Kimi K3:
 * architecture, training and inference systems", sections 11.2 and 13.2), taken
 * in the delta form of section 3.1:
 *     S <- D S + beta k (v^T - k^T D S),  D = Diag(exp(g)),   o = S^T q.
 *
 *   q, k     [N][H][dk], dtype;  v [N][H][dv], dtype;  beta [N][H], dtype
 *   g        [N][H][dk] fp32, any values <= 0
 *   S        [N][H][dv][dk] fp32, read and overwritten in place
 *   o        [N][H][dv], dtype, written
 */
kda_status_t kda_recurrent_step(const void* q, const void* k, const void* v, int dtype,
                                const float* g, const void* beta, float* S, void* o, int N, int H,
                                int dk, int dv, kda_stream_t stream);

/*
 * kda_recurrent_multi_step -- T (1..KDA_MULTI_STEP_MAX_T) tokens per sequence in
 * one pass over the states, for speculative decoding: the verify pass needs the
 * outputs of every draft token, the commit advances the state over the accepted
 * ones only ("Kimi K3: architecture, training and inference systems", section
 * 13.2, speculative verify and replay).  Each token is the recurrence of
 * kda_recurrent_step, applied to the T tokens in order.
 *   q, k, v  [N][T][H][128] of `dtype` (token t of sequence n at row n*T + t)
 *   g        [N][T][H][128] fp32 log-decays (any g <= 0);  beta [N][T][H], dtype
 *   S        [N][H][dv][dk] fp32, in place: the state after the first
 *            n_advance[n] tokens (n_advance: device int32 [N], values clamped to
 *            [0, T]; NULL = all T tokens; 0 leaves the state unchanged)
 *   o        [N][T][H][dv] of `dtype`: outputs of all T tokens computed with the
 *            state evolving through them, whatever n_advance is; may be NULL
 * Errors: as kda_recurrent_step; T outside 1..KDA_MULTI_STEP_MAX_T ->
 * KDA_ERR_UNSUPPORTED_SHAPE (longer runs are prefills: kda_chunk_fwd).
 */
#define KDA_MULTI_STEP_MAX_T 16
kda_status_t kda_recurrent_multi_step(const void* q, const void* k, const void* v, int dtype,
                                      const float* g, const void* beta, float* S, void* o,
                                      const int32_t* n_advance, int N, int T, int H, int dk,
                                      int dv, kda_stream_t stream);

/* Message for the last non-OK status returned on this thread (never NULL). */
const char* kda_last_error_string(void);

/* Reads and clears the device error flag set by the kernels.  Synchronizes
 * `stream`.  Returns KDA_OK; KDA_ERR_DEVICE_TIMEOUT when a bounded device-side
 * wait gave up; KDA_ERR_INVALID_ARG when cu_seqlens was malformed (clamped on
 * the device), more checkpoints than slots were asked for, or the input check
 * (KDA_CHUNK_CHECK_INPUTS) found an out-of-range g or beta. */
kda_status_t kda_get_device_error(kda_stream_t stream);

/*
 * kda_selftest_wait_timeout -- exercises the bounded-wait path that every
 * tensor-core kernel uses (no counterpart on the KDA pages: it is the library's
 * failure-detection self-test).  One CTA of four warps waits, through the same
 * wait routine as the prefill kernels, on a barrier that nothing signals, with
 * a limit of timeout_us microseconds (1 .. 1,000,000), while a real bulk copy is
 * in flight.  The first wait to run out records KDA_ERR_DEVICE_TIMEOUT in the
 * device error flag and raises the CTA's abort word, the other warps stop, the
 * copy is drained, and the kernel returns: nothing is left waiting and the
 * context stays usable.  Synchronizes `stream`; *warps_gave_up (host int) is
 * the number of warps (4 expected) whose wait ended unsatisfied.  The flag is
 * left set for kda_get_device_error to read.
 */
kda_status_t kda_selftest_wait_timeout(uint32_t timeout_us, int* warps_gave_up,
                                       kda_stream_t stream);

/*
 * Per-kernel timing with CUDA events (a tracing aid; off by default).
 * kda_profile_enable(1) clears earlier records and makes every kernel launch of
 * the library record a start and a stop event on the stream it is launched on;
 * kda_profile_enable(0) stops recording (and also clears).  kda_profile_collect()
 * waits for the recorded events and aggregates them per kernel name, returning
 * the number of distinct kernels (or -1 on a CUDA error); kda_profile_get(i, ...)
 * returns kernel i's name (static storage), launch count and total milliseconds.
 * Host-side state is global to the process and guarded by a mutex.
 */
int kda_profile_enable(int on);
int kda_profile_collect(void);
int kda_profile_get(int i, const char** name, int* launches, double* total_ms);

/* Library version, "major.minor.patch". */
const char* kda_version(void);

#ifdef __cplusplus
}
#endif
#endif /* KDA_H_ */
