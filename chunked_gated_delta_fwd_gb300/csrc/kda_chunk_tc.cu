// kda_chunk_tc.cu -- bf16 tensor-core (tcgen05) chunk path: not yet enabled;
// bf16 inputs are evaluated by the fp32 CUDA-core kernels meanwhile.
#include "kda_internal.cuh"

namespace kda {

size_t tc_workspace_bytes(int64_t n_tokens, int n_seqs, int H) {
  return simt_workspace_bytes(n_tokens, n_seqs, H);
}

cudaError_t launch_chunk_tc(const void* q, const void* k, const void* v, const float* g,
                            const void* beta, const float* h0, void* o, float* hT,
                            int64_t n_tokens, int n_seqs, int H, void* ws, int* err_flag,
                            cudaStream_t s) {
  (void)err_flag;
  return launch_chunk_simt(q, k, v, 1, g, beta, h0, o, hT, n_tokens, n_seqs, H, ws, s);
}

}  // namespace kda
