// Tensor-core (tcgen05 / TMEM) split-KV verify attention: placeholder until
// the kernel lands; AUTO resolves to the CUDA-core kernel meanwhile.
#include "common.cuh"

namespace mlav {

int tc_rows_per_group() { return 128; }
int tc_tokens_per_tile() { return 64; }
int tc_units_auto(int sm_count) { return sm_count / 2; }
int tc_default_for(int dtype) { (void)dtype; return MLA_ALGO_SIMT; }

cudaError_t launch_attn_tc(const Params& p, cudaStream_t stream) {
  (void)p;
  (void)stream;
  return cudaErrorNotSupported;
}

}  // namespace mlav
