// tc_stub.cu - placeholder bf16 entry points routed to the CUDA-core kernels
// until the tensor-core kernels land.
#include "internal.h"

namespace mha {
mha_status gemm_tc(const GemmProblem* probs, int nprob, int32_t*, cudaStream_t s) {
  return gemm_simt(probs, nprob, MHA_DTYPE_BF16, s);
}
mha_status attention_tc(const AttnArgs& a, cudaStream_t s) {
  return attention_simt(a, MHA_DTYPE_BF16, s);
}
}  // namespace mha
