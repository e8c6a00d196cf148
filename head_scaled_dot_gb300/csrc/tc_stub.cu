// tc_stub.cu - placeholder bf16 attention entry point routed to the CUDA-core
// kernel until the tensor-core attention kernel lands.
#include "internal.h"

namespace mha {
mha_status attention_tc(const AttnArgs& a, cudaStream_t s) {
  return attention_simt(a, MHA_DTYPE_BF16, s);
}
}  // namespace mha
