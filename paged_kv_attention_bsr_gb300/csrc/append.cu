// append.cu -- causal / non-causal append (prefill) attention on tcgen05.
#include "internal.h"

namespace attn {

int append_ctas_per_sm() { return 1; }

cudaError_t launch_append(const AppendArgs& a, cudaStream_t stream, const char** msg) {
  (void)a;
  (void)stream;
  *msg = "attn_append_run: the append kernel is not built yet";
  return cudaErrorNotSupported;
}

}  // namespace attn
