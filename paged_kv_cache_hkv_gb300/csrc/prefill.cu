// Tensor-core (tcgen05) causal prefill attention over the paged cache: not
// built yet; the launcher reports the path as unsupported.
#include "common.cuh"
#include "launch.h"

namespace pkv {

static __device__ uint32_t g_errors_prefill;

cudaError_t launch_prefill(const AttnArgs&, const AttnWorkspace&, const CUtensorMap&,
                           const CUtensorMap&, int, cudaStream_t) {
  return cudaErrorNotSupported;
}

cudaError_t read_errors_prefill(uint32_t* out, bool clear) {
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_errors_prefill, sizeof(v));
  if (e != cudaSuccess) return e;
  *out |= v;
  if (clear) {
    const uint32_t z = 0;
    e = cudaMemcpyToSymbol(g_errors_prefill, &z, sizeof(z));
  }
  return e;
}

}  // namespace pkv
