// pa_tile.cu -- tensor-core (tcgen05) tile kernel for bf16 extend/prefill.
// Until it lands, extend/prefill rows take the row-streaming kernel.
#include "pa_internal.h"

namespace pa {

bool tile_kernel_supported(int, int, int) { return false; }

cudaError_t launch_tile_kernel(const FwdParams &, const CUtensorMap &, const CUtensorMap &,
                               const CUtensorMap &, int, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace pa
