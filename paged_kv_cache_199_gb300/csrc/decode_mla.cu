// MLA decode kernel (filled in after the GQA path).
#include "kernels.h"
namespace pd {
cudaError_t launch_mla_decode(const CUtensorMap&, const MlaParams&, int, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace pd
