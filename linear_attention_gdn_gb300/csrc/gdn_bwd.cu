// gdn_bwd.cu -- backward kernels (placeholder until they land)
#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn.h"
namespace gdn {
void setup_bwd_attrs() {}
gdn_status run_bwd(const Plan&, const gdn_problem&, const void*, const void*, const void*, const float*,
                   const float*, const int32_t*, const void*, const void*, void*, void*, void*, float*, float*,
                   uint8_t*, cudaStream_t) {
  return GDN_ERR_UNSUPPORTED;
}
}  // namespace gdn
