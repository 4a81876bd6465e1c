// gdn_prof.h -- launch bookkeeping for the optional per-kernel timing of the
// C ABI (gdn_profile_*): every kernel launch of the library goes through
// prof_begin / prof_end, which count it and, while profiling is on, record a
// CUDA event pair on the launching stream around it.
#pragma once
#include <cuda_runtime.h>

namespace gdn {
enum KernelId {
  K_TABLES_SCAN = 0, K_TABLES_FILL, K_PREP, K_FWD_WALK, K_FWD_MERGE, K_FWD_SCAN,
  K_CHECK_SAVED, K_BWD_WALK, K_BWD_MERGE, K_BWD_SCAN, K_GRAD, K_PASS, K_CONV_FWD, K_CONV_BWD, K_VNEW,
  K_KDA_PREP, K_KDA_OUT, K_KDA_GRAD, K_WALK_ORDER, K_NUM
};
void prof_begin(int id, cudaStream_t s);
void prof_end(int id, cudaStream_t s);
}  // namespace gdn
