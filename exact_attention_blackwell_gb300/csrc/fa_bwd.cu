// fa_bwd.cu — fused attention backward for sm_103a (in progress).
#include "fa_internal.h"

namespace fa {

int launch_bwd(const BwdParams &, int, bool, const void *, const void *, const float *, void *, float *, float *,
               cudaStream_t) {
  return FA_ERR_UNSUPPORTED;
}

}  // namespace fa
