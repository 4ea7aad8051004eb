// nvfp4.cu -- NVFP4 attention launcher (the tcgen05 kind::mxf4nvf4 kernel is not built yet; the
// call returns FA_LP_ERR_UNSUPPORTED, never a fallback).
#include "fa_lp_internal.h"

namespace falp {

int launch_nvfp4_attention(const fa_lp_plan&, uint8_t*, void*, int64_t, int64_t, cudaStream_t) {
  return FA_LP_ERR_UNSUPPORTED;
}

}  // namespace falp
