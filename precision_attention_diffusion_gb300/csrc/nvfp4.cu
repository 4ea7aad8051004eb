// nvfp4.cu -- NVFP4 (SageAttention3-style) quantize and attention launchers.
#include "fa_lp_internal.h"

namespace falp {

int launch_nvfp4_quantize(const fa_lp_plan&, uint8_t*, const void*, int64_t, int64_t, const void*,
                          int64_t, int64_t, const void*, int64_t, int64_t, cudaStream_t) {
  return FA_LP_ERR_UNSUPPORTED;
}

int launch_nvfp4_attention(const fa_lp_plan&, uint8_t*, void*, int64_t, int64_t, cudaStream_t) {
  return FA_LP_ERR_UNSUPPORTED;
}

}  // namespace falp
