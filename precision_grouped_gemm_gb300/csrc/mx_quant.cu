// MX quantize kernels (row-wise and group-aware column-wise).
#include "internal.h"

namespace pgg {
int launch_mx_quantize_rowwise(const void*, int64_t, int64_t, int, uint8_t*, uint8_t*, cudaStream_t) {
  return PGG_ERR_UNSUPPORTED;
}
int launch_mx_quantize_colwise(const void*, int64_t, int64_t, const int32_t*, int, int, uint8_t*,
                               uint8_t*, int64_t, int32_t*, cudaStream_t) {
  return PGG_ERR_UNSUPPORTED;
}
}  // namespace pgg
