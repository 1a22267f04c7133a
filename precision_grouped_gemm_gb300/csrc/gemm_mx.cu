// Block-scaled (MX) grouped GEMM.
#include "internal.h"

namespace pgg {
int launch_mx_gemm(const MxCall&) { return PGG_ERR_UNSUPPORTED; }
}  // namespace pgg
