// Tensor-core backward (tcgen05 + TMA) -- not compiled for any shape yet.
#include "fa_internal.h"

namespace fa {
bool have_bwd_tc(int64_t, fa_dtype) { return false; }
fa_status launch_bwd_tc(const BwdParams&, cudaStream_t) { return FA_ERR_ARG; }
}  // namespace fa
