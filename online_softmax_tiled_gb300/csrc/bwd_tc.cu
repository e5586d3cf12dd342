// bf16 backward entry (tcgen05 kernel under construction; routes to the FFMA kernel).
#include "common.cuh"
#include "launchers.h"

namespace attn {
ATTN_DEFINE_ERROR_WORD(take_error_bwd_tc)
cudaError_t launch_bwd_tc(const BwdArgs& a) { return launch_bwd_simt(a); }
}  // namespace attn
