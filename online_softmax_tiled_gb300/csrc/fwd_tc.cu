// bf16 forward entry (tcgen05 kernel under construction; routes to the FFMA kernel).
#include "common.cuh"
#include "launchers.h"

namespace attn {
ATTN_DEFINE_ERROR_WORD(take_error_fwd_tc)
cudaError_t launch_fwd_tc(const FwdArgs& a) { return launch_fwd_simt(a); }
}  // namespace attn
