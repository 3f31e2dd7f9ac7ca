// Prefill sink attention (placeholder until the tcgen05 kernel lands).
#include "attn_internal.h"
#include "kernels.h"

namespace attn {
attn_status launch_prefill(attn_plan_s*, const void*, const void*, const float*, void*, float*,
                           cudaStream_t) {
    return ATTN_ERR_UNSUPPORTED;
}
}  // namespace attn
