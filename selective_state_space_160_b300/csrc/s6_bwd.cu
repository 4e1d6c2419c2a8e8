// s6_bwd.cu -- S6 backward (placeholder until the kernel lands).
#include "msc_common.cuh"
#include "msc_internal.h"

namespace msc_host {
size_t s6_bwd_workspace(int64_t, int64_t, int64_t, int64_t) { return 0; }
msc_status s6_bwd_launch(const S6BwdArgs&, cudaStream_t) {
    return fail(MSC_ERR_UNSUPPORTED, "S6 backward not built yet");
}
}  // namespace msc_host
