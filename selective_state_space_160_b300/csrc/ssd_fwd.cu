// ssd_fwd.cu -- SSD chunked forward (placeholder until the kernels land).
#include "msc_common.cuh"
#include "msc_internal.h"

namespace msc_host {
size_t ssd_workspace(int64_t, int64_t, int64_t, int64_t, int64_t, int64_t, int64_t) { return 1024; }
msc_status ssd_take_status(unsigned int* code, unsigned int* site) {
    *code = 0;
    *site = 0;
    return MSC_OK;
}
msc_status ssd_launch(const SsdArgs&, cudaStream_t) {
    return fail(MSC_ERR_UNSUPPORTED, "SSD forward not built yet");
}
}  // namespace msc_host
