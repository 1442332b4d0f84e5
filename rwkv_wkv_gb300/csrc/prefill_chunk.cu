// Chunked WKV-7 prefill (placeholder: routes to the sequential kernel until the
// tensor-core chunked kernel lands).
#include "wkv7_internal.h"

namespace wkv7 {
cudaError_t launch_prefill_chunked(const PrefillArgs &a, cudaStream_t s, int *launches) {
    return launch_prefill_sequential(a, s, launches);
}
}  // namespace wkv7
