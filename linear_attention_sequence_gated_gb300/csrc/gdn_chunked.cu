// Chunked path placeholder: not built yet, so AUTO never selects it.
#include "gdn_internal.h"

namespace gdn {
bool chunked_supports(int) { return false; }
size_t chunked_workspace_bytes(int, int, int, int, int) { return 0; }
cudaError_t launch_chunked(const Problem &, void *, size_t, cudaStream_t) {
    return cudaErrorNotSupported;
}
}  // namespace gdn
