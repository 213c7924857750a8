// tcgen05 / TMEM / TMA chunkwise GLA forward (placeholder until the kernel lands).
#include "gla_internal.h"

namespace gla {

bool tc_supported(const Problem &) { return false; }
int tc_auto_splits(const Problem &, int) { return 1; }
size_t tc_workspace_bytes(const Problem &, int) { return 0; }
cudaError_t launch_tc(const Problem &, int, void *, size_t, unsigned int *, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace gla
