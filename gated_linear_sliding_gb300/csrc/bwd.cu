// Backward of the Lizard token mixer: not built yet.
#include "internal.h"

namespace lz {

size_t bwd_workspace_bytes(const Plan&) { return kHeaderBytes; }

cudaError_t launch_bwd(const Plan&, const BwdArgs&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace lz
