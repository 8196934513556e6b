// Tensor-core (tcgen05 / TMEM / TMA) forward of the Lizard token mixer: not built yet.
#include "internal.h"

namespace lz {

bool fwd_tc_supported(const Plan&) { return false; }

cudaError_t launch_fwd_tc(const Plan&, const FwdArgs&, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace lz
