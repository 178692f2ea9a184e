// Placeholder until the tcgen05 chunk kernel lands: routes to the CUDA-core kernel.
#include "internal.cuh"
namespace efla {
cudaError_t launch_chunk_tc(const FwdArgs &a, const char **why) {
    *why = "recurrent kernel launch";
    return launch_recurrent(a);
}
}  // namespace efla
