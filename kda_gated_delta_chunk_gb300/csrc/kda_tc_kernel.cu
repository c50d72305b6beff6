// tcgen05 + TMA chunk kernel (KDA_KERNEL_TC) -- under construction.
#include "kda_internal.cuh"

namespace kda {
cudaError_t launch_tc(const Params&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace kda
