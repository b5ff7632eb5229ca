// Tensor-core (tcgen05/TMEM) chunkwise prefill: not built yet.
#include "kda_internal.cuh"

namespace kda {

bool prefill_tc_supported(const PrefillArgs &) { return false; }

cudaError_t launch_prefill_tc(const PrefillArgs &, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace kda
