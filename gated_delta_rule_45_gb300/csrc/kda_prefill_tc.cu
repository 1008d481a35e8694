// Tensor-core (tcgen05 / TMEM / TMA) chunkwise KDA prefill: placeholder until
// the kernel lands; reports every shape as not covered.
#include "kda_internal.h"

namespace kda {

bool prefill_tc_supports(const PrefillArgs&) { return false; }

cudaError_t launch_prefill_tc(const PrefillArgs&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace kda
