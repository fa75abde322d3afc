// Instantiations: any block size / any percentile rank, 8-bit m and v, stochastic rounding.
#include "psadam_kernels.cuh"

namespace psadam {
#define PSADAM_INST(GB, CAP) template cudaError_t launch_step_any<kModeQ8, GB, true, CAP>(const LaunchArgs<CAP>&, cudaStream_t);
PSADAM_INST(false, kCapSmall)
PSADAM_INST(true, kCapSmall)
PSADAM_INST(false, kCapLarge)
PSADAM_INST(true, kCapLarge)
#undef PSADAM_INST
}  // namespace psadam
