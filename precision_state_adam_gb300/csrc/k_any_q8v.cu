// Instantiations: any block size / any percentile rank, fp32 m with 8-bit v.
#include "psadam_kernels.cuh"

namespace psadam {
#define PSADAM_INST(GB, SR, CAP) template cudaError_t launch_step_any<kModeQ8V, GB, SR, CAP>(const LaunchArgs<CAP>&, cudaStream_t);
#define PSADAM_INST_CAP(GB, SR) PSADAM_INST(GB, SR, kCapSmall) PSADAM_INST(GB, SR, kCapLarge)
PSADAM_INST_CAP(false, false)
PSADAM_INST_CAP(false, true)
PSADAM_INST_CAP(true, false)
PSADAM_INST_CAP(true, true)
#undef PSADAM_INST_CAP
#undef PSADAM_INST
}  // namespace psadam
