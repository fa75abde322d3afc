// Instantiations: fused AdamW step with 8-bit moments, Philox stochastic rounding.
#include "psadam_kernels.cuh"

namespace psadam {
#define PSADAM_INST(GB, K, CAP) template cudaError_t launch_step<kModeQ8, GB, true, K, CAP>(const LaunchArgs<CAP>&, cudaStream_t);
#define PSADAM_INST_K(GB, CAP) PSADAM_INST(GB, 1, CAP) PSADAM_INST(GB, 3, CAP) PSADAM_INST(GB, 4, CAP) PSADAM_INST(GB, kRankSel, CAP)
PSADAM_INST_K(false, kCapSmall)
PSADAM_INST_K(true, kCapSmall)
PSADAM_INST_K(false, kCapLarge)
PSADAM_INST_K(true, kCapLarge)
#undef PSADAM_INST_K
#undef PSADAM_INST
}  // namespace psadam
