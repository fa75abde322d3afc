// Instantiations: fused AdamW step with an fp32 first moment and an 8-bit second moment,
// stochastic rounding.
#include "psadam_kernels.cuh"

namespace psadam {
#define PSADAM_INST(GB, K, CAP) template cudaError_t launch_step<kModeQ8V, GB, true, K, CAP>(const LaunchArgs<CAP>&, cudaStream_t);
#define PSADAM_INST_K(GB, CAP) PSADAM_INST(GB, 1, CAP) PSADAM_INST(GB, 3, CAP) PSADAM_INST(GB, 4, CAP) PSADAM_INST(GB, kRankSel, CAP)
PSADAM_INST_K(false, kCapSmall)
PSADAM_INST_K(true, kCapSmall)
PSADAM_INST_K(false, kCapLarge)
PSADAM_INST_K(true, kCapLarge)
#undef PSADAM_INST_K
#undef PSADAM_INST
}  // namespace psadam
