// Instantiations: fused AdamW step with an fp32 first moment and an 8-bit second moment.
#include "psadam_kernels.cuh"

namespace psadam {
#define PSADAM_INST(GB, SR, K, CAP) template cudaError_t launch_step<kModeQ8V, GB, SR, K, CAP>(const LaunchArgs<CAP>&, cudaStream_t);
#define PSADAM_INST_K(GB, SR, CAP) PSADAM_INST(GB, SR, 1, CAP) PSADAM_INST(GB, SR, 3, CAP) PSADAM_INST(GB, SR, 4, CAP)
PSADAM_INST_K(false, false, kCapSmall)
PSADAM_INST_K(true, false, kCapSmall)
PSADAM_INST_K(false, false, kCapLarge)
PSADAM_INST_K(true, false, kCapLarge)
PSADAM_INST_K(false, true, kCapSmall)
PSADAM_INST_K(true, true, kCapSmall)
PSADAM_INST_K(false, true, kCapLarge)
PSADAM_INST_K(true, true, kCapLarge)
#undef PSADAM_INST_K
#undef PSADAM_INST
}  // namespace psadam
