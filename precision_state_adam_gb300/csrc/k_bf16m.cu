// Instantiations: fused AdamW step with bf16 moments (fp32 or bf16 grads).
#include "psadam_kernels.cuh"

namespace psadam {
#define PSADAM_INST(GB, CAP) template cudaError_t launch_step<kModeBF16, GB, false, 1, CAP>(const LaunchArgs<CAP>&, cudaStream_t);
PSADAM_INST(false, kCapSmall)
PSADAM_INST(true, kCapSmall)
PSADAM_INST(false, kCapLarge)
PSADAM_INST(true, kCapLarge)
#undef PSADAM_INST
}  // namespace psadam
