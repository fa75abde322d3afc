// Instantiations: fused AdamW step, 8-bit m and v, power-of-two quantization blocks of 16..1024
// elements inside the persistent kernel's 2048-element tiles.
#include "psadam_kernels.cuh"

namespace psadam {
#define PSADAM_INST(GB, SR, CAP) template cudaError_t launch_step_sub<kModeQ8, GB, SR, CAP>(const LaunchArgs<CAP>&, cudaStream_t);
#define PSADAM_INST_SR(GB, CAP) PSADAM_INST(GB, false, CAP) PSADAM_INST(GB, true, CAP)
PSADAM_INST_SR(false, kCapSmall)
PSADAM_INST_SR(true, kCapSmall)
PSADAM_INST_SR(false, kCapLarge)
PSADAM_INST_SR(true, kCapLarge)
#undef PSADAM_INST_SR
#undef PSADAM_INST
}  // namespace psadam
