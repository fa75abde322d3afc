// Instantiations: any block size / any percentile rank (8-bit moments, both layouts).
#include "psadam_kernels.cuh"

namespace psadam {
#define PSADAM_INST(MODE, GB, SR, CAP) template cudaError_t launch_step_any<MODE, GB, SR, CAP>(const LaunchArgs<CAP>&, cudaStream_t);
#define PSADAM_INST_CAP(MODE, GB, SR) PSADAM_INST(MODE, GB, SR, kCapSmall) PSADAM_INST(MODE, GB, SR, kCapLarge)
PSADAM_INST_CAP(kModeQ8, false, false)
PSADAM_INST_CAP(kModeQ8, false, true)
PSADAM_INST_CAP(kModeQ8, true, false)
PSADAM_INST_CAP(kModeQ8, true, true)
#undef PSADAM_INST_CAP
#undef PSADAM_INST
template cudaError_t launch_quantize_any<false, kCapSmall>(const LaunchArgs<kCapSmall>&, cudaStream_t);
template cudaError_t launch_quantize_any<true, kCapSmall>(const LaunchArgs<kCapSmall>&, cudaStream_t);
template cudaError_t launch_quantize_any<false, kCapLarge>(const LaunchArgs<kCapLarge>&, cudaStream_t);
template cudaError_t launch_quantize_any<true, kCapLarge>(const LaunchArgs<kCapLarge>&, cudaStream_t);
template cudaError_t launch_dequantize_any<kCapSmall>(const LaunchArgs<kCapSmall>&, cudaStream_t);
template cudaError_t launch_dequantize_any<kCapLarge>(const LaunchArgs<kCapLarge>&, cudaStream_t);
}  // namespace psadam
