// Instantiations: any block size / any percentile rank, 8-bit m and v, round to nearest even;
// quantize-only and dequantize-only for any block size.
#include "psadam_kernels.cuh"

namespace psadam {
#define PSADAM_INST(GB, CAP) template cudaError_t launch_step_any<kModeQ8, GB, false, CAP>(const LaunchArgs<CAP>&, cudaStream_t);
PSADAM_INST(false, kCapSmall)
PSADAM_INST(true, kCapSmall)
PSADAM_INST(false, kCapLarge)
PSADAM_INST(true, kCapLarge)
#undef PSADAM_INST
template cudaError_t launch_quantize_any<false, kCapSmall>(const LaunchArgs<kCapSmall>&, cudaStream_t);
template cudaError_t launch_quantize_any<true, kCapSmall>(const LaunchArgs<kCapSmall>&, cudaStream_t);
template cudaError_t launch_quantize_any<false, kCapLarge>(const LaunchArgs<kCapLarge>&, cudaStream_t);
template cudaError_t launch_quantize_any<true, kCapLarge>(const LaunchArgs<kCapLarge>&, cudaStream_t);
template cudaError_t launch_dequantize_any<kCapSmall>(const LaunchArgs<kCapSmall>&, cudaStream_t);
template cudaError_t launch_dequantize_any<kCapLarge>(const LaunchArgs<kCapLarge>&, cudaStream_t);
}  // namespace psadam
