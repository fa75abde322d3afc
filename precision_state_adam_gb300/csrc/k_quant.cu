// Instantiations: quantize-only / dequantize-only kernels of the 8-bit moment format and the
// non-finite grad check.
#include "psadam_kernels.cuh"

namespace psadam {
#define PSADAM_INST(SR, K, CAP) template cudaError_t launch_quantize<SR, K, CAP>(const LaunchArgs<CAP>&, cudaStream_t);
#define PSADAM_INST_K(SR, CAP) PSADAM_INST(SR, 1, CAP) PSADAM_INST(SR, 4, CAP)
PSADAM_INST_K(false, kCapSmall)
PSADAM_INST_K(true, kCapSmall)
PSADAM_INST_K(false, kCapLarge)
PSADAM_INST_K(true, kCapLarge)
#undef PSADAM_INST_K
#undef PSADAM_INST
template cudaError_t launch_dequantize<kCapSmall>(const LaunchArgs<kCapSmall>&, cudaStream_t);
template cudaError_t launch_dequantize<kCapLarge>(const LaunchArgs<kCapLarge>&, cudaStream_t);
template cudaError_t launch_check_grads<false, kCapSmall>(const LaunchArgs<kCapSmall>&, int*, cudaStream_t);
template cudaError_t launch_check_grads<true, kCapSmall>(const LaunchArgs<kCapSmall>&, int*, cudaStream_t);
template cudaError_t launch_check_grads<false, kCapLarge>(const LaunchArgs<kCapLarge>&, int*, cudaStream_t);
template cudaError_t launch_check_grads<true, kCapLarge>(const LaunchArgs<kCapLarge>&, int*, cudaStream_t);
}  // namespace psadam
