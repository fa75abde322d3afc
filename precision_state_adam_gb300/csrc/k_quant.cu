// Instantiations: quantize-only / dequantize-only kernels of the 8-bit moment format and the
// non-finite grad check.
#include "psadam_kernels.cuh"

namespace psadam {
#define PSADAM_INST(SR, K, CAP) template cudaError_t launch_quantize<SR, K, CAP>(const LaunchArgs<CAP>&, cudaStream_t);
#define PSADAM_INST_K(SR, CAP) PSADAM_INST(SR, 1, CAP) PSADAM_INST(SR, 3, CAP) PSADAM_INST(SR, 4, CAP) PSADAM_INST(SR, kRankSel, CAP)
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

// ------------------------------------------------------------------ bounded-wait self-test
// One thread waits on an mbarrier that nothing arrives at: the wait gives up after `cycles`
// and the kernel reports it in the fault word, as the step kernels do. Nothing faults and
// nothing hangs; the host then reads the word.
__global__ void psadam_wait_selftest_kernel(int* fault, long long cycles) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_init_fence();
    if (!mbar_wait(&bar, 0u, cycles) && fault != nullptr) atomicExch(fault, 1);
  }
}

cudaError_t launch_wait_selftest(int* fault, long long cycles, cudaStream_t s) {
  psadam_wait_selftest_kernel<<<1, 32, 0, s>>>(fault, cycles);
  return cudaGetLastError();
}
}  // namespace psadam
