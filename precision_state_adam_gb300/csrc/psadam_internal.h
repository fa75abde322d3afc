// psadam_internal.h — launch-argument layout shared by the host API and the kernel
// translation units of libpsadam.so (not installed; the public ABI is include/psadam.h).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace psadam {

constexpr int kBlock = 2048;   // quantization block = elements handled by one CTA
constexpr int kThreads = 256;  // threads per CTA
constexpr int kVec = 4;        // consecutive elements per thread per group (one 16-byte fp32 vector)
constexpr int kGroups = kBlock / (kThreads * kVec);  // 2 groups of 4 elements per thread
constexpr int kWarps = kThreads / 32;

// Tensor-list capacities of one launch: small lists use a small kernel-parameter block,
// long lists the largest block that stays under the 32,764-byte parameter limit.
constexpr int kCapSmall = 8;
constexpr int kCapLarge = 440;
// Largest percentile rank k the 2048-block kernels select: ranks 2 and 3 by per-lane top-3
// lists and warp extraction, rank 4 by top-4 lists, ranks 5..32 from sorted thread maxima and
// a gathered candidate set (block_rank_stats); higher ranks run the general kernel's radix
// select.
constexpr int kMaxRank = 32;
constexpr int kRankSel = 32;  // rank template of ranks 5..32
// Largest quantization block of the any-block-size kernels (its fp32 m', v' are staged in
// shared memory: 128 KB for both moments).
constexpr int kMaxAnyBlock = 16384;
// The general kernels' CTA takes a tile of whole blocks: as many as fit 2048 elements, at
// most kAnyMaxQ of them (one block when B > 2048).
constexpr int kAnyMaxQ = 64;
constexpr int kAnyTile = 2048;
constexpr int any_blocks_per_tile(int B) {
  return B >= kAnyTile ? 1 : (kAnyTile / B < kAnyMaxQ ? kAnyTile / B : kAnyMaxQ);
}
// Blocks larger than the general kernel's tile with absmax scales (rank 1), whose C channels
// would take more than 32 KB of staging (fewer than 4 CTAs per SM), are not staged in shared
// memory: the kernel reads each block twice instead (moments, then the whole update).
__host__ __device__ constexpr bool any_recompute(int tile, int k_full, int channels) {
  return tile > kAnyTile && k_full == 1 && tile * channels > 8192;
}

enum Mode : int { kModeF32 = 0, kModeBF16 = 1, kModeQ8 = 2, kModeQ8V = 3 };  // Q8V: fp32 m, 8-bit v

// Per-step fp32 constants (formed in double on the host, rounded once).
struct StepConsts {
  float b1, omb1, b2, omb2, decay, step_size, inv_sqrt_bc2, eps;
  int fast_root;  // eps and inv_sqrt_bc2 allow the update's fused root and quotient (adamw_n)
};

// One non-empty tensor of the list. For the quantize-only kernel p/g are unused and
// m/v are the fp32 inputs; for dequantize-only m/v are the fp32 outputs and the codes
// travel in g (m codes) and p (v codes).
struct TensorRef {
  float* p;
  const void* g;
  void* m;
  void* v;
  float* ms;
  float* vs;
  long long numel;
  int block_begin;  // index of this tensor's first CTA within the launch
  int k_last;       // percentile rank of the tensor's last block (may be partial)
  int list_idx;     // position in the caller's list (stochastic-rounding stream)
  int grp_off;      // first element / 4 within the caller's whole tensor (nonzero for a slice
                    // of one): added to the stochastic-rounding counter
};

template <int CAP>
struct LaunchArgs {
  StepConsts c;
  uint32_t seed_lo, seed_hi, step_lo;
  int k_full;       // percentile rank of a full 2048-element block
  int n_tensors;
  int total_blocks;
  float g_unscale;  // grads are multiplied by this before use (1: unchanged)
  int zero_grads;   // nonzero: overwrite each grad with zero after reading it
  const int* skip;  // device flag or null: a nonzero value makes the launch a no-op
  int* fault;       // device word set to 1 when a bounded wait gives up (see psadam_device_fault)
  int static_scales;  // 8-bit: a block's nonzero scale is kept instead of recomputed
  int block_size;     // 8-bit quantization block (the 2048-block kernels assume 2048)
  int block_shift;    // log2(block_size) when it is a power of two (the sub-block path)
  int tile;           // elements per CTA (a whole number of blocks)
  int approx;         // nonzero: approximate square root and division in the update
  TensorRef t[CAP];
};
static_assert(sizeof(LaunchArgs<kCapLarge>) <= 32764, "kernel parameter block too large");

// Rank templates: K = 1 (absmax), 3 (k-th largest for k = 2, 3: percentile 99.9 on full
// blocks), 4 (k = 4) or kRankSel (k = 5 .. 32: percentile 98.5 and up on full blocks).
constexpr int rank_template(int k) { return k <= 1 ? 1 : (k <= 3 ? 3 : (k == 4 ? 4 : kRankSel)); }

// Launchers, explicitly instantiated in the kernel translation units.
template <int MODE, bool GBF16, bool SR, int K, int CAP>
cudaError_t launch_step(const LaunchArgs<CAP>& a, cudaStream_t s);

template <bool SR, int K, int CAP>
cudaError_t launch_quantize(const LaunchArgs<CAP>& a, cudaStream_t s);

template <int CAP>
cudaError_t launch_dequantize(const LaunchArgs<CAP>& a, cudaStream_t s);

// Power-of-two block sizes in [kMinSubBlock, kMaxSubBlock] with rank 1 and the plain or
// approximate update: the persistent kernel, several blocks per 2048-element tile.
constexpr int kMinSubBlock = 16;
constexpr int kMaxSubBlock = 1024;
template <int MODE, bool GBF16, bool SR, int CAP>
cudaError_t launch_step_sub(const LaunchArgs<CAP>& a, cudaStream_t s);

// Any block size in [1, kMaxAnyBlock] and any percentile rank: one CTA per quantization block.
template <int MODE, bool GBF16, bool SR, int CAP>
cudaError_t launch_step_any(const LaunchArgs<CAP>& a, cudaStream_t s);

template <bool SR, int CAP>
cudaError_t launch_quantize_any(const LaunchArgs<CAP>& a, cudaStream_t s);

template <int CAP>
cudaError_t launch_dequantize_any(const LaunchArgs<CAP>& a, cudaStream_t s);

// Bounded-wait self-test: a wait that nothing completes gives up after `cycles`, sets *fault.
cudaError_t launch_wait_selftest(int* fault, long long cycles, cudaStream_t s);
cudaError_t launch_math_selftest(int full, const StepConsts* c, int n_c, unsigned long long* out, cudaStream_t s);

// Non-finite grad check: sets *flag = 1 if any grad (times g_unscale) is inf or NaN.
template <bool GBF16, int CAP>
cudaError_t launch_check_grads(const LaunchArgs<CAP>& a, int* flag, cudaStream_t s);

}  // namespace psadam
