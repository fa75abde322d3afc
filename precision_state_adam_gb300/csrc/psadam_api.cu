// psadam_api.cu — the C ABI declared in include/psadam.h: argument validation, the
// per-step constants, tensor-list packing into launch-parameter blocks, and dispatch to
// the kernel instantiations. No device memory is allocated here.
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#include "psadam.h"
#include "psadam_internal.h"

using namespace psadam;

// Set to 1 by a kernel whose bounded wait gave up (read and cleared by psadam_device_fault).
// A module variable: the library still allocates no device memory.
__device__ int g_psadam_fault = 0;
// Where psadam_device_fault's one-thread kernel leaves the value it took out of g_psadam_fault.
__device__ int g_psadam_fault_taken = 0;

// Read and clear the fault word in one atomic exchange, so a fault set meanwhile is either
// taken now or left for the next read.
__global__ void psadam_take_fault_kernel() { g_psadam_fault_taken = atomicExch(&g_psadam_fault, 0); }

namespace {

thread_local int32_t g_last_cuda_error = 0;

// Device address of g_psadam_fault in the current context. Looked up on every call (no cache,
// so a context made anew after cudaDeviceReset gets its own address).
int* fault_word() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_psadam_fault) != cudaSuccess) return nullptr;
  return static_cast<int*>(p);
}

// The step kernels' own limit on a bounded wait, in SM cycles (about a second).
constexpr long long kMaxWaitCycles = 1LL << 31;

// Largest tensor whose block count fits a grid dimension.
constexpr long long kMaxNumel = (long long)INT_MAX * kBlock;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool finite(float x) { return std::isfinite(x); }

struct Entry {
  float* p;
  const void* g;
  void* m;
  void* v;
  float* ms;
  float* vs;
  long long numel;
  int list_idx;
  long long elem_off = 0;  // a slice's first element within its whole tensor (a multiple of 4)
};

int check_hparams(const psadam_hparams* hp, int64_t step) {
  if (!hp || step < 1) return PSADAM_ERR_INVALID_ARG;
  if (!finite(hp->lr) || !finite(hp->beta1) || !finite(hp->beta2) || !finite(hp->eps) ||
      !finite(hp->weight_decay))
    return PSADAM_ERR_INVALID_ARG;
  if (hp->beta1 < 0.f || hp->beta1 >= 1.f || hp->beta2 < 0.f || hp->beta2 >= 1.f || hp->eps < 0.f)
    return PSADAM_ERR_INVALID_ARG;
  return PSADAM_OK;
}

int check_block_size(int32_t bs) {
  if (bs < 1) return PSADAM_ERR_INVALID_ARG;
  if (bs > kMaxAnyBlock) return PSADAM_ERR_UNSUPPORTED;
  return PSADAM_OK;
}

int check_q8(const psadam_q8_opts* q) {
  if (!q) return PSADAM_ERR_INVALID_ARG;
  const int st = check_block_size(q->block_size);
  if (st != PSADAM_OK) return st;
  if (q->stochastic_rounding != 0 && q->stochastic_rounding != 1) return PSADAM_ERR_INVALID_ARG;
  if (!finite(q->percentile) || !(q->percentile > 0.f) || q->percentile > 100.f) return PSADAM_ERR_INVALID_ARG;
  if (q->static_scales != 0 && q->static_scales != 1) return PSADAM_ERR_INVALID_ARG;
  return PSADAM_OK;
}

// Per-step constants: bias corrections 1 - beta^t from pow() in double (the 8-bit Adam
// PR's UpdateParameters forms them with Math.Pow on doubles), each constant rounded
// once to fp32.
StepConsts make_consts(const psadam_hparams& hp, int64_t t) {
  const double lr = hp.lr, b1 = hp.beta1, b2 = hp.beta2, wd = hp.weight_decay;
  const double bc1 = 1.0 - std::pow(b1, (double)t);
  const double bc2 = 1.0 - std::pow(b2, (double)t);
  StepConsts c;
  c.b1 = hp.beta1;
  c.omb1 = (float)(1.0 - b1);
  c.b2 = hp.beta2;
  c.omb2 = (float)(1.0 - b2);
  c.decay = (float)(1.0 - lr * wd);
  c.step_size = (float)(lr / bc1);
  c.inv_sqrt_bc2 = (float)(1.0 / std::sqrt(bc2));
  c.eps = hp.eps;
  // the domain of the update's own correctly rounded root and quotient (psadam_kernels.cuh)
  c.fast_root = c.eps >= 0x1p-60f && c.eps <= 0x1p20f && c.inv_sqrt_bc2 >= 0x1p-20f && c.inv_sqrt_bc2 <= 0x1p20f;
  return c;
}

// Nearest-rank percentile as a position from the top: k = n - ceil(pct*n/100) + 1.
int percentile_rank(float pct, long long n) {
  long long from_bottom = (long long)std::ceil((double)pct * (double)n / 100.0);
  long long k = n - from_bottom + 1;
  if (k < 1) k = 1;
  if (k > n) k = n;
  return (int)k;
}

long long n_blocks(long long n, int bs = kBlock) { return (n + bs - 1) / bs; }
int last_block_len(long long n, int bs = kBlock) { return (int)(n - (n_blocks(n, bs) - 1) * bs); }

// Validate one tensor's pointers. `ptrs` lists the ones that must be present.
int check_tensor(long long numel, std::initializer_list<const void*> ptrs) {
  if (numel < 0) return PSADAM_ERR_INVALID_ARG;
  if (numel == 0) return PSADAM_OK;
  if (numel > kMaxNumel) return PSADAM_ERR_UNSUPPORTED;
  for (const void* p : ptrs)
    if (!p) return PSADAM_ERR_INVALID_ARG;
  for (const void* p : ptrs)
    if (!aligned16(p)) return PSADAM_ERR_MISALIGNED;
  return PSADAM_OK;
}

// Highest percentile rank any block of the list needs.
int max_rank(const std::vector<Entry>& es, float pct, int bs) {
  int k = 1;
  for (const Entry& e : es) {
    if (e.numel >= bs) k = std::max(k, percentile_rank(pct, bs));
    k = std::max(k, percentile_rank(pct, last_block_len(e.numel, bs)));
  }
  return k;
}

// Every tensor's block count must fit a grid dimension.
int check_block_counts(const std::vector<Entry>& es, int bs) {
  for (const Entry& e : es)
    if (n_blocks(e.numel, bs) > INT_MAX) return PSADAM_ERR_UNSUPPORTED;
  return PSADAM_OK;
}

template <int CAP>
using Launcher = cudaError_t (*)(const LaunchArgs<CAP>&, cudaStream_t);

// Grad-side options of a step (see psadam_list).
struct GradSide {
  float unscale = 1.0f;
  int zero = 0;
  const int* skip = nullptr;
  int static_scales = 0;  // not grad-side, but carried the same way into the launch
  int approx = 0;         // likewise: approximate square root and division in the update
};

// Pack the list into as few launches as fit and run `fn` on each.
// bs: quantization block; unit: elements per CTA (bs for the 2048-block kernels, a tile of
// whole blocks for the general ones).
template <int CAP, typename Fn>
int run_launches(const std::vector<Entry>& es, const StepConsts& c, uint64_t seed, int64_t step, float pct,
                 const GradSide& gs, Fn fn, cudaStream_t stream, int bs = kBlock, int unit = 0) {
  if (unit == 0) unit = bs;
  static thread_local LaunchArgs<CAP> a;  // ~32 KB: keep it off the stack
  std::memset(&a, 0, sizeof a);
  a.c = c;
  a.g_unscale = gs.unscale;
  a.zero_grads = gs.zero;
  a.skip = gs.skip;
  a.static_scales = gs.static_scales;
  a.approx = gs.approx;
  a.fault = fault_word();
  a.seed_lo = (uint32_t)(seed & 0xFFFFFFFFu);
  a.seed_hi = (uint32_t)(seed >> 32);
  a.step_lo = (uint32_t)step;
  a.block_size = bs;
  a.block_shift = 0;
  while ((1 << a.block_shift) < bs && a.block_shift < 30) ++a.block_shift;
  a.tile = unit;
  a.k_full = percentile_rank(pct, bs);
  size_t i = 0;
  while (i < es.size()) {
    int nt = 0;
    long long blocks = 0;
    while (i < es.size() && nt < CAP) {
      const long long nb = n_blocks(es[i].numel, unit);
      if (blocks + nb > INT_MAX) break;
      TensorRef& t = a.t[nt++];
      t.p = es[i].p;
      t.g = es[i].g;
      t.m = es[i].m;
      t.v = es[i].v;
      t.ms = es[i].ms;
      t.vs = es[i].vs;
      t.numel = es[i].numel;
      t.block_begin = (int)blocks;
      t.k_last = percentile_rank(pct, last_block_len(es[i].numel, bs));
      t.list_idx = es[i].list_idx;
      t.grp_off = (int)(es[i].elem_off / 4);
      blocks += nb;
      ++i;
    }
    a.n_tensors = nt;
    a.total_blocks = (int)blocks;
    const cudaError_t err = fn(a, stream);
    if (err != cudaSuccess) {
      g_last_cuda_error = (int32_t)err;
      return PSADAM_ERR_CUDA;
    }
  }
  return PSADAM_OK;
}

#define PSADAM_STEP_FN(MODE, GB, SR, K, CAP) &launch_step<MODE, GB, SR, K, CAP>

template <int CAP>
Launcher<CAP> pick_step(int mode, bool gb, bool sr, int K) {
  if (mode == kModeF32) return gb ? PSADAM_STEP_FN(kModeF32, true, false, 1, CAP) : PSADAM_STEP_FN(kModeF32, false, false, 1, CAP);
  if (mode == kModeBF16) return gb ? PSADAM_STEP_FN(kModeBF16, true, false, 1, CAP) : PSADAM_STEP_FN(kModeBF16, false, false, 1, CAP);
#define PSADAM_PICK_K(MODE, GB, SR)                                 \
  if (K == 1) return PSADAM_STEP_FN(MODE, GB, SR, 1, CAP);          \
  if (K == 3) return PSADAM_STEP_FN(MODE, GB, SR, 3, CAP);          \
  if (K == 4) return PSADAM_STEP_FN(MODE, GB, SR, 4, CAP);          \
  return PSADAM_STEP_FN(MODE, GB, SR, kRankSel, CAP);
#define PSADAM_PICK_MODE(MODE)                                      \
  if (gb) {                                                         \
    if (sr) { PSADAM_PICK_K(MODE, true, true) } else { PSADAM_PICK_K(MODE, true, false) } \
  } else {                                                          \
    if (sr) { PSADAM_PICK_K(MODE, false, true) } else { PSADAM_PICK_K(MODE, false, false) } \
  }
  if (mode == kModeQ8V) { PSADAM_PICK_MODE(kModeQ8V) }
  PSADAM_PICK_MODE(kModeQ8)
#undef PSADAM_PICK_MODE
#undef PSADAM_PICK_K
}

template <int CAP>
Launcher<CAP> pick_step_any(int mode, bool gb, bool sr) {
  if (mode == kModeQ8V) {
    if (gb) return sr ? &launch_step_any<kModeQ8V, true, true, CAP> : &launch_step_any<kModeQ8V, true, false, CAP>;
    return sr ? &launch_step_any<kModeQ8V, false, true, CAP> : &launch_step_any<kModeQ8V, false, false, CAP>;
  }
  if (gb) return sr ? &launch_step_any<kModeQ8, true, true, CAP> : &launch_step_any<kModeQ8, true, false, CAP>;
  return sr ? &launch_step_any<kModeQ8, false, true, CAP> : &launch_step_any<kModeQ8, false, false, CAP>;
}

template <int CAP>
Launcher<CAP> pick_step_sub(int mode, bool gb, bool sr) {
  if (mode == kModeQ8V) {
    if (gb) return sr ? &launch_step_sub<kModeQ8V, true, true, CAP> : &launch_step_sub<kModeQ8V, true, false, CAP>;
    return sr ? &launch_step_sub<kModeQ8V, false, true, CAP> : &launch_step_sub<kModeQ8V, false, false, CAP>;
  }
  if (gb) return sr ? &launch_step_sub<kModeQ8, true, true, CAP> : &launch_step_sub<kModeQ8, true, false, CAP>;
  return sr ? &launch_step_sub<kModeQ8, false, true, CAP> : &launch_step_sub<kModeQ8, false, false, CAP>;
}

template <int CAP>
Launcher<CAP> pick_quantize(bool sr, int K) {
  if (sr) {
    if (K == 1) return &launch_quantize<true, 1, CAP>;
    if (K == 3) return &launch_quantize<true, 3, CAP>;
    return K == 4 ? &launch_quantize<true, 4, CAP> : &launch_quantize<true, kRankSel, CAP>;
  }
  if (K == 1) return &launch_quantize<false, 1, CAP>;
  if (K == 3) return &launch_quantize<false, 3, CAP>;
  return K == 4 ? &launch_quantize<false, 4, CAP> : &launch_quantize<false, kRankSel, CAP>;
}

// Dispatch on list length: short lists use the small parameter block.
int dispatch(const std::vector<Entry>& es, const StepConsts& c, uint64_t seed, int64_t step, float pct,
             Launcher<kCapSmall> small, Launcher<kCapLarge> large, cudaStream_t stream,
             const GradSide& gs = GradSide{}, int bs = kBlock, int unit = 0) {
  if (es.empty()) return PSADAM_OK;
  if (es.size() <= (size_t)kCapSmall)
    return run_launches<kCapSmall>(es, c, seed, step, pct, gs, small, stream, bs, unit);
  return run_launches<kCapLarge>(es, c, seed, step, pct, gs, large, stream, bs, unit);
}

// Elements per CTA of the general kernels for block size bs.
int any_tile(int bs) { return any_blocks_per_tile(bs) * bs; }

// The list's grad-side options; 0 as an unscale factor reads as 1 (a zeroed struct changes nothing).
int grad_side(const psadam_list* list, GradSide& gs) {
  gs.unscale = list->grad_unscale == 0.0f ? 1.0f : list->grad_unscale;
  if (!finite(gs.unscale)) return PSADAM_ERR_INVALID_ARG;
  gs.zero = list->zero_grads != 0;
  gs.skip = list->skip_if_set;
  gs.approx = list->approx_update != 0;
  if (gs.skip && (reinterpret_cast<uintptr_t>(gs.skip) & 3u)) return PSADAM_ERR_MISALIGNED;
  return PSADAM_OK;
}

// Shared front half of the step entry points. need_ms / need_vs: the mode keeps 8-bit m / v
// codes and so needs their scale arrays.
int collect_list(const psadam_list* list, const void* const* m, const void* const* v, const float* const* ms,
                 const float* const* vs, bool need_ms, bool need_vs, std::vector<Entry>& out) {
  if (!list || list->n_tensors < 0) return PSADAM_ERR_INVALID_ARG;
  if (list->n_tensors == 0) return PSADAM_OK;
  if (list->grad_dtype != PSADAM_GRAD_F32 && list->grad_dtype != PSADAM_GRAD_BF16) return PSADAM_ERR_INVALID_ARG;
  if (!list->numel || !list->param || !list->grad || !m || !v || (need_ms && !ms) || (need_vs && !vs))
    return PSADAM_ERR_INVALID_ARG;
  out.reserve(list->n_tensors);
  for (int i = 0; i < list->n_tensors; ++i) {
    const long long n = list->numel[i];
    const int st = need_ms ? check_tensor(n, {list->param[i], list->grad[i], m[i], v[i], ms[i], vs[i]})
                   : need_vs ? check_tensor(n, {list->param[i], list->grad[i], m[i], v[i], vs[i]})
                             : check_tensor(n, {list->param[i], list->grad[i], m[i], v[i]});
    if (st != PSADAM_OK) return st;
    if (n == 0) continue;
    out.push_back(Entry{list->param[i], list->grad[i], const_cast<void*>(m[i]), const_cast<void*>(v[i]),
                        need_ms ? const_cast<float*>(ms[i]) : nullptr, need_vs ? const_cast<float*>(vs[i]) : nullptr,
                        n, i});
  }
  return PSADAM_OK;
}

// A validated step: everything the launches need.
struct StepCall {
  int mode = 0;
  bool q8mode = false, sr = false, gb = false;
  float pct = 100.f;
  uint64_t seed = 0;
  int bs = kBlock;
  GradSide gs;
  StepConsts c{};
  int64_t step = 1;
};

int prepare_step(int mode, const psadam_list* list, const void* const* m, const void* const* v, const float* const* ms,
                 const float* const* vs, int64_t step, const psadam_hparams* hp, const psadam_q8_opts* q8,
                 std::vector<Entry>& es, StepCall& call) {
  int st = check_hparams(hp, step);
  if (st != PSADAM_OK) return st;
  call.mode = mode;
  call.q8mode = mode == kModeQ8 || mode == kModeQ8V;
  if (call.q8mode && (st = check_q8(q8)) != PSADAM_OK) return st;
  if ((st = collect_list(list, m, v, ms, vs, mode == kModeQ8, call.q8mode, es)) != PSADAM_OK) return st;
  call.pct = call.q8mode ? q8->percentile : 100.f;
  call.sr = call.q8mode && q8->stochastic_rounding;
  call.seed = call.q8mode ? q8->seed : 0;
  call.bs = call.q8mode ? q8->block_size : kBlock;
  if ((st = check_block_counts(es, call.bs)) != PSADAM_OK) return st;
  if ((st = grad_side(list, call.gs)) != PSADAM_OK) return st;
  call.gs.static_scales = call.q8mode && q8->static_scales != 0;
  call.gb = list->grad_dtype == PSADAM_GRAD_BF16;
  call.c = make_consts(*hp, step);
  call.step = step;
  return PSADAM_OK;
}

// Launch the step over es (the whole list, or slices of it: every per-block decision below
// depends only on each block's own elements, its tensor's last-block length and rank).
int launch_prepared(const std::vector<Entry>& es, const StepCall& call, cudaStream_t s) {
  const int kmax = max_rank(es, call.pct, call.bs);
  // Power-of-two blocks of 16..1024 elements at rank 1 without the runtime options: several
  // blocks per tile of the persistent kernel
  const bool pow2 = (call.bs & (call.bs - 1)) == 0;
  const bool opts = call.gs.unscale != 1.0f || call.gs.zero != 0 || call.gs.static_scales != 0;
  if (call.q8mode && pow2 && call.bs >= kMinSubBlock && call.bs <= kMaxSubBlock && kmax == 1 && !opts)
    return dispatch(es, call.c, call.seed, call.step, call.pct, pick_step_sub<kCapSmall>(call.mode, call.gb, call.sr),
                    pick_step_sub<kCapLarge>(call.mode, call.gb, call.sr), s, call.gs, call.bs, kBlock);
  // 2048-element blocks with rank <= kMaxRank: the specialised kernels; otherwise the general one
  if (call.q8mode && (call.bs != kBlock || kmax > kMaxRank))
    return dispatch(es, call.c, call.seed, call.step, call.pct, pick_step_any<kCapSmall>(call.mode, call.gb, call.sr),
                    pick_step_any<kCapLarge>(call.mode, call.gb, call.sr), s, call.gs, call.bs, any_tile(call.bs));
  const int K = rank_template(kmax);
  return dispatch(es, call.c, call.seed, call.step, call.pct, pick_step<kCapSmall>(call.mode, call.gb, call.sr, K),
                  pick_step<kCapLarge>(call.mode, call.gb, call.sr, K), s, call.gs);
}

int step_common(int mode, const psadam_list* list, const void* const* m, const void* const* v,
                const float* const* ms, const float* const* vs, int64_t step, const psadam_hparams* hp,
                const psadam_q8_opts* q8, void* stream) {
  if (!list || list->n_tensors < 0) return PSADAM_ERR_INVALID_ARG;
  if (list->n_tensors == 0) return PSADAM_OK;
  std::vector<Entry> es;
  StepCall call;
  const int st = prepare_step(mode, list, m, v, ms, vs, step, hp, q8, es, call);
  if (st != PSADAM_OK) return st;
  return launch_prepared(es, call, static_cast<cudaStream_t>(stream));
}

// Events for the host pipeline, created once per thread and reused.
struct EventPool {
  std::vector<cudaEvent_t> ev;
  ~EventPool() {
    for (cudaEvent_t e : ev) cudaEventDestroy(e);
  }
  cudaError_t get(size_t n, cudaEvent_t** out) {
    while (ev.size() < n) {
      cudaEvent_t e;
      const cudaError_t err = cudaEventCreateWithFlags(&e, cudaEventDisableTiming);
      if (err != cudaSuccess) return err;
      ev.push_back(e);
    }
    *out = ev.data();
    return cudaSuccess;
  }
};

int cuda_fail(cudaError_t e) {
  g_last_cuda_error = (int32_t)e;
  return PSADAM_ERR_CUDA;
}

// Copies of consecutive pieces merged while both the source and the destination continue
// where the previous piece ended (tensors laid out back to back in flat buffers): one
// cudaMemcpyAsync per run instead of one per tensor.
struct CopyRun {
  cudaMemcpyKind kind;
  cudaStream_t stream;
  char* dst = nullptr;
  const char* src = nullptr;
  size_t bytes = 0;
  CopyRun(cudaMemcpyKind k, cudaStream_t s) : kind(k), stream(s) {}
  cudaError_t add(void* d, const void* sp, size_t n) {
    if (bytes != 0 && static_cast<char*>(d) == dst + bytes && static_cast<const char*>(sp) == src + bytes) {
      bytes += n;
      return cudaSuccess;
    }
    const cudaError_t e = flush();
    dst = static_cast<char*>(d);
    src = static_cast<const char*>(sp);
    bytes = n;
    return e;
  }
  cudaError_t flush() {
    if (bytes == 0) return cudaSuccess;
    const cudaError_t e = cudaMemcpyAsync(dst, src, bytes, kind, stream);
    bytes = 0;
    return e;
  }
};

// A slice's first element / 4 reaches the kernels as an int (the stochastic-rounding counter
// offset, TensorRef::grp_off), so no cut lies past 4 * INT_MAX elements of a tensor: the rest
// of a larger tensor stays in one slice.
constexpr long long kMaxCut = 4LL * INT_MAX;

// The list cut into chunks of about total/n_chunks elements: whole tensors in order, a tensor
// that does not fit the current chunk cut at a multiple of `unit` elements from its start.
std::vector<std::vector<Entry>> make_chunks(const std::vector<Entry>& es, int n_chunks, long long unit, int mode,
                                            int bs, size_t grad_bytes) {
  long long total = 0;
  for (const Entry& e : es) total += e.numel;
  long long target = (total / n_chunks + unit - 1) / unit * unit;
  if (target < unit) target = unit;
  const int mb = mode == kModeF32 || mode == kModeQ8V ? 4 : (mode == kModeBF16 ? 2 : 1);  // m bytes / element
  const int vb = mode == kModeF32 ? 4 : (mode == kModeBF16 ? 2 : 1);
  std::vector<std::vector<Entry>> chunks(1);
  long long size = 0;
  for (const Entry& e : es) {
    long long lo = 0;
    while (lo < e.numel) {
      long long hi = e.numel - lo <= target - size ? e.numel : lo + (target - size) / unit * unit;
      if (hi < e.numel && e.elem_off + hi > kMaxCut) hi = e.numel;
      if (hi <= lo) {  // not even one unit fits: close the chunk first
        chunks.emplace_back();
        size = 0;
        continue;
      }
      Entry piece = e;
      piece.p = e.p + lo;
      piece.g = static_cast<const char*>(e.g) + lo * (long long)grad_bytes;
      piece.m = static_cast<char*>(e.m) + lo * mb;
      piece.v = static_cast<char*>(e.v) + lo * vb;
      piece.ms = e.ms ? e.ms + lo / bs : nullptr;
      piece.vs = e.vs ? e.vs + lo / bs : nullptr;
      piece.numel = hi - lo;
      piece.elem_off = e.elem_off + lo;
      chunks.back().push_back(piece);
      size += hi - lo;
      lo = hi;
      if (size >= target || lo < e.numel) {
        chunks.emplace_back();
        size = 0;
      }
    }
  }
  if (chunks.back().empty()) chunks.pop_back();
  return chunks;
}

}  // namespace

extern "C" {

int psadam_step_from_host(int32_t mode, const psadam_list* list, const void* const* host_grad, float* const* host_param,
                          void* const* m, void* const* v, float* const* m_scale, float* const* v_scale, int64_t step,
                          const psadam_hparams* hp, const psadam_q8_opts* q8, int32_t n_chunks, void* stream,
                          void* stream_in, void* stream_out) {
  if (mode < kModeF32 || mode > kModeQ8V || !list || list->n_tensors < 0 || n_chunks < 1)
    return PSADAM_ERR_INVALID_ARG;
  if (list->n_tensors == 0) return PSADAM_OK;
  if (!host_grad || !host_param) return PSADAM_ERR_INVALID_ARG;
  for (int i = 0; i < list->n_tensors; ++i)
    if (list->numel && list->numel[i] > 0 && (!host_grad[i] || !host_param[i])) return PSADAM_ERR_INVALID_ARG;
  std::vector<Entry> es;
  StepCall call;
  int st = prepare_step(mode, list, reinterpret_cast<const void* const*>(m), reinterpret_cast<const void* const*>(v),
                        m_scale, v_scale, step, hp, q8, es, call);
  if (st != PSADAM_OK) return st;
  if (es.empty()) return PSADAM_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool piped = stream_in != nullptr && stream_out != nullptr;
  cudaStream_t sin = piped ? static_cast<cudaStream_t>(stream_in) : s;
  cudaStream_t sout = piped ? static_cast<cudaStream_t>(stream_out) : s;
  const size_t gsz = call.gb ? 2 : 4;
  // cut points keep every slice 16-byte aligned: a multiple of 4 blocks (scales) and of 16
  // elements (8-bit codes)
  long long unit = 4LL * call.bs;
  while (unit % 16 != 0) unit *= 2;
  const std::vector<std::vector<Entry>> chunks = make_chunks(es, piped ? n_chunks : 1, unit, mode, call.bs, gsz);
  static thread_local EventPool pool;
  cudaEvent_t* ev = nullptr;
  cudaError_t e = pool.get(2 * chunks.size() + 2, &ev);
  if (e != cudaSuccess) return cuda_fail(e);
  // the uploads overwrite the device grads: they wait for the caller's earlier work
  if (piped) {
    if ((e = cudaEventRecord(ev[0], s)) != cudaSuccess || (e = cudaStreamWaitEvent(sin, ev[0], 0)) != cudaSuccess)
      return cuda_fail(e);
  }
  for (size_t c = 0; c < chunks.size(); ++c) {
    CopyRun up(cudaMemcpyHostToDevice, sin);
    for (const Entry& pc : chunks[c]) {
      const char* src = static_cast<const char*>(host_grad[pc.list_idx]) + pc.elem_off * (long long)gsz;
      if ((e = up.add(const_cast<void*>(pc.g), src, (size_t)pc.numel * gsz)) != cudaSuccess) return cuda_fail(e);
    }
    if ((e = up.flush()) != cudaSuccess) return cuda_fail(e);
    if (piped) {
      if ((e = cudaEventRecord(ev[2 + 2 * c], sin)) != cudaSuccess || (e = cudaStreamWaitEvent(s, ev[2 + 2 * c], 0)) != cudaSuccess)
        return cuda_fail(e);
    }
    if ((st = launch_prepared(chunks[c], call, s)) != PSADAM_OK) return st;
    if (piped) {
      if ((e = cudaEventRecord(ev[3 + 2 * c], s)) != cudaSuccess ||
          (e = cudaStreamWaitEvent(sout, ev[3 + 2 * c], 0)) != cudaSuccess)
        return cuda_fail(e);
    }
    CopyRun down(cudaMemcpyDeviceToHost, sout);
    for (const Entry& pc : chunks[c]) {
      float* dst = host_param[pc.list_idx] + pc.elem_off;
      if ((e = down.add(dst, pc.p, (size_t)pc.numel * sizeof(float))) != cudaSuccess) return cuda_fail(e);
    }
    if ((e = down.flush()) != cudaSuccess) return cuda_fail(e);
  }
  // the caller's stream sees the whole step, downloads included
  if (piped) {
    if ((e = cudaEventRecord(ev[1], sout)) != cudaSuccess || (e = cudaStreamWaitEvent(s, ev[1], 0)) != cudaSuccess)
      return cuda_fail(e);
  }
  return PSADAM_OK;
}


int adam_step_fp32(const psadam_list* list, float* const* m, float* const* v, int64_t step,
                   const psadam_hparams* hp, void* stream) {
  return step_common(kModeF32, list, reinterpret_cast<const void* const*>(m), reinterpret_cast<const void* const*>(v),
                     nullptr, nullptr, step, hp, nullptr, stream);
}

int adam_step_bf16m(const psadam_list* list, uint16_t* const* m, uint16_t* const* v, int64_t step,
                    const psadam_hparams* hp, void* stream) {
  return step_common(kModeBF16, list, reinterpret_cast<const void* const*>(m), reinterpret_cast<const void* const*>(v),
                     nullptr, nullptr, step, hp, nullptr, stream);
}

int adam_step_q8(const psadam_list* list, int8_t* const* m_code, uint8_t* const* v_code, float* const* m_scale,
                 float* const* v_scale, int64_t step, const psadam_hparams* hp, const psadam_q8_opts* q8,
                 void* stream) {
  return step_common(kModeQ8, list, reinterpret_cast<const void* const*>(m_code),
                     reinterpret_cast<const void* const*>(v_code), m_scale, v_scale, step, hp, q8, stream);
}

int adam_step_q8v(const psadam_list* list, float* const* m, uint8_t* const* v_code, float* const* v_scale,
                  int64_t step, const psadam_hparams* hp, const psadam_q8_opts* q8, void* stream) {
  return step_common(kModeQ8V, list, reinterpret_cast<const void* const*>(m),
                     reinterpret_cast<const void* const*>(v_code), nullptr, v_scale, step, hp, q8, stream);
}

int psadam_q8_quantize(int32_t n_tensors, const int64_t* numel, const float* const* m, const float* const* v,
                       int8_t* const* m_code, uint8_t* const* v_code, float* const* m_scale, float* const* v_scale,
                       const psadam_q8_opts* q8, int64_t step, void* stream) {
  if (n_tensors < 0) return PSADAM_ERR_INVALID_ARG;
  if (n_tensors == 0) return PSADAM_OK;
  int st = check_q8(q8);
  if (st != PSADAM_OK) return st;
  if (!numel || !m || !v || !m_code || !v_code || !m_scale || !v_scale || step < 1) return PSADAM_ERR_INVALID_ARG;
  std::vector<Entry> es;
  for (int i = 0; i < n_tensors; ++i) {
    if ((st = check_tensor(numel[i], {m[i], v[i], m_code[i], v_code[i], m_scale[i], v_scale[i]})) != PSADAM_OK)
      return st;
    if (numel[i] == 0) continue;
    // codes travel in the p (m codes) and g (v codes) slots
    es.push_back(Entry{reinterpret_cast<float*>(m_code[i]), v_code[i], const_cast<float*>(m[i]),
                       const_cast<float*>(v[i]), m_scale[i], v_scale[i], numel[i], i});
  }
  const int bs = q8->block_size;
  if ((st = check_block_counts(es, bs)) != PSADAM_OK) return st;
  const int kmax = max_rank(es, q8->percentile, bs);
  const bool sr = q8->stochastic_rounding != 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (bs != kBlock || kmax > kMaxRank)
    return dispatch(es, StepConsts{}, q8->seed, step, q8->percentile,
                    sr ? &launch_quantize_any<true, kCapSmall> : &launch_quantize_any<false, kCapSmall>,
                    sr ? &launch_quantize_any<true, kCapLarge> : &launch_quantize_any<false, kCapLarge>, s, GradSide{},
                    bs, any_tile(bs));
  const int K = rank_template(kmax);
  return dispatch(es, StepConsts{}, q8->seed, step, q8->percentile, pick_quantize<kCapSmall>(sr, K),
                  pick_quantize<kCapLarge>(sr, K), s);
}

int psadam_q8_dequantize(int32_t n_tensors, const int64_t* numel, const int8_t* const* m_code,
                         const uint8_t* const* v_code, const float* const* m_scale, const float* const* v_scale,
                         float* const* m, float* const* v, int32_t block_size, void* stream) {
  if (n_tensors < 0) return PSADAM_ERR_INVALID_ARG;
  if (n_tensors == 0) return PSADAM_OK;
  const int bst = check_block_size(block_size);
  if (bst != PSADAM_OK) return bst;
  if (!numel || !m || !v || !m_code || !v_code || !m_scale || !v_scale) return PSADAM_ERR_INVALID_ARG;
  std::vector<Entry> es;
  for (int i = 0; i < n_tensors; ++i) {
    const int st = check_tensor(numel[i], {m[i], v[i], m_code[i], v_code[i], m_scale[i], v_scale[i]});
    if (st != PSADAM_OK) return st;
    if (numel[i] == 0) continue;
    es.push_back(Entry{reinterpret_cast<float*>(const_cast<int8_t*>(m_code[i])), v_code[i], m[i], v[i],
                       const_cast<float*>(m_scale[i]), const_cast<float*>(v_scale[i]), numel[i], i});
  }
  if (check_block_counts(es, block_size) != PSADAM_OK) return PSADAM_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (block_size != kBlock)
    return dispatch(es, StepConsts{}, 0, 1, 100.f, &launch_dequantize_any<kCapSmall>, &launch_dequantize_any<kCapLarge>,
                    s, GradSide{}, block_size, any_tile(block_size));
  return dispatch(es, StepConsts{}, 0, 1, 100.f, &launch_dequantize<kCapSmall>, &launch_dequantize<kCapLarge>, s);
}

int psadam_check_grads(const psadam_list* list, int32_t* found_nonfinite, void* stream) {
  if (!list || list->n_tensors < 0 || !found_nonfinite) return PSADAM_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(found_nonfinite) & 3u) return PSADAM_ERR_MISALIGNED;
  if (list->grad_dtype != PSADAM_GRAD_F32 && list->grad_dtype != PSADAM_GRAD_BF16) return PSADAM_ERR_INVALID_ARG;
  if (list->n_tensors > 0 && (!list->numel || !list->grad)) return PSADAM_ERR_INVALID_ARG;
  GradSide gs;
  int st = grad_side(list, gs);
  if (st != PSADAM_OK) return st;
  std::vector<Entry> es;
  for (int i = 0; i < list->n_tensors; ++i) {
    if ((st = check_tensor(list->numel[i], {list->grad[i]})) != PSADAM_OK) return st;
    if (list->numel[i] == 0) continue;
    es.push_back(Entry{nullptr, list->grad[i], nullptr, nullptr, nullptr, nullptr, list->numel[i], i});
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t e0 = cudaMemsetAsync(found_nonfinite, 0, sizeof(int32_t), s);
  if (e0 != cudaSuccess) {
    g_last_cuda_error = (int32_t)e0;
    return PSADAM_ERR_CUDA;
  }
  if (es.empty()) return PSADAM_OK;
  const bool gb = list->grad_dtype == PSADAM_GRAD_BF16;
  int* flag = found_nonfinite;
  auto small = [&](const LaunchArgs<kCapSmall>& a, cudaStream_t ss) {
    return gb ? launch_check_grads<true, kCapSmall>(a, flag, ss) : launch_check_grads<false, kCapSmall>(a, flag, ss);
  };
  auto large = [&](const LaunchArgs<kCapLarge>& a, cudaStream_t ss) {
    return gb ? launch_check_grads<true, kCapLarge>(a, flag, ss) : launch_check_grads<false, kCapLarge>(a, flag, ss);
  };
  if (es.size() <= (size_t)kCapSmall) return run_launches<kCapSmall>(es, StepConsts{}, 0, 1, 100.f, gs, small, s);
  return run_launches<kCapLarge>(es, StepConsts{}, 0, 1, 100.f, gs, large, s);
}

size_t psadam_state_bytes(int32_t mode, int64_t numel, int32_t block_size) {
  if (numel < 0) return 0;
  const size_t n = (size_t)numel;
  if ((mode == 2 || mode == 3) && block_size < 1) return 0;
  switch (mode) {
    case 0: return 8 * n;
    case 1: return 4 * n;
    case 2: return 2 * n + 8 * (size_t)n_blocks(numel, block_size);
    case 3: return 5 * n + 4 * (size_t)n_blocks(numel, block_size);
    default: return 0;
  }
}

int psadam_selftest_bounded_wait(int64_t cycles, void* stream) {
  if (cycles < 0 || cycles > kMaxWaitCycles) return PSADAM_ERR_INVALID_ARG;
  int* fault = fault_word();
  if (fault == nullptr) return PSADAM_ERR_CUDA;
  const cudaError_t e = launch_wait_selftest(fault, cycles, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PSADAM_OK : cuda_fail(e);
}

int psadam_selftest_update_math(int32_t full, uint64_t* mismatches, void* stream) {
  if (mismatches == nullptr || (full != 0 && full != 1)) return PSADAM_ERR_INVALID_ARG;
  // three launches' constants: the pages' defaults at the first step, a late step of another
  // setting, and eps = 0 (outside the fused domain: the IEEE path throughout)
  psadam_hparams h0{1e-3f, 0.9f, 0.999f, 1e-8f, 0.01f}, h1{3e-4f, 0.9f, 0.95f, 1e-6f, 0.1f}, h2{1e-3f, 0.9f, 0.999f, 0.0f, 0.0f};
  const StepConsts c[3] = {make_consts(h0, 1), make_consts(h1, 1000), make_consts(h2, 7)};
  unsigned long long out[4] = {0, 0, 0, 0};
  const cudaError_t e = launch_math_selftest(full, c, 3, out, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  for (int i = 0; i < 4; ++i) mismatches[i] = out[i];
  return PSADAM_OK;
}

int32_t psadam_device_fault(void) {
  // every stream of the device, non-blocking ones included, has finished what it was given
  if (cudaDeviceSynchronize() != cudaSuccess) return -1;
  psadam_take_fault_kernel<<<1, 1>>>();
  if (cudaGetLastError() != cudaSuccess) return -1;
  int v = 0;
  // ordered after the kernel on the legacy default stream
  if (cudaMemcpyFromSymbol(&v, g_psadam_fault_taken, sizeof v) != cudaSuccess) return -1;
  return v != 0 ? 1 : 0;
}

const char* psadam_status_string(int32_t status) {
  switch (status) {
    case PSADAM_OK: return "PSADAM_OK";
    case PSADAM_ERR_INVALID_ARG: return "PSADAM_ERR_INVALID_ARG";
    case PSADAM_ERR_MISALIGNED: return "PSADAM_ERR_MISALIGNED";
    case PSADAM_ERR_UNSUPPORTED: return "PSADAM_ERR_UNSUPPORTED";
    case PSADAM_ERR_CUDA: return "PSADAM_ERR_CUDA";
    default: return "PSADAM_ERR_UNKNOWN";
  }
}

int32_t psadam_last_cuda_error(void) { return g_last_cuda_error; }

}  // extern "C"
