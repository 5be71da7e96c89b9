// moe_permute_static: the dispatch step (moe_permute) for callers that cannot
// allocate device memory and have no workspace to hand over.
//
// Who needs it: code that runs where allocation is not allowed or not
// possible - for example inside an inference engine's plugin callback that
// owns all device memory and forbids allocation on its execution path, or a
// real-time service that reserves every byte at start-up so that no request
// can fail on a cudaMalloc.  Such callers still pass their inputs and
// outputs; the scratch space moe_permute would take from the workspace comes
// instead from one fixed array in device memory, placed there when this
// module is loaded on a device and held until the process exits.  With
// CUDA's default lazy module loading the module is loaded by the first
// cudaGetSymbolAddress below, i.e. inside the first call on each device:
// callers make that call at start-up, before they reserve all memory.
//
// The page's method has no counterpart to this entry point; it changes where
// the scratch lives, not what is computed (the same kernels run).
#include <climits>
#include <cmath>
#include <mutex>

#include "common.cuh"
#include "kernels.cuh"

#define MOE_API extern "C" __attribute__((visibility("default")))

namespace moe {
namespace {

constexpr int64_t kMaxAssign = MOE_STATIC_MAX_ASSIGNMENTS;
constexpr int64_t kMaxExperts = MOE_STATIC_MAX_EXPERTS;
constexpr int64_t kMaxBlocks = (kMaxAssign + kPermuteChunk - 1) / kPermuteChunk;
// local ranks [A] + per-chunk histograms [blocks, N] + per-chunk bases [blocks, N]
constexpr int64_t kScratchInts = kMaxAssign + 2 * kMaxBlocks * kMaxExperts;

}  // namespace
}  // namespace moe

// The shared scratch: 768 KiB of int32 on every device that loads the library.
static __device__ __align__(256) int32_t g_permute_scratch[moe::kScratchInts];

namespace moe {
namespace {

std::mutex g_setup_mutex;
int32_t* g_scratch_addr[256] = {};

// Device address of the scratch array for the current device.  In host code
// `g_permute_scratch` only names a host-side stand-in; the real address is
// looked up once per device, with that device current.
moe_status_t scratch_for_current_device(int32_t** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) return MOE_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_permute_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
    g_scratch_addr[dev] = static_cast<int32_t*>(p);
  }
  *out = g_scratch_addr[dev];
  return MOE_OK;
}

bool misaligned(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u); }

}  // namespace
}  // namespace moe

using namespace moe;

MOE_API moe_status_t moe_permute_static(const moe_config_t* cfg, const int32_t* topk_idx,
                                        const float* p_mean, int32_t* counts, int32_t* offsets,
                                        int32_t* perm, int32_t* inv, float* f, float* l_aux,
                                        void* stream) {
  if (!cfg) return MOE_ERR_INVALID_ARG;
  const moe_config_t& c = *cfg;
  if (c.T < 0 || c.H <= 0 || c.F <= 0 || c.N <= 0 || c.k <= 0 || c.k > c.N || c.F_shared < 0 ||
      std::isnan(c.capacity_factor) || std::isnan(c.aux_alpha) ||
      c.routing != MOE_ROUTING_TOKEN_CHOICE || c.min_capacity < 0 ||
      (c.drop_order != MOE_DROP_TOKEN_MAJOR && c.drop_order != MOE_DROP_SLOT_MAJOR))
    return MOE_ERR_INVALID_ARG;
  const int64_t A = (int64_t)c.T * c.k;
  // the fixed scratch bounds the problem size
  if (A > kMaxAssign || c.N > kMaxExperts || c.k > MOE_MAX_TOP_K) return MOE_ERR_UNSUPPORTED;
  int64_t C = -1;
  if (c.capacity_factor > 0.0f) {
    const double v = std::floor((double)c.T / (double)c.N * (double)c.capacity_factor);
    C = v < 0 ? 0 : (int64_t)v;
    if (C < c.min_capacity) C = c.min_capacity;
  }
  const int64_t R = C < 0 ? A : (C * c.N < A ? C * c.N : A);
  if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
  if (A > 0 && (!topk_idx || !inv)) return MOE_ERR_INVALID_ARG;
  if (R > 0 && !perm) return MOE_ERR_INVALID_ARG;
  if (l_aux && !p_mean) return MOE_ERR_INVALID_ARG;
  if (misaligned(topk_idx) || misaligned(p_mean) || misaligned(counts) || misaligned(offsets) ||
      misaligned(perm) || misaligned(inv) || misaligned(f) || misaligned(l_aux))
    return MOE_ERR_UNSUPPORTED;

  int32_t* scratch = nullptr;
  moe_status_t s = scratch_for_current_device(&scratch);
  if (s != MOE_OK) return s;

  PermuteLaunch a;
  a.topk_idx = topk_idx;
  a.p_mean = p_mean;
  a.counts = counts;
  a.offsets = offsets;
  a.perm = perm;
  a.inv = inv;
  a.f = f;
  a.l_aux = l_aux;
  // Every scratch entry a call reads is written earlier in the same call
  // (ranks and histograms by the rank kernel, bases by the scan kernel), so
  // nothing has to be cleared between calls.
  a.local_rank = scratch;
  a.blk_hist = scratch + kMaxAssign;
  a.blk_base = scratch + kMaxAssign + kMaxBlocks * kMaxExperts;
  a.T = c.T;
  a.N = c.N;
  a.k = c.k;
  a.capacity = C;
  a.alpha = c.aux_alpha;
  a.slot_major = c.drop_order == MOE_DROP_SLOT_MAJOR ? 1 : 0;
  return launch_permute(a, static_cast<cudaStream_t>(stream), nullptr) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}
