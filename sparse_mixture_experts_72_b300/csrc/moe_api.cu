// C ABI of the MoE FFN forward pass: argument checks, workspace layout and
// the stream-ordered launch sequence.  Declarations and the contract of each
// entry point are in include/moe.h.
#include <climits>
#include <cmath>
#include <cstring>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "kernels.cuh"

#define MOE_API extern "C" __attribute__((visibility("default")))

namespace moe {
namespace {

constexpr size_t kAlign = 256;

inline size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t capacity_of(const moe_config_t& c) {
  if (!(c.capacity_factor > 0.0f)) return -1;
  // floor(T / N * cf), in double, in that order; then the min_capacity floor
  const double v = std::floor((double)c.T / (double)c.N * (double)c.capacity_factor);
  const int64_t C = v < 0 ? 0 : (int64_t)v;
  return C < c.min_capacity ? (int64_t)c.min_capacity : C;
}

bool expert_choice(const moe_config_t& c) { return c.routing == MOE_ROUTING_EXPERT_CHOICE; }

// Slots per token S: assignment a = t*S + j (j the slot, or the expert for
// expert choice).
int slots_of(const moe_config_t& c) { return expert_choice(c) ? c.N : c.k; }

// Tokens each expert takes under expert choice: the capacity, at most T.
int64_t ec_tokens(const moe_config_t& c) {
  const int64_t C = capacity_of(c);
  return C < 0 ? 0 : (C < c.T ? C : (int64_t)c.T);
}

int64_t max_rows_of(const moe_config_t& c) {
  if (expert_choice(c)) return ec_tokens(c) * c.N;
  const int64_t A = (int64_t)c.T * c.k;
  const int64_t C = capacity_of(c);
  if (C < 0) return A;
  const int64_t cap = C * c.N;
  return cap < A ? cap : A;
}

// Rows of W1 per expert: F, or 2F (gate and up) for SwiGLU.
int64_t w1_rows(const moe_config_t& c, int64_t F) { return c.activation == MOE_ACT_SWIGLU ? 2 * F : F; }

// Rows one expert can hold: its capacity, at most one per token.
int64_t group_rows_max(const moe_config_t& c) {
  const int64_t cap = capacity_of(c);
  return expert_choice(c) ? ec_tokens(c) : (cap >= 0 && cap < c.T ? cap : (int64_t)c.T);
}

// The expert FFN runs with the operands swapped (decode_tc.cu: weights as
// the MMA's 128-row operand, routed and shared experts in one launch) when
// the experts hold few rows on average: a 128-row token tile would then be
// mostly padding.
constexpr int64_t kDecodeAvgRows = 64;
bool decode_ffn(const moe_config_t& c) {
  if (c.T == 0) return false;
  return max_rows_of(c) <= kDecodeAvgRows * c.N;
}

struct WsLayout {
  size_t status, status_bytes, rows_done, rows_done_s, w3, logits, p_part, local_rank, blk_hist,
      blk_base;
  size_t topk_idx, topk_w, p_mean, counts, offsets, perm, inv, f, l_aux, z_loss, probs;
  size_t xp, hid, y, hid_s, y_s;
  size_t total;
};

WsLayout layout_of(const moe_config_t& c) {
  WsLayout L;
  const int64_t T = c.T, N = c.N, A = T * slots_of(c), R = max_rows_of(c);
  const int64_t Ak = expert_choice(c) ? 0 : T * c.k;   // top-k outputs (token choice)
  const int64_t nsel = router_num_select_blocks(c.T);
  int64_t nblk = permute_num_blocks(A);
  if (T > 0 && c.N <= kRouterTcMaxExperts) {
    // a fused router's chunks use the same histogram / base arrays
    const int64_t ch = router_fused_chunks(c.T, c.N, c.H);
    if (ch > nblk) nblk = ch;
  }
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o += align_up(bytes > 0 ? bytes : 1); return at; };
  // The header every call zeroes first: [0] status word, [1] router ticket,
  // [2] permute ticket (or the fused dispatch's flag), [3] the expert FFN
  // launch's tile counter, then the row-block counters of the routed and the
  // shared expert FFN (phase 0 -> phase 1 hand-over).
  int64_t nrd = R > 0 ? gemm_rows_done_len(R, (int)N) : 0;
  const int64_t nrd_s = (c.F_shared > 0 && T > 0) ? gemm_rows_done_len(T, 1) : 0;
  if (T > 0 && decode_ffn(c)) {
    const int64_t nd = decode_rows_done_len(R, (int)N, c.F_shared > 0 ? T : 0);
    if (nd > nrd) nrd = nd;
  }
  L.status_bytes = align_up(sizeof(int32_t) * (4 + nrd + nrd_s));
  L.status = take(L.status_bytes);
  L.rows_done = L.status + 16;
  L.rows_done_s = L.rows_done + sizeof(int32_t) * nrd;
  const bool tc = c.N <= kRouterTcMaxExperts;
  L.w3 = take(tc ? router_w3_bytes(c.N, c.H) : 0);
  // logits: the SIMT router's scratch; expert choice selects on them
  L.logits = take((tc && !expert_choice(c)) ? 0 : sizeof(float) * T * N);
  const int64_t pblocks = tc ? router_tc_num_ctas(c.T, c.N, c.H) : nsel;
  L.p_part = take(sizeof(float) * (pblocks > 0 ? pblocks : 1) * (N + 1));
  L.local_rank = take(sizeof(int32_t) * A);
  L.blk_hist = take(sizeof(int32_t) * (nblk > 0 ? nblk : 1) * N);
  L.blk_base = take(sizeof(int32_t) * (nblk > 0 ? nblk : 1) * N);
  L.topk_idx = take(sizeof(int32_t) * Ak);
  L.topk_w = take(sizeof(float) * Ak);
  // expert choice weights its rows by the softmax itself
  L.probs = take(expert_choice(c) ? sizeof(float) * T * N : 0);
  L.p_mean = take(sizeof(float) * N);
  L.counts = take(sizeof(int32_t) * N);
  L.offsets = take(sizeof(int32_t) * (N + 1));
  L.perm = take(sizeof(int32_t) * R);
  L.inv = take(sizeof(int32_t) * A);
  L.f = take(sizeof(float) * N);
  L.l_aux = take(sizeof(float));
  L.z_loss = take(sizeof(float));
  L.xp = take(2 * (size_t)R * c.H);
  L.hid = take(2 * (size_t)R * c.F);   // the activation's output: F columns
  L.y = take(2 * (size_t)R * c.H);
  L.hid_s = take(c.F_shared > 0 ? 2 * (size_t)T * c.F_shared : 0);
  L.y_s = take(c.F_shared > 0 ? 2 * (size_t)T * c.H : 0);
  L.total = o;
  return L;
}

moe_status_t check_config(const moe_config_t* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->T < 0 || c->H <= 0 || c->F <= 0 || c->N <= 0 || c->k <= 0 || c->F_shared < 0)
    return MOE_ERR_INVALID_ARG;
  if (c->k > c->N) return MOE_ERR_INVALID_ARG;
  if (c->routing != MOE_ROUTING_TOKEN_CHOICE && c->routing != MOE_ROUTING_EXPERT_CHOICE)
    return MOE_ERR_INVALID_ARG;
  if (c->activation != MOE_ACT_GELU && c->activation != MOE_ACT_SILU &&
      c->activation != MOE_ACT_SWIGLU)
    return MOE_ERR_INVALID_ARG;
  if (c->drop_order != MOE_DROP_TOKEN_MAJOR && c->drop_order != MOE_DROP_SLOT_MAJOR)
    return MOE_ERR_INVALID_ARG;
  if (c->min_capacity < 0) return MOE_ERR_INVALID_ARG;
  if (c->weight_dtype != MOE_WEIGHTS_BF16 && c->weight_dtype != MOE_WEIGHTS_E4M3)
    return MOE_ERR_INVALID_ARG;
  if (c->routing == MOE_ROUTING_EXPERT_CHOICE) {
    if (!(c->capacity_factor > 0.0f)) return MOE_ERR_INVALID_ARG;
    if (c->T > kExpertChoiceMaxTokens) return MOE_ERR_UNSUPPORTED;
    if ((int64_t)c->T * c->N > INT32_MAX / 2) return MOE_ERR_UNSUPPORTED;
  }
  if (c->N > MOE_MAX_EXPERTS || c->k > MOE_MAX_TOP_K) return MOE_ERR_UNSUPPORTED;
  if (c->H % 8 || c->F % 8 || c->F_shared % 8) return MOE_ERR_UNSUPPORTED;
  if (c->weight_dtype == MOE_WEIGHTS_E4M3 && (c->H % 16 || c->F % 16 || c->F_shared % 16))
    return MOE_ERR_UNSUPPORTED;  // E4M3 rows must start on 16-byte boundaries
  if ((int64_t)c->T * c->k > INT32_MAX / 2) return MOE_ERR_UNSUPPORTED;
  if (std::isnan(c->capacity_factor) || std::isnan(c->aux_alpha)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

// 16-byte alignment of every non-null pointer; `required` ones must be non-null
template <typename... P>
moe_status_t check_ptrs(bool required, P... ps) {
  const void* arr[] = {static_cast<const void*>(ps)...};
  for (const void* p : arr) {
    if (!p) {
      if (required) return MOE_ERR_INVALID_ARG;
      continue;
    }
    if (!aligned16(p)) return MOE_ERR_UNSUPPORTED;
  }
  return MOE_OK;
}

moe_status_t check_ws(const moe_config_t& c, void* ws, size_t ws_bytes) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) % kAlign)) return MOE_ERR_WORKSPACE;
  if (ws_bytes < layout_of(c).total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

struct DeviceInfo {
  int sms = 0;
  bool ok = false;
};

// Per-process cache for the current device (one GPU per process here).
moe_status_t device_info(DeviceInfo* out) {
  static DeviceInfo cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_NO_DEVICE;
  DeviceInfo& d = cached[dev];
  if (!d.ok) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MOE_ERR_NO_DEVICE;
    if (major != 10 || minor != 3) return MOE_ERR_NO_DEVICE;
    if (!tensor_map_encoder_available()) return MOE_ERR_NO_DEVICE;
    d.sms = sms;
    d.ok = true;
  }
  *out = d;
  return MOE_OK;
}

inline moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

#define MOE_TRY(expr)                    \
  do {                                   \
    moe_status_t _s = (expr);            \
    if (_s != MOE_OK) return _s;         \
  } while (0)

#define MOE_CUDA(expr)                                   \
  do {                                                   \
    if ((expr) != cudaSuccess) return MOE_ERR_CUDA;      \
  } while (0)

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

moe_status_t clear_status(void* ws, const WsLayout& L, cudaStream_t st, LaunchTrace* tr) {
  trace_mark(tr, st);
  return cuda_status(cudaMemsetAsync(at<int>(ws, L.status), 0, L.status_bytes, st));
}

// ---------------------------------------------------------------- stages
// The tensor-core router's first kernel can zero the status header itself.
// Token choice with token-major claims on the tensor-core router: the
// router's CTAs also rank their chunk's assignments per expert and count
// them, and the scatter launch scans the counts (no rank launch).
bool fused_dispatch(const moe_config_t& c) {
  return !expert_choice(c) && c.drop_order == MOE_DROP_TOKEN_MAJOR &&
         c.N <= kRouterTcMaxExperts && c.T > 0;
}

// Whether the router's first kernel zeroes the header itself: the W_g split
// kernel does (planes along K); with stacked planes there is no split kernel
// and the router's CTA 0 does it, but only when the router uses no ticket
// (a fused dispatch).
bool router_clears_status(const moe_config_t& c, bool fused) {
  return c.N <= kRouterTcMaxExperts && c.T > 0 && (!router_own_split(c.T, c.N, c.H) || fused);
}

// Zeroes the status word and router ticket, unless the router's first kernel
// does it (router_clears_status).
moe_status_t begin_call(const moe_config_t& c, bool fused, void* ws, const WsLayout& L,
                        cudaStream_t st, LaunchTrace* tr) {
  if (router_clears_status(c, fused)) return MOE_OK;
  return clear_status(ws, L, st, tr);
}

// idx / w nullptr: no per-token selection (expert choice).
moe_status_t do_route(const moe_config_t& c, const uint16_t* x, const float* Wg, const float* bg,
                      const float* sel, int32_t* idx, float* w, float* probs, float* logits,
                      float* p_mean, float* z_loss, void* ws, const WsLayout& L, cudaStream_t st,
                      LaunchTrace* tr, bool fused = false) {
  RouterLaunch a;
  a.x = reinterpret_cast<const __nv_bfloat16*>(x);
  a.Wg = Wg;
  a.bg = bg;
  a.sel_bias = sel;
  a.topk_idx = idx;
  a.topk_w = w;
  a.probs = probs;
  a.p_mean = p_mean;
  a.logits = at<float>(ws, L.logits);
  a.logits_out = logits;
  a.z_loss = z_loss;
  a.p_part = at<float>(ws, L.p_part);
  a.T = c.T;
  a.H = c.H;
  a.N = c.N;
  a.k = idx ? c.k : 1;
  if (c.N <= kRouterTcMaxExperts) {
    RouterFused fz{at<int32_t>(ws, L.local_rank), at<int32_t>(ws, L.blk_hist)};
    return cuda_status(launch_router_tc(
        a, at<__nv_bfloat16>(ws, L.w3), at<int>(ws, L.status) + 1, at<int>(ws, L.status),
        router_clears_status(c, fused) ? at<int>(ws, L.status) : nullptr,
        (int)(L.status_bytes / 4), fused ? &fz : nullptr, st, tr));
  }
  return cuda_status(launch_router(a, st, tr));
}

moe_status_t do_permute(const moe_config_t& c, const int32_t* idx, const float* p_mean,
                        int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv, float* f,
                        float* l_aux, void* ws, const WsLayout& L, cudaStream_t st,
                        LaunchTrace* tr, const uint16_t* gather_x = nullptr) {
  PermuteLaunch a;
  a.topk_idx = idx;
  a.p_mean = p_mean;
  a.counts = counts;
  a.offsets = offsets;
  a.perm = perm;
  a.inv = inv;
  a.f = f;
  a.l_aux = l_aux;
  a.local_rank = at<int32_t>(ws, L.local_rank);
  a.blk_hist = at<int32_t>(ws, L.blk_hist);
  a.blk_base = at<int32_t>(ws, L.blk_base);
  a.T = c.T;
  a.N = c.N;
  a.k = c.k;
  a.capacity = capacity_of(c);
  a.alpha = c.aux_alpha;
  a.slot_major = c.drop_order == MOE_DROP_SLOT_MAJOR ? 1 : 0;
  a.ticket = at<int>(ws, L.status) + 2;  // zeroed with the status word
  if (gather_x && max_rows_of(c) > 0) {
    a.x = reinterpret_cast<const __nv_bfloat16*>(gather_x);
    a.xp = at<__nv_bfloat16>(ws, L.xp);
    a.H = c.H;
  }
  return cuda_status(launch_permute(a, st, tr));
}

// The scatter launch after a fused router (fused_dispatch).
moe_status_t do_dispatch_fused(const moe_config_t& c, const int32_t* idx, float* p_mean,
                               float* z_loss, int32_t* counts, int32_t* offsets, int32_t* perm,
                               int32_t* inv, float* f, float* l_aux, const uint16_t* x, void* ws,
                               const WsLayout& L, cudaStream_t st, LaunchTrace* tr) {
  DispatchFusedLaunch a{};
  a.topk_idx = idx;
  a.local_rank = at<int32_t>(ws, L.local_rank);
  a.blk_hist = at<int32_t>(ws, L.blk_hist);
  a.blk_base = at<int32_t>(ws, L.blk_base);
  a.p_part = at<float>(ws, L.p_part);
  a.counts = counts;
  a.offsets = offsets;
  a.perm = perm;
  a.inv = inv;
  a.f = f;
  a.p_mean = p_mean;
  a.z_loss = z_loss;
  a.l_aux = l_aux;
  a.flag = at<int>(ws, L.status) + 2;   // zeroed with the header by the router
  a.status = at<int>(ws, L.status);
  a.x = reinterpret_cast<const __nv_bfloat16*>(x);
  a.xp = max_rows_of(c) > 0 ? at<__nv_bfloat16>(ws, L.xp) : nullptr;
  a.T = c.T;
  a.N = c.N;
  a.k = c.k;
  a.H = c.H;
  a.chunks = router_fused_chunks(c.T, c.N, c.H);
  a.chunk_tokens = router_fused_chunk_tokens(c.T, c.N, c.H);
  a.capacity = capacity_of(c);
  a.alpha = c.aux_alpha;
  return cuda_status(launch_dispatch_fused(a, st, tr));
}

// Two events per device for moe_forward_host's stream hand-overs.  A wait
// takes the state of the event's latest record at the time it is enqueued,
// so one pair serves every call.
moe_status_t host_events(cudaEvent_t* in, cudaEvent_t* out) {
  static std::mutex mu;
  static cudaEvent_t evs[64][2] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < 2; ++i)
    if (!evs[dev][i] && cudaEventCreateWithFlags(&evs[dev][i], cudaEventDisableTiming) != cudaSuccess)
      return MOE_ERR_CUDA;
  *in = evs[dev][0];
  *out = evs[dev][1];
  return MOE_OK;
}

// Failure-injection count (moe_debug_suppress_gemm_producer): each GEMM
// launch consumes one unit while it is positive.
std::atomic<int> g_suppress_producer{0};

int32_t take_suppress_producer() {
  int v = g_suppress_producer.load();
  while (v > 0 && !g_suppress_producer.compare_exchange_weak(v, v - 1)) {
  }
  return v > 0 ? 1 : 0;
}

moe_status_t do_ffn(const moe_config_t& c, const uint16_t* x, const int32_t* perm,
                    const int32_t* offsets, const float* topk_w, const moe_weights_t& W,
                    uint16_t* y, uint16_t* y_shared, void* ws, const WsLayout& L, int sms,
                    cudaStream_t st, LaunchTrace* tr, bool gathered = false) {
  using bf = __nv_bfloat16;
  const int64_t R = max_rows_of(c);
  int* status = at<int>(ws, L.status);
  const bool fp8 = c.weight_dtype == MOE_WEIGHTS_E4M3;
  const int32_t act_mode = c.activation == MOE_ACT_SWIGLU ? EPI_SWIGLU
                           : c.activation == MOE_ACT_SILU ? EPI_SILU
                                                          : EPI_GELU;
  if (decode_ffn(c) && (R > 0 || (c.F_shared > 0 && c.T > 0))) {
    // routed and shared experts in one operand-swapped launch
    bf* xp = at<bf>(ws, L.xp);
    if (!gathered && R > 0)
      MOE_CUDA(launch_gather(reinterpret_cast<const bf*>(x), perm, offsets, c.N, slots_of(c), R,
                             c.H, xp, st, tr));
    const bool sh = c.F_shared > 0;
    DecodeArgs a{};
    a.offsets = offsets;
    a.num_groups = c.N;
    a.shared_rows = sh ? c.T : 0;
    a.H = c.H;
    a.F = c.F;
    a.Fs = sh ? c.F_shared : 0;
    a.mode0 = act_mode;
    a.b1 = reinterpret_cast<const bf*>(W.b1);
    a.b2 = reinterpret_cast<const bf*>(W.b2);
    a.b1s = reinterpret_cast<const bf*>(W.b1s);
    a.b2s = reinterpret_cast<const bf*>(W.b2s);
    if (fp8) {
      a.s1 = W.s1;
      a.s2 = W.s2;
      a.s1s = W.s1s;
      a.s2s = W.s2s;
    }
    a.out0 = at<bf>(ws, L.hid);
    a.out1 = reinterpret_cast<bf*>(y);
    a.out0s = sh ? at<bf>(ws, L.hid_s) : nullptr;
    a.out1s = reinterpret_cast<bf*>(y_shared);
    a.topk_w = topk_w;
    a.perm = perm;
    a.rows_done = at<int32_t>(ws, L.rows_done);
    a.status = status;
    a.skip_producer = take_suppress_producer();
    DecodeTensors t{};
    t.W1 = W.W1;
    t.W2 = W.W2;
    t.W1s = W.W1s;
    t.W2s = W.W2s;
    t.xp = xp;
    t.hid = at<bf>(ws, L.hid);
    t.R = R;
    t.x = reinterpret_cast<const bf*>(x);
    t.hid_s = sh ? at<bf>(ws, L.hid_s) : nullptr;
    DecodePlan p;
    MOE_CUDA(make_decode_plan(&p, a, t, fp8, group_rows_max(c), sms));
    MOE_CUDA(launch_decode(p, st, tr));
    return MOE_OK;
  }
  const bool sh = c.F_shared > 0 && c.T > 0;
  if (R > 0 || sh) {
    bf* xp = at<bf>(ws, L.xp);
    bf* hid = at<bf>(ws, L.hid);
    if (!gathered && R > 0)
      MOE_CUDA(launch_gather(reinterpret_cast<const bf*>(x), perm, offsets, c.N, slots_of(c), R,
                             c.H, xp, st, tr));
    // one persistent launch: Hid = act(X_perm W1_e^T + b1_e), then
    // y = w * (Hid W2_e^T + b2_e), row block by row block; the shared expert
    // is group N of the same launch (all T rows, weight 1)
    GemmArgs g{};
    g.offsets = offsets;
    g.num_groups = c.N;
    g.num_phases = 2;
    g.ph[0].n_out = c.F;
    g.ph[0].K = c.H;
    g.ph[0].mode = act_mode;
    g.ph[0].bias = reinterpret_cast<const bf*>(W.b1);
    g.ph[0].out = hid;
    g.ph[0].ld_out = c.F;
    g.ph[1].n_out = c.H;
    g.ph[1].K = c.F;
    g.ph[1].mode = EPI_SCALE;
    g.ph[1].bias = reinterpret_cast<const bf*>(W.b2);
    g.ph[1].topk_w = topk_w;
    g.ph[1].perm = perm;
    g.ph[1].out = reinterpret_cast<bf*>(y);
    g.ph[1].ld_out = c.H;
    if (fp8) {
      g.ph[0].b_scale = W.s1;
      g.ph[1].b_scale = W.s2;
    }
    g.rows_done = at<int32_t>(ws, L.rows_done);
    g.status = status;
    g.tile_counter = fp8 ? nullptr : status + 3;   // zeroed with the header
    g.skip_producer = take_suppress_producer();
    const void* Bs[2] = {W.W1s, W.W2s};
    int64_t b_rows_s[2] = {0, 0};
    if (sh) {
      g.shared_rows = c.T;
      g.shp[0].n_out = c.F_shared;
      g.shp[0].K = c.H;
      g.shp[0].mode = act_mode;
      g.shp[0].bias = reinterpret_cast<const bf*>(W.b1s);
      g.shp[0].out = at<bf>(ws, L.hid_s);
      g.shp[0].ld_out = c.F_shared;
      g.shp[1].n_out = c.H;
      g.shp[1].K = c.F_shared;
      g.shp[1].mode = EPI_SCALE;
      g.shp[1].bias = reinterpret_cast<const bf*>(W.b2s);
      g.shp[1].out = reinterpret_cast<bf*>(y_shared);
      g.shp[1].ld_out = c.H;
      if (fp8) {
        g.shp[0].b_scale = W.s1s;
        g.shp[1].b_scale = W.s2s;
      }
      g.rows_done_s = at<int32_t>(ws, L.rows_done_s);
      b_rows_s[0] = w1_rows(c, c.F_shared);
      b_rows_s[1] = c.H;
    }
    const void* B[2] = {W.W1, W.W2};
    const int64_t b_rows[2] = {(int64_t)c.N * w1_rows(c, c.F), (int64_t)c.N * c.H};
    GemmPlan p;
    // the rows one group can hold: an expert's (capacity, at most one per
    // token) or the shared expert's T
    const int64_t gmax = sh ? (int64_t)c.T : group_rows_max(c);
    MOE_CUDA(make_gemm_plan(&p, g, xp, R, B, b_rows, fp8, gmax, sms,
                            reinterpret_cast<const bf*>(x), Bs, b_rows_s));
    MOE_CUDA(launch_gemm(p, st, tr));
  }
  return MOE_OK;
}

int ffn_num_launches(const moe_config_t& c, bool gathered) {
  // [gather] + one launch for the routed and the shared experts
  const bool rows = max_rows_of(c) > 0, sh = c.F_shared > 0 && c.T > 0;
  return (rows && !gathered ? 1 : 0) + (rows || sh ? 1 : 0);
}

// Names of the launches moe_forward makes, in order (moe_forward_launch_name).
int forward_launch_names(const moe_config_t& c, const char** names, int cap) {
  int n = 0;
  auto add = [&](const char* s) {
    if (n < cap) names[n] = s;
    ++n;
  };
  const bool tc = c.N <= kRouterTcMaxExperts;
  const bool fz = fused_dispatch(c);
  if (!router_clears_status(c, fz)) add("status_memset");
  if (c.T == 0) add("router_pmean");
  else if (tc) {
    if (!router_own_split(c.T, c.N, c.H)) add("router_split");
    add("router_tc");
  } else { add("router_logits"); add("router_select"); add("router_pmean"); }
  const bool rows = max_rows_of(c) > 0, sh = c.F_shared > 0 && c.T > 0;
  bool gathered = true;
  if (expert_choice(c)) {
    add("expert_choice");
    gathered = false;
  } else if (fz) {
    add("dispatch_scatter");
  } else if ((int64_t)c.T * c.k > 0) {
    add("permute_rank_scan");
    add("scatter_gather");
  } else {
    add("permute_scan");
  }
  if (rows && !gathered) add("gather_rows");
  if (rows || sh) add(decode_ffn(c) ? "expert_ffn_decode" : "expert_ffn");
  if (c.T > 0) add("combine");
  return n;
}

moe_status_t check_weights(const moe_config_t& c, const moe_weights_t* W, bool need_router,
                           bool need_experts) {
  if (!W) return MOE_ERR_INVALID_ARG;
  if (need_router) {
    MOE_TRY(check_ptrs(true, W->Wg));
    MOE_TRY(check_ptrs(false, W->bg, W->sel_bias));
  }
  if (need_experts) {
    const bool fp8 = c.weight_dtype == MOE_WEIGHTS_E4M3;
    MOE_TRY(check_ptrs(true, W->W1, W->W2));
    MOE_TRY(check_ptrs(false, W->b1, W->b2));
    MOE_TRY(check_ptrs(fp8, W->s1, W->s2));
    if (c.F_shared > 0) {
      MOE_TRY(check_ptrs(true, W->W1s, W->W2s));
      MOE_TRY(check_ptrs(false, W->b1s, W->b2s));
      MOE_TRY(check_ptrs(fp8, W->s1s, W->s2s));
    }
  }
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

MOE_API size_t moe_workspace_size(const moe_config_t* cfg) {
  if (check_config(cfg) != MOE_OK) return 0;
  return layout_of(*cfg).total;
}

MOE_API int64_t moe_max_rows(const moe_config_t* cfg) {
  if (check_config(cfg) != MOE_OK) return -1;
  return max_rows_of(*cfg);
}

MOE_API int64_t moe_capacity(const moe_config_t* cfg) {
  if (check_config(cfg) != MOE_OK) return -1;
  return capacity_of(*cfg);
}

MOE_API int32_t moe_forward_num_launches(const moe_config_t* cfg) {
  if (check_config(cfg) != MOE_OK) return -1;
  const moe_config_t& c = *cfg;
  const bool fz = fused_dispatch(c);
  int n = router_clears_status(c, fz) ? 0 : 1;  // status clear
  n += router_num_launches(c.T, c.N, c.H);
  if (expert_choice(c)) {
    n += 1;                                 // expert-choice selection
    n += ffn_num_launches(c, false);        // gather + expert FFN (+ shared)
  } else if (fz) {
    n += 1;                                 // scan + scatter + gather
    n += ffn_num_launches(c, true);
  } else {
    n += permute_num_launches(c.T, c.k, true);  // the scatter also gathers the rows
    n += ffn_num_launches(c, true);
  }
  if (c.T > 0) n += 1;  // combine
  return n;
}

MOE_API const char* moe_forward_launch_name(const moe_config_t* cfg, int32_t i) {
  if (check_config(cfg) != MOE_OK || i < 0) return nullptr;
  const char* names[MOE_TRACE_MAX_EVENTS];
  const int n = forward_launch_names(*cfg, names, MOE_TRACE_MAX_EVENTS);
  return i < n && i < MOE_TRACE_MAX_EVENTS ? names[i] : nullptr;
}

MOE_API moe_status_t moe_route(const moe_config_t* cfg, const uint16_t* x, const float* Wg,
                               const float* bg, const float* sel_bias, int32_t* topk_idx,
                               float* topk_w, float* probs, float* logits, float* p_mean,
                               float* z_loss, void* ws, size_t ws_bytes, void* stream) {
  MOE_TRY(check_config(cfg));
  const moe_config_t& c = *cfg;
  const bool has_t = c.T > 0;
  MOE_TRY(check_ptrs(true, Wg, p_mean));
  if (expert_choice(c)) {
    topk_idx = nullptr;
    topk_w = nullptr;
  } else if (has_t) {
    MOE_TRY(check_ptrs(true, x, topk_idx, topk_w));
  }
  if (has_t) MOE_TRY(check_ptrs(true, x));
  MOE_TRY(check_ptrs(false, bg, sel_bias, probs, logits, z_loss));
  MOE_TRY(check_ws(c, ws, ws_bytes));
  DeviceInfo d;
  MOE_TRY(device_info(&d));
  const WsLayout L = layout_of(c);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MOE_TRY(begin_call(c, false, ws, L, st, nullptr));
  return do_route(c, x, Wg, bg, sel_bias, topk_idx, topk_w, probs, logits, p_mean, z_loss, ws, L,
                  st, nullptr);
}

MOE_API moe_status_t moe_expert_choice(const moe_config_t* cfg, const float* logits,
                                       const float* p_mean, int32_t* counts, int32_t* offsets,
                                       int32_t* perm, int32_t* inv, float* f, float* l_aux,
                                       void* stream) {
  MOE_TRY(check_config(cfg));
  const moe_config_t& c = *cfg;
  if (!expert_choice(c)) return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_ptrs(true, counts, offsets));
  if (c.T > 0) MOE_TRY(check_ptrs(true, logits, inv));
  if (max_rows_of(c) > 0) MOE_TRY(check_ptrs(true, perm));
  if (l_aux) MOE_TRY(check_ptrs(true, p_mean));
  MOE_TRY(check_ptrs(false, logits, p_mean, perm, inv, f, l_aux));
  DeviceInfo d;
  MOE_TRY(device_info(&d));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return cuda_status(launch_expert_choice(logits, p_mean, c.T, c.N, (int)ec_tokens(c),
                                          c.aux_alpha, counts, offsets, perm, inv, f, l_aux, st,
                                          nullptr));
}

MOE_API moe_status_t moe_update_sel_bias(const moe_config_t* cfg, const int32_t* counts,
                                         float* sel_bias, float gamma, void* stream) {
  MOE_TRY(check_config(cfg));
  if (std::isnan(gamma)) return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_ptrs(true, counts, sel_bias));
  DeviceInfo d;
  MOE_TRY(device_info(&d));
  return cuda_status(
      launch_update_sel_bias(counts, sel_bias, cfg->N, gamma, static_cast<cudaStream_t>(stream)));
}

MOE_API moe_status_t moe_permute(const moe_config_t* cfg, const int32_t* topk_idx,
                                 const float* p_mean, int32_t* counts, int32_t* offsets,
                                 int32_t* perm, int32_t* inv, float* f, float* l_aux, void* ws,
                                 size_t ws_bytes, void* stream) {
  MOE_TRY(check_config(cfg));
  const moe_config_t& c = *cfg;
  if (expert_choice(c)) return MOE_ERR_INVALID_ARG;  // moe_expert_choice dispatches those
  MOE_TRY(check_ptrs(true, counts, offsets));
  if ((int64_t)c.T * c.k > 0) MOE_TRY(check_ptrs(true, topk_idx, inv));
  if (max_rows_of(c) > 0) MOE_TRY(check_ptrs(true, perm));
  if (l_aux) MOE_TRY(check_ptrs(true, p_mean));
  MOE_TRY(check_ptrs(false, f, l_aux, p_mean));
  MOE_TRY(check_ws(c, ws, ws_bytes));
  DeviceInfo d;
  MOE_TRY(device_info(&d));
  const WsLayout L = layout_of(c);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MOE_TRY(clear_status(ws, L, st, nullptr));
  return do_permute(c, topk_idx, p_mean, counts, offsets, perm, inv, f, l_aux, ws, L, st,
                    nullptr);
}

MOE_API moe_status_t moe_expert_ffn(const moe_config_t* cfg, const uint16_t* x,
                                    const int32_t* perm, const int32_t* offsets,
                                    const float* topk_w, const moe_weights_t* weights,
                                    uint16_t* y, uint16_t* y_shared, void* ws, size_t ws_bytes,
                                    void* stream) {
  MOE_TRY(check_config(cfg));
  const moe_config_t& c = *cfg;
  MOE_TRY(check_weights(c, weights, false, true));
  if (c.T > 0) MOE_TRY(check_ptrs(true, x));
  if (max_rows_of(c) > 0) MOE_TRY(check_ptrs(true, perm, offsets, topk_w, y));
  if (c.F_shared > 0 && c.T > 0) MOE_TRY(check_ptrs(true, y_shared));
  MOE_TRY(check_ptrs(false, y, y_shared));
  MOE_TRY(check_ws(c, ws, ws_bytes));
  DeviceInfo d;
  MOE_TRY(device_info(&d));
  const WsLayout L = layout_of(c);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MOE_TRY(clear_status(ws, L, st, nullptr));
  return do_ffn(c, x, perm, offsets, topk_w, *weights, y, y_shared, ws, L, d.sms, st, nullptr);
}

MOE_API moe_status_t moe_combine(const moe_config_t* cfg, const uint16_t* y, const int32_t* inv,
                                 const uint16_t* y_shared, uint16_t* out, void* stream) {
  MOE_TRY(check_config(cfg));
  const moe_config_t& c = *cfg;
  if (c.T > 0) MOE_TRY(check_ptrs(true, inv, out));
  if (max_rows_of(c) > 0 && c.T > 0) MOE_TRY(check_ptrs(true, y));
  MOE_TRY(check_ptrs(false, y, y_shared));
  if (c.F_shared > 0 && c.T > 0 && !y_shared) return MOE_ERR_INVALID_ARG;
  DeviceInfo d;
  MOE_TRY(device_info(&d));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  using bf = __nv_bfloat16;
  return cuda_status(launch_combine(reinterpret_cast<const bf*>(y), inv,
                                    c.F_shared > 0 ? reinterpret_cast<const bf*>(y_shared) : nullptr,
                                    reinterpret_cast<bf*>(out), c.T, slots_of(c), c.H, st,
                                    nullptr));
}

MOE_API moe_status_t moe_forward(const moe_config_t* cfg, const moe_weights_t* weights,
                                 const uint16_t* x, uint16_t* out, const moe_outputs_t* outputs,
                                 void* ws, size_t ws_bytes, void* stream,
                                 void* const* trace_events) {
  MOE_TRY(check_config(cfg));
  const moe_config_t& c = *cfg;
  MOE_TRY(check_weights(c, weights, true, true));
  if (c.T > 0) MOE_TRY(check_ptrs(true, x, out));
  moe_outputs_t o;
  std::memset(&o, 0, sizeof(o));
  if (outputs) o = *outputs;
  MOE_TRY(check_ptrs(false, o.topk_idx, o.topk_w, o.probs, o.p_mean, o.counts, o.offsets, o.perm,
                     o.inv, o.f, o.l_aux, o.z_loss, o.logits));
  MOE_TRY(check_ws(c, ws, ws_bytes));
  DeviceInfo d;
  MOE_TRY(device_info(&d));
  const WsLayout L = layout_of(c);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  LaunchTrace trace{reinterpret_cast<cudaEvent_t*>(const_cast<void**>(trace_events)),
                    MOE_TRACE_MAX_EVENTS, 0};
  LaunchTrace* tr = trace_events ? &trace : nullptr;

  int32_t* idx = o.topk_idx ? o.topk_idx : at<int32_t>(ws, L.topk_idx);
  float* w = o.topk_w ? o.topk_w : at<float>(ws, L.topk_w);
  float* p_mean = o.p_mean ? o.p_mean : at<float>(ws, L.p_mean);
  int32_t* counts = o.counts ? o.counts : at<int32_t>(ws, L.counts);
  int32_t* offsets = o.offsets ? o.offsets : at<int32_t>(ws, L.offsets);
  int32_t* perm = o.perm ? o.perm : at<int32_t>(ws, L.perm);
  int32_t* inv = o.inv ? o.inv : at<int32_t>(ws, L.inv);
  float* f = o.f ? o.f : at<float>(ws, L.f);
  float* l_aux = o.l_aux ? o.l_aux : at<float>(ws, L.l_aux);
  float* z_loss = o.z_loss ? o.z_loss : at<float>(ws, L.z_loss);
  uint16_t* y = at<uint16_t>(ws, L.y);
  uint16_t* ys = c.F_shared > 0 ? at<uint16_t>(ws, L.y_s) : nullptr;

  const bool fz = fused_dispatch(c);
  MOE_TRY(begin_call(c, fz, ws, L, st, tr));
  if (expert_choice(c)) {
    // route (logits + softmax) -> each expert takes its top-C tokens ->
    // gather -> expert FFN weighted by P[t, e] -> combine over the N experts
    float* logits = o.logits ? o.logits : at<float>(ws, L.logits);
    float* probs = o.probs ? o.probs : at<float>(ws, L.probs);
    MOE_TRY(do_route(c, x, weights->Wg, weights->bg, nullptr, nullptr, nullptr, probs, logits,
                     p_mean, z_loss, ws, L, st, tr));
    MOE_CUDA(launch_expert_choice(logits, p_mean, c.T, c.N, (int)ec_tokens(c), c.aux_alpha,
                                  counts, offsets, perm, inv, f, l_aux, st, tr));
    MOE_TRY(do_ffn(c, x, perm, offsets, probs, *weights, y, ys, ws, L, d.sms, st, tr, false));
  } else {
    MOE_TRY(do_route(c, x, weights->Wg, weights->bg, weights->sel_bias, idx, w, o.probs, o.logits,
                     p_mean, z_loss, ws, L, st, tr, fz));
    if (fz)
      MOE_TRY(do_dispatch_fused(c, idx, p_mean, z_loss, counts, offsets, perm, inv, f, l_aux, x,
                                ws, L, st, tr));
    else
      MOE_TRY(do_permute(c, idx, p_mean, counts, offsets, perm, inv, f, l_aux, ws, L, st, tr, x));
    MOE_TRY(do_ffn(c, x, perm, offsets, w, *weights, y, ys, ws, L, d.sms, st, tr, true));
  }
  if (c.T > 0) {
    using bf = __nv_bfloat16;
    MOE_CUDA(launch_combine(reinterpret_cast<const bf*>(y), inv, reinterpret_cast<const bf*>(ys),
                            reinterpret_cast<bf*>(out), c.T, slots_of(c), c.H, st, tr));
  }
  trace_mark(tr, st);
  return MOE_OK;
}

MOE_API moe_status_t moe_forward_host(const moe_config_t* cfg, const moe_weights_t* weights,
                                      const uint16_t* x_host, uint16_t* x_dev, uint16_t* out_dev,
                                      uint16_t* out_host, const moe_outputs_t* outputs, void* ws,
                                      size_t ws_bytes, void* h2d_stream, void* compute_stream,
                                      void* d2h_stream) {
  MOE_TRY(check_config(cfg));
  const moe_config_t& c = *cfg;
  if (c.T > 0 && (!x_host || !out_host)) return MOE_ERR_INVALID_ARG;
  // validate everything the forward checks before the first copy is enqueued
  MOE_TRY(check_weights(c, weights, true, true));
  if (c.T > 0) MOE_TRY(check_ptrs(true, x_dev, out_dev));
  MOE_TRY(check_ws(c, ws, ws_bytes));
  DeviceInfo d;
  MOE_TRY(device_info(&d));
  cudaStream_t is = static_cast<cudaStream_t>(h2d_stream);
  cudaStream_t ks = static_cast<cudaStream_t>(compute_stream);
  cudaStream_t os = static_cast<cudaStream_t>(d2h_stream);
  cudaEvent_t ev_in = nullptr, ev_out = nullptr;
  if (is != ks || os != ks) MOE_TRY(host_events(&ev_in, &ev_out));
  const size_t bytes = sizeof(uint16_t) * (size_t)c.T * c.H;
  if (bytes > 0) MOE_CUDA(cudaMemcpyAsync(x_dev, x_host, bytes, cudaMemcpyHostToDevice, is));
  if (is != ks) {
    MOE_CUDA(cudaEventRecord(ev_in, is));
    MOE_CUDA(cudaStreamWaitEvent(ks, ev_in, 0));
  }
  MOE_TRY(moe_forward(cfg, weights, x_dev, out_dev, outputs, ws, ws_bytes, ks, nullptr));
  if (os != ks) {
    MOE_CUDA(cudaEventRecord(ev_out, ks));
    MOE_CUDA(cudaStreamWaitEvent(os, ev_out, 0));
  }
  if (bytes > 0) MOE_CUDA(cudaMemcpyAsync(out_host, out_dev, bytes, cudaMemcpyDeviceToHost, os));
  return MOE_OK;
}

MOE_API moe_status_t moe_workspace_status(const void* ws, void* stream) {
  if (!ws) return MOE_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int v = 0;
  // the status word sits at offset 0 of every layout
  if (cudaMemcpyAsync(&v, ws, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  return v == 0 ? MOE_OK : static_cast<moe_status_t>(v);
}

MOE_API moe_status_t moe_debug_suppress_gemm_producer(int launches) {
  if (launches < 0) return MOE_ERR_INVALID_ARG;
  g_suppress_producer.store(launches);
  return MOE_OK;
}

MOE_API const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape or alignment";
    case MOE_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_TIMEOUT: return "device-side wait timed out";
    case MOE_ERR_NO_DEVICE: return "no usable sm_103 device";
  }
  return "unknown status";
}

MOE_API const char* moe_version(void) { return "moe_b300 0.1 (sm_103a)"; }
