// Host-side launch descriptions of the MoE kernels (one translation unit
// per pipeline stage; moe_api.cu strings them together).
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda.h>
#include <stdint.h>

namespace moe {

// Launches `kern` with programmatic stream serialisation (the kernel calls
// pdl_wait() before its first global memory access) and, for cluster > 1,
// thread-block clusters of that many CTAs along x.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, unsigned cluster, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  int n = 1;
  if (cluster > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    n = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Optional per-launch event trace: event i is recorded before launch i.
struct LaunchTrace {
  cudaEvent_t* events;
  int n_events;
  int next;
};

// While the stream is being captured into a CUDA graph the events become
// event-record nodes of the graph (so replays carry the timestamps).
inline void trace_mark(LaunchTrace* tr, cudaStream_t st) {
  if (tr && tr->events && tr->next < tr->n_events) {
    cudaEvent_t e = tr->events[tr->next++];
    if (!e) return;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
      cudaEventRecordWithFlags(e, st, cudaEventRecordExternal);
    else
      cudaEventRecord(e, st);
  }
}

// ---------------------------------------------------------------- router
struct RouterLaunch {
  const __nv_bfloat16* x;
  const float* Wg;
  const float* bg;
  const float* sel_bias;
  int32_t* topk_idx;
  float* topk_w;
  float* probs;     // nullable
  float* p_mean;
  float* logits;    // [T, N]: scratch of the SIMT router; written by the
                    // tensor-core router only when logits_out is set
  float* p_part;    // scratch [blocks, N + 1]: per-block column sums of P,
                    // then the block's sum of logsumexp(l_t)^2
  float* z_loss;    // nullable: mean over tokens of logsumexp(l_t)^2
  float* logits_out;  // nullable [T, N] (tensor-core router)
  int T, H, N, k;   // topk_idx == nullptr: no selection (expert choice)
};
int router_num_select_blocks(int T);
int router_num_launches(int T, int N, int H);
// fp32 SIMT router (any N <= MOE_MAX_EXPERTS)
cudaError_t launch_router(const RouterLaunch& a, cudaStream_t st, LaunchTrace* tr);
// p_mean[0..N) = 0 and *z_loss = 0 (nullable) in one launch (an empty batch)
cudaError_t launch_router_stats_zero(float* p_mean, float* z_loss, int N, cudaStream_t st);

// tensor-core router (N <= kRouterTcMaxExperts): split kernel + fused kernel
constexpr int kRouterTcMaxExperts = 256;
struct RouterTcArgs {
  const float* bg;
  const float* sel_bias;
  int32_t* topk_idx;
  float* topk_w;
  float* probs;     // nullable
  float* logits_out;  // nullable [T, N]
  float* z_loss;    // nullable
  float* p_part;    // [m_tiles * splits, N + 1] per-CTA column sums of P, then sum of lse^2
  float* p_mean;
  int* ticket;      // CTAs done; zero on entry
  int* status;
  int T, N, N_pad, H_pad, k, tmem_cols;
  int stacked;           // 1: planes stacked along N; 0: planes along K
  int nacc;              // independent TMEM accumulators
  int planes_per_stage;  // planes along K: B tiles per stage (1 or 3)
  int stages;
  int kb_per_split;      // x tiles (64 wide) per K split
  int splits;            // K splits = cluster size (1, 2, 4 or 8)
  int work_bytes;        // ring / logits-tile shared memory
  // stacked planes: the epilogue warps split W_g (fp32 [N, H]) into the
  // three bf16 planes of each ring slot themselves (no W3, no split kernel)
  const float* Wg;
  int H;
  // dispatch fused into the router (moe_forward, token choice, token-major
  // claims): each CTA writes its chunk's local ranks (local_rank[t*k + j],
  // the rank of the assignment among the chunk's assignments to the same
  // expert in token order) and expert histogram (blk_hist[cta][N]) instead
  // of reducing p_mean; `clear` (clear_n ints) is zeroed by CTA 0 first.
  int32_t* local_rank;   // nullptr: not fused (the last CTA reduces p_mean)
  int32_t* blk_hist;
  int* clear;
  int clear_n;
};
struct RouterTcPlan {
  int N_pad, H_pad, stacked, pp, nacc, tmem_cols, stage_bytes, stages, m_tiles, splits,
      kb_per_split, work_bytes, smem;
};
RouterTcPlan router_tc_plan(int T, int N, int H);
int router_tc_num_ctas(int T, int N, int H);
inline size_t router_w3_bytes(int N, int H) {
  const size_t N_pad = (N + 15) / 16 * 16, H_pad = (H + 63) / 64 * 64;
  return N_pad * 3 * H_pad * 2;
}
// `clear` (nullable, clear_n ints) is zeroed by the first kernel of the
// router, before the router kernel itself runs (with stacked planes and no
// split kernel: by the router's CTA 0; the router then uses no ticket, so
// `clear` must not hold one it needs - see router_stacked()).
// fused (nullable): the dispatch histogram outputs of a fused router.
struct RouterFused {
  int32_t* local_rank;   // [T * k]
  int32_t* blk_hist;     // [chunks, N]
};
cudaError_t launch_router_tc(const RouterLaunch& a, __nv_bfloat16* W3, int* ticket, int* status,
                             int* clear, int clear_n, const RouterFused* fused, cudaStream_t st,
                             LaunchTrace* tr);
// whether the tensor-core router splits W_g itself (stacked planes, few x
// tiles per CTA): no split kernel then
bool router_own_split(int T, int N, int H);
// chunks (router CTAs) and tokens per chunk of a fused router launch
int router_fused_chunks(int T, int N, int H);
int router_fused_chunk_tokens(int T, int N, int H);

// TMA map of a row-major bf16 matrix [rows, K], box 64 (K) x box_rows, 128B swizzle
bool encode_tensor_map_bf16(CUtensorMap* map, const void* base, int64_t rows, int64_t K,
                            int box_cols, int box_rows);

// ---------------------------------------------------------------- permute
struct PermuteLaunch {
  const int32_t* topk_idx;
  const float* p_mean;  // nullable when l_aux == nullptr
  int32_t* counts;
  int32_t* offsets;
  int32_t* perm;
  int32_t* inv;
  float* f;             // nullable
  float* l_aux;         // nullable
  int32_t* local_rank;  // scratch [T*k]
  int32_t* blk_hist;    // scratch [nblk, N]
  int32_t* blk_base;    // scratch [nblk, N]
  int T, N, k;
  int64_t capacity;     // < 0: no limit
  float alpha;
  int slot_major = 0;   // claim order: 0 a = t*k + j; 1 j-major, then t
  int* ticket = nullptr;  // zeroed int: the rank launch's last block also scans
  // optional fused gather: xp[row] = x[perm[row] / k] for every kept row
  const __nv_bfloat16* x = nullptr;
  __nv_bfloat16* xp = nullptr;
  int H = 0;
};
// Dispatch after a fused router (router_tc with RouterFused): the scatter
// launch's CTA 0 scans the router's chunk histograms (counts, capacity,
// offsets, chunk bases, f, p_mean from the router's partial sums, z-loss,
// L_aux) and releases a flag; every CTA then scatters and gathers its tokens.
struct DispatchFusedLaunch {
  const int32_t* topk_idx;
  const int32_t* local_rank;  // [T * k] from the router
  const int32_t* blk_hist;    // [chunks, N] from the router
  int32_t* blk_base;          // scratch [chunks, N]
  const float* p_part;        // [chunks, N + 1] from the router
  int32_t* counts;
  int32_t* offsets;
  int32_t* perm;
  int32_t* inv;
  float* f;                   // nullable
  float* p_mean;
  float* z_loss;              // nullable
  float* l_aux;               // nullable
  int* flag;                  // zeroed by the router's CTA 0
  int* status;
  const __nv_bfloat16* x;
  __nv_bfloat16* xp;
  int T, N, k, H, chunks, chunk_tokens;
  int64_t capacity;
  float alpha;
};
cudaError_t launch_dispatch_fused(const DispatchFusedLaunch& a, cudaStream_t st, LaunchTrace* tr);

constexpr int kPermuteChunk = 256;  // assignments per block
inline int permute_num_blocks(int64_t A) { return (int)((A + kPermuteChunk - 1) / kPermuteChunk); }
int permute_num_launches(int T, int k, bool fused_scan);
cudaError_t launch_permute(const PermuteLaunch& a, cudaStream_t st, LaunchTrace* tr);

// ---------------------------------------------------------------- gather / combine
cudaError_t launch_gather(const __nv_bfloat16* x, const int32_t* perm, const int32_t* offsets,
                          int N, int k, int64_t max_rows, int H, __nv_bfloat16* xp,
                          cudaStream_t st, LaunchTrace* tr);
cudaError_t launch_combine(const __nv_bfloat16* y, const int32_t* inv,
                           const __nv_bfloat16* y_shared, __nv_bfloat16* out, int T, int k,
                           int H, cudaStream_t st, LaunchTrace* tr);

// ---------------------------------------------------------------- expert choice
constexpr int kExpertChoiceMaxTokens = 51200;  // one expert's column in shared memory
// One CTA per expert: counts, offsets, perm, inv [T*N], f, l_aux (nullable).
cudaError_t launch_expert_choice(const float* logits, const float* p_mean, int T, int N, int C,
                                 float alpha, int32_t* counts, int32_t* offsets, int32_t* perm,
                                 int32_t* inv, float* f, float* l_aux, cudaStream_t st,
                                 LaunchTrace* tr);
// sel_bias[e] += gamma * sign(counts[e] - mean(counts)), one launch
cudaError_t launch_update_sel_bias(const int32_t* counts, float* sel_bias, int N, float gamma,
                                   cudaStream_t st);

// ---------------------------------------------------------------- grouped tcgen05 GEMM
// EPI_SWIGLU: B holds 2*n_out rows per group (gate rows, then up rows); a
// tile covers 128 output columns, its accumulator the 128 gate and the 128
// up columns, and the output is SiLU(gate) * up.
enum EpilogueMode : int32_t { EPI_GELU = 0, EPI_SCALE = 1, EPI_SILU = 2, EPI_SWIGLU = 3 };

// One GEMM of a launch: out = epilogue(A_rows . B_g^T) for every group g.
struct GemmPhase {
  int32_t n_out;                 // output columns per group (B rows per group: n_out, or
                                 // 2 * n_out for EPI_SWIGLU)
  int32_t K;                     // reduction length
  int32_t mode;                  // EpilogueMode
  int32_t ld_out;
  const __nv_bfloat16* bias;     // [G, n_out] ([G, 2 * n_out] for EPI_SWIGLU) or nullptr
  const float* topk_w;           // EPI_SCALE: weight per assignment, or nullptr (weight 1)
  const int32_t* perm;           // EPI_SCALE: row -> assignment (with topk_w)
  __nv_bfloat16* out;            // [rows, ld_out]
  const float* b_scale;          // FP8 B: per B row (output column) scale, same layout as
                                 // bias but fp32; nullptr for bf16 B
};

// A launch runs one phase, or two where phase 1 reads phase 0's output rows
// as its A operand (the expert FFN's Linear -> GELU -> Linear in one
// persistent grid).  Both phases share the row segments of the groups.
struct GemmArgs {
  const int32_t* offsets;        // [G+1] row segments of A per group, or nullptr
  int32_t num_groups;            // G (routed experts), or 1 with offsets == nullptr
  int32_t rows_single;           // rows of the single group when offsets == nullptr
  int32_t num_phases;            // 1 or 2
  GemmPhase ph[2];
  int32_t* rows_done;            // num_phases == 2: per row block, phase-0 epilogue arrivals
                                 // (zeroed before the launch; gemm_rows_done_len() entries)
  int* status;                   // device status word
  int32_t skip_producer;         // failure injection: the TMA producer issues nothing
  int32_t a_box;                 // rows per A copy (set by make_gemm_plan): 128, or for
                                 // FP8 single-CTA tiles the bound on a group's rows
  int32_t swap_tail;             // CTA pairs: a group's last row block of at most this
                                 // many rows (and fewer than 256) runs operand-swapped;
                                 // 0: none (set by make_gemm_plan)
  // the always-on shared expert as group G of the same launch: shared_rows
  // rows (T; 0 = none) of its own A tensors (x, then its Hid), its own
  // weights, outputs (shp[p].out) and row-block counters; weight 1
  int32_t shared_rows;
  GemmPhase shp[2];
  int32_t* rows_done_s;
  // bf16 weights: a launch-wide tile counter (zeroed before the launch) from
  // which the CTAs (pairs) take their next tile as they finish the last one;
  // nullptr: tile t runs on CTA (pair) t % grid.  make_gemm_plan keeps it
  // only for bf16 launches of many tiles per CTA (pair).
  int32_t* tile_counter;
};

struct GemmPlan {
  CUtensorMap tmS[4];  // shared expert: A phase 0 (x), B phase 0 (W1s), A phase 1 (its Hid), B phase 1
  CUtensorMap tmA[2];  // per phase: A [rows, K] bf16, box 64 x 128, 128B swizzle
  CUtensorMap tmB[2];  // per phase: B [G * n_out, K] bf16, box 64 x (256 / pair), 128B
                       // swizzle; FP8 B: E4M3 bytes, the same box unswizzled
  GemmArgs args;
  int grid;
  int pair;         // 1: one CTA per 128-row tile; 2: a CTA pair per 256-row tile
  bool fp8;         // B operands are E4M3 codes with per-row scales (ph[p].b_scale)
};

// Upper bound of the row blocks (tiles along M) of a launch over a_rows rows
// in G groups: the length of GemmArgs::rows_done.
inline int64_t gemm_rows_done_len(int64_t a_rows, int G) { return (a_rows + 127) / 128 + G; }

// Encodes the tensor maps (phase 1's A is phase 0's output when num_phases
// is 2); returns cudaErrorInvalidValue if encoding fails.
// B[p] points at bf16 weights, or with fp8 set at E4M3 codes (one byte per
// weight; K a multiple of 16 so that rows start on 16-byte boundaries).
// group_rows_max bounds the rows of any one group (tokens per expert); FP8
// launches of small groups copy only that many A rows per k-block (a group
// that exceeds it records MOE_ERR_INVALID_ARG in the status word).
// With args.shared_rows > 0, A_s is its phase-0 A tensor (x) and
// B_s / b_rows_s its weights (W1s, W2s); a_rows may then be 0.
cudaError_t make_gemm_plan(GemmPlan* plan, const GemmArgs& args, const __nv_bfloat16* A,
                           int64_t a_rows, const void* const B[2], const int64_t b_rows[2],
                           bool fp8, int64_t group_rows_max, int num_sms,
                           const __nv_bfloat16* A_s = nullptr, const void* const* B_s = nullptr,
                           const int64_t* b_rows_s = nullptr);
cudaError_t launch_gemm(const GemmPlan& plan, cudaStream_t st, LaunchTrace* tr);
bool tensor_map_encoder_available();
// TMA map of a row-major byte matrix [rows, K] (E4M3 codes), 128B swizzle
bool encode_tensor_map_u8(CUtensorMap* map, const void* base, int64_t rows, int64_t K,
                          int box_cols, int box_rows);

// ---------------------------------------------------------------- decode expert FFN
// The expert FFN with the operands swapped (weights as the 128-row MMA
// operand, an expert's few token rows as N), routed experts and the shared
// expert in one launch.  For batches whose experts hold few rows.
struct DecodeMaps {
  CUtensorMap wa0, wa1;   // routed weights: W1 [G * w1_rows, H], W2 [G * H, F]
  CUtensorMap ws0, ws1;   // shared weights: W1s [w1_rows_s, H], W2s [H, Fs]
  CUtensorMap xa0, xa1;   // routed activations: X_perm [R, H], Hid [R, F] (boxes of 16 rows)
  CUtensorMap xs0, xs1;   // shared activations: x [T, H], Hid_s [T, Fs]
};
struct DecodeArgs {
  const int32_t* offsets;        // [G + 1] row segments of the routed experts
  int32_t num_groups;            // G
  int32_t shared_rows;           // T with a shared expert, else 0
  int32_t H, F, Fs;              // hidden, routed and shared inner sizes (output columns of phase 0)
  int32_t mode0;                 // EPI_GELU / EPI_SILU / EPI_SWIGLU (phase 1 is EPI_SCALE)
  const __nv_bfloat16 *b1, *b2, *b1s, *b2s;   // biases or nullptr
  const float *s1, *s2, *s1s, *s2s;           // E4M3 row scales (nullptr for bf16 weights)
  __nv_bfloat16 *out0, *out1, *out0s, *out1s; // Hid, y, Hid_s, y_s
  const float* topk_w;           // routed rows' gate weights (through perm)
  const int32_t* perm;
  int32_t* rows_done;            // per token chunk: phase-0 tiles stored (zeroed before the launch)
  int* status;
  int32_t skip_producer;         // failure injection: the TMA producer issues nothing
  // set by make_decode_plan
  int32_t nt, w_stages, x_stages, q_stages, tmem_cols;
};
struct DecodeTensors {
  const void *W1, *W2, *W1s, *W2s;            // weights (bf16 or E4M3 codes)
  const __nv_bfloat16* xp;                    // [R, H] permuted token rows
  const __nv_bfloat16* hid;                   // [R, F]
  int64_t R;                                  // rows of xp / hid (0: no routed rows)
  const __nv_bfloat16* x;                     // [T, H]
  const __nv_bfloat16* hid_s;                 // [T, Fs]
};
struct DecodePlan {
  DecodeMaps maps;
  DecodeArgs args;
  int grid, smem;
  bool fp8;
};
// token rows per tile for groups of at most group_rows_max rows (16..32)
int decode_token_tile(int64_t group_rows_max);
// Upper bound of the token chunks (phase-1 counters) of a decode launch.
inline int64_t decode_rows_done_len(int64_t R, int G, int64_t T) { return (R + 15) / 16 + G + (T + 15) / 16 + 1; }
cudaError_t make_decode_plan(DecodePlan* plan, const DecodeArgs& args, const DecodeTensors& t,
                             bool fp8, int64_t group_rows_max, int num_sms);
cudaError_t launch_decode(const DecodePlan& plan, cudaStream_t st, LaunchTrace* tr);

}  // namespace moe
