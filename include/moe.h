/*
 * moe.h - C ABI of the B300 (sm_103a) sparse Mixture-of-Experts FFN forward pass.
 *
 * One MoE FFN layer ("AI-Research-SKILLs MoE 训练实战：稀疏专家模型的架构、路由、
 * 负载均衡与推理优化全指南", §3.1 MoELayer; "混合专家模型 MoE 架构深度解析：从路由
 * 机制到生产级推理部署", §1.2-§3):
 *
 *   l     = x . W_g^T + b_g                       gate Linear, fp32
 *   P     = softmax(l)                            over the N experts
 *   idx   = top-k of (l - b_sel)                  b_sel: selection-only bias
 *   w     = P[idx] / sum_j P[idx_j]               renormalised over the k
 *   C     = floor(T / N * capacity_factor)        capacity, overflow dropped
 *   y     = W2_e . GELU(W1_e . x_t + b1_e) + b2_e  per kept assignment
 *   out_t = sum_j w_tj y_tj  (+ shared expert)    dropped slots add zero
 *   L_aux = alpha * N * sum_i f_i p_i
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library
 *    never allocates device memory.  Scratch comes from the caller's
 *    workspace `ws` of at least moe_workspace_size(cfg) bytes.
 *  - bf16 tensors are passed as uint16_t bit patterns.  Layouts are row-major;
 *    weights use the nn.Linear [out, in] layout (K contiguous):
 *      W_g [N, H] fp32, W1 [N, F, H], W2 [N, H, F], W1s [Fs, H], W2s [H, Fs].
 *  - Every pointer must be 16-byte aligned; H, F and F_shared must be
 *    multiples of 8 (of 16 with E4M3 weights).  Violations return
 *    MOE_ERR_UNSUPPORTED before any launch.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream).  Arguments are validated on the host before anything
 *    is launched; a non-OK return means nothing was enqueued, except
 *    MOE_ERR_CUDA, which reports a failed launch.
 *  - Device-side failures never trap.  A kernel whose bounded wait runs out
 *    records MOE_ERR_TIMEOUT in a status word inside `ws` and returns; every
 *    entry point that takes `ws` clears that word first, and
 *    moe_workspace_status() reads it.
 *  - Calls are stateless and re-entrant; concurrent calls need distinct `ws`.
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,  /* null required pointer, negative size, k < 1 or k > N, ... */
  MOE_ERR_UNSUPPORTED = 2,  /* misaligned pointer, H/F not a multiple of 8, N > MOE_MAX_EXPERTS */
  MOE_ERR_WORKSPACE = 3,    /* ws is NULL, misaligned or smaller than moe_workspace_size() */
  MOE_ERR_CUDA = 4,         /* a CUDA runtime call or kernel launch failed */
  MOE_ERR_TIMEOUT = 5,      /* a device-side bounded wait ran out (see moe_workspace_status) */
  MOE_ERR_NO_DEVICE = 6     /* no usable sm_103 device or driver entry point */
} moe_status_t;

#define MOE_MAX_EXPERTS 1024
#define MOE_MAX_TOP_K 32
/* moe_forward records at most this many events when given a trace array. */
#define MOE_TRACE_MAX_EVENTS 32

/* Layer shape and routing parameters. */
/* routing: who chooses.  Token choice is the pages' top-k router
 * ("混合专家模型 MoE 架构深度解析" §1.3); expert choice lets each expert take
 * its C highest-scoring tokens ("AI-Research-SKILLs MoE 训练实战" §4.2, §7.3). */
#define MOE_ROUTING_TOKEN_CHOICE 0
#define MOE_ROUTING_EXPERT_CHOICE 1
/* activation of the expert FFN: GELU (§3.1's MoELayer), SiLU (the two-Linear
 * expert printed in §6.1) or SwiGLU (the gated form §6.1's text names for
 * Mixtral: W1 then holds [N, 2F, H], gate rows first, up rows second). */
#define MOE_ACT_GELU 0
#define MOE_ACT_SILU 1
#define MOE_ACT_SWIGLU 2
/* which assignments claim capacity first: token-major (a = t*k + j in
 * increasing a) or slot-major (every token's first choice, then every
 * token's second choice, ...). */
#define MOE_DROP_TOKEN_MAJOR 0
#define MOE_DROP_SLOT_MAJOR 1
/* storage of the expert weights W1, W2, W1s, W2s: bf16, or FP8 ("AI-Research-
 * SKILLs MoE 训练实战" §9.2 FP8 quantisation, which names no format: read as
 * E4M3 codes, 1 sign, 4 exponent bits with bias 7, 3 mantissa bits) with one
 * fp32 scale per weight row:
 *   W[r, c] = scale[r] * E4M3(code[r, c])
 * Activations stay bf16; each weight is widened to bf16 (exactly) on chip and
 * the products accumulate in fp32, as for bf16 weights. */
#define MOE_WEIGHTS_BF16 0
#define MOE_WEIGHTS_E4M3 1

typedef struct {
  int32_t T;                /* tokens (rows of x); 0 is allowed */
  int32_t H;                /* hidden size */
  int32_t F;                /* routed expert FFN inner size */
  int32_t N;                /* routed experts, 1..MOE_MAX_EXPERTS */
  int32_t k;                /* experts per token, 1..min(N, MOE_MAX_TOP_K); token choice */
  float capacity_factor;    /* > 0: C = floor(T / N * capacity_factor); <= 0: no limit */
  int32_t F_shared;         /* shared expert inner size; 0 = no shared expert */
  float aux_alpha;          /* alpha of L_aux (the pages use 0.01) */
  int32_t routing;          /* MOE_ROUTING_*; expert choice needs capacity_factor > 0 */
  int32_t activation;       /* MOE_ACT_*; the shared expert uses the same one */
  int32_t min_capacity;     /* >= 0: C = max(C, min_capacity) when a capacity applies
                               (the DeepSpeed moe block's min_capacity, §5.1) */
  int32_t drop_order;       /* MOE_DROP_* (token choice with a capacity) */
  int32_t weight_dtype;     /* MOE_WEIGHTS_*; E4M3 needs H, F, F_shared multiples of 16 */
} moe_config_t;

/* Layer parameters (device pointers).  The expert weights W1, W2, W1s, W2s
 * hold one element per weight of the type weight_dtype names: bf16 bit
 * patterns (2 bytes) or E4M3 codes (1 byte); with E4M3 each has a row scale
 * array (fp32, one per row of the [out, in] matrix), required. */
typedef struct {
  const float* Wg;          /* [N, H] fp32 gate weight, required */
  const float* bg;          /* [N] fp32 gate bias, or NULL (= 0) */
  const float* sel_bias;    /* [N] fp32 selection-only bias b_i, or NULL (= 0) */
  const void* W1;           /* [N, F, H] ([N, 2F, H] for SwiGLU), required */
  const uint16_t* b1;       /* [N, F] ([N, 2F] for SwiGLU) bf16 or NULL */
  const void* W2;           /* [N, H, F], required */
  const uint16_t* b2;       /* [N, H] bf16 or NULL */
  const void* W1s;          /* [Fs, H] ([2Fs, H] for SwiGLU), required iff F_shared > 0 */
  const uint16_t* b1s;      /* [Fs] ([2Fs] for SwiGLU) bf16 or NULL */
  const void* W2s;          /* [H, Fs], required iff F_shared > 0 */
  const uint16_t* b2s;      /* [H] bf16 or NULL */
  const float* s1;          /* E4M3: [N, F] ([N, 2F] for SwiGLU) row scales of W1 */
  const float* s2;          /* E4M3: [N, H] row scales of W2 */
  const float* s1s;         /* E4M3 with F_shared > 0: [Fs] ([2Fs]) row scales of W1s */
  const float* s2s;         /* E4M3 with F_shared > 0: [H] row scales of W2s */
} moe_weights_t;

/* Optional device outputs of moe_forward; each may be NULL (kept in ws).
 * "Slots per token" S is k for token choice and N for expert choice, where
 * assignment a = t*N + e means expert e took token t. */
typedef struct {
  int32_t* topk_idx;        /* [T, k] (token choice) */
  float* topk_w;            /* [T, k] (token choice) */
  float* probs;             /* [T, N] full softmax; written only when non-NULL */
  float* p_mean;            /* [N]   p_i = mean_t P[t, i] */
  int32_t* counts;          /* [N]   assignments per expert before capacity drops */
  int32_t* offsets;         /* [N+1] expert-contiguous row offsets after drops */
  int32_t* perm;            /* [moe_max_rows(cfg)] row -> assignment t*S+j */
  int32_t* inv;             /* [T*S] assignment -> row, -1 if dropped / not taken */
  float* f;                 /* [N]   f_i = counts_i / sum_e counts_e */
  float* l_aux;             /* [1]   alpha * N * sum f_i p_i */
  float* z_loss;            /* [1]   router z-loss, mean_t logsumexp(l_t)^2 */
  float* logits;            /* [T, N] gate logits l = x W_g^T + b_g */
} moe_outputs_t;

/* Bytes of workspace the entry points need for this configuration. */
size_t moe_workspace_size(const moe_config_t* cfg);

/* Upper bound on kept rows R: T*k, or min(T*k, N*C) with a capacity limit;
 * N*min(C, T) for expert choice. */
int64_t moe_max_rows(const moe_config_t* cfg);

/* Capacity C of "混合专家模型 MoE 架构深度解析" §2.3, computed in double as
 * floor((double)T / N * capacity_factor), then raised to min_capacity; -1
 * when there is no limit. */
int64_t moe_capacity(const moe_config_t* cfg);

/* Number of kernel launches (and memsets) one moe_forward call enqueues. */
int32_t moe_forward_num_launches(const moe_config_t* cfg);

/* Name of launch i (0 <= i < moe_forward_num_launches(cfg)) of moe_forward,
 * e.g. "router_tc", "expert_ffn", "expert_ffn_decode", "combine": the
 * intervals a trace_events array times.  A static string; NULL for an
 * invalid configuration or index.  No device access. */
const char* moe_forward_launch_name(const moe_config_t* cfg, int32_t i);

/*
 * moe_route - gate, softmax, top-k selection and renormalisation.
 * ("混合专家模型 MoE 架构深度解析" §1.2 gate formula, §1.3 top-K steps 1-3,
 *  §2.4 selection bias; "AI-Research-SKILLs MoE 训练实战" §3.1 MoELayer gate,
 *  §4.3 router z-loss.)
 *   x        [T, H] bf16          Wg [N, H] fp32, bg [N] fp32 or NULL
 *   sel_bias [N] fp32 or NULL     subtracted from the logits for selection only
 *   topk_idx [T, k] int32 out     experts in descending (l - b_sel); ties -> lower index
 *   topk_w   [T, k] fp32 out      unbiased softmax at idx, renormalised to sum 1
 *            (both NULL, and not computed, for expert choice)
 *   probs    [T, N] fp32 out or NULL   full softmax
 *   logits   [T, N] fp32 out or NULL   l = x W_g^T + b_g
 *   p_mean   [N] fp32 out         mean over tokens of the softmax (p_i of L_aux)
 *   z_loss   [1] fp32 out or NULL mean over tokens of logsumexp(l_t)^2
 * Logits accumulate in fp32.
 */
moe_status_t moe_route(const moe_config_t* cfg, const uint16_t* x, const float* Wg,
                       const float* bg, const float* sel_bias, int32_t* topk_idx,
                       float* topk_w, float* probs, float* logits, float* p_mean,
                       float* z_loss, void* ws, size_t ws_bytes, void* stream);

/*
 * moe_expert_choice - expert-choice dispatch ("AI-Research-SKILLs MoE 训练实战"
 * §4.2: expert_scores = router(x) transposed, top-k along the tokens with
 * k = capacity_per_expert; §7.3: perfect balance, no token dropped for load).
 * Expert e takes the C = moe_capacity(cfg) (at most T) tokens with the largest
 * logits[:, e]; equal logits take the lower token first.  Its rows are
 * [e*C, (e+1)*C), tokens in increasing order; assignment a = t*N + e.
 *   logits [T, N] fp32 in (moe_route); p_mean [N] fp32 in, or NULL when l_aux is NULL
 *   counts [N] int32 out (C each)  offsets [N+1] int32 out (e*C)
 *   perm [N*C] int32 out           inv [T*N] int32 out (row, or -1: not taken)
 *   f [N] fp32 out or NULL (1/N)   l_aux [1] fp32 out or NULL (alpha * N * sum f_i p_i)
 * Needs routing = MOE_ROUTING_EXPERT_CHOICE, capacity_factor > 0 and
 * T <= 51200 (the per-expert column is staged in shared memory); otherwise
 * MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED before any launch.  One launch,
 * no workspace.
 */
moe_status_t moe_expert_choice(const moe_config_t* cfg, const float* logits,
                               const float* p_mean, int32_t* counts, int32_t* offsets,
                               int32_t* perm, int32_t* inv, float* f, float* l_aux,
                               void* stream);

/*
 * moe_update_sel_bias - one auxiliary-loss-free balancing step
 * ("混合专家模型 MoE 架构深度解析" §2.4): the selection bias of an expert that
 * received more than the mean number of assignments rises by gamma, that of
 * one that received fewer falls by gamma, an expert at the mean keeps its
 * bias:  sel_bias[e] += gamma * sign(counts[e] - sum(counts) / N).
 * The pages give no rate; gamma is the caller's.
 *   counts [N] int32 in (moe_permute / moe_forward), sel_bias [N] fp32 in/out
 * One launch, no workspace.
 */
moe_status_t moe_update_sel_bias(const moe_config_t* cfg, const int32_t* counts,
                                 float* sel_bias, float gamma, void* stream);

/*
 * moe_permute - histogram, capacity, stable expert-contiguous dispatch and L_aux.
 * ("混合专家模型 MoE 架构深度解析" §2.3 capacity and overflow, §2.2 L_aux;
 *  "AI-Research-SKILLs MoE 训练实战" §4.3 expert fraction, §4.4 drop_tokens.)
 * Assignments a = t*k + j claim slots in increasing a (drop_order token-
 * major) or j-major then t (slot-major); rank within its expert >= C means
 * dropped.  Token choice only.
 *   topk_idx [T, k] int32 in; values must lie in [0, N) (not checked on device:
 *            out-of-range indices are ignored by the histogram and dropped)
 *   p_mean   [N] fp32 in (from moe_route); may be NULL when l_aux is NULL
 *   counts   [N] int32 out        offsets [N+1] int32 out
 *   perm     [moe_max_rows] int32 out (first offsets[N] entries written)
 *   inv      [T*k] int32 out      -1 for dropped assignments
 *   f        [N] fp32 out or NULL l_aux [1] fp32 out or NULL
 */
moe_status_t moe_permute(const moe_config_t* cfg, const int32_t* topk_idx, const float* p_mean,
                         int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv,
                         float* f, float* l_aux, void* ws, size_t ws_bytes, void* stream);

/*
 * moe_expert_ffn - gather, expert Linear -> activation -> Linear, gate weighting.
 * ("AI-Research-SKILLs MoE 训练实战" §3.1 expert = Linear(H,F), GELU, Linear(F,H);
 *  §6.1 SiLU / SwiGLU; §7.1 and "混合专家模型 MoE 架构深度解析" §3 shared expert.)
 *   y[r]        = bf16( w_a * (W2_e . bf16(act(W1_e . x_t + b1_e)) + b2_e) )
 *                 for rows r < offsets[N], a = perm[r], t = a / S, e the expert of r
 *                 (S = k, or N for expert choice)
 *   y_shared[t] = bf16( W2s . bf16(act(W1s . x_t + b1s)) + b2s )   when F_shared > 0
 *   act: GELU(z), SiLU(z), or SiLU(z[:F]) * z[F:] for SwiGLU
 *   x [T, H] bf16; perm/offsets from moe_permute or moe_expert_choice;
 *   topk_w [T, S] fp32 (the renormalised top-k weights, or the softmax
 *   probs [T, N] for expert choice)
 *   y [moe_max_rows, H] bf16 out; y_shared [T, H] bf16 out (NULL iff F_shared == 0)
 * bf16 x bf16 products accumulate in fp32 on the tensor cores; E4M3 weights
 * are widened to bf16 in shared memory and their row scale multiplies the
 * fp32 sum before the bias.
 * Both Linears run in one persistent launch whose second-Linear tiles wait
 * (bounded) for the first Linear's rows; it sizes its grid to the CTAs that
 * fit on the GPU at once, so two such launches running at the same time on
 * different streams can starve each other: keep the layers of concurrent
 * batches on one stream (moe_forward_host shows the pattern); if they do
 * overlap, the waits run out and MOE_ERR_TIMEOUT is recorded, nothing hangs.
 * Two kernels serve it.  When the experts hold at most 64 rows on average
 * (moe_max_rows(cfg) <= 64 N: decode-sized batches) the operands are
 * swapped: each expert's weights are the 128-row operand of the tensor-core
 * MMA and its token rows the narrow one; any row count per expert is
 * computed.  Otherwise token rows are the 128- or 256-row operand (CTA pairs
 * for groups of 192 rows or more on average).  In both kernels the shared
 * expert is one more group of the same launch (T rows, weight 1).  In the
 * token-row kernel, offsets must give no expert more rows than the config allows
 * (at most T for token choice, since a token picks distinct experts, and at
 * most the capacity when one applies), as moe_permute and moe_expert_choice
 * produce: FP8 launches with groups below 128 rows copy only that many rows
 * per expert; an expert with more records MOE_ERR_INVALID_ARG in the status
 * word (its extra rows are not computed; nothing is read or written out of
 * bounds).
 */
moe_status_t moe_expert_ffn(const moe_config_t* cfg, const uint16_t* x, const int32_t* perm,
                            const int32_t* offsets, const float* topk_w,
                            const moe_weights_t* weights, uint16_t* y, uint16_t* y_shared,
                            void* ws, size_t ws_bytes, void* stream);

/*
 * moe_combine - weighted sum back per token ("AI-Research-SKILLs MoE 训练实战"
 * §3.1 output[mask] += score * expert_out; §6.1 index_add_ combine).
 *   out[t] = bf16( sum_{j<S, inv[t*S+j] >= 0} y[inv[t*S+j]] (+ y_shared[t]) )
 * summed in fp32 in the order j = 0..S-1, then the shared term (S = k, or N
 * for expert choice).  A token whose every slot was dropped (or that no
 * expert took) gets 0 (+ its shared term).
 *   y [moe_max_rows, H] bf16, inv [T*S] int32, y_shared [T, H] bf16 or NULL
 *   out [T, H] bf16
 */
moe_status_t moe_combine(const moe_config_t* cfg, const uint16_t* y, const int32_t* inv,
                         const uint16_t* y_shared, uint16_t* out, void* stream);

/*
 * moe_forward - the whole layer: route, permute, experts, combine, stream-
 * ordered with no host synchronisation.
 *   x [T, H] bf16 in; out [T, H] bf16 out; weights as moe_weights_t;
 *   outputs: optional device copies of the intermediate results, or NULL.
 *   trace_events: NULL, or an array of MOE_TRACE_MAX_EVENTS cudaEvent_t
 *   (NULL entries are skipped); when given, event i is recorded on `stream`
 *   just before launch i and event moe_forward_num_launches(cfg) just after
 *   the last one.
 */
moe_status_t moe_forward(const moe_config_t* cfg, const moe_weights_t* weights,
                         const uint16_t* x, uint16_t* out, const moe_outputs_t* outputs,
                         void* ws, size_t ws_bytes, void* stream, void* const* trace_events);

/*
 * moe_forward_host - moe_forward for a batch that lives in host memory:
 * copies x_host into x_dev, runs the layer, copies out_dev back into
 * out_host, with cudaMemcpyAsync and no host synchronisation.  The input
 * copy goes on h2d_stream, the layer on compute_stream and the output copy
 * on d2h_stream (any of them may be the same stream); the layer waits for
 * the input copy and the output copy for the layer through events the
 * library keeps per device.  x_host / out_host should be page-locked
 * (pinned) for the copies to be asynchronous; pageable memory works but
 * each copy then waits.
 * Pipelining: successive calls with three streams overlap batch i+1's input
 * copy and batch i-1's output copy with batch i's layer; the layers stay in
 * order on the one compute stream (the expert-FFN launch assumes it is the
 * only one of its kind on the GPU at a time).  The caller owns buffer reuse:
 * x_dev / out_dev / out_host of a call must not be reused before its output
 * copy has completed (three sets of staging buffers keep all three engines
 * busy).
 *   x_host [T, H] bf16 (host), out_host [T, H] bf16 (host)
 *   x_dev, out_dev [T, H] bf16 (device staging), the rest as moe_forward.
 */
moe_status_t moe_forward_host(const moe_config_t* cfg, const moe_weights_t* weights,
                              const uint16_t* x_host, uint16_t* x_dev, uint16_t* out_dev,
                              uint16_t* out_host, const moe_outputs_t* outputs, void* ws,
                              size_t ws_bytes, void* h2d_stream, void* compute_stream,
                              void* d2h_stream);

/*
 * moe_permute_static - moe_permute for callers that cannot allocate device
 * memory and have no workspace to give: for example a plugin running inside
 * an inference engine that owns all device memory and forbids allocation on
 * its execution path, or a service that reserves all memory at start-up.
 * The source pages have no counterpart to this entry point: it computes
 * exactly what moe_permute computes (same arithmetic, same outputs), but its
 * scratch is one fixed array in device memory that the library holds on
 * every device it is loaded on until the process exits.
 *   Arguments and outputs are those of moe_permute, without ws/ws_bytes.
 *   Limits: T*k <= MOE_STATIC_MAX_ASSIGNMENTS and N <= MOE_STATIC_MAX_EXPERTS;
 *   larger sizes return MOE_ERR_UNSUPPORTED before anything is enqueued.
 *   The call allocates nothing (no cudaMalloc/cudaFree).  Its first call on a
 *   device looks up the array's device address (cudaGetSymbolAddress) with
 *   that device current.  Under CUDA's default lazy module loading that
 *   first call is also when the library's code and this 768 KiB array are
 *   placed in that device's memory, so it can fail with MOE_ERR_CUDA in a
 *   process that has already reserved all device memory: make one call on
 *   each device at start-up, before reserving memory and before any stream
 *   capture; later calls take no device memory.  Every call shares the one
 *   array, which keeps the last call's contents (nothing in it needs
 *   clearing: each call writes every entry it reads); calls that overlap on
 *   the GPU - on different streams, or from different threads - race on it
 *   and must be serialised.
 */
#define MOE_STATIC_MAX_ASSIGNMENTS 65536
#define MOE_STATIC_MAX_EXPERTS 256
moe_status_t moe_permute_static(const moe_config_t* cfg, const int32_t* topk_idx,
                                const float* p_mean, int32_t* counts, int32_t* offsets,
                                int32_t* perm, int32_t* inv, float* f, float* l_aux,
                                void* stream);

/* Synchronises `stream` and returns the device status word of `ws`
 * (MOE_OK or MOE_ERR_TIMEOUT), or MOE_ERR_CUDA if the synchronisation fails. */
moe_status_t moe_workspace_status(const void* ws, void* stream);

/* Failure-injection hook for tests; the source pages have no counterpart.
 * The next `launches` expert-GEMM launches enqueued by this process (by
 * moe_expert_ffn or moe_forward, on any device) run with their TMA producer
 * issuing nothing, as if its signals were lost.  The MMA issuer and the
 * epilogue warps then wait until their bound runs out (about 2 s of SM
 * clocks), record MOE_ERR_TIMEOUT in the workspace status word and return
 * without touching the output; the CUDA context stays usable.  The count is
 * process-wide and is consumed at launch time, so a graph captured while it
 * is non-zero keeps the suppressed launches.  0 switches the hook off.
 * Returns MOE_ERR_INVALID_ARG for launches < 0, else MOE_OK. */
moe_status_t moe_debug_suppress_gemm_producer(int launches);

/* Static description of a status code. */
const char* moe_status_string(moe_status_t status);

/* Library version string. */
const char* moe_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_H */
