// Router: gate Linear in fp32, softmax over the N experts, top-k selection on
// the logits minus the selection-only bias, renormalisation of the k weights,
// and the per-expert mean gate probability p_i.
//
// "混合专家模型 MoE 架构深度解析" §1.2 (gate_weights = Softmax(x . W_g)), §1.3
// (steps 1-3 of top-K routing), §2.4 (adjusted_logits_i = logits_i - b_i used
// for selection); "AI-Research-SKILLs MoE 训练实战" §3.1 (gate is nn.Linear
// with bias; softmax, topk, divide by the sum) and §4.3 (p = mean softmax).
#include "common.cuh"
#include "kernels.cuh"

namespace moe {

// ---------------------------------------------------------------------------
// logits[T, N] = x[T, H] (bf16 -> fp32) . Wg[N, H]^T + bg   (fp32 FFMA)
//
// 64 tokens x 64 experts per 256-thread block, K staged through shared memory
// 32 at a time, 4 x 4 outputs per thread.

constexpr int RL_BT = 64, RL_BE = 64, RL_BK = 32;

__global__ void __launch_bounds__(256) router_logits_kernel(const __nv_bfloat16* __restrict__ x,
                                                            const float* __restrict__ Wg,
                                                            const float* __restrict__ bg,
                                                            float* __restrict__ logits, int T,
                                                            int H, int N) {
  __shared__ float xs[RL_BK][RL_BT + 4];
  __shared__ float wsm[RL_BK][RL_BE + 4];
  pdl_launch_dependents();
  pdl_wait();
  const int tid = threadIdx.x;
  const int t0 = blockIdx.x * RL_BT;
  const int e0 = blockIdx.y * RL_BE;
  const int tx = tid % 16, ty = tid / 16;  // tx -> experts, ty -> tokens
  float acc[4][4] = {};
  for (int k0 = 0; k0 < H; k0 += RL_BK) {
    // x tile: 64 rows x 32 cols, 8 bf16 per thread (one 16-byte load)
    {
      const int r = tid / 4, c = (tid % 4) * 8;
      const int t = t0 + r, kk = k0 + c;
      float v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      if (t < T && kk < H) {  // H % 8 == 0, so the 8-vector is all in or all out
        const uint4 u = *reinterpret_cast<const uint4*>(x + (size_t)t * H + kk);
        v[0] = bf16lo(u.x); v[1] = bf16hi(u.x); v[2] = bf16lo(u.y); v[3] = bf16hi(u.y);
        v[4] = bf16lo(u.z); v[5] = bf16hi(u.z); v[6] = bf16lo(u.w); v[7] = bf16hi(u.w);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) xs[c + i][r] = v[i];
    }
    // W tile: 64 experts x 32 cols fp32, 8 per thread (two 16-byte loads)
    {
      const int r = tid / 4, c = (tid % 4) * 8;
      const int e = e0 + r, kk = k0 + c;
      float v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      if (e < N && kk < H) {
        const float4 a = *reinterpret_cast<const float4*>(Wg + (size_t)e * H + kk);
        const float4 b = *reinterpret_cast<const float4*>(Wg + (size_t)e * H + kk + 4);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) wsm[c + i][r] = v[i];
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < RL_BK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = xs[kk][ty + 16 * i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = wsm[kk][tx + 16 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + ty + 16 * i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + tx + 16 * j;
      if (e < N) logits[(size_t)t * N + e] = acc[i][j] + (bg ? bg[e] : 0.0f);
    }
  }
}

// ---------------------------------------------------------------------------
// softmax + top-k + renormalise: one warp per token; lane l holds experts
// l, l+32, ...  Each block also writes its column sums of P for p_i.

constexpr int RS_WARPS = 8, RS_TOK_PER_WARP = 4;
constexpr int RS_TOK_PER_BLOCK = RS_WARPS * RS_TOK_PER_WARP;

template <int NPL>
__global__ void __launch_bounds__(RS_WARPS * 32) router_select_kernel(
    const float* __restrict__ logits, const float* __restrict__ sel_bias,
    int32_t* __restrict__ topk_idx, float* __restrict__ topk_w, float* __restrict__ probs,
    float* __restrict__ p_part, int T, int N, int k) {
  __shared__ float psum[RS_WARPS][NPL * 32];
  __shared__ float zsum[RS_WARPS];
  pdl_launch_dependents();
  pdl_wait();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  float zacc = 0.0f;  // this warp's sum of logsumexp(l_t)^2 (router z-loss)
  float pacc[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) pacc[i] = 0.0f;
  for (int it = 0; it < RS_TOK_PER_WARP; ++it) {
    const int t = blockIdx.x * RS_TOK_PER_BLOCK + warp * RS_TOK_PER_WARP + it;
    if (t >= T) break;
    float l[NPL], s[NPL];
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const int e = lane + 32 * i;
      l[i] = (e < N) ? logits[(size_t)t * N + e] : -INFINITY;
      s[i] = (e < N) ? (sel_bias ? l[i] - sel_bias[e] : l[i]) : -INFINITY;
      m = fmaxf(m, l[i]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float z = 0.0f;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      l[i] = (lane + 32 * i < N) ? expf(l[i] - m) : 0.0f;  // l now holds exp(l - m)
      z += l[i];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    {
      const float lse = m + logf(z);
      zacc += lse * lse;
    }
    const float inv_z = 1.0f / z;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      l[i] *= inv_z;  // l now holds P
      pacc[i] += l[i];
      const int e = lane + 32 * i;
      if (probs && e < N) probs[(size_t)t * N + e] = l[i];
    }
    if (topk_idx == nullptr) continue;  // expert choice: no per-token selection
    // k rounds of warp arg-max on s; ties go to the lower expert index
    float selp[MOE_MAX_TOP_K > 32 ? 32 : MOE_MAX_TOP_K];
    int seli[MOE_MAX_TOP_K > 32 ? 32 : MOE_MAX_TOP_K];
    float psel = 0.0f;
    for (int j = 0; j < k; ++j) {
      float bv = -INFINITY;
      int be = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < NPL; ++i) {
        const int e = lane + 32 * i;
        if (e < N && (s[i] > bv || (s[i] == bv && e < be))) { bv = s[i]; be = e; }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        if (ov > bv || (ov == bv && oe < be)) { bv = ov; be = oe; }
      }
      // owner lane knocks the winner out and broadcasts its probability
      float pw = 0.0f;
#pragma unroll
      for (int i = 0; i < NPL; ++i) {
        if (lane + 32 * i == be) { pw = l[i]; s[i] = -INFINITY; }
      }
      pw = __shfl_sync(0xffffffffu, pw, be % 32);
      if (j < 32) { selp[j] = pw; seli[j] = be; }
      psel += pw;
    }
    if (lane == 0) {
      const float inv_sel = 1.0f / psel;
      for (int j = 0; j < k; ++j) {
        topk_idx[(size_t)t * k + j] = seli[j];
        topk_w[(size_t)t * k + j] = selp[j] * inv_sel;
      }
    }
  }
#pragma unroll
  for (int i = 0; i < NPL; ++i) psum[warp][lane + 32 * i] = pacc[i];
  if (lane == 0) zsum[warp] = zacc;
  __syncthreads();
  for (int e = threadIdx.x; e <= N; e += blockDim.x) {
    float acc = 0.0f;
#pragma unroll
    for (int w = 0; w < RS_WARPS; ++w) acc += e < N ? psum[w][e] : zsum[w];
    p_part[(size_t)blockIdx.x * (N + 1) + e] = acc;
  }
}

// p_mean[e] = column sum over the blocks / T; column N of the block sums is
// the router z-loss numerator.  One block; with nblocks = 0 it zeroes both.
__global__ void __launch_bounds__(256) router_pmean_kernel(const float* __restrict__ p_part,
                                                           float* __restrict__ p_mean,
                                                           float* __restrict__ z_loss, int nblocks,
                                                           int N, int T) {
  __shared__ float red[256];
  pdl_launch_dependents();
  pdl_wait();
  if (N + 1 <= 256) {
    reduce_router_partials(p_part, nblocks, N, T, p_mean, z_loss, red);
    return;
  }
  for (int e = threadIdx.x; e <= N; e += blockDim.x) {  // many experts: one thread per column
    float acc = 0.0f;
    for (int b = 0; b < nblocks; ++b) acc += p_part[(size_t)b * (N + 1) + e];
    const float mean = T > 0 ? acc / (float)T : 0.0f;
    if (e < N) p_mean[e] = mean;
    else if (z_loss) *z_loss = mean;
  }
}

cudaError_t launch_router_stats_zero(float* p_mean, float* z_loss, int N, cudaStream_t st) {
  return launch_pdl(router_pmean_kernel, dim3(1), dim3(256), 0, st, 1,
                    static_cast<const float*>(nullptr), p_mean, z_loss, 0, N, 0);
}

// ---------------------------------------------------------------------------
// host launchers

int router_num_select_blocks(int T) { return (T + RS_TOK_PER_BLOCK - 1) / RS_TOK_PER_BLOCK; }

cudaError_t launch_router(const RouterLaunch& a, cudaStream_t st, LaunchTrace* tr) {
  const int T = a.T, N = a.N;
  const int nsel = router_num_select_blocks(T);
  if (T > 0) {
    dim3 grid((T + RL_BT - 1) / RL_BT, (N + RL_BE - 1) / RL_BE);
    trace_mark(tr, st);
    float* lg = a.logits_out ? a.logits_out : a.logits;
    cudaError_t err = launch_pdl(router_logits_kernel, grid, dim3(256), 0, st, 1, a.x, a.Wg, a.bg,
                                 lg, T, a.H, N);
    if (err != cudaSuccess) return err;
    const int npl = (N + 31) / 32;
    trace_mark(tr, st);
#define MOE_SEL(NPLV)                                                                      \
  err = launch_pdl(router_select_kernel<NPLV>, dim3(nsel), dim3(RS_WARPS * 32), 0, st, 1,        \
                   static_cast<const float*>(lg), a.sel_bias, a.topk_idx, a.topk_w, a.probs,      \
                   a.p_part, T, N, a.k)
    if (npl <= 1) MOE_SEL(1);
    else if (npl <= 2) MOE_SEL(2);
    else if (npl <= 4) MOE_SEL(4);
    else if (npl <= 8) MOE_SEL(8);
    else if (npl <= 16) MOE_SEL(16);
    else MOE_SEL(32);
#undef MOE_SEL
    if (err != cudaSuccess) return err;
  }
  trace_mark(tr, st);
  return launch_pdl(router_pmean_kernel, dim3(1), dim3(256), 0, st, 1,
                    static_cast<const float*>(a.p_part), a.p_mean, a.z_loss, nsel, N, T);
}

int router_num_launches(int T, int N, int H) {
  // tensor-core router: [W_g split kernel, unless the router splits itself] + router
  if (N <= kRouterTcMaxExperts) return T > 0 ? (router_own_split(T, N, H) ? 1 : 2) : 1;
  return T > 0 ? 3 : 1;
}

}  // namespace moe
