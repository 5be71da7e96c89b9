// Expert-choice dispatch: each expert takes the C tokens with the largest
// router logits in its column.
//
// "AI-Research-SKILLs MoE 训练实战" §4.2 (expert_scores = router(x) with the
// token and expert axes swapped, top-k along the tokens with k =
// capacity_per_expert) and §7.3 (perfect balance, no token dropped for
// load); the capacity is "混合专家模型 MoE 架构深度解析" §2.3's formula.
//
// One CTA per expert.  The column of logits is staged in shared memory as
// order-preserving 32-bit keys; a 4-pass radix select (8 bits per pass,
// histograms in shared memory) finds the C-th largest key K and how many of
// the keys equal to K must be taken.  Equal logits take the lower token
// first, so the chosen set is unique; two block-wide scans over contiguous
// token segments then give every chosen token its row, in token order:
//   rows of expert e: [e*C, (e+1)*C), perm[row] = t*N + e, inv[t*N + e] = row
// Integer work only after the keys are formed: the result is bit-exact.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {

constexpr int EC_THREADS = 1024;

// Larger float -> larger key; -0 and +0 get the same key (they compare equal).
__device__ __forceinline__ uint32_t ec_key(float v) {
  const uint32_t u = __float_as_uint(v == 0.0f ? 0.0f : v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive scan of one value per thread over the block (EC_THREADS threads);
// `total` receives the sum.  `sh` holds 32 ints.
__device__ __forceinline__ int ec_block_scan(int v, int* sh, int& total) {
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) sh[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = sh[lane];
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += u;
    }
    sh[lane] = wi - w;                      // exclusive prefix of the warps
    if (lane == 31) sh[32] = wi;            // block total
  }
  __syncthreads();
  const int r = sh[warp] + incl - v;
  total = sh[32];
  __syncthreads();  // sh is reused by the next scan
  return r;
}

__global__ void __launch_bounds__(EC_THREADS) expert_choice_kernel(
    const float* __restrict__ logits, const float* __restrict__ p_mean, int T, int N, int C,
    float alpha, int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
    int32_t* __restrict__ perm, int32_t* __restrict__ inv, float* __restrict__ f,
    float* __restrict__ l_aux) {
  extern __shared__ uint32_t keys[];  // [T]
  __shared__ int hist[256];
  __shared__ int sh[33];
  __shared__ uint32_t s_prefix;
  __shared__ int s_remaining;
  const int e = blockIdx.x;
  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  pdl_launch_dependents();
  pdl_wait();

  if (tid == 0) {
    counts[e] = C;
    offsets[e] = e * C;
    if (e == N - 1) offsets[N] = N * C;
    if (f) f[e] = 1.0f / (float)N;
    if (e == 0 && l_aux) {
      // every expert takes the same share: f_i = 1/N; fixed order in double
      double s = 0.0;
      for (int i = 0; i < N; ++i) s += (1.0 / (double)N) * (double)p_mean[i];
      *l_aux = (float)((double)alpha * (double)N * s);
    }
  }
  if (C == 0) {
    for (int t = tid; t < T; t += EC_THREADS) inv[(size_t)t * N + e] = -1;
    return;
  }
  for (int t = tid; t < T; t += EC_THREADS) keys[t] = ec_key(logits[(size_t)t * N + e]);

  // ---- radix select: the C-th largest key, 8 bits per pass from the top
  uint32_t prefix = 0u, mask = 0u;
  int remaining = C;  // keys still to take among those matching the prefix
  for (int shift = 24; shift >= 0; shift -= 8) {
    if (tid < 256) hist[tid] = 0;
    __syncthreads();
    for (int t = tid; t < T; t += EC_THREADS) {
      const uint32_t k = keys[t];
      if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1);
    }
    __syncthreads();
    if (warp == 0) {
      // lane l owns the digits 255-8l .. 248-8l (descending)
      int cnt = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) cnt += hist[255 - 8 * lane - j];
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
      }
      const unsigned hit = __ballot_sync(0xffffffffu, incl >= remaining);
      const int L = __ffs(hit) - 1;  // remaining <= keys matching the prefix, so hit != 0
      if (lane == L) {
        int run = incl - cnt;
        for (int j = 0; j < 8; ++j) {
          const int d = 255 - 8 * lane - j;
          const int c = hist[d];
          if (run + c >= remaining) {
            s_prefix = prefix | ((uint32_t)d << shift);
            s_remaining = remaining - run;
            break;
          }
          run += c;
        }
      }
    }
    __syncthreads();
    prefix = s_prefix;
    remaining = s_remaining;
    mask |= 255u << shift;
  }
  const uint32_t K = prefix;    // the C-th largest key
  const int need_eq = remaining;  // keys equal to K that are taken (lowest tokens first)

  // ---- rows in token order: contiguous token segments per thread
  const int seg = (T + EC_THREADS - 1) / EC_THREADS;
  const int ta = min(T, tid * seg), tb = min(T, ta + seg);
  int n_eq = 0;
  for (int t = ta; t < tb; ++t) n_eq += keys[t] == K ? 1 : 0;
  int tot;
  int eq_rank = ec_block_scan(n_eq, sh, tot);
  int n_sel = 0;
  {
    int r = eq_rank;
    for (int t = ta; t < tb; ++t) {
      const uint32_t k = keys[t];
      if (k > K) ++n_sel;
      else if (k == K) { if (r < need_eq) ++n_sel; ++r; }
    }
  }
  int row = e * C + ec_block_scan(n_sel, sh, tot);
  {
    int r = eq_rank;
    for (int t = ta; t < tb; ++t) {
      const uint32_t k = keys[t];
      bool take = k > K;
      if (k == K) { take = r < need_eq; ++r; }
      const int64_t a = (int64_t)t * N + e;
      if (take) {
        perm[row] = (int32_t)a;
        inv[a] = row;
        ++row;
      } else {
        inv[a] = -1;
      }
    }
  }
}

cudaError_t launch_expert_choice(const float* logits, const float* p_mean, int T, int N, int C,
                                 float alpha, int32_t* counts, int32_t* offsets, int32_t* perm,
                                 int32_t* inv, float* f, float* l_aux, cudaStream_t st,
                                 LaunchTrace* tr) {
  const size_t smem = sizeof(uint32_t) * (size_t)(T > 0 ? T : 1);
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(expert_choice_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(sizeof(uint32_t) * kExpertChoiceMaxTokens));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  trace_mark(tr, st);
  return launch_pdl(expert_choice_kernel, dim3(N), dim3(EC_THREADS), smem, st, 1, logits, p_mean,
                    T, N, C, alpha, counts, offsets, perm, inv, f, l_aux);
}

// ---------------------------------------------------------------------------
// Auxiliary-loss-free balancing step ("混合专家模型 MoE 架构深度解析" §2.4):
// sel_bias[e] += gamma * sign(counts[e] - mean), compared exactly in
// integers as counts[e] * N against the total.  One block.
__global__ void __launch_bounds__(1024) update_sel_bias_kernel(const int32_t* __restrict__ counts,
                                                               float* __restrict__ sel_bias, int N,
                                                               float gamma) {
  __shared__ long long part[32];
  pdl_launch_dependents();
  pdl_wait();
  long long s = 0;
  for (int e = threadIdx.x; e < N; e += blockDim.x) s += counts[e];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (threadIdx.x % 32 == 0) part[threadIdx.x / 32] = s;
  __syncthreads();
  long long total = 0;
  for (int w = 0; w < (int)(blockDim.x + 31) / 32; ++w) total += part[w];
  for (int e = threadIdx.x; e < N; e += blockDim.x) {
    const long long d = (long long)counts[e] * N - total;
    const float step = d > 0 ? gamma : (d < 0 ? -gamma : 0.0f);
    sel_bias[e] += step;
  }
}

cudaError_t launch_update_sel_bias(const int32_t* counts, float* sel_bias, int N, float gamma,
                                   cudaStream_t st) {
  return launch_pdl(update_sel_bias_kernel, dim3(1), dim3(1024), 0, st, 1, counts, sel_bias, N,
                    gamma);
}

}  // namespace moe
