// Row gather into the expert-contiguous layout, and the per-token weighted
// combine back through the inverse permutation.
//
// "AI-Research-SKILLs MoE 训练实战" §3.1 (x_flat[mask] gathers the tokens of an
// expert; output[mask] += score * expert_output sums them back) and §6.1
// (hidden_states[idx] gather, index_add_ combine).  The gate weight is
// applied in the second GEMM's epilogue, so the combine is a plain sum of at
// most k rows per token, in slot order, with a single writer per output.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {

// xp[r] = x[perm[r] / k] for r < offsets[N]; one warp per row, 16-byte copies.
__global__ void __launch_bounds__(256) gather_rows_kernel(const __nv_bfloat16* __restrict__ x,
                                                          const int32_t* __restrict__ perm,
                                                          const int32_t* __restrict__ offsets,
                                                          int N, int k, int64_t max_rows, int H,
                                                          __nv_bfloat16* __restrict__ xp) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t R = offsets[N];
  const int lane = threadIdx.x % 32;
  const int64_t nvec = H / 8;
  for (int64_t r = (int64_t)blockIdx.x * 8 + threadIdx.x / 32; r < R && r < max_rows;
       r += (int64_t)gridDim.x * 8) {
    const int64_t t = perm[r] / k;
    const uint4* src = reinterpret_cast<const uint4*>(x + t * H);
    uint4* dst = reinterpret_cast<uint4*>(xp + r * H);
    for (int64_t v = lane; v < nvec; v += 32) dst[v] = __ldg(src + v);
  }
}

// out[t, c:c+8] = sum_j y[inv[t*k+j], c:c+8] (+ y_shared[t, c:c+8]), fp32 sum.
__global__ void __launch_bounds__(256) combine_kernel(const __nv_bfloat16* __restrict__ y,
                                                      const int32_t* __restrict__ inv,
                                                      const __nv_bfloat16* __restrict__ ys,
                                                      __nv_bfloat16* __restrict__ out, int T,
                                                      int k, int H) {
  pdl_launch_dependents();
  pdl_wait();
  const int nvec = H / 8;
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (gid >= (int64_t)T * nvec) return;
  const int64_t t = gid / nvec;
  const int c = (int)(gid % nvec) * 8;
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  auto add8 = [&](const __nv_bfloat16* p) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    acc[0] += bf16lo(u.x); acc[1] += bf16hi(u.x);
    acc[2] += bf16lo(u.y); acc[3] += bf16hi(u.y);
    acc[4] += bf16lo(u.z); acc[5] += bf16hi(u.z);
    acc[6] += bf16lo(u.w); acc[7] += bf16hi(u.w);
  };
  for (int j = 0; j < k; ++j) {
    const int32_t r = inv[t * k + j];
    if (r >= 0) add8(y + (int64_t)r * H + c);
  }
  if (ys) add8(ys + t * H + c);
  uint4 o;
  o.x = pack_bf16x2(acc[0], acc[1]);
  o.y = pack_bf16x2(acc[2], acc[3]);
  o.z = pack_bf16x2(acc[4], acc[5]);
  o.w = pack_bf16x2(acc[6], acc[7]);
  *reinterpret_cast<uint4*>(out + t * H + c) = o;
}

cudaError_t launch_gather(const __nv_bfloat16* x, const int32_t* perm, const int32_t* offsets,
                          int N, int k, int64_t max_rows, int H, __nv_bfloat16* xp,
                          cudaStream_t st, LaunchTrace* tr) {
  int64_t blocks = (max_rows + 7) / 8;
  if (blocks > 148 * 16) blocks = 148 * 16;
  if (blocks < 1) blocks = 1;
  trace_mark(tr, st);
  return launch_pdl(gather_rows_kernel, dim3((unsigned)blocks), dim3(256), 0, st, 1, x, perm,
                    offsets, N, k, max_rows, H, xp);
}

cudaError_t launch_combine(const __nv_bfloat16* y, const int32_t* inv,
                           const __nv_bfloat16* y_shared, __nv_bfloat16* out, int T, int k,
                           int H, cudaStream_t st, LaunchTrace* tr) {
  const int64_t n = (int64_t)T * (H / 8);
  if (n == 0) return cudaSuccess;
  trace_mark(tr, st);
  return launch_pdl(combine_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, st, 1, y, inv,
                    y_shared, out, T, k, H);
}

}  // namespace moe
