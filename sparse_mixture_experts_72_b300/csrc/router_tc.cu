// Router on the tensor cores: fp32 gate logits from an exact three-way bf16
// split of W_g, with softmax, top-k, renormalisation and the per-expert mean
// probability fused into the TMEM epilogue.
//
// "混合专家模型 MoE 架构深度解析" §1.2 (gate_weights = Softmax(x . W_g)), §1.3
// (top-K steps 1-3), §2.4 (selection on logits_i - b_i); "AI-Research-SKILLs
// MoE 训练实战" §3.1 (gate Linear with bias, softmax, topk, renormalise) and
// §4.3 (p = mean softmax, for L_aux).
//
// Exactness of the logits: x is bf16 and W_g is fp32.  W_g = hi + mid + lo
// with hi, mid, lo bf16 (round-to-nearest at each step) is exact, because
// each residual has at most 24 - 8k significant bits.  Each product of two
// bf16 values is exact in fp32, so x . W_g^T = x.hi^T + x.mid^T + x.lo^T is
// an fp32-accumulated sum of exact products: the same accuracy class as an
// fp32 FFMA dot product.  The three planes are stored side by side along K,
// W3 [N_pad, 3 * H_pad], and the MMA walks K three times over the x tile.
//
// One CTA per 128 tokens, 192 threads:
//   warp 0     TMA producer (x tile 128 x 64, W3 tile N_pad x 64, 4 stages)
//   warp 1     TMEM allocator and MMA issuer (M=128, N=N_pad, K=16)
//   warps 2-5  epilogue, one token per thread (TMEM lane = token row):
//              pass 1 streams the token's N logits in 16-column chunks,
//              keeping an online max/sum for the softmax and a sorted top-k
//              of l - b_sel in registers; pass 2 re-reads the logits to form
//              P for the optional probs output and the CTA's column sums.
// The last CTA to finish (integer ticket) reduces the per-CTA column sums in
// CTA order into p_mean, so the result does not depend on scheduling.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {

constexpr int RT_BM = 128, RT_BK = 64, RT_STAGES = 4;
constexpr int RT_THREADS = 192;
constexpr int RT_A_BYTES = RT_BM * RT_BK * 2;

// W3[e, p * H_pad + h] = plane p of W_g[e, h]; zero outside [0,N) x [0,H).
__global__ void __launch_bounds__(256) router_split_kernel(const float* __restrict__ Wg,
                                                           __nv_bfloat16* __restrict__ W3, int N,
                                                           int H, int N_pad, int H_pad) {
  const int64_t total = (int64_t)N_pad * H_pad;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int e = (int)(i / H_pad), h = (int)(i % H_pad);
    const float w = (e < N && h < H) ? Wg[(size_t)e * H + h] : 0.0f;
    const __nv_bfloat16 hi = __float2bfloat16_rn(w);
    const float r1 = w - __bfloat162float(hi);
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(mid);
    const __nv_bfloat16 lo = __float2bfloat16_rn(r2);
    __nv_bfloat16* row = W3 + (size_t)e * 3 * H_pad;
    row[h] = hi;
    row[H_pad + h] = mid;
    row[2 * H_pad + h] = lo;
  }
}

template <int KMAX>
__global__ void __launch_bounds__(RT_THREADS, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                     RouterTcArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int N = args.N, N_pad = args.N_pad, k = args.k;
  const int b_bytes = N_pad * RT_BK * 2;
  const int stage_bytes = RT_A_BYTES + b_bytes;
  const uint32_t s0 = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + RT_STAGES * stage_bytes);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (RT_STAGES + s); };
  const uint32_t tfull_bar = bar0 + 8u * (2 * RT_STAGES);
  const uint32_t drain_bar = bar0 + 8u * (2 * RT_STAGES + 1);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * RT_STAGES + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* is_last = reinterpret_cast<int*>(tmem_holder + 2);
  float* psum = reinterpret_cast<float*>(tmem_holder + 4);  // [4][N_pad]

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int t0 = blockIdx.x * RT_BM;
  const int KB = args.H_pad / RT_BK;
  const int nkb = 3 * KB;
  int* status = args.status;

  if (threadIdx.x == 0) {
    for (int s = 0; s < RT_STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(tfull_bar, 1);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmW);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), args.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  long long tma_issued = 0;

  if (warp == 0) {
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      for (int kb = 0; kb < nkb; ++kb) {
        if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, status)) break;
        const int kx = kb / 3, p = kb % 3;  // x tile reused by three consecutive planes
        const uint32_t sa = s0 + stage * stage_bytes;
        mbar_arrive_expect_tx(full_bar(stage), stage_bytes);
        tma_load_2d(sa, &tmX, full_bar(stage), kx * RT_BK, t0);
        tma_load_2d(sa + RT_A_BYTES, &tmW, full_bar(stage), p * args.H_pad + kx * RT_BK, 0);
        ++tma_issued;
        if (++stage == RT_STAGES) { stage = 0; phase ^= 1u; }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(RT_BM, N_pad);
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int kb = 0; kb < nkb; ++kb) {
        if (!mbar_wait_bounded(full_bar(stage), phase, abort_flag, status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t sa = s0 + stage * stage_bytes;
        const uint64_t adesc = sdesc_kmajor_sw128(sa);
        const uint64_t bdesc = sdesc_kmajor_sw128(sa + RT_A_BYTES);
#pragma unroll
        for (int kk = 0; kk < RT_BK / 16; ++kk)
          umma_bf16(tmem_base, adesc + 2 * kk, bdesc + 2 * kk, idesc, (kb | kk) != 0 ? 1u : 0u);
        umma_commit(empty_bar(stage));
        if (++stage == RT_STAGES) { stage = 0; phase ^= 1u; }
      }
      if (ok) umma_commit(tfull_bar);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int t = t0 + row;
    const bool valid = t < args.T;
    const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
    int ok = 1;
    if (lane == 0) ok = mbar_wait_bounded(tfull_bar, 0, abort_flag, status) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) {
      tc_fence_after();
      float m = -INFINITY, z = 0.0f;
      float tv[KMAX], tl[KMAX];
      int ti[KMAX];
#pragma unroll
      for (int j = 0; j < KMAX; ++j) { tv[j] = -INFINITY; tl[j] = -INFINITY; ti[j] = 0x7fffffff; }
      // pass 1: online softmax statistics and the top-k of l - b_sel
      for (int c = 0; c < N_pad; c += 16) {
        uint32_t r[16];
        tmem_ld_32x32b_x16(tmem_base + lane_addr + c, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int e = c + i;
          if (e >= N) break;
          const float l = __uint_as_float(r[i]) + (args.bg ? args.bg[e] : 0.0f);
          if (l > m) {
            z = z * expf(m - l) + 1.0f;
            m = l;
          } else {
            z += expf(l - m);
          }
          float sv = args.sel_bias ? l - args.sel_bias[e] : l;
          float lv = l;
          int ei = e;
          // insertion into the descending list; an equal score stays behind
          // the earlier (lower-index) expert
#pragma unroll
          for (int j = 0; j < KMAX; ++j) {
            if (sv > tv[j]) {
              const float a = tv[j], b = tl[j];
              const int c2 = ti[j];
              tv[j] = sv; tl[j] = lv; ti[j] = ei;
              sv = a; lv = b; ei = c2;
            }
          }
        }
      }
      // renormalised weights of the k chosen experts (unbiased softmax)
      float wsum = 0.0f;
#pragma unroll
      for (int j = 0; j < KMAX; ++j)
        if (j < k) wsum += expf(tl[j] - m);
      if (valid) {
        const float inv = 1.0f / wsum;
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
          if (j < k) {
            args.topk_idx[(size_t)t * k + j] = ti[j];
            args.topk_w[(size_t)t * k + j] = expf(tl[j] - m) * inv;
          }
        }
      }
      // pass 2: P = exp(l - m) / z for the probs output and the column sums
      const float inv_z = 1.0f / z;
      for (int c = 0; c < N_pad; c += 16) {
        uint32_t r[16];
        tmem_ld_32x32b_x16(tmem_base + lane_addr + c, r);
        tmem_ld_wait();
        float pv[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int e = c + i;
          const float l = __uint_as_float(r[i]) + ((args.bg && e < N) ? args.bg[e] : 0.0f);
          pv[i] = (valid && e < N) ? expf(l - m) * inv_z : 0.0f;
        }
        if (args.probs && valid) {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (c + i < N) args.probs[(size_t)t * N + c + i] = pv[i];
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float v = pv[i];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          if (lane == 0) psum[q * N_pad + c + i] = v;
        }
      }
    }
    tc_fence_before();
    // column sums over the 4 epilogue warps, in warp order
    named_barrier(1, 128);
    if (!*abort_flag) {
      for (int e = threadIdx.x - 64; e < N; e += 128)
        args.p_part[(size_t)blockIdx.x * N + e] =
            ((psum[0 * N_pad + e] + psum[1 * N_pad + e]) + psum[2 * N_pad + e]) + psum[3 * N_pad + e];
    }
    __threadfence();
    named_barrier(1, 128);
    if (threadIdx.x == 64) *is_last = (atomicAdd(args.ticket, 1) == (int)gridDim.x - 1) ? 1 : 0;
    named_barrier(1, 128);
    if (*is_last) {
      __threadfence();
      const int nb = gridDim.x;
      for (int e = threadIdx.x - 64; e < N; e += 128) {
        // fixed association: 8 interleaved partial sums, then a fixed tree
        float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        int b = 0;
        for (; b + 8 <= nb; b += 8) {
#pragma unroll
          for (int u = 0; u < 8; ++u) acc[u] += __ldcg(args.p_part + (size_t)(b + u) * N + e);
        }
        for (int u = 0; b < nb; ++b, ++u) acc[u] += __ldcg(args.p_part + (size_t)b * N + e);
        const float s = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
        args.p_mean[e] = args.T > 0 ? s / (float)args.T : 0.0f;
      }
      if (threadIdx.x == 64) *args.ticket = 0;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    if (warp == 0 && lane == 0) {
      const long long first = tma_issued > RT_STAGES ? tma_issued - RT_STAGES : 0;
      for (long long j = first; j < tma_issued; ++j) {
        const long long t0c = clock64();
        while (!mbar_try_wait(full_bar((int)(j % RT_STAGES)), (uint32_t)((j / RT_STAGES) & 1)))
          if (clock64() - t0c > 200000000LL) break;
      }
    }
    if (warp == 1 && lane == 0) {
      umma_commit(drain_bar);
      const long long t0c = clock64();
      while (!mbar_try_wait(drain_bar, 0))
        if (clock64() - t0c > 200000000LL) break;
    }
    __syncwarp();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, args.tmem_cols);
  }
}

// ---------------------------------------------------------------------------
// host side

int router_tc_smem_bytes(int N_pad) {
  return 1024 + RT_STAGES * (RT_A_BYTES + N_pad * RT_BK * 2) + (2 * RT_STAGES + 2) * 8 + 16 +
         4 * N_pad * 4;
}

cudaError_t launch_router_tc(const RouterLaunch& a, __nv_bfloat16* W3, int* ticket, int* status,
                             cudaStream_t st, LaunchTrace* tr) {
  const int N_pad = (a.N + 15) / 16 * 16;
  const int H_pad = (a.H + RT_BK - 1) / RT_BK * RT_BK;
  if (a.T == 0) {
    trace_mark(tr, st);
    return cudaMemsetAsync(a.p_mean, 0, sizeof(float) * a.N, st);
  }
  {
    const int64_t total = (int64_t)N_pad * H_pad;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 148 * 8) blocks = 148 * 8;
    trace_mark(tr, st);
    router_split_kernel<<<(unsigned)blocks, 256, 0, st>>>(a.Wg, W3, a.N, a.H, N_pad, H_pad);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  CUtensorMap tmX, tmW;
  if (!encode_tensor_map_bf16(&tmX, a.x, a.T, a.H, RT_BK, RT_BM)) return cudaErrorInvalidValue;
  if (!encode_tensor_map_bf16(&tmW, W3, N_pad, 3 * H_pad, RT_BK, N_pad)) return cudaErrorInvalidValue;
  RouterTcArgs args;
  args.bg = a.bg;
  args.sel_bias = a.sel_bias;
  args.topk_idx = a.topk_idx;
  args.topk_w = a.topk_w;
  args.probs = a.probs;
  args.p_part = a.p_part;
  args.p_mean = a.p_mean;
  args.ticket = ticket;
  args.status = status;
  args.T = a.T;
  args.N = a.N;
  args.N_pad = N_pad;
  args.H_pad = H_pad;
  args.k = a.k;
  int cols = 32;
  while (cols < N_pad) cols <<= 1;
  args.tmem_cols = cols;
  const int smem = router_tc_smem_bytes(N_pad);
  const int grid = (a.T + RT_BM - 1) / RT_BM;
  trace_mark(tr, st);
#define MOE_RTC(KM)                                                                            \
  do {                                                                                         \
    cudaError_t e = cudaFuncSetAttribute(router_tc_kernel<KM>,                                 \
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);   \
    if (e != cudaSuccess) return e;                                                            \
    router_tc_kernel<KM><<<grid, RT_THREADS, smem, st>>>(tmX, tmW, args);                      \
  } while (0)
  if (a.k <= 1) MOE_RTC(1);
  else if (a.k <= 2) MOE_RTC(2);
  else if (a.k <= 4) MOE_RTC(4);
  else if (a.k <= 8) MOE_RTC(8);
  else if (a.k <= 16) MOE_RTC(16);
  else MOE_RTC(32);
#undef MOE_RTC
  return cudaGetLastError();
}

}  // namespace moe
