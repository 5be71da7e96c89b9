// Dispatch: per-expert histogram, capacity, stable expert-contiguous scatter,
// and the load-balance statistic.
//
// "混合专家模型 MoE 架构深度解析" §2.3 (Capacity = floor(T/N * capacity_factor);
// tokens over capacity pass through with no expert output), §2.2
// (L_aux = alpha * N * sum f_i p_i); "AI-Research-SKILLs MoE 训练实战" §4.3
// (f from bincount of the top-k indices over their count), §4.4 (drop_tokens).
//
// Assignments claim slots in a fixed order of positions p: p = a = t*k + j
// (token-major) or p = j*T + t (slot-major: every token's first choice
// first).  Each is ranked within its expert in increasing p (a stable
// scatter), so the first C claimants of each expert keep a row.
// Two launches, all integer work and no atomics on values:
//   1. rank + scan: per 256-assignment chunk, rank of each assignment among
//               the chunk's assignments to the same expert + the chunk
//               histogram; the last block to finish (integer ticket) then
//               scans: chunk bases per expert (in chunk order), counts,
//               capacity, row offsets, f and L_aux
//   2. scatter: row = offsets[e] + base + local rank, or dropped
// (Without a ticket, e.g. for the workspace-free entry point, the scan is a
// launch of its own.)  In a forward pass with token-major claims the router
// ranks and counts the assignments of its chunks instead, and one launch
// (dispatch_fused_kernel) scans and scatters.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {

constexpr int PR_THREADS = kPermuteChunk;
constexpr int PR_WARPS = PR_THREADS / 32;

// position p of assignment a (and back): the claim order
__device__ __forceinline__ int64_t claim_pos(int64_t a, int T, int k, int slot_major) {
  return slot_major ? (a % k) * T + a / k : a;
}
__device__ __forceinline__ int64_t claim_assignment(int64_t p, int T, int k, int slot_major) {
  return slot_major ? (p % T) * k + p / T : p;
}

// The scan over the chunk histograms, by one block of any multiple of 32
// threads.  Thread e takes experts e, e + blockDim, ... and walks the chunks
// in order (loads coalesced across the experts, eight in flight), so the
// bases come out in chunk order.  Then warp 0 turns the kept counts into row
// offsets and reduces L_aux in a fixed order.  `s_kept` holds N ints of
// shared memory.
__device__ void scan_experts_block(const int32_t* __restrict__ blk_hist,
                                   int32_t* __restrict__ blk_base, int32_t* __restrict__ counts,
                                   int32_t* __restrict__ offsets,
                                   const float* __restrict__ p_mean, float* __restrict__ f,
                                   float* __restrict__ l_aux, int nblk, int N, int64_t A,
                                   int64_t capacity, float alpha, int32_t* s_kept) {
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  constexpr int U = 8;
  for (int e = threadIdx.x; e < N; e += blockDim.x) {
    int run = 0;
    int b = 0;
    for (; b + U <= nblk; b += U) {
      int c[U];
#pragma unroll
      for (int u = 0; u < U; ++u) c[u] = __ldcg(blk_hist + (size_t)(b + u) * N + e);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        blk_base[(size_t)(b + u) * N + e] = run;
        run += c[u];
      }
    }
    for (; b < nblk; ++b) {
      const int c = __ldcg(blk_hist + (size_t)b * N + e);
      blk_base[(size_t)b * N + e] = run;
      run += c;
    }
    counts[e] = run;
    s_kept[e] = (int)((capacity >= 0 && run > capacity) ? capacity : run);
    if (f) f[e] = A > 0 ? (float)((double)run / (double)A) : 0.0f;
  }
  __syncthreads();
  if (warp == 0) {
    // offsets: exclusive scan of kept over the experts, contiguous per lane
    const int epl = (N + 31) / 32;
    const int e0 = min(N, lane * epl), e1 = min(N, e0 + epl);
    int sum = 0;
    double term = 0.0;
    for (int e = e0; e < e1; ++e) {
      sum += s_kept[e];
      if (l_aux) term += (A > 0 ? (double)counts[e] / (double)A : 0.0) * (double)p_mean[e];
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - sum;
    for (int e = e0; e < e1; ++e) {
      offsets[e] = run;
      run += s_kept[e];
    }
    if (lane == 31) offsets[N] = incl;
    // fixed-order reduction of the per-lane L_aux terms
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) term += __shfl_xor_sync(0xffffffffu, term, o);
    if (lane == 0 && l_aux) *l_aux = (float)((double)alpha * (double)N * term);
  }
}

// local_rank and the chunk histograms are indexed by claim position p.
// With a ticket, the last block to finish also runs the scan.
__global__ void __launch_bounds__(PR_THREADS) permute_rank_kernel(
    const int32_t* __restrict__ idx, int32_t* __restrict__ local_rank,
    int32_t* __restrict__ blk_hist, int64_t A, int N, int T, int k, int slot_major,
    int* __restrict__ ticket, int32_t* __restrict__ blk_base, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, const float* __restrict__ p_mean, float* __restrict__ f,
    float* __restrict__ l_aux, int64_t capacity, float alpha) {
  extern __shared__ int32_t wcnt[];  // [PR_WARPS][N]; later the scan's kept counts
  __shared__ int s_last;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  pdl_launch_dependents();
  for (int i = tid; i < PR_WARPS * N; i += PR_THREADS) wcnt[i] = 0;
  pdl_wait();
  __syncthreads();
  const int64_t a = (int64_t)blockIdx.x * PR_THREADS + tid;   // claim position p
  int e = (a < A) ? idx[claim_assignment(a, T, k, slot_major)] : -1;
  if (e < 0 || e >= N) e = -1;  // out-of-range indices take no slot
  const uint32_t peers = __match_any_sync(0xffffffffu, e);
  const int wrank = __popc(peers & ((1u << lane) - 1u));
  if (e >= 0 && wrank == 0) wcnt[warp * N + e] = __popc(peers);
  __syncthreads();
  // exclusive scan over the warps, per expert; the chunk total is the histogram
  for (int ex = tid; ex < N; ex += PR_THREADS) {
    int run = 0;
#pragma unroll
    for (int w = 0; w < PR_WARPS; ++w) {
      const int c = wcnt[w * N + ex];
      wcnt[w * N + ex] = run;
      run += c;
    }
    blk_hist[(size_t)blockIdx.x * N + ex] = run;
  }
  __syncthreads();
  if (a < A) local_rank[a] = (e >= 0) ? wcnt[warp * N + e] + wrank : -1;
  if (ticket == nullptr) return;
  // last block: every histogram is written (release by each block's fence
  // before its ticket, acquire by the last one after)
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(ticket, 1) == (int)gridDim.x - 1 ? 1 : 0;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  scan_experts_block(blk_hist, blk_base, counts, offsets, p_mean, f, l_aux, (int)gridDim.x, N, A,
                     capacity, alpha, wcnt);
}

// The scan as a launch of its own (one block of 1024 threads).
__global__ void __launch_bounds__(1024) permute_scan_kernel(
    const int32_t* __restrict__ blk_hist, int32_t* __restrict__ blk_base,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets, const float* __restrict__ p_mean,
    float* __restrict__ f, float* __restrict__ l_aux, int nblk, int N, int64_t A,
    int64_t capacity, float alpha) {
  __shared__ int32_t s_kept[MOE_MAX_EXPERTS];
  pdl_launch_dependents();
  pdl_wait();
  scan_experts_block(blk_hist, blk_base, counts, offsets, p_mean, f, l_aux, nblk, N, A, capacity,
                     alpha, s_kept);
}

__global__ void __launch_bounds__(256) permute_scatter_kernel(
    const int32_t* __restrict__ idx, const int32_t* __restrict__ local_rank,
    const int32_t* __restrict__ blk_base, const int32_t* __restrict__ offsets,
    int32_t* __restrict__ perm, int32_t* __restrict__ inv, int64_t A, int N, int64_t capacity,
    int T, int k, int slot_major) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t a = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (a >= A) return;
  const int e = idx[a];
  if (e < 0 || e >= N) { inv[a] = -1; return; }
  const int64_t p = claim_pos(a, T, k, slot_major);
  const int64_t pos = (int64_t)blk_base[(p / kPermuteChunk) * N + e] + local_rank[p];
  if (capacity >= 0 && pos >= capacity) { inv[a] = -1; return; }
  const int32_t row = offsets[e] + (int32_t)pos;
  perm[row] = (int32_t)a;
  inv[a] = row;
}

// The scatter fused with the row gather of the expert GEMMs' A operand: one
// warp per token writes perm / inv of its k assignments, reads x[t] once and
// copies it into each kept slot's expert-contiguous row xp[row] (16-byte
// vectors across lanes).
__global__ void __launch_bounds__(256) permute_scatter_gather_kernel(
    const int32_t* __restrict__ idx, const int32_t* __restrict__ local_rank,
    const int32_t* __restrict__ blk_base, const int32_t* __restrict__ offsets,
    int32_t* __restrict__ perm, int32_t* __restrict__ inv, int T, int N, int k,
    int64_t capacity, const __nv_bfloat16* __restrict__ x, __nv_bfloat16* __restrict__ xp, int H,
    int slot_major) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x % 32;
  const int64_t nvec = H / 8;
  for (int64_t t = (int64_t)blockIdx.x * 8 + threadIdx.x / 32; t < T; t += (int64_t)gridDim.x * 8) {
    // rows of the token's slots: lane j computes slot j (k <= 32)
    int32_t row = -1;
    if (lane < k) {
      const int64_t a = t * k + lane;
      const int e = idx[a];
      if (e >= 0 && e < N) {
        const int64_t p = slot_major ? (int64_t)lane * T + t : a;
        const int64_t pos = (int64_t)blk_base[(p / kPermuteChunk) * N + e] + local_rank[p];
        if (capacity < 0 || pos < capacity) row = offsets[e] + (int32_t)pos;
      }
      inv[a] = row;
      if (row >= 0) perm[row] = (int32_t)a;
    }
    const unsigned kept_mask = __ballot_sync(0xffffffffu, row >= 0);
    if (kept_mask == 0u) continue;
    const uint4* src = reinterpret_cast<const uint4*>(x + t * H);
    for (int64_t v = lane; v < nvec; v += 32) {
      const uint4 val = __ldg(src + v);
      unsigned m = kept_mask;
      while (m) {
        const int j = __ffs(m) - 1;
        m &= m - 1;
        const int32_t r = __shfl_sync(0xffffffffu, row, j);
        reinterpret_cast<uint4*>(xp + (int64_t)r * H)[v] = val;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Dispatch after a fused router (token choice, token-major claims).  The
// router's CTAs each wrote, for their chunk of consecutive tokens, the
// local rank of every assignment and the chunk's expert histogram.  CTA 0
// of this launch scans them: per expert the chunk bases (prefix over chunks,
// in chunk order), the counts, the capacity, the row offsets, f_i; p_i and
// the z-loss from the router's per-chunk partial sums (fixed order); L_aux.
// It then releases a flag (zeroed by the router), and every CTA - which
// waits for the flag, bounded - scatters its tokens: row = offsets[e] +
// base[chunk][e] + local rank, or dropped past the capacity, with the token's
// x row copied into each kept row.  The grid never exceeds the CTAs that fit
// at once, so CTA 0 always runs.
constexpr int DF_THREADS = 512;

__device__ __forceinline__ void st_release_gpu(int* p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__global__ void __launch_bounds__(DF_THREADS) dispatch_fused_kernel(const DispatchFusedLaunch a) {
  __shared__ int32_t s_part[DF_THREADS];
  __shared__ int32_t s_cnt[kRouterTcMaxExperts];
  __shared__ float s_red[DF_THREADS];
  __shared__ int s_ok;
  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const int N = a.N, C = a.chunks;
  const int64_t A = (int64_t)a.T * a.k;
  pdl_launch_dependents();
  pdl_wait();
  if (blockIdx.x == 0) {
    // chunk bases: P threads per expert, each over a run of chunks
    const int P = DF_THREADS / N > 0 ? DF_THREADS / N : 1;
    const int cp = (C + P - 1) / P;
    const int e = tid / P, part = tid % P;
    const bool act = e < N;
    const int c0 = part * cp, c1 = min(C, c0 + cp);
    int sum = 0;
    if (act)
      for (int c = c0; c < c1; ++c) sum += __ldcg(a.blk_hist + (size_t)c * N + e);
    s_part[tid] = sum;
    __syncthreads();
    if (act) {
      int base = 0;
      for (int p2 = 0; p2 < part; ++p2) base += s_part[e * P + p2];
      for (int c = c0; c < c1; ++c) {
        a.blk_base[(size_t)c * N + e] = base;
        base += __ldcg(a.blk_hist + (size_t)c * N + e);
      }
      if (part == P - 1) s_cnt[e] = base;   // every chunk: the expert's count
    }
    __syncthreads();
    // p_i and the z-loss from the router's per-chunk sums (fixed order)
    reduce_router_partials(a.p_part, C, N, a.T, a.p_mean, a.z_loss, s_red);
    if (warp == 0) {
      // counts, f, capacity, offsets (exclusive scan of the kept counts,
      // contiguous runs of experts per lane) and L_aux (fixed order, double)
      const int epl = (N + 31) / 32;
      const int e0 = min(N, lane * epl), e1 = min(N, e0 + epl);
      int run_k = 0;
      double term = 0.0;
      for (int e2 = e0; e2 < e1; ++e2) {
        const int cnt = s_cnt[e2];
        a.counts[e2] = cnt;
        const double fe = A > 0 ? (double)cnt / (double)A : 0.0;
        if (a.f) a.f[e2] = (float)fe;
        term += fe * (double)a.p_mean[e2];
        run_k += (int)((a.capacity >= 0 && cnt > a.capacity) ? a.capacity : cnt);
      }
      int incl = run_k;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      int run = incl - run_k;
      for (int e2 = e0; e2 < e1; ++e2) {
        a.offsets[e2] = run;
        const int cnt = s_cnt[e2];
        run += (int)((a.capacity >= 0 && cnt > a.capacity) ? a.capacity : cnt);
      }
      if (lane == 31) a.offsets[N] = incl;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) term += __shfl_xor_sync(0xffffffffu, term, o);
      if (lane == 0 && a.l_aux) *a.l_aux = (float)((double)a.alpha * (double)N * term);
    }
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      st_release_gpu(a.flag, 1);
    }
  } else {
    if (tid == 0) {
      int ok = 1;
      const long long t0 = clock64();
      while (ld_acquire_gpu(a.flag) == 0) {
        if (clock64() - t0 > kWaitLimitCycles) {
          atomicExch(a.status, (int)MOE_ERR_TIMEOUT);
          ok = 0;
          break;
        }
      }
      s_ok = ok;
    }
    __syncthreads();
    if (!s_ok) return;
  }
  // scatter and gather: one warp per token, lane j < k for slot j
  const int64_t nvec = a.H / 8;
  constexpr int WPB = DF_THREADS / 32;
  for (int64_t t = (int64_t)blockIdx.x * WPB + warp; t < a.T; t += (int64_t)gridDim.x * WPB) {
    int32_t row = -1;
    if (lane < a.k) {
      const int64_t as = t * a.k + lane;
      const int e = a.topk_idx[as];
      if (e >= 0 && e < N) {
        const int64_t pos = (int64_t)__ldcg(a.blk_base + (t / a.chunk_tokens) * N + e) +
                            a.local_rank[as];
        if (a.capacity < 0 || pos < a.capacity) row = __ldcg(a.offsets + e) + (int32_t)pos;
      }
      a.inv[as] = row;
      if (row >= 0) a.perm[row] = (int32_t)as;
    }
    const unsigned kept_mask = __ballot_sync(0xffffffffu, row >= 0);
    if (kept_mask == 0u || a.xp == nullptr) continue;
    const uint4* src = reinterpret_cast<const uint4*>(a.x + t * a.H);
    // four 16-byte loads in flight per lane, then their copies into every kept row
    for (int64_t v0 = lane; v0 < nvec; v0 += 4 * 32) {
      uint4 val[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (v0 + u * 32 < nvec) val[u] = __ldg(src + v0 + u * 32);
      unsigned mk = kept_mask;
      while (mk) {
        const int j = __ffs(mk) - 1;
        mk &= mk - 1;
        const int32_t r = __shfl_sync(0xffffffffu, row, j);
        uint4* dst = reinterpret_cast<uint4*>(a.xp + (int64_t)r * a.H);
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (v0 + u * 32 < nvec) dst[v0 + u * 32] = val[u];
      }
    }
  }
}

cudaError_t launch_dispatch_fused(const DispatchFusedLaunch& a, cudaStream_t st, LaunchTrace* tr) {
  // at most two CTAs per SM (the kernel's registers allow that many):
  // every CTA is resident while CTA 0 scans
  int64_t blocks = ((int64_t)a.T + DF_THREADS / 32 - 1) / (DF_THREADS / 32);
  if (blocks > 148 * 2) blocks = 148 * 2;
  if (blocks < 1) blocks = 1;
  trace_mark(tr, st);
  return launch_pdl(dispatch_fused_kernel, dim3((unsigned)blocks), dim3(DF_THREADS), 0, st, 1, a);
}

int permute_num_launches(int T, int k, bool fused_scan) {
  if ((int64_t)T * k == 0) return 1;  // the scan alone
  return fused_scan ? 2 : 3;
}

cudaError_t launch_permute(const PermuteLaunch& a, cudaStream_t st, LaunchTrace* tr) {
  const int64_t A = (int64_t)a.T * a.k;
  const int nblk = permute_num_blocks(A);
  const bool fused = a.ticket != nullptr && A > 0;
  const size_t rank_smem = sizeof(int32_t) * (size_t)PR_WARPS * a.N;
  if (A > 0) {
    trace_mark(tr, st);
    cudaError_t err = launch_pdl(permute_rank_kernel, dim3(nblk), dim3(PR_THREADS), rank_smem, st,
                                 1, a.topk_idx, a.local_rank, a.blk_hist, A, a.N, a.T, a.k,
                                 a.slot_major, fused ? a.ticket : static_cast<int*>(nullptr),
                                 a.blk_base, a.counts, a.offsets, a.p_mean, a.f, a.l_aux,
                                 a.capacity, a.alpha);
    if (err != cudaSuccess) return err;
  }
  if (!fused) {
    trace_mark(tr, st);
    cudaError_t err = launch_pdl(permute_scan_kernel, dim3(1), dim3(1024), 0, st, 1, a.blk_hist,
                                 a.blk_base, a.counts, a.offsets, a.p_mean, a.f, a.l_aux, nblk,
                                 a.N, A, a.capacity, a.alpha);
    if (err != cudaSuccess || A == 0) return err;
  }
  trace_mark(tr, st);
  if (a.x != nullptr) {
    int64_t blocks = ((int64_t)a.T + 7) / 8;
    if (blocks > 148 * 16) blocks = 148 * 16;
    return launch_pdl(permute_scatter_gather_kernel, dim3((unsigned)blocks), dim3(256), 0, st, 1,
                      a.topk_idx, a.local_rank, a.blk_base, a.offsets, a.perm, a.inv, a.T, a.N,
                      a.k, a.capacity, a.x, a.xp, a.H, a.slot_major);
  } else {
    return launch_pdl(permute_scatter_kernel, dim3((unsigned)((A + 255) / 256)), dim3(256), 0, st,
                      1, a.topk_idx, a.local_rank, a.blk_base, a.offsets, a.perm, a.inv, A, a.N,
                      a.capacity, a.T, a.k, a.slot_major);
  }
  return cudaGetLastError();
}

}  // namespace moe
