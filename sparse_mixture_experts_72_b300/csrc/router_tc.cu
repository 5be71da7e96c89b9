// Router on the tensor cores: fp32 gate logits from an exact three-way bf16
// split of W_g, with softmax, top-k, renormalisation and the per-expert mean
// probability fused into the epilogue.
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
// fp32 FFMA dot product.
//
// Layout of the three planes:
//   stacked (3 N_pad <= 256): rows p*N_pad + e of each ring slot's B tile, so
//            one MMA with N = 3 N_pad covers all planes; when a CTA streams
//            at most 16 x tiles the epilogue warps, idle during the main
//            loop, split W_g's slice of every slot into shared memory
//            themselves (no split kernel, no W3), else router_split_kernel
//            writes W3 as a [3 N_pad, H_pad] matrix;
//   along K (wider routers): W3[e, p*H_pad + h] written by
//            router_split_kernel, one plane per MMA.
// Consecutive k-steps go round-robin to `nacc` independent TMEM accumulators
// so that the MMAs of a stage do not wait on one another; the epilogue adds
// accumulators and planes back up in a fixed order.
//
// One CTA per (128-token tile, K split).  With few token tiles the K range is
// split over the CTAs of a thread-block cluster (up to 8): each CTA parks its
// partial logits in its own shared memory, and after a cluster barrier CTA s
// sums rows [s*128/S, (s+1)*128/S) of all the partials in split order through
// distributed shared memory, so the result does not depend on scheduling.
//
// 192 threads: warp 0 TMA producer (also prefetching x tiles into L2 one
// ring ahead), warp 1 TMEM allocator and MMA issuer, warps 2-5 epilogue with
// one token per thread: the logits go TMEM -> shared memory, then pass 1
// keeps an online max/sum for the softmax and a sorted top-k of l - b_sel in
// registers and pass 2 forms P for the optional probs output and the CTA's
// column sums.  The last CTA to finish (integer ticket) reduces the per-CTA
// column sums in CTA order into p_mean.  In a forward pass with token-major
// claims the router also starts the dispatch ("混合专家模型 MoE 架构深度解析"
// §2.3): each CTA ranks its chunk's assignments per expert from per-expert
// token bitmasks and writes the chunk's histogram, and the scatter launch
// (dispatch_fused_kernel) reduces p_mean, so no ticket is needed.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {

constexpr int RT_BM = 128, RT_BK = 64, RT_MAX_STAGES = 8;
constexpr int RT_THREADS = 192;
constexpr int RT_A_BYTES = RT_BM * RT_BK * 2;
constexpr int kRouterTcSmemMax = 227 * 1024;

// Plane p of W_g: hi, mid, lo with W_g = hi + mid + lo exactly.
// It also zeroes `clear` (the header of a forward pass's workspace: status
// word, router ticket and the expert FFN's row-block counters), which saves
// a separate memset launch.
__global__ void __launch_bounds__(256) router_split_kernel(const float* __restrict__ Wg,
                                                           __nv_bfloat16* __restrict__ W3, int N,
                                                           int H, int N_pad, int H_pad,
                                                           int stacked, int* clear, int clear_n) {
  pdl_launch_dependents();
  pdl_wait();
  if (clear && blockIdx.x == 0)
    for (int i = threadIdx.x; i < clear_n; i += blockDim.x) clear[i] = 0;
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
    if (stacked) {
      W3[((size_t)0 * N_pad + e) * H_pad + h] = hi;
      W3[((size_t)1 * N_pad + e) * H_pad + h] = mid;
      W3[((size_t)2 * N_pad + e) * H_pad + h] = lo;
    } else {
      __nv_bfloat16* row = W3 + (size_t)e * 3 * H_pad;
      row[h] = hi;
      row[H_pad + h] = mid;
      row[2 * H_pad + h] = lo;
    }
  }
}


__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t cluster_addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(cluster_addr)
               : "memory");
  return v;
}

template <int KMAX>
__global__ void __launch_bounds__(RT_THREADS, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                     RouterTcArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int N = args.N, N_pad = args.N_pad, k = args.k;
  const bool stacked = args.stacked != 0;
  const int mma_n = stacked ? 3 * N_pad : N_pad;     // N of one MMA
  const int b_bytes = mma_n * RT_BK * 2;             // one B tile
  const int PP = stacked ? 1 : args.planes_per_stage;  // B tiles per stage
  const int STAGES = args.stages;
  const int stage_bytes = RT_A_BYTES + PP * b_bytes;
  const int nacc = args.nacc;
  const int acc_cols = mma_n;                        // TMEM columns per accumulator
  const int ld = N_pad + 4;                          // row stride of the logits tile (floats)
  const uint32_t s0 = smem_u32(smem);
  float* ltile = reinterpret_cast<float*>(smem);     // [128][ld], reuses the ring afterwards
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + args.work_bytes);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (RT_MAX_STAGES + s); };
  const uint32_t tfull_bar = bar0 + 8u * (2 * RT_MAX_STAGES);
  const uint32_t drain_bar = bar0 + 8u * (2 * RT_MAX_STAGES + 1);
  // W_g planes of a ring slot written by the epilogue warps (in-kernel split)
  auto bfull_bar = [&](int s) { return bar0 + 8u * (2 * RT_MAX_STAGES + 2 + s); };
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 3 * RT_MAX_STAGES + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* flags = reinterpret_cast<int*>(tmem_holder + 2);      // [0] last CTA
  float* psum = reinterpret_cast<float*>(tmem_holder + 4);   // [4][N_pad]
  float* zsum = psum + 4 * N_pad;                            // [4]
  uint32_t* tmask = reinterpret_cast<uint32_t*>(zsum + 4);   // [N_pad][4]: tokens per expert
  const bool own_split = args.Wg != nullptr;                 // stacked planes split here
  const bool fused = args.local_rank != nullptr;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  pdl_launch_dependents();
  const int S = args.splits;                                 // cluster size
  const int split = S > 1 ? (int)cluster_ctarank() : 0;      // K split
  const int mt = blockIdx.x / S;                             // token tile
  const int t0 = mt * RT_BM;
  const int KB = args.H_pad / RT_BK;
  const int kx0 = split * args.kb_per_split;
  const int kx1 = min(KB, kx0 + args.kb_per_split);
  // stages this CTA streams: one per x tile (stacked, or all planes per
  // stage), or three (one per plane)
  const int per_x = stacked ? 1 : 3 / PP;
  const int nst = (kx1 > kx0 ? kx1 - kx0 : 0) * per_x;
  const int rows_per = RT_BM / S;                            // rows this CTA finishes
  const int row_lo = split * rows_per;
  int* status = args.status;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
      mbar_init(bfull_bar(s), 4);   // the four epilogue warps
    }
    mbar_init(tfull_bar, 1);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmX);
    if (!own_split) tma_prefetch_desc(&tmW);
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
  pdl_wait();  // the W_g planes, x and the ticket come from earlier launches
  if (args.clear && blockIdx.x == 0 && warp >= 2) {
    // the forward pass's header (status word, dispatch flag, the expert
    // FFN's counters): no kernel before this one in the call clears it
    for (int i = threadIdx.x - 64; i < args.clear_n; i += RT_THREADS - 64) args.clear[i] = 0;
  }

  if (warp == 0) {
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      for (int st = 0; st < nst; ++st) {
        // x tiles a ring ahead go to L2 now, so their loads hit L2 later
        const int pf = st + STAGES;
        if (pf < nst && pf % per_x == 0) tma_prefetch_l2_2d(&tmX, (kx0 + pf / per_x) * RT_BK, t0);
        if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, status)) break;
        const int kx = kx0 + st / per_x;
        const uint32_t sa = s0 + stage * stage_bytes;
        mbar_arrive_expect_tx(full_bar(stage), own_split ? RT_A_BYTES : stage_bytes);
        tma_load_2d(sa, &tmX, full_bar(stage), kx * RT_BK, t0);
        for (int pp = 0; pp < (own_split ? 0 : PP); ++pp) {
          // stacked: all planes in one tile at column kx*64;
          // along K: plane p's tile at column p*H_pad + kx*64
          const int p = PP == 3 ? pp : st % per_x;
          const int col = stacked ? kx * RT_BK : p * args.H_pad + kx * RT_BK;
          tma_load_2d(sa + RT_A_BYTES + pp * b_bytes, &tmW, full_bar(stage), col, 0);
        }
        ++tma_issued;
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(RT_BM, mma_n);
      uint32_t stage = 0, phase = 0;
      uint32_t step = 0;  // MMA counter: accumulator = step % nacc
      bool ok = true;
      for (int st = 0; st < nst; ++st) {
        if (!mbar_wait_bounded(full_bar(stage), phase, abort_flag, status)) { ok = false; break; }
        if (own_split && !mbar_wait_bounded(bfull_bar(stage), phase, abort_flag, status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = s0 + stage * stage_bytes;
        const uint64_t adesc = sdesc_kmajor_sw128(sa);
        for (int pp = 0; pp < PP; ++pp) {
          const uint64_t bdesc = sdesc_kmajor_sw128(sa + RT_A_BYTES + pp * b_bytes);
#pragma unroll
          for (int kk = 0; kk < RT_BK / 16; ++kk, ++step) {
            const uint32_t a = step % (uint32_t)nacc;
            umma_bf16(tmem_base + a * acc_cols, adesc + 2 * kk, bdesc + 2 * kk, idesc,
                      step >= (uint32_t)nacc ? 1u : 0u);
          }
        }
        umma_commit(empty_bar(stage));
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
      if (ok) umma_commit(tfull_bar);
    }
    __syncwarp();
  } else {
    if (own_split) {
      // ---- E0: the three bf16 planes of W_g for each ring slot, written in
      // the 128-byte swizzled layout the MMA reads (rows p * N_pad + e of 64
      // values; 16-byte chunk c of row r at c ^ (r % 8)).  hi = bf16(w),
      // mid = bf16(w - hi), lo = bf16(w - hi - mid): hi + mid + lo = w
      // exactly, so x . W_g^T accumulates exact products in fp32.
      const int et = threadIdx.x - 64;
      uint32_t stage = 0, phase = 0;
      for (int st = 0; st < nst; ++st) {
        int ok = 1;
        if (lane == 0) ok = mbar_wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, status) ? 1 : 0;
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        const int col0 = (kx0 + st) * RT_BK;
        uint8_t* bt = smem + stage * stage_bytes + RT_A_BYTES;
        for (int it = et; it < N_pad * 8; it += 128) {
          const int e = it >> 3, c = it & 7;
          const int col = col0 + c * 8;
          float w[8];
          if (e < N && col < args.H) {
            const float4 a = __ldg(reinterpret_cast<const float4*>(args.Wg + (size_t)e * args.H + col));
            const float4 b = __ldg(reinterpret_cast<const float4*>(args.Wg + (size_t)e * args.H + col + 4));
            w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w; w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
          } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) w[i] = 0.0f;
          }
          uint32_t ph[3][4];
#pragma unroll
          for (int i = 0; i < 8; i += 2) {
            float r0 = w[i], r1 = w[i + 1];
#pragma unroll
            for (int pl = 0; pl < 3; ++pl) {
              const __nv_bfloat16 h0 = __float2bfloat16_rn(r0), h1 = __float2bfloat16_rn(r1);
              ph[pl][i / 2] = (uint32_t)__bfloat16_as_ushort(h0) |
                              ((uint32_t)__bfloat16_as_ushort(h1) << 16);
              r0 -= __bfloat162float(h0);
              r1 -= __bfloat162float(h1);
            }
          }
#pragma unroll
          for (int pl = 0; pl < 3; ++pl) {
            const int r = pl * N_pad + e;
            *reinterpret_cast<uint4*>(bt + (r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4)) =
                make_uint4(ph[pl][0], ph[pl][1], ph[pl][2], ph[pl][3]);
          }
        }
        fence_proxy_async_shared();   // the tensor cores read what the threads wrote
        __syncwarp();
        if (lane == 0) mbar_arrive(bfull_bar(stage));
        if (++stage == (uint32_t)STAGES) { stage = 0; phase ^= 1u; }
      }
    }
    // ---- E1: this CTA's (partial) logits, TMEM -> shared-memory tile.  The
    // ring is idle once every MMA has completed (tmem_full), so the tile
    // reuses its space.  Accumulators and planes are added in a fixed order.
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
    const int nplanes_cols = stacked ? 3 : 1;
    const int nld = nacc * nplanes_cols;  // 3 (stacked) or 2 (along K)
    int ok = 1;
    if (lane == 0) ok = mbar_wait_bounded(tfull_bar, 0, abort_flag, status) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) {
      tc_fence_after();
      for (int c = 0; c < N_pad; c += 16) {
        uint32_t r0[16], r1[16], r2[16];
        tmem_ld_32x32b_x16(tmem_base + lane_addr + c, r0);
        const uint32_t off1 = nplanes_cols == 3 ? (uint32_t)N_pad : (uint32_t)acc_cols;
        tmem_ld_32x32b_x16(tmem_base + lane_addr + off1 + c, r1);
        if (nld == 3) tmem_ld_32x32b_x16(tmem_base + lane_addr + 2 * N_pad + c, r2);
        tmem_ld_wait();
        float l[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          l[i] = __uint_as_float(r0[i]) + __uint_as_float(r1[i]);
          if (nld == 3) l[i] += __uint_as_float(r2[i]);
        }
        float4* dst = reinterpret_cast<float4*>(ltile + (size_t)row * ld + c);
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[i] = make_float4(l[4 * i], l[4 * i + 1], l[4 * i + 2], l[4 * i + 3]);
      }
    }
    tc_fence_before();
  }

  // ---- E2: with a K split, CTA s sums rows [row_lo, row_lo + rows_per) of
  // every CTA's partial tile, in split order, into its own tile.
  __syncthreads();
  if (S > 1) {
    cluster_sync_all();  // every partial tile of the cluster is complete
    const int q4 = N_pad / 4;
    const uint32_t my_base = smem_u32(ltile);
    for (int i = threadIdx.x; i < rows_per * q4; i += RT_THREADS) {
      const int r = row_lo + i / q4, c = (i % q4) * 4;
      const uint32_t off = (uint32_t)((r * ld + c) * 4);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int s2 = 0; s2 < S; ++s2) {
        const float4 v = ld_dsmem_f4(mapa_shared(my_base + off, (uint32_t)s2));
        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
      }
      *reinterpret_cast<float4*>(ltile + (size_t)r * ld + c) = acc;
    }
    cluster_sync_all();  // no CTA overwrites or leaves while others still read it
  }

  if (warp >= 2) {
    if (args.logits_out && !*abort_flag) {
      // the finished logits of this CTA's rows, row-contiguous stores
      for (int i = threadIdx.x - 64; i < rows_per * N; i += 128) {
        const int r = row_lo + i / N, e = i % N;
        if (t0 + r < args.T)
          args.logits_out[(size_t)(t0 + r) * N + e] =
              ltile[(size_t)r * ld + e] + (args.bg ? args.bg[e] : 0.0f);
      }
    }
    // ---- E3: one token per thread for this CTA's rows
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int t = t0 + row;
    const bool mine = row >= row_lo && row < row_lo + rows_per;
    const bool valid = mine && t < args.T && !*abort_flag;
    const float* lrow = ltile + (size_t)row * ld;
    float m = -INFINITY, z = 0.0f;
    float tv[KMAX], tl[KMAX];
    int ti[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) { tv[j] = -INFINITY; tl[j] = -INFINITY; ti[j] = 0x7fffffff; }
    if (valid) {
      // pass 1: online softmax statistics and the top-k of l - b_sel
      for (int e = 0; e < N; ++e) {
        const float l = lrow[e] + (args.bg ? args.bg[e] : 0.0f);
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
      // renormalised weights of the k chosen experts (unbiased softmax)
      if (args.topk_idx) {
        float wsum = 0.0f;
#pragma unroll
        for (int j = 0; j < KMAX; ++j)
          if (j < k) wsum += expf(tl[j] - m);
        const float inv = 1.0f / wsum;
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
          if (j < k) {
            args.topk_idx[(size_t)t * k + j] = ti[j];
            args.topk_w[(size_t)t * k + j] = expf(tl[j] - m) * inv;
          }
        }
      }
    }
    if (fused) {
      // dispatch ranks of this CTA's chunk (its rows, in token order): the
      // rank of (t, j) among the chunk's assignments to expert e is the
      // number of earlier chunk tokens that chose e (a token's k experts
      // are distinct), read from a per-expert token bitmask
      const int et = threadIdx.x - 64;
      for (int i = et; i < N_pad * 4; i += 128) tmask[i] = 0u;
      named_barrier(1, 128);
      const int lr = row - row_lo;   // token index inside the chunk (< 128)
      if (valid) {
#pragma unroll
        for (int j = 0; j < KMAX; ++j)
          if (j < k) atomicOr(&tmask[ti[j] * 4 + (lr >> 5)], 1u << (lr & 31));
      }
      named_barrier(1, 128);
      if (valid) {
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
          if (j < k) {
            const uint32_t* mk = tmask + ti[j] * 4;
            int rank = __popc(mk[lr >> 5] & ((1u << (lr & 31)) - 1u));
            for (int wd = 0; wd < (lr >> 5); ++wd) rank += __popc(mk[wd]);
            args.local_rank[(size_t)t * k + j] = rank;
          }
        }
      }
      for (int e = et; e < N; e += 128)
        args.blk_hist[(size_t)blockIdx.x * N + e] =
            __popc(tmask[e * 4]) + __popc(tmask[e * 4 + 1]) + __popc(tmask[e * 4 + 2]) +
            __popc(tmask[e * 4 + 3]);
    }
    // router z-loss term of the token: logsumexp(l_t)^2
    {
      float zt = 0.0f;
      if (valid) {
        const float lse = m + logf(z);
        zt = lse * lse;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) zt += __shfl_xor_sync(0xffffffffu, zt, o);
      if (lane == 0) zsum[q] = zt;
    }
    // pass 2: P = exp(l - m) / z for the probs output and the column sums
    // (every lane takes part in the shuffles; rows not finished here add 0)
    const float inv_z = valid ? 1.0f / z : 0.0f;
    for (int c = 0; c < N_pad; c += 16) {
      float pv[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int e = c + i;
        pv[i] = (valid && e < N) ? expf(lrow[e] + (args.bg ? args.bg[e] : 0.0f) - m) * inv_z : 0.0f;
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
    // column sums over the 4 epilogue warps, in warp order
    named_barrier(1, 128);
    if (!*abort_flag) {
      for (int e = threadIdx.x - 64; e < N; e += 128)
        args.p_part[(size_t)blockIdx.x * (N + 1) + e] =
            ((psum[0 * N_pad + e] + psum[1 * N_pad + e]) + psum[2 * N_pad + e]) +
            psum[3 * N_pad + e];
      if (threadIdx.x == 64)
        args.p_part[(size_t)blockIdx.x * (N + 1) + N] = ((zsum[0] + zsum[1]) + zsum[2]) + zsum[3];
    }
    if (!fused) {
    __threadfence();
    named_barrier(1, 128);
    if (threadIdx.x == 64) flags[0] = (atomicAdd(args.ticket, 1) == (int)gridDim.x - 1) ? 1 : 0;
    named_barrier(1, 128);
    if (flags[0]) {
      __threadfence();
      const int nb = gridDim.x;
      const int W = N + 1;
      for (int e = threadIdx.x - 64; e <= N; e += 128) {
        // fixed association: 8 interleaved partial sums, then a fixed tree
        float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        int b = 0;
        for (; b + 8 <= nb; b += 8) {
#pragma unroll
          for (int u = 0; u < 8; ++u) acc[u] += __ldcg(args.p_part + (size_t)(b + u) * W + e);
        }
        for (int u = 0; b < nb; ++b, ++u) acc[u] += __ldcg(args.p_part + (size_t)b * W + e);
        const float s2 = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
        const float mean = args.T > 0 ? s2 / (float)args.T : 0.0f;
        if (e < N) args.p_mean[e] = mean;
        else if (args.z_loss) *args.z_loss = mean;
      }
    }
    }  // !fused
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    if (warp == 0 && lane == 0) {
      const long long first = tma_issued > STAGES ? tma_issued - STAGES : 0;
      for (long long j = first; j < tma_issued; ++j) {
        const long long t0c = clock64();
        while (!mbar_try_wait(full_bar((int)(j % STAGES)), (uint32_t)((j / STAGES) & 1)))
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

RouterTcPlan router_tc_plan(int T, int N, int H) {
  RouterTcPlan p;
  p.N_pad = (N + 15) / 16 * 16;
  p.H_pad = (H + RT_BK - 1) / RT_BK * RT_BK;
  p.stacked = 3 * p.N_pad <= 256 ? 1 : 0;
  const int mma_n = p.stacked ? 3 * p.N_pad : p.N_pad;
  p.pp = p.stacked ? 1 : (p.N_pad <= 128 ? 3 : 1);
  // stacked planes: one accumulator; planes along K: two, alternating per
  // k-step (the epilogue reads all of them in one TMEM round trip)
  p.nacc = p.stacked ? 1 : 2;
  int cols = 32;
  while (cols < p.nacc * mma_n) cols <<= 1;
  p.tmem_cols = cols;
  p.stage_bytes = RT_A_BYTES + p.pp * mma_n * RT_BK * 2;
  int st = (200 * 1024) / p.stage_bytes;
  p.stages = st > RT_MAX_STAGES ? RT_MAX_STAGES : (st < 2 ? 2 : st);
  p.m_tiles = (T + RT_BM - 1) / RT_BM;
  // split K over a cluster while the token tiles alone leave SMs idle:
  // S in {1, 2, 4, 8}, at least two x tiles per split
  const int KB = p.H_pad / RT_BK;
  int S = 1;
  while (S < 8 && p.m_tiles > 0 && p.m_tiles * S * 2 <= 148 && KB / (S * 2) >= 2) S *= 2;
  p.kb_per_split = (KB + S - 1) / S;
  p.splits = S;
  // shared memory: the ring, later reused for the [128][N_pad + 4] logits tile
  const int ring = p.stages * p.stage_bytes;
  const int tile = RT_BM * (p.N_pad + 4) * 4;
  p.work_bytes = ((ring > tile ? ring : tile) + 1023) / 1024 * 1024;
  p.smem = 1024 + p.work_bytes + (3 * RT_MAX_STAGES + 2) * 8 + 16 + 4 * p.N_pad * 4 + 16 +
           p.N_pad * 16;
  return p;
}

int router_tc_num_ctas(int T, int N, int H) {
  const RouterTcPlan p = router_tc_plan(T, N, H);
  return p.m_tiles * p.splits;
}

// The epilogue warps split W_g for each ring slot with a dependent L2 round
// trip per slot; that pays off against a separate split launch only while a
// CTA streams few x tiles.
constexpr int kOwnSplitMaxTiles = 16;

bool router_own_split(int T, int N, int H) {
  const RouterTcPlan p = router_tc_plan(T, N, H);
  return p.stacked && p.kb_per_split <= kOwnSplitMaxTiles;
}

int router_fused_chunks(int T, int N, int H) { return router_tc_num_ctas(T, N, H); }

int router_fused_chunk_tokens(int T, int N, int H) {
  return RT_BM / router_tc_plan(T, N, H).splits;
}

cudaError_t launch_router_tc(const RouterLaunch& a, __nv_bfloat16* W3, int* ticket, int* status,
                             int* clear, int clear_n, const RouterFused* fused, cudaStream_t st,
                             LaunchTrace* tr) {
  const RouterTcPlan P = router_tc_plan(a.T, a.N, a.H);
  if (a.T == 0) {
    trace_mark(tr, st);
    return launch_router_stats_zero(a.p_mean, a.z_loss, a.N, st);  // p_mean = 0, z_loss = 0
  }
  // stacked planes over few x tiles per CTA: the router's epilogue warps
  // split W_g per ring slot and (fused only, where it uses no ticket) its
  // CTA 0 clears the header; otherwise a split kernel writes W3 first
  const bool own = router_own_split(a.T, a.N, a.H);
  if (!own) {
    const int64_t total = (int64_t)P.N_pad * P.H_pad;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 148 * 8) blocks = 148 * 8;
    trace_mark(tr, st);
    cudaError_t e = launch_pdl(router_split_kernel, dim3((unsigned)blocks), dim3(256), 0, st, 1,
                               a.Wg, W3, a.N, a.H, P.N_pad, P.H_pad, P.stacked, clear, clear_n);
    if (e != cudaSuccess) return e;
  }
  CUtensorMap tmX, tmW;
  if (!encode_tensor_map_bf16(&tmX, a.x, a.T, a.H, RT_BK, RT_BM)) return cudaErrorInvalidValue;
  if (own) {
    tmW = tmX;   // not read: the planes are written in shared memory
  } else if (P.stacked) {
    if (!encode_tensor_map_bf16(&tmW, W3, 3 * P.N_pad, P.H_pad, RT_BK, 3 * P.N_pad))
      return cudaErrorInvalidValue;
  } else {
    if (!encode_tensor_map_bf16(&tmW, W3, P.N_pad, 3 * P.H_pad, RT_BK, P.N_pad))
      return cudaErrorInvalidValue;
  }
  RouterTcArgs args;
  args.bg = a.bg;
  args.sel_bias = a.sel_bias;
  args.topk_idx = a.topk_idx;
  args.topk_w = a.topk_w;
  args.probs = a.probs;
  args.logits_out = a.logits_out;
  args.z_loss = a.z_loss;
  args.p_part = a.p_part;
  args.p_mean = a.p_mean;
  args.ticket = ticket;
  args.status = status;
  args.T = a.T;
  args.N = a.N;
  args.N_pad = P.N_pad;
  args.H_pad = P.H_pad;
  args.k = a.k;
  args.tmem_cols = P.tmem_cols;
  args.stacked = P.stacked;
  args.nacc = P.nacc;
  args.planes_per_stage = P.pp;
  args.stages = P.stages;
  args.kb_per_split = P.kb_per_split;
  args.splits = P.splits;
  args.work_bytes = P.work_bytes;
  args.Wg = own ? a.Wg : nullptr;
  args.H = a.H;
  args.local_rank = fused ? fused->local_rank : nullptr;
  args.blk_hist = fused ? fused->blk_hist : nullptr;
  args.clear = (own && fused) ? clear : nullptr;
  args.clear_n = clear_n;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(P.m_tiles * P.splits);
  cfg.blockDim = dim3(RT_THREADS);
  cfg.dynamicSmemBytes = P.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = P.splits;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see pdl_wait()
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  trace_mark(tr, st);
  // the largest ring needs ~203 KB; the attribute is set once per kernel
#define MOE_RTC(KM)                                                                            \
  do {                                                                                         \
    static bool attr_set = false;                                                              \
    if (!attr_set) {                                                                           \
      cudaError_t e = cudaFuncSetAttribute(router_tc_kernel<KM>,                               \
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,        \
                                           kRouterTcSmemMax);                                  \
      if (e != cudaSuccess) return e;                                                          \
      attr_set = true;                                                                         \
    }                                                                                          \
    cudaError_t le = cudaLaunchKernelEx(&cfg, router_tc_kernel<KM>, tmX, tmW, args);           \
    if (le != cudaSuccess) return le;                                                          \
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
