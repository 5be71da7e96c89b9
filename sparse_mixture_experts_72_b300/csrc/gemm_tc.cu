// Grouped bf16 GEMM on the 5th-generation tensor cores (tcgen05 + TMEM),
// fed by TMA, with the expert FFN epilogues fused:
//
//   EPI_GELU :  out[r, n] = bf16( GELU_erf(acc[r, n] + bias_g[n]) )        (Linear -> GELU)
//   EPI_SCALE:  out[r, n] = bf16( w_r * (acc[r, n] + bias_g[n]) )          (Linear, gate weight)
//
// acc[r, :] = A[r, :] . B_g[:, :]^T over the K dimension, where group g (an
// expert) owns the A rows [offsets[g], offsets[g+1]) and the B rows
// [g * n_out, (g+1) * n_out).  The experts are "AI-Research-SKILLs MoE 训练实战"
// §3.1's Linear(H, 4H) -> GELU -> Linear(4H, H); the weighting by the
// renormalised gate score is its output[mask] += score * expert_output.
//
// Structure (one persistent CTA per SM, 320 threads):
//   warp 0      TMA producer: A tile 128 x 64 and B tile 256 x 64 per stage,
//               4-stage ring of full/empty mbarriers
//   warp 1      TMEM allocator and single-thread MMA issuer:
//               tcgen05.mma kind::f16, M=128 N=256 K=16, fp32 accumulators in
//               TMEM, double-buffered (2 x 256 columns)
//   warps 2..9  epilogue: tcgen05.ld -> bias -> GELU or scale -> bf16 stores;
//               warp w reads TMEM lanes 32*(w%4).. and column half (w-2)/4
// Tiles are ordered expert-major, then output block, then row block, so the
// CTAs working at one time share the same weight slab through L2.
// Every wait is bounded: on expiry the CTA records MOE_ERR_TIMEOUT, drains
// its in-flight copies and MMAs, frees TMEM and exits.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int EPI_WARPS = 8;
constexpr int GEMM_THREADS = 64 + EPI_WARPS * 32;
constexpr int TMEM_COLS = 2 * BN;
constexpr int MAX_GROUPS = MOE_MAX_EXPERTS;
constexpr int NUM_BARS = 2 * STAGES + 5;
constexpr int SMEM_TILES = STAGES * STAGE_BYTES;
constexpr int SMEM_BYTES =
    1024 + SMEM_TILES + NUM_BARS * 8 + 16 + 2 * (MAX_GROUPS + 1) * 4;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
constexpr long long kDrainLimitCycles = 200000000LL;  // ~0.1 s

// Wait used only while draining after an abort: ignores the abort flag.
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kDrainLimitCycles) return false;
  }
  return true;
}

struct TileCursor {
  int g = 0;
  __device__ __forceinline__ void locate(int tile, const int32_t* tile_start, const int32_t* seg,
                                         int n_out, int& a_row, int& rows_left, int& m, int& n) {
    while (tile >= tile_start[g + 1]) ++g;
    const int local = tile - tile_start[g];
    const int rows = seg[g + 1] - seg[g];
    const int mt = (rows + BM - 1) / BM;
    n = local / mt;
    m = local - n * mt;
    a_row = seg[g] + m * BM;
    rows_left = rows - m * BM;
    (void)n_out;
  }
};

__global__ void __launch_bounds__(GEMM_THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB, const GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sA = smem_u32(smem);
  const uint32_t sB = sA + STAGES * A_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SMEM_TILES);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int32_t* seg = reinterpret_cast<int32_t*>(tmem_holder + 4);   // [G+1] row offsets
  int32_t* tile_start = seg + (MAX_GROUPS + 1);                 // [G+1] tile prefix

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int G = args.num_groups;
  const int n_out = args.n_out;
  const int n_tiles = (n_out + BN - 1) / BN;
  const int nkb = (args.K + BK - 1) / BK;
  int* status = args.status;

  // ---- set-up: group table, barriers, TMEM
  for (int i = threadIdx.x; i <= G; i += GEMM_THREADS)
    seg[i] = args.offsets ? args.offsets[i] : (i == 0 ? 0 : args.rows_single);
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), EPI_WARPS);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), TMEM_COLS);
    tmem_relinquish();
  }
  __syncthreads();  // seg[] visible
  if (warp == 2) {
    // tile_start = exclusive prefix over groups of (row blocks * n_tiles)
    const int per = (G + 31) / 32;
    const int g0 = lane * per;
    int local = 0;
    for (int g = g0; g < g0 + per && g < G; ++g)
      local += ((seg[g + 1] - seg[g] + BM - 1) / BM) * n_tiles;
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - local;
    for (int g = g0; g < g0 + per && g < G; ++g) {
      tile_start[g] = run;
      run += ((seg[g + 1] - seg[g] + BM - 1) / BM) * n_tiles;
    }
    if (lane == 31) tile_start[G] = incl;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int total = tile_start[G];
  long long tma_issued = 0;  // producer thread only

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      long long issued = 0;
      bool ok = true;
      TileCursor cur;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        int a_row, rows_left, m, n;
        cur.locate(tile, tile_start, seg, n_out, a_row, rows_left, m, n);
        const int b_row = cur.g * n_out + n * BN;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full_bar(stage), STAGE_BYTES);
          tma_load_2d(sA + stage * A_BYTES, &tmA, full_bar(stage), kb * BK, a_row);
          tma_load_2d(sB + stage * B_BYTES, &tmB, full_bar(stage), kb * BK, b_row);
          ++issued;
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      tma_issued = issued;
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        if (!mbar_wait_bounded(tempty_bar(acc), acc_phase ^ 1u, abort_flag, status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait_bounded(full_bar(stage), phase, abort_flag, status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = sdesc_kmajor_sw128(sA + stage * A_BYTES);
          const uint64_t bdesc = sdesc_kmajor_sw128(sB + stage * B_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            // +32 bytes along K per step of 16 bf16 inside the 128-byte swizzle atom
            umma_bf16(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          umma_commit(empty_bar(stage));
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        umma_commit(tfull_bar(acc));
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;            // TMEM lane quarter this warp may access
    const int h = (warp - 2) >> 2;     // column half of the 256-wide tile
    const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
    uint32_t acc = 0, acc_phase = 0;
    TileCursor cur;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      int a_row, rows_left, m, n;
      cur.locate(tile, tile_start, seg, n_out, a_row, rows_left, m, n);
      int ok = 1;
      if (lane == 0) ok = mbar_wait_bounded(tfull_bar(acc), acc_phase, abort_flag, status) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const int r_in = q * 32 + lane;
      const bool row_ok = r_in < rows_left;
      const int64_t out_row = (int64_t)a_row + r_in;
      float wscale = 1.0f;
      if (args.mode == EPI_SCALE && args.topk_w != nullptr && row_ok)
        wscale = args.topk_w[args.perm[out_row]];
      const __nv_bfloat16* bias = args.bias ? args.bias + (size_t)cur.g * n_out : nullptr;
      __nv_bfloat16* orow = args.out + out_row * args.ld_out;
#pragma unroll 1
      for (int c = 0; c < (BN / 2) / 32; ++c) {
        const int tcol = h * (BN / 2) + c * 32;  // column inside the tile
        const int col = n * BN + tcol;           // column inside the group's n_out
        if (col >= n_out) break;                 // warp-uniform
        uint32_t r[32];
        tmem_ld_32x32b_x32(tmem_base + lane_addr + acc * BN + tcol, r);
        tmem_ld_wait();
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
        if (bias) {
#pragma unroll
          for (int j8 = 0; j8 < 4; ++j8) {
            if (col + 8 * j8 < n_out) {
              const uint4 u = __ldg(reinterpret_cast<const uint4*>(bias + col + 8 * j8));
              v[8 * j8 + 0] += bf16lo(u.x); v[8 * j8 + 1] += bf16hi(u.x);
              v[8 * j8 + 2] += bf16lo(u.y); v[8 * j8 + 3] += bf16hi(u.y);
              v[8 * j8 + 4] += bf16lo(u.z); v[8 * j8 + 5] += bf16hi(u.z);
              v[8 * j8 + 6] += bf16lo(u.w); v[8 * j8 + 7] += bf16hi(u.w);
            }
          }
        }
        if (args.mode == EPI_GELU) {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = gelu_erf(v[i]);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= wscale;
        }
        if (row_ok) {
#pragma unroll
          for (int j8 = 0; j8 < 4; ++j8) {
            if (col + 8 * j8 < n_out) {
              uint4 o;
              o.x = pack_bf16x2(v[8 * j8 + 0], v[8 * j8 + 1]);
              o.y = pack_bf16x2(v[8 * j8 + 2], v[8 * j8 + 3]);
              o.z = pack_bf16x2(v[8 * j8 + 4], v[8 * j8 + 5]);
              o.w = pack_bf16x2(v[8 * j8 + 6], v[8 * j8 + 7]);
              *reinterpret_cast<uint4*>(orow + col + 8 * j8) = o;
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(acc));
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  // ---- teardown: every MMA has completed (observed through tmem_full or
  // the drain barrier) and every TMEM load has been waited for.
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // Some role gave up, so copies or MMAs may still be in flight.  Let the
    // copies (at most the last STAGES issued) land and the MMAs finish
    // before the shared memory and TMEM go away.
    if (warp == 0 && lane == 0) {
      const long long first = tma_issued > STAGES ? tma_issued - STAGES : 0;
      for (long long j = first; j < tma_issued; ++j)
        mbar_wait_drain(full_bar((int)(j % STAGES)), (uint32_t)((j / STAGES) & 1));
    }
    if (warp == 1 && lane == 0) {
      umma_commit(drain_bar);
      mbar_wait_drain(drain_bar, 0);
    }
    __syncwarp();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encoder() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

bool tensor_map_encoder_available() { return get_encoder() != nullptr; }

bool encode_tensor_map_bf16(CUtensorMap* map, const void* base, int64_t rows, int64_t K,
                            int box_cols, int box_rows) {
  EncodeTiledFn enc = get_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

cudaError_t make_gemm_plan(GemmPlan* plan, const __nv_bfloat16* A, int64_t a_rows,
                           const __nv_bfloat16* B, int64_t b_rows, const GemmArgs& args,
                           int num_sms) {
  if (a_rows <= 0 || b_rows <= 0 || args.K <= 0 || args.n_out <= 0) return cudaErrorInvalidValue;
  if (!encode_tensor_map_bf16(&plan->tmA, A, a_rows, args.K, BK, BM)) return cudaErrorInvalidValue;
  if (!encode_tensor_map_bf16(&plan->tmB, B, b_rows, args.K, BK, BN)) return cudaErrorInvalidValue;
  plan->args = args;
  const int64_t n_tiles = (args.n_out + BN - 1) / BN;
  const int64_t max_tiles = ((a_rows + BM - 1) / BM + args.num_groups) * n_tiles;
  plan->grid = (int)(max_tiles < num_sms ? max_tiles : num_sms);
  return cudaSuccess;
}

cudaError_t launch_gemm(const GemmPlan& plan, cudaStream_t st, LaunchTrace* tr) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  trace_mark(tr, st);
  grouped_gemm_kernel<<<plan.grid, GEMM_THREADS, SMEM_BYTES, st>>>(plan.tmA, plan.tmB, plan.args);
  return cudaGetLastError();
}

}  // namespace moe
