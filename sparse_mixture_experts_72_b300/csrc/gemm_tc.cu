// Grouped bf16 GEMM on the 5th-generation tensor cores (tcgen05 + TMEM),
// fed by TMA, with the expert FFN epilogues fused:
//
//   EPI_GELU  : out[r, n] = bf16( GELU_erf(acc[r, n] + bias_g[n]) )        (Linear -> GELU)
//   EPI_SILU  : out[r, n] = bf16( SiLU(acc[r, n] + bias_g[n]) )            (Linear -> SiLU)
//   EPI_SWIGLU: out[r, n] = bf16( SiLU(gate[r, n]) * up[r, n] )            (gated Linear)
//               gate / up = acc against B rows n and n_out + n (+ bias)
//   EPI_SCALE : out[r, n] = bf16( w_r * (acc[r, n] + bias_g[n]) )          (Linear, gate weight)
//
// acc[r, :] = A[r, :] . B_g[:, :]^T over the K dimension, where group g (an
// expert) owns the A rows [offsets[g], offsets[g+1]) and the B rows
// [g * n_out, (g+1) * n_out).  The experts are "AI-Research-SKILLs MoE 训练实战"
// §3.1's Linear(H, 4H) -> GELU -> Linear(4H, H); the weighting by the
// renormalised gate score is its output[mask] += score * expert_output.
//
// One launch runs the whole expert FFN as two phases over one persistent
// grid: phase 0 (Hid = GELU(X W1^T + b1)) and phase 1 (y = w (Hid W2^T +
// b2)), for the routed experts and, as group G with its own tensors and
// weight 1, the always-on shared expert ("混合专家模型 MoE 架构深度解析" §3).
// The tile list is phase 0's tiles followed by phase 1's; CTAs (pairs) take
// them round-robin or, in long bf16 launches, from a launch-wide counter
// (dynamic order).  When the last of a CTA's epilogue warps has stored a
// phase-0 tile (a CTA-scope acquire-release count in shared memory), it
// releases a per-row-block counter in global memory (red.release.gpu), and
// the TMA producer acquires the counter of a phase-1 tile's row block
// (ld.acquire.gpu, then fence.proxy.async) before loading its Hid rows.  The second Linear of an expert therefore
// starts as soon as its rows are ready, with no kernel boundary, and the
// second Linear's few large tiles fill the gaps of the first's tail instead
// of forming a partial last wave.
//
// Two shapes of the same persistent, warp-specialised kernel, each for bf16
// or FP8 (E4M3) weights:
//
//   PAIR = 1  one CTA per tile of 128 rows x 256 columns: A tile 128 x 64 and
//             B tile 256 x 64 per stage, 4 stages; tcgen05.mma.cta_group::1,
//             M = 128.  Used when experts hold few rows (decode batches).
//   PAIR = 2  a cluster of two CTAs per tile of 256 rows x 256 columns:
//             each CTA loads its own 128 rows of A and 128 rows of B per
//             stage (32 KB, 6 stages), the even CTA issues
//             tcgen05.mma.cta_group::2 with M = 256 over both CTAs' shared
//             memory, and each CTA's TMEM receives its 128 rows.  Two thirds
//             of the shared-memory bytes per FLOP of PAIR = 1, so the same
//             ring hides 1.5x more load latency.
//
// Roles: warp 0 TMA producer; warp 1 TMEM allocator and single-thread MMA
// issuer (even CTA only for PAIR = 2) into one of two 256-column fp32
// accumulators; then EPI_WARPS epilogue warps (tcgen05.ld -> scale -> bias ->
// activation or gate weight -> bf16 stores; warp w reads TMEM lanes
// 32*(w%4).. and the EPI_COLS-wide column slice (w-2)/4 of the tile); with
// FP8 weights, then CONV_WARPS converter warps that fetch the E4M3 weight
// rows and widen them to the bf16 B tiles (8 epilogue + 8 converter warps;
// 576 threads in every shape).
// The grid never exceeds the CTAs (pairs) that can be resident at once, so a
// phase-1 tile only ever waits for tiles that running CTAs will finish.
// Every wait is bounded: on expiry the CTA records MOE_ERR_TIMEOUT, lets its
// in-flight copies land, drains its MMAs, frees TMEM and exits.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {

constexpr int BK = 64, BN = 256;
constexpr int TMEM_COLS = 2 * BN;
constexpr int MAX_GROUPS = MOE_MAX_EXPERTS;
constexpr int A_BYTES = 128 * BK * 2;  // 128 rows of A per CTA and stage
constexpr long long kDrainLimitCycles = 200000000LL;  // ~0.1 s

// Shared-memory rings of one CTA.  bf16 weights: one ring of STAGES k-blocks
// holding A and B, filled by the TMA producer and freed by the MMA.  FP8
// weights: three rings, so that the weight bytes in flight do not wait for
// the MMA:
//   A ring   STAGES   x A tile                producer TMA -> MMA
//   Q ring   Q_STAGES x E4M3 B tile, 2 k-blocks  the converter warps' own TMA -> converters
//   B ring   B_STAGES x bf16 B tile           converters -> MMA
// A Q slot holds 128 bytes of each weight row (two k-blocks): the copies
// read whole 128-byte row segments, as the bf16 tiles do.  The Q ring runs
// up to 2 * Q_STAGES + B_STAGES k-blocks ahead of the MMA, and phase-1
// weights stream in while the producer still waits for phase-0 rows.
template <int PAIR, bool FP8>
struct GemmShape {
  static constexpr int TILE_M = 128 * PAIR;              // rows per tile (whole pair)
  static constexpr int B_ROWS = BN / PAIR;               // B rows each CTA loads
  static constexpr int B_BYTES = B_ROWS * BK * 2;        // bf16 B tile the MMA reads
  static constexpr int BKQ = 2 * BK;                     // K columns (bytes) of a Q slot
  static constexpr int BQ_BYTES = FP8 ? B_ROWS * BKQ : 0; // E4M3 B rows as loaded (row-major)
  // bytes the full barrier of an A-ring slot counts per CTA
  static constexpr int TX_BYTES = FP8 ? A_BYTES : A_BYTES + B_BYTES;
  static constexpr int STAGES = FP8 ? (PAIR == 2 ? 6 : 3) : (PAIR == 2 ? 6 : 4);
  // FP8, single CTA: the A ring's bytes are cut into slots of the launch's A
  // copy height (GemmArgs::a_box rows), up to A_SLOTS_MAX of them; elsewhere
  // STAGES slots of 128 rows
  static constexpr int A_SLOTS_MAX = FP8 && PAIR == 1 ? 12 : STAGES;
  static constexpr int B_STAGES = FP8 ? (PAIR == 2 ? 4 : 2) : STAGES;
  static constexpr int Q_STAGES = FP8 ? 3 : 0;
  // Epilogue warps: 4 per TMEM lane quarter, EPI_COLS columns each.  FP8:
  // warps widening E4M3 to bf16 in shared memory.  Widening a k-block takes
  // a warp longer than the MMA step it feeds unless many warps share it, so
  // FP8 kernels give half of the epilogue warps to the conversion (8 + 8;
  // with 2 converter warps a pair's CTA ran 3.5x slower than bf16 weights).
  static constexpr int EPI_WARPS = FP8 ? 8 : 16;
  static constexpr int EPI_COLS = BN / (EPI_WARPS / 4);
  static constexpr int CONV_WARPS = FP8 ? 8 : 0;
  static constexpr int THREADS = 64 + EPI_WARPS * 32 + CONV_WARPS * 32;
  // bf16 weights: slots of each tile-index queue (dynamic tile order)
  static constexpr int QD = FP8 ? 0 : 4;
  // full, empty, tmem full / empty, drain (+ FP8: Q full / empty, B full /
  // empty; bf16: pair and local tile queues, full / empty)
  static constexpr int NUM_BARS =
      2 * A_SLOTS_MAX + 5 + (FP8 ? 2 * Q_STAGES + 2 * B_STAGES : 0) + 4 * QD;
  static constexpr int SMEM_TILES = STAGES * A_BYTES + B_STAGES * B_BYTES + Q_STAGES * BQ_BYTES;
  // tiles (1024-aligned), barriers, TMEM address / flags, bias staging, then
  // the two group tables of G + 1 ints: sized per launch, the unused
  // shared memory is left to L1 (measured 2-3 % faster than a fixed size)
  // CTA pairs: a transpose buffer per epilogue warp for swapped tail tiles
  // (8 token rows x 32 output columns of bf16)
  static constexpr int TRANS_BYTES = PAIR == 2 ? EPI_WARPS * 8 * 32 * 2 : 0;
  static constexpr int SMEM_FIXED = SMEM_TILES + NUM_BARS * 8 + 16 + 2 * QD * 4 + 16 +
                                    EPI_WARPS * EPI_COLS * 2 +              // bias staging
                                    (FP8 ? EPI_WARPS * EPI_COLS * 4 : 0) +  // scale staging
                                    TRANS_BYTES;
  static constexpr int smem_bytes(int G) { return SMEM_FIXED + 2 * (G + 1) * 4; }
  static_assert(SMEM_FIXED + 2 * (MAX_GROUPS + 1) * 4 <= 232448, "shared memory budget");
};

// Wait used only while draining after an abort: ignores the abort flag.
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kDrainLimitCycles) return false;
  }
  return true;
}

// Walks the tiles of a launch in increasing order: phase 0's tiles, then
// phase 1's; inside a phase expert-major, then column block, then row block
// (row block fastest, so the CTAs working at one time share a weight slab),
// and after the routed experts the shared expert (group G: rows_s rows in
// mt_s row blocks of its own tensors).
template <int TILE_M>
struct TileCursor {
  int phase = 0, g = 0;
  __device__ __forceinline__ void locate(int tile, int tiles0, int nt0, int nt1,
                                         const int32_t* mt_pre, const int32_t* seg, int G,
                                         int mt_s, int rows_s, int& a_row, int& rows_left,
                                         int& n, int& rb) {
    int local = tile;
    if (tile >= tiles0) {
      if (phase == 0) { phase = 1; g = 0; }
      local = tile - tiles0;
    }
    const int ntp = phase ? nt1 : nt0;
    const int routed = mt_pre[G] * ntp;
    if (local >= routed) {
      g = G;
      const int ls = local - routed;
      n = ls / mt_s;
      const int m = ls - n * mt_s;
      rb = m;   // index into the shared expert's own counters
      a_row = m * TILE_M;
      rows_left = rows_s - m * TILE_M;
      return;
    }
    while (local >= mt_pre[g + 1] * ntp) ++g;   // groups without rows own no tiles
    const int mt = mt_pre[g + 1] - mt_pre[g];
    const int lg = local - mt_pre[g] * ntp;
    n = lg / mt;
    const int m = lg - n * mt;
    rb = mt_pre[g] + m;
    a_row = seg[g] + m * TILE_M;
    rows_left = seg[g + 1] - seg[g] - m * TILE_M;
  }
};

// Per-tile view of a phase's parameters, read field by field from the
// kernel parameters (no dynamic indexing into parameter space).
struct PhaseView {
  int n_out, K, mode, ld_out;
  const __nv_bfloat16* bias;
  const float* topk_w;
  const int32_t* perm;
  __nv_bfloat16* out;
  const float* b_scale;
  __device__ __forceinline__ PhaseView(const GemmArgs& a, int p, bool sh) {
    if (sh) {   // the shared expert: its own tensors, weight 1
      n_out = p ? a.shp[1].n_out : a.shp[0].n_out;
      K = p ? a.shp[1].K : a.shp[0].K;
      mode = p ? a.shp[1].mode : a.shp[0].mode;
      ld_out = p ? a.shp[1].ld_out : a.shp[0].ld_out;
      bias = p ? a.shp[1].bias : a.shp[0].bias;
      topk_w = nullptr;
      perm = nullptr;
      out = p ? a.shp[1].out : a.shp[0].out;
      b_scale = p ? a.shp[1].b_scale : a.shp[0].b_scale;
      return;
    }
    n_out = p ? a.ph[1].n_out : a.ph[0].n_out;
    K = p ? a.ph[1].K : a.ph[0].K;
    mode = p ? a.ph[1].mode : a.ph[0].mode;
    ld_out = p ? a.ph[1].ld_out : a.ph[0].ld_out;
    bias = p ? a.ph[1].bias : a.ph[0].bias;
    topk_w = p ? a.ph[1].topk_w : a.ph[0].topk_w;
    perm = p ? a.ph[1].perm : a.ph[0].perm;
    out = p ? a.ph[1].out : a.ph[0].out;
    b_scale = p ? a.ph[1].b_scale : a.ph[0].b_scale;
  }
};

template <int PAIR, bool FP8>
__global__ void __launch_bounds__(GemmShape<PAIR, FP8>::THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA0,
                        const __grid_constant__ CUtensorMap tmB0,
                        const __grid_constant__ CUtensorMap tmA1,
                        const __grid_constant__ CUtensorMap tmB1,
                        const __grid_constant__ CUtensorMap tmSA0,
                        const __grid_constant__ CUtensorMap tmSB0,
                        const __grid_constant__ CUtensorMap tmSA1,
                        const __grid_constant__ CUtensorMap tmSB1, const GemmArgs args) {
  using S = GemmShape<PAIR, FP8>;
  constexpr int STAGES = S::STAGES;
  constexpr int GEMM_THREADS = S::THREADS;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {
    // the 128-byte swizzled tiles need a 1024-byte aligned base; never seen,
    // but refuse rather than compute garbage
    if (threadIdx.x == 0) atomicExch(args.status, (int)MOE_ERR_UNSUPPORTED);
    return;
  }
  uint8_t* smem = smem_raw;
  const uint32_t sA = smem_u32(smem);
  const uint32_t sB = sA + STAGES * A_BYTES;               // B ring (bf16)
  const uint32_t sBq = sB + S::B_STAGES * S::B_BYTES;      // Q ring (FP8 only)
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::SMEM_TILES);
  const uint32_t bar0 = smem_u32(bars);
  constexpr int AS = S::A_SLOTS_MAX;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (AS + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * AS + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * AS + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * AS + 4);
  // FP8: E4M3 tile landed / read by every converter warp; bf16 tile written
  // by every converter warp of the pair / read by the MMA
  constexpr int QB = 2 * AS + 5, CB = QB + 2 * S::Q_STAGES;
  auto qfull_bar = [&](int s) { return bar0 + 8u * (QB + s); };
  auto qempty_bar = [&](int s) { return bar0 + 8u * (QB + S::Q_STAGES + s); };
  auto cfull_bar = [&](int s) { return bar0 + 8u * (CB + s); };
  auto cempty_bar = [&](int s) { return bar0 + 8u * (CB + S::B_STAGES + s); };
  // bf16 tile queues: the pair queue (the leader's producer to the peer's,
  // barriers used in the receiving CTA: full in the peer, empty in the
  // leader) and the local queue (this CTA's producer to its MMA issuer and
  // epilogue warps)
  constexpr int QD = S::QD, TB = CB + (FP8 ? 2 * S::B_STAGES : 0);
  auto pqfull_bar = [&](int s) { return bar0 + 8u * (TB + s); };
  auto pqempty_bar = [&](int s) { return bar0 + 8u * (TB + QD + s); };
  auto lqfull_bar = [&](int s) { return bar0 + 8u * (TB + 2 * QD + s); };
  auto lqempty_bar = [&](int s) { return bar0 + 8u * (TB + 3 * QD + s); };
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + S::NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  uint32_t* stored_cnt = tmem_holder + 2;  // [2]: epilogue warps done with the tile in acc
  volatile int* pq = reinterpret_cast<volatile int*>(tmem_holder + 4);   // [QD] pair queue
  volatile int* lq = pq + QD;                                             // [QD] local queue
  constexpr int EPI_WARPS = S::EPI_WARPS, EPI_COLS = S::EPI_COLS;
  uint16_t* bias_stage = reinterpret_cast<uint16_t*>(  // [EPI_WARPS][EPI_COLS], 16-B aligned
      (reinterpret_cast<uintptr_t>(tmem_holder + 4 + 2 * QD) + 15) & ~static_cast<uintptr_t>(15));
  float* scale_stage = reinterpret_cast<float*>(bias_stage + EPI_WARPS * EPI_COLS);  // FP8 only
  uint16_t* trans_stage = reinterpret_cast<uint16_t*>(   // [EPI_WARPS][8][32] (CTA pairs)
      reinterpret_cast<uint8_t*>(scale_stage) + (FP8 ? EPI_WARPS * EPI_COLS * 4 : 0));
  int32_t* seg = reinterpret_cast<int32_t*>(
      reinterpret_cast<uint8_t*>(trans_stage) + S::TRANS_BYTES);  // [G+1]
  int32_t* mt_pre = seg + (args.num_groups + 1);                          // [G+1]

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const uint32_t rank = PAIR == 2 ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  const int unit = PAIR == 2 ? (int)cluster_id_x() : (int)blockIdx.x;   // pair (or CTA) index
  const int units = PAIR == 2 ? (int)num_clusters_x() : (int)gridDim.x;
  const int G = args.num_groups;
  const bool two = args.num_phases == 2;
  // output columns per tile: 256, or 128 for SwiGLU (gate + up fill the 256
  // accumulator columns)
  const int bno0 = args.ph[0].mode == EPI_SWIGLU ? BN / 2 : BN;
  const int bno1 = two && args.ph[1].mode == EPI_SWIGLU ? BN / 2 : BN;
  const int nt0 = (args.ph[0].n_out + bno0 - 1) / bno0;
  const int nt1 = two ? (args.ph[1].n_out + bno1 - 1) / bno1 : 0;
  const int nkb0 = (args.ph[0].K + BK - 1) / BK;
  const int nkb1 = two ? (args.ph[1].K + BK - 1) / BK : 0;
  // the shared expert (group G): row blocks, and its phase-1 reduction length
  const int rows_s = args.shared_rows;
  const int mt_s = rows_s > 0 ? (rows_s + S::TILE_M - 1) / S::TILE_M : 0;
  const int nt0s = mt_s > 0 ? (args.shp[0].n_out + bno0 - 1) / bno0 : 0;
  const int nt1s = mt_s > 0 && two ? nt1 : 0;
  const int nkb1s = mt_s > 0 && two ? (args.shp[1].K + BK - 1) / BK : 0;
  // releases that complete one row block: one per CTA of the tile for every
  // column block
  const int rows_done_target = nt0 * PAIR, rows_done_target_s = nt0s * PAIR;
  // per-tile choices between a routed expert and the shared one
  auto map_a = [&](int ph, bool sh) { return sh ? (ph ? &tmSA1 : &tmSA0) : (ph ? &tmA1 : &tmA0); };
  auto map_b = [&](int ph, bool sh) { return sh ? (ph ? &tmSB1 : &tmSB0) : (ph ? &tmB1 : &tmB0); };
  auto nkb_of = [&](int ph, bool sh) { return ph ? (sh ? nkb1s : nkb1) : nkb0; };
  auto n_out_of = [&](int ph, bool sh) {
    return sh ? (ph ? args.shp[1].n_out : args.shp[0].n_out) : (ph ? args.ph[1].n_out : args.ph[0].n_out);
  };
  // A copies: a_box rows each (the 128-row MMA also reads the rows after
  // them, which belong to no row of the tile and are never stored)
  constexpr bool SMALL_A = FP8 && PAIR == 1;
  const int a_box = SMALL_A ? args.a_box : 128;
  const uint32_t a_slot = (uint32_t)a_box * BK * 2;
  const int a_slots = SMALL_A ? min(AS, (int)(STAGES * A_BYTES / a_slot)) : STAGES;
  int* status = args.status;
  // Tail tiles of CTA pairs: the last row block of a group with fewer than
  // 256 rows runs with the operands swapped - the 256 weight rows of the tile
  // (the B rows, split 128 per CTA as usual) are the MMA's M operand and the
  // group's remaining token rows, rounded up to 16 and split in halves
  // across the pair, its N operand - so the tensor cores skip the padding
  // rows.  The accumulator then holds output columns in TMEM lanes and tokens
  // in columns.  Not for SwiGLU first Linears (gate and up rows would land in
  // different CTAs).
  auto swapped_tail = [&](int ph, int rows_left) {
    return PAIR == 2 && rows_left <= args.swap_tail && rows_left < S::TILE_M &&
           (ph ? args.ph[1].mode : args.ph[0].mode) != EPI_SWIGLU;
  };

  // ---- set-up: barriers, TMEM (CTA-local, may overlap the previous kernel),
  // then the group table
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < AS; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), EPI_WARPS * PAIR);
    }
    mbar_init(drain_bar, 1);
    if constexpr (FP8) {
      for (int s2 = 0; s2 < S::Q_STAGES; ++s2) {
        mbar_init(qfull_bar(s2), 1);
        mbar_init(qempty_bar(s2), S::CONV_WARPS);
      }
      for (int s2 = 0; s2 < S::B_STAGES; ++s2) {
        mbar_init(cfull_bar(s2), S::CONV_WARPS * PAIR);  // every converter warp of the pair
        mbar_init(cempty_bar(s2), 1);
      }
    }
    for (int s2 = 0; s2 < QD; ++s2) {
      mbar_init(pqfull_bar(s2), 1);
      mbar_init(pqempty_bar(s2), 1);
      mbar_init(lqfull_bar(s2), 1);
      // read by the epilogue warps and, in the leader, the MMA issuer
      mbar_init(lqempty_bar(s2), EPI_WARPS + (leader ? 1 : 0));
    }
    *abort_flag = 0;
    stored_cnt[0] = stored_cnt[1] = 0u;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA0);
    tma_prefetch_desc(&tmB0);
    if (two) {
      tma_prefetch_desc(&tmA1);
      tma_prefetch_desc(&tmB1);
    }
    if (args.shared_rows > 0) {
      tma_prefetch_desc(&tmSA0);
      tma_prefetch_desc(&tmSB0);
      if (two) {
        tma_prefetch_desc(&tmSA1);
        tma_prefetch_desc(&tmSB1);
      }
    }

  }
  if (warp == 1) {
    if constexpr (PAIR == 2) {
      tmem_alloc_pair(smem_u32(tmem_holder), TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_holder), TMEM_COLS);
      tmem_relinquish();
    }
  }
  pdl_wait();  // offsets, the A rows and the row-block counters come from earlier launches
  for (int i = threadIdx.x; i <= G; i += GEMM_THREADS)
    seg[i] = args.offsets ? args.offsets[i] : (i == 0 ? 0 : args.rows_single);
  __syncthreads();  // seg[] visible
  if (warp == 2) {
    // mt_pre = exclusive prefix over groups of their row blocks
    const int per = (G + 31) / 32;
    const int g0 = lane * per;
    int local = 0;
    for (int g = g0; g < g0 + per && g < G; ++g)
      local += (seg[g + 1] - seg[g] + S::TILE_M - 1) / S::TILE_M;
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - local;
    for (int g = g0; g < g0 + per && g < G; ++g) {
      mt_pre[g] = run;
      run += (seg[g + 1] - seg[g] + S::TILE_M - 1) / S::TILE_M;
    }
    if (lane == 31) mt_pre[G] = incl;
  }
  tc_fence_before();
  if constexpr (PAIR == 2) {
    cluster_sync_all();  // barriers of both CTAs initialised before any cross-CTA use
  } else {
    __syncthreads();
  }
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int tiles0 = mt_pre[G] * nt0 + mt_s * nt0s;
  const int total = tiles0 + (two ? mt_pre[G] * nt1 + mt_s * nt1s : 0);
  long long tma_issued = 0;  // producer thread only
  long long q_issued = 0;    // FP8: the converters' issuing thread only

  // ---- tile order.  Static: tile t runs on unit t % units.  Dynamic (bf16
  // weights with a tile counter): the leader's producer draws the tiles from
  // the launch-wide counter; each CTA's producer hands them on through a
  // QD-slot queue to its own MMA issuer and epilogue warps, the leader's
  // through a second one to the peer's producer.  Units that drew cheap
  // tiles (swapped tails, short groups) then take more.  Counter values only
  // grow, so every role sees its tiles in increasing order and every phase-0
  // tile is taken before any phase-1 tile.
  const bool dyn = !FP8 && args.tile_counter != nullptr;
  const bool drawer = dyn && leader;   // on the producer thread
  struct TileQueue { int next; uint32_t slot, phase; };
  auto advance = [&](TileQueue& q) {
    if (++q.slot == (uint32_t)QD) { q.slot = 0; q.phase ^= 1u; }
  };
  // the MMA issuer and the epilogue warps: the next tile index, total when
  // none is left, or -1 when the role must give up (a bounded wait ran out
  // or the CTA aborted)
  auto take_tile = [&](TileQueue& q) -> int {
    if (!dyn) {
      const int t = q.next;
      q.next += units;
      return t < total ? t : total;
    }
    if (!mbar_wait_bounded(lqfull_bar(q.slot), q.phase, abort_flag, status)) return -1;
    const int t = lq[q.slot];
    mbar_arrive(lqempty_bar(q.slot));
    advance(q);
    return t;
  };
  // the producers: the next tile (the drawer's: `drawn`), passed on to the
  // peer's producer and to this CTA's consumers; -1 to give up
  auto producer_next = [&](TileQueue& pqs, TileQueue& lqs, int drawn) -> int {
    if (!dyn) return take_tile(pqs);
    int t;
    if (leader) {
      t = min(drawn, total);
      if constexpr (PAIR == 2) {
        if (!mbar_wait_bounded_cluster(pqempty_bar(pqs.slot), pqs.phase ^ 1u, abort_flag, status))
          return -1;
        st_shared_cluster_s32(mapa_shared(smem_u32(const_cast<const int*>(pq + pqs.slot)), 1), t);
        mbar_arrive_cluster(mapa_shared(pqfull_bar(pqs.slot), 1));
        advance(pqs);
      }
    } else {
      if (!mbar_wait_bounded_cluster(pqfull_bar(pqs.slot), pqs.phase, abort_flag, status))
        return -1;
      t = pq[pqs.slot];
      mbar_arrive_cluster(mapa_shared(pqempty_bar(pqs.slot), 0));
      advance(pqs);
    }
    if (!mbar_wait_bounded(lqempty_bar(lqs.slot), lqs.phase ^ 1u, abort_flag, status)) return -1;
    lq[lqs.slot] = t;
    mbar_arrive(lqfull_bar(lqs.slot));
    advance(lqs);
    return t;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    // (with skip_producer set no copy and no full-barrier arrival is issued:
    // the consumers' bounded waits run out, and tma_issued stays 0 so the
    // abort path drains nothing)
    if (lane == 0 && !args.skip_producer) {
      uint32_t stage = 0, phase = 0;
      long long issued = 0;
      bool ok = true;
      TileCursor<S::TILE_M> cur;
      TileQueue pqs{unit, 0u, 0u}, lqs{unit, 0u, 0u};
      int tile = producer_next(pqs, lqs, drawer ? atomicAdd(args.tile_counter, 1) : 0);
      while (true) {
        if (tile < 0) { ok = false; break; }
        if (tile >= total) break;
        // the drawer takes the following tile now and publishes it once this
        // tile's copies are issued: the atomic's round trip overlaps them
        int drawn = 0;
        if (drawer) drawn = atomicAdd(args.tile_counter, 1);
        int a_row, rows_left, n, rb;
        cur.locate(tile, tiles0, nt0, nt1, mt_pre, seg, G, mt_s, rows_s, a_row, rows_left, n, rb);
        const int ph = cur.phase;
        const bool sh = cur.g == G;
        const int gi = sh ? 0 : cur.g;   // weight / bias block of the group
        const CUtensorMap* mA = map_a(ph, sh);
        const CUtensorMap* mB = map_b(ph, sh);
        const int nkb = nkb_of(ph, sh);
        const int n_out = n_out_of(ph, sh);
        if (SMALL_A && min(rows_left, S::TILE_M) > a_box) {
          // more rows in a group than the launch was planned for: the rows
          // past a_box are not loaded; report it (the tile is still run)
          atomicExch(status, (int)MOE_ERR_INVALID_ARG);
        }
        if (ph == 1) {
          // the A rows of this tile are phase 0's output: wait until every
          // phase-0 tile of the row block has been stored and released
          const int* cnt = sh ? args.rows_done_s + rb : args.rows_done + rb;
          const int target = sh ? rows_done_target_s : rows_done_target;
          const long long t0 = clock64();
          while (ld_acquire_gpu(cnt) < target) {
            if (*abort_flag) { ok = false; break; }
            if (clock64() - t0 > kWaitLimitCycles) {
              *abort_flag = 1;
              atomicExch(status, (int)MOE_ERR_TIMEOUT);
              ok = false;
              break;
            }
          }
          if (!ok) break;
          fence_proxy_async_global();  // the TMA reads below see those plain stores
        }
        const bool glu = (ph ? args.ph[1].mode : args.ph[0].mode) == EPI_SWIGLU;
        // B rows of the tile: n_out-row blocks per group, or for SwiGLU 128
        // gate rows and the 128 matching up rows (the odd CTA of a pair, or
        // the second half of a single CTA's B tile, takes the up rows)
        const int b_row = glu ? gi * 2 * n_out + (int)rank * n_out + n * (BN / 2)
                              : gi * n_out + n * BN + (int)rank * S::B_ROWS;
        const int a_row_cta = a_row + (int)rank * 128;
        // swapped tail tile: each CTA copies the usual 128-row token box,
        // starting at its half of the rows (the MMA's N reads only that half)
        const bool sw = swapped_tail(ph, rows_left);
        const int half = sw ? (rows_left + 15) / 16 * 8 : 0;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, status)) {
            ok = false;
            break;
          }
          if constexpr (PAIR == 2) {
            // both CTAs' copies complete on the even CTA's full barrier
            const uint32_t fb = mapa_shared(full_bar(stage), 0);
            if (leader) mbar_arrive_expect_tx(full_bar(stage), 2 * S::TX_BYTES);
            tma_load_2d_pair(sA + stage * A_BYTES, mA, fb, kb * BK,
                             sw ? a_row + (int)rank * half : a_row_cta);
            if constexpr (!FP8) tma_load_2d_pair(sB + stage * S::B_BYTES, mB, fb, kb * BK, b_row);
          } else if constexpr (FP8) {
            mbar_arrive_expect_tx(full_bar(stage), a_slot);
            tma_load_2d(sA + stage * a_slot, mA, full_bar(stage), kb * BK, a_row_cta);
          } else {
            mbar_arrive_expect_tx(full_bar(stage), S::TX_BYTES);
            tma_load_2d(sA + stage * A_BYTES, mA, full_bar(stage), kb * BK, a_row_cta);
            if (glu) {
              // two 128-row boxes: gate rows, then up rows (128 * BK * 2 bytes further)
              tma_load_2d(sB + stage * S::B_BYTES, mB, full_bar(stage), kb * BK, b_row);
              tma_load_2d(sB + stage * S::B_BYTES + 128 * BK * 2, mB, full_bar(stage), kb * BK,
                          b_row + n_out);
            } else {
              tma_load_2d(sB + stage * S::B_BYTES, mB, full_bar(stage), kb * BK, b_row);
            }
          }
          ++issued;
          if (++stage == a_slots) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tile = producer_next(pqs, lqs, drawn);
      }
      tma_issued = issued;
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && leader) {
      constexpr uint32_t idesc_full = idesc_bf16_f32(128 * PAIR, BN);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      uint32_t cstage = 0, cphase = 0;  // FP8: B ring
      bool ok = true;
      TileCursor<S::TILE_M> cur;
      TileQueue tqs{unit, 0u, 0u};
      while (ok) {
        const int tile = take_tile(tqs);
        if (tile < 0) { ok = false; break; }
        if (tile >= total) break;
        int a_row, rows_left, n, rb;
        cur.locate(tile, tiles0, nt0, nt1, mt_pre, seg, G, mt_s, rows_s, a_row, rows_left, n, rb);
        const int nkb = nkb_of(cur.phase, cur.g == G);
        // swapped tail tile: M = the 256 weight rows, N = the token rows rounded to 16
        const bool sw = swapped_tail(cur.phase, rows_left);
        const uint32_t idesc =
            sw ? idesc_bf16_f32(128 * PAIR, (rows_left + 15) / 16 * 16) : idesc_full;
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
          if constexpr (FP8) {
            // the converted B tiles of both CTAs (the peer's arrivals are
            // cluster-scope releases)
            if (!mbar_wait_bounded_cluster(cfull_bar(cstage), cphase, abort_flag, status)) {
              ok = false;
              break;
            }
          }
          tc_fence_after();
          const uint64_t tdesc = sdesc_kmajor_sw128(sA + stage * a_slot);   // token rows
          const uint64_t wdesc =
              sdesc_kmajor_sw128(sB + (FP8 ? cstage : stage) * S::B_BYTES);  // weight rows
          const uint64_t adesc = sw ? wdesc : tdesc;
          const uint64_t bdesc = sw ? tdesc : wdesc;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            // +32 bytes along K per step of 16 bf16 inside the 128-byte swizzle atom
            const uint32_t accum = (kb | kk) != 0 ? 1u : 0u;
            if constexpr (PAIR == 2)
              umma_bf16_pair(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, accum);
            else
              umma_bf16(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, accum);
          }
          if constexpr (PAIR == 2) umma_commit_pair_mc(empty_bar(stage), 0x3);
          else umma_commit(empty_bar(stage));
          if (++stage == a_slots) { stage = 0; phase ^= 1u; }
          if constexpr (FP8) {
            if constexpr (PAIR == 2) umma_commit_pair_mc(cempty_bar(cstage), 0x3);
            else umma_commit(cempty_bar(cstage));
            if (++cstage == S::B_STAGES) { cstage = 0; cphase ^= 1u; }
          }
        }
        if (!ok) break;
        if constexpr (PAIR == 2) umma_commit_pair_mc(tfull_bar(acc), 0x3);
        else umma_commit(tfull_bar(acc));
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
    }
    __syncwarp();
  } else if (FP8 && warp >= 2 + EPI_WARPS) {
    // ------------------------------------------------------------ E4M3 -> bf16
    // The converter warps fetch the E4M3 B rows themselves (lane 0 of the
    // first one issues the copies, Q_STAGES slots of two k-blocks ahead) and
    // widen each k-block's [B_ROWS][64] codes into the bf16 tile the MMA
    // reads.  Both tiles are in the 128-byte swizzled layout (8-row groups of
    // 1024 bytes, 16-byte chunk c of row r at c ^ (r % 8)): the Q rows as the
    // copies write them (128 codes a row), the bf16 rows as the MMA reads
    // them (64 values a row).
    const int cw = warp - (2 + EPI_WARPS);
    const bool issuer = cw == 0 && lane == 0;
    // position of the next copy: tile, k-block and its B rows
    TileCursor<S::TILE_M> lcur;
    int l_tile = unit, l_kq = 0, l_nkq = 0, l_brow = 0, l_n_out = 0;
    bool l_glu = false;
    const CUtensorMap* l_map = &tmB0;
    auto l_locate = [&]() {
      int a_row, rows_left, n, rb;
      lcur.locate(l_tile, tiles0, nt0, nt1, mt_pre, seg, G, mt_s, rows_s, a_row, rows_left, n, rb);
      const int ph = lcur.phase;
      const bool sh = lcur.g == G;
      const int gi = sh ? 0 : lcur.g;
      l_map = map_b(ph, sh);
      l_nkq = (nkb_of(ph, sh) + 1) / 2;  // Q slots of the tile
      l_n_out = n_out_of(ph, sh);
      l_glu = (ph ? args.ph[1].mode : args.ph[0].mode) == EPI_SWIGLU;
      // the B rows the producer of a bf16 tile would load (see above)
      l_brow = l_glu ? gi * 2 * l_n_out + (int)rank * l_n_out + n * (BN / 2)
                     : gi * l_n_out + n * BN + (int)rank * S::B_ROWS;
    };
    auto issue = [&](int slot) {
      const uint32_t dq = sBq + slot * S::BQ_BYTES;
      mbar_arrive_expect_tx(qfull_bar(slot), S::BQ_BYTES);
      if (l_glu && PAIR == 1) {
        tma_load_2d(dq, l_map, qfull_bar(slot), l_kq * S::BKQ, l_brow);
        tma_load_2d(dq + 128 * S::BKQ, l_map, qfull_bar(slot), l_kq * S::BKQ,
                    l_brow + l_n_out);
      } else {
        tma_load_2d(dq, l_map, qfull_bar(slot), l_kq * S::BKQ, l_brow);
      }
      ++q_issued;
      if (++l_kq == l_nkq) {
        l_kq = 0;
        l_tile += units;
        if (l_tile < total) l_locate();
      }
    };
    if (issuer && l_tile < total) {
      l_locate();
      for (int s2 = 0; s2 < S::Q_STAGES && l_tile < total; ++s2) issue(s2);
    }
    uint32_t qs = 0, qph = 0, cs = 0, cph = 0;
    bool ok = true;
    TileCursor<S::TILE_M> ccur;
    for (int tile = unit; tile < total && ok; tile += units) {
      int a_row_c, rows_left_c, n_c, rb_c;
      ccur.locate(tile, tiles0, nt0, nt1, mt_pre, seg, G, mt_s, rows_s, a_row_c, rows_left_c, n_c,
                  rb_c);
      const int nkb = nkb_of(ccur.phase, ccur.g == G);
      for (int kb = 0; kb < nkb; ++kb) {
        // k-block kb is half kb % 2 of Q slot kb / 2 of the tile
        bool got = (kb & 1) ? true : mbar_wait_bounded(qfull_bar(qs), qph, abort_flag, status);
        if (got) got = mbar_wait_bounded(cempty_bar(cs), cph ^ 1u, abort_flag, status);
        if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
        const uint8_t* q = smem + (sBq - sA) + qs * S::BQ_BYTES;
        uint8_t* b = smem + (sB - sA) + cs * S::B_BYTES;
        const int h4 = (kb & 1) * 4;  // first 16-byte chunk of this k-block in a Q row
#pragma unroll 2
        for (int g8 = cw; g8 < S::B_ROWS / 8; g8 += S::CONV_WARPS) {
          // 8-row group g8; each quarter-warp takes rows rr and rr ^ 5 of it
          // (they differ in bits 0 and 2, so neither the swizzled Q reads nor
          // the swizzled bf16 writes of a quarter-warp share a bank), and lane
          // c4 the 16 codes at K columns 16*c4 .. of the k-block
          const int rr = (lane & 4) ? ((lane >> 3) ^ 5) : (lane >> 3);
          const int c4 = lane & 3;
          const uint4 in = *reinterpret_cast<const uint4*>(
              q + (g8 * 8 + rr) * S::BKQ + (((h4 + c4) ^ rr) << 4));
          uint8_t* row = b + g8 * 1024 + rr * 128;
          uint4 o0, o1;
          e4m3x4_to_bf16x4(in.x, o0.x, o0.y);
          e4m3x4_to_bf16x4(in.y, o0.z, o0.w);
          e4m3x4_to_bf16x4(in.z, o1.x, o1.y);
          e4m3x4_to_bf16x4(in.w, o1.z, o1.w);
          *reinterpret_cast<uint4*>(row + (((2 * c4) ^ rr) << 4)) = o0;
          *reinterpret_cast<uint4*>(row + (((2 * c4 + 1) ^ rr) << 4)) = o1;
        }
        fence_proxy_async_shared();  // the tensor cores read what the threads wrote
        __syncwarp();
        const bool slot_done = (kb & 1) || kb == nkb - 1;
        if (lane == 0) {
          if (slot_done) mbar_arrive(qempty_bar(qs));
          if (PAIR == 2 && !leader) mbar_arrive_cluster(mapa_shared(cfull_bar(cs), 0));
          else mbar_arrive(cfull_bar(cs));
        }
        if (++cs == S::B_STAGES) { cs = 0; cph ^= 1u; }
        if (!slot_done) continue;
        if (cw == 0) {
          // once every converter warp has read slot qs, refill it
          int refill_ok = 1;
          if (issuer && l_tile < total) {
            if (mbar_wait_bounded(qempty_bar(qs), qph, abort_flag, status)) issue((int)qs);
            else refill_ok = 0;
          }
          if (!__shfl_sync(0xffffffffu, refill_ok, 0)) { ok = false; break; }
        }
        if (++qs == S::Q_STAGES) { qs = 0; qph ^= 1u; }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                  // TMEM lane quarter this warp may access
    const int cpart = (warp - 2) >> 2;       // which EPI_COLS-wide column slice of the tile
    const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
    const int warp_row0 = (int)rank * 128 + q * 32;  // first tile row of this warp
    uint16_t* my_bias = bias_stage + (warp - 2) * EPI_COLS;
    float* my_scale = scale_stage + (warp - 2) * EPI_COLS;  // FP8: per output column
    uint32_t acc = 0, acc_phase = 0;
    TileCursor<S::TILE_M> cur;
    TileQueue tqs{unit, 0u, 0u};
    while (true) {
      int tile = 0;
      if (lane == 0) tile = take_tile(tqs);
      tile = __shfl_sync(0xffffffffu, tile, 0);
      if (tile < 0 || tile >= total) break;
      int a_row, rows_left, n, rb;
      cur.locate(tile, tiles0, nt0, nt1, mt_pre, seg, G, mt_s, rows_s, a_row, rows_left, n, rb);
      const bool sh = cur.g == G;
      const int gi = sh ? 0 : cur.g;   // weight / bias block of the group
      const PhaseView P(args, cur.phase, sh);
      const int n_out = P.n_out;
      if (swapped_tail(cur.phase, rows_left)) {
        // Swapped tail tile: output columns in TMEM lanes, token rows in
        // columns.  This warp takes the 32 output columns of its lane quarter
        // and every (EPI_WARPS / 4)-th 8-token chunk, transposed through its
        // shared buffer into 16-byte stores along the output rows.
        const int n16 = (rows_left + 15) / 16 * 16;
        const int colq = n * BN + (int)rank * S::B_ROWS + q * 32;   // the warp's first column
        const int colw = colq + lane;
        float bz = 0.0f, sz = 1.0f;
        if (colw < n_out) {
          if (P.bias) bz = __bfloat162float(P.bias[(size_t)gi * n_out + colw]);
          if (FP8 && P.b_scale) sz = P.b_scale[(size_t)gi * n_out + colw];
        }
        // this warp's chunks: 8 tokens at c = cpart * 8 + i * CSTEP, two per
        // TMEM round trip; lane l holds the gate weight of token c + l % 8.
        // The loop stays rolled (an unrolled one, with every activation
        // inlined, made the whole launch slower through its code size); the
        // weights of the next two chunks are fetched one pass ahead, those
        // of the first two before the accumulator is ready.
        constexpr int CSTEP = 8 * (EPI_WARPS / 4);
        const bool gate_w = P.mode == EPI_SCALE && P.topk_w != nullptr;
        auto gate_of = [&](int c) {
          const int tok = c + (lane & 7);
          return gate_w && tok < rows_left ? P.topk_w[P.perm[a_row + tok]] : 1.0f;
        };
        float wn0 = gate_of(cpart * 8), wn1 = gate_of(cpart * 8 + CSTEP);
        int ok = 1;
        if (lane == 0) ok = mbar_wait_bounded(tfull_bar(acc), acc_phase, abort_flag, status) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        tc_fence_after();
        uint16_t* tb = trans_stage + (warp - 2) * 8 * 32;
        const uint32_t taddr = tmem_base + lane_addr + acc * BN;
        // one 8-token chunk: activation (or gate weight), then the transpose
        // into 16-byte stores along the output rows
        auto chunk = [&](const uint32_t* r, int c, float wv) {
          float o[8];
          if (P.mode == EPI_GELU) {
#pragma unroll
            for (int t = 0; t < 8; ++t) o[t] = gelu_erf(__uint_as_float(r[t]) * sz + bz);
          } else if (P.mode == EPI_SILU) {
#pragma unroll
            for (int t = 0; t < 8; ++t) o[t] = silu_f(__uint_as_float(r[t]) * sz + bz);
          } else {
#pragma unroll
            for (int t = 0; t < 8; ++t)
              o[t] = __shfl_sync(0xffffffffu, wv, t) * (__uint_as_float(r[t]) * sz + bz);
          }
#pragma unroll
          for (int t = 0; t < 8; ++t) tb[t * 32 + lane] = __bfloat16_as_ushort(__float2bfloat16_rn(o[t]));
          __syncwarp();
          const int t = lane >> 2, c8 = (lane & 3) * 8;
          if (c + t < rows_left && colq + c8 < n_out)
            *reinterpret_cast<uint4*>(P.out + (int64_t)(a_row + c + t) * P.ld_out + colq + c8) =
                *reinterpret_cast<const uint4*>(tb + t * 32 + c8);
          __syncwarp();
        };
#pragma unroll 1
        for (int c0 = cpart * 8; c0 < n16; c0 += 2 * CSTEP) {
          const int c1 = c0 + CSTEP;
          const float w0 = wn0, w1 = wn1;
          if (c0 + 2 * CSTEP < n16) {
            wn0 = gate_of(c0 + 2 * CSTEP);
            wn1 = gate_of(c1 + 2 * CSTEP);
          }
          uint32_t r0[8], r1[8];
          tmem_ld_32x32b_x8(taddr + c0, r0);
          if (c1 < n16) tmem_ld_32x32b_x8(taddr + c1, r1);
          tmem_ld_wait();
          chunk(r0, c0, w0);
          if (c1 < n16) chunk(r1, c1, w1);
        }
      } else {
      const int r_in = warp_row0 + lane;
      const bool row_ok = r_in < rows_left;
      const int64_t out_row = (int64_t)a_row + r_in;
      const bool glu = P.mode == EPI_SWIGLU;
      // this warp's output columns: EPI_COLS of a 256-wide tile, or half as
      // many of a 128-wide SwiGLU tile (whose accumulator holds 128 gate +
      // 128 up)
      const int wcols = glu ? EPI_COLS / 2 : EPI_COLS;
      const int col0 = n * (glu ? BN / 2 : BN) + cpart * wcols;
      // everything that does not need the accumulator is fetched before waiting
      float wscale = 1.0f;
      if (P.mode == EPI_SCALE && P.topk_w != nullptr && row_ok)
        wscale = P.topk_w[P.perm[out_row]];
      const bool has_bias = P.bias != nullptr;
      const bool has_scale = FP8 && P.b_scale != nullptr;
      if (has_bias || has_scale) {
        // EPI_COLS staged values per warp, 2 per lane and pass: the slice's
        // biases (and FP8 column scales), or for SwiGLU its wcols gate values
        // followed by its wcols up values
#pragma unroll
        for (int j2 = lane * 2; j2 < EPI_COLS; j2 += 64) {
          int c2 = col0 + j2;
          size_t off = (size_t)gi * n_out + c2;
          if (glu) {
            const bool up = j2 >= wcols;
            c2 = col0 + (up ? j2 - wcols : j2);
            off = (size_t)gi * 2 * n_out + (up ? n_out : 0) + c2;
          }
          if (has_bias) {
            uint32_t b = 0u;
            if (c2 < n_out) b = __ldg(reinterpret_cast<const uint32_t*>(P.bias + off));
            *reinterpret_cast<uint32_t*>(my_bias + j2) = b;
          }
          if (has_scale) {
            float2 sc = make_float2(0.0f, 0.0f);
            if (c2 < n_out) sc = __ldg(reinterpret_cast<const float2*>(P.b_scale + off));
            *reinterpret_cast<float2*>(my_scale + j2) = sc;
          }
        }
        __syncwarp();
      }
      int ok = 1;
      if (lane == 0) ok = mbar_wait_bounded(tfull_bar(acc), acc_phase, abort_flag, status) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      __nv_bfloat16* orow = P.out + out_row * P.ld_out;
      const bool warp_has_rows = warp_row0 < rows_left;     // warp-uniform
      const bool full_cols = col0 + wcols <= n_out;         // warp-uniform
      if (warp_has_rows && col0 < n_out && glu) {
        // wcols output columns in pieces of 16: gate and up accumulators
        const uint32_t tg = tmem_base + lane_addr + acc * BN + cpart * wcols;
#pragma unroll 1
        for (int h = 0; h < EPI_COLS / 32; ++h) {
          uint32_t rg[16], ru[16];
          tmem_ld_32x32b_x16(tg + h * 16, rg);
          tmem_ld_32x32b_x16(tg + BN / 2 + h * 16, ru);
          tmem_ld_wait();
          float v[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float g = __uint_as_float(rg[i]), u = __uint_as_float(ru[i]);
            if (has_scale) {
              g *= my_scale[h * 16 + i];
              u *= my_scale[EPI_COLS / 2 + h * 16 + i];
            }
            if (has_bias) {
              const uint16_t bgate = my_bias[h * 16 + i], bup = my_bias[EPI_COLS / 2 + h * 16 + i];
              g += __uint_as_float((uint32_t)bgate << 16);
              u += __uint_as_float((uint32_t)bup << 16);
            }
            v[i] = silu_f(g) * u;
          }
          uint4 o[2];
#pragma unroll
          for (int j8 = 0; j8 < 2; ++j8) {
            o[j8].x = pack_bf16x2(v[8 * j8 + 0], v[8 * j8 + 1]);
            o[j8].y = pack_bf16x2(v[8 * j8 + 2], v[8 * j8 + 3]);
            o[j8].z = pack_bf16x2(v[8 * j8 + 4], v[8 * j8 + 5]);
            o[j8].w = pack_bf16x2(v[8 * j8 + 6], v[8 * j8 + 7]);
          }
          const int col = col0 + h * 16;
          uint4* dst = reinterpret_cast<uint4*>(orow + col);
          if (row_ok) {
#pragma unroll
            for (int j8 = 0; j8 < 2; ++j8)
              if (full_cols || col + 8 * j8 < n_out) dst[j8] = o[j8];
          }
        }
      } else if (warp_has_rows && col0 < n_out) {
        const uint32_t taddr = tmem_base + lane_addr + acc * BN + cpart * EPI_COLS;
        // CW = 16 columns per TMEM load: half the inlined activation code of
        // 32-wide passes, which matters for the instruction cache
        constexpr int CW = 16;
#pragma unroll 1
        for (int c = 0; c < EPI_COLS / CW; ++c) {
          uint32_t r[CW];
          tmem_ld_32x32b_x16(taddr + c * CW, r);
          tmem_ld_wait();
          float v[CW];
#pragma unroll
          for (int i = 0; i < CW; ++i) v[i] = __uint_as_float(r[i]);
          if (has_scale) {
#pragma unroll
            for (int i = 0; i < CW; ++i) v[i] *= my_scale[c * CW + i];
          }
          if (has_bias) {
#pragma unroll
            for (int j8 = 0; j8 < CW / 8; ++j8) {
              const uint4 u = *reinterpret_cast<const uint4*>(my_bias + c * CW + 8 * j8);
              v[8 * j8 + 0] += bf16lo(u.x); v[8 * j8 + 1] += bf16hi(u.x);
              v[8 * j8 + 2] += bf16lo(u.y); v[8 * j8 + 3] += bf16hi(u.y);
              v[8 * j8 + 4] += bf16lo(u.z); v[8 * j8 + 5] += bf16hi(u.z);
              v[8 * j8 + 6] += bf16lo(u.w); v[8 * j8 + 7] += bf16hi(u.w);
            }
          }
          if (P.mode == EPI_GELU) {
#pragma unroll
            for (int i = 0; i < CW; ++i) v[i] = gelu_erf(v[i]);
          } else if (P.mode == EPI_SILU) {
#pragma unroll
            for (int i = 0; i < CW; ++i) v[i] = silu_f(v[i]);
          } else {
#pragma unroll
            for (int i = 0; i < CW; ++i) v[i] *= wscale;
          }
          uint4 o[CW / 8];
#pragma unroll
          for (int j8 = 0; j8 < CW / 8; ++j8) {
            o[j8].x = pack_bf16x2(v[8 * j8 + 0], v[8 * j8 + 1]);
            o[j8].y = pack_bf16x2(v[8 * j8 + 2], v[8 * j8 + 3]);
            o[j8].z = pack_bf16x2(v[8 * j8 + 4], v[8 * j8 + 5]);
            o[j8].w = pack_bf16x2(v[8 * j8 + 6], v[8 * j8 + 7]);
          }
          const int col = col0 + c * CW;
          uint4* dst = reinterpret_cast<uint4*>(orow + col);
          if (row_ok) {
            if (full_cols) {
#pragma unroll
              for (int j8 = 0; j8 < CW / 8; ++j8) dst[j8] = o[j8];
            } else {
#pragma unroll
              for (int j8 = 0; j8 < CW / 8; ++j8)
                if (col + 8 * j8 < n_out) dst[j8] = o[j8];
            }
          }
        }
      }
      }  // normal tile
      if (two && cur.phase == 0) {
        // Hand the row block's stores to phase 1: the last of this CTA's
        // epilogue warps to finish the tile (a CTA-scope acquire-release
        // count) releases them at GPU scope with one red.release.  This
        // comes before the warp frees the accumulator, so every count of
        // this tile precedes any count of the next tile on the same buffer.
        __syncwarp();
        if (lane == 0 && atom_add_acqrel_cta(&stored_cnt[acc], 1u) == EPI_WARPS - 1) {
          stored_cnt[acc] = 0u;
          fence_proxy_async_global();
          red_release_gpu_add((sh ? args.rows_done_s : args.rows_done) + rb, 1);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (PAIR == 2) {
          if (leader) mbar_arrive(tempty_bar(acc));
          else mbar_arrive_cluster(mapa_shared(tempty_bar(acc), 0));
        } else {
          mbar_arrive(tempty_bar(acc));
        }
      }

      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  // ---- teardown: every MMA has completed (observed through tmem_full or
  // the drain barrier) and every TMEM load has been waited for.
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // Some role gave up, so copies or MMAs may still be in flight.  Let them
    // land / finish before shared memory and TMEM go away.
    if (warp == 0 && lane == 0) {
      if (PAIR == 1 || leader) {
        // the full barriers count every byte issued to this CTA's ring
        const long long first = tma_issued > a_slots ? tma_issued - a_slots : 0;
        for (long long j = first; j < tma_issued; ++j)
          mbar_wait_drain(full_bar((int)(j % a_slots)), (uint32_t)((j / a_slots) & 1));
      } else {
        // the odd CTA's copies complete on its peer's barriers: give them a
        // bounded grace period (they land within microseconds)
        const long long t0 = clock64();
        while (clock64() - t0 < 4000000LL) {
        }
      }
    }
    if constexpr (FP8) {
      if (warp == 2 + EPI_WARPS && lane == 0) {
        // the converters' E4M3 copies complete on this CTA's Q ring
        constexpr int QS = S::Q_STAGES;
        const long long first = q_issued > QS ? q_issued - QS : 0;
        for (long long j = first; j < q_issued; ++j)
          mbar_wait_drain(qfull_bar((int)(j % QS)), (uint32_t)((j / QS) & 1));
      }
    }
    if (warp == 1 && lane == 0 && leader) {
      if constexpr (PAIR == 2) umma_commit_pair_mc(drain_bar, 0x1);
      else umma_commit(drain_bar);
      mbar_wait_drain(drain_bar, 0);
    }
    __syncwarp();
  }
  if constexpr (PAIR == 2) {
    // neither CTA leaves while its peer may still touch its shared memory,
    // barriers or TMEM
    cluster_sync_all();
  }
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR == 2) tmem_dealloc_pair(tmem_base, TMEM_COLS);
    else tmem_dealloc(tmem_base, TMEM_COLS);
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

// E4M3 codes [rows, K] (K bytes per row), boxes of 128 codes a row in the
// 128-byte swizzled layout; the converter warps write the bf16 tile.
bool encode_tensor_map_u8(CUtensorMap* map, const void* base, int64_t rows, int64_t K,
                          int box_cols, int box_rows) {
  EncodeTiledFn enc = get_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// CTA pairs: a group's last row block runs operand-swapped when it holds at
// most this many rows.
constexpr int kSwapTailRows = 255;

// Launches with at least this many tiles (row blocks without tails x column
// blocks) per CTA pair (or CTA) take their tiles in dynamic order.
constexpr int64_t kDynamicTilesPerUnit = 100;

cudaError_t make_gemm_plan(GemmPlan* plan, const GemmArgs& args_in, const __nv_bfloat16* A,
                           int64_t a_rows, const void* const B[2], const int64_t b_rows[2],
                           bool fp8, int64_t group_rows_max, int num_sms,
                           const __nv_bfloat16* A_s, const void* const* B_s,
                           const int64_t* b_rows_s) {
  GemmArgs args = args_in;
  const int np = args.num_phases;
  const bool sh = args.shared_rows > 0;
  if (np < 1 || np > 2 || a_rows < 0 || (a_rows == 0 && !sh)) return cudaErrorInvalidValue;
  if (sh && (A_s == nullptr || B_s == nullptr || b_rows_s == nullptr || args.shp[0].out == nullptr))
    return cudaErrorInvalidValue;
  for (int p = 0; p < np; ++p) {
    if ((a_rows > 0 && b_rows[p] <= 0) || args.ph[p].K <= 0 || args.ph[p].n_out <= 0 ||
        (fp8 && (args.ph[p].K % 16 != 0 || (a_rows > 0 && args.ph[p].b_scale == nullptr))))
      return cudaErrorInvalidValue;
    if (sh && (b_rows_s[p] <= 0 || args.shp[p].K <= 0 || args.shp[p].n_out <= 0 ||
               (fp8 && (args.shp[p].K % 16 != 0 || args.shp[p].b_scale == nullptr))))
      return cudaErrorInvalidValue;
  }
  if (np == 2 && (args.rows_done == nullptr || args.ph[1].K != args.ph[0].n_out ||
                  args.ph[0].ld_out != args.ph[0].n_out))
    return cudaErrorInvalidValue;
  if (np == 2 && sh && (args.rows_done_s == nullptr || args.shp[1].K != args.shp[0].n_out ||
                        args.shp[0].ld_out != args.shp[0].n_out || args.shp[1].n_out != args.ph[1].n_out))
    return cudaErrorInvalidValue;
  // CTA pairs (256-row tiles) once the average group holds enough rows to
  // fill them; single CTAs (128-row tiles) for decode-sized groups.
  const int64_t avg_rows = a_rows > 0 ? a_rows / (args.num_groups > 0 ? args.num_groups : 1)
                                      : (int64_t)args.shared_rows;
  const int pair = (avg_rows >= 192 && num_sms >= 2) ? 2 : 1;
  // FP8 single-CTA tiles copy the A rows a group can hold, in steps of 16
  int a_box = 128;
  if (fp8 && pair == 1 && group_rows_max > 0 && group_rows_max < 128)
    a_box = (int)((group_rows_max + 15) / 16 * 16);
  args.a_box = a_box;
  auto encode_b = [&](CUtensorMap* m, const void* b, int64_t rows, int p, int K) {
    // SwiGLU tiles load 128 gate and 128 up rows: two 128-row boxes
    const int box_b = args.ph[p].mode == EPI_SWIGLU ? BN / 2 : BN / pair;
    return fp8 ? encode_tensor_map_u8(m, b, rows, K, 2 * BK, box_b)
               : encode_tensor_map_bf16(m, b, rows, K, BK, box_b);
  };
  for (int p = 0; p < np; ++p) {
    if (a_rows > 0) {
      // phase 1 reads phase 0's output [a_rows, n_out0] as its A operand
      const __nv_bfloat16* a = p == 0 ? A : args.ph[0].out;
      if (!encode_tensor_map_bf16(&plan->tmA[p], a, a_rows, args.ph[p].K, BK, a_box))
        return cudaErrorInvalidValue;
      if (!encode_b(&plan->tmB[p], B[p], b_rows[p], p, args.ph[p].K)) return cudaErrorInvalidValue;
    }
    if (sh) {
      const __nv_bfloat16* a = p == 0 ? A_s : args.shp[0].out;
      if (!encode_tensor_map_bf16(&plan->tmS[2 * p], a, args.shared_rows, args.shp[p].K, BK, a_box))
        return cudaErrorInvalidValue;
      if (!encode_b(&plan->tmS[2 * p + 1], B_s[p], b_rows_s[p], p, args.shp[p].K))
        return cudaErrorInvalidValue;
    }
  }
  if (np == 1) {
    plan->tmA[1] = plan->tmA[0];
    plan->tmB[1] = plan->tmB[0];
    plan->tmS[2] = plan->tmS[0];
    plan->tmS[3] = plan->tmS[1];
  }
  // maps a launch never reads still have to be valid descriptors
  if (a_rows == 0) {
    plan->tmA[0] = plan->tmS[0];
    plan->tmB[0] = plan->tmS[1];
    plan->tmA[1] = plan->tmS[2];
    plan->tmB[1] = plan->tmS[3];
  }
  if (!sh) {
    plan->tmS[0] = plan->tmA[0];
    plan->tmS[1] = plan->tmB[0];
    plan->tmS[2] = plan->tmA[1];
    plan->tmS[3] = plan->tmB[1];
  }
  args.swap_tail = pair == 2 ? kSwapTailRows : 0;
  plan->args = args;
  plan->pair = pair;
  plan->fp8 = fp8;
  const int64_t tile_m = 128 * pair;
  int64_t n_tiles = 0, n_tiles_s = 0;
  for (int p = 0; p < np; ++p) {
    const int bno = args.ph[p].mode == EPI_SWIGLU ? BN / 2 : BN;
    n_tiles += (args.ph[p].n_out + bno - 1) / bno;
    if (sh) n_tiles_s += (args.shp[p].n_out + bno - 1) / bno;
  }
  const int64_t max_tiles = ((a_rows + tile_m - 1) / tile_m + args.num_groups) * n_tiles +
                            (sh ? (args.shared_rows + tile_m - 1) / tile_m * n_tiles_s : 0);
  const int64_t max_units = num_sms / pair;
  const int64_t units = max_tiles < max_units ? max_tiles : max_units;
  plan->grid = (int)(units * pair);
  // Dynamic tile order only for long launches: measured on one B300 it took
  // 4-5 % off the Mixtral- and DeepSeek-sized prefill launches (about 125
  // tiles per CTA pair without tails, both under the power cap) and added
  // 2-3 % to the MoELayer and Switch-sized ones (9 and 69 per pair).
  const int64_t tiles_est = (a_rows + tile_m - 1) / tile_m * n_tiles +
                            (sh ? (args.shared_rows + tile_m - 1) / tile_m * n_tiles_s : 0);
  if (fp8 || units <= 0 || tiles_est < kDynamicTilesPerUnit * units) plan->args.tile_counter = nullptr;
  return cudaSuccess;
}

template <int PAIR, bool FP8>
static cudaError_t launch_gemm_t(const GemmPlan& plan, cudaStream_t st) {
  using S = GemmShape<PAIR, FP8>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<PAIR, FP8>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         S::smem_bytes(MAX_GROUPS));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(plan.grid);
  cfg.blockDim = dim3(S::THREADS);
  cfg.dynamicSmemBytes = S::smem_bytes(plan.args.num_groups);
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = PAIR;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see pdl_wait()
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  // A persistent grid must be co-resident: phase-1 tiles wait for phase-0
  // tiles owned by other CTAs.  No more CTAs (pairs) than fit at once.
  static int max_units = -1;
  if (max_units < 0) {
    int n = 0;
    if (PAIR == 2) {
      if (cudaOccupancyMaxActiveClusters(&n, grouped_gemm_kernel<PAIR, FP8>, &cfg) != cudaSuccess)
        n = 0;
    } else {
      int dev = 0, sms = 0, per_sm = 0;
      if (cudaGetDevice(&dev) == cudaSuccess &&
          cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, grouped_gemm_kernel<PAIR, FP8>,
                                                        S::THREADS,
                                                        S::smem_bytes(MAX_GROUPS)) == cudaSuccess)
        n = sms * per_sm;
    }
    max_units = n > 0 ? n : 1;
  }
  if ((int)cfg.gridDim.x > PAIR * max_units) cfg.gridDim.x = PAIR * max_units;
  return cudaLaunchKernelEx(&cfg, grouped_gemm_kernel<PAIR, FP8>, plan.tmA[0], plan.tmB[0],
                            plan.tmA[1], plan.tmB[1], plan.tmS[0], plan.tmS[1], plan.tmS[2],
                            plan.tmS[3], plan.args);
}

cudaError_t launch_gemm(const GemmPlan& plan, cudaStream_t st, LaunchTrace* tr) {
  trace_mark(tr, st);
  cudaError_t e;
  if (plan.fp8)
    e = plan.pair == 2 ? launch_gemm_t<2, true>(plan, st) : launch_gemm_t<1, true>(plan, st);
  else
    e = plan.pair == 2 ? launch_gemm_t<2, false>(plan, st) : launch_gemm_t<1, false>(plan, st);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace moe
