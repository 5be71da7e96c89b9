// Expert FFN for decode-sized batches, operands swapped: the expert weights
// are the 128-row M operand of tcgen05.mma and the few token rows an expert
// holds are the narrow N operand, so that the tensor cores do no work on
// padding rows and the launch streams the weights at the memory rate.
//
//   phase 0: Hid^T[f, j] = act( W1_e[f, :] . X_e[j, :] + b1_e[f] )
//   phase 1: y^T[h, j]   = w_j ( W2_e[h, :] . Hid_e[j, :] + b2_e[h] )
//
// for expert e's token rows j ("AI-Research-SKILLs MoE 训练实战" §3.1:
// Linear(H, 4H) -> GELU -> Linear(4H, H), the output weighted by the
// renormalised gate score; §6.1 SiLU / SwiGLU).  The always-on shared expert
// ("混合专家模型 MoE 架构深度解析" §3, Output = Shared(x) + sum_j w_j Routed_j(x))
// is one more group of the same launch: all T token rows, weight 1, its own
// weights and outputs.  Decode is bound by the weight bytes (INFER "FP8 量化":
// weight streaming dominates small batches), so with E4M3 weights converter
// warps widen the codes to bf16 in shared memory as they stream in.
//
// A tile is (phase, group, 256 weight rows, up to NT token rows): two M=128
// MMAs per k-step, half 0 into accumulator columns [0, NT) and half 1 into
// [NT, 2 NT), TMEM lanes holding weight rows.  The halves are 256
// consecutive weight rows (256 output columns, one copy of 32 KB per
// k-block), or for SwiGLU's first Linear the 128 gate rows and the 128
// matching up rows of 128 output columns.  Each copy instruction carries
// 16-32 KB of weights: the per-copy cost, not the bytes in flight, bounded
// an earlier 128-row version at 4.2 TB/s.
// Tiles are ordered phase 0 before phase 1, then group, weight block and
// token chunk (fastest); CTAs take them round-robin.  A phase-1 tile reads
// Hid rows of its group's token chunk, which every phase-0 tile of that
// chunk writes: each phase-0 tile releases a per-chunk counter in global
// memory (red.release.gpu after the last epilogue warp's stores), and the
// token producer of a phase-1 tile acquires it (bounded spin) before its
// Hid copies.
//
// Decode streams every expert weight once.  The weights have a ring of
// their own, filled by a producer that does not wait for the phase-1
// hand-over (bf16: 32 KB slots; E4M3: 32 KB slots of codes feeding a short
// bf16 ring), and the token rows a ring of small slots of their own.
//
// Roles: warp 0 token producer (TMA), warp 1 TMEM allocator and MMA issuer,
// warps 2-5 epilogue (TMEM lane quarter warp % 4: 32 weight rows each, all
// token columns, transposed through shared memory 16 tokens at a time into
// 16-byte stores along the output rows), then the weight producer: warp 6
// (TMA) with bf16 weights, or warps 6-13 with E4M3 weights, which copy the
// codes and widen them to bf16.
// Every wait is bounded: on expiry the CTA records MOE_ERR_TIMEOUT, lets its
// copies land, drains its MMAs, frees TMEM and exits.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {

namespace {

constexpr int DK = 64;                     // K per k-block: one 128-byte swizzled bf16 row
constexpr int DM = 128;                    // weight rows per MMA (M); a tile has two halves
constexpr int DBOX = 16;                   // token rows per activation copy
constexpr int D_A_BYTES = DM * DK * 2;     // one bf16 weight tile
constexpr int D_Q_BYTES = DM * 2 * DK;     // E4M3 codes of one half: 128 rows x 128 codes (two k-blocks)
constexpr int D_W_MAX = 8;                 // weight ring slots (bf16 tiles of both halves)
constexpr int D_X_MAX = 16;                // token ring slots
constexpr int D_Q_MAX = 8;                 // E4M3 ring slots (both halves)
constexpr int D_EPI_WARPS = 4;
constexpr int D_CONV_WARPS = 8;
constexpr int D_NT_MAX = 32;               // token rows per tile
constexpr long long kDecodeDrainCycles = 200000000LL;

// warps: 0 token producer, 1 MMA, 2-5 epilogue, then the weight producer
// (one warp with bf16 weights, the E4M3 converters otherwise)
template <bool FP8>
struct DShape {
  static constexpr int W_WARPS = FP8 ? D_CONV_WARPS : 1;
  static constexpr int THREADS = (2 + D_EPI_WARPS + W_WARPS) * 32;
};

__device__ __forceinline__ bool d_wait_drain(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kDecodeDrainCycles) return false;
  }
  return true;
}

// Tile position: phase, group, weight block, token chunk.  Tiles are visited
// in increasing order by each role, so the group only moves forward.
struct DCursor {
  int phase = 0, g = 0;
  __device__ __forceinline__ void locate(int tile, int tiles0, const int32_t* tp0,
                                         const int32_t* tp1, const int32_t* nch, int& wb,
                                         int& tc) {
    int local = tile;
    if (tile >= tiles0) {
      if (phase == 0) { phase = 1; g = 0; }
      local = tile - tiles0;
    }
    const int32_t* tp = phase ? tp1 : tp0;
    while (local >= tp[g + 1]) ++g;
    const int lg = local - tp[g];
    const int c = nch[g];
    wb = lg / c;
    tc = lg - wb * c;
  }
};

}  // namespace

// Per-group view of one tile's operands and outputs (routed expert g < G,
// or the shared expert g == G).
struct DTileView {
  bool shared;
  int rows;       // token rows of the group
  int row0;       // first activation / output row of the chunk
  int n_valid;    // token rows in this chunk
  int n_out;      // output columns of the phase (F, Fs or H)
  int K;          // reduction length of the phase
  int w_row;      // first weight row of half 0 (256 rows, or SwiGLU's 128 gate rows)
  int w_row_up;   // SwiGLU phase 0: first of half 1's 128 up rows
  int cols;       // output columns of the tile: 256, or 128 for SwiGLU
  int col0;       // first output column
};

__device__ __forceinline__ DTileView d_view(const DecodeArgs& a, const int32_t* seg, int phase,
                                            int g, int wb, int tc, int nt) {
  DTileView v;
  v.shared = g == a.num_groups;
  const int base = v.shared ? 0 : seg[g];
  v.rows = v.shared ? a.shared_rows : seg[g + 1] - seg[g];
  v.row0 = base + tc * nt;
  v.n_valid = min(nt, v.rows - tc * nt);
  const bool glu = phase == 0 && a.mode0 == EPI_SWIGLU;
  v.cols = glu ? DM : 2 * DM;
  v.col0 = wb * v.cols;
  if (phase == 0) {
    v.n_out = v.shared ? a.Fs : a.F;
    v.K = a.H;
    const int wrows = glu ? 2 * v.n_out : v.n_out;   // weight rows of one expert
    const int gbase = v.shared ? 0 : g * wrows;
    v.w_row = gbase + v.col0;
    v.w_row_up = gbase + v.n_out + v.col0;
  } else {
    v.n_out = a.H;
    v.K = v.shared ? a.Fs : a.F;
    v.w_row = (v.shared ? 0 : g * a.H) + v.col0;
    v.w_row_up = 0;
  }
  return v;
}

template <bool FP8>
__global__ void __launch_bounds__(DShape<FP8>::THREADS, 1)
    decode_ffn_kernel(const __grid_constant__ DecodeMaps maps, const DecodeArgs args) {
  constexpr int THREADS = DShape<FP8>::THREADS;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) atomicExch(args.status, (int)MOE_ERR_UNSUPPORTED);
    return;
  }
  const int NT = args.nt;
  const bool glu = args.mode0 == EPI_SWIGLU;
  const int WST = args.w_stages, XST = args.x_stages, QST = args.q_stages;
  constexpr int a_stage = 2 * D_A_BYTES;                 // bf16 weights of both halves
  const int x_stage = NT * DK * 2;                       // token bytes per ring slot
  constexpr int qslot = 2 * D_Q_BYTES;                   // E4M3 codes of both halves
  const int acc_cols = 2 * NT;                           // half 0's NT columns, then half 1's
  uint8_t* smem = smem_raw;
  const uint32_t sW = smem_u32(smem);
  const uint32_t sQ = sW + WST * a_stage;                // E4M3 slots (FP8)
  const uint32_t sX = sQ + (FP8 ? QST * qslot : 0);
  uint16_t* tbuf = reinterpret_cast<uint16_t*>(smem + (sX - sW) + XST * x_stage);  // [4][16][32]
  float* wv = reinterpret_cast<float*>(tbuf + D_EPI_WARPS * 16 * 32);              // [4][NT]
  uint64_t* bars = reinterpret_cast<uint64_t*>(wv + D_EPI_WARPS * D_NT_MAX);
  const uint32_t bar0 = smem_u32(bars);
  auto wfull_bar = [&](int s) { return bar0 + 8u * s; };
  auto wempty_bar = [&](int s) { return bar0 + 8u * (D_W_MAX + s); };
  auto xfull_bar = [&](int s) { return bar0 + 8u * (2 * D_W_MAX + s); };
  auto xempty_bar = [&](int s) { return bar0 + 8u * (2 * D_W_MAX + D_X_MAX + s); };
  auto qfull_bar = [&](int s) { return bar0 + 8u * (2 * D_W_MAX + 2 * D_X_MAX + s); };
  auto qempty_bar = [&](int s) { return bar0 + 8u * (2 * D_W_MAX + 2 * D_X_MAX + D_Q_MAX + s); };
  constexpr int TB = 2 * D_W_MAX + 2 * D_X_MAX + 2 * D_Q_MAX;
  auto tfull_bar = [&](int a) { return bar0 + 8u * (TB + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (TB + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (TB + 4);
  constexpr int NUM_BARS = TB + 5;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  uint32_t* stored_cnt = tmem_holder + 2;   // [2]
  const int G = args.num_groups;
  const int NG = G + (args.shared_rows > 0 ? 1 : 0);   // groups incl. the shared one
  int32_t* seg = reinterpret_cast<int32_t*>(tmem_holder + 4);   // [G + 2]
  int32_t* nch = seg + (G + 2);      // [G + 1] token chunks per group
  int32_t* cpre = nch + (G + 1);     // [G + 2] first chunk counter of each group
  int32_t* tp0 = cpre + (G + 2);     // [G + 2] phase-0 tile prefix
  int32_t* tp1 = tp0 + (G + 2);      // [G + 2] phase-1 tile prefix

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int unit = blockIdx.x, units = gridDim.x;
  constexpr int WW0 = 2 + D_EPI_WARPS;   // first weight-producer warp
  int* status = args.status;

  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < D_W_MAX; ++s) {
      mbar_init(wfull_bar(s), FP8 ? D_CONV_WARPS : 1);
      mbar_init(wempty_bar(s), 1);
    }
    for (int s = 0; s < D_X_MAX; ++s) {
      mbar_init(xfull_bar(s), 1);
      mbar_init(xempty_bar(s), 1);
    }
    for (int s = 0; s < D_Q_MAX; ++s) {
      mbar_init(qfull_bar(s), 1);
      mbar_init(qempty_bar(s), D_CONV_WARPS);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), D_EPI_WARPS);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    stored_cnt[0] = stored_cnt[1] = 0u;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&maps.wa0);
    tma_prefetch_desc(&maps.wa1);
    tma_prefetch_desc(&maps.xa0);
    tma_prefetch_desc(&maps.xa1);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), args.tmem_cols);
    tmem_relinquish();
  }
  pdl_wait();   // offsets, the token rows and the chunk counters come from earlier launches
  for (int i = threadIdx.x; i <= G; i += THREADS) seg[i] = args.offsets ? args.offsets[i] : 0;
  __syncthreads();
  if (warp == 2) {
    // per group: token chunks, and prefixes over the groups of the chunks
    // and of both phases' tiles (one lane per run of groups, then a warp scan)
    const int cw0 = glu ? DM : 2 * DM;   // output columns per phase-0 tile
    const int nwb0 = (args.F + cw0 - 1) / cw0, nwb0s = (args.Fs + cw0 - 1) / cw0;
    const int nwb1 = (args.H + 2 * DM - 1) / (2 * DM);
    const int per = (NG + 31) / 32;
    const int g0 = lane * per;
    int c_loc = 0, t0_loc = 0, t1_loc = 0;
    for (int g = g0; g < g0 + per && g < NG; ++g) {
      const int rows = g == G ? args.shared_rows : seg[g + 1] - seg[g];
      const int c = rows > 0 ? (rows + NT - 1) / NT : 0;
      nch[g] = c;
      c_loc += c;
      t0_loc += c * (g == G ? nwb0s : nwb0);
      t1_loc += c * nwb1;
    }
    int ci = c_loc, ti0 = t0_loc, ti1 = t1_loc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a = __shfl_up_sync(0xffffffffu, ci, o);
      const int b = __shfl_up_sync(0xffffffffu, ti0, o);
      const int c = __shfl_up_sync(0xffffffffu, ti1, o);
      if (lane >= o) { ci += a; ti0 += b; ti1 += c; }
    }
    int rc = ci - c_loc, r0 = ti0 - t0_loc, r1 = ti1 - t1_loc;
    for (int g = g0; g < g0 + per && g < NG; ++g) {
      cpre[g] = rc;
      tp0[g] = r0;
      tp1[g] = r1;
      rc += nch[g];
      r0 += nch[g] * (g == G ? nwb0s : nwb0);
      r1 += nch[g] * nwb1;
    }
    if (lane == 31) {
      cpre[NG] = ci;
      tp0[NG] = ti0;
      tp1[NG] = ti1;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int tiles0 = tp0[NG], total = tiles0 + tp1[NG];
  const int cw0 = glu ? DM : 2 * DM;
  const int nwb0 = (args.F + cw0 - 1) / cw0, nwb0s = (args.Fs + cw0 - 1) / cw0;
  long long x_issued = 0, w_issued = 0, q_issued = 0;

  if (warp == 0) {
    // ------------------------------------------------------------ token producer
    // (with skip_producer set nothing is issued: the consumers' bounded waits
    // run out and the abort path drains nothing)
    if (lane == 0 && !args.skip_producer) {
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      DCursor cur;
      for (int tile = unit; tile < total && ok; tile += units) {
        int wb, tc;
        cur.locate(tile, tiles0, tp0, tp1, nch, wb, tc);
        const int ph = cur.phase, g = cur.g;
        const DTileView v = d_view(args, seg, ph, g, wb, tc, NT);
        const CUtensorMap* mX = v.shared ? (ph ? &maps.xs1 : &maps.xs0) : (ph ? &maps.xa1 : &maps.xa0);
        const int nb = (v.n_valid + DBOX - 1) / DBOX;
        const uint32_t tx = (uint32_t)nb * DBOX * DK * 2;
        const int nkb = (v.K + DK - 1) / DK;
        if (ph == 1) {
          // the Hid rows of this chunk come from phase-0 tiles: wait until
          // each of them has stored and released its part
          const int target = v.shared ? nwb0s : nwb0;
          const int* cnt = args.rows_done + cpre[g] + tc;
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
          fence_proxy_async_global();   // the TMA reads below see those plain stores
        }
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait_bounded(xempty_bar(stage), phase ^ 1u, abort_flag, status)) { ok = false; break; }
          mbar_arrive_expect_tx(xfull_bar(stage), tx);
          for (int b = 0; b < nb; ++b)
            tma_load_2d(sX + stage * x_stage + b * DBOX * DK * 2, mX, xfull_bar(stage), kb * DK,
                        v.row0 + b * DBOX);
          ++x_issued;
          if (++stage == (uint32_t)XST) { stage = 0; phase ^= 1u; }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t ws = 0, wph = 0, xs = 0, xph = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      DCursor cur;
      for (int tile = unit; tile < total && ok; tile += units) {
        int wb, tc;
        cur.locate(tile, tiles0, tp0, tp1, nch, wb, tc);
        const DTileView v = d_view(args, seg, cur.phase, cur.g, wb, tc, NT);
        const int n16 = (v.n_valid + 15) / 16 * 16;
        const uint32_t idesc = idesc_bf16_f32(DM, n16);
        const int nkb = (v.K + DK - 1) / DK;
        if (!mbar_wait_bounded(tempty_bar(acc), acc_phase ^ 1u, abort_flag, status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * acc_cols;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait_bounded(wfull_bar(ws), wph, abort_flag, status) ||
              !mbar_wait_bounded(xfull_bar(xs), xph, abort_flag, status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = sdesc_kmajor_sw128(sW + ws * a_stage);
          const uint64_t bdesc = sdesc_kmajor_sw128(sX + xs * x_stage);
#pragma unroll
          for (int kk = 0; kk < DK / 16; ++kk) {
            const uint32_t accum = (kb | kk) != 0 ? 1u : 0u;
            // half 0 (weight rows 0-127 / gate rows) into columns [0, NT),
            // half 1 (rows 128-255 / up rows) into [NT, 2 NT)
            const uint64_t udesc = sdesc_kmajor_sw128(sW + ws * a_stage + D_A_BYTES);
            umma_bf16(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, accum);
            umma_bf16(d_tmem + NT, udesc + 2 * kk, bdesc + 2 * kk, idesc, accum);
          }
          umma_commit(wempty_bar(ws));
          umma_commit(xempty_bar(xs));
          if (++ws == (uint32_t)WST) { ws = 0; wph ^= 1u; }
          if (++xs == (uint32_t)XST) { xs = 0; xph ^= 1u; }
        }
        if (!ok) break;
        umma_commit(tfull_bar(acc));
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
    }
    __syncwarp();
  } else if (!FP8 && warp == WW0) {
    // ------------------------------------------------------------ weight producer
    // independent of the phase-1 hand-over, so the weight copies of the
    // next tiles stream in while the token producer waits for Hid rows
    if (lane == 0 && !args.skip_producer) {
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      DCursor cur;
      for (int tile = unit; tile < total && ok; tile += units) {
        int wb, tc;
        cur.locate(tile, tiles0, tp0, tp1, nch, wb, tc);
        const int ph = cur.phase;
        const DTileView v = d_view(args, seg, ph, cur.g, wb, tc, NT);
        const CUtensorMap* mW = v.shared ? (ph ? &maps.ws1 : &maps.ws0) : (ph ? &maps.wa1 : &maps.wa0);
        const bool tglu = glu && ph == 0;
        const int nkb = (v.K + DK - 1) / DK;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait_bounded(wempty_bar(stage), phase ^ 1u, abort_flag, status)) { ok = false; break; }
          mbar_arrive_expect_tx(wfull_bar(stage), (uint32_t)a_stage);
          // 256 consecutive weight rows in one copy (the map's box), or
          // SwiGLU's gate and up rows in two 128-row copies
          tma_load_2d(sW + stage * a_stage, mW, wfull_bar(stage), kb * DK, v.w_row);
          if (tglu) tma_load_2d(sW + stage * a_stage + D_A_BYTES, mW, wfull_bar(stage), kb * DK, v.w_row_up);
          ++w_issued;
          if (++stage == (uint32_t)WST) { stage = 0; phase ^= 1u; }
        }
      }
    }
    __syncwarp();
  } else if (FP8 && warp >= WW0) {
    // ------------------------------------------------------------ E4M3 -> bf16
    // The converter warps copy the E4M3 weight rows themselves (lane 0 of
    // the first one issues the copies, QST slots of two k-blocks ahead: the
    // bytes in flight from memory) and widen each k-block's [128][64] codes
    // (gate and up: [256][64]) into the bf16 weight tile of the ring slot
    // the MMA reads.
    const int cw = warp - WW0;
    const bool issuer = cw == 0 && lane == 0;
    DCursor lcur;
    int l_tile = unit, l_kq = 0, l_nkq = 0, l_row = 0, l_row_up = 0;
    bool l_glu = false, l_shared = false;
    int l_ph = 0;
    auto l_locate = [&]() {
      int wb, tc;
      lcur.locate(l_tile, tiles0, tp0, tp1, nch, wb, tc);
      l_ph = lcur.phase;
      const DTileView v = d_view(args, seg, l_ph, lcur.g, wb, tc, NT);
      l_nkq = ((v.K + DK - 1) / DK + 1) / 2;
      l_row = v.w_row;
      l_row_up = v.w_row_up;
      l_glu = glu && l_ph == 0;
      l_shared = v.shared;
    };
    auto issue = [&](int slot) {
      const uint32_t dq = sQ + slot * qslot;
      const CUtensorMap* m = l_shared ? (l_ph ? &maps.ws1 : &maps.ws0) : (l_ph ? &maps.wa1 : &maps.wa0);
      mbar_arrive_expect_tx(qfull_bar(slot), (uint32_t)qslot);
      tma_load_2d(dq, m, qfull_bar(slot), l_kq * 2 * DK, l_row);
      if (l_glu) tma_load_2d(dq + D_Q_BYTES, m, qfull_bar(slot), l_kq * 2 * DK, l_row_up);
      ++q_issued;
      if (++l_kq == l_nkq) {
        l_kq = 0;
        l_tile += units;
        if (l_tile < total) l_locate();
      }
    };
    if (issuer && !args.skip_producer && l_tile < total) {
      l_locate();
      for (int s2 = 0; s2 < QST && l_tile < total; ++s2) issue(s2);
    }
    uint32_t qs = 0, qph = 0, stage = 0, phase = 0;
    bool ok = true;
    DCursor cur;
    for (int tile = unit; tile < total && ok; tile += units) {
      int wb, tc;
      cur.locate(tile, tiles0, tp0, tp1, nch, wb, tc);
      const DTileView v = d_view(args, seg, cur.phase, cur.g, wb, tc, NT);
      const int nkb = (v.K + DK - 1) / DK;
      for (int kb = 0; kb < nkb; ++kb) {
        bool got = (kb & 1) ? true : mbar_wait_bounded(qfull_bar(qs), qph, abort_flag, status);
        if (got) got = mbar_wait_bounded(wempty_bar(stage), phase ^ 1u, abort_flag, status);
        if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
        const int h4 = (kb & 1) * 4;   // first 16-byte chunk of this k-block in a code row
        for (int half = 0; half < 2; ++half) {
          const uint8_t* q = smem + (sQ - sW) + qs * qslot + half * D_Q_BYTES;
          uint8_t* b = smem + stage * a_stage + half * D_A_BYTES;
#pragma unroll 2
          for (int g8 = cw; g8 < DM / 8; g8 += D_CONV_WARPS) widen_e4m3_rows8(q, b, g8, h4, lane);
        }
        fence_proxy_async_shared();   // the tensor cores read what the threads wrote
        __syncwarp();
        const bool slot_done = (kb & 1) || kb == nkb - 1;
        if (lane == 0) {
          if (slot_done) mbar_arrive(qempty_bar(qs));
          mbar_arrive(wfull_bar(stage));
        }
        if (++stage == (uint32_t)WST) { stage = 0; phase ^= 1u; }
        if (!slot_done) continue;
        if (cw == 0) {
          int refill_ok = 1;
          if (issuer && !args.skip_producer && l_tile < total) {
            if (mbar_wait_bounded(qempty_bar(qs), qph, abort_flag, status)) issue((int)qs);
            else refill_ok = 0;
          }
          if (!__shfl_sync(0xffffffffu, refill_ok, 0)) { ok = false; break; }
        }
        if (++qs == (uint32_t)QST) { qs = 0; qph ^= 1u; }
      }
    }
  } else if (warp >= 2 && warp < 2 + D_EPI_WARPS) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                       // TMEM lane quarter
    const int ew = warp - 2;
    const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
    uint16_t* tb = tbuf + ew * 16 * 32;            // [16][32] bf16: 16 tokens x this warp's rows
    float* wj = wv + ew * D_NT_MAX;                // [NT] gate weight of each token column
    uint32_t acc = 0, acc_phase = 0;
    DCursor cur;
    for (int tile = unit; tile < total; tile += units) {
      int wb, tc;
      cur.locate(tile, tiles0, tp0, tp1, nch, wb, tc);
      const int ph = cur.phase, g = cur.g;
      const DTileView v = d_view(args, seg, ph, g, wb, tc, NT);
      const bool tglu = glu && ph == 0;
      const int mode = ph ? EPI_SCALE : args.mode0;
      // per-row constants of this thread's two weight rows (half 0 and half
      // 1: rows q*32 + lane of each, or for SwiGLU the gate and up rows of
      // one output column): bias and E4M3 row scale
      const __nv_bfloat16* bias = v.shared ? (ph ? args.b2s : args.b1s) : (ph ? args.b2 : args.b1);
      const float* scale = v.shared ? (ph ? args.s2s : args.s1s) : (ph ? args.s2 : args.s1);
      const int wrows = tglu ? 2 * v.n_out : v.n_out;
      const int64_t rbase = v.shared ? 0 : (int64_t)g * wrows;
      float bh[2] = {0.0f, 0.0f}, sh[2] = {1.0f, 1.0f};
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int c = tglu ? v.col0 + q * 32 + lane : v.col0 + h * DM + q * 32 + lane;
        const int64_t r = tglu ? rbase + h * v.n_out + c : rbase + c;
        if (c < v.n_out) {
          if (bias) bh[h] = __bfloat162float(bias[r]);
          if (FP8 && scale) sh[h] = scale[r];
        }
      }
      if (ph == 1) {
        for (int j = lane; j < v.n_valid; j += 32)
          wj[j] = (v.shared || args.topk_w == nullptr) ? 1.0f : args.topk_w[args.perm[v.row0 + j]];
        __syncwarp();
      }
      int ok = 1;
      if (lane == 0) ok = mbar_wait_bounded(tfull_bar(acc), acc_phase, abort_flag, status) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + lane_addr + acc * acc_cols;
      const int n16 = (v.n_valid + 15) / 16 * 16;
      __nv_bfloat16* out = v.shared ? (ph ? args.out1s : args.out0s) : (ph ? args.out1 : args.out0);
      const int ld = v.n_out;
      // SwiGLU combines the halves into one set of 32 output columns; other
      // tiles store each half's 32 columns
      for (int h = 0; h < (tglu ? 1 : 2); ++h) {
        const int colw = v.col0 + h * DM + q * 32;   // this warp's first output column
        for (int c = 0; c < n16; c += 16) {
          uint32_t r[16], ru[16];
          tmem_ld_32x32b_x16(taddr + h * NT + c, r);
          if (tglu) tmem_ld_32x32b_x16(taddr + NT + c, ru);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int j = c + i;
            const float z = __uint_as_float(r[i]) * sh[h] + bh[h];
            float o;
            if (mode == EPI_GELU) o = gelu_erf(z);
            else if (mode == EPI_SILU) o = silu_f(z);
            else if (mode == EPI_SWIGLU) o = silu_f(z) * (__uint_as_float(ru[i]) * sh[1] + bh[1]);
            else o = (j < v.n_valid ? wj[j] : 0.0f) * z;
            tb[i * 32 + lane] = __bfloat16_as_ushort(__float2bfloat16_rn(o));
          }
          __syncwarp();
          // 16 token rows of 32 consecutive output columns: 16-byte stores
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const int i = (lane >> 2) + 8 * h2, c8 = (lane & 3) * 8;
            if (c + i < v.n_valid && colw + c8 < v.n_out)
              *reinterpret_cast<uint4*>(out + (int64_t)(v.row0 + c + i) * ld + colw + c8) =
                  *reinterpret_cast<const uint4*>(tb + i * 32 + c8);
          }
          __syncwarp();
        }
      }
      if (ph == 0) {
        // the last epilogue warp of the tile releases the chunk's counter
        if (lane == 0 && atom_add_acqrel_cta(&stored_cnt[acc], 1u) == D_EPI_WARPS - 1) {
          stored_cnt[acc] = 0u;
          fence_proxy_async_global();
          red_release_gpu_add(args.rows_done + cpre[g] + tc, 1);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(acc));
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  // ---- teardown
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // let every copy still in flight land before shared memory goes away
    if (warp == 0 && lane == 0) {
      const long long first = x_issued > XST ? x_issued - XST : 0;
      for (long long j = first; j < x_issued; ++j)
        d_wait_drain(xfull_bar((int)(j % XST)), (uint32_t)((j / XST) & 1));
    }
    if (!FP8 && warp == WW0 && lane == 0) {
      const long long first = w_issued > WST ? w_issued - WST : 0;
      for (long long j = first; j < w_issued; ++j)
        d_wait_drain(wfull_bar((int)(j % WST)), (uint32_t)((j / WST) & 1));
    }
    if (FP8 && warp == WW0 && lane == 0) {
      const long long first = q_issued > QST ? q_issued - QST : 0;
      for (long long j = first; j < q_issued; ++j)
        d_wait_drain(qfull_bar((int)(j % QST)), (uint32_t)((j / QST) & 1));
    }
    if (warp == 1 && lane == 0) {
      umma_commit(drain_bar);
      d_wait_drain(drain_bar, 0);
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

int decode_token_tile(int64_t group_rows_max) {
  int64_t nt = (group_rows_max + 15) / 16 * 16;
  if (nt < 16) nt = 16;
  if (nt > D_NT_MAX) nt = D_NT_MAX;
  return (int)nt;
}

cudaError_t make_decode_plan(DecodePlan* plan, const DecodeArgs& args_in, const DecodeTensors& t,
                             bool fp8, int64_t group_rows_max, int num_sms) {
  DecodeArgs a = args_in;
  const bool glu = a.mode0 == EPI_SWIGLU;
  a.nt = decode_token_tile(group_rows_max);
  const int NT = a.nt;
  const int acc_cols = 2 * NT;
  int cols = 32;
  while (cols < 2 * acc_cols) cols <<= 1;
  if (cols > 512) return cudaErrorInvalidValue;
  a.tmem_cols = cols;
  const bool has_routed = t.R > 0;
  const bool has_shared = a.shared_rows > 0;
  if (!has_routed && !has_shared) return cudaErrorInvalidValue;
  const int w1r = glu ? 2 * a.F : a.F, w1rs = glu ? 2 * a.Fs : a.Fs;
  DecodeMaps& m = plan->maps;
  // weight copies: 256 consecutive rows (both halves of a tile), or 128
  // rows for SwiGLU's first Linear (gate and up rows are copied apart)
  auto wmap = [&](CUtensorMap* mp, const void* base, int64_t rows, int64_t K, int box_rows) {
    return fp8 ? encode_tensor_map_u8(mp, base, rows, K, 2 * DK, box_rows)
               : encode_tensor_map_bf16(mp, base, rows, K, DK, box_rows);
  };
  const int box0 = glu ? DM : 2 * DM;
  auto xmap = [&](CUtensorMap* mp, const void* base, int64_t rows, int64_t K) {
    return encode_tensor_map_bf16(mp, base, rows, K, DK, DBOX);
  };
  bool ok = true;
  if (has_routed) {
    ok = ok && wmap(&m.wa0, t.W1, (int64_t)a.num_groups * w1r, a.H, box0);
    ok = ok && wmap(&m.wa1, t.W2, (int64_t)a.num_groups * a.H, a.F, 2 * DM);
    ok = ok && xmap(&m.xa0, t.xp, t.R, a.H);
    ok = ok && xmap(&m.xa1, t.hid, t.R, a.F);
  }
  if (has_shared) {
    ok = ok && wmap(&m.ws0, t.W1s, w1rs, a.H, box0);
    ok = ok && wmap(&m.ws1, t.W2s, a.H, a.Fs, 2 * DM);
    ok = ok && xmap(&m.xs0, t.x, a.shared_rows, a.H);
    ok = ok && xmap(&m.xs1, t.hid_s, a.shared_rows, a.Fs);
  }
  if (!ok) return cudaErrorInvalidValue;
  if (!has_routed) { m.wa0 = m.ws0; m.wa1 = m.ws1; m.xa0 = m.xs0; m.xa1 = m.xs1; }
  if (!has_shared) { m.ws0 = m.wa0; m.ws1 = m.wa1; m.xs0 = m.xa0; m.xs1 = m.xa1; }
  // shared memory: the token ring, the weight ring (bf16: as deep as fits;
  // E4M3: a short bf16 ring and as many code slots as fit, since those are
  // the bytes in flight from memory), the transpose buffers, gate weights,
  // barriers and group tables
  const int a_stage = 2 * D_A_BYTES;
  const int x_stage = NT * DK * 2;
  const int qslot = 2 * D_Q_BYTES;
  const int G = a.num_groups;
  const int n_bars = 2 * D_W_MAX + 2 * D_X_MAX + 2 * D_Q_MAX + 5;
  const int fixed = D_EPI_WARPS * 16 * 32 * 2 + D_EPI_WARPS * D_NT_MAX * 4 + n_bars * 8 + 16 +
                    5 * (G + 2) * 4;
  const int budget = 232448 - 1024 - fixed;
  const int x_stages = fp8 ? D_X_MAX / 2 : D_X_MAX;   // E4M3: room for more code slots
  int w_stages, q_stages = 0;
  if (fp8) {
    w_stages = 2;
    q_stages = (budget - x_stages * x_stage - w_stages * a_stage) / qslot;
    if (q_stages > D_Q_MAX) q_stages = D_Q_MAX;
    if (q_stages < 2) return cudaErrorInvalidValue;
  } else {
    w_stages = (budget - x_stages * x_stage) / a_stage;
    if (w_stages > D_W_MAX) w_stages = D_W_MAX;
    if (w_stages < 2) return cudaErrorInvalidValue;
  }
  a.w_stages = w_stages;
  a.x_stages = x_stages;
  a.q_stages = q_stages;
  plan->smem = w_stages * a_stage + q_stages * qslot + x_stages * x_stage + fixed;
  plan->args = a;
  plan->fp8 = fp8;
  plan->grid = num_sms;
  return cudaSuccess;
}

template <bool FP8>
static cudaError_t launch_decode_t(const DecodePlan& plan, cudaStream_t st) {
  using S = DShape<FP8>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(decode_ffn_kernel<FP8>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(plan.grid);
  cfg.blockDim = dim3(S::THREADS);
  cfg.dynamicSmemBytes = plan.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see pdl_wait()
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // phase-1 tiles wait for phase-0 tiles of other CTAs: every CTA must be
  // resident at once (one per SM with this much shared memory)
  int per_sm = 0, dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_ffn_kernel<FP8>, S::THREADS,
                                                    plan.smem) != cudaSuccess ||
      per_sm < 1)
    return cudaErrorInvalidConfiguration;
  if ((int)cfg.gridDim.x > sms * per_sm) cfg.gridDim.x = sms * per_sm;
  return cudaLaunchKernelEx(&cfg, decode_ffn_kernel<FP8>, plan.maps, plan.args);
}

cudaError_t launch_decode(const DecodePlan& plan, cudaStream_t st, LaunchTrace* tr) {
  trace_mark(tr, st);
  cudaError_t e = plan.fp8 ? launch_decode_t<true>(plan, st) : launch_decode_t<false>(plan, st);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace moe
