// Backward pass of tiled exact attention on sm_103a.
//
// Method ("What Ordinary Autograd Saves", section "Why this is
// FlashAttention's second idea"; "Backward Pass Implementation", section "The
// Recomputation Strategy"): only O and the row statistic L survive the
// forward; every score/probability tile is rebuilt on chip from Q, K and L.
// With D_i = rowsum(dO_i * O_i):
//     P = exp(scale * Q K^T - L),  dP = dO V^T,  dS = P * (dP - D),
//     dV += P^T dO,  dK += dS^T Q * scale,  dQ += dS K * scale.
//
// Three kernels:
//   fa_bwd_pre   D = rowsum(dO * O), L in log2 units (+inf on padding rows so
//                that their probabilities vanish), zero the fp32 dQ
//                accumulator and the split items' counters.  HBM-bound, a row
//                per group of dv / 8 lanes.
//   fa_bwd_main  one CTA per (batch, kv head, 128-key tile) -- without a causal
//                mask, a short last round of tiles runs as two CTAs per tile,
//                each over half of its query tiles, whose fp32 dK / dV meet in
//                the workspace -- K and V stay in
//                shared memory; the CTA walks the G query heads of its group
//                and the 128-row query tiles that can see its keys (causal:
//                from the diagonal on; with a sliding window of W keys, up to
//                the last row whose window still reaches the tile), keeping dK
//                and dV in TMEM for the whole walk and adding each tile's dQ
//                into the fp32 accumulator in global memory.
//   fa_dq_cast   dQ = bf16(scale * accumulator).  HBM-bound.
//
// fa_bwd_main roles (512 threads, four warpgroups):
//   warp 0      TMA: K, V once; then Q_t (+ the tile's L and D slices by 1-D
//               bulk copy) through a 2-deep ring and dO_t through one buffer
//               (3-deep and 2 buffers at d = dv = 64).
//   warp 1      tcgen05 issuer, per tile t:
//                 dP^T = V dO_t^T       -> TMEM [128,256)
//                 dV  += P^T dO_t       A = P^T from TMEM (bf16, written over S^T)
//                 S^T(t+1) = K Q_{t+1}^T -> TMEM [0,128)     (key rows = lanes)
//                 dK  += dS^T Q_t       A = dS^T from TMEM (bf16, written over dP^T)
//                 dQ_t = dS K           -> TMEM [128,128+d), or at d = 64 the free
//                                        columns after dK; A = the dS bytes in
//                                        shared memory read MN-major; B = K read MN-major
//               relying on in-order MMA execution, not on waits, wherever a
//               later MMA overwrites columns an earlier one reads.  At
//               d = dv = 64 it checks only P and dS per tile: one elementwise
//               thread and the dQ warps vouch for Q_{t+1}, dO_{t+1} and the
//               drained dQ columns.
//   warps 4..11 two elementwise warpgroups (thread = key row = TMEM lane; group
//               w owns query columns [64w, 64w+64)): P = exp2(S*scale*log2e - L2)
//               with masks -> TMEM; dS = P * (dP - D) -> shared memory (for the
//               dQ MMA) and, packed, into TMEM over dP^T (for the dK MMA).
//               Epilogue: dV and dK*scale -> bf16 -> TMA store.
//   warps 12..15 dQ warpgroup (thread = query row): each warp copies its 32
//               rows of dQ_t out of TMEM into registers, releases the columns,
//               then stages two 32-column chunks at a time in its own
//               128B-swizzled fp32 slots and adds each chunk into the fp32
//               accumulator in global memory with one TMA bulk reduce-add
//               (32 x 32 box); no cross-warp synchronisation.  At d = 128 it
//               takes registers from the producer / MMA warpgroup (setmaxnreg)
//               to hold a whole dQ row.
// TMEM columns: S^T/P^T [0,128), dP^T/dS^T/dQ [128,256), dV [256,256+dv), dK [256+dv, 256+dv+d);
// at d = 64 dQ moves to [256+dv+d, 256+dv+2d).
#include <cstdint>

#include "fa_internal.h"
#include "sm103_ptx.cuh"

using namespace fa_ptx;

namespace {

constexpr int BM = fa::kTile;  // query rows per tile
constexpr int BN = fa::kTile;  // keys per CTA
constexpr int kThreads = 512;
// Register split of fa_bwd_main at d = 128 (see the kernel): every thread
// starts with kRegsLaunch; the producer / MMA warpgroup drops to kRegsLow and
// the dQ warpgroup rises to kRegsHigh, the two elementwise warpgroups keep
// kRegsLaunch.
constexpr int kRegsLaunch = 65536 / kThreads;  // 128
constexpr int kRegsLow = 80;
constexpr int kRegsHigh = 2 * kRegsLaunch - kRegsLow;  // 176
template <int HD>
constexpr bool kSplitRegs = HD == 128;
static_assert(kRegsLow % 8 == 0 && kRegsHigh % 8 == 0 && kRegsHigh <= 256, "setmaxnreg operands");

// HD: head size of Q and K; HDV: head size of V, O and dO.
template <int HD, int HDV>
struct BwdCfg {
  // d = dv = 64 leaves shared memory for deeper Q and dO rings.  Loads then
  // land a tile earlier, and other roles can vouch for three of the MMA
  // thread's five checks per tile (see the kernel): one elementwise thread
  // checks Q(t+1) before it releases P(t) and dO(t+1) before it releases
  // dS(t), and the dQ warps arrive on ds_ready(t+1) once dQ(t) is drained.
  static constexpr bool VOUCH = HD == 64 && HDV == 64;
  static constexpr int NQ = VOUCH ? 3 : 2;   // Q tiles (with their L and D slices) in flight
  static constexpr int NDO = VOUCH ? 2 : 1;  // dO tiles in flight
  static constexpr int QK_TILE = 128 * HD * 2;   // one Q or K tile (bf16)
  static constexpr int VO_TILE = 128 * HDV * 2;  // one V or dO tile (bf16)
  static constexpr int DS_BYTES = BN * BM * 2;
  static constexpr int STG_SLOT = 32 * 32 * 4;  // one warp's 32 rows x 32 fp32 columns
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + QK_TILE;
  static constexpr int OFF_Q = OFF_V + VO_TILE;         // [NQ]
  static constexpr int OFF_DO = OFF_Q + NQ * QK_TILE;   // [NDO]
  static constexpr int OFF_DS = OFF_DO + NDO * VO_TILE;
  // Epilogue staging of dV and dK over the Q ring and the dO buffer (idle by then).
  static constexpr int OFF_DV_STAGE = OFF_Q;
  static constexpr int OFF_DK_STAGE = OFF_Q + (QK_TILE > VO_TILE ? QK_TILE : VO_TILE);
  static_assert(OFF_DK_STAGE + QK_TILE <= OFF_DS, "dV / dK staging fits in the Q ring and dO buffer");
  static constexpr int OFF_STG = OFF_DS + DS_BYTES;       // [4 warps][2] dQ staging slots
  static constexpr int OFF_LSE = OFF_STG + 8 * STG_SLOT;  // [NQ][128] fp32
  static constexpr int OFF_DELTA = OFF_LSE + NQ * 512;   // [NQ][128] fp32
  static constexpr int OFF_BAR = OFF_DELTA + NQ * 512;
  static constexpr int NBAR = 24;
  static_assert(1 + 2 * NQ + 2 * NDO + 8 <= NBAR, "barrier slots");
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 16;
  static_assert(SMEM <= 232448, "shared memory budget");
};

// Epilogue of one fp32 accumulator of W columns in TMEM (dV or dK): this
// thread's key row r, the warpgroup's half of the columns (wg), times `mul`,
// as bf16 into a 128-row, 128B-swizzled staging tile for the TMA store.
// `have` is false when the CTA saw no query tile: the rows are zero.
// `add` (optional): the same row's partial sums from the other half of a
// split item, this warpgroup's columns, added before the scaling.
template <int W>
__device__ __forceinline__ void stage_rows_bf16(uint32_t src, uint8_t* stage, int r, int wg, float mul, bool have,
                                                const float* add = nullptr) {
  constexpr int HALF = W / 2;
#pragma unroll
  for (int c = 0; c < HALF / 32; ++c) {
    uint32_t v[32];
    if (have) {
      tmem_ld32(src + c * 32, v);
      tmem_wait_ld();
    } else {
#pragma unroll
      for (int e = 0; e < 32; ++e) v[e] = 0u;
    }
    if (add) {
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 a = __ldcg(reinterpret_cast<const float4*>(add + c * 32) + q);
        v[4 * q] = __float_as_uint(__uint_as_float(v[4 * q]) + a.x);
        v[4 * q + 1] = __float_as_uint(__uint_as_float(v[4 * q + 1]) + a.y);
        v[4 * q + 2] = __float_as_uint(__uint_as_float(v[4 * q + 2]) + a.z);
        v[4 * q + 3] = __float_as_uint(__uint_as_float(v[4 * q + 3]) + a.w);
      }
    }
    const int col0 = wg * HALF + c * 32;  // first column of this chunk
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        w[e] = pack_bf16x2(__uint_as_float(v[8 * q + 2 * e]) * mul, __uint_as_float(v[8 * q + 2 * e + 1]) * mul);
      const int col = col0 + 8 * q;
      st_shared_v4(smem_u32(stage + (col >> 6) * (BN * 128) + sw128_offset(r, (col & 63) >> 3)), w[0], w[1], w[2],
                   w[3]);
    }
  }
}

// This row's fp32 sums of one accumulator (W columns in TMEM at src, this
// warpgroup's half of them) into a split item's partial area (zeros if the
// half saw no tile).
template <int W>
__device__ __forceinline__ void write_partial(uint32_t src, float* dst, bool have) {
  constexpr int HALF = W / 2;
#pragma unroll
  for (int c = 0; c < HALF / 32; ++c) {
    uint32_t v[32];
    if (have) {
      tmem_ld32(src + c * 32, v);
      tmem_wait_ld();
    } else {
#pragma unroll
      for (int e = 0; e < 32; ++e) v[e] = 0u;
    }
#pragma unroll
    for (int q = 0; q < 8; ++q)
      __stcg(reinterpret_cast<float4*>(dst + c * 32) + q,
             make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]), __uint_as_float(v[4 * q + 2]),
                         __uint_as_float(v[4 * q + 3])));
  }
}

struct BwdParams {
  const float* lse2;
  const float* delta;
  int* status;
  int Hq, Hkv, G, Tq, Tk, causal_off, q_tiles, kv_tiles;
  int sb_groups;  // (batch, kv head) groups per super-batch of the grid order; divides B * Hkv
  int window;     // causal sliding window in keys, 0 = none
  long long Tq_pad;
  float scale_log2, scale;
  int test_withhold_do;  // test build only: never issue the dO loads (the CTA's waits then time out)
  // Split items: the last n_split items of the grid order run as two CTAs
  // each (CTAs n_whole + 2 s and n_whole + 2 s + 1 for item n_whole + s),
  // each walking half of the item's query tiles; the halves' fp32 dK / dV
  // meet in `part`, and whichever half finishes second adds the other's and
  // stores them (split_counters, zeroed by fa_bwd_pre, tell them apart).
  int n_whole, n_split;
  float* part;                    // [n_split][2 halves][128 key rows][d + dv]
  unsigned int* split_counters;   // [n_split]
};

// WINDOW (causal only): the sliding-window terms are compiled in only where
// a window is set, so the plain causal and full masks keep their lean code.
template <int HD, int HDV, bool CAUSAL, bool WINDOW>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_main(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                const __grid_constant__ CUtensorMap tmdK, const __grid_constant__ CUtensorMap tmdV,
                const __grid_constant__ CUtensorMap tmAcc, const BwdParams p) {
  using C = BwdCfg<HD, HDV>;
  extern __shared__ __align__(1024) uint8_t smem[];
  constexpr int NQ = C::NQ, NDO = C::NDO;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* kv_full = bars + 0;
  uint64_t* q_full = bars + 1;         // [NQ]
  uint64_t* q_empty = q_full + NQ;     // [NQ]
  uint64_t* do_full = q_empty + NQ;    // [NDO]
  uint64_t* do_empty = do_full + NDO;  // [NDO]
  uint64_t* s_full = do_empty + NDO;
  uint64_t* dp_full = s_full + 1;
  uint64_t* p_ready = s_full + 2;
  uint64_t* ds_ready = s_full + 3;
  uint64_t* dq_full = s_full + 4;
  uint64_t* dq_empty = s_full + 5;
  uint64_t* acc_done = s_full + 6;
  uint64_t* drain = s_full + 7;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile unsigned int* split_seen = reinterpret_cast<volatile unsigned int*>(tmem_slot + 2);  // halves counted before

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // One linear grid in super-batches of sb_groups (batch, kv head) groups;
  // within a super-batch the key tile is slowest: its groups' tile 0 runs
  // first, then tile 1, ...  Causal low key tiles see the most query rows, so
  // each super-batch runs heaviest-first and the next one's heavy CTAs fill
  // the SMs its light ones free, which keeps the tail short.  Only a few
  // groups' Q, dO and fp32 dQ accumulator are live at a time, so they stay in
  // L2.  (One group at a time keeps even less live, but its late heavy CTAs
  // make the causal step ~12% longer.)
  // Split items exist only without a causal mask (equal-work items); the
  // causal instances compile none of their code.
  constexpr bool SPLIT = !CAUSAL;
  int item = blockIdx.x, split = -1, half = 0;
  if (SPLIT && item >= p.n_whole) {
    split = (item - p.n_whole) >> 1;
    half = (item - p.n_whole) & 1;
    item = p.n_whole + split;
  }
  const int per_sb = p.sb_groups * p.kv_tiles;
  const int sb = item / per_sb;
  const int in_sb = item - sb * per_sb;
  const int n = in_sb / p.sb_groups;  // key tile
  const int bkv = sb * p.sb_groups + (in_sb - n * p.sb_groups);
  const int b = bkv / p.Hkv, hk = bkv - b * p.Hkv;
  const int k0 = n * BN;

  int m_begin = 0, m_end = p.q_tiles;
  if (CAUSAL) {
    const int first_row = k0 - p.causal_off;  // first query row that sees key k0
    m_begin = first_row <= 0 ? 0 : min(p.q_tiles, first_row / BM);
    if (WINDOW) {
      // last query row whose window reaches the tile's last key
      const long long last_row = (long long)k0 + BN - 1 - p.causal_off + p.window - 1;
      m_end = last_row < 0 ? 0 : (int)min((long long)p.q_tiles, last_row / BM + 1);
    }
  }
  const int n_m = max(0, m_end - m_begin);
  const int T_item = p.G * n_m;  // the item's tiles
  // this CTA's tiles: [t0, t0 + T) of the item's
  const int t0 = split >= 0 && half ? T_item / 2 : 0;
  const int T = split >= 0 ? (half ? T_item - T_item / 2 : T_item / 2) : T_item;

  if (threadIdx.x == 0) {
    *abort_flag = (smem_u32(smem) & 1023u) ? 1 : 0;
    mbar_init(kv_full, 1);
    for (int s = 0; s < NQ; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
    }
    for (int s = 0; s < NDO; ++s) {
      mbar_init(&do_full[s], 1);
      mbar_init(&do_empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    mbar_init(p_ready, 256);
    // with VOUCH the dQ warps arrive too, once the previous dQ tile is drained
    mbar_init(ds_ready, C::VOUCH ? 384 : 256);
    mbar_init(dq_full, 1);
    mbar_init(dq_empty, 128);
    mbar_init(acc_done, 1);
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool run = (*abort_flag == 0) && T > 0;
  // d = 128: the dQ warpgroup holds a whole 128-column dQ row in registers so
  // that it can release dQ's TMEM columns before staging it; it takes the
  // registers the producer / MMA warpgroup does not need (setmaxnreg at the
  // top of both roles).  The launch gives every thread kRegsLaunch registers
  // (the launcher checks this), and the shares add up to that total:
  // kRegsLow + kRegsHigh = 2 * kRegsLaunch.
  const uint32_t T_S = tmem, T_DP = tmem + 128, T_DV = tmem + 256, T_DK = tmem + 256 + HDV;
  // dQ shares dP^T's columns unless there is room for columns of its own
  // (d = 64: dK ends at 384 or 448); then dP^T(t+1) need not wait for dQ(t)'s
  // drain, only dQ(t+1) does.
  constexpr bool kOwnDQ = 256 + HDV + 2 * HD <= 512;
  const uint32_t T_DQ = kOwnDQ ? T_DK + HD : T_DP;

  if (warp < 4) {
    if (kSplitRegs<HD>) setmaxnreg_dec<kRegsLow>();
    if (warp == 0 && lane == 0 && run) {
      // ---------------------------------------------------------- producer
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmdO);
      mbar_arrive_expect_tx(kv_full, C::QK_TILE + C::VO_TILE);
#pragma unroll
      for (int cb = 0; cb < HD / 64; ++cb) tma_load_3d(smem + C::OFF_K + cb * BN * 128, &tmK, kv_full, cb * 64, k0, bkv);
#pragma unroll
      for (int cb = 0; cb < HDV / 64; ++cb) tma_load_3d(smem + C::OFF_V + cb * BN * 128, &tmV, kv_full, cb * 64, k0, bkv);
      int last_q[NQ], last_do[NDO];
      for (int s = 0; s < NQ; ++s) last_q[s] = -1;
      for (int s = 0; s < NDO; ++s) last_do[s] = -1;
      for (int t = 0; t < T; ++t) {
        const int st = t % NQ, u = t / NQ;
        const int g = (t0 + t) / n_m, m = m_begin + ((t0 + t) - g * n_m);
        const int bh = b * p.Hq + hk * p.G + g;
        if (!mbar_wait(&q_empty[st], (u & 1) ^ 1, abort_flag)) break;
        mbar_arrive_expect_tx(&q_full[st], C::QK_TILE + 1024);
#pragma unroll
        for (int cb = 0; cb < HD / 64; ++cb)
          tma_load_3d(smem + C::OFF_Q + st * C::QK_TILE + cb * BM * 128, &tmQ, &q_full[st], cb * 64, m * BM, bh);
        const long long row0 = (long long)bh * p.Tq_pad + (long long)m * BM;
        bulk_load(smem + C::OFF_LSE + st * 512, p.lse2 + row0, 512, &q_full[st]);
        bulk_load(smem + C::OFF_DELTA + st * 512, p.delta + row0, 512, &q_full[st]);
        last_q[st] = u;
        // A dO slot is refilled only once dV of the tile before is done: pull
        // the tile into L2 now so that its load later does not stall the dP MMA.
#pragma unroll
        for (int cb = 0; cb < HDV / 64; ++cb) tma_prefetch_l2_3d(&tmdO, cb * 64, m * BM, bh);
        const int so = t % NDO, uo = t / NDO;
        if (!mbar_wait(&do_empty[so], (uo & 1) ^ 1, abort_flag)) break;
#ifdef FA_TEST_HOOKS
        if (p.test_withhold_do) continue;
#endif
        mbar_arrive_expect_tx(&do_full[so], C::VO_TILE);
#pragma unroll
        for (int cb = 0; cb < HDV / 64; ++cb)
          tma_load_3d(smem + C::OFF_DO + so * C::VO_TILE + cb * BM * 128, &tmdO, &do_full[so], cb * 64, m * BM, bh);
        last_do[so] = uo;
      }
      mbar_wait_bounded(kv_full, 0);
      for (int s = 0; s < NQ; ++s)
        if (last_q[s] >= 0) mbar_wait_bounded(&q_full[s], last_q[s] & 1);
      for (int s = 0; s < NDO; ++s)
        if (last_do[s] >= 0) mbar_wait_bounded(&do_full[s], last_do[s] & 1);
    } else if (warp == 1 && lane == 0 && run) {
      // ---------------------------------------------------------- MMA issuer
      constexpr uint32_t id_sdp = idesc_bf16(BN, BM, 0, 0);  // S^T, dP^T: M = keys, N = queries
      constexpr uint32_t id_dv = idesc_bf16(BN, HDV, 0, 1);  // dV: M = keys, N = dv, B MN-major
      constexpr uint32_t id_dk = idesc_bf16(BN, HD, 0, 1);   // dK: M = keys, N = d, B MN-major
      constexpr uint32_t id_q = idesc_bf16(BM, HD, 1, 1);    // dQ: M = queries (A MN-major), N = d
      const uint32_t k_base = smem_u32(smem + C::OFF_K), v_base = smem_u32(smem + C::OFF_V);
      const uint32_t ds_base = smem_u32(smem + C::OFF_DS);
      // S^T(t) = K Q_t^T into T_S
      auto mma_s = [&](int t) {
        const uint32_t q_base = smem_u32(smem + C::OFF_Q + (t % NQ) * C::QK_TILE);
#pragma unroll
        for (int k = 0; k < HD / 16; ++k)
          mma_ss(T_S, desc_kmajor(k_base + (k >> 2) * (BN * 128) + (k & 3) * 32),
                 desc_kmajor(q_base + (k >> 2) * (BM * 128) + (k & 3) * 32), id_sdp, k > 0 ? 1u : 0u);
        mma_commit(s_full);
      };
      // Issue order per tile t: dP^T(t), dV(t), S^T(t+1), dK(t), dQ(t).  S^T(t+1)
      // overwrites the P^T(t) columns dV(t) reads, and dQ(t) (d = 128) the dS^T(t)
      // columns dK(t) reads; one thread's MMAs execute in issue order, so both
      // have been read by then.  With S^T(t+1) right behind dV(t), the
      // elementwise warps go from tile t's dS phase straight to tile t+1's P
      // phase while dK(t), dQ(t) and dP^T(t+1) run.
      // With VOUCH the thread checks only p_ready(t) and ds_ready(t) per tile
      // (and dO(0)): those barriers also stand for Q(t+1) (before S^T(t+1)),
      // for dO(t+1) and for the drain of dQ(t) (before dQ(t+1) and dP^T(t+1)),
      // so dK(t), dQ(t) and dP^T(t+1) go out as one run of MMAs.
      bool ok = mbar_wait(kv_full, 0, abort_flag) && mbar_wait(&q_full[0], 0, abort_flag);
      if (ok) {
        tc_fence_after();
        mma_s(0);
      }
      for (int t = 0; ok && t < T; ++t) {
        const int st = t % NQ, so = t % NDO;
        const uint32_t q_base = smem_u32(smem + C::OFF_Q + st * C::QK_TILE);
        const uint32_t do_base = smem_u32(smem + C::OFF_DO + so * C::VO_TILE);
        if ((!C::VOUCH || t == 0) && !mbar_wait(&do_full[so], (t / NDO) & 1, abort_flag)) { ok = false; break; }
        // dP^T shares its TMEM columns with dQ (d = 128): the previous tile's dQ must be drained
        if (!kOwnDQ && t > 0 && !mbar_wait(dq_empty, (t - 1) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < HDV / 16; ++k)
          mma_ss(T_DP, desc_kmajor(v_base + (k >> 2) * (BN * 128) + (k & 3) * 32),
                 desc_kmajor(do_base + (k >> 2) * (BM * 128) + (k & 3) * 32), id_sdp, k > 0 ? 1u : 0u);
        mma_commit(dp_full);
        if (!mbar_wait(p_ready, t & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        // P^T lives in TMEM as packed bf16 over S^T: query columns [0,64) at TMEM
        // columns [0,32), query columns [64,128) at [64,96) (each elementwise
        // warpgroup overwrote its own half of S^T).
#pragma unroll
        for (int k = 0; k < BM / 16; ++k)
          mma_ts(T_DV, T_S + (k >> 2) * 64 + (k & 3) * 8, desc_mnmajor(do_base + k * 2048, BM * 128), id_dv,
                 (t > 0 || k > 0) ? 1u : 0u);
        mma_commit(&do_empty[so]);
        if (t + 1 < T) {
          if (!C::VOUCH) {
            if (!mbar_wait(&q_full[(t + 1) % NQ], ((t + 1) / NQ) & 1, abort_flag)) { ok = false; break; }
            tc_fence_after();
          }
          mma_s(t + 1);
        }
        // dS^T lives in TMEM as packed bf16 over dP^T, in the same column
        // pattern as P^T: query columns [0,64) at [128,160), [64,128) at
        // [192,224).  (dK waits for all of it: by the time S^T(t+1) is
        // queued the elementwise warps have finished both halves, and every
        // extra barrier check would leave the tensor pipe idle for a
        // shared-memory round trip.)
        if (!mbar_wait(ds_ready, t & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < BM / 16; ++k)
          mma_ts(T_DK, T_DP + (k >> 2) * 64 + (k & 3) * 8, desc_mnmajor(q_base + k * 2048, BM * 128), id_dk,
                 (t > 0 || k > 0) ? 1u : 0u);
        mma_commit(&q_empty[st]);
        if (kOwnDQ && !C::VOUCH && t > 0) {  // dQ(t-1) drained from its columns
          if (!mbar_wait(dq_empty, (t - 1) & 1, abort_flag)) { ok = false; break; }
          tc_fence_after();
        }
#pragma unroll
        for (int k = 0; k < BN / 16; ++k)
          mma_ss(T_DQ, desc_mnmajor(ds_base + k * 2048, BN * 128), desc_mnmajor(k_base + k * 2048, BN * 128), id_q,
                 k > 0 ? 1u : 0u);
        mma_commit(dq_full);
      }
      mma_commit(acc_done);
      mma_commit(drain);
      mbar_wait_bounded(drain, 0);
    }
  } else if (warp < 12) {
    // ------------------------------------------------------------ elementwise warpgroups
    const int wg = (warp - 4) >> 2;  // 0 or 1
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // TMEM lane = key row
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const int key = k0 + r;
    const bool key_valid = key < p.Tk;
    const float sl2 = p.scale_log2;
    bool ok = run;
    // With VOUCH one thread checks the next tile's Q before releasing P and
    // its dO before releasing dS, standing in for the MMA thread's checks.
    const bool voucher = C::VOUCH && warp == 4 && lane == 0;
    for (int t = 0; ok && t < T; ++t) {
      const int st = t % NQ, u = t / NQ;
      const int g = (t0 + t) / n_m, m = m_begin + ((t0 + t) - g * n_m);
      const int q0 = m * BM;
      const float* lse_s = reinterpret_cast<const float*>(smem + C::OFF_LSE + st * 512);
      const float* del_s = reinterpret_cast<const float*>(smem + C::OFF_DELTA + st * 512);
      // Each warp agrees on the outcome of the waits before its collective
      // TMEM loads and stores, so a timeout never splits a warp.
      bool got = mbar_wait(&q_full[st], u & 1, abort_flag) && mbar_wait(s_full, t & 1, abort_flag);
      if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
      tc_fence_after();
      // ---- P = exp2(S * scale * log2e - L2), masked; 32 query columns at a time.
      // The packed bf16 P of chunk c is stored over S columns this thread has
      // already read (each thread only touches its own TMEM lane); the fp32 P
      // stays in registers for dS.
      const bool need_mask = !key_valid || (CAUSAL && k0 + BN - 1 > q0 + p.causal_off) ||
                             (WINDOW && q0 + BM - 1 + p.causal_off - p.window + 1 > k0);
      // key row `key` is visible to query q0 + c iff vis_from <= c <= vis_to:
      // key <= q0 + c + off, and with a window also key > q0 + c + off - W
      const int vis_from = key_valid ? (CAUSAL ? key - p.causal_off - q0 : -0x40000000) : 0x40000000;
      const int vis_to = WINDOW ? key - p.causal_off - q0 + p.window - 1 : 0x40000000;
      const float4* lse4 = reinterpret_cast<const float4*>(lse_s + wg * 64);
      const uint64_t sl2x2 = f2_pack(sl2, sl2);
      float pr[64];
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        uint32_t sr[32];
        tmem_ld32(T_S + lane_base + wg * 64 + ch * 32, sr);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
          const float4 l4 = ld_shared_f4(lse4 + ((ch * 32 + c) >> 2));  // 16-byte broadcast: 4 columns
          const uint64_t x01 = f2_fma(f2_pack(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), sl2x2,
                                      f2_pack(-l4.x, -l4.y));
          const uint64_t x23 = f2_fma(f2_pack(__uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3])), sl2x2,
                                      f2_pack(-l4.z, -l4.w));
          float v0 = ex2(f2_lo(x01)), v1 = ex2(f2_hi(x01)), v2 = ex2(f2_lo(x23)), v3 = ex2(f2_hi(x23));
          if (need_mask) {
            const int qc = wg * 64 + ch * 32 + c;
            if (qc < vis_from || (WINDOW && qc > vis_to)) v0 = 0.f;
            if (qc + 1 < vis_from || (WINDOW && qc + 1 > vis_to)) v1 = 0.f;
            if (qc + 2 < vis_from || (WINDOW && qc + 2 > vis_to)) v2 = 0.f;
            if (qc + 3 < vis_from || (WINDOW && qc + 3 > vis_to)) v3 = 0.f;
          }
          pr[ch * 32 + c] = v0;
          pr[ch * 32 + c + 1] = v1;
          pr[ch * 32 + c + 2] = v2;
          pr[ch * 32 + c + 3] = v3;
          pk[c / 2] = pack_bf16x2(v0, v1);
          pk[c / 2 + 1] = pack_bf16x2(v2, v3);
        }
        tmem_st16(T_S + lane_base + wg * 64 + ch * 16, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      if (voucher && t + 1 < T && !mbar_wait(&q_full[(t + 1) % NQ], ((t + 1) / NQ) & 1, abort_flag)) ok = false;
      mbar_arrive(p_ready);
      if (C::VOUCH && !__all_sync(0xffffffffu, ok)) { ok = false; break; }  // the warp stops as one
      // ---- dS = P * (dP - D) -> shared memory (row = key, 128B-swizzled, query-contiguous)
      // dP^T is in TMEM.  The previous tile's dQ MMA, which reads dS from shared
      // memory, was issued before this tile's dP^T by the same thread, so the
      // dP^T commit covers it too.
      got = mbar_wait(dp_full, t & 1, abort_flag);
      if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
      tc_fence_after();
      uint8_t* ds_blk = smem + C::OFF_DS + wg * (BN * 128);
      const float4* del4 = reinterpret_cast<const float4*>(del_s + wg * 64);
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        uint32_t dr[32];
        tmem_ld32(T_DP + lane_base + wg * 64 + ch * 32, dr);
        tmem_wait_ld();
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; e += 2) {
            const int c = cc * 8 + 2 * e;  // column inside the chunk (4 per step)
            const float4 d4 = ld_shared_f4(del4 + ((ch * 32 + c) >> 2));
            const uint64_t g01 = f2_sub(f2_pack(__uint_as_float(dr[c]), __uint_as_float(dr[c + 1])), f2_pack(d4.x, d4.y));
            const uint64_t g23 = f2_sub(f2_pack(__uint_as_float(dr[c + 2]), __uint_as_float(dr[c + 3])), f2_pack(d4.z, d4.w));
            const uint64_t s01 = f2_mul(g01, f2_pack(pr[ch * 32 + c], pr[ch * 32 + c + 1]));
            const uint64_t s23 = f2_mul(g23, f2_pack(pr[ch * 32 + c + 2], pr[ch * 32 + c + 3]));
            w[e] = pack_bf16x2(f2_lo(s01), f2_hi(s01));
            w[e + 1] = pack_bf16x2(f2_lo(s23), f2_hi(s23));
          }
          st_shared_v4(smem_u32(ds_blk + sw128_offset(r, ch * 4 + cc)), w[0], w[1], w[2], w[3]);
          // packed dS^T of these 8 columns, for the dK MMA (A from TMEM), over
          // dP^T columns this thread has already read
          tmem_st4(T_DP + lane_base + wg * 64 + ch * 16 + cc * 4, w[0], w[1], w[2], w[3]);
        }
      }
      tmem_wait_st();
      fence_async_smem();
      tc_fence_before();
      if (voucher && t + 1 < T && !mbar_wait(&do_full[(t + 1) % NDO], ((t + 1) / NDO) & 1, abort_flag)) ok = false;
      mbar_arrive(ds_ready);
      if (C::VOUCH && !__all_sync(0xffffffffu, ok)) { ok = false; break; }
    }
    // ---- epilogue: dV, dK * scale -> bf16 -> shared (the Q ring, idle now) -> TMA store
    if (ok && T > 0) {
      if (!__all_sync(0xffffffffu, mbar_wait(acc_done, 0, abort_flag))) ok = false;
      tc_fence_after();
    }
    const bool mine = (T == 0 || ok) && *abort_flag == 0;
    if (named_bar_and(1, 256, mine)) {
      // A split item's halves: each writes its fp32 sums to the partial area
      // and counts itself in; the one that comes second adds the other's sums
      // to its own and stores the item's dV and dK.  Neither waits for the other.
      const float* other = nullptr;
      bool finish = true;
      if (split >= 0) {
        float* own = p.part + (((size_t)split * 2 + half) * BN + r) * (HD + HDV);
        write_partial<HDV>(T_DV + lane_base + wg * (HDV / 2), own + wg * (HDV / 2), T > 0);
        write_partial<HD>(T_DK + lane_base + wg * (HD / 2), own + HDV + wg * (HD / 2), T > 0);
        __threadfence();
        named_bar_sync(3, 256);
        if (warp == 4 && lane == 0) *split_seen = atomicAdd(&p.split_counters[split], 1u);
        named_bar_sync(3, 256);
        finish = *split_seen == 1u;
        if (finish) {
          __threadfence();
          other = p.part + (((size_t)split * 2 + (half ^ 1)) * BN + r) * (HD + HDV);
        }
      }
      if (!finish) goto epilogue_done;
      stage_rows_bf16<HDV>(T_DV + lane_base + wg * (HDV / 2), smem + C::OFF_DV_STAGE, r, wg, 1.f, T > 0,
                           other ? other + wg * (HDV / 2) : nullptr);
      stage_rows_bf16<HD>(T_DK + lane_base + wg * (HD / 2), smem + C::OFF_DK_STAGE, r, wg, p.scale, T > 0,
                          other ? other + HDV + wg * (HD / 2) : nullptr);
      fence_async_smem();
      named_bar_sync(2, 256);
      if (warp == 4 && lane == 0) {
        prefetch_tmap(&tmdV);
        prefetch_tmap(&tmdK);
#pragma unroll
        for (int cb = 0; cb < HDV / 64; ++cb)
          tma_store_3d(&tmdV, smem + C::OFF_DV_STAGE + cb * BN * 128, cb * 64, k0, bkv);
#pragma unroll
        for (int cb = 0; cb < HD / 64; ++cb)
          tma_store_3d(&tmdK, smem + C::OFF_DK_STAGE + cb * BN * 128, cb * 64, k0, bkv);
        bulk_commit();
        bulk_wait0();
      }
    }
  epilogue_done:;
  } else {
    // ------------------------------------------------------------ dQ warpgroup
    if (kSplitRegs<HD>) setmaxnreg_inc<kRegsHigh>();
    // Each warp drains its own 32 query rows (its TMEM lanes).  It copies all
    // of its rows of dQ_t out of TMEM first and releases the columns at once
    // (dP^T of the next tile waits for them at d = 128), then adds them into
    // the fp32 accumulator two 32-column chunks at a time: two 4 KB staging
    // slots per warp (32 rows x 32 fp32, 128B-swizzled), one 32x32 TMA
    // reduce-add per slot; only warp-local ordering is needed.
    const int quad = warp & 3;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const bool leader = (lane == 0);
    uint8_t* wslot = smem + C::OFF_STG + quad * (2 * C::STG_SLOT);
    constexpr int NCH = HD / 32;  // 32-column chunks per tile
    bool ok = run;
    // With VOUCH the drain is announced on ds_ready(t+1) (which the MMA thread
    // waits for before dQ(t+1) anyway); there is nothing to drain before dQ(0).
    if (C::VOUCH && ok) mbar_arrive(ds_ready);
    for (int t = 0; ok && t < T; ++t) {
      const int g = (t0 + t) / n_m, m = m_begin + ((t0 + t) - g * n_m);
      const int bh = b * p.Hq + hk * p.G + g;
      if (!__all_sync(0xffffffffu, mbar_wait(dq_full, t & 1, abort_flag))) { ok = false; break; }
      tc_fence_after();
      uint32_t v[NCH][32];
#pragma unroll
      for (int c = 0; c < NCH; ++c) tmem_ld32(T_DQ + lane_base + c * 32, v[c]);
      tmem_wait_ld();
      tc_fence_before();
      // all of dQ_t is out of TMEM: it may take dP_{t+1} (or dQ_{t+1})
      if (!C::VOUCH)
        mbar_arrive(dq_empty);
      else if (t + 1 < T)
        mbar_arrive(ds_ready);
#pragma unroll
      for (int c = 0; c < NCH; c += 2) {
        if (leader) bulk_wait_read0();  // both slots read by the previous reduce-adds
        __syncwarp();
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          st_shared_v4(smem_u32(wslot + sw128_offset(lane, q)), v[c][4 * q], v[c][4 * q + 1], v[c][4 * q + 2],
                       v[c][4 * q + 3]);
          st_shared_v4(smem_u32(wslot + C::STG_SLOT + sw128_offset(lane, q)), v[c + 1][4 * q], v[c + 1][4 * q + 1],
                       v[c + 1][4 * q + 2], v[c + 1][4 * q + 3]);
        }
        fence_async_smem();
        __syncwarp();
        if (leader) {
          tma_reduce_add_3d(&tmAcc, wslot, c * 32, m * BM + quad * 32, bh);
          tma_reduce_add_3d(&tmAcc, wslot + C::STG_SLOT, (c + 1) * 32, m * BM + quad * 32, bh);
          bulk_commit();
        }
      }
    }
    if (leader) bulk_wait0();  // every reduce-add has landed before the kernel ends
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicExch(p.status, DEV_TIMEOUT);
}

// D = rowsum(dO * O) and L2 = L * log2(e) per padded query row (padding rows:
// D = 0, L2 = +inf); zeroes the row of the fp32 dQ accumulator (and the main
// kernel's split-item counters).  HD: columns
// of the accumulator (d); HDV: columns of O and dO (dv).  A row is HDV / 8
// lanes with 16 bytes of O and of dO each; a warp takes two groups of
// 32 / (HDV / 8) rows per step, so that every lane has four 16-byte loads in
// flight (the kernel is short and bound by memory latency as much as by
// bandwidth).
template <int HD, int HDV>
__global__ void __launch_bounds__(256) fa_bwd_pre(const uint16_t* __restrict__ O, const uint16_t* __restrict__ dO,
                                                  const float* __restrict__ L, float* __restrict__ lse2,
                                                  float* __restrict__ delta, float* __restrict__ dq_acc,
                                                  unsigned int* __restrict__ split_counters, int n_counters,
                                                  long long rows_pad, int Tq, long long Tq_pad) {
  if (blockIdx.x == 0)
    for (int c = threadIdx.x; c < n_counters; c += blockDim.x) split_counters[c] = 0u;
  constexpr int LPR = HDV / 8;   // lanes per row
  constexpr int RPG = 32 / LPR;  // rows per group
  constexpr int UNR = 2;         // groups per warp step
  constexpr int ZF4 = HD / (4 * LPR);  // float4 of the accumulator row each lane zeroes
  const int lane = threadIdx.x & 31, sub = lane / LPR, part = lane - sub * LPR;
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  const long long wid = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  for (long long base = wid * (RPG * UNR); base < rows_pad; base += warps * (RPG * UNR)) {
    uint4 a[UNR], g[UNR];
    long long row[UNR], src_row[UNR];
    bool real[UNR];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      row[u] = base + u * RPG + sub;
      const long long bh = row[u] / Tq_pad;
      const long long q = row[u] - bh * Tq_pad;
      real[u] = row[u] < rows_pad && q < Tq;
      src_row[u] = bh * Tq + q;
      a[u] = g[u] = make_uint4(0u, 0u, 0u, 0u);
      if (real[u]) {
        a[u] = *reinterpret_cast<const uint4*>(O + src_row[u] * HDV + part * 8);
        g[u] = *reinterpret_cast<const uint4*>(dO + src_row[u] * HDV + part * 8);
      }
    }
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const uint32_t aw[4] = {a[u].x, a[u].y, a[u].z, a[u].w}, gw[4] = {g[u].x, g[u].y, g[u].z, g[u].w};
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        dot += __uint_as_float(aw[e] << 16) * __uint_as_float(gw[e] << 16);
        dot += __uint_as_float(aw[e] & 0xffff0000u) * __uint_as_float(gw[e] & 0xffff0000u);
      }
#pragma unroll
      for (int off = LPR / 2; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
      if (row[u] < rows_pad) {
        if (part == 0) {
          delta[row[u]] = dot;
          lse2[row[u]] = real[u] ? L[src_row[u]] * 1.4426950408889634f : __int_as_float(0x7f800000);
        }
        float4* acc = reinterpret_cast<float4*>(dq_acc + row[u] * HD) + part * ZF4;
#pragma unroll
        for (int z = 0; z < ZF4; ++z) acc[z] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  }
}

// dQ = bf16(scale * accumulator).  A row is HD / 8 lanes with 8 fp32 each;
// a warp takes two groups of 32 / (HD / 8) rows per step (four 16-byte loads
// in flight per lane).
template <int HD>
__global__ void __launch_bounds__(256) fa_dq_cast(const float* __restrict__ dq_acc, uint16_t* __restrict__ dQ,
                                                  long long q_rows, int Tq, long long Tq_pad, float scale) {
  constexpr int LPR = HD / 8;
  constexpr int RPG = 32 / LPR;
  constexpr int UNR = 2;
  const int lane = threadIdx.x & 31, sub = lane / LPR, part = lane - sub * LPR;
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  const long long wid = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  for (long long base = wid * (RPG * UNR); base < q_rows; base += warps * (RPG * UNR)) {
    float4 x[UNR], y[UNR];
    long long row[UNR];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      row[u] = base + u * RPG + sub;
      x[u] = y[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (row[u] < q_rows) {
        const long long bh = row[u] / Tq;
        const float* src = dq_acc + (bh * Tq_pad + (row[u] - bh * Tq)) * HD + part * 8;
        x[u] = *reinterpret_cast<const float4*>(src);
        y[u] = *reinterpret_cast<const float4*>(src + 4);
      }
    }
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      if (row[u] >= q_rows) continue;
      uint4 o;
      o.x = pack_bf16x2(x[u].x * scale, x[u].y * scale);
      o.y = pack_bf16x2(x[u].z * scale, x[u].w * scale);
      o.z = pack_bf16x2(y[u].x * scale, y[u].y * scale);
      o.w = pack_bf16x2(y[u].z * scale, y[u].w * scale);
      *reinterpret_cast<uint4*>(dQ + row[u] * HD + part * 8) = o;
    }
  }
}

__global__ void fa_zero_words(uint32_t* p, size_t n) {
  for (size_t t = blockIdx.x * (size_t)blockDim.x + threadIdx.x; t < n; t += (size_t)gridDim.x * blockDim.x) p[t] = 0u;
}

template <int HD, int HDV, bool CAUSAL, bool WINDOW>
cudaError_t launch_main_t(const fa::Problem& pr, const CUtensorMap* maps, const BwdParams& bp, cudaStream_t stream) {
  using C = BwdCfg<HD, HDV>;
  const void* fn = reinterpret_cast<const void*>(fa_bwd_main<HD, HDV, CAUSAL, WINDOW>);
  cudaError_t e = fa::allow_dynamic_smem(fn, C::SMEM);
  if (e != cudaSuccess) return e;
  if (kSplitRegs<HD>) {
    // The register split only balances if every thread was launched with
    // exactly kRegsLaunch registers; otherwise the dQ warpgroup's request
    // could never be met, so refuse to launch.
    cudaFuncAttributes fa_attr;
    e = cudaFuncGetAttributes(&fa_attr, fn);
    if (e != cudaSuccess) return e;
    if (fa_attr.numRegs != kRegsLaunch) return cudaErrorInvalidConfiguration;
  }
  // one CTA per item, two per split item (within int range: checked by the API, n_split <= kMaxSplitItems)
  dim3 grid((unsigned)(bp.n_whole + 2 * bp.n_split));
  fa_bwd_main<HD, HDV, CAUSAL, WINDOW><<<grid, kThreads, C::SMEM, stream>>>(maps[0], maps[1], maps[2], maps[3], maps[4], maps[5],
                                                               maps[6], bp);
  return cudaGetLastError();
}

template <int HD, int HDV>
cudaError_t launch_main_dims(const fa::Problem& pr, const CUtensorMap* maps, const BwdParams& bp,
                             cudaStream_t stream) {
  if (!pr.causal) return launch_main_t<HD, HDV, false, false>(pr, maps, bp, stream);
  if (pr.window) return launch_main_t<HD, HDV, true, true>(pr, maps, bp, stream);
  return launch_main_t<HD, HDV, true, false>(pr, maps, bp, stream);
}

// Groups per super-batch of fa_bwd_main's grid order: the smallest divisor of
// the group count whose super-batch holds at least 1.5 CTAs per SM, so that
// one super-batch fills the GPU with a heaviest-first queue of its own while
// few groups' data is live in L2.  0 if the SM count cannot be read.
int backward_super_batch(int n_groups, int kv_tiles) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                 cudaSuccess)
    return 0;
  return fa::super_batch_groups(n_groups, kv_tiles, sms);
}

inline int grid_for(long long work, int per_block) {
  long long g = (work + per_block - 1) / per_block;
  if (g > 152LL * 32) g = 152LL * 32;
  return (int)(g < 1 ? 1 : g);
}

}  // namespace

namespace fa {

BwdWorkspace backward_workspace_layout(const Problem& p) {
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  const size_t rows = (size_t)p.B * p.Hq * (size_t)p.Tq_pad();
  BwdWorkspace w;
  w.dq_acc = 0;
  w.lse2 = up(w.dq_acc + rows * p.d * sizeof(float));
  w.delta = up(w.lse2 + rows * sizeof(float));
  w.part = up(w.delta + rows * sizeof(float));
  w.total_min = w.part;
  // Items have equal work without a causal mask: then a short last round may
  // be split (up to kMaxSplitItems items).  (With a window the last key
  // tiles of each head are lighter, and splitting did not pay.)
  const long long n_items = (long long)p.B * p.Hkv * p.kv_tiles();
  w.split_cap = !p.causal ? (int)(n_items < kMaxSplitItems ? n_items : kMaxSplitItems) : 0;
  w.counters = up(w.part + (size_t)w.split_cap * 2 * kTile * (p.d + p.dv) * sizeof(float));
  w.total = up(w.counters + (size_t)w.split_cap * sizeof(unsigned int));
  return w;
}

// Items of the backward main kernel run as two halves (each half walks half
// of the item's query tiles and the halves' dK / dV are added): the last
// n_items mod sms items, where items have equal work and that last round
// fills at most half of the SMs, so its halves run on twice as many SMs.
int backward_split_items(const Problem& p, int split_cap) {
  int dev = 0, sms = 0;
  if (split_cap <= 0 || cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return 0;
  const long long n_items = (long long)p.B * p.Hkv * p.kv_tiles();
  const long long r = n_items % sms;
  return (r > 0 && 2 * r <= sms && r <= split_cap) ? (int)r : 0;
}

cudaError_t launch_backward(const Problem& pr, const void* Q, const void* K, const void* V, const void* O,
                            const void* dO, const float* L, void* dQ, void* dK, void* dV, void* workspace,
                            size_t workspace_bytes, int stages, cudaStream_t stream, int* launches) {
  const long long q_rows = (long long)pr.B * pr.Hq * pr.Tq;
  const long long k_rows = (long long)pr.B * pr.Hkv * pr.Tk;
  if (q_rows == 0 && k_rows == 0) return cudaSuccess;
  if (q_rows == 0 || pr.Tk == 0) {
    if (!(stages & FA_BWD_MAIN)) return cudaSuccess;
    // No query rows: dK = dV = 0.  No keys: dQ = 0.
    if (k_rows) {
      fa_zero_words<<<grid_for(k_rows * pr.d / 2, 256), 256, 0, stream>>>(static_cast<uint32_t*>(dK),
                                                                         (size_t)k_rows * pr.d / 2);
      fa_zero_words<<<grid_for(k_rows * pr.dv / 2, 256), 256, 0, stream>>>(static_cast<uint32_t*>(dV),
                                                                          (size_t)k_rows * pr.dv / 2);
      *launches += 2;
    }
    if (q_rows) {
      fa_zero_words<<<grid_for(q_rows * pr.d / 2, 256), 256, 0, stream>>>(static_cast<uint32_t*>(dQ),
                                                                         (size_t)q_rows * pr.d / 2);
      *launches += 1;
    }
    return cudaGetLastError();
  }
  const BwdWorkspace w = backward_workspace_layout(pr);
  // the split items' area is used only where the caller's workspace holds it
  const int split_cap = workspace_bytes >= w.total ? w.split_cap : 0;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* dq_acc = reinterpret_cast<float*>(ws + w.dq_acc);
  float* lse2 = reinterpret_cast<float*>(ws + w.lse2);
  float* delta = reinterpret_cast<float*>(ws + w.delta);
  float* part = reinterpret_cast<float*>(ws + w.part);
  unsigned int* split_counters = reinterpret_cast<unsigned int*>(ws + w.counters);
  const long long rows_pad = (long long)pr.B * pr.Hq * pr.Tq_pad();

  cudaError_t e = cudaSuccess;
  // 1. preprocess
  if (stages & FA_BWD_PRE) {
  auto pre = pr.d == 64 ? (pr.dv == 64 ? fa_bwd_pre<64, 64> : fa_bwd_pre<64, 128>)
                        : (pr.dv == 64 ? fa_bwd_pre<128, 64> : fa_bwd_pre<128, 128>);
  pre<<<grid_for(rows_pad, 8 * 2 * (32 / (pr.dv / 8))), 256, 0, stream>>>(static_cast<const uint16_t*>(O), static_cast<const uint16_t*>(dO), L,
                                                 lse2, delta, dq_acc, split_counters, split_cap, rows_pad, pr.Tq,
                                                 pr.Tq_pad());
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ++*launches;
  }

  // 2. main
  if (stages & FA_BWD_MAIN) {
  CUtensorMap maps[7];
  if (!encode_rows_bf16(&maps[0], Q, pr.d, pr.Tq, (long long)pr.B * pr.Hq) ||
      !encode_rows_bf16(&maps[1], K, pr.d, pr.Tk, (long long)pr.B * pr.Hkv) ||
      !encode_rows_bf16(&maps[2], V, pr.dv, pr.Tk, (long long)pr.B * pr.Hkv) ||
      !encode_rows_bf16(&maps[3], dO, pr.dv, pr.Tq, (long long)pr.B * pr.Hq) ||
      !encode_rows_bf16(&maps[4], dK, pr.d, pr.Tk, (long long)pr.B * pr.Hkv) ||
      !encode_rows_bf16(&maps[5], dV, pr.dv, pr.Tk, (long long)pr.B * pr.Hkv) ||
      !encode_acc_f32(&maps[6], dq_acc, pr.d, pr.Tq_pad(), (long long)pr.B * pr.Hq, 32))
    return cudaErrorInvalidValue;
  BwdParams bp;
  bp.lse2 = lse2;
  bp.delta = delta;
  bp.status = device_status_word();
  bp.Hq = pr.Hq;
  bp.Hkv = pr.Hkv;
  bp.G = pr.G();
  bp.Tq = pr.Tq;
  bp.Tk = pr.Tk;
  bp.causal_off = pr.Tk - pr.Tq;
  bp.window = pr.causal ? pr.window : 0;
  bp.q_tiles = pr.q_tiles();
  bp.kv_tiles = pr.kv_tiles();
  bp.sb_groups = backward_super_batch(pr.B * pr.Hkv, pr.kv_tiles());
  if (bp.sb_groups < 1) return cudaErrorInvalidValue;
  bp.Tq_pad = pr.Tq_pad();
  bp.scale = pr.scale;
  bp.scale_log2 = pr.scale * 1.4426950408889634f;
  bp.test_withhold_do = fa::test_withhold() == fa::kWithholdBwdDO;
  bp.n_split = backward_split_items(pr, split_cap);
  bp.n_whole = (int)((long long)pr.B * pr.Hkv * pr.kv_tiles()) - bp.n_split;
  bp.part = part;
  bp.split_counters = split_counters;
  if (pr.d == 64)
    e = pr.dv == 64 ? launch_main_dims<64, 64>(pr, maps, bp, stream) : launch_main_dims<64, 128>(pr, maps, bp, stream);
  else
    e = pr.dv == 64 ? launch_main_dims<128, 64>(pr, maps, bp, stream)
                    : launch_main_dims<128, 128>(pr, maps, bp, stream);
  if (e != cudaSuccess) return e;
  ++*launches;
  }

  // 3. dQ cast
  if (!(stages & FA_BWD_CAST)) return cudaSuccess;
  const int rows_per_block = 8 * 2 * (32 / (pr.d / 8));  // 8 warps, two row groups each
  if (pr.d == 64)
    fa_dq_cast<64><<<grid_for(q_rows, rows_per_block), 256, 0, stream>>>(dq_acc, static_cast<uint16_t*>(dQ), q_rows,
                                                                         pr.Tq, pr.Tq_pad(), pr.scale);
  else
    fa_dq_cast<128><<<grid_for(q_rows, rows_per_block), 256, 0, stream>>>(dq_acc, static_cast<uint16_t*>(dQ),
                                                                          q_rows, pr.Tq, pr.Tq_pad(), pr.scale);
  e = cudaGetLastError();
  if (e == cudaSuccess) ++*launches;
  return e;
}

}  // namespace fa
