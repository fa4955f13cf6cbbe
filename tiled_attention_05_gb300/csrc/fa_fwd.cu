// Forward pass of tiled exact attention on sm_103a.
//
// Method ("What Ordinary Autograd Saves: Tiling the Forward Pass Is Only Half
// the Algorithm", section "The implementation under test"): for one block of
// query rows, walk the key/value blocks keeping per row a running maximum m,
// a running sum of exponentials l and an unnormalised output; rescale the
// output when the maximum moves; normalise once at the end and emit
// L = m + log(l) beside O.  Nothing of size Tq x Tk is ever stored.
//
// GB300 mapping: a persistent grid of one CTA per SM.  A work item is two
// 128-row query tiles (A and B) of one (batch, head), sharing every K/V tile
// the CTA loads for it; each CTA walks its items (heaviest causal rows first,
// in a snake order over the CTAs so that their totals even out) and starts
// the next item's loads and first MMAs while the current one finishes.
// Without a causal mask (items of equal work) a last round with at most half
// as many items as SMs is run as single-tile items (tile B left empty) on
// twice as many SMs.
//   warp 0       TMA producer: Q_A, Q_B per item (each as soon as the last
//                S of the previous item's tile has read its buffer), then the
//                item's K_j / V_j through NS-deep rings that run on across items.
//   warp 1       tcgen05 issuer.  Per key tile j it issues, in this order,
//                  O_A += P_A(j) V_j,  S_A(j+1) = Q_A K_{j+1}^T,
//                  O_B += P_B(j) V_j,  S_B(j+1) = Q_B K_{j+1}^T,
//                so while one softmax warpgroup works on its tile the tensor
//                pipe runs the other tile's two MMAs (ping-pong).  P is read
//                straight from TMEM (A operand); the MMAs of one thread execute
//                in issue order, so S_X(j+1) overwrites P_X(j) only after the
//                P.V that reads it.  An item's first S MMAs follow the previous
//                item's last P.V at once, while the softmax warpgroups write
//                that item's output.
//   warps 4..7   softmax of tile A, warps 8..11 softmax of tile B (thread =
//                query row = TMEM lane): load the score row, mask, row max,
//                exp2, row sum, write P as packed bf16 over the scores in TMEM;
//                rescale the O row in TMEM when the max grows by more than 2^8
//                (lazy rescaling, exact after the final normalisation);
//                epilogue O / l -> bf16 -> global (each thread its row), L -> global.
//                The next item's first P.V into O_X waits for this warpgroup's
//                first P of that item, which it writes only after its epilogue
//                has read O_X out of TMEM.
//                The two softmax warpgroups take registers from the producer /
//                MMA warpgroup (setmaxnreg), so that a whole score row stays in
//                registers without spilling.
// TMEM columns: S_A/P_A [0,128), S_B/P_B [128,256), O_A [256,256+dv), O_B [384,384+dv).
// Scores are kept in log2 units (scale * log2(e) folded into one FMA).
//
// Each tile visits the key tiles [beg, end) its rows can see (causal: up to
// the diagonal; with a sliding window of W keys also from the first row's
// window start on).  The CTA loads the union of the two ranges once; a key
// tile inside the union that one tile does not need is skipped by that tile's
// MMAs and softmax.  Every barrier phase (and ring position) is counted from
// the start of the CTA, not of the item.
#include <cstdint>

#include "fa_internal.h"
#include "sm103_ptx.cuh"

using namespace fa_ptx;

namespace {

constexpr int BM = fa::kTile;  // query rows per tile (two tiles per work item)
constexpr int BN = fa::kTile;  // keys per tile
constexpr int kThreads = 384;
// Register split: every thread starts with kRegsLaunch; the producer / MMA
// warpgroup drops to kRegsLow and the two softmax warpgroups rise to
// kRegsHigh (one score row of 128 fp32 values and its packed P in registers
// without spilling).  kRegsLow + 2 * kRegsHigh = 3 * kRegsLaunch.
constexpr int kRegsLaunch = 168;  // 65536 / 384 rounded down to a multiple of 8
constexpr int kRegsLow = 88;
constexpr int kRegsHigh = (3 * kRegsLaunch - kRegsLow) / 2;  // 208
static_assert(kRegsLow + 2 * kRegsHigh == 3 * kRegsLaunch && kRegsHigh % 8 == 0, "setmaxnreg operands");
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P stays <= 256 between rescales

// The forward's waits: mbar_wait with a suspend-time hint on try_wait.  A
// thread that finds the phase incomplete then sleeps until it completes (or
// the hint runs out) and is woken ~80 cycles after the completing arrival,
// against 100-160 with the default limit (measured).  Same bounds and abort
// behaviour as mbar_wait.
constexpr uint32_t kSuspendHintNs = 100000u;
__device__ __forceinline__ bool try_wait_hinted(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool fwd_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                         uint64_t timeout_ns = 2000000000ull) {
  if (try_wait_hinted(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t spins = 0;
  while (true) {
    if (try_wait_hinted(bar, parity)) return true;
    if ((++spins & 63u) == 0) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > timeout_ns) {
        *abort = 1;
        return false;
      }
    }
  }
}

// HD: head size of Q and K (the score contraction); HDV: head size of V and O.
template <int HD, int HDV>
struct FwdCfg {
  static constexpr int NS = (HD == 64 && HDV == 64) ? 4 : 2;  // K/V ring depth
  // With a 4-deep ring K_{j+1} / V_{j+1} have landed long before tile j's P is
  // ready, so the softmax checks them and the MMA thread saves a barrier
  // check per key tile.  With a 2-deep ring they often land later than that,
  // and tying P_X(j).V to them would stall the tensor pipe.
  static constexpr bool KV_VIA_SOFTMAX = NS >= 3;
  static constexpr int Q_BYTES = BM * HD * 2;
  static constexpr int K_BYTES = BN * HD * 2;
  static constexpr int V_BYTES = BN * HDV * 2;
  static constexpr int OFF_Q = 0;  // [2]: tile A, tile B
  static constexpr int OFF_K = OFF_Q + 2 * Q_BYTES;
  static constexpr int OFF_V = OFF_K + NS * K_BYTES;
  static constexpr int OFF_BAR = OFF_V + NS * V_BYTES;
  static constexpr int NBAR = 2 + 2 + 3 * NS + 2 + 2 + 2 + 1;
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 16;
  static_assert(SMEM <= 232448, "shared memory budget");
};

struct FwdParams {
  uint16_t* O;  // bf16 [B, Hq, Tq, dv]
  float* L;
  int* status;
  int Hq, Hkv, G, Tq, Tk;
  int causal_off;  // Tk - Tq
  int window;      // causal sliding window in keys, 0 = none
  int kv_tiles;
  int n_bh;            // B * Hq
  int n_pairs;         // query-tile pairs per (batch, head)
  long long n_full;    // work items that are pairs of query tiles
  long long n_items;   // all work items: n_full pairs, then single query tiles
  float scale_log2;  // scale * log2(e)
  int test_withhold_q;  // test build only: never issue the Q loads (every wait then times out)
};

// Key tiles [*beg, *end) that query rows [qa, qa+128) must visit (empty: 0, 0).
template <bool CAUSAL, bool WINDOW>
__device__ __forceinline__ void kv_range_for(const FwdParams& p, int qa, int* beg, int* end) {
  *beg = *end = 0;
  if (qa >= p.Tq) return;
  if (!CAUSAL) {
    *end = p.kv_tiles;
    return;
  }
  const int last_key = min(qa + BM, p.Tq) - 1 + p.causal_off;  // last key the tile's last row sees
  if (last_key < 0) return;
  const int e = min(p.kv_tiles, last_key / BN + 1);
  int bg = 0;
  if (WINDOW) {
    const int first_key = qa + p.causal_off - p.window + 1;  // first key the tile's first row sees
    bg = first_key > 0 ? first_key / BN : 0;
  }
  if (bg < e) {
    *beg = bg;
    *end = e;
  }
}

// One work item: query tiles A = [q0, q0 + 128) and B = [q0 + 128, q0 + 256)
// of (batch, head) bh, and the key tiles each must visit.
struct FwdItem {
  int bh, q0, bkv;
  int kb[2], ke[2];  // key-tile range of tile A and tile B
  int ub, ue;        // their union, loaded once
  bool single;       // tile B is not part of the item (its rows belong to another item)
};

// The n-th item of this CTA, or false past its last.  Items are numbered
// heaviest causal rows first (the pair index slowest); round n of the grid
// takes items [n * G, n * G + G), CTA c the c-th of them in even rounds and
// the (G - 1 - c)-th in odd ones, so each CTA's heavy and light items pair up.
// Past n_full, every pair is split into two single-tile items (tile B empty),
// which spreads a short last round of equal-weight items over twice as many
// CTAs.
template <bool CAUSAL, bool WINDOW>
__device__ __forceinline__ bool fwd_item(const FwdParams& p, int n, FwdItem* it) {
  const long long G = gridDim.x, c = blockIdx.x;
  const long long k = n * G + ((n & 1) ? G - 1 - c : c);
  if (k >= p.n_items) return false;
  const bool single = k >= p.n_full;
  it->single = single;
  const long long kp = single ? p.n_full + ((k - p.n_full) >> 1) : k;  // the pair
  const int y = (int)(kp / p.n_bh);
  it->bh = (int)(kp - (long long)y * p.n_bh);
  const int b = it->bh / p.Hq, h = it->bh - b * p.Hq;
  it->q0 = (p.n_pairs - 1 - y) * (2 * BM) + (single ? (int)((k - p.n_full) & 1) * BM : 0);
  it->bkv = b * p.Hkv + h / p.G;
  kv_range_for<CAUSAL, WINDOW>(p, it->q0, &it->kb[0], &it->ke[0]);
  if (single) {
    it->kb[1] = it->ke[1] = 0;
  } else {
    kv_range_for<CAUSAL, WINDOW>(p, it->q0 + BM, &it->kb[1], &it->ke[1]);
  }
  // Tile B's rows follow tile A's, so B's range starts and ends no earlier
  // than A's, and starts no later than A's end: the union has no gap and
  // every key tile in it is needed by A or B.
  it->ub = it->ke[0] > it->kb[0] ? it->kb[0] : it->kb[1];
  it->ue = max(it->ke[0], it->ke[1]);
  return true;
}

// WINDOW (causal only): the sliding-window terms are compiled in only where
// a window is set, so the plain causal and full masks keep their lean code.
template <int HD, int HDV, bool CAUSAL, bool WINDOW>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using C = FwdCfg<HD, HDV>;
  constexpr int NS = C::NS;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;           // [2] per tile
  uint64_t* q_empty = q_full + 2;    // [2]
  // One "full" barrier per ring slot covers both K_j and V_j, so the MMA
  // thread checks a key tile once; K and V are released separately (K after
  // the last S that reads it, V after the last P.V), so K_{j+NS} can load
  // before V_j's readers are done.
  uint64_t* kv_full = q_empty + 2;
  uint64_t* k_empty = kv_full + NS;
  uint64_t* v_empty = k_empty + NS;
  uint64_t* s_full = v_empty + NS;  // [2] per tile
  uint64_t* p_full = s_full + 2;    // [2]
  uint64_t* o_done = p_full + 2;    // [2]
  uint64_t* drain = o_done + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t q_buf = smem_u32(smem + C::OFF_Q);
  const uint32_t k_base = smem_u32(smem + C::OFF_K);
  const uint32_t v_base = smem_u32(smem + C::OFF_V);
  bool withhold_q = false;
#ifdef FA_TEST_HOOKS
  withhold_q = p.test_withhold_q != 0;
#endif

  // Producer state; the first item's Q and its first NS key/value tiles (the
  // ring slots are all free) are issued during set-up, before TMEM allocation
  // and the CTA-wide barrier, so their memory latency overlaps the set-up.
  int nq[2] = {0, 0};  // Q_X loads issued (the producer) / waited for (the MMA thread)
  int pre_kv = 0;      // key/value tiles of item 0 issued during set-up
  auto load_q = [&](const FwdItem& it, int x) {
    if (!withhold_q) {
      mbar_arrive_expect_tx(&q_full[x], C::Q_BYTES);
#pragma unroll
      for (int cb = 0; cb < HD / 64; ++cb)
        tma_load_3d(smem + C::OFF_Q + x * C::Q_BYTES + cb * BM * 128, &tmQ, &q_full[x], cb * 64, it.q0 + x * BM,
                    it.bh);
    }
    ++nq[x];
  };
  auto load_k = [&](const FwdItem& it, int jj, int s) {
    mbar_arrive_expect_tx(&kv_full[s], C::K_BYTES + C::V_BYTES);
#pragma unroll
    for (int cb = 0; cb < HD / 64; ++cb)
      tma_load_3d(smem + C::OFF_K + s * C::K_BYTES + cb * BN * 128, &tmK, &kv_full[s], cb * 64,
                  (it.ub + jj) * BN, it.bkv);
  };
  auto load_v = [&](const FwdItem& it, int jj, int s) {
#pragma unroll
    for (int cb = 0; cb < HDV / 64; ++cb)
      tma_load_3d(smem + C::OFF_V + s * C::V_BYTES + cb * BN * 128, &tmV, &kv_full[s], cb * 64,
                  (it.ub + jj) * BN, it.bkv);
  };

  if (threadIdx.x == 0) {
    *abort_flag = (smem_u32(smem) & 1023u) ? 1 : 0;  // swizzled tiles need 1024 B alignment
    for (int x = 0; x < 2; ++x) {
      mbar_init(&q_full[x], 1);
      mbar_init(&q_empty[x], 1);
      mbar_init(&s_full[x], 1);
      mbar_init(&p_full[x], 128);
      mbar_init(&o_done[x], 1);
    }
    for (int s = 0; s < NS; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    mbar_init(drain, 1);
    fence_mbar_init();
    FwdItem it;
    if (*abort_flag == 0 && fwd_item<CAUSAL, WINDOW>(p, 0, &it)) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
#pragma unroll
      for (int x = 0; x < 2; ++x)
        if (it.ke[x] > it.kb[x]) load_q(it, x);
      for (; pre_kv < NS && pre_kv < it.ue - it.ub; ++pre_kv) {
        load_k(it, pre_kv, pre_kv);
        load_v(it, pre_kv, pre_kv);
      }
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool run = *abort_flag == 0;

  if (warp < 4) {
    setmaxnreg_dec<kRegsLow>();
    if (warp == 0) {
      // ------------------------------------------------------------ producer
      if (lane == 0 && run) {
        int g = pre_kv;     // ring position of the next key/value tile (running over items)
        int kv_last[NS];    // last ring pass whose K and V loads were both issued, per slot
        bool half = false;  // a K load was issued whose V load was not (abort in between)
#pragma unroll
        for (int s = 0; s < NS; ++s) kv_last[s] = s < pre_kv ? 0 : -1;
        bool ok = true;
        FwdItem it;
        for (int n = 0; ok && fwd_item<CAUSAL, WINDOW>(p, n, &it); ++n) {
          if (n > 0) {
#pragma unroll
            for (int x = 0; x < 2; ++x) {
              if (it.ke[x] <= it.kb[x]) continue;
              // Q_X's buffer is free once the previous item's last S_X has read it.
              if (nq[x] > 0 && !fwd_wait(&q_empty[x], (nq[x] - 1) & 1, abort_flag)) { ok = false; break; }
              load_q(it, x);
            }
          }
          for (int jj = n == 0 ? pre_kv : 0; ok && jj < it.ue - it.ub; ++jj, ++g) {
            const int s = g % NS, u = g / NS;
            if (!fwd_wait(&k_empty[s], (u & 1) ^ 1, abort_flag)) { ok = false; break; }
            load_k(it, jj, s);
            half = true;
            if (!fwd_wait(&v_empty[s], (u & 1) ^ 1, abort_flag)) { ok = false; break; }
            load_v(it, jj, s);
            half = false;
            kv_last[s] = u;
          }
        }
        // Every issued copy must land before the CTA releases its shared memory.
        if (!withhold_q)
#pragma unroll
          for (int x = 0; x < 2; ++x)
            if (nq[x] > 0) mbar_wait_bounded(&q_full[x], (nq[x] - 1) & 1);
#pragma unroll
        for (int s = 0; s < NS; ++s)
          if (kv_last[s] >= 0) mbar_wait_bounded(&kv_full[s], kv_last[s] & 1);
        // A K load whose V never followed leaves its barrier short of bytes:
        // give the copy in flight time to land before the CTA exits.
        if (half) {
          const uint64_t t0 = globaltimer_ns();
          while (globaltimer_ns() - t0 < 1000000ull) {
          }
        }
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      if (lane == 0 && run) {
        constexpr uint32_t idS = idesc_bf16(BM, BN, 0, 0);
        constexpr uint32_t idPV = idesc_bf16(BM, HDV, 0, 1);
        int np[2] = {0, 0};  // p_full phases waited for, per tile
        int base = 0;        // ring position of the current item's first key tile
        bool ok = true;
        FwdItem it;
        for (int n = 0; ok && fwd_item<CAUSAL, WINDOW>(p, n, &it); ++n) {
          auto active = [&](int x, int j) { return j >= it.kb[x] && j < it.ke[x]; };
          // S_X(j) = Q_X K_j^T into TMEM [128 X, 128 X + 128).  Every barrier
          // check here costs the tensor pipe a shared-memory round trip, so
          // K_j / V_j are checked only where nothing else vouches for them
          // (wait_kv): tile B's S uses the key tile tile A has just waited
          // for, and with KV_VIA_SOFTMAX, inside an item, the P_X(j-1)
          // barrier waited for just before covers them too (the softmax
          // checks K_j / V_j before it arrives).
          auto issue_s = [&](int x, int j, bool wait_kv) -> bool {
            const int pos = base + (j - it.ub), s = pos % NS;
            if (j == it.kb[x]) {  // the tile's first S of this item: wait for its Q
              if (!fwd_wait(&q_full[x], nq[x] & 1, abort_flag)) return false;
              ++nq[x];
            }
            if (wait_kv && !fwd_wait(&kv_full[s], (pos / NS) & 1, abort_flag)) return false;
            tc_fence_after();
            const uint32_t q_base = q_buf + x * C::Q_BYTES;
#pragma unroll
            for (int k = 0; k < HD / 16; ++k) {
              const uint64_t a = desc_kmajor(q_base + (k >> 2) * (BM * 128) + (k & 3) * 32);
              const uint64_t bd = desc_kmajor(k_base + s * C::K_BYTES + (k >> 2) * (BN * 128) + (k & 3) * 32);
              mma_ss(tmem + x * 128, a, bd, idS, k > 0 ? 1u : 0u);
            }
            mma_commit(&s_full[x]);
            if (j == it.ke[x] - 1) mma_commit(&q_empty[x]);  // last reader of Q_X in this item
            return true;
          };
          // O_X += P_X(j) V_j with P_X read from TMEM (packed bf16 over S_X)
          auto issue_pv = [&](int x, int j) -> bool {
            const int s = (base + j - it.ub) % NS;
            // V_j landed with K_j: the S(j) MMA before this P.V waited for both.
            if (!fwd_wait(&p_full[x], np[x] & 1, abort_flag)) return false;
            ++np[x];
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < BN / 16; ++k) {
              const uint64_t bd = desc_mnmajor(v_base + s * C::V_BYTES + k * 2048, BN * 128);
              mma_ts(tmem + 256 + x * 128, tmem + x * 128 + k * 8, bd, idPV, (j > it.kb[x] || k > 0) ? 1u : 0u);
            }
            return true;
          };
          if (it.ue > it.ub) {
            // A tile whose range starts at ub gets its first S up front; tile B,
            // if it starts later, gets it in the loop below one step before its range.
            if (ok && active(0, it.ub)) ok = issue_s(0, it.ub, true);
            if (ok && active(1, it.ub)) ok = issue_s(1, it.ub, !active(0, it.ub));
            if (ok) mma_commit(&k_empty[base % NS]);
          }
          for (int j = it.ub; ok && j < it.ue; ++j) {
#pragma unroll
            for (int x = 0; x < 2; ++x) {
              if (active(x, j)) {
                if (!issue_pv(x, j)) { ok = false; break; }
                if (x == 1 || !active(1, j)) mma_commit(&v_empty[(base + j - it.ub) % NS]);  // last reader of V_j
              }
              if (active(x, j + 1)) {
                // Tile B relies on tile A's wait (or, with KV_VIA_SOFTMAX, on
                // A's P_A(j) when A goes on to j + 1); with KV_VIA_SOFTMAX a
                // tile's own P_X(j), just waited for, vouches for K_{j+1} / V_{j+1}.
                const bool covered = (x == 1 && active(0, j + 1) && (!C::KV_VIA_SOFTMAX || active(0, j))) ||
                                     (C::KV_VIA_SOFTMAX && active(x, j));
                if (!issue_s(x, j + 1, !covered)) { ok = false; break; }
                if (x == 1 || !active(1, j + 1))
                  mma_commit(&k_empty[(base + j + 1 - it.ub) % NS]);  // last reader of K_{j+1}
              } else if (active(x, j)) {
                mma_commit(&o_done[x]);
              }
            }
          }
          base += it.ue - it.ub;
        }
        // Let every MMA issued above finish before TMEM is released.
        mma_commit(drain);
        mbar_wait_bounded(drain, 0);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue of tile x
    setmaxnreg_inc<kRegsHigh>();
    const int x = (warp - 4) >> 2;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // row inside the tile == TMEM lane
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const uint32_t tS = tmem + x * 128 + lane_base;
    const uint32_t tO = tmem + 256 + x * 128 + lane_base;
    const float sl2 = p.scale_log2;
    const float NEG_INF = -__int_as_float(0x7f800000);
    int ns = 0, no = 0;  // s_full / o_done phases waited for
    int base = 0;        // ring position of the current item's first key tile
    bool ok = run;
    FwdItem it;
    for (int n = 0; ok && fwd_item<CAUSAL, WINDOW>(p, n, &it); ++n) {
      const int item_base = base;
      base += it.ue - it.ub;
      const int kbx = x ? it.kb[1] : it.kb[0];  // first key tile of this tile's range
      const int nkv = (x ? it.ke[1] : it.ke[0]) - kbx;
      const int qx0 = it.q0 + x * BM;
      const int i = qx0 + r;  // query row
      float m_ref = NEG_INF;  // reference max (log2 units) the P values are taken against
      float l = 0.f;
      for (int jx = 0; ok && jx < nkv; ++jx) {  // jx-th key tile of this tile's range
        // the warp agrees on the outcome before its collective TMEM loads
        if (!__all_sync(0xffffffffu, fwd_wait(&s_full[x], ns & 1, abort_flag))) { ok = false; break; }
        ++ns;
        tc_fence_after();
        uint32_t sr[BN];
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) tmem_ld32(tS + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[c * 32]));
        tmem_wait_ld();
        const int kv0 = (kbx + jx) * BN;
        // window: the tile's last row starts its window past this key tile's start
        const bool win_mask = WINDOW && qx0 + BM - 1 + p.causal_off - p.window + 1 > kv0;
        const bool need_mask = (kv0 + BN > p.Tk) || (CAUSAL && kv0 + BN - 1 > qx0 + p.causal_off) || win_mask;
        if (need_mask) {
          int lim = p.Tk - kv0;  // columns [lo, lim) are visible to row i
          if (CAUSAL) lim = min(lim, i + p.causal_off + 1 - kv0);
          const int lo = win_mask ? i + p.causal_off - p.window + 1 - kv0 : -BN;
#pragma unroll
          for (int c = 0; c < BN; ++c)
            if (c >= lim || c < lo) sr[c] = __float_as_uint(NEG_INF);
        }
        // row max: eight independent three-input max chains (short dependency depth)
        float pm[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) pm[k] = __uint_as_float(sr[k]);
#pragma unroll
        for (int c = 8; c < BN; c += 16)
#pragma unroll
          for (int k = 0; k < 8; ++k) pm[k] = fmax3(pm[k], __uint_as_float(sr[c + k]), __uint_as_float(sr[c + 8 + k]));
        const float mt = fmax3(fmax3(pm[0], pm[1], pm[2]), fmax3(pm[3], pm[4], pm[5]), fmaxf(pm[6], pm[7]));
        const float mt2 = mt * sl2;
        float m_new = m_ref;
        if (mt2 > m_ref + kRescaleThreshold) m_new = mt2;  // also taken when m_ref == -inf
        // Does this row's O need rescaling, and does any row of the warp's?  (The
        // vote is taken here, where fewer registers are live than after exp2.)
        const bool rescale = jx > 0 && m_new != m_ref && m_ref != NEG_INF;
        const bool warp_rescale = __any_sync(0xffffffffu, rescale);
        const float base = (m_new == NEG_INF) ? 0.f : m_new;
        const uint64_t sl2x2 = f2_pack(sl2, sl2), nbase2 = f2_pack(-base, -base);
        // exponentials (argument and row sum on packed pairs); P (packed bf16)
        // goes over the already-loaded scores in TMEM 16 columns at a time
        uint64_t rs[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const uint64_t xv = f2_fma(
                f2_pack(__uint_as_float(sr[32 * c + 2 * e]), __uint_as_float(sr[32 * c + 2 * e + 1])), sl2x2, nbase2);
            const float e0 = ex2(f2_lo(xv)), e1 = ex2(f2_hi(xv));
            rs[e & 3] = f2_add(rs[e & 3], f2_pack(e0, e1));
            pk[e] = pack_bf16x2(e0, e1);
          }
          tmem_st16(tS + 16 * c, pk);
        }
        const uint64_t rs2 = f2_add(f2_add(rs[0], rs[1]), f2_add(rs[2], rs[3]));
        const float rowsum = f2_lo(rs2) + f2_hi(rs2);
        // O_X is idle here: the P.V of tile j-1 completed before S_X(j) did.
        const float alpha = (m_new == m_ref) ? 1.f : (m_ref == NEG_INF ? 0.f : ex2(m_ref - m_new));
        l = l * alpha + rowsum;
        // TMEM loads and stores are warp-collective: when any row of the warp
        // must rescale its O row, every lane takes part (factor 1 where not).
        if (warp_rescale) {
          const float a = rescale ? alpha : 1.f;
#pragma unroll
          for (int c = 0; c < HDV / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * a);
            tmem_st32(tO + c * 32, o);
          }
        }
        m_ref = m_new;
        tmem_wait_st();
        tc_fence_before();
        // The MMA thread takes this barrier as word that K / V of this tile's
        // next key tile have landed too (it issues that S right after this
        // tile's P.V without checking them), so one thread checks them first.
        if (C::KV_VIA_SOFTMAX && r == 0 && jx + 1 < nkv) {
          const int pos = item_base + kbx + jx + 1 - it.ub;
          if (!fwd_wait(&kv_full[pos % NS], (pos / NS) & 1, abort_flag)) ok = false;
        }
        mbar_arrive(&p_full[x]);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      }
      // ---- epilogue: O / l -> bf16 -> global (one row per thread); L -> global
      if (ok && nkv > 0) {
        if (!__all_sync(0xffffffffu, fwd_wait(&o_done[x], no & 1, abort_flag))) ok = false;
        ++no;
        tc_fence_after();
      }
      // (a tile past the last row, or tile B of a single-tile item, has nothing to write)
      if (!ok || qx0 >= p.Tq || (x == 1 && it.single)) continue;
      const bool row_ok = i < p.Tq;
      if (row_ok) p.L[(size_t)it.bh * p.Tq + i] = l > 0.f ? (m_ref + __log2f(l)) * 0.69314718055994531f : NEG_INF;
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      uint4* orow = reinterpret_cast<uint4*>(p.O + ((size_t)it.bh * p.Tq + (row_ok ? i : 0)) * HDV);
#pragma unroll
      for (int c = 0; c < HDV / 32; ++c) {
        uint32_t o[32];
        if (nkv > 0) {
          tmem_ld32(tO + c * 32, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0u;
        }
        if (row_ok) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(o[8 * q + 0]) * inv_l, __uint_as_float(o[8 * q + 1]) * inv_l);
            w.y = pack_bf16x2(__uint_as_float(o[8 * q + 2]) * inv_l, __uint_as_float(o[8 * q + 3]) * inv_l);
            w.z = pack_bf16x2(__uint_as_float(o[8 * q + 4]) * inv_l, __uint_as_float(o[8 * q + 5]) * inv_l);
            w.w = pack_bf16x2(__uint_as_float(o[8 * q + 6]) * inv_l, __uint_as_float(o[8 * q + 7]) * inv_l);
            orow[c * 4 + q] = w;
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicExch(p.status, DEV_TIMEOUT);
}

// SM count of the current device (the persistent grid's size); 0 if unknown.
int sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                 cudaSuccess)
    return 0;
  return sms;
}

template <int HD, int HDV, bool CAUSAL, bool WINDOW>
cudaError_t launch_fwd_t(const fa::Problem& pr, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                         void* O, float* L, cudaStream_t stream) {
  using C = FwdCfg<HD, HDV>;
  const void* fn = reinterpret_cast<const void*>(fa_fwd_kernel<HD, HDV, CAUSAL, WINDOW>);
  cudaError_t e = fa::allow_dynamic_smem(fn, C::SMEM);
  if (e != cudaSuccess) return e;
  // The register split only balances if every thread was launched with
  // exactly kRegsLaunch registers; otherwise the softmax warpgroups' request
  // could never be met, so refuse to launch.
  cudaFuncAttributes fa_attr;
  e = cudaFuncGetAttributes(&fa_attr, fn);
  if (e != cudaSuccess) return e;
  if (fa_attr.numRegs != kRegsLaunch) return cudaErrorInvalidConfiguration;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  FwdParams p;
  p.O = static_cast<uint16_t*>(O);
  p.L = L;
  p.status = fa::device_status_word();
  p.Hq = pr.Hq;
  p.Hkv = pr.Hkv;
  p.G = pr.G();
  p.Tq = pr.Tq;
  p.Tk = pr.Tk;
  p.causal_off = pr.Tk - pr.Tq;
  p.window = pr.causal ? pr.window : 0;
  p.kv_tiles = pr.kv_tiles();
  p.n_bh = pr.B * pr.Hq;
  p.n_pairs = (pr.q_tiles() + 1) / 2;
  const long long n_pair_items = (long long)p.n_bh * p.n_pairs;
  // Without a causal mask every item has the same work.  A last round with at
  // most half as many items as SMs then runs them as single tiles on twice
  // as many SMs (a tile alone takes ~0.65 of a pair's time: no ping-pong).
  const long long r = n_pair_items % sms;
  p.n_full = (!pr.causal && r > 0 && 2 * r <= sms) ? n_pair_items - r : n_pair_items;
  p.n_items = p.n_full + 2 * (n_pair_items - p.n_full);
  p.scale_log2 = pr.scale * 1.4426950408889634f;
  p.test_withhold_q = fa::test_withhold() == fa::kWithholdFwdQ;
  const int grid = (int)(p.n_items < sms ? p.n_items : sms);
  fa_fwd_kernel<HD, HDV, CAUSAL, WINDOW><<<grid, kThreads, C::SMEM, stream>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

template <int HD, int HDV>
cudaError_t launch_fwd_dims(const fa::Problem& pr, const CUtensorMap& mq, const CUtensorMap& mk,
                            const CUtensorMap& mv, void* O, float* L, cudaStream_t stream) {
  if (!pr.causal) return launch_fwd_t<HD, HDV, false, false>(pr, mq, mk, mv, O, L, stream);
  if (pr.window) return launch_fwd_t<HD, HDV, true, true>(pr, mq, mk, mv, O, L, stream);
  return launch_fwd_t<HD, HDV, true, false>(pr, mq, mk, mv, O, L, stream);
}

__global__ void fa_fwd_empty_keys(uint32_t* O_words, size_t n_words, float* L, size_t n_rows) {
  const float NEG_INF = -__int_as_float(0x7f800000);
  for (size_t t = blockIdx.x * (size_t)blockDim.x + threadIdx.x; t < n_words || t < n_rows;
       t += (size_t)gridDim.x * blockDim.x) {
    if (t < n_words) O_words[t] = 0u;
    if (t < n_rows) L[t] = NEG_INF;
  }
}

}  // namespace

namespace fa {

cudaError_t launch_forward(const Problem& pr, const void* Q, const void* K, const void* V, void* O, float* L,
                           cudaStream_t stream, int* launches) {
  const long long rows = (long long)pr.B * pr.Hq * pr.Tq;
  if (rows == 0) return cudaSuccess;
  if (pr.Tk == 0) {
    const size_t words = (size_t)rows * pr.dv / 2;
    fa_fwd_empty_keys<<<1216, 256, 0, stream>>>(static_cast<uint32_t*>(O), words, L, (size_t)rows);
    ++*launches;
    return cudaGetLastError();
  }
  CUtensorMap mq, mk, mv;
  if (!encode_rows_bf16(&mq, Q, pr.d, pr.Tq, (long long)pr.B * pr.Hq) ||
      !encode_rows_bf16(&mk, K, pr.d, pr.Tk, (long long)pr.B * pr.Hkv) ||
      !encode_rows_bf16(&mv, V, pr.dv, pr.Tk, (long long)pr.B * pr.Hkv))
    return cudaErrorInvalidValue;
  cudaError_t e;
  if (pr.d == 64)
    e = pr.dv == 64 ? launch_fwd_dims<64, 64>(pr, mq, mk, mv, O, L, stream)
                    : launch_fwd_dims<64, 128>(pr, mq, mk, mv, O, L, stream);
  else
    e = pr.dv == 64 ? launch_fwd_dims<128, 64>(pr, mq, mk, mv, O, L, stream)
                    : launch_fwd_dims<128, 128>(pr, mq, mk, mv, O, L, stream);
  if (e == cudaSuccess) ++*launches;
  return e;
}

}  // namespace fa
