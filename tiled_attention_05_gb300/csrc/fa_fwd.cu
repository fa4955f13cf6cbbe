// Forward pass of tiled exact attention on sm_103a.
//
// Method ("What Ordinary Autograd Saves: Tiling the Forward Pass Is Only Half
// the Algorithm", section "The implementation under test"): for one block of
// query rows, walk the key/value blocks keeping per row a running maximum m,
// a running sum of exponentials l and an unnormalised output; rescale the
// output when the maximum moves; normalise once at the end and emit
// L = m + log(l) beside O.  Nothing of size Tq x Tk is ever stored.
//
// GB300 mapping (one CTA = one 128-row query tile of one (batch, head)):
//   warp 0      TMA producer: Q once, then K_j / V_j through an NS-deep ring.
//   warp 1      tcgen05 issuer: S_j = Q K_j^T into one of two TMEM score
//               buffers, then O += P_{j-1} V_{j-1} into the TMEM accumulator.
//   warps 2..5  softmax (thread = query row = TMEM lane): load the score row
//               from TMEM, mask, row max, exp2, row sum, write P (bf16) to
//               shared memory in the 128B-swizzled K-major layout the next
//               MMA reads; rescale the O row in TMEM when its max grows by
//               more than 2^8 (lazy rescaling: exact after normalisation);
//               epilogue O / l -> bf16 -> TMA store, L -> global.
// TMEM: S buffers at columns [0,128) and [128,256), O at [256, 256+d).
// Scores are kept in log2 units (scale * log2(e) folded into one FMA).
#include <cstdint>

#include "fa_internal.h"
#include "sm103_ptx.cuh"

using namespace fa_ptx;

namespace {

constexpr int BM = fa::kTile;  // query rows per CTA
constexpr int BN = fa::kTile;  // keys per tile
constexpr int kThreads = 192;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P stays <= 256 between rescales

template <int HD>
struct FwdCfg {
  static constexpr int NS = HD == 64 ? 4 : 2;  // K/V ring depth
  static constexpr int Q_BYTES = BM * HD * 2;
  static constexpr int KV_BYTES = BN * HD * 2;
  static constexpr int P_BYTES = BM * BN * 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int OFF_V = OFF_K + NS * KV_BYTES;
  static constexpr int OFF_P = OFF_V + NS * KV_BYTES;
  static constexpr int OFF_BAR = OFF_P + P_BYTES;
  static constexpr int NBAR = 1 + 4 * NS + 2 + 2 + 1 + 1 + 1;
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 16;
  static_assert(SMEM <= 232448, "shared memory budget");
};

struct FwdParams {
  float* L;
  int* status;
  int Hq, Hkv, G, Tq, Tk;
  int causal_off;  // Tk - Tq
  int kv_tiles;
  float scale_log2;  // scale * log2(e)
};

template <int HD, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                  const FwdParams p) {
  using C = FwdCfg<HD>;
  constexpr int NS = C::NS;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* k_full = q_full + 1;
  uint64_t* k_empty = k_full + NS;
  uint64_t* v_full = k_empty + NS;
  uint64_t* v_empty = v_full + NS;
  uint64_t* s_full = v_empty + NS;  // [2]
  uint64_t* s_empty = s_full + 2;   // [2]
  uint64_t* p_full = s_empty + 2;
  uint64_t* pv_done = p_full + 1;
  uint64_t* drain = pv_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.x;
  const int b = bh / p.Hq, h = bh - b * p.Hq;
  const int qt = gridDim.y - 1 - blockIdx.y;  // longest causal rows first
  const int q0 = qt * BM;
  const int bkv = b * p.Hkv + h / p.G;

  int nkv = p.kv_tiles;
  if (CAUSAL) {
    const int last_key = min(q0 + BM, p.Tq) - 1 + p.causal_off;  // last key the tile's last row sees
    nkv = last_key < 0 ? 0 : min(nkv, last_key / BN + 1);
  }

  if (threadIdx.x == 0) {
    *abort_flag = (smem_u32(smem) & 1023u) ? 1 : 0;  // swizzled tiles need 1024 B alignment
    mbar_init(q_full, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&s_empty[s], 128);
    }
    mbar_init(p_full, 128);
    mbar_init(pv_done, 1);
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
  const bool run = (*abort_flag == 0) && nkv > 0;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && run) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      mbar_arrive_expect_tx(q_full, C::Q_BYTES);
#pragma unroll
      for (int cb = 0; cb < HD / 64; ++cb) tma_load_3d(smem + C::OFF_Q + cb * BM * 128, &tmQ, q_full, cb * 64, q0, bh);
      int k_last[NS], v_last[NS];
#pragma unroll
      for (int s = 0; s < NS; ++s) k_last[s] = v_last[s] = -1;
      for (int j = 0; j < nkv; ++j) {
        const int s = j % NS, u = j / NS;
        if (!mbar_wait(&k_empty[s], (u & 1) ^ 1, abort_flag)) break;
        mbar_arrive_expect_tx(&k_full[s], C::KV_BYTES);
#pragma unroll
        for (int cb = 0; cb < HD / 64; ++cb)
          tma_load_3d(smem + C::OFF_K + s * C::KV_BYTES + cb * BN * 128, &tmK, &k_full[s], cb * 64, j * BN, bkv);
        k_last[s] = u;
        if (!mbar_wait(&v_empty[s], (u & 1) ^ 1, abort_flag)) break;
        mbar_arrive_expect_tx(&v_full[s], C::KV_BYTES);
#pragma unroll
        for (int cb = 0; cb < HD / 64; ++cb)
          tma_load_3d(smem + C::OFF_V + s * C::KV_BYTES + cb * BN * 128, &tmV, &v_full[s], cb * 64, j * BN, bkv);
        v_last[s] = u;
      }
      // Every issued copy must land before the CTA releases its shared memory.
      mbar_wait_bounded(q_full, 0);
#pragma unroll
      for (int s = 0; s < NS; ++s) {
        if (k_last[s] >= 0) mbar_wait_bounded(&k_full[s], k_last[s] & 1);
        if (v_last[s] >= 0) mbar_wait_bounded(&v_full[s], v_last[s] & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && run) {
      constexpr uint32_t idS = idesc_bf16(BM, BN, 0, 0);
      constexpr uint32_t idPV = idesc_bf16(BM, HD, 0, 1);
      const uint32_t tO = tmem + 256;
      const uint32_t q_base = smem_u32(smem + C::OFF_Q);
      const uint32_t k_base = smem_u32(smem + C::OFF_K);
      const uint32_t v_base = smem_u32(smem + C::OFF_V);
      const uint32_t p_base = smem_u32(smem + C::OFF_P);
      auto issue_pv = [&](int t) -> bool {
        const int s = t % NS, u = t / NS;
        if (!mbar_wait(p_full, t & 1, abort_flag)) return false;
        if (!mbar_wait(&v_full[s], u & 1, abort_flag)) return false;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < BN / 16; ++k) {
          const uint64_t a = desc_kmajor(p_base + (k >> 2) * (BM * 128) + (k & 3) * 32);
          const uint64_t bd = desc_mnmajor(v_base + s * C::KV_BYTES + k * 2048, BN * 128);
          mma_ss(tO, a, bd, idPV, (t > 0 || k > 0) ? 1u : 0u);
        }
        mma_commit(pv_done);
        mma_commit(&v_empty[s]);
        return true;
      };
      bool ok = mbar_wait(q_full, 0, abort_flag);
      if (ok) tc_fence_after();
      for (int j = 0; ok && j < nkv; ++j) {
        const int s = j % NS, u = j / NS, sb = j & 1;
        if (!mbar_wait(&k_full[s], u & 1, abort_flag)) { ok = false; break; }
        if (!mbar_wait(&s_empty[sb], ((j >> 1) & 1) ^ 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < HD / 16; ++k) {
          const uint64_t a = desc_kmajor(q_base + (k >> 2) * (BM * 128) + (k & 3) * 32);
          const uint64_t bd = desc_kmajor(k_base + s * C::KV_BYTES + (k >> 2) * (BN * 128) + (k & 3) * 32);
          mma_ss(tmem + sb * 128, a, bd, idS, k > 0 ? 1u : 0u);
        }
        mma_commit(&s_full[sb]);
        mma_commit(&k_empty[s]);
        if (j > 0 && !issue_pv(j - 1)) { ok = false; break; }
      }
      if (ok) issue_pv(nkv - 1);
      // Let every MMA issued above finish before TMEM is released.
      mma_commit(drain);
      mbar_wait_bounded(drain, 0);
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // row inside the tile == TMEM lane
    const int i = q0 + r;            // query row
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const float sl2 = p.scale_log2;
    const float NEG_INF = -__int_as_float(0x7f800000);
    float m_ref = NEG_INF;  // reference max (log2 units) the P values are taken against
    float l = 0.f;
    bool ok = run;
    uint8_t* Ps = smem + C::OFF_P;
    for (int j = 0; ok && j < nkv; ++j) {
      const int sb = j & 1;
      if (!mbar_wait(&s_full[sb], (j >> 1) & 1, abort_flag)) { ok = false; break; }
      tc_fence_after();
      uint32_t sr[BN];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c)
        tmem_ld32(tmem + sb * 128 + lane_base + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[c * 32]));
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&s_empty[sb]);
      float s[BN];
#pragma unroll
      for (int c = 0; c < BN; ++c) s[c] = __uint_as_float(sr[c]);
      const int kv0 = j * BN;
      const bool need_mask = (kv0 + BN > p.Tk) || (CAUSAL && kv0 + BN - 1 > q0 + p.causal_off);
      if (need_mask) {
        int lim = p.Tk - kv0;
        if (CAUSAL) lim = min(lim, i + p.causal_off + 1 - kv0);
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (c >= lim) s[c] = NEG_INF;
      }
      float mt = s[0];
#pragma unroll
      for (int c = 1; c < BN; ++c) mt = fmaxf(mt, s[c]);
      const float mt2 = mt * sl2;
      float m_new = m_ref;
      if (mt2 > m_ref + kRescaleThreshold) m_new = mt2;  // also taken when m_ref == -inf
      const float base = (m_new == NEG_INF) ? 0.f : m_new;
      uint32_t pk[BN / 2];
      float rowsum = 0.f;
#pragma unroll
      for (int c = 0; c < BN; c += 2) {
        const float e0 = ex2(fmaf(s[c], sl2, -base));
        const float e1 = ex2(fmaf(s[c + 1], sl2, -base));
        rowsum += e0 + e1;
        pk[c / 2] = pack_bf16x2(e0, e1);
      }
      // The previous P.V must be done before P is overwritten or O rescaled.
      if (j > 0) {
        if (!mbar_wait(pv_done, (j - 1) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
      }
      if (m_new != m_ref) {
        const float alpha = (m_ref == NEG_INF) ? 0.f : ex2(m_ref - m_new);
        l *= alpha;
        if (j > 0 && m_ref != NEG_INF) {
#pragma unroll
          for (int c = 0; c < HD / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tmem + 256 + lane_base + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(tmem + 256 + lane_base + c * 32, o);
          }
          tmem_wait_st();
        }
        m_ref = m_new;
      }
      l += rowsum;
#pragma unroll
      for (int cc = 0; cc < BN / 8; ++cc)
        st_shared_v4(smem_u32(Ps + (cc >> 3) * (BM * 128) + sw128_offset(r, cc & 7)), pk[4 * cc], pk[4 * cc + 1],
                     pk[4 * cc + 2], pk[4 * cc + 3]);
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(p_full);
    }
    // ---- epilogue: O / l -> bf16 -> shared (Q's buffer, free now) -> TMA store; L -> global
    if (ok) {
      if (!mbar_wait(pv_done, (nkv - 1) & 1, abort_flag)) ok = false;
      tc_fence_after();
    }
    // All 128 softmax threads agree on whether to write (a timeout anywhere in
    // the CTA cancels the epilogue), so the barriers below can never split.
    const bool mine = ((nkv == 0) || ok) && *abort_flag == 0;
    if (named_bar_and(1, 128, mine)) {
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      if (i < p.Tq) p.L[(size_t)bh * p.Tq + i] = l > 0.f ? (m_ref + __log2f(l)) * 0.69314718055994531f : NEG_INF;
      uint8_t* Os = smem + C::OFF_Q;
#pragma unroll
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t o[32];
        if (nkv > 0) {
          tmem_ld32(tmem + 256 + lane_base + c * 32, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0u;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t w0 = pack_bf16x2(__uint_as_float(o[8 * q + 0]) * inv_l, __uint_as_float(o[8 * q + 1]) * inv_l);
          const uint32_t w1 = pack_bf16x2(__uint_as_float(o[8 * q + 2]) * inv_l, __uint_as_float(o[8 * q + 3]) * inv_l);
          const uint32_t w2 = pack_bf16x2(__uint_as_float(o[8 * q + 4]) * inv_l, __uint_as_float(o[8 * q + 5]) * inv_l);
          const uint32_t w3 = pack_bf16x2(__uint_as_float(o[8 * q + 6]) * inv_l, __uint_as_float(o[8 * q + 7]) * inv_l);
          st_shared_v4(smem_u32(Os + (c >> 1) * (BM * 128) + sw128_offset(r, (c & 1) * 4 + q)), w0, w1, w2, w3);
        }
      }
      fence_async_smem();
      named_bar_sync(2, 128);
      if (warp == 2 && lane == 0) {
        prefetch_tmap(&tmO);
#pragma unroll
        for (int cb = 0; cb < HD / 64; ++cb) tma_store_3d(&tmO, Os + cb * BM * 128, cb * 64, q0, bh);
        bulk_commit();
        bulk_wait0();
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

template <int HD, bool CAUSAL>
cudaError_t launch_fwd_t(const fa::Problem& pr, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                         const CUtensorMap& mo, float* L, cudaStream_t stream) {
  using C = FwdCfg<HD>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(fa_fwd_kernel<HD, CAUSAL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  FwdParams p;
  p.L = L;
  p.status = fa::device_status_word();
  p.Hq = pr.Hq;
  p.Hkv = pr.Hkv;
  p.G = pr.G();
  p.Tq = pr.Tq;
  p.Tk = pr.Tk;
  p.causal_off = pr.Tk - pr.Tq;
  p.kv_tiles = pr.kv_tiles();
  p.scale_log2 = pr.scale * 1.4426950408889634f;
  dim3 grid(pr.B * pr.Hq, pr.q_tiles());
  fa_fwd_kernel<HD, CAUSAL><<<grid, kThreads, C::SMEM, stream>>>(mq, mk, mv, mo, p);
  return cudaGetLastError();
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
    const size_t words = (size_t)rows * pr.d / 2;
    fa_fwd_empty_keys<<<1216, 256, 0, stream>>>(static_cast<uint32_t*>(O), words, L, (size_t)rows);
    ++*launches;
    return cudaGetLastError();
  }
  CUtensorMap mq, mk, mv, mo;
  if (!encode_rows_bf16(&mq, Q, pr.d, pr.Tq, (long long)pr.B * pr.Hq) ||
      !encode_rows_bf16(&mk, K, pr.d, pr.Tk, (long long)pr.B * pr.Hkv) ||
      !encode_rows_bf16(&mv, V, pr.d, pr.Tk, (long long)pr.B * pr.Hkv) ||
      !encode_rows_bf16(&mo, O, pr.d, pr.Tq, (long long)pr.B * pr.Hq))
    return cudaErrorInvalidValue;
  cudaError_t e;
  if (pr.d == 64)
    e = pr.causal ? launch_fwd_t<64, true>(pr, mq, mk, mv, mo, L, stream)
                  : launch_fwd_t<64, false>(pr, mq, mk, mv, mo, L, stream);
  else
    e = pr.causal ? launch_fwd_t<128, true>(pr, mq, mk, mv, mo, L, stream)
                  : launch_fwd_t<128, false>(pr, mq, mk, mv, mo, L, stream);
  if (e == cudaSuccess) ++*launches;
  return e;
}

}  // namespace fa
