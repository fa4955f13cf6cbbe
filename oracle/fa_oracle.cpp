// Float64 CPU oracle for tiled exact attention (forward + recompute backward).
//
// TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
// load this file; only the tests, the smoke check and the benchmark's CPU
// baseline leg use it.  It shares no code, header or constant with the CUDA
// library.
//
// What it computes is the plain definition of attention, not the tiled
// algorithm ("What Ordinary Autograd Saves", section "The implementation
// under test": `dense_attention` = softmax(Q K^T / sqrt(d)) V; "Backward Pass
// Implementation", section "Limitations of PyTorch Autograd", the three-line
// `standard_attention`).  Per (batch b, query head h), with key/value head
// kvh = h / (Hq / Hkv) (the repeat_interleave grouping of "The Autograd
// Memory Trap", section "The GQA Expansion Question"), row by row:
//
//   s_j  = scale * q_i . k_j          for every visible key j
//   m    = max_j s_j,  l = sum_j exp(s_j - m)
//   p_j  = exp(s_j - m) / l
//   O_i  = sum_j p_j v_j
//   L_i  = m + ln l                   (natural-log logsumexp of the scaled
//                                      scores: the row statistic L that the
//                                      tiled forward returns as `mi + log(li)`)
//
// Visible keys: j < Tk, and with causal masking j <= i + (Tk - Tq)
// (bottom-right alignment; identical to top-left when Tq == Tk).  With a
// sliding window of W >= 1 keys (causal only; the local-attention layers of
// "The Autograd Memory Trap", section "Assumptions and Uncertainties", item 3,
// which see a bounded number of keys), also j > i + (Tk - Tq) - W: the row sees
// at most its last W keys.  A row with no visible key gets O_i = 0,
// L_i = -inf and no gradient.
//
// Backward, derived by hand from the softmax Jacobian dp_j/ds_k = p_j(d_jk - p_k)
// for a loss with upstream gradient dO (no equations survive on the pages;
// this is the derivation written out):
//   dP_ij = dO_i . v_j
//   D_i   = sum_j p_ij dP_ij
//   dS_ij = p_ij (dP_ij - D_i)
//   dQ_i  = scale * sum_j dS_ij k_j
//   dK_j += scale * dS_ij q_i         (summed over every query head of the group)
//   dV_j += p_ij dO_i                 (likewise)
//
// All arithmetic is IEEE double.  Layouts: Q [B,Hq,Tq,d], K [B,Hkv,Tk,d],
// V [B,Hkv,Tk,dv], O/dO [B,Hq,Tq,dv], L/D [B,Hq,Tq], row-major contiguous.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

struct Dims {
  int B, Hq, Hkv, Tq, Tk, d, dv, causal, window;
  double scale;
};

// Last visible key index + 1 for query row i.
inline int64_t visible_end(const Dims& z, int64_t i) {
  if (!z.causal) return z.Tk;
  int64_t e = i + (int64_t)(z.Tk - z.Tq) + 1;
  if (e < 0) e = 0;
  if (e > z.Tk) e = z.Tk;
  return e;
}

// First visible key index for query row i (0 unless a sliding window is set).
inline int64_t visible_begin(const Dims& z, int64_t i) {
  if (!z.causal || z.window <= 0) return 0;
  int64_t b = i + (int64_t)(z.Tk - z.Tq) - z.window + 1;
  return b < 0 ? 0 : b;
}

// Scores, probabilities and logsumexp of one query row.  Visible keys are
// [j0, n); returns n with p[j0..n) filled, *j0 set, *lse set (-inf when the
// range is empty).
int64_t row_probs(const Dims& z, const double* q, const double* Kh, int64_t i, double* p, double* lse,
                  int64_t* j0) {
  const int64_t n = visible_end(z, i);
  *j0 = visible_begin(z, i);
  if (*j0 >= n) {
    *lse = -std::numeric_limits<double>::infinity();
    *j0 = n;
    return n;
  }
  double m = -std::numeric_limits<double>::infinity();
  for (int64_t j = *j0; j < n; ++j) {
    const double* k = Kh + j * z.d;
    double s = 0.0;
    for (int c = 0; c < z.d; ++c) s += q[c] * k[c];
    s *= z.scale;
    p[j] = s;
    if (s > m) m = s;
  }
  double l = 0.0;
  for (int64_t j = *j0; j < n; ++j) {
    p[j] = std::exp(p[j] - m);
    l += p[j];
  }
  for (int64_t j = *j0; j < n; ++j) p[j] /= l;
  *lse = m + std::log(l);
  return n;
}

}  // namespace

extern "C" {

// Forward on rows [row_lo, row_hi) of every (b, h); other rows of O and L are
// left untouched.  nthreads <= 0 uses the OpenMP default.
void fa_oracle_forward(const double* Q, const double* K, const double* V, int B, int Hq, int Hkv, int Tq, int Tk,
                       int d, int dv, int causal, int window, double scale, int row_lo, int row_hi, double* O,
                       double* L, int nthreads) {
  const Dims z{B, Hq, Hkv, Tq, Tk, d, dv, causal, window, scale};
  const int G = Hq / Hkv;
  if (row_lo < 0) row_lo = 0;
  if (row_hi > Tq) row_hi = Tq;
  const int64_t nrows = row_hi > row_lo ? row_hi - row_lo : 0;
  const int64_t total = (int64_t)B * Hq * nrows;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel
#endif
  {
    std::vector<double> p(Tk > 0 ? Tk : 1);
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 8)
#endif
    for (int64_t t = 0; t < total; ++t) {
      const int64_t bh = t / nrows, i = row_lo + t % nrows;
      const int64_t b = bh / Hq, h = bh % Hq, kvh = h / G;
      const double* q = Q + ((b * Hq + h) * (int64_t)Tq + i) * d;
      const double* Kh = K + (b * Hkv + kvh) * (int64_t)Tk * d;
      const double* Vh = V + (b * Hkv + kvh) * (int64_t)Tk * dv;
      double* o = O + ((b * Hq + h) * (int64_t)Tq + i) * dv;
      double lse;
      int64_t j0;
      const int64_t n = row_probs(z, q, Kh, i, p.data(), &lse, &j0);
      for (int c = 0; c < dv; ++c) o[c] = 0.0;
      for (int64_t j = j0; j < n; ++j) {
        const double* v = Vh + j * dv;
        for (int c = 0; c < dv; ++c) o[c] += p[j] * v[c];
      }
      L[(b * Hq + h) * (int64_t)Tq + i] = lse;
    }
  }
}

// Full backward for every (b, h).  dQ [B,Hq,Tq,d], dK [B,Hkv,Tk,d],
// dV [B,Hkv,Tk,dv] are overwritten.  D_out (nullable) receives D_i.
void fa_oracle_backward(const double* Q, const double* K, const double* V, const double* dO, int B, int Hq, int Hkv,
                        int Tq, int Tk, int d, int dv, int causal, int window, double scale, double* dQ, double* dK,
                        double* dV, double* D_out, int nthreads) {
  const Dims z{B, Hq, Hkv, Tq, Tk, d, dv, causal, window, scale};
  const int G = Hq / Hkv;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
  std::memset(dQ, 0, sizeof(double) * (size_t)B * Hq * Tq * d);
  std::memset(dK, 0, sizeof(double) * (size_t)B * Hkv * Tk * d);
  std::memset(dV, 0, sizeof(double) * (size_t)B * Hkv * Tk * dv);
  // One (b, kv-head) group at a time; its G*Tq query rows are spread over the
  // threads, each thread summing dK/dV into a private buffer that is added to
  // the group's slice at the end.
  for (int64_t grp = 0; grp < (int64_t)B * Hkv; ++grp) {
    const int64_t b = grp / Hkv, kvh = grp % Hkv;
    const double* Kh = K + grp * (int64_t)Tk * d;
    const double* Vh = V + grp * (int64_t)Tk * dv;
    double* dKh = dK + grp * (int64_t)Tk * d;
    double* dVh = dV + grp * (int64_t)Tk * dv;
    const int64_t rows = (int64_t)G * Tq;
#ifdef _OPENMP
#pragma omp parallel
#endif
    {
      std::vector<double> p(Tk > 0 ? Tk : 1), dP(Tk > 0 ? Tk : 1);
      std::vector<double> dKp((size_t)Tk * d, 0.0), dVp((size_t)Tk * dv, 0.0);
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 4)
#endif
      for (int64_t t = 0; t < rows; ++t) {
        const int64_t h = kvh * G + t / Tq, i = t % Tq;
        const int64_t row = (b * Hq + h) * (int64_t)Tq + i;
        const double* q = Q + row * d;
        const double* g = dO + row * dv;
        double lse;
        int64_t j0;
        const int64_t n = row_probs(z, q, Kh, i, p.data(), &lse, &j0);
        double Di = 0.0;
        for (int64_t j = j0; j < n; ++j) {
          const double* v = Vh + j * dv;
          double s = 0.0;
          for (int c = 0; c < dv; ++c) s += g[c] * v[c];
          dP[j] = s;
          Di += p[j] * s;
        }
        if (D_out) D_out[row] = Di;
        double* dq = dQ + row * d;
        for (int64_t j = j0; j < n; ++j) {
          const double dS = p[j] * (dP[j] - Di);
          const double* k = Kh + j * d;
          double* dk = dKp.data() + j * d;
          double* dvv = dVp.data() + j * dv;
          for (int c = 0; c < d; ++c) {
            dq[c] += scale * dS * k[c];
            dk[c] += scale * dS * q[c];
          }
          for (int c = 0; c < dv; ++c) dvv[c] += p[j] * g[c];
        }
      }
#ifdef _OPENMP
#pragma omp critical
#endif
      {
        for (size_t e = 0; e < dKp.size(); ++e) dKh[e] += dKp[e];
        for (size_t e = 0; e < dVp.size(); ++e) dVh[e] += dVp[e];
      }
    }
  }
}

// Bytes each strategy keeps alive for the backward pass, per attention call
// ("What Ordinary Autograd Saves", sections "The measurement" and "Why this is
// FlashAttention's second idea"):
//   dense autograd: Q, K, V plus the Tq x Tk softmax output of every head;
//   checkpointed:   Q, K, V only;
//   custom backward (this method): Q, K, V plus O and the row statistic L.
// elem_bytes: size of one Q/K/V/O element; stat_bytes: size of one L element;
// prob_bytes: size of one softmax-output element.
int64_t fa_oracle_saved_bytes(int strategy, int B, int Hq, int Hkv, int Tq, int Tk, int d, int dv, int elem_bytes,
                              int stat_bytes, int prob_bytes) {
  const int64_t qkv = ((int64_t)B * Hq * Tq * d + (int64_t)B * Hkv * Tk * d + (int64_t)B * Hkv * Tk * dv) * elem_bytes;
  switch (strategy) {
    case 0:  // dense
      return qkv + (int64_t)B * Hq * Tq * Tk * prob_bytes;
    case 1:  // checkpointed
      return qkv;
    case 2:  // keep O and L
      return qkv + (int64_t)B * Hq * Tq * dv * elem_bytes + (int64_t)B * Hq * Tq * stat_bytes;
    default:
      return -1;
  }
}

int fa_oracle_abi_version(void) { return 1; }

}  // extern "C"
