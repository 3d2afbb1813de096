// fp64 CPU oracle for exact softmax attention and its gradients.
//
// TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call
// this file: only the tests, the smoke check and the CPU-baseline leg of the
// benchmark use it. It shares no code, header, table or helper with the CUDA
// library under exact_io_aware_27_gb300/csrc.
//
// What it computes, and where the pages define it:
//  * standard attention  S = Q K^T * scale, causal mask "key k visible from
//    query q iff k <= q" (top-left), P = softmax(S) row-wise, O = P V
//    -- "05_flash_attention.py" (page 1), function standard_attention;
//    the softmax formula exp(x - max x) / sum exp(x - max x) is the one the
//    CSDN post (page 2) states under "block normalisation".
//  * logsumexp L_i = m_i + log l_i, natural log -- page 1,
//    flash_attention_forward docstring ("L_i = m_i + log(l_i)").
//  * gradients of a scalar loss with upstream dO:  dV = P^T dO,
//    dP = dO V^T, D_i = sum_j P_ij dP_ij, dS = P o (dP - D),
//    dQ = dS K * scale, dK = dS^T Q * scale -- page 1,
//    flash_attention_backward docstring; the two matrix-calculus rules
//    (O = PV and P = softmax(S)) in "Flash Attention" notes (page 3),
//    section 1.5 "Matrix Calculus Cheatsheet".
//  * the score and probability matrices themselves (S and P of standard
//    attention, which the materialised baseline writes to memory) -- page 1,
//    standard_attention.
//  * the online (one-pass) max / rescaled-sum recurrence -- page 1,
//    online_softmax_stats; page 3, section 1.1 "Online Softmax".
//
// Everything is evaluated directly from those definitions in double precision:
// a full score row per query, a two-pass max / log-sum-exp, no tiling and no
// fusion. D is computed from its definition sum_j P_ij dP_ij, not from the
// rowsum(dO o O) shortcut (the tests check that identity separately).
// dQ is formed query row by query row and dK, dV key row by key row, each
// recomputing P_ij from the same definitions, so no reduction across threads
// is needed. The *_rows variants evaluate the same definitions on a chosen
// subset of query / key rows (used for the long workloads); the full
// functions are those variants called with every row.
//
// All arrays are one head, row-major: Q, dO, O, dQ are n x d; K, V, dK, dV are
// m x d; L and D have n entries.

#include <cmath>
#include <cstdlib>
#include <cstring>
#include <limits>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

const double kNegInf = -std::numeric_limits<double>::infinity();

// Score s_ij = scale * <Q_i, K_j>, or -inf where the causal mask hides key j
// from query i (j > i).
double score(const double* Q, const double* K, long d, long i, long j, int causal,
             double scale) {
  if (causal && j > i) return kNegInf;
  double acc = 0.0;
  for (long c = 0; c < d; ++c) acc += Q[i * d + c] * K[j * d + c];
  return scale * acc;
}

// Direct two-pass log-sum-exp of one score row: max first, then the sum of
// exp(s - max). Returns the natural-log value L_i.
double row_logsumexp(const double* s, long m) {
  double mx = kNegInf;
  for (long j = 0; j < m; ++j)
    if (s[j] > mx) mx = s[j];
  double sum = 0.0;
  for (long j = 0; j < m; ++j) sum += std::exp(s[j] - mx);
  return mx + std::log(sum);
}

}  // namespace

extern "C" {

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void oracle_set_num_threads(int t) {
#ifdef _OPENMP
  if (t > 0) omp_set_num_threads(t);
#else
  (void)t;
#endif
}

// One-pass running statistics over x[0..len) read `block` entries at a time:
//   m_new = max(m, max(chunk));  l = l * exp(m - m_new) + sum exp(chunk - m_new)
// starting from m = -inf, l = 0. block = 1 is the per-element form of page 3.
// Afterwards softmax(x)_i = exp(x_i - m) / l and logsumexp(x) = m + log l.
int oracle_online_softmax_stats(const double* x, long len, long block, double* m_out,
                                double* l_out) {
  if (!x || !m_out || !l_out || len < 1 || block < 1) return -1;
  double m = kNegInf, l = 0.0;
  for (long s = 0; s < len; s += block) {
    long e = s + block < len ? s + block : len;
    double cmax = kNegInf;
    for (long i = s; i < e; ++i)
      if (x[i] > cmax) cmax = x[i];
    double m_new = m > cmax ? m : cmax;
    double csum = 0.0;
    for (long i = s; i < e; ++i) csum += std::exp(x[i] - m_new);
    // exp(-inf - finite) = 0 on the first chunk, so l starts from the chunk sum.
    l = l * std::exp(m - m_new) + csum;
    m = m_new;
  }
  *m_out = m;
  *l_out = l;
  return 0;
}

// Forward of one head on selected query rows: for r < nrows, row rows[r] of
// O goes to O[r * d ...] and its natural-log logsumexp to L[r].
int oracle_attention_forward_rows(const double* Q, const double* K, const double* V, long n,
                                  long m, long d, int causal, double scale, const long* rows,
                                  long nrows, double* O, double* L) {
  if (!Q || !K || !V || !O || !L || !rows || n < 1 || m < 1 || d < 1 || nrows < 0) return -1;
  for (long r = 0; r < nrows; ++r)
    if (rows[r] < 0 || rows[r] >= n) return -1;
#pragma omp parallel
  {
    std::vector<double> s(m);
#pragma omp for schedule(dynamic, 4)
    for (long r = 0; r < nrows; ++r) {
      const long i = rows[r];
      for (long j = 0; j < m; ++j) s[j] = score(Q, K, d, i, j, causal, scale);
      const double Li = row_logsumexp(s.data(), m);
      L[r] = Li;
      double* Oi = O + r * d;
      for (long c = 0; c < d; ++c) Oi[c] = 0.0;
      for (long j = 0; j < m; ++j) {
        if (s[j] == kNegInf) continue;  // P_ij = 0 exactly
        const double p = std::exp(s[j] - Li);
        for (long c = 0; c < d; ++c) Oi[c] += p * V[j * d + c];
      }
    }
  }
  return 0;
}

// The intermediates of standard attention for one head ("05_flash_attention.py",
// standard_attention): the score matrix S (n x m; -inf where the causal mask
// hides a key) and P = softmax(S) row-wise (n x m; 0 where hidden), each row's
// P_ij = exp(s_ij - L_i) with L_i the row's direct log-sum-exp.
int oracle_attention_probabilities(const double* Q, const double* K, long n, long m, long d,
                                   int causal, double scale, double* S, double* P) {
  if (!Q || !K || !S || !P || n < 1 || m < 1 || d < 1) return -1;
#pragma omp parallel for schedule(dynamic, 4)
  for (long i = 0; i < n; ++i) {
    double* si = S + i * m;
    for (long j = 0; j < m; ++j) si[j] = score(Q, K, d, i, j, causal, scale);
    const double Li = row_logsumexp(si, m);
    for (long j = 0; j < m; ++j) P[i * m + j] = si[j] == kNegInf ? 0.0 : std::exp(si[j] - Li);
  }
  return 0;
}

// Forward of one head: O (n x d) and natural-log logsumexp L (n).
int oracle_attention_forward(const double* Q, const double* K, const double* V, long n,
                             long m, long d, int causal, double scale, double* O, double* L) {
  if (n < 1) return -1;
  std::vector<long> all(n);
  for (long i = 0; i < n; ++i) all[i] = i;
  return oracle_attention_forward_rows(Q, K, V, n, m, d, causal, scale, all.data(), n, O, L);
}

// Backward of one head for the scalar f = sum(O o dO), evaluated on selected
// rows: dQ for query rows qrows[0..nq) (into dQ[r * d ...]) and dK, dV for key
// rows krows[0..nk). D_out (n entries, all rows) receives D_i = sum_j P_ij dP_ij
// when not NULL. L_i and D_i are always formed for every query row, since each
// key's gradient sums over all of them.
int oracle_attention_backward_rows(const double* Q, const double* K, const double* V,
                                   const double* dO, long n, long m, long d, int causal,
                                   double scale, const long* qrows, long nq, const long* krows,
                                   long nk, double* dQ, double* dK, double* dV, double* D_out) {
  if (!Q || !K || !V || !dO || n < 1 || m < 1 || d < 1 || nq < 0 || nk < 0) return -1;
  if ((nq > 0 && (!qrows || !dQ)) || (nk > 0 && (!krows || !dK || !dV))) return -1;
  for (long r = 0; r < nq; ++r)
    if (qrows[r] < 0 || qrows[r] >= n) return -1;
  for (long r = 0; r < nk; ++r)
    if (krows[r] < 0 || krows[r] >= m) return -1;
  std::vector<double> Lrow(n), Drow(n);

  // Pass 1, every query row: L_i and D_i = sum_j P_ij dP_ij, dP_ij = <dO_i, V_j>.
#pragma omp parallel
  {
    std::vector<double> s(m);
#pragma omp for schedule(dynamic, 4)
    for (long i = 0; i < n; ++i) {
      for (long j = 0; j < m; ++j) s[j] = score(Q, K, d, i, j, causal, scale);
      const double Li = row_logsumexp(s.data(), m);
      double Di = 0.0;
      for (long j = 0; j < m; ++j) {
        if (s[j] == kNegInf) continue;
        const double p = std::exp(s[j] - Li);
        double dp = 0.0;
        for (long c = 0; c < d; ++c) dp += dO[i * d + c] * V[j * d + c];
        Di += p * dp;
      }
      Lrow[i] = Li;
      Drow[i] = Di;
    }
  }

  // Selected query rows: dQ_i = scale * sum_j dS_ij K_j, dS_ij = P_ij (dP_ij - D_i).
#pragma omp parallel for schedule(dynamic, 4)
  for (long r = 0; r < nq; ++r) {
    const long i = qrows[r];
    double* dQi = dQ + r * d;
    for (long c = 0; c < d; ++c) dQi[c] = 0.0;
    for (long j = 0; j < m; ++j) {
      const double sij = score(Q, K, d, i, j, causal, scale);
      if (sij == kNegInf) continue;
      const double p = std::exp(sij - Lrow[i]);
      double dp = 0.0;
      for (long c = 0; c < d; ++c) dp += dO[i * d + c] * V[j * d + c];
      const double dS = p * (dp - Drow[i]);
      for (long c = 0; c < d; ++c) dQi[c] += scale * dS * K[j * d + c];
    }
  }

  // Selected key rows: dV_j = sum_i P_ij dO_i and dK_j = scale * sum_i dS_ij Q_i.
#pragma omp parallel for schedule(dynamic, 4)
  for (long r = 0; r < nk; ++r) {
    const long j = krows[r];
    double* dKj = dK + r * d;
    double* dVj = dV + r * d;
    for (long c = 0; c < d; ++c) dKj[c] = dVj[c] = 0.0;
    for (long i = 0; i < n; ++i) {
      const double sij = score(Q, K, d, i, j, causal, scale);
      if (sij == kNegInf) continue;
      const double p = std::exp(sij - Lrow[i]);
      double dp = 0.0;
      for (long c = 0; c < d; ++c) dp += dO[i * d + c] * V[j * d + c];
      const double dS = p * (dp - Drow[i]);
      for (long c = 0; c < d; ++c) {
        dVj[c] += p * dO[i * d + c];
        dKj[c] += scale * dS * Q[i * d + c];
      }
    }
  }
  if (D_out) std::memcpy(D_out, Drow.data(), sizeof(double) * n);
  return 0;
}

// Backward of one head for the scalar f = sum(O o dO): dQ (n x d), dK, dV (m x d).
int oracle_attention_backward(const double* Q, const double* K, const double* V,
                              const double* dO, long n, long m, long d, int causal,
                              double scale, double* dQ, double* dK, double* dV,
                              double* D_out) {
  if (n < 1 || m < 1) return -1;
  std::vector<long> qa(n), ka(m);
  for (long i = 0; i < n; ++i) qa[i] = i;
  for (long j = 0; j < m; ++j) ka[j] = j;
  return oracle_attention_backward_rows(Q, K, V, dO, n, m, d, causal, scale, qa.data(), n,
                                        ka.data(), m, dQ, dK, dV, D_out);
}

}  // extern "C"
