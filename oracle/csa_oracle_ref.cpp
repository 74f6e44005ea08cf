// CPU oracle of the CSA / HCA path in plain C++17, double precision -- TEST
// INFRASTRUCTURE ONLY (the tests, the smoke check and the benchmark's CPU
// baseline may call it; the CUDA library never does and shares no code with
// it).  Each function restates its definition in order, in loops:
//
// "DeepSeek V4 technical review" (takeshell.com), section 2.1 CSA: each
// compressed entry is a weighted sum over m tokens; the indexer rates the
// compressed entries for each query and keeps the k best; attention runs over
// those entries only.  Section 2.2 HCA: m' = 128, every entry attended.
// Octagono "Hybrid Attention: CSA and HCA": a window over the most recent raw
// tokens is attended together with the selected entries.  The workload
// specification fixes the compressor (per-channel softmax of the gate logits
// times the raw vectors), the score sum_h w_h ReLU(q_h . k), the lowest-index
// tie rule, the visibility (b+1) m - 1 <= t and the scale 1/sqrt(d).
//
// Built by the repository's build step as oracle/liboracle_ref.so; called
// through oracle/ref_cpp.py.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <limits>
#include <numeric>
#include <vector>

extern "C" {

// Block compression of one stream x [T][D] with gate logits g [T][D]:
// out[b][c] = sum_j softmax_j(g[b m + j][c]) x[b m + j][c], j < m; the T mod m
// trailing tokens are dropped.  Returns the number of entries T / m.
int oref_compress(const double* x, const double* g, int T, int D, int m, double* out) {
  const int nb = T / m;
  for (int b = 0; b < nb; ++b) {
    for (int c = 0; c < D; ++c) {
      double mx = -std::numeric_limits<double>::infinity();
      for (int j = 0; j < m; ++j) mx = std::max(mx, g[static_cast<size_t>(b * m + j) * D + c]);
      double den = 0.0, num = 0.0;
      for (int j = 0; j < m; ++j) {
        const size_t i = static_cast<size_t>(b * m + j) * D + c;
        const double p = std::exp(g[i] - mx);
        den += p;
        num += p * x[i];
      }
      out[static_cast<size_t>(b) * D + c] = num / den;
    }
  }
  return nb;
}

// Visible blocks at position t: block b (tokens b m .. b m + m - 1) is visible
// iff (b + 1) m - 1 <= t, at most N of them.
int oref_n_visible(int t, int m, int N) {
  const int n = (t + 1) / m;
  return std::max(0, std::min(N, n));
}

// Indexer scores of one query: S[b] = sum_h w[h] ReLU(q[h] . k[b]) for the
// visible blocks.  q [H][dI], k [N][dI], w [H].  Returns n_vis.
int oref_indexer_scores(const double* q, const double* k, const double* w, int H, int dI, int N, int t, int m,
                        double* S) {
  const int n = oref_n_visible(t, m, N);
  for (int b = 0; b < n; ++b) {
    double s = 0.0;
    for (int h = 0; h < H; ++h) {
      double dot = 0.0;
      for (int c = 0; c < dI; ++c) dot += q[static_cast<size_t>(h) * dI + c] * k[static_cast<size_t>(b) * dI + c];
      s += w[h] * std::max(dot, 0.0);
    }
    S[b] = s;
  }
  return n;
}

// Top-k of n scores: the min(k, n) largest, equal scores to the lower index;
// out [k] holds the kept indices ascending, then -1.
void oref_topk(const double* S, int n, int k, int32_t* out) {
  std::vector<int> order(n);
  std::iota(order.begin(), order.end(), 0);
  std::sort(order.begin(), order.end(), [&](int a, int b) { return S[a] > S[b] || (S[a] == S[b] && a < b); });
  const int kept = std::min(k, n);
  std::sort(order.begin(), order.begin() + kept);
  for (int i = 0; i < k; ++i) out[i] = i < kept ? order[i] : -1;
}

// Attention of one query (all heads) over one softmax of the keys
// k_cmp[sel[i]] (sel[i] >= 0) followed by the window rows k_raw[win[i]]:
// O[h] = sum_j softmax_j(scale q[h] . K_j) V_j, lse[h] = log sum_j exp(.).
// q [H][d]; k_cmp, v_cmp [*][d]; k_raw, v_raw [*][d].  No key: O = 0,
// lse = -inf.
void oref_attend_one(const double* q, int H, int d, const double* k_cmp, const double* v_cmp, const int32_t* sel,
                     int n_sel, const double* k_raw, const double* v_raw, const int32_t* win, int n_win,
                     double scale, double* O, double* lse) {
  std::vector<const double*> K, V;
  for (int i = 0; i < n_sel; ++i)
    if (sel[i] >= 0) {
      K.push_back(k_cmp + static_cast<size_t>(sel[i]) * d);
      V.push_back(v_cmp + static_cast<size_t>(sel[i]) * d);
    }
  for (int i = 0; i < n_win; ++i) {
    K.push_back(k_raw + static_cast<size_t>(win[i]) * d);
    V.push_back(v_raw + static_cast<size_t>(win[i]) * d);
  }
  const size_t L = K.size();
  std::vector<double> s(L);
  for (int h = 0; h < H; ++h) {
    double* o = O + static_cast<size_t>(h) * d;
    std::fill(o, o + d, 0.0);
    if (L == 0) {
      lse[h] = -std::numeric_limits<double>::infinity();
      continue;
    }
    double mx = -std::numeric_limits<double>::infinity();
    for (size_t j = 0; j < L; ++j) {
      double dot = 0.0;
      for (int c = 0; c < d; ++c) dot += q[static_cast<size_t>(h) * d + c] * K[j][c];
      s[j] = scale * dot;
      mx = std::max(mx, s[j]);
    }
    double den = 0.0;
    for (size_t j = 0; j < L; ++j) {
      const double p = std::exp(s[j] - mx);
      den += p;
      for (int c = 0; c < d; ++c) o[c] += p * V[j][c];
    }
    for (int c = 0; c < d; ++c) o[c] /= den;
    lse[h] = mx + std::log(den);
  }
}

}  // extern "C"
