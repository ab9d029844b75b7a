// MiTA forward oracle -- TEST INFRASTRUCTURE ONLY.
//
// A plain, slow, fp64 CPU restatement of the Mixture-of-Top-k Attention
// forward pass.  Only the tests, the smoke check and the bench's CPU-baseline
// leg may load it.  It shares no code, header or constant with the CUDA
// library; it reads the same (already rounded) Q, K, V the GPU sees and widens
// them exactly to double.
//
// Sources (cited per function below):
//   [TUT]  MiTA tutorial, iwxt.cn/tutorials/mita-attention (8 chapters; the
//          chapter 4 step list restates paper Sec. 3.2, eq. 5-12).
//   [GIST] gist.science summary of arXiv 2602.01219, Sec. 2.2-2.3
//          (Algorithm 1).
//   [NEWS] bit.fan news article on MiTA, section on expert construction
//          (Algorithm 1: group queries by routing result, online softmax).
//
// Readings where the pages are silent (all listed in the design notes):
//   * scores use the same 1/sqrt(d) scaling for shared and raw pairs
//     ([TUT] ch. 5 and ch. 8 caveat 3); on request the joint softmax's shared
//     logits take 1/d instead, q . q~ / d, the temperature [TUT] ch. 8 caveat 3
//     reads out of the official code (raw logits and the landmark softmax
//     behind v~ keep 1/sqrt(d));
//   * top-k and top-s order is (score descending, index ascending), so ties go
//     to the lowest index; expert index lists are stored ascending;
//   * the landmark queries are materialised in the input dtype: an fp64 window
//     mean rounded once (round-to-nearest-even);
//   * 2D pooling uses the adaptive-average-pool window rule, the landmark grid
//     is sqrt(m) x sqrt(m) unless a grid of mh x mw = m landmarks is given; 1D
//     pooling (grid_h == 1) uses the same rule on a 1 x N grid pooled to 1 x m;
//   * no mask, no dropout, no special self term.
//
// Parity pins: every function is pinned by tests that do not call back into
// this file's arithmetic (worked counterexample, brute-force sorts, textbook
// dense attention, adaptive_avg_pool2d, merge identity, convex hull).
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <numeric>
#include <utility>
#include <vector>

#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

enum DType { DT_F32 = 0, DT_BF16 = 1, DT_F64 = 2 };

// Exact widening of one stored element to double.
double widen(const void* p, int dt, size_t i) {
  if (dt == DT_F32) return (double)((const float*)p)[i];
  if (dt == DT_BF16) {
    uint32_t bits = (uint32_t)((const uint16_t*)p)[i] << 16;
    float f;
    std::memcpy(&f, &bits, 4);
    return (double)f;
  }
  return ((const double*)p)[i];
}

// Round a double once to the nearest bfloat16 (ties to even) and return that
// value as a double.  bfloat16 keeps 8 significant bits, min exponent -126,
// subnormal quantum 2^-133.
double round_to_bf16(double x) {
  if (x == 0.0 || !std::isfinite(x)) return x;
  int e;
  std::frexp(x, &e);            // |x| = f * 2^e, f in [0.5, 1)
  int q = e - 8;                // quantum for 8 significant bits
  if (q < -133) q = -133;       // subnormal range
  double r = std::nearbyint(std::ldexp(x, -q));  // default mode: ties to even
  double y = std::ldexp(r, q);
  if (std::fabs(y) >= std::ldexp(1.0, 128)) return std::copysign(INFINITY, x);
  return y;
}

double round_to_dtype(double x, int dt) {
  if (dt == DT_BF16) return round_to_bf16(x);
  if (dt == DT_F32) return (double)(float)x;
  return x;
}

// Half-open adaptive window [floor(i*in/out), ceil((i+1)*in/out)).
void window(long i, long in, long out, long* lo, long* hi) {
  *lo = (i * in) / out;
  *hi = ((i + 1) * in + out - 1) / out;
}

int isqrt_exact(int m) {
  int r = (int)std::lround(std::sqrt((double)m));
  return (r * r == m) ? r : -1;
}

// Lexicographic "better than": higher score, then lower index.
struct Better {
  const double* s;
  bool operator()(int a, int b) const {
    if (s[a] != s[b]) return s[a] > s[b];
    return a < b;
  }
};

double dot(const void* a, int dta, size_t oa, const void* b, int dtb, size_t ob,
           int d) {
  double acc = 0.0;
  for (int l = 0; l < d; ++l) acc += widen(a, dta, oa + l) * widen(b, dtb, ob + l);
  return acc;
}

}  // namespace

extern "C" {

// Step 1, landmark queries: average-pool Q into m landmark queries.
// [TUT] ch. 4 step 1 (paper eq. 5): each landmark is the mean of a group of
// queries (not of keys); [NEWS]: "local average pooling"; [TUT] ch. 5 pools a
// 2 x 4 token grid in 2D.  Output is rounded once to `out_dt` and returned as
// doubles in q_tilde[B, H, m, d].
// Pooling onto an explicit mh x mw landmark grid (row-major landmark index).
int orc_pool_grid(const void* q, int dt, int B, int H, int N, int d, int grid_h,
                  int grid_w, int mh, int mw, int out_dt, double* q_tilde) {
  if ((long)grid_h * grid_w != N || mh < 1 || mw < 1) return 1;
  const int m = mh * mw;
#pragma omp parallel for collapse(2) schedule(static)
  for (int bh = 0; bh < B * H; ++bh) {
    for (int i = 0; i < m; ++i) {
      long r0, r1, c0, c1;
      window(i / mw, grid_h, mh, &r0, &r1);
      window(i % mw, grid_w, mw, &c0, &c1);
      double cnt = (double)((r1 - r0) * (c1 - c0));
      for (int l = 0; l < d; ++l) {
        double sum = 0.0;
        for (long r = r0; r < r1; ++r)
          for (long c = c0; c < c1; ++c)
            sum += widen(q, dt, ((size_t)bh * N + (size_t)(r * grid_w + c)) * d + l);
        q_tilde[((size_t)bh * m + i) * d + l] = round_to_dtype(sum / cnt, out_dt);
      }
    }
  }
  return 0;
}

int orc_pool(const void* q, int dt, int B, int H, int N, int d, int grid_h,
             int grid_w, int m, int out_dt, double* q_tilde) {
  if ((long)grid_h * grid_w != N || m < 1 || m > N) return 1;
  int mh = 1, mw = m;
  if (grid_h != 1) {
    int r = isqrt_exact(m);
    if (r < 0) return 1;
    mh = mw = r;
  }
  return orc_pool_grid(q, dt, B, H, N, d, grid_h, grid_w, mh, mw, out_dt, q_tilde);
}

// Steps 2-3 for a list of landmark rows (flat row id = bh * m + i).
// [TUT] ch. 4 step 2 (eq. 6-7): s_ij = q~_i . k_j / sqrt(d) over all N keys,
// the top-k keys form routed expert i ([NEWS]: experts may overlap and span
// any positions).  [TUT] ch. 4 step 3 (eq. 8-9): the same N scores, softmax,
// weight all of V -> v~_i (not an average over the top-k only).
// Outputs per row: topk_idx[k] ascending, v_tilde[d], gap = (s_(k) - s_(k+1))
// / max_j |s_j| (the relative margin at the selection boundary; 1e300 when
// k == N).
int orc_landmark_rows(const double* q_tilde, const void* k, const void* v,
                      int dt, int B, int H, int N, int d, int m, int topk,
                      long nrows, const int64_t* rows, int32_t* topk_idx,
                      double* v_tilde, double* gap) {
  (void)B; (void)H;
  if (topk < 1 || topk > N) return 1;
  const double sqrt_d = std::sqrt((double)d);
  // requested rows grouped by head, so each head's K and V are widened once
  std::vector<std::pair<long, long>> order(nrows);  // (head, position in request)
  for (long r = 0; r < nrows; ++r) order[r] = {(rows ? rows[r] : r) / m, r};
  std::sort(order.begin(), order.end());
  std::vector<double> kd((size_t)N * d), vd((size_t)N * d);
  for (long g0 = 0; g0 < nrows;) {
    long g1 = g0;
    const long bh = order[g0].first;
    while (g1 < nrows && order[g1].first == bh) ++g1;
    const size_t kv0 = (size_t)bh * N * d;
#pragma omp parallel for schedule(static)
    for (long t = 0; t < (long)N * d; ++t) {
      kd[t] = widen(k, dt, kv0 + t);
      vd[t] = widen(v, dt, kv0 + t);
    }
#pragma omp parallel
    {
      std::vector<double> s(N);
      std::vector<int> ord(N);
      std::vector<double> acc(d);
#pragma omp for schedule(dynamic, 1)
      for (long g = g0; g < g1; ++g) {
        const long r = order[g].second;
        const long row = rows ? rows[r] : r;
        const double* qt = q_tilde + (size_t)row * d;
        double smax = -INFINITY, amax = 0.0;
        for (int j = 0; j < N; ++j) {
          const double* kr = kd.data() + (size_t)j * d;
          double a = 0.0;
          for (int l = 0; l < d; ++l) a += qt[l] * kr[l];
          s[j] = a / sqrt_d;
          smax = std::max(smax, s[j]);
          amax = std::max(amax, std::fabs(s[j]));
        }
        // Top-k selection with the (score desc, index asc) order.
        std::iota(ord.begin(), ord.end(), 0);
        Better better{s.data()};
        if (topk < N)
          std::nth_element(ord.begin(), ord.begin() + topk, ord.end(), better);
        std::vector<int> sel(ord.begin(), ord.begin() + topk);
        int kth = *std::max_element(sel.begin(), sel.end(),
                                    [&](int a, int b) { return better(a, b); });
        if (topk < N) {
          int next = ord[topk];  // nth_element puts the (k+1)-th best here
          gap[r] = amax > 0 ? (s[kth] - s[next]) / amax : 0.0;
        } else {
          gap[r] = 1e300;
        }
        std::sort(sel.begin(), sel.end());
        for (int t = 0; t < topk; ++t) topk_idx[(size_t)r * topk + t] = sel[t];
        // Shared landmark value: full softmax over all N scores.
        double z = 0.0;
        std::fill(acc.begin(), acc.end(), 0.0);
        for (int j = 0; j < N; ++j) {
          double w = std::exp(s[j] - smax);
          z += w;
          const double* vr = vd.data() + (size_t)j * d;
          for (int l = 0; l < d; ++l) acc[l] += w * vr[l];
        }
        for (int l = 0; l < d; ++l) v_tilde[(size_t)r * d + l] = acc[l] / z;
      }
    }
    g0 = g1;
  }
  return 0;
}

// Step 4: route every query to its top-s landmarks by q . q~_i.
// [TUT] ch. 4 step 4 (eq. 10): compare q . q~_i and keep the top-s indices;
// scores select, there is no gate.  [GIST] Sec. 2.2: s = 1 in practice.
// route[., s] lists the chosen landmarks best first; gap = margin between the
// s-th and (s+1)-th logits relative to max_i |q . q~_i|.
int orc_route_rows(const void* q, int dt, const double* q_tilde, int B, int H,
                   int N, int d, int m, int s, long nq, const int64_t* qsel,
                   int32_t* route, double* gap) {
  (void)B; (void)H;
  if (s < 1 || s > m) return 1;
#pragma omp parallel
  {
    std::vector<double> sc(m);
    std::vector<int> ord(m);
#pragma omp for schedule(static)
    for (long r = 0; r < nq; ++r) {
      long qi = qsel ? qsel[r] : r;
      long bh = qi / N;
      double amax = 0.0;
      for (int i = 0; i < m; ++i) {
        double acc = 0.0;
        for (int l = 0; l < d; ++l)
          acc += widen(q, dt, (size_t)qi * d + l) * q_tilde[((size_t)bh * m + i) * d + l];
        sc[i] = acc;
        amax = std::max(amax, std::fabs(acc));
      }
      std::iota(ord.begin(), ord.end(), 0);
      Better better{sc.data()};
      std::sort(ord.begin(), ord.end(), better);
      for (int t = 0; t < s; ++t) route[(size_t)r * s + t] = ord[t];
      gap[r] = (s < m) ? (amax > 0 ? (sc[ord[s - 1]] - sc[ord[s]]) / amax : 0.0) : 1e300;
    }
  }
  return 0;
}

// Step 5: group queries by routed expert (Algorithm 1, [NEWS]).  A stable
// counting sort: bucket_off[B, H, m + 1] is the exclusive prefix sum of the
// per-expert counts; bucket_qidx[B, H, N * s] lists, per expert, the query
// indices in ascending order.
int orc_bucket(const int32_t* route, int B, int H, int N, int m, int s,
               int32_t* bucket_off, int32_t* bucket_qidx) {
  for (long bh = 0; bh < (long)B * H; ++bh) {
    std::vector<int32_t> cnt(m, 0);
    const int32_t* r = route + (size_t)bh * N * s;
    for (long n = 0; n < (long)N * s; ++n) {
      if (r[n] < 0 || r[n] >= m) return 1;
      cnt[r[n]]++;
    }
    int32_t* off = bucket_off + (size_t)bh * (m + 1);
    off[0] = 0;
    for (int i = 0; i < m; ++i) off[i + 1] = off[i] + cnt[i];
    std::vector<int32_t> fill(off, off + m);
    for (long n = 0; n < N; ++n)
      for (int t = 0; t < s; ++t)
        bucket_qidx[(size_t)bh * N * s + fill[r[n * s + t]]++] = (int32_t)n;
  }
  return 0;
}

// Step 6: one joint softmax over the concatenated entries.
// [TUT] ch. 4 steps 5-6 (eq. 11-12): every query sees the m shared pairs
// (q~_i, v~_i) plus the s*k raw pairs of its chosen experts, m + s*k entries,
// all scaled by 1/sqrt(d) and normalised together ([TUT] ch. 4: the shared
// and routed parts compete for one total weight of 1).  Experts are
// concatenated in route order; overlapping experts (s > 1) contribute their
// rows again, as the literal concatenation V* = [V~, V(e1), ..., V(es)] does.
// shared_temp = 0: every logit / sqrt(d); 1: the shared logits q . q~_i / d.
// routed_only = 1: the model without the shared (compression) branch that
// [NEWS] (LRA section) compares against at an equal number of entries per
// query: the softmax runs over the s*k raw pairs alone.
int orc_attend_rows_v(const void* q, const void* k, const void* v, int dt,
                      const double* q_tilde, const double* v_tilde,
                      const int32_t* topk_idx, const int32_t* route, int B, int H,
                      int N, int d, int m, int topk, int s, long nq,
                      const int64_t* qsel, int shared_temp, int routed_only, double* out) {
  (void)B; (void)H;
  if (shared_temp != 0 && shared_temp != 1) return 1;
  if (routed_only != 0 && routed_only != 1) return 1;
  const double sqrt_d = std::sqrt((double)d);
  const double shared_div = shared_temp ? (double)d : sqrt_d;
  const int m_used = routed_only ? 0 : m;
  const long E = (long)m_used + (long)s * topk;
#pragma omp parallel
  {
    std::vector<double> logit(E);
    std::vector<const double*> vrow_d(E);
    std::vector<long> vrow_raw(E);
    std::vector<double> acc(d);
#pragma omp for schedule(static)
    for (long r = 0; r < nq; ++r) {
      long qi = qsel ? qsel[r] : r;
      long bh = qi / N;
      size_t kv0 = (size_t)bh * N * d;
      long e = 0;
      for (int i = 0; i < m_used; ++i, ++e) {
        const double* qt = q_tilde + ((size_t)bh * m + i) * d;
        double a = 0.0;
        for (int l = 0; l < d; ++l) a += widen(q, dt, (size_t)qi * d + l) * qt[l];
        logit[e] = a / shared_div;
        vrow_d[e] = v_tilde + ((size_t)bh * m + i) * d;
        vrow_raw[e] = -1;
      }
      for (int t = 0; t < s; ++t) {
        int ex = route[(size_t)r * s + t];
        const int32_t* idx = topk_idx + ((size_t)bh * m + ex) * topk;
        for (int j = 0; j < topk; ++j, ++e) {
          logit[e] = dot(q, dt, (size_t)qi * d, k, dt, kv0 + (size_t)idx[j] * d, d) / sqrt_d;
          vrow_d[e] = nullptr;
          vrow_raw[e] = (long)idx[j];
        }
      }
      double mx = *std::max_element(logit.begin(), logit.end());
      double z = 0.0;
      std::fill(acc.begin(), acc.end(), 0.0);
      for (long t = 0; t < E; ++t) {
        double w = std::exp(logit[t] - mx);
        z += w;
        for (int l = 0; l < d; ++l)
          acc[l] += w * (vrow_d[t] ? vrow_d[t][l]
                                   : widen(v, dt, kv0 + (size_t)vrow_raw[t] * d + l));
      }
      for (int l = 0; l < d; ++l) out[(size_t)r * d + l] = acc[l] / z;
    }
  }
  return 0;
}

int orc_attend_rows(const void* q, const void* k, const void* v, int dt,
                    const double* q_tilde, const double* v_tilde,
                    const int32_t* topk_idx, const int32_t* route, int B, int H,
                    int N, int d, int m, int topk, int s, long nq,
                    const int64_t* qsel, double* out) {
  return orc_attend_rows_v(q, k, v, dt, q_tilde, v_tilde, topk_idx, route, B, H, N, d, m,
                           topk, s, nq, qsel, 0, 0, out);
}

// Dense softmax attention, softmax(q . k_j / sqrt(d)) over all N keys of the
// query's head, weighting V: the baseline of the long-sequence inference
// throughput comparison ([TUT] ch. 7, figure 5; [NEWS] throughput section).
int orc_dense_rows(const void* q, const void* k, const void* v, int dt, int B, int H, int N,
                   int d, long nq, const int64_t* qsel, double* out) {
  (void)B; (void)H;
  const double sqrt_d = std::sqrt((double)d);
#pragma omp parallel
  {
    std::vector<double> logit(N);
    std::vector<double> acc(d);
#pragma omp for schedule(static)
    for (long r = 0; r < nq; ++r) {
      long qi = qsel ? qsel[r] : r;
      long bh = qi / N;
      size_t kv0 = (size_t)bh * N * d;
      double mx = -INFINITY;
      for (long j = 0; j < N; ++j) {
        logit[j] = dot(q, dt, (size_t)qi * d, k, dt, kv0 + (size_t)j * d, d) / sqrt_d;
        mx = std::max(mx, logit[j]);
      }
      double z = 0.0;
      std::fill(acc.begin(), acc.end(), 0.0);
      for (long j = 0; j < N; ++j) {
        double w = std::exp(logit[j] - mx);
        z += w;
        for (int l = 0; l < d; ++l) acc[l] += w * widen(v, dt, kv0 + (size_t)j * d + l);
      }
      for (int l = 0; l < d; ++l) out[(size_t)r * d + l] = acc[l] / z;
    }
  }
  return 0;
}

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void orc_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

}  // extern "C"
