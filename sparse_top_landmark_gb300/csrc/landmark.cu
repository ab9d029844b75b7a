// Steps 2-3: routed experts (per-landmark top-k keys) and shared landmark
// values, from one sweep over the keys.
//
// MiTA tutorial (iwxt.cn), ch. 4 step 2 (paper eq. 6-7): landmark i scores
// all N keys with q~_i . k_j / sqrt(d) and keeps the top-k raw KV rows as
// routed expert i (bit.fan article: experts may overlap and span any
// positions).  Ch. 4 step 3 (eq. 8-9): the same N scores go through a
// softmax over all N that weights all of V into the shared value v~_i.
//
// Pipeline (split-N, flash-decoding style, to fill the GPU when B*H*m is
// small):
//   1. landmark_partial_kernel: CTA = (head, tile of RT landmarks, key split).
//      One thread per landmark row.  Scores are fp32 dots; an online softmax
//      accumulates (max, sum, sum p v); a per-row min-heap in shared memory
//      keeps the split's best Tcap (score, index) pairs.
//   2. landmark_merge_kernel: CTA = one landmark row.  Merges the softmax
//      partials (the merge identity of tutorial ch. 4) and selects the top-k
//      exactly: the fp32 candidates fix a threshold tau; keys whose fp32
//      score is within 2E of tau (E bounds the fp32 error) are re-scored with
//      exact-product fp32 arithmetic (two-product + two-sum; fp64 runs at a
//      small fraction of the fp32 rate here), so the selected set is the one
//      exact scores give, ties to the lowest index.  Rows where a split might
//      have dropped a qualifying key, or with too many near-ties, go to
//   3. landmark_exact_kernel: fp64 scores for all N keys of the row and a
//      radix select on (score, index) -- slow, used only for degenerate inputs
//      (mass ties, adversarial key order).
#include "common.cuh"
#include "kernels.h"

#include <algorithm>
#include <type_traits>

namespace mita {
namespace {

// Scaled log2-domain softmax constant log2(e) / sqrt(d).
__host__ __device__ inline float softmax_scale_log2(int D) {
  return (float)(1.4426950408889634 / sqrt((double)D));
}

// ---------------------------------------------------------------------------
// Per-row min-heap (worst kept candidate at the root) in shared memory,
// transposed as [slot][row] so that lanes never share a bank.
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool worse(float sa, int ia, float sb, int ib) {
  return sa < sb || (sa == sb && ia > ib);
}

template <int RT>
__device__ __forceinline__ void heap_offer(float* hs, int* hi, int lane, int& cnt, int cap,
                                           float s, int j) {
  if (cnt < cap) {
    int pos = cnt++;
    while (pos > 0) {
      int par = (pos - 1) >> 1;
      float ps = hs[par * RT + lane];
      int pi = hi[par * RT + lane];
      if (!worse(s, j, ps, pi)) break;
      hs[pos * RT + lane] = ps;
      hi[pos * RT + lane] = pi;
      pos = par;
    }
    hs[pos * RT + lane] = s;
    hi[pos * RT + lane] = j;
  } else if (s > hs[lane]) {
    // keys arrive in increasing index order, so an equal score is worse
    int pos = 0;
    for (;;) {
      int ch = 2 * pos + 1;
      if (ch >= cap) break;
      float cs = hs[ch * RT + lane];
      int ci = hi[ch * RT + lane];
      if (ch + 1 < cap) {
        float cs2 = hs[(ch + 1) * RT + lane];
        int ci2 = hi[(ch + 1) * RT + lane];
        if (worse(cs2, ci2, cs, ci)) { ch = ch + 1; cs = cs2; ci = ci2; }
      }
      if (!worse(cs, ci, s, j)) break;
      hs[pos * RT + lane] = cs;
      hi[pos * RT + lane] = ci;
      pos = ch;
    }
    hs[pos * RT + lane] = s;
    hi[pos * RT + lane] = j;
  }
}

template <typename T, int D, int RT>
__global__ void __launch_bounds__(RT)
landmark_partial_kernel(const T* __restrict__ q_tilde, const T* __restrict__ k,
                        const T* __restrict__ v, int N, int m, int S, int split_len,
                        int Tcap, LandmarkWs ws) {
  constexpr int KT = kKeyTile;
  constexpr int VEC = Vec<T>::N;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  float* ks = reinterpret_cast<float*>(smem_raw);           // [KT][D]
  float* vs = ks + KT * D;                                  // [KT][D]
  float* hs = vs + KT * D;                                  // [Tcap][RT]
  int* hi = reinterpret_cast<int*>(hs + Tcap * RT);         // [Tcap][RT]

  const int nrt = (m + RT - 1) / RT;
  long long b = blockIdx.x;
  const int split = (int)(b % S); b /= S;
  const int tile = (int)(b % nrt);
  const long long bh = b / nrt;
  const int tid = threadIdx.x;
  const int row = tile * RT + tid;
  const bool live = row < m;
  const int j0 = split * split_len;
  const int j1 = min(N, j0 + split_len);

  float qr[D];
  if (live) load_row<T, D>(q_tilde + (bh * m + row) * D, qr);
  else {
#pragma unroll
    for (int l = 0; l < D; ++l) qr[l] = 0.f;
  }
  const float c = softmax_scale_log2(D);
  float mrun = -INFINITY, lsum = 0.f;
  float acc[D];
#pragma unroll
  for (int l = 0; l < D; ++l) acc[l] = 0.f;
  int hcnt = 0;
  float kmax2 = 0.f;

  const T* kb = k + (size_t)bh * N * D;
  const T* vb = v + (size_t)bh * N * D;
  for (int jt = j0; jt < j1; jt += KT) {
    const int nk = min(KT, j1 - jt);
    __syncthreads();
    for (int e = tid; e < KT * (D / VEC); e += RT) {
      const int key = e / (D / VEC), part = (e % (D / VEC)) * VEC;
      float xk[VEC], xv[VEC];
      if (key < nk) {
        Vec<T>::load(kb + (size_t)(jt + key) * D + part, xk);
        Vec<T>::load(vb + (size_t)(jt + key) * D + part, xv);
      } else {
#pragma unroll
        for (int t = 0; t < VEC; ++t) { xk[t] = 0.f; xv[t] = 0.f; }
      }
#pragma unroll
      for (int t = 0; t < VEC; ++t) { ks[key * D + part + t] = xk[t]; vs[key * D + part + t] = xv[t]; }
    }
    __syncthreads();
    if (live) {
      for (int t = 0; t < nk; ++t) {
        const float* kr = ks + t * D;
        float sdot = 0.f;
#pragma unroll
        for (int l = 0; l < D; ++l) sdot = fmaf(qr[l], kr[l], sdot);
        heap_offer<RT>(hs, hi, tid, hcnt, Tcap, sdot, jt + t);
        const float x = sdot * c;
        if (x > mrun) {
          const float sc = exp2f(mrun - x);
          lsum *= sc;
#pragma unroll
          for (int l = 0; l < D; ++l) acc[l] *= sc;
          mrun = x;
        }
        const float p = exp2f(x - mrun);
        lsum += p;
        const float* vr = vs + t * D;
#pragma unroll
        for (int l = 0; l < D; ++l) acc[l] = fmaf(p, vr[l], acc[l]);
      }
    }
    if (tid < nk) {
      const float* kr = ks + tid * D;
      float n2 = 0.f;
#pragma unroll
      for (int l = 0; l < D; ++l) n2 = fmaf(kr[l], kr[l], n2);
      kmax2 = fmaxf(kmax2, n2);
    }
  }

  if (tid < 32) {
    float km = warp_max(kmax2);
    if (tid == 0 && tile == 0) ws.kmax2[bh * S + split] = km;
  }
  if (!live) return;
  const size_t rs = (size_t)(bh * m + row) * S + split;
  ws.M[rs] = mrun;
  ws.L[rs] = lsum;
  float* A = ws.A + rs * D;
#pragma unroll
  for (int l = 0; l < D; ++l) A[l] = acc[l];
  ws.cn[rs] = hcnt;
  ws.theta[rs] = (j1 - j0 > Tcap) ? hs[tid] : -INFINITY;
  float* cs = ws.cs + rs * Tcap;
  int* ci = ws.ci + rs * Tcap;
  for (int t = 0; t < hcnt; ++t) { cs[t] = hs[t * RT + tid]; ci[t] = hi[t * RT + tid]; }
}

// Exact top-k from fp32 candidates sorted best first (us/ui; `total` real
// entries).  tau = the k-th fp32 score.  Keys above tau + 2E are members,
// keys below tau - 2E are not (E bounds the fp32 error; the caller guarantees
// every key that could reach tau - 2E is among the candidates); the band in
// between is re-scored with exact-product arithmetic and ranked (score desc,
// index asc).  With `slow` set, or a band too wide to rank here, the row goes
// to the exact fallback.  Writes the member indices ascending.
template <typename T, int D>
__device__ void finish_topk(float* us, int* ui, int total, int topk, float E, bool slow,
                            const float* qd, const T* kb, F2* bx, int* bi, int* ired,
                            long long rowflat, const LandmarkWs& ws,
                            int32_t* __restrict__ topk_idx) {
  const int tid = threadIdx.x;
  int a = 0, bnd_end = 0;
  if (!slow) {
    const float tau = us[topk - 1];
    const float lo_band = tau - 2.f * E, hi_band = tau + 2.f * E;
    // us is sorted best first: [0, a) above the band, [a, bnd_end) in it
    int ca = 0, cb = 0;
    for (int t = tid; t < total; t += blockDim.x) {
      ca += us[t] > hi_band;
      cb += us[t] >= lo_band;
    }
    block_excl_scan(ca, ired, &a);
    __syncthreads();
    block_excl_scan(cb, ired, &bnd_end);
    if (bnd_end - a > kBandCap) slow = true;
  }
  if (slow) {
    if (tid == 0) {
      const int p = atomicAdd(ws.nslow, 1);
      ws.slow_rows[p] = (int)rowflat;
    }
    return;
  }
  // --- exact re-scoring of the band -------------------------------------------
  const int nb = bnd_end - a;
  const int PB = next_pow2(max(nb, 1));
  for (int t = tid; t < PB; t += blockDim.x) {
    if (t < nb) {
      const int j = ui[a + t];
      float kr[D];
      load_row<T, D>(kb + (size_t)j * D, kr);
      bx[t] = dot_f2<D>(qd, kr);
      bi[t] = j;
    } else {
      bx[t] = F2{-INFINITY, 0.f};
      bi[t] = 0x7fffffff;
    }
  }
  bitonic_sort_desc(bx, bi, PB);
  // --- the a sure members plus the best (topk - a) of the band, ascending ----
  const int PK = next_pow2(topk);
  __syncthreads();
  int* outset = reinterpret_cast<int*>(us);   // us is no longer needed
  for (int t = tid; t < PK; t += blockDim.x) {
    int val;
    if (t < a) val = ui[t];
    else if (t < topk) val = bi[t - a];
    else val = 0x7fffffff;
    outset[t] = val;
  }
  bitonic_sort_int_asc(outset, PK);
  for (int t = tid; t < topk; t += blockDim.x) topk_idx[rowflat * topk + t] = outset[t];
}

template <typename T, int D>
__global__ void __launch_bounds__(256)
landmark_merge_kernel(const T* __restrict__ q_tilde, const T* __restrict__ k, int N, int m,
                      int topk, int S, int Tcap, int P, LandmarkWs ws,
                      int32_t* __restrict__ topk_idx, float* __restrict__ v_tilde) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  float* us = reinterpret_cast<float*>(smem_raw);           // [P]
  int* ui = reinterpret_cast<int*>(us + P);                 // [P]
  F2* bx = reinterpret_cast<F2*>(ui + P);                   // [kBandCap]
  int* bi = reinterpret_cast<int*>(bx + kBandCap);          // [kBandCap]
  __shared__ float qd[D];
  __shared__ int soff[257];
  __shared__ float red[8];
  __shared__ int ired[9];
  __shared__ int s_slow;

  const long long rowflat = blockIdx.x;                     // bh * m + i
  const long long bh = rowflat / m;
  const int tid = threadIdx.x;
  const size_t r0 = (size_t)rowflat * S;

  // --- shared value: merge the split softmax partials -----------------------
  float mx = -INFINITY;
  for (int s = tid; s < S; s += blockDim.x) mx = fmaxf(mx, ws.M[r0 + s]);
  mx = block_max(mx, red);
  for (int l = tid; l < D; l += blockDim.x) {
    float num = 0.f, den = 0.f;
    for (int s = 0; s < S; ++s) {
      const float w = exp2f(ws.M[r0 + s] - mx);
      num = fmaf(w, ws.A[(r0 + s) * D + l], num);
      den = fmaf(w, ws.L[r0 + s], den);
    }
    v_tilde[rowflat * D + l] = num / den;
    if (l == 0 && ws.lse_out) ws.lse_out[rowflat] = (mx + log2f(den)) * 0.6931471805599453f;
  }

  // --- gather the kept candidates of every split -----------------------------
  if (tid == 0) {
    int run = 0;
    for (int s = 0; s < S; ++s) { soff[s] = run; run += ws.cn[r0 + s]; }
    soff[S] = run;
    s_slow = 0;
  }
  for (int l = tid; l < D; l += blockDim.x) qd[l] = to_f(q_tilde[rowflat * D + l]);
  __syncthreads();
  const int total = soff[S];
  for (int s = 0; s < S; ++s) {
    const int n = soff[s + 1] - soff[s];
    for (int t = tid; t < n; t += blockDim.x) {
      us[soff[s] + t] = ws.cs[(r0 + s) * Tcap + t];
      ui[soff[s] + t] = ws.ci[(r0 + s) * Tcap + t];
    }
  }
  for (int t = total + tid; t < P; t += blockDim.x) { us[t] = -INFINITY; ui[t] = 0x7fffffff; }
  bitonic_sort_desc(us, ui, P);

  // --- threshold and fp32 error bound ---------------------------------------
  float qn2 = 0.f;
  for (int l = tid; l < D; l += blockDim.x) qn2 += qd[l] * qd[l];
  qn2 = block_sum(qn2, red);
  float km2 = 0.f;
  for (int s = tid; s < S; s += blockDim.x) km2 = fmaxf(km2, ws.kmax2[bh * S + s]);
  km2 = block_max(km2, red);
  const float E = err_gamma(D) * sqrtf(qn2) * sqrtf(km2);
  bool slow = total < topk;
  if (!slow) {
    // a split that dropped keys scoring at or above tau - 2E may hide a member
    const float lo_band = us[topk - 1] - 2.f * E;
    for (int s = tid; s < S; s += blockDim.x)
      if (ws.theta[r0 + s] >= lo_band) s_slow = 1;
  }
  __syncthreads();
  slow = slow || s_slow;
  finish_topk<T, D>(us, ui, total, topk, E, slow, qd, k + (size_t)bh * N * D, bx, bi, ired,
                    rowflat, ws, topk_idx);
}

// Exact-product dot of qd (shared memory, fp32) with one key row, by a whole warp: lane l
// takes the products of elements l, l + 32 (split exactly with an FMA), and the 32
// partial (sum, error) pairs are combined with error-free two-sums across the lanes.
// Returns hi + lo on every lane; like dot_f2, exact up to ~2^-48 relative.
template <typename T, int D>
__device__ __forceinline__ F2 dot_f2_warp(const float* qd, const T* krow, int lane) {
  static_assert(D <= 128, "row split over the warp's lanes");   // lanes past D add zeros
  float s = 0.f, c = 0.f;
#pragma unroll
  for (int l = lane; l < D; l += 32) {
    const float a = qd[l], b = to_f(krow[l]);
    const float p = __fmul_rn(a, b);
    const float e = fmaf(a, b, -p);
    two_sum_acc(s, c, p);
    c = __fadd_rn(c, e);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o), c2 = __shfl_xor_sync(0xffffffffu, c, o);
    two_sum_acc(s, c, s2);
    c = __fadd_rn(c, c2);
  }
  return f2_normalize(s, c);
}

// Candidates of the tensor-core path: the keys whose fp32 score reached the
// row's collection threshold, gathered by the collect kernel (in no particular
// order).  tau, the k-th largest fp32 score, comes from a radix select over
// the order-preserving 32-bit keys (four 8-bit digits, most significant first,
// warp-aggregated shared-memory histograms); the keys above tau + 2E are
// members, the band [tau - 2E, tau + 2E] is re-scored exactly and ranked
// (score desc, index asc), and the member indices are sorted ascending --
// the same rule as finish_topk without sorting every candidate.
template <typename T, int D>
__global__ void __launch_bounds__(256)
landmark_select_kernel(const T* __restrict__ q_tilde, const T* __restrict__ k, int N, int m,
                       int topk, int cap, int P, LandmarkWs ws, int32_t* __restrict__ topk_idx) {
  griddep_wait();
  extern __shared__ __align__(16) unsigned char smem_raw[];
  float* us = reinterpret_cast<float*>(smem_raw);           // [cap]
  int* ui = reinterpret_cast<int*>(us + cap);               // [cap]
  F2* bx = reinterpret_cast<F2*>(ui + cap);                 // [kBandCap]
  int* bi = reinterpret_cast<int*>(bx + kBandCap);          // [kBandCap]
  int* outset = bi + kBandCap;                              // [next_pow2(topk)]
  __shared__ float qd[D];
  __shared__ int hist[256];
  __shared__ int s_cnt[2];
  __shared__ uint32_t s_prefix;
  __shared__ int s_need;
  (void)P;
  const long long rowflat = blockIdx.x;
  const long long bh = rowflat / m;
  const int tid = threadIdx.x, lane = tid & 31;
  const int cnt = ws.cnt[rowflat];
  const int total = min(cnt, cap);
  if (cnt > cap || cnt < topk) {                             // to the exact fallback
    if (tid == 0) ws.slow_rows[atomicAdd(ws.nslow, 1)] = (int)rowflat;
    return;
  }
  for (int l = tid; l < D; l += blockDim.x) qd[l] = to_f(q_tilde[rowflat * D + l]);
  const float* cs = ws.cand_s + (size_t)rowflat * cap;
  const int* ci = ws.cand_i + (size_t)rowflat * cap;
  for (int t = tid; t < total; t += blockDim.x) {
    us[t] = cs[t];
    ui[t] = ci[t];
  }
  if (tid == 0) {
    s_prefix = 0u;
    s_need = topk;
    s_cnt[0] = 0;
    s_cnt[1] = 0;
  }
  const int iters = (total + blockDim.x - 1) / blockDim.x;
  // ---- tau: the k-th largest key, digit by digit
  uint32_t mask = 0u;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    hist[tid] = 0;
    __syncthreads();
    const uint32_t prefix = s_prefix;
    for (int j = 0; j < iters; ++j) {
      const int t = j * blockDim.x + tid;
      int dg = -1;
      if (t < total) {
        const uint32_t key = fkey(us[t]);
        if ((key & mask) == prefix) dg = (int)((key >> shift) & 255u);
      }
      const unsigned peers = __match_any_sync(0xffffffffu, dg);
      if (dg >= 0 && lane == __ffs(peers) - 1) atomicAdd(&hist[dg], __popc(peers));
    }
    __syncthreads();
    if (tid < 32) {
      // lane l holds digits 255 - 8l down to 248 - 8l; counts accumulate from the top
      int c[8], sum = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        c[i] = hist[255 - 8 * lane - i];
        sum += c[i];
      }
      int inc = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
      }
      const int need = s_need, before = inc - sum;
      if (before < need && inc >= need) {                    // exactly one lane
        int run = before, dg = -1;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (dg < 0) {
            if (run + c[i] >= need) dg = 255 - 8 * lane - i;
            else run += c[i];
          }
        }
        s_need = need - run;
        s_prefix = prefix | ((uint32_t)dg << shift);
      }
    }
    mask |= 255u << shift;
    __syncthreads();
  }
  const float tau = fkey_inv(s_prefix);
  const float E = ws.E[rowflat];
  const float lo_band = tau - 2.f * E, hi_band = tau + 2.f * E;
  // ---- members above the band, and the band (both unordered)
  for (int j = 0; j < iters; ++j) {
    const int t = j * blockDim.x + tid;
    const float x = t < total ? us[t] : -INFINITY;
    const int id = t < total ? ui[t] : 0;
    const bool above = t < total && x > hi_band;
    const bool inband = t < total && !above && x >= lo_band;
    const unsigned ma = __ballot_sync(0xffffffffu, above), mb = __ballot_sync(0xffffffffu, inband);
    int ba = 0, bb = 0;
    if (lane == 0) {
      if (ma) ba = atomicAdd(&s_cnt[0], __popc(ma));
      if (mb) bb = atomicAdd(&s_cnt[1], __popc(mb));
    }
    ba = __shfl_sync(0xffffffffu, ba, 0);
    bb = __shfl_sync(0xffffffffu, bb, 0);
    const unsigned lt = (1u << lane) - 1u;
    if (above) outset[ba + __popc(ma & lt)] = id;           // fewer than topk keys exceed tau
    if (inband) {
      const int pb = bb + __popc(mb & lt);
      if (pb < kBandCap) bi[pb] = id;
    }
  }
  __syncthreads();
  const int a = s_cnt[0], nb = s_cnt[1];
  if (nb > kBandCap) {
    if (tid == 0) ws.slow_rows[atomicAdd(ws.nslow, 1)] = (int)rowflat;
    return;
  }
  // ---- exact re-scoring and ranking of the band
  const T* kb = k + (size_t)bh * N * D;
  const int PB = next_pow2(max(nb, 1));
  for (int t = nb + tid; t < PB; t += blockDim.x) {
    bx[t] = F2{-INFINITY, 0.f};
    bi[t] = 0x7fffffff;
  }
  // one warp per band entry
  for (int t = tid >> 5; t < nb; t += blockDim.x >> 5) {
    const F2 x = dot_f2_warp<T, D>(qd, kb + (size_t)bi[t] * D, lane);
    if (lane == 0) bx[t] = x;
  }
  bitonic_sort_desc(bx, bi, PB);
  // ---- the a members above the band plus the best (topk - a) of it, ascending
  const int PK = next_pow2(topk);
  for (int t = a + tid; t < PK; t += blockDim.x) outset[t] = t < topk ? bi[t - a] : 0x7fffffff;
  bitonic_sort_int_asc(outset, PK);
  for (int t = tid; t < topk; t += blockDim.x) topk_idx[rowflat * topk + t] = outset[t];
}

// Exact fallback: fp64 scores of all N keys, radix select on the monotone
// 64-bit key, ties at the k-th value resolved by the lowest index.
template <typename T, int D>
__global__ void __launch_bounds__(512)
landmark_exact_kernel(const T* __restrict__ q_tilde, const T* __restrict__ k, int N, int m,
                      int topk, LandmarkWs ws, int32_t* __restrict__ topk_idx) {
  griddep_wait();
  __shared__ double qd[D];
  __shared__ int hist[256];
  __shared__ int ired[17];
  __shared__ unsigned long long s_prefix;
  __shared__ int s_need;
  double* sc = ws.exact + (size_t)blockIdx.x * N;
  const int tid = threadIdx.x;
  const int nslow = *ws.nslow;
  for (int w = blockIdx.x; w < nslow; w += gridDim.x) {
    const long long rowflat = ws.slow_rows[w];
    const long long bh = rowflat / m;
    __syncthreads();
    for (int l = tid; l < D; l += blockDim.x) qd[l] = to_f(q_tilde[rowflat * D + l]);
    __syncthreads();
    const T* kb = k + (size_t)bh * N * D;
    for (int j = tid; j < N; j += blockDim.x) sc[j] = dot_exact<T, D>(qd, kb + (size_t)j * D);
    if (tid == 0) { s_prefix = 0ull; s_need = topk; }
    unsigned long long mask = 0ull;
    for (int pass = 0; pass < 8; ++pass) {
      const int shift = 56 - 8 * pass;
      for (int t = tid; t < 256; t += blockDim.x) hist[t] = 0;
      __syncthreads();
      const unsigned long long prefix = s_prefix;
      for (int j = tid; j < N; j += blockDim.x) {
        const unsigned long long u = order_key(sc[j]);
        if ((u & mask) == prefix) atomicAdd(&hist[(u >> shift) & 255], 1);
      }
      __syncthreads();
      if (tid == 0) {
        int need = s_need, cum = 0, dg = 255;
        for (; dg > 0; --dg) {
          if (cum + hist[dg] >= need) break;
          cum += hist[dg];
        }
        s_need = need - cum;
        s_prefix = prefix | ((unsigned long long)dg << shift);
      }
      mask |= 0xffull << shift;
      __syncthreads();
    }
    const unsigned long long kstar = s_prefix;
    const int need_eq = s_need;           // how many keys equal to kstar to take
    int out_base = 0, eq_base = 0;
    for (int j0 = 0; j0 < N; j0 += blockDim.x) {
      const int j = j0 + tid;
      unsigned long long u = 0ull;
      if (j < N) u = order_key(sc[j]);
      const int is_eq = (j < N && u == kstar) ? 1 : 0;
      int eq_tot;
      const int eq_rank = eq_base + block_excl_scan(is_eq, ired, &eq_tot);
      const int take = (j < N) && (u > kstar || (is_eq && eq_rank < need_eq));
      int take_tot;
      const int pos = out_base + block_excl_scan(take, ired, &take_tot);
      if (take && pos < topk) topk_idx[rowflat * topk + pos] = j;
      out_base += take_tot;
      eq_base += eq_tot;
    }
  }
}

template <typename T, int D, int RT>
cudaError_t run_partial(const T* qt, const T* k, const T* v, int BH, int N, int m,
                        const LandmarkPlan& p, const LandmarkWs& ws, cudaStream_t st) {
  const size_t smem = (size_t)2 * kKeyTile * D * sizeof(float) + (size_t)p.Tcap * RT * 8;
  auto kern = landmark_partial_kernel<T, D, RT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const long long blocks = (long long)BH * p.nrt * p.S;
  kern<<<(unsigned)blocks, RT, smem, st>>>(qt, k, v, N, m, p.S, p.split_len, p.Tcap, ws);
  count_launch();
  return cudaGetLastError();
}

// Short sequences (N <= kSmallMaxN, too few key tiles for the tensor-core two-pass
// selection): one CTA holds up to kSmallRows landmark rows of one head and takes all N keys
// through shared memory twice -- K for the fp32 scores, then V for the shared values v~
// (tutorial ch. 4 steps 2-3) -- in chunks staged by cp.async into a double buffer.  The
// score block S[key][row] stays in shared memory; between the two passes each warp selects
// its row's top-k exactly (the landmark_select_kernel rule: tau, the k-th largest fp32 score,
// by a radix select over the order-preserving keys; keys above tau + 2E are members, the band
// [tau - 2E, tau + 2E] is re-scored exactly and ranked by (score desc, index asc)) and turns
// its scores into softmax weights in place.  Rows whose band holds more than 32 keys go to
// the exact fallback.
constexpr int kSmallMaxN = 1024;
constexpr int kSmallRows = 8;              // landmark rows per CTA, one warp each
constexpr int kSmallThreads = 256;
constexpr int kSmallSP = kSmallRows + 1;   // S row stride in floats (odd: no bank conflicts)

template <typename T, int D>
struct SmallCfg {
  static constexpr int VEC = Vec<T>::N;                       // elements per 16-byte slice
  static constexpr int NS = D / VEC;                          // slices per row
  static constexpr int KC0 = 16384 / (D * (int)sizeof(T));
  static constexpr int KC = KC0 > 256 ? 256 : KC0;            // keys per staged chunk
  static constexpr int RS = D * (int)sizeof(T) + 16;          // staged row stride (bytes)
  static constexpr size_t BUF = (size_t)KC * RS;
  static_assert((size_t)kSmallThreads / 32 * kSmallRows * D * 4 <= 2 * BUF,
                "the cross-warp reduction fits in the staging buffers");
};

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// S[N][kSmallSP] floats, rounded up to keep what follows 16-byte aligned
__host__ __device__ inline size_t small_s_floats(int N) {
  return ((size_t)N * kSmallSP + 3) & ~(size_t)3;
}

// four consecutive elements as floats (8-byte aligned for bf16, 16-byte for fp32)
__device__ __forceinline__ void load4(const bf16* p, float* o) {
  const uint2 x = *reinterpret_cast<const uint2*>(p);
  o[0] = __uint_as_float(x.x << 16);
  o[1] = __uint_as_float(x.x & 0xffff0000u);
  o[2] = __uint_as_float(x.y << 16);
  o[3] = __uint_as_float(x.y & 0xffff0000u);
}
__device__ __forceinline__ void load4(const float* p, float* o) {
  const float4 x = *reinterpret_cast<const float4*>(p);
  o[0] = x.x; o[1] = x.y; o[2] = x.z; o[3] = x.w;
}

template <typename T, int D>
size_t small_smem_bytes(int N) {
  using C = SmallCfg<T, D>;
  return 2 * C::BUF + small_s_floats(N) * 4 + (size_t)kSmallRows * D * (4 + sizeof(T)) +
         (size_t)kSmallRows * 256 * 4 + (size_t)kSmallRows * 32 * 8 + 64;
}

// The topk-th largest of a warp's n order keys (lane l holds items l + 32 i, i < NI; 0 marks
// no item: below every key), bit by bit from the top (the largest prefix that at least topk
// keys reach).  Bits 31..16 count every key; the keys sharing the 16-bit prefix found are then
// the only ones the low bits can still order, so they are listed in `al` (256 words of
// scratch): up to 32 of them are ranked directly, up to 256 finish the bit search alone.
template <int NI>
__device__ __forceinline__ uint32_t warp_kth_key(const uint32_t (&u)[NI], int n, int topk,
                                                 uint32_t* al, int lane) {
  const int N = n;
  uint32_t prefix = 0u;
#pragma unroll 1
  for (int b = 31; b >= 16; --b) {
    const uint32_t cand = prefix | (1u << b);
    int c = 0;
#pragma unroll
    for (int i = 0; i < NI; ++i) c += u[i] >= cand ? 1 : 0;
    if ((int)__reduce_add_sync(0xffffffffu, (unsigned)c) >= topk) prefix = cand;
  }
  {
    const uint32_t top = prefix >> 16;
    int c = 0;
#pragma unroll
    for (int i = 0; i < NI; ++i) c += (u[i] >> 16) > top ? 1 : 0;
    const int need = topk - (int)__reduce_add_sync(0xffffffffu, (unsigned)c);
    int na16 = 0;
    const unsigned lt16 = (1u << lane) - 1u;
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      if (32 * i < N) {
        const bool in = (u[i] >> 16) == top && u[i] != 0u;
        const unsigned bm = __ballot_sync(0xffffffffu, in);
        if (in && na16 + __popc(bm & lt16) < 256) al[na16 + __popc(bm & lt16)] = u[i];
        na16 += __popc(bm);
      }
    }
    __syncwarp();
    if (na16 <= 32) {
      // at most one listed key a lane: tau is the one whose rank among them brackets need
      const uint32_t mine = lane < na16 ? al[lane] : 0u;
      int gt = 0, eq = 0;
      for (int f = 0; f < na16; ++f) {
        const uint32_t o = al[f];
        gt += o > mine ? 1 : 0;
        eq += o == mine ? 1 : 0;
      }
      const bool hit = lane < na16 && gt < need && need <= gt + eq;
      prefix = __shfl_sync(0xffffffffu, mine, __ffs(__ballot_sync(0xffffffffu, hit)) - 1);
    } else if (na16 <= 256) {
      uint32_t v[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) v[t] = lane + 32 * t < na16 ? al[lane + 32 * t] : 0u;
#pragma unroll 1
      for (int b = 15; b >= 0; --b) {
        const uint32_t cand = prefix | (1u << b);
        int cc = 0;
#pragma unroll
        for (int t = 0; t < 8; ++t) cc += v[t] >= cand ? 1 : 0;
        if ((int)__reduce_add_sync(0xffffffffu, (unsigned)cc) >= need) prefix = cand;
      }
    } else {
#pragma unroll 1
      for (int b = 15; b >= 0; --b) {
        const uint32_t cand = prefix | (1u << b);
        int cc = 0;
#pragma unroll
        for (int i = 0; i < NI; ++i) cc += u[i] >= cand ? 1 : 0;
        if ((int)__reduce_add_sync(0xffffffffu, (unsigned)cc) >= topk) prefix = cand;
      }
    }
    __syncwarp();
  }
  return prefix;
}

// One landmark row of landmark_small_kernel, on one warp: the exact top-k of the row's N fp32
// scores (key j at Sw[j * kSmallSP]), then the softmax weights in place of the scores.  Lane
// l holds keys l + 32 i for i < NI (32 NI >= N) in registers.
template <typename T, int D, int NI>
__device__ __forceinline__ void small_row(float* Sw, const float* qd, const T* kb, int N, int topk,
                                          long long row, float km2, int* hist, int* bjw,
                                          unsigned* sw, float* lsum_out, const LandmarkWs& ws,
                                          int32_t* __restrict__ topk_idx, int lane) {
  // the scores as order keys (fkey is a bijection: fkey_inv gives the score back)
  uint32_t u[NI];
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const int j = lane + 32 * i;
    const float x = j < N ? Sw[(size_t)j * kSmallSP] : -INFINITY;
    mx = fmaxf(mx, x);
    u[i] = j < N ? fkey(x) : 0u;             // 0: below every key
  }
  const uint32_t prefix = warp_kth_key<NI>(u, N, topk, reinterpret_cast<uint32_t*>(hist), lane);
  const float tau = fkey_inv(prefix);
  float qn2 = 0.f;
  for (int l = lane; l < D; l += 32) qn2 = fmaf(qd[l], qd[l], qn2);
  qn2 = warp_sum(qn2);
  const float E = err_gamma(D) * sqrtf(qn2) * sqrtf(km2);
  const float hi_band = tau + 2.f * E, lo_band = tau - 2.f * E;
  const unsigned lt = (1u << lane) - 1u;
  // members above the band (bit i: key lane + 32 i), and the band listed by ascending key
  sw[lane] = 0u;
  uint32_t above = 0u;
  int nb = 0, na = 0;
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    if (32 * i < N) {
      const bool ok = lane + 32 * i < N;
      const float x = fkey_inv(u[i]);
      const bool ab = ok && x > hi_band, in = ok && !ab && x >= lo_band;
      above |= (uint32_t)ab << i;
      na += __popc(__ballot_sync(0xffffffffu, ab));
      const unsigned bm = __ballot_sync(0xffffffffu, in);
      if (in && nb + __popc(bm & lt) < 32) bjw[nb + __popc(bm & lt)] = lane + 32 * i;
      nb += __popc(bm);
    }
  }
  if (nb > 32) {
    if (lane == 0) ws.slow_rows[atomicAdd(ws.nslow, 1)] = (int)row;
  } else {
    __syncwarp();
    F2 mine{-INFINITY, 0.f};
    int mj = 0x7fffffff;
    for (int e = 0; e < nb; ++e) {
      const int j = bjw[e];
      const F2 x = dot_f2_warp<T, D>(qd, kb + (size_t)j * D, lane);
      if (lane == e) { mine = x; mj = j; }
    }
    int rank = 0;
    for (int f = 0; f < nb; ++f) {
      const F2 y{__shfl_sync(0xffffffffu, mine.hi, f), __shfl_sync(0xffffffffu, mine.lo, f)};
      const int jf = __shfl_sync(0xffffffffu, mj, f);
      if (f != lane && ranks_before(y, jf, mine, mj)) ++rank;
    }
    if (lane < nb && rank < topk - na) atomicOr(&sw[mj & 31], 1u << (mj >> 5));
    __syncwarp();
    const uint32_t mem = above | sw[lane];
    int32_t* out = topk_idx + row * topk;
    int pos = 0;
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      if (32 * i < N) {
        const bool take = (mem >> i) & 1u;
        const unsigned mm = __ballot_sync(0xffffffffu, take);
        if (take && pos + __popc(mm & lt) < topk) out[pos + __popc(mm & lt)] = lane + 32 * i;
        pos += __popc(mm);
      }
    }
  }
  const float cl = softmax_scale_log2(D);
  const float M = warp_max(mx) * cl;         // log2 units
  float ls = 0.f;
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const int j = lane + 32 * i;
    if (32 * i < N && j < N) {
      const float p = exp2f(fkey_inv(u[i]) * cl - M);
      Sw[(size_t)j * kSmallSP] = p;
      ls += p;
    }
  }
  const float lsum = warp_sum(ls);
  if (lane == 0) {
    *lsum_out = lsum;
    if (ws.lse_out) ws.lse_out[row] = (M + log2f(lsum)) * 0.6931471805599453f;
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(kSmallThreads, 3)
landmark_small_kernel(const T* __restrict__ q_tilde, const T* __restrict__ k,
                      const T* __restrict__ v, int N, int m, int groups, int rpg, int topk,
                      LandmarkWs ws, int32_t* __restrict__ topk_idx, float* __restrict__ v_tilde) {
  using C = SmallCfg<T, D>;
  constexpr int VEC = C::VEC, NS = C::NS, KC = C::KC;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  unsigned char* buf = smem_raw;                                       // [2][KC][RS]
  float* S = reinterpret_cast<float*>(smem_raw + 2 * C::BUF);          // [N][kSmallSP]
  float* qs = S + small_s_floats(N);                                   // [rows][D]
  T* qsT = reinterpret_cast<T*>(qs + kSmallRows * D);                  // [rows][D]
  int* whist = reinterpret_cast<int*>(qsT + kSmallRows * D);           // [rows][256]
  int* bj = whist + kSmallRows * 256;                                  // [rows][32]
  unsigned* selw = reinterpret_cast<unsigned*>(bj + kSmallRows * 32);  // [rows][32]
  float* lsum_s = reinterpret_cast<float*>(selw + kSmallRows * 32);    // [rows]
  unsigned* km2_s = reinterpret_cast<unsigned*>(lsum_s + kSmallRows);  // [1]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long bh = blockIdx.x / groups;
  const int r0 = (int)(blockIdx.x % groups) * rpg;
  const int nrows = min(rpg, m - r0);
  const long long row0 = bh * m + r0;
  const T* kb = k + (size_t)bh * N * D;
  const T* vb = v + (size_t)bh * N * D;
  const int nc = (N + KC - 1) / KC;

  auto stage = [&](int c) {                  // chunk c < nc: K rows; c >= nc: V rows
    const T* src = c < nc ? kb : vb;
    const int j0 = (c < nc ? c : c - nc) * KC;
    unsigned char* dst = buf + (size_t)(c & 1) * C::BUF;
    for (int t = tid; t < KC * NS; t += kSmallThreads) {
      const int jl = t / NS, s = t % NS;
      if (j0 + jl < N)
        cp_async16(dst + (size_t)jl * C::RS + s * 16, src + (size_t)(j0 + jl) * D + s * VEC);
    }
    cp_async_commit();
  };

  griddep_wait();
  stage(0);
  for (int t = tid; t < kSmallRows * D; t += kSmallThreads) {
    const int r = t / D;
    const T x = r < nrows ? q_tilde[(row0 + r) * D + t % D] : T(0.f);
    qsT[t] = x;
    qs[t] = to_f(x);
  }
  if (tid == 0) *km2_s = 0u;

  // ---- pass 1: S[j][r] = q~_r . k_j (fp32), and the largest squared key norm; a thread
  // takes keys jl and jl + KC / 2 of the chunk, on every TPP-th slice
  constexpr int KP = KC / 2, TPP = kSmallThreads / KP;
  static_assert(NS % TPP == 0 && TPP <= 32, "pair threads split a row's slices");
  float km2 = 0.f;
  for (int c = 0; c < nc; ++c) {
    stage(c + 1);
    cp_async_wait<1>();
    __syncthreads();
    const unsigned char* kbuf = buf + (size_t)(c & 1) * C::BUF;
    const int kp = tid / TPP, part = tid % TPP;
    const int j0 = c * KC + kp, j1 = j0 + KP;
    float a0[kSmallRows], a1[kSmallRows];
#pragma unroll
    for (int r = 0; r < kSmallRows; ++r) { a0[r] = 0.f; a1[r] = 0.f; }
    float n0 = 0.f, n1 = 0.f;
    if (j0 < N) {
#pragma unroll
      for (int s = part; s < NS; s += TPP) {
        float x0[VEC], x1[VEC];
        Vec<T>::load(reinterpret_cast<const T*>(kbuf + (size_t)kp * C::RS + s * 16), x0);
        Vec<T>::load(reinterpret_cast<const T*>(kbuf + (size_t)(kp + KP) * C::RS + s * 16), x1);
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          n0 = fmaf(x0[e], x0[e], n0);
          n1 = fmaf(x1[e], x1[e], n1);
        }
#pragma unroll
        for (int r = 0; r < kSmallRows; ++r) {
          float q[VEC];
          Vec<T>::load(qsT + r * D + s * VEC, q);
#pragma unroll
          for (int e = 0; e < VEC; ++e) {
            a0[r] = fmaf(q[e], x0[e], a0[r]);
            a1[r] = fmaf(q[e], x1[e], a1[r]);
          }
        }
      }
    }
#pragma unroll
    for (int o = 1; o < TPP; o <<= 1) {
      n0 += __shfl_xor_sync(0xffffffffu, n0, o);
      n1 += __shfl_xor_sync(0xffffffffu, n1, o);
#pragma unroll
      for (int r = 0; r < kSmallRows; ++r) {
        a0[r] += __shfl_xor_sync(0xffffffffu, a0[r], o);
        a1[r] += __shfl_xor_sync(0xffffffffu, a1[r], o);
      }
    }
    if (part == 0) {
      if (j0 < N) {
#pragma unroll
        for (int r = 0; r < kSmallRows; ++r) S[(size_t)j0 * kSmallSP + r] = a0[r];
        km2 = fmaxf(km2, n0);
      }
      if (j1 < N) {              // the second key's staged row is stale past N: unused then
#pragma unroll
        for (int r = 0; r < kSmallRows; ++r) S[(size_t)j1 * kSmallSP + r] = a1[r];
        km2 = fmaxf(km2, n1);
      }
    }
    __syncthreads();
  }
  km2 = warp_max(km2);
  if (lane == 0) atomicMax(km2_s, __float_as_uint(km2));   // non-negative: bits order as values
  __syncthreads();

  // ---- per row (one warp): exact top-k, then softmax weights in place of the scores
  if (warp < nrows) {
    const float km2h = __uint_as_float(*km2_s);
    float* Sw = S + warp;
    if (N <= 256)
      small_row<T, D, 8>(Sw, qs + warp * D, kb, N, topk, row0 + warp, km2h, whist + warp * 256,
                         bj + warp * 32, selw + warp * 32, lsum_s + warp, ws, topk_idx, lane);
    else
      small_row<T, D, 32>(Sw, qs + warp * D, kb, N, topk, row0 + warp, km2h, whist + warp * 256,
                          bj + warp * 32, selw + warp * 32, lsum_s + warp, ws, topk_idx, lane);
  }
  __syncthreads();

  // ---- pass 2: sum_j p_rj v_j; thread = (key group g, 4-element piece s of the row)
  constexpr int NP = D / 4;                  // pieces per row
  constexpr int GP = kSmallThreads / NP;     // key groups
  static_assert(NP <= 32 && 32 % NP == 0, "a warp spans whole rows in the V pass");
  const int s = tid % NP, g = tid / NP;
  float acc[kSmallRows][4];
#pragma unroll
  for (int r = 0; r < kSmallRows; ++r)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[r][e] = 0.f;
  for (int c = nc; c < 2 * nc; ++c) {
    if (c + 1 < 2 * nc) stage(c + 1);
    if (c + 1 < 2 * nc) cp_async_wait<1>();
    else cp_async_wait<0>();
    __syncthreads();
    const unsigned char* vbuf = buf + (size_t)(c & 1) * C::BUF;
    const int jn = min(KC, N - (c - nc) * KC);
    const float* Sc = S + (size_t)(c - nc) * KC * kSmallSP;
#pragma unroll 4
    for (int jl = g; jl < jn; jl += GP) {
      float x[4];
      load4(reinterpret_cast<const T*>(vbuf + (size_t)jl * C::RS) + 4 * s, x);
      const float* pj = Sc + (size_t)jl * kSmallSP;
#pragma unroll
      for (int r = 0; r < kSmallRows; ++r) {
        const float p = pj[r];
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[r][e] = fmaf(p, x[e], acc[r][e]);
      }
    }
    __syncthreads();
  }
  // lanes of a warp that share a piece, then the warps through shared memory
#pragma unroll
  for (int o = NP; o < 32; o <<= 1)
#pragma unroll
    for (int r = 0; r < kSmallRows; ++r)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[r][e] += __shfl_xor_sync(0xffffffffu, acc[r][e], o);
  float* red = reinterpret_cast<float*>(buf);                          // [warps][rows][D]
  if (lane < NP) {
#pragma unroll
    for (int r = 0; r < kSmallRows; ++r)
      *reinterpret_cast<float4*>(red + ((size_t)warp * kSmallRows + r) * D + 4 * s) =
          make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
  }
  __syncthreads();
  for (int t = tid; t < nrows * D; t += kSmallThreads) {
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < kSmallThreads / 32; ++w) sum += red[(size_t)w * kSmallRows * D + t];
    const int r = t / D;
    v_tilde[(row0 + r) * D + t % D] = sum / lsum_s[r];
  }
}

template <typename T, int D>
cudaError_t run(const T* qt, const T* k, const T* v, int BH, int N, int m, int topk,
                const LandmarkPlan& p, const LandmarkWs& ws, int32_t* topk_idx, float* vt,
                int* status, cudaStream_t st, bool prezeroed) {
  cudaError_t e = cudaSuccess;
  if (!prezeroed && (e = cudaMemsetAsync(ws.nslow, 0, sizeof(int), st)) != cudaSuccess) return e;
  if constexpr (std::is_same<T, bf16>::value && D == 64) {
    if (p.tc) {
      e = launch_landmark_tc_passes(qt, k, v, BH, N, m, topk, p, ws, vt, status, st);
      if (e != cudaSuccess) return e;
      const size_t ssmem = (size_t)p.cap * 8 + (size_t)kBandCap * (sizeof(F2) + 4) +
                           (size_t)next_pow2(topk) * 4;
      auto sk = landmark_select_kernel<T, D>;
      e = cudaFuncSetAttribute(sk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ssmem);
      if (e != cudaSuccess) return e;
      e = launch_pdl(sk, dim3((unsigned)((long long)BH * m)), dim3(256), ssmem, st, qt, k, N, m,
                     topk, p.cap, p.P, ws, topk_idx);
      count_launch();
      if (e != cudaSuccess) return e;
      e = launch_pdl(landmark_exact_kernel<T, D>, dim3(kExactCtas), dim3(512), 0, st, qt, k, N, m,
                     topk, ws, topk_idx);
      count_launch();
      return e;
    }
  }
  (void)status;
  if (p.small) {
    const int groups = (m + kSmallRows - 1) / kSmallRows;
    const int rpg = (m + groups - 1) / groups;
    const size_t smem = small_smem_bytes<T, D>(N);
    auto kern = landmark_small_kernel<T, D>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(kern, dim3((unsigned)((long long)BH * groups)), dim3(kSmallThreads), smem, st,
                   qt, k, v, N, m, groups, rpg, topk, ws, topk_idx, vt);
    count_launch();
    if (e != cudaSuccess) return e;
    e = launch_pdl(landmark_exact_kernel<T, D>, dim3(kExactCtas), dim3(512), 0, st, qt, k, N, m,
                   topk, ws, topk_idx);
    count_launch();
    return e;
  }
  switch (p.RT) {
    case 32: e = run_partial<T, D, 32>(qt, k, v, BH, N, m, p, ws, st); break;
    case 64: e = run_partial<T, D, 64>(qt, k, v, BH, N, m, p, ws, st); break;
    default: e = run_partial<T, D, 128>(qt, k, v, BH, N, m, p, ws, st); break;
  }
  if (e != cudaSuccess) return e;
  const size_t msmem = (size_t)p.P * 8 + (size_t)kBandCap * (sizeof(F2) + 4);
  auto mk = landmark_merge_kernel<T, D>;
  e = cudaFuncSetAttribute(mk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)msmem);
  if (e != cudaSuccess) return e;
  mk<<<(unsigned)((long long)BH * m), 256, msmem, st>>>(qt, k, N, m, topk, p.S, p.Tcap, p.P,
                                                        ws, topk_idx, vt);
  count_launch();
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  landmark_exact_kernel<T, D><<<kExactCtas, 512, 0, st>>>(qt, k, N, m, topk, ws, topk_idx);
  count_launch();
  return cudaGetLastError();
}

}  // namespace

LandmarkPlan plan_landmark(int BH, int N, int d, int m, int topk, int num_sms, bool bf16_input) {
  LandmarkPlan p{};
  if (bf16_input && landmark_tc_eligible(d, N, topk)) {
    plan_landmark_tc(p, BH, N, m, topk, num_sms);
    return p;
  }
  p.tc = false;
  if (N <= kSmallMaxN) {
    // one CTA per block of landmark rows of a head, all N keys staged through shared memory
    p.small = true;
    p.RT = kSmallRows;
    p.nrt = 1;
    p.S = 1;
    p.split_len = N;
    p.Tcap = 0;
    p.cap = 0;
    p.P = 0;
    p.ntiles = 0;
    return p;
  }
  p.RT = m >= 128 ? 128 : (m > 32 ? 64 : 32);
  p.nrt = (m + p.RT - 1) / p.RT;
  p.Tcap = std::min(kTcapMax, topk + 32);
  const long long ctas_per_split = (long long)BH * p.nrt;
  const long long target = 2LL * std::max(num_sms, 1);
  int s_occ = (int)std::max(1LL, (target + ctas_per_split - 1) / ctas_per_split);
  int s_need = (p.Tcap < topk + 32) ? (2 * (topk + 32) + p.Tcap - 1) / p.Tcap : 1;
  int S = std::max(s_occ, s_need);
  S = std::min(S, std::max(1, (N + 31) / 32));      // at least 32 keys per split
  S = std::min(S, std::max(s_need, 256));
  p.split_len = (N + S - 1) / S;
  p.S = (N + p.split_len - 1) / p.split_len;        // no empty split
  p.P = next_pow2(std::max(p.S * p.Tcap, 2));
  return p;
}

size_t landmark_ws_bytes(const LandmarkPlan& p, int BH, int N, int d, int m) {
  const size_t rows = (size_t)BH * m;
  const size_t parts = rows * (p.tc ? 2 * p.S : p.S);
  size_t b = 0;
  auto add = [&](size_t n) { b += (n + 255) / 256 * 256; };
  add(parts * 4); add(parts * 4); add(parts * d * 4);
  if (!p.tc && !p.small) {
    add(parts * p.Tcap * 4); add(parts * p.Tcap * 4); add(parts * 4); add(parts * 4);
  }
  add((size_t)BH * p.S * std::max(1, p.nrt) * 4);
  add(4); add(rows * 4);
  add((size_t)kExactCtas * N * 8);
  if (p.tc) {
    add((size_t)p.ntiles * rows * 4);
    add(rows * 4); add(rows * 4); add(rows * 4);
    add(rows * p.cap * 4); add(rows * p.cap * 4);
  }
  return b;
}

LandmarkWs carve_landmark_ws(void* base, const LandmarkPlan& p, int BH, int N, int d, int m) {
  const size_t rows = (size_t)BH * m;
  const size_t parts = rows * (p.tc ? 2 * p.S : p.S);
  char* c = static_cast<char*>(base);
  auto take = [&](size_t n) { char* r = c; c += (n + 255) / 256 * 256; return r; };
  LandmarkWs w{};
  w.M = (float*)take(parts * 4);
  w.L = (float*)take(parts * 4);
  w.A = (float*)take(parts * d * 4);
  if (!p.tc && !p.small) {
    w.cs = (float*)take(parts * p.Tcap * 4);
    w.ci = (int*)take(parts * p.Tcap * 4);
    w.cn = (int*)take(parts * 4);
    w.theta = (float*)take(parts * 4);
  }
  w.kmax2 = (float*)take((size_t)BH * p.S * std::max(1, p.nrt) * 4);
  w.nslow = (int*)take(4);
  w.slow_rows = (int*)take(rows * 4);
  w.exact = (double*)take((size_t)kExactCtas * N * 8);
  if (p.tc) {
    w.bm = (float*)take((size_t)p.ntiles * rows * 4);
    w.thr = (float*)take(rows * 4);
    w.E = (float*)take(rows * 4);
    w.cnt = (int*)take(rows * 4);
    w.cand_s = (float*)take(rows * p.cap * 4);
    w.cand_i = (int*)take(rows * p.cap * 4);
  }
  return w;
}

template <typename T>
cudaError_t launch_landmark(const T* q_tilde, const T* k, const T* v, int BH, int N, int d,
                            int m, int topk, const LandmarkPlan& plan, const LandmarkWs& ws,
                            int32_t* topk_idx, float* v_tilde, int* status, cudaStream_t st,
                            bool prezeroed) {
#define MITA_LM_CASE(DD)                                                                     \
  case DD:                                                                                   \
    return run<T, DD>(q_tilde, k, v, BH, N, m, topk, plan, ws, topk_idx, v_tilde, status, st, \
                      prezeroed);
  switch (d) {
    MITA_LM_CASE(16)
    MITA_LM_CASE(32)
    MITA_LM_CASE(64)
    MITA_LM_CASE(128)
    default: return cudaErrorInvalidValue;
  }
#undef MITA_LM_CASE
}

template cudaError_t launch_landmark<float>(const float*, const float*, const float*, int, int,
                                            int, int, int, const LandmarkPlan&,
                                            const LandmarkWs&, int32_t*, float*, int*,
                                            cudaStream_t, bool);
template cudaError_t launch_landmark<bf16>(const bf16*, const bf16*, const bf16*, int, int, int,
                                           int, int, const LandmarkPlan&, const LandmarkWs&,
                                           int32_t*, float*, int*, cudaStream_t, bool);

}  // namespace mita
