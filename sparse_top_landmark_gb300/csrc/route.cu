// Step 4: route each query to its top-s landmarks.
//
// MiTA tutorial (iwxt.cn), ch. 4 step 4 (paper eq. 10): a query compares
// q . q~_i over the m landmarks and keeps the top-s indices, best first; the
// scores only select (no gate).  gist.science summary Sec. 2.2: s = 1 in
// practice.  The bit.fan article notes that the query-landmark logits are
// reused as the shared-branch logits; this kernel can emit that branch's
// partial (log-sum-exp and normalised output over the m shared pairs), its
// logits scaled by 1/sqrt(d) or, on request, by 1/d (the official code's
// temperature, tutorial ch. 8 caveat 3).
//
// Exactness: each thread keeps its s + 1 best fp32 scores in a sorted
// register list.  The list is accepted when every neighbouring pair in it
// differs by more than 2E (E bounds the fp32 dot error), i.e. neither the
// order of the s chosen landmarks nor the cut after the s-th can change in
// exact arithmetic; otherwise every landmark within 2E of the s-th score is
// re-scored with exact-product fp32 arithmetic and the exact top-s wins, ties
// to the lowest landmark index.
#include "common.cuh"
#include "kernels.h"

namespace mita {
namespace {

constexpr int kRouteThreads = 128;   // one query per thread
constexpr int kLmChunk = 32;         // landmarks staged per smem chunk

// Insert (x, i) into the descending list (v, id)[0..L); equal scores keep the
// earlier entry first (landmarks arrive in ascending index order).
template <int L, typename S>
__device__ __forceinline__ void list_insert(S (&v)[L], int (&id)[L], S x, int i) {
#pragma unroll
  for (int t = 0; t < L; ++t) {
    const bool take = x > v[t];
    const S tv = take ? v[t] : x;
    const int ti = take ? id[t] : i;
    v[t] = take ? x : v[t];
    id[t] = take ? i : id[t];
    x = tv;
    i = ti;
  }
}

// L = length of the kept list: 2 for s = 1 (best and runner-up), kMaxRouteS + 1 otherwise.
template <typename T, int D, int L>
__global__ void __launch_bounds__(kRouteThreads)
route_kernel(const T* __restrict__ q, const T* __restrict__ q_tilde,
             const float* __restrict__ v_tilde, int N, int m, int s, float c,
             int32_t* __restrict__ route, float* __restrict__ shared_lse,
             float* __restrict__ shared_o) {
  __shared__ __align__(16) float qs[kLmChunk][D];
  __shared__ __align__(16) float vs[kLmChunk][D];
  __shared__ float red[kRouteThreads / 32];
  const bool want_shared = shared_o != nullptr || shared_lse != nullptr;
  const int nqt = (N + kRouteThreads - 1) / kRouteThreads;
  const long long bh = blockIdx.x / nqt;
  const int n = (blockIdx.x % nqt) * kRouteThreads + threadIdx.x;
  const bool live = n < N;
  const T* qtb = q_tilde + (size_t)bh * m * D;

  // max landmark norm of this head (for the error bound)
  float qt2 = 0.f;
  for (int i = threadIdx.x; i < m; i += kRouteThreads) {
    float r[D];
    load_row<T, D>(qtb + (size_t)i * D, r);
    float nn = 0.f;
#pragma unroll
    for (int l = 0; l < D; ++l) nn = fmaf(r[l], r[l], nn);
    qt2 = fmaxf(qt2, nn);
  }
  qt2 = block_max(qt2, red);

  float qr[D];
  if (live) load_row<T, D>(q + ((size_t)bh * N + n) * D, qr);
  else {
#pragma unroll
    for (int l = 0; l < D; ++l) qr[l] = 0.f;
  }
  float qn2 = 0.f;
#pragma unroll
  for (int l = 0; l < D; ++l) qn2 = fmaf(qr[l], qr[l], qn2);

  float bv[L];
  int bi[L];
#pragma unroll
  for (int t = 0; t < L; ++t) { bv[t] = -INFINITY; bi[t] = 0; }
  float mrun = -INFINITY, lsum = 0.f;
  float acc[D];
#pragma unroll
  for (int l = 0; l < D; ++l) acc[l] = 0.f;

  for (int i0 = 0; i0 < m; i0 += kLmChunk) {
    const int nc = min(kLmChunk, m - i0);
    __syncthreads();
    for (int e = threadIdx.x; e < nc * D; e += kRouteThreads) {
      const int t = e / D, l = e % D;
      qs[t][l] = to_f(qtb[(size_t)(i0 + t) * D + l]);
      if (want_shared) vs[t][l] = v_tilde[((size_t)bh * m + i0 + t) * D + l];
    }
    __syncthreads();
    if (!live) continue;
    for (int t = 0; t < nc; ++t) {
      float sc0 = 0.f;
#pragma unroll
      for (int l = 0; l < D; ++l) sc0 = fmaf(qr[l], qs[t][l], sc0);
      if (sc0 > bv[L - 1]) list_insert<L>(bv, bi, sc0, i0 + t);
      if (want_shared) {
        const float x = sc0 * c;
        if (x > mrun) {
          const float sc = exp2f(mrun - x);
          lsum *= sc;
#pragma unroll
          for (int l = 0; l < D; ++l) acc[l] *= sc;
          mrun = x;
        }
        const float p = exp2f(x - mrun);
        lsum += p;
#pragma unroll
        for (int l = 0; l < D; ++l) acc[l] = fmaf(p, vs[t][l], acc[l]);
      }
    }
  }
  if (!live) return;

  const float E = err_gamma(D) * sqrtf(qn2) * sqrtf(qt2);
  // the s-th kept score, and whether any neighbouring pair up to the (s+1)-th is within 2E
  float cut = bv[0];
  bool near = false;
#pragma unroll
  for (int t = 0; t + 1 < L; ++t) {
    if (t < s) {
      cut = bv[t];
      near = near || (bv[t] - bv[t + 1] <= 2.f * E);
    }
  }
  const size_t qi = (size_t)bh * N + n;
  if (near) {
    // near tie: re-score every landmark that can still be among the exact top-s
    F2 xv[L];
    int xi[L];
#pragma unroll
    for (int t = 0; t < L; ++t) { xv[t] = F2{-INFINITY, 0.f}; xi[t] = 0; }
    for (int i = 0; i < m; ++i) {
      float r[D];
      load_row<T, D>(qtb + (size_t)i * D, r);
      float sf = 0.f;
#pragma unroll
      for (int l = 0; l < D; ++l) sf = fmaf(qr[l], r[l], sf);
      if (sf >= cut - 2.f * E) {
        F2 x = dot_f2<D>(qr, r);
        int ix = i;
#pragma unroll
        for (int t = 0; t < L; ++t) {
          const bool take = f2_greater(x, xv[t]);
          const F2 tv = take ? xv[t] : x;
          const int ti = take ? xi[t] : ix;
          xv[t] = take ? x : xv[t];
          xi[t] = take ? ix : xi[t];
          x = tv;
          ix = ti;
        }
      }
    }
#pragma unroll
    for (int t = 0; t < L; ++t) bi[t] = xi[t];
  }
#pragma unroll
  for (int t = 0; t < L; ++t)
    if (t < s) route[qi * s + t] = bi[t];
  if (want_shared) {
    const float inv = 1.f / lsum;
    if (shared_lse) shared_lse[qi] = (mrun + log2f(lsum)) * 0.6931471805599453f;  // natural log
    if (shared_o) {
#pragma unroll
      for (int l = 0; l < D; ++l) shared_o[qi * D + l] = acc[l] * inv;
    }
  }
}

template <typename T, int D>
cudaError_t run(const T* q, const T* qt, const float* vt, int BH, int N, int m, int s,
                int32_t* route, float* lse, float* o, int temp, cudaStream_t st) {
  const long long nqt = (N + kRouteThreads - 1) / kRouteThreads;
  const dim3 grid((unsigned)(BH * nqt));
  // shared logits in log2 units: log2(e) / sqrt(d), or log2(e) / d
  const float c = (float)(1.4426950408889634 / (temp ? (double)D : sqrt((double)D)));
  if (s == 1)
    route_kernel<T, D, 2><<<grid, kRouteThreads, 0, st>>>(q, qt, vt, N, m, 1, c, route, lse, o);
  else
    route_kernel<T, D, kMaxRouteS + 1><<<grid, kRouteThreads, 0, st>>>(q, qt, vt, N, m, s, c,
                                                                        route, lse, o);
  count_launch();
  return cudaGetLastError();
}

}  // namespace

template <typename T>
cudaError_t launch_route(const T* q, const T* q_tilde, const float* v_tilde, int BH, int N,
                         int d, int m, int s, int32_t* route_idx, float* shared_lse,
                         float* shared_o, cudaStream_t st, int shared_temp) {
  if (s < 1 || s > kMaxRouteS || s > m) return cudaErrorInvalidValue;
  switch (d) {
    case 16: return run<T, 16>(q, q_tilde, v_tilde, BH, N, m, s, route_idx, shared_lse, shared_o, shared_temp, st);
    case 32: return run<T, 32>(q, q_tilde, v_tilde, BH, N, m, s, route_idx, shared_lse, shared_o, shared_temp, st);
    case 64: return run<T, 64>(q, q_tilde, v_tilde, BH, N, m, s, route_idx, shared_lse, shared_o, shared_temp, st);
    case 128: return run<T, 128>(q, q_tilde, v_tilde, BH, N, m, s, route_idx, shared_lse, shared_o, shared_temp, st);
    default: return cudaErrorInvalidValue;
  }
}

template cudaError_t launch_route<float>(const float*, const float*, const float*, int, int, int,
                                         int, int, int32_t*, float*, float*, cudaStream_t, int);
template cudaError_t launch_route<bf16>(const bf16*, const bf16*, const float*, int, int, int,
                                        int, int, int32_t*, float*, float*, cudaStream_t, int);

}  // namespace mita
