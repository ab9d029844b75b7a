// Step 4: route each query to its best landmark (s = 1).
//
// MiTA tutorial (iwxt.cn), ch. 4 step 4 (paper eq. 10): a query compares
// q . q~_i over the m landmarks and keeps the top-s indices; the scores only
// select (no gate).  gist.science summary Sec. 2.2: s = 1 in practice.
// The bit.fan article notes that the query-landmark logits are reused as the
// shared-branch logits; this kernel can emit that branch's partial
// (log-sum-exp and normalised output over the m shared pairs).
//
// Exactness: the fp32 argmax is accepted when it beats the runner-up by more
// than 2E (E bounds the fp32 dot error); otherwise every landmark within 2E of
// the best is re-scored with exact-product fp32 arithmetic and the exact
// maximum wins, ties to the lowest landmark index.
#include "common.cuh"
#include "kernels.h"

namespace mita {
namespace {

constexpr int kRouteThreads = 128;   // one query per thread
constexpr int kLmChunk = 32;         // landmarks staged per smem chunk

template <typename T, int D>
__global__ void __launch_bounds__(kRouteThreads)
route_kernel(const T* __restrict__ q, const T* __restrict__ q_tilde,
             const float* __restrict__ v_tilde, int N, int m, int32_t* __restrict__ route,
             float* __restrict__ shared_lse, float* __restrict__ shared_o) {
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
    float s = 0.f;
#pragma unroll
    for (int l = 0; l < D; ++l) s = fmaf(r[l], r[l], s);
    qt2 = fmaxf(qt2, s);
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

  const float c = (float)(1.4426950408889634 / sqrt((double)D));
  float best = -INFINITY, second = -INFINITY;
  int ib = 0;
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
      float s = 0.f;
#pragma unroll
      for (int l = 0; l < D; ++l) s = fmaf(qr[l], qs[t][l], s);
      if (s > best) { second = best; best = s; ib = i0 + t; }
      else if (s > second) second = s;
      if (want_shared) {
        const float x = s * c;
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
  if (best - second <= 2.f * E) {
    // near tie: re-score the candidates exactly
    F2 bx{-INFINITY, 0.f};
    int bi = ib;
    for (int i = 0; i < m; ++i) {
      float r[D];
      load_row<T, D>(qtb + (size_t)i * D, r);
      float s = 0.f;
#pragma unroll
      for (int l = 0; l < D; ++l) s = fmaf(qr[l], r[l], s);
      if (s >= best - 2.f * E) {
        const F2 x = dot_f2<D>(qr, r);
        if (f2_greater(x, bx)) { bx = x; bi = i; }
      }
    }
    ib = bi;
  }
  const size_t qi = (size_t)bh * N + n;
  route[qi] = ib;
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
cudaError_t run(const T* q, const T* qt, const float* vt, int BH, int N, int m, int32_t* route,
                float* lse, float* o, cudaStream_t st) {
  const long long nqt = (N + kRouteThreads - 1) / kRouteThreads;
  route_kernel<T, D><<<(unsigned)(BH * nqt), kRouteThreads, 0, st>>>(q, qt, vt, N, m, route,
                                                                      lse, o);
  count_launch();
  return cudaGetLastError();
}

}  // namespace

template <typename T>
cudaError_t launch_route(const T* q, const T* q_tilde, const float* v_tilde, int BH, int N,
                         int d, int m, int32_t* route_idx, float* shared_lse, float* shared_o,
                         cudaStream_t st) {
  switch (d) {
    case 16: return run<T, 16>(q, q_tilde, v_tilde, BH, N, m, route_idx, shared_lse, shared_o, st);
    case 32: return run<T, 32>(q, q_tilde, v_tilde, BH, N, m, route_idx, shared_lse, shared_o, st);
    case 64: return run<T, 64>(q, q_tilde, v_tilde, BH, N, m, route_idx, shared_lse, shared_o, st);
    case 128: return run<T, 128>(q, q_tilde, v_tilde, BH, N, m, route_idx, shared_lse, shared_o, st);
    default: return cudaErrorInvalidValue;
  }
}

template cudaError_t launch_route<float>(const float*, const float*, const float*, int, int, int,
                                         int, int32_t*, float*, float*, cudaStream_t);
template cudaError_t launch_route<bf16>(const bf16*, const bf16*, const float*, int, int, int,
                                        int, int32_t*, float*, float*, cudaStream_t);

}  // namespace mita
