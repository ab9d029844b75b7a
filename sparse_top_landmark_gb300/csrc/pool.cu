// Step 1: landmark queries by local average pooling of Q.
//
// MiTA tutorial (iwxt.cn), ch. 4 step 1 (paper Sec. 3.2, eq. 5): every
// landmark query is the mean of a group of queries; the bit.fan article calls
// it local average pooling; tutorial ch. 5 pools a 2 x 4 token grid in 2D.
// Windows follow the adaptive-average-pool rule on the grid_h x grid_w token
// grid onto an mh x mw landmark grid (1D: 1 x N pooled to 1 x m; 2D: by
// default sqrt(m) x sqrt(m), or any mh x mw = m the caller gives).
//
// HBM-bound: one CTA per landmark streams its window once with 16-byte loads
// (one warp per landmark when windows are small).
// Sums are error-free (fp32 two-sum per thread and across threads; one fp64
// division per output), so the mean is rounded once into the input dtype --
// the same value an fp64 mean
// rounded to nearest gives.
#include "common.cuh"
#include "kernels.h"

#include <algorithm>

namespace mita {
namespace {

// 128 threads, up to eight CTAs per SM: the B*H*m windows of the long workloads (1 024)
// then run in a single wave on 152 SMs instead of 1.7 waves of 256-thread CTAs
constexpr int kPoolThreads = 128;

template <typename T, int D>
__global__ void __launch_bounds__(kPoolThreads, 8)
pool_kernel(const T* __restrict__ q, int N, int grid_h, int grid_w, int mh, int mw,
            T* __restrict__ q_tilde) {
  griddep_wait();
  constexpr int VEC = Vec<T>::N;
  constexpr int NV = D / VEC;              // 16-byte vectors per row
  constexpr int TL = kPoolThreads / NV;    // token lanes
  constexpr int UNR = 8;                   // 16-byte loads in flight per thread
  static_assert(D % VEC == 0, "row must be a whole number of 16-byte vectors");
  __shared__ float red_s[TL][D], red_c[TL][D];

  const int m = mh * mw;
  const long long flat = blockIdx.x;       // bh * m + i
  const int i = (int)(flat % m);
  const long long bh = flat / m;
  int r0, r1, c0, c1;
  adaptive_window(i / mw, grid_h, mh, &r0, &r1);
  adaptive_window(i % mw, grid_w, mw, &c0, &c1);
  const int nc = c1 - c0;
  const int cnt = (r1 - r0) * nc;
  const bool one_row = r1 - r0 == 1;       // 1D windows are contiguous

  const int vlane = threadIdx.x % NV, tl = threadIdx.x / NV;
  float s[VEC], c[VEC];
#pragma unroll
  for (int e = 0; e < VEC; ++e) { s[e] = 0.f; c[e] = 0.f; }
  const T* base = q + (size_t)bh * N * D + vlane * VEC;
  for (int t0 = tl; t0 < cnt; t0 += TL * UNR) {
    uint4 raw[UNR];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int t = t0 + u * TL;
      if (t < cnt) {
        const size_t tok = one_row ? (size_t)r0 * grid_w + c0 + t
                                   : (size_t)(r0 + t / nc) * grid_w + c0 + t % nc;
        raw[u] = *reinterpret_cast<const uint4*>(base + tok * D);
      } else {
        raw[u] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      float x[VEC];
      Vec<T>::load(reinterpret_cast<const T*>(&raw[u]), x);
#pragma unroll
      for (int e = 0; e < VEC; ++e) two_sum_acc(s[e], c[e], x[e]);
    }
  }
#pragma unroll
  for (int e = 0; e < VEC; ++e) {
    red_s[tl][vlane * VEC + e] = s[e];
    red_c[tl][vlane * VEC + e] = c[e];
  }
  __syncthreads();
  for (int l = threadIdx.x; l < D; l += kPoolThreads) {
    // error-free combination of the token lanes, then one rounding
    float S = 0.f, C = 0.f;
    for (int t = 0; t < TL; ++t) {
      two_sum_acc(S, C, red_s[t][l]);
      C = __fadd_rn(C, red_c[t][l]);
    }
    q_tilde[flat * D + l] = round_double<T>(((double)S + (double)C) / (double)cnt);
  }
}

// Small windows (the image grids: a few to a few dozen tokens per landmark): one warp per
// landmark and no shared memory or block barrier.  Lanes split into NV 16-byte column slices
// x 32 / NV token lanes; the token lanes' error-free partial sums meet by shuffles.
constexpr int kWarpWindow = 64;

template <typename T, int D>
__global__ void __launch_bounds__(kPoolThreads)
pool_warp_kernel(const T* __restrict__ q, long long rows, int N, int grid_h, int grid_w, int mh,
                 int mw, T* __restrict__ q_tilde) {
  griddep_wait();
  constexpr int VEC = Vec<T>::N;
  constexpr int NV = D / VEC;
  constexpr int TL = 32 / NV;              // token lanes of a warp
  constexpr int UNR = 4;
  static_assert(NV <= 32 && 32 % NV == 0, "a warp spans whole rows");
  const int lane = threadIdx.x & 31;
  const long long flat = (long long)blockIdx.x * (kPoolThreads / 32) + (threadIdx.x >> 5);
  if (flat >= rows) return;                // whole warps
  const int m = mh * mw;
  const int i = (int)(flat % m);
  const long long bh = flat / m;
  int r0, r1, c0, c1;
  adaptive_window(i / mw, grid_h, mh, &r0, &r1);
  adaptive_window(i % mw, grid_w, mw, &c0, &c1);
  const int nc = c1 - c0;
  const int cnt = (r1 - r0) * nc;
  const int vlane = lane % NV, tl = lane / NV;
  float s[VEC], c[VEC];
#pragma unroll
  for (int e = 0; e < VEC; ++e) { s[e] = 0.f; c[e] = 0.f; }
  const T* base = q + (size_t)bh * N * D + vlane * VEC;
  for (int t0 = tl; t0 < cnt; t0 += TL * UNR) {
    uint4 raw[UNR];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int t = t0 + u * TL;
      raw[u] = make_uint4(0u, 0u, 0u, 0u);
      if (t < cnt) {
        const size_t tok = (size_t)(r0 + t / nc) * grid_w + c0 + t % nc;
        raw[u] = *reinterpret_cast<const uint4*>(base + tok * D);
      }
    }
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      float x[VEC];
      Vec<T>::load(reinterpret_cast<const T*>(&raw[u]), x);
#pragma unroll
      for (int e = 0; e < VEC; ++e) two_sum_acc(s[e], c[e], x[e]);
    }
  }
#pragma unroll
  for (int o = NV; o < 32; o <<= 1) {
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
      const float so = __shfl_xor_sync(0xffffffffu, s[e], o);
      const float co = __shfl_xor_sync(0xffffffffu, c[e], o);
      two_sum_acc(s[e], c[e], so);
      c[e] = __fadd_rn(c[e], co);
    }
  }
  // every token lane now holds the slice's sums: lane (tl, vlane) rounds elements
  // tl, tl + TL, ... of the slice, so the fp64 divisions run on all 32 lanes at once
#pragma unroll
  for (int e0 = 0; e0 < VEC; e0 += TL) {
    const int e = e0 + tl;
    float se = s[0], ce = c[0];
#pragma unroll
    for (int u = 1; u < VEC; ++u)
      if (e == u) { se = s[u]; ce = c[u]; }
    if (e < VEC)
      q_tilde[flat * D + vlane * VEC + e] = round_double<T>(((double)se + (double)ce) / (double)cnt);
  }
}

// largest window of the adaptive pooling of an `in`-long axis onto `out` cells
inline int max_window(int in, int out) {
  int w = 0;
  for (int i = 0; i < out; ++i) {
    int lo, hi;
    adaptive_window(i, in, out, &lo, &hi);
    w = std::max(w, hi - lo);
  }
  return w;
}

template <typename T, int D>
cudaError_t run(const T* q, int BH, int N, int grid_h, int grid_w, int mh, int mw, T* qt,
                cudaStream_t st) {
  const long long blocks = (long long)BH * mh * mw;
  cudaError_t e;
  if ((long long)max_window(grid_h, mh) * max_window(grid_w, mw) <= kWarpWindow) {
    const long long wpb = kPoolThreads / 32;
    e = launch_pdl(pool_warp_kernel<T, D>, dim3((unsigned)((blocks + wpb - 1) / wpb)),
                   dim3(kPoolThreads), 0, st, q, blocks, N, grid_h, grid_w, mh, mw, qt);
  } else {
    e = launch_pdl(pool_kernel<T, D>, dim3((unsigned)blocks), dim3(kPoolThreads), 0, st, q, N,
                   grid_h, grid_w, mh, mw, qt);
  }
  count_launch();
  return e;
}

}  // namespace

template <typename T>
cudaError_t launch_pool(const T* q, int BH, int N, int d, int grid_h, int grid_w, int mh,
                        int mw, T* q_tilde, cudaStream_t st) {
  if (mh < 1 || mw < 1) return cudaErrorInvalidValue;
  switch (d) {
    case 16: return run<T, 16>(q, BH, N, grid_h, grid_w, mh, mw, q_tilde, st);
    case 32: return run<T, 32>(q, BH, N, grid_h, grid_w, mh, mw, q_tilde, st);
    case 64: return run<T, 64>(q, BH, N, grid_h, grid_w, mh, mw, q_tilde, st);
    case 128: return run<T, 128>(q, BH, N, grid_h, grid_w, mh, mw, q_tilde, st);
    default: return cudaErrorInvalidValue;
  }
}

template cudaError_t launch_pool<float>(const float*, int, int, int, int, int, int, int, float*,
                                        cudaStream_t);
template cudaError_t launch_pool<bf16>(const bf16*, int, int, int, int, int, int, int, bf16*,
                                       cudaStream_t);

}  // namespace mita
