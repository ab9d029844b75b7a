// Step 4 on the tensor cores: route each query to its best landmark (s = 1),
// bf16, d = 64, m <= 512.
//
// MiTA tutorial (iwxt.cn), ch. 4 step 4 (paper eq. 10): q . q~_i over the m
// landmarks selects the expert; there is no gate.
//
// One CTA owns a head's landmark block q~ (TMA, resident in shared memory)
// and walks query tiles of 128 rows of that head:
//   warp 0      TMA producer: query tiles into a 3-stage ring;
//   warp 1      MMA issuer: S = Q_tile . q~^T into tensor memory, in chunks of
//               W <= 256 landmarks, two chunk buffers (ping-pong);
//   warps 4-11  epilogue: TMEM lane quadrant = warp % 4 (one query row per
//               thread), two warps per quadrant split each chunk's columns.
// Each thread keeps the best and runner-up fp32 scores of its query with
// branch-free min/max (the index of the best is looked up only in the rare
// 16-score group that raises it).  If the runner-up is
// within 2E of the best (E bounds the fp32 dot error), the warp re-scores the
// query's plausible winners with exact-product fp32 arithmetic (no fp64: it
// runs at a small fraction of the fp32 rate here).  The result is the exact
// argmax, ties to the lowest landmark index.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"

namespace mita {
namespace {
using namespace sm100;

constexpr int kQStages = 3;
constexpr int kEpiWarps = 8;
constexpr int kThreads = (4 + kEpiWarps) * 32;
constexpr int kMaxM = 512;

struct Cand {
  float v1, v2;   // best and runner-up fp32 scores
  int i1;         // lowest index reaching v1
};

struct alignas(1024) RouteSmem {
  bf16 qt[kMaxM * 64];                 // landmark rows, 128B-swizzled
  bf16 q[kQStages][128 * 64];          // query tiles, 128B-swizzled
  uint64_t q_full[kQStages], q_empty[kQStages];
  uint64_t qt_full, drain;
  uint64_t s_full[2], s_empty[2];
  Cand cand[2][128];                   // half-1 partial results, by tile parity
  float red[kEpiWarps];
  float qtmax2;
  uint32_t tmem;
};

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// Row r (128 bytes) of a 128B-swizzled bf16 tile -> 64 floats.
__device__ __forceinline__ void load_swizzled_row(const bf16* tile, int r, float* out) {
  const char* base = reinterpret_cast<const char*>(tile);
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    uint4 x = *reinterpret_cast<const uint4*>(base + sw128_offset(r, c));
    uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      out[c * 8 + 2 * i] = __uint_as_float(w[i] << 16);
      out[c * 8 + 2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
}

// Exact-enough score of swizzled row ra of `ta` against row rb of `tb`.
__device__ __forceinline__ F2 dot_rows_f2(const bf16* ta, int ra, const bf16* tb, int rb) {
  float a[64], b[64];
  load_swizzled_row(ta, ra, a);
  load_swizzled_row(tb, rb, b);
  return dot_f2<64>(a, b);
}

// Whole-warp exact argmax for every lane that flagged a near tie: the warp
// splits the m landmarks, screens them with fp32 dots (a landmark can win only
// if its fp32 score is within 2E of the tensor-core best), re-scores the
// survivors with dot_f2 and reduces (score desc, index asc).
__device__ void resolve_near_ties(const bf16* qtile, const bf16* qt, int m, int row, bool need,
                                  float best, float twoE, int& ib) {
  const int lane = threadIdx.x & 31;
  unsigned mask = __ballot_sync(0xffffffffu, need);
  while (mask) {
    const int src = __ffs(mask) - 1;
    mask &= mask - 1;
    const int srow = __shfl_sync(0xffffffffu, row, src);
    const float sbest = __shfl_sync(0xffffffffu, best, src);
    const float stwoE = __shfl_sync(0xffffffffu, twoE, src);
    float qr[64];
    load_swizzled_row(qtile, srow, qr);
    F2 bv{-INFINITY, 0.f};
    int bi = 0x7fffffff;
    for (int i = lane; i < m; i += 32) {
      float r[64];
      load_swizzled_row(qt, i, r);
      float d = 0.f;
#pragma unroll
      for (int l = 0; l < 64; ++l) d = fmaf(qr[l], r[l], d);
      if (d >= sbest - stwoE) {
        const F2 x = dot_f2<64>(qr, r);
        if (ranks_before(x, i, bv, bi)) { bv = x; bi = i; }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const F2 ov{__shfl_xor_sync(0xffffffffu, bv.hi, o), __shfl_xor_sync(0xffffffffu, bv.lo, o)};
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ranks_before(ov, oi, bv, bi)) { bv = ov; bi = oi; }
    }
    if (lane == src) ib = bi;
  }
}

__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Running best value v1 (at index i1, the lowest index reaching it) and
// runner-up value v2, over 16 scores starting at index i0.  Branch-free except
// for the rare group that raises v1, where the index is looked up.
__device__ __forceinline__ void top2_group(Cand& c, const float* v, int i0, int nvalid) {
  const float before = c.v1;
#pragma unroll
  for (int i = 0; i < 16; i += 2) {
    const float a = (i < nvalid) ? v[i] : -INFINITY;
    const float b = (i + 1 < nvalid) ? v[i + 1] : -INFINITY;
    const float hi = fmaxf(a, b), lo = fminf(a, b);
    c.v2 = max3f(c.v2, lo, fminf(c.v1, hi));
    c.v1 = fmaxf(c.v1, hi);
  }
  if (c.v1 > before) {
    int k = 0;
#pragma unroll
    for (int i = 15; i >= 0; --i)
      if (i < nvalid && v[i] == c.v1) k = i;
    c.i1 = i0 + k;
  }
}

__global__ void __launch_bounds__(kThreads, 1)
route_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_qt,
                int N, int m, int W, int nch, int G_h, uint32_t tmem_cols,
                int32_t* __restrict__ route, int* status) {
  extern __shared__ unsigned char smem_raw[];
  RouteSmem& s = *reinterpret_cast<RouteSmem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.x / G_h, c0 = blockIdx.x % G_h;
  const int nqt = (N + 127) / 128;
  const int ntiles = (c0 < nqt) ? (nqt - c0 + G_h - 1) / G_h : 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kQStages; ++i) {
      mbar_init(&s.q_full[i], 1);
      mbar_init(&s.q_empty[i], 1 + kEpiWarps);
    }
    mbar_init(&s.qt_full, 1);
    mbar_init(&s.drain, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s.s_full[b], 1);
      mbar_init(&s.s_empty[b], kEpiWarps);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&s.tmem, tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = s.tmem;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&map_q);
      prefetch_tmap(&map_qt);
      mbar_expect_tx(&s.qt_full, (uint32_t)(nch * W * 128));
      for (int ch = 0; ch < nch; ++ch)
        tma_load_3d(s.qt + ch * W * 64, &map_qt, &s.qt_full, 0, ch * W, bh);
      for (int it = 0; it < ntiles; ++it) {
        const int st = it % kQStages;
        if (!mbar_wait(&s.q_empty[st], ((it / kQStages) & 1) ^ 1)) {
          flag_error(status, kDevErrTimeout);
          break;
        }
        mbar_expect_tx(&s.q_full[st], 128 * 128);
        tma_load_3d(s.q[st], &map_q, &s.q_full[st], 0, (c0 + it * G_h) * 128, bh);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(128, W, false);
      bool ok = mbar_wait(&s.qt_full, 0);
      int gch = 0;
      for (int it = 0; it < ntiles && ok; ++it) {
        const int st = it % kQStages;
        if (!mbar_wait(&s.q_full[st], (it / kQStages) & 1)) { ok = false; break; }
        tc_fence_after();
        for (int ch = 0; ch < nch; ++ch, ++gch) {
          const int b = gch & 1;
          if (!mbar_wait(&s.s_empty[b], ((gch >> 1) & 1) ^ 1)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t da = smem_desc_sw128(smem_u32(s.q[st]) + kk * 32, 1024);
            const uint64_t db = smem_desc_sw128(smem_u32(s.qt + ch * W * 64) + kk * 32, 1024);
            mma_ss(tbase + b * W, da, db, idesc, kk > 0);
          }
          mma_commit(&s.s_full[b]);
        }
        mma_commit(&s.q_empty[st]);
      }
      if (!ok) flag_error(status, kDevErrTimeout);
      mma_commit(&s.drain);
      mbar_wait(&s.drain, 0);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue
    const int et = threadIdx.x - 128;              // 0..255
    const int quad = warp & 3, half = (warp - 4) >> 2;
    const int row = quad * 32 + lane;
    const uint32_t taddr_lane = (uint32_t)(quad * 32) << 16;
    bool ok = mbar_wait(&s.qt_full, 0);
    // largest landmark norm of the head (error bound)
    float n2max = 0.f;
    if (ok) {
      for (int i = et; i < m; i += 256) {
        float r[64];
        load_swizzled_row(s.qt, i, r);
        float a = 0.f;
#pragma unroll
        for (int l = 0; l < 64; ++l) a = fmaf(r[l], r[l], a);
        n2max = fmaxf(n2max, a);
      }
    }
    n2max = warp_max(n2max);
    if (lane == 0) s.red[warp - 4] = n2max;
    epi_bar();
    float qtmax2 = 0.f;
    for (int i = 0; i < kEpiWarps; ++i) qtmax2 = fmaxf(qtmax2, s.red[i]);
    const float gam = err_gamma(64);
    const int cols_half = W / 2;
    int gch = 0;
    for (int it = 0; it < ntiles; ++it) {
      const int st = it % kQStages;
      if (ok && !mbar_wait(&s.q_full[st], (it / kQStages) & 1)) ok = false;
      Cand c{-INFINITY, -INFINITY, 0x7fffffff};
      for (int ch = 0; ch < nch; ++ch, ++gch) {
        const int b = gch & 1;
        if (ok && !mbar_wait(&s.s_full[b], (gch >> 1) & 1)) ok = false;
        tc_fence_after();
        if (ok) {
          const int col0 = half * cols_half;
          for (int cc = 0; cc < cols_half; cc += 16) {
            float v[16];
            tmem_ld16(tbase + taddr_lane + (uint32_t)(b * W + col0 + cc), v);
            tmem_ld_wait();
            const int i0 = ch * W + col0 + cc;
            top2_group(c, v, i0, m - i0);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.s_empty[b]);
      }
      if (half == 1) {
        s.cand[it & 1][row] = c;
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.q_empty[st]);
      }
      epi_bar();
      if (half == 0) {
        const Cand o = s.cand[it & 1][row];
        // merge the two halves: best (ties to the lower index) and runner-up
        Cand r = c;
        const bool w1 = o.v1 > c.v1 || (o.v1 == c.v1 && o.i1 < c.i1);
        r.v2 = max3f(c.v2, o.v2, fminf(c.v1, o.v1));
        if (w1) { r.v1 = o.v1; r.i1 = o.i1; }
        const int n = (c0 + it * G_h) * 128 + row;
        const bool live = ok && n < N;
        float twoE = 0.f;
        if (live) {
          float qr[64];
          load_swizzled_row(s.q[st], row, qr);
          float qn2 = 0.f;
#pragma unroll
          for (int l = 0; l < 64; ++l) qn2 = fmaf(qr[l], qr[l], qn2);
          twoE = 2.f * gam * sqrtf(qn2) * sqrtf(qtmax2);
        }
        int ib = r.i1;
        resolve_near_ties(s.q[st], s.qt, m, row, live && (r.v1 - r.v2 <= twoE), r.v1, twoE, ib);
        if (live) route[(size_t)bh * N + n] = ib;
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.q_empty[st]);
      }
    }
    if (!ok) flag_error(status, kDevErrTimeout);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, tmem_cols);
}

}  // namespace

size_t route_tc_smem_bytes() { return sizeof(RouteSmem) + 1024; }

bool route_tc_supported(int d, int m) { return d == 64 && m >= 1 && m <= kMaxM; }

cudaError_t launch_route_tc(const bf16* q, const bf16* q_tilde, int BH, int N, int m,
                            int num_sms, int32_t* route, int* status, cudaStream_t st) {
  const int W = std::min(256, (m + 31) / 32 * 32);
  const int nch = (m + W - 1) / W;
  uint32_t cols = 32;
  while (cols < (uint32_t)(2 * W)) cols <<= 1;
  CUtensorMap mq, mqt;
  if (!make_tmap_rows64(&mq, q, (uint64_t)N, (uint64_t)BH, 128) ||
      !make_tmap_rows64(&mqt, q_tilde, (uint64_t)m, (uint64_t)BH, (uint32_t)W))
    return cudaErrorInvalidValue;
  const int nqt = (N + 127) / 128;
  int G_h = std::max(1, (num_sms + BH - 1) / BH);
  G_h = std::min(G_h, nqt);
  const size_t smem = route_tc_smem_bytes();
  cudaError_t e = cudaFuncSetAttribute(route_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  route_tc_kernel<<<(unsigned)(BH * G_h), kThreads, smem, st>>>(mq, mqt, N, m, W, nch, G_h, cols,
                                                                 route, status);
  return cudaGetLastError();
}

}  // namespace mita
