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
// Each thread keeps the exact best and runner-up fp32 scores of its query
// (branch-free min/max) and a register copy of the 32-score block holding the
// running best, so the best's index (lowest on ties) is looked up once at the
// end.  When the best beats the runner-up by more than 2E (E bounds the fp32
// dot error) it is the exact argmax; otherwise the query goes on an
// "ambiguous" list and route_fixup_kernel re-routes it exactly (fp32
// screening + exact-product re-scoring, ties to the lowest index) -- about
// 0.2% of the queries on the long-sequence workloads.
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
  float v1, v2;   // best and runner-up scores
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

__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Top-2 update over a block of 32 scores starting at index i0 (entries at or
// past nvalid ignored); bb keeps a copy of the block that holds the best.
__device__ __forceinline__ void top2_block(Cand& c, float* bb, int& bb0, const float* v, int i0,
                                           int nvalid) {
  const float before = c.v1;
  if (nvalid >= 32) {
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      const float hi = fmaxf(v[i], v[i + 1]), lo = fminf(v[i], v[i + 1]);
      c.v2 = max3f(c.v2, lo, fminf(c.v1, hi));
      c.v1 = fmaxf(c.v1, hi);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      const float a = (i < nvalid) ? v[i] : -INFINITY;
      const float b = (i + 1 < nvalid) ? v[i + 1] : -INFINITY;
      const float hi = fmaxf(a, b), lo = fminf(a, b);
      c.v2 = max3f(c.v2, lo, fminf(c.v1, hi));
      c.v1 = fmaxf(c.v1, hi);
    }
  }
  const bool up = c.v1 > before;
#pragma unroll
  for (int i = 0; i < 32; ++i) bb[i] = up ? v[i] : bb[i];
  bb0 = up ? i0 : bb0;
}

// lowest index in the saved block whose score equals the best
__device__ __forceinline__ int block_argmax(const float* bb, int bb0, float v1) {
  int k = 31;
#pragma unroll
  for (int i = 31; i >= 0; --i) k = (bb[i] == v1) ? i : k;
  return bb0 + k;
}

__global__ void __launch_bounds__(kThreads, 1)
route_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_qt,
                int N, int m, int W, int nch, int G_h, uint32_t tmem_cols,
                int32_t* __restrict__ route, int* __restrict__ amb, int* status) {
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
      mma_commit(&s.drain);
      if (!mbar_wait(&s.drain, 0)) ok = false;
      if (!ok) flag_error(status, kDevErrTimeout);
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
      float bb[32];
      int bb0 = 0;
#pragma unroll
      for (int i = 0; i < 32; ++i) bb[i] = -INFINITY;
      for (int ch = 0; ch < nch; ++ch, ++gch) {
        const int b = gch & 1;
        if (ok && !mbar_wait(&s.s_full[b], (gch >> 1) & 1)) ok = false;
        tc_fence_after();
        if (ok) {
          const int col0 = half * cols_half;
          for (int cc = 0; cc < cols_half; cc += 32) {
            float v[32];
            const uint32_t ta = tbase + taddr_lane + (uint32_t)(b * W + col0 + cc);
            tmem_ld16(ta, v);                 // cols_half is a multiple of 16
            if (cols_half - cc > 16) tmem_ld16(ta + 16, v + 16);
            tmem_ld_wait();
            const int i0 = ch * W + col0 + cc;
            top2_block(c, bb, bb0, v, i0, min(m - i0, cols_half - cc));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.s_empty[b]);
      }
      if (c.v1 > -INFINITY) c.i1 = block_argmax(bb, bb0, c.v1);
      if (half == 1) {
        s.cand[it & 1][row] = c;
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.q_empty[st]);
      }
      epi_bar();
      if (half == 0) {
        const Cand o = s.cand[it & 1][row];
        const bool w1 = o.v1 > c.v1 || (o.v1 == c.v1 && o.i1 < c.i1);
        const float v1 = w1 ? o.v1 : c.v1;
        const int i1 = w1 ? o.i1 : c.i1;
        const float v2 = max3f(c.v2, o.v2, fminf(c.v1, o.v1));
        const int n = (c0 + it * G_h) * 128 + row;
        const bool live = ok && n < N;
        bool ambiguous = false;
        if (live) {
          float qr[64];
          load_swizzled_row(s.q[st], row, qr);
          float qn2 = 0.f;
#pragma unroll
          for (int l = 0; l < 64; ++l) qn2 = fmaf(qr[l], qr[l], qn2);
          const float twoE = 2.f * gam * sqrtf(qn2) * sqrtf(qtmax2);
          ambiguous = !(v1 - v2 > twoE);
          route[(size_t)bh * N + n] = i1;
        }
        // append ambiguous queries (one reservation per warp)
        const unsigned am = __ballot_sync(0xffffffffu, ambiguous);
        if (am) {
          int base = 0;
          if (lane == 0) base = atomicAdd(amb, __popc(am));
          base = __shfl_sync(0xffffffffu, base, 0);
          if (ambiguous) amb[1 + base + __popc(am & ((1u << lane) - 1u))] = (int)((size_t)bh * N + n);
        }
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

// Exact routing of the ambiguous queries: one warp per query.  Lanes screen
// all m landmarks with fp32 dots (only those within 2E of the fp32 best can
// win), re-score the survivors with exact-product arithmetic and reduce
// (score desc, index asc).
__global__ void __launch_bounds__(256)
route_fixup_kernel(const bf16* __restrict__ q, const bf16* __restrict__ q_tilde, int N, int m,
                   const int* __restrict__ amb, int32_t* __restrict__ route) {
  const int lane = threadIdx.x & 31;
  const int nwarps = gridDim.x * 8;
  const int count = amb[0];
  for (int w = blockIdx.x * 8 + (threadIdx.x >> 5); w < count; w += nwarps) {
    const int qflat = amb[1 + w];
    const int bh = qflat / N;
    float qr[64];
    load_row<bf16, 64>(q + (size_t)qflat * 64, qr);
    float qn2 = 0.f, best = -INFINITY, qt2 = 0.f;
#pragma unroll
    for (int l = 0; l < 64; ++l) qn2 = fmaf(qr[l], qr[l], qn2);
    const bf16* qtb = q_tilde + (size_t)bh * m * 64;
    for (int i = lane; i < m; i += 32) {
      float r[64];
      load_row<bf16, 64>(qtb + (size_t)i * 64, r);
      float d = 0.f, n2 = 0.f;
#pragma unroll
      for (int l = 0; l < 64; ++l) { d = fmaf(qr[l], r[l], d); n2 = fmaf(r[l], r[l], n2); }
      best = fmaxf(best, d);
      qt2 = fmaxf(qt2, n2);
    }
    best = warp_max(best);
    qt2 = warp_max(qt2);
    const float twoE = 2.f * err_gamma(64) * sqrtf(qn2) * sqrtf(qt2);
    F2 bv{-INFINITY, 0.f};
    int bi = 0x7fffffff;
    for (int i = lane; i < m; i += 32) {
      float r[64];
      load_row<bf16, 64>(qtb + (size_t)i * 64, r);
      float d = 0.f;
#pragma unroll
      for (int l = 0; l < 64; ++l) d = fmaf(qr[l], r[l], d);
      if (d >= best - twoE) {
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
    if (lane == 0) route[qflat] = bi;
  }
}

}  // namespace

size_t route_tc_smem_bytes() { return sizeof(RouteSmem) + 1024; }

bool route_tc_supported(int d, int m) { return d == 64 && m >= 1 && m <= kMaxM; }

cudaError_t launch_route_tc(const bf16* q, const bf16* q_tilde, int BH, int N, int m,
                            int num_sms, int32_t* route, int* amb, int* status, cudaStream_t st) {
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
  e = cudaMemsetAsync(amb, 0, sizeof(int), st);
  if (e != cudaSuccess) return e;
  route_tc_kernel<<<(unsigned)(BH * G_h), kThreads, smem, st>>>(mq, mqt, N, m, W, nch, G_h, cols,
                                                                 route, amb, status);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  route_fixup_kernel<<<std::max(num_sms, 1) * 4, 256, 0, st>>>(q, q_tilde, N, m, amb, route);
  return cudaGetLastError();
}

}  // namespace mita
