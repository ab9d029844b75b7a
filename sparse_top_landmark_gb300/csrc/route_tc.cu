// Step 4 on the tensor cores: route each query to its best landmark (s = 1),
// bf16, d = 64, m <= 512.
//
// MiTA tutorial (iwxt.cn), ch. 4 step 4 (paper eq. 10): q . q~_i over the m
// landmarks selects the expert; there is no gate.
//
// One CTA owns a head's landmark block q~ (TMA, resident in shared memory)
// and walks query tiles of 128 rows of that head:
//   warp 0      TMA producer: query tiles into a 3-stage ring;
//   warp 1      MMA issuer (whole warp, one elected lane issues): S = Q_tile .
//               q~^T into tensor memory, in chunks of W <= 256 landmarks, two
//               chunk buffers (ping-pong);
//   warps 4-11  epilogue: TMEM lane quadrant = warp % 4 (one query row per
//               thread), two warps per quadrant split each chunk's columns and
//               meet on a 64-thread barrier per tile.
// Each thread keeps, over blocks of 32 scores, the running best with a
// register copy of the block holding it, and the maxima of all other blocks;
// the exact best, runner-up and the best's index (lowest on ties) follow at
// the end of the row.  When the best beats the runner-up by more than 2E (E bounds the fp32
// dot error) it is the exact argmax; otherwise the query goes on its head's
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
  // (drain: completion of the issuer's last products before tensor memory is freed)
  Cand cand[2][128];                   // half-1 partial results, by tile parity
  float4 bbuf[256][8];                 // per epilogue thread: copy of its best 32-score block
  float red[kEpiWarps];
  float qtmax2;
  uint32_t tmem;
};

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
// the two epilogue warps of one TMEM lane quadrant
__device__ __forceinline__ void quad_bar(int quad) {
  asm volatile("bar.sync %0, 64;" ::"r"(2 + quad) : "memory");
}

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

// Running best over blocks of 32 scores.  Per block only its maximum is
// computed; the block holding the running best is kept in registers (bb,
// first index bb0) and every other block contributes its maximum to v2c.  At
// the end the best's index (lowest on ties) and the runner-up come from bb:
// the runner-up of the whole row is the larger of v2c and the second largest
// entry of bb.
struct RowTop {
  float v1 = -INFINITY, v2c = -INFINITY;
  int bb0 = 0;
};

// bb: this thread's 32-float block copy in shared memory, eight 16-byte chunks
// stored at chunk c ^ sw (sw = thread % 8), so a warp's 16-byte accesses spread
// over all banks.  The copy goes through shared memory (a few stores, only when
// the block improves the best) instead of 32 register selects per block.
__device__ __forceinline__ void top_block(RowTop& t, float* v, int i0, int nvalid, float4* bb,
                                          int sw) {
  if (nvalid < 32) {                 // ragged last block (uniform across the warp)
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = i < nvalid ? v[i] : -INFINITY;
  }
  float a[11];
#pragma unroll
  for (int i = 0; i < 10; ++i) a[i] = max3f(v[3 * i], v[3 * i + 1], v[3 * i + 2]);
  a[10] = fmaxf(v[30], v[31]);
  const float b0 = max3f(a[0], a[1], a[2]), b1 = max3f(a[3], a[4], a[5]);
  const float b2 = max3f(a[6], a[7], a[8]), b3 = fmaxf(a[9], a[10]);
  const float mb = fmaxf(max3f(b0, b1, b2), b3);
  const bool up = mb > t.v1;
  t.v2c = fmaxf(t.v2c, up ? t.v1 : mb);
  t.v1 = up ? mb : t.v1;
  if (up) {
#pragma unroll
    for (int c = 0; c < 8; ++c)
      bb[c ^ sw] = make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
    t.bb0 = i0;
  }
}

// (best, runner-up, lowest index of the best) of a finished row
__device__ __forceinline__ Cand finish_top(const RowTop& t, const float4* bbs, int sw) {
  Cand c{t.v1, t.v2c, 0x7fffffff};
  if (t.v1 == -INFINITY) return c;
  float bb[32];
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const float4 x = bbs[q ^ sw];
    bb[4 * q] = x.x; bb[4 * q + 1] = x.y; bb[4 * q + 2] = x.z; bb[4 * q + 3] = x.w;
  }
  int k = 31;
#pragma unroll
  for (int i = 31; i >= 0; --i) k = (bb[i] == t.v1) ? i : k;
  float s2 = -INFINITY;
#pragma unroll
  for (int i = 0; i < 32; ++i) s2 = (i == k) ? s2 : fmaxf(s2, bb[i]);
  c.v2 = fmaxf(c.v2, s2);
  c.i1 = t.bb0 + k;
  return c;
}

__global__ void __launch_bounds__(kThreads, 1)
route_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_qt,
                int N, int m, int W, int nch, int G_h, uint32_t tmem_cols,
                int32_t* __restrict__ route, int* __restrict__ amb, int* status) {
  // amb: per head, [count, query ids...] at amb + bh * (N + 1)
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

  // registers: the launch grants 384 x 168; warps 0-3 keep 56 each, the two epilogue
  // warpgroups take 224 each (128*56 + 2*128*224 = 384*168)
  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 56;\n" ::: "memory");
    if (warp == 0) {
      // ---------------------------------------------------------- producer
      bool ok = true;
      if (elect_one()) {
        prefetch_tmap(&map_q);
        prefetch_tmap(&map_qt);
        mbar_expect_tx(&s.qt_full, (uint32_t)(nch * W * 128));
        for (int ch = 0; ch < nch; ++ch)
          tma_load_3d(s.qt + ch * W * 64, &map_qt, &s.qt_full, 0, ch * W, bh);
      }
      __syncwarp();
      for (int it = 0; it < ntiles; ++it) {
        const int st = it % kQStages;
        if (!mbar_wait_warp(&s.q_empty[st], ((it / kQStages) & 1) ^ 1)) { ok = false; break; }
        if (elect_one()) {
          mbar_expect_tx(&s.q_full[st], 128 * 128);
          tma_load_3d(s.q[st], &map_q, &s.q_full[st], 0, (c0 + it * G_h) * 128, bh);
        }
        __syncwarp();
      }
      if (!ok && lane == 0) flag_error(status, kDevErrTimeout);
    } else if (warp == 1) {
      // ---------------------------------------------------------- MMA issuer
      const uint32_t idesc = idesc_f16(128, W, false);
      const uint32_t qtb = smem_u32(s.qt);
      bool ok = mbar_wait_warp(&s.qt_full, 0);
      int gch = 0;
      for (int it = 0; it < ntiles && ok; ++it) {
        const int st = it % kQStages;
        if (!mbar_wait_warp(&s.q_full[st], (it / kQStages) & 1)) { ok = false; break; }
        const uint32_t qa = smem_u32(s.q[st]);
        for (int ch = 0; ch < nch; ++ch, ++gch) {
          const int b = gch & 1;
          if (!mbar_wait_warp(&s.s_empty[b], ((gch >> 1) & 1) ^ 1)) { ok = false; break; }
          tc_fence_after();
          const uint32_t qb = qtb + ch * W * 128;
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ss(tbase + b * W, smem_desc_sw128(qa + kk * 32, 1024),
                     smem_desc_sw128(qb + kk * 32, 1024), idesc, kk > 0);
            mma_commit(&s.s_full[b]);
            if (ch == nch - 1) mma_commit(&s.q_empty[st]);
          }
          __syncwarp();
        }
      }
      if (elect_one()) mma_commit(&s.drain);
      __syncwarp();
      if (!mbar_wait_warp(&s.drain, 0)) ok = false;
      if (!ok && lane == 0) flag_error(status, kDevErrTimeout);
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 224;\n" ::: "memory");
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
    const int cols_half = W / 2;                   // a multiple of 16, at most 128
    int* hamb = amb + (size_t)bh * (N + 1);
    int gch = 0;
    for (int it = 0; it < ntiles; ++it) {
      const int st = it % kQStages;
      if (ok && !mbar_wait(&s.q_full[st], (it / kQStages) & 1)) ok = false;
      // the query's error bound first (half 0), while the scores are computed
      const int n = (c0 + it * G_h) * 128 + row;
      const bool live = ok && n < N;
      float twoE = 0.f;
      if (half == 0 && live) {
        float qr[64];
        load_swizzled_row(s.q[st], row, qr);
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
        for (int l = 0; l < 64; l += 4) {
          a0 = fmaf(qr[l], qr[l], a0);
          a1 = fmaf(qr[l + 1], qr[l + 1], a1);
          a2 = fmaf(qr[l + 2], qr[l + 2], a2);
          a3 = fmaf(qr[l + 3], qr[l + 3], a3);
        }
        twoE = 2.f * gam * sqrtf((a0 + a1) + (a2 + a3)) * sqrtf(qtmax2);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.q_empty[st]);   // this warp is done with the query tile
      RowTop top;
      for (int ch = 0; ch < nch; ++ch, ++gch) {
        const int b = gch & 1;
        if (ok && !mbar_wait(&s.s_full[b], (gch >> 1) & 1)) ok = false;
        tc_fence_after();
        const int col0 = half * cols_half;
        float v[128];
        if (ok) {
          const uint32_t ta = tbase + taddr_lane + (uint32_t)(b * W + col0);
          if (cols_half >= 64) {
            tmem_ld64(ta, v);
          } else {
#pragma unroll
            for (int cc = 0; cc < 64; cc += 16)
              if (cc < cols_half) tmem_ld16(ta + cc, v + cc);
          }
          if (cols_half >= 128) {
            tmem_ld64(ta + 64, v + 64);
          } else {
#pragma unroll
            for (int cc = 64; cc < 128; cc += 16)
              if (cc < cols_half) tmem_ld16(ta + cc, v + cc);
          }
          tmem_ld_wait();
          tmem_fence_regs<128>(v);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.s_empty[b]);   // the buffer may be overwritten now
        if (ok) {
#pragma unroll
          for (int cc = 0; cc < 128; cc += 32) {
            if (cc < cols_half) {
              const int i0 = ch * W + col0 + cc;
              top_block(top, v + cc, i0, min(m - i0, cols_half - cc), s.bbuf[et], et & 7);
            }
          }
        }
      }
      const Cand c = finish_top(top, s.bbuf[et], et & 7);
      if (half == 1) s.cand[it & 1][row] = c;
      quad_bar(quad);
      if (half == 0) {
        const Cand o = s.cand[it & 1][row];
        const bool w1 = o.v1 > c.v1 || (o.v1 == c.v1 && o.i1 < c.i1);
        const float v1 = w1 ? o.v1 : c.v1;
        const int i1 = w1 ? o.i1 : c.i1;
        const float v2 = max3f(c.v2, o.v2, fminf(c.v1, o.v1));
        const bool ambiguous = live && !(v1 - v2 > twoE);
        if (live) route[(size_t)bh * N + n] = i1;
        // append ambiguous queries to the head's list (one reservation per warp)
        const unsigned am = __ballot_sync(0xffffffffu, ambiguous);
        if (am) {
          int base = 0;
          if (lane == 0) base = atomicAdd(hamb, __popc(am));
          base = __shfl_sync(0xffffffffu, base, 0);
          if (ambiguous) hamb[1 + base + __popc(am & ((1u << lane) - 1u))] = n;
        }
      }
    }
    if (!ok) flag_error(status, kDevErrTimeout);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, tmem_cols);
}

// Exact routing of the ambiguous queries.  CTA = (head, slice of the head's
// list) with the head's q~ block in shared memory (rows padded to 144 bytes:
// a warp's 16-byte reads of 32 different rows then hit every bank evenly);
// one warp per query: lanes screen the landmarks with fp32 dots (only those
// within 2E of the fp32 best can win), re-score the survivors with
// exact-product arithmetic and reduce (score desc, index asc).
constexpr int kFixRow = 72;            // bf16 per padded landmark row

__global__ void __launch_bounds__(256)
route_fixup_kernel(const bf16* __restrict__ q, const bf16* __restrict__ q_tilde, int N, int m,
                   int per_head, const int* __restrict__ amb, int32_t* __restrict__ route) {
  extern __shared__ __align__(16) unsigned char fix_raw[];
  bf16* qt = reinterpret_cast<bf16*>(fix_raw);       // [m][kFixRow]
  __shared__ float red[8];
  const int bh = blockIdx.x / per_head, part = blockIdx.x % per_head;
  const int* hamb = amb + (size_t)bh * (N + 1);
  const int count = hamb[0];
  if (count <= part * 8) return;                      // no query for this CTA
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bf16* qtb = q_tilde + (size_t)bh * m * 64;
  float n2 = 0.f;
  for (int t = threadIdx.x; t < m * 8; t += 256) {
    const int i = t >> 3, c = t & 7;
    const uint4 x = reinterpret_cast<const uint4*>(qtb + (size_t)i * 64)[c];
    *reinterpret_cast<uint4*>(qt + i * kFixRow + c * 8) = x;
    float f[8];
    Vec<bf16>::load(reinterpret_cast<const bf16*>(&x), f);
#pragma unroll
    for (int e = 0; e < 8; ++e) n2 = fmaf(f[e], f[e], n2);
  }
  // largest squared landmark norm: per-row sums of 8 lanes' partials
  n2 += __shfl_xor_sync(0xffffffffu, n2, 1);
  n2 += __shfl_xor_sync(0xffffffffu, n2, 2);
  n2 += __shfl_xor_sync(0xffffffffu, n2, 4);
  n2 = warp_max(n2);
  if (lane == 0) red[warp] = n2;
  __syncthreads();
  float qt2 = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) qt2 = fmaxf(qt2, red[w]);
  for (int w = part * 8 + warp; w < count; w += per_head * 8) {
    const int n = hamb[1 + w];
    if (n < 0 || n >= N) continue;
    float qr[64];
    load_row<bf16, 64>(q + ((size_t)bh * N + n) * 64, qr);
    float qn2 = 0.f;
#pragma unroll
    for (int l = 0; l < 64; ++l) qn2 = fmaf(qr[l], qr[l], qn2);
    // pass 1: the fp32 best (the landmark loops stay rolled: unrolled copies of
    // these bodies overflow the instruction cache)
    float best = -INFINITY;
#pragma unroll 1
    for (int i = lane; i < m; i += 32) {
      float r[64];
      load_row<bf16, 64>(qt + i * kFixRow, r);
      float a = 0.f;
#pragma unroll
      for (int l = 0; l < 64; ++l) a = fmaf(qr[l], r[l], a);
      best = fmaxf(best, a);
    }
    best = warp_max(best);
    const float twoE = 2.f * err_gamma(64) * sqrtf(qn2) * sqrtf(qt2);
    // pass 2: exact re-scoring of the landmarks within 2E of it
    F2 bv{-INFINITY, 0.f};
    int bi = 0x7fffffff;
#pragma unroll 1
    for (int i = lane; i < m; i += 32) {
      float r[64];
      load_row<bf16, 64>(qt + i * kFixRow, r);
      float a = 0.f;
#pragma unroll
      for (int l = 0; l < 64; ++l) a = fmaf(qr[l], r[l], a);
      if (a >= best - twoE) {
        const F2 x = dot_f2<64, 64>(qr, r);   // fully unrolled: qr, r stay in registers
        if (ranks_before(x, i, bv, bi)) { bv = x; bi = i; }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const F2 ov{__shfl_xor_sync(0xffffffffu, bv.hi, o), __shfl_xor_sync(0xffffffffu, bv.lo, o)};
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ranks_before(ov, oi, bv, bi)) { bv = ov; bi = oi; }
    }
    if (lane == 0) route[(size_t)bh * N + n] = bi;
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
  for (int b = 0; b < BH; ++b) {
    e = cudaMemsetAsync(amb + (size_t)b * (N + 1), 0, sizeof(int), st);
    if (e != cudaSuccess) return e;
  }
  route_tc_kernel<<<(unsigned)(BH * G_h), kThreads, smem, st>>>(mq, mqt, N, m, W, nch, G_h, cols,
                                                                 route, amb, status);
  count_launch();
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int per_head = std::max(1, std::max(num_sms, 1) / BH);
  const size_t fsm = (size_t)m * kFixRow * 2;
  e = cudaFuncSetAttribute(route_fixup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)fsm);
  if (e != cudaSuccess) return e;
  route_fixup_kernel<<<(unsigned)(BH * per_head), 256, fsm, st>>>(q, q_tilde, N, m, per_head, amb,
                                                                 route);
  count_launch();
  return cudaGetLastError();
}

}  // namespace mita
