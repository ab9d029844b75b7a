// Step 4 on the tensor cores: route each query to its best landmark (s = 1),
// bf16, d = 64, m <= 512.
//
// MiTA tutorial (iwxt.cn), ch. 4 step 4 (paper eq. 10): q . q~_i over the m
// landmarks selects the expert; there is no gate.
//
// One CTA owns a head's landmark block q~ (TMA, resident in shared memory)
// and walks query tiles of 128 rows of that head:
//   warp 0       TMA producer: query tiles into a ring of kQStages;
//   warp 1       MMA issuer (whole warp, one elected lane issues): S = Q_tile .
//                q~^T into tensor memory, in chunks of W <= 128 landmarks;
//   warps 4-19   epilogue, four groups of four warps; group g owns the tiles
//                it = g, g + 4, ... and one W-column tensor-memory buffer; in a
//                group, warp w serves TMEM lane quadrant w % 4, one query row per
//                thread, whole rows (no partner to merge with).
// The issuer walks the tiles in rounds of four (one per group) and, inside a
// round, chunk by chunk over the four groups, so each group's next chunk is
// computed while the group reads the previous one and the other three groups'
// products keep the tensor pipe busy.
// Each thread keeps, over blocks of 32 scores, the running best with a
// shared-memory copy of the block holding it, and the maxima of all other
// blocks; the exact best, runner-up and the best's index (lowest on ties)
// follow at the end of the row.  When the best beats the runner-up by more
// than 2E (E bounds the fp32 dot error) it is the exact argmax; otherwise the
// query goes on its head's "ambiguous" list and route_fixup_kernel re-routes it
// exactly (fp32 screening + exact-product re-scoring, ties to the lowest
// index) -- about 0.2% of the queries on the long-sequence workloads.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"

namespace mita {
namespace {
using namespace sm100;

constexpr int kQStages = 6;
constexpr int kGroups = 4;
constexpr int kEpiWarps = 4 * kGroups;
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kThreads = (4 + kEpiWarps) * 32;
constexpr int kMaxM = 512;
constexpr int kMaxW = 128;

struct Cand {
  float v1, v2;   // best and runner-up scores
  int i1;         // lowest index reaching v1
};

struct alignas(1024) RouteSmem {
  bf16 qt[kMaxM * 64];                 // landmark rows, 128B-swizzled
  bf16 q[kQStages][128 * 64];          // query tiles, 128B-swizzled
  float4 bbuf[kEpiThreads][8];         // per epilogue thread: copy of its best 32-score block
  uint64_t q_full[kQStages], q_empty[kQStages];
  uint64_t qt_full, drain;
  uint64_t s_full[kGroups], s_empty[kGroups];
  // (drain: completion of the issuer's last products before tensor memory is freed)
  float red[kEpiWarps];
  uint32_t tmem;
};

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory"); }

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
// mb_hw: the block's maximum from the reducing tensor-memory load; a ragged last block (its
// columns past m hold zeros, uniform across the warp) recomputes it over its valid entries.
__device__ __forceinline__ void top_block(RowTop& t, float* v, float mb_hw, int i0, int nvalid,
                                          float4* bb, int sw) {
  float mb = mb_hw;
  if (nvalid < 32) {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = i < nvalid ? v[i] : -INFINITY;
    float a[11];
#pragma unroll
    for (int i = 0; i < 10; ++i) a[i] = max3f(v[3 * i], v[3 * i + 1], v[3 * i + 2]);
    a[10] = fmaxf(v[30], v[31]);
    const float b0 = max3f(a[0], a[1], a[2]), b1 = max3f(a[3], a[4], a[5]);
    const float b2 = max3f(a[6], a[7], a[8]), b3 = fmaxf(a[9], a[10]);
    mb = fmaxf(max3f(b0, b1, b2), b3);
  }
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

// (best, runner-up, lowest index of the best) of a finished row.  In the best
// block: the entries equal to the best form a bit mask (its lowest bit is the
// index, two or more bits make the runner-up equal to the best), and the
// runner-up of the block is the largest entry below the best -- independent
// comparisons and a max3 tree, no serial chain over the 32 entries.
__device__ __forceinline__ Cand finish_top(const RowTop& t, const float4* bbs, int sw) {
  Cand c{t.v1, t.v2c, 0x7fffffff};
  if (t.v1 == -INFINITY) return c;
  float bb[32];
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const float4 x = bbs[q ^ sw];
    bb[4 * q] = x.x; bb[4 * q + 1] = x.y; bb[4 * q + 2] = x.z; bb[4 * q + 3] = x.w;
  }
  uint32_t eq[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const bool e = bb[i] == t.v1;
    eq[i & 3] |= e ? (1u << i) : 0u;
    bb[i] = e ? -INFINITY : bb[i];
  }
  const uint32_t mask = (eq[0] | eq[1]) | (eq[2] | eq[3]);
  float a[11];
#pragma unroll
  for (int i = 0; i < 10; ++i) a[i] = max3f(bb[3 * i], bb[3 * i + 1], bb[3 * i + 2]);
  a[10] = fmaxf(bb[30], bb[31]);
  const float s2 = fmaxf(max3f(max3f(a[0], a[1], a[2]), max3f(a[3], a[4], a[5]), max3f(a[6], a[7], a[8])),
                         fmaxf(a[9], a[10]));
  c.v2 = (__popc(mask) > 1) ? t.v1 : fmaxf(c.v2, s2);
  c.i1 = t.bb0 + (__ffs(mask) - 1);
  return c;
}

__global__ void __launch_bounds__(kThreads, 1)
route_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_qt,
                int N, int m, int W, int nch, int G_h, uint32_t tmem_cols,
                int32_t* __restrict__ route, int* __restrict__ amb, int* status,
                int* __restrict__ hist) {
  griddep_wait();
  // amb: the heads' counts at amb[0, BH), then head bh's query ids at amb + BH + bh * N,
  // then (as floats) their fp32 best scores at amb + BH + BH * N + bh * N
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
      mbar_init(&s.q_empty[i], 1 + 4);   // the last chunk's MMA + the tile's four warps
    }
    mbar_init(&s.qt_full, 1);
    mbar_init(&s.drain, 1);
    for (int g = 0; g < kGroups; ++g) {
      mbar_init(&s.s_full[g], 1);
      mbar_init(&s.s_empty[g], 4);
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

  // registers: the launch grants 640 x 96; warps 0-3 keep 56 each, the sixteen
  // epilogue warps take 104 each (128*56 + 512*104 <= 640*96)
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
      // rounds of kGroups tiles; in a round, chunk by chunk over the groups
      const uint32_t idesc = idesc_f16(128, W, false);
      const uint32_t qtb = smem_u32(s.qt);
      bool ok = mbar_wait_warp(&s.qt_full, 0);
      const int nrounds = (ntiles + kGroups - 1) / kGroups;
      for (int r = 0; r < nrounds && ok; ++r) {
        const int ng = min(kGroups, ntiles - r * kGroups);
        for (int ch = 0; ch < nch && ok; ++ch) {
          const uint32_t qb = qtb + ch * W * 128;
          const int u = r * nch + ch;                  // this buffer's use count
          for (int g = 0; g < ng; ++g) {
            const int it = r * kGroups + g, st = it % kQStages;
            if (ch == 0 && !mbar_wait_warp(&s.q_full[st], (it / kQStages) & 1)) { ok = false; break; }
            if (!mbar_wait_warp(&s.s_empty[g], (u & 1) ^ 1)) { ok = false; break; }
            tc_fence_after();
            const uint32_t qa = smem_u32(s.q[st]);
            if (elect_one()) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_ss(tbase + g * W, smem_desc_sw128(qa + kk * 32, 1024),
                       smem_desc_sw128(qb + kk * 32, 1024), idesc, kk > 0);
              mma_commit(&s.s_full[g]);
              if (ch == nch - 1) mma_commit(&s.q_empty[st]);
            }
            __syncwarp();
          }
        }
      }
      if (elect_one()) mma_commit(&s.drain);
      __syncwarp();
      if (!mbar_wait_warp(&s.drain, 0)) ok = false;
      if (!ok && lane == 0) flag_error(status, kDevErrTimeout);
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 104;\n" ::: "memory");
    // ------------------------------------------------------------ epilogue
    const int et = threadIdx.x - 128;              // 0..511
    const int quad = warp & 3, grp = (warp - 4) >> 2;
    const int row = quad * 32 + lane;
    const uint32_t tb = tbase + ((uint32_t)(quad * 32) << 16) + (uint32_t)(grp * W);
    float4* bb = s.bbuf[et];
    const int sw = et & 7;
    bool ok = mbar_wait(&s.qt_full, 0);
    // largest landmark norm of the head (error bound)
    float n2max = 0.f;
    if (ok) {
      for (int i = et; i < m; i += kEpiThreads) {
        float r[64];
        load_swizzled_row(s.qt, i, r);
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int l = 0; l < 64; l += 2) {
          a0 = fmaf(r[l], r[l], a0);
          a1 = fmaf(r[l + 1], r[l + 1], a1);
        }
        n2max = fmaxf(n2max, a0 + a1);
      }
    }
    n2max = warp_max(n2max);
    if (lane == 0) s.red[warp - 4] = n2max;
    epi_bar();
    float qtmax2 = 0.f;
#pragma unroll
    for (int i = 0; i < kEpiWarps; ++i) qtmax2 = fmaxf(qtmax2, s.red[i]);
    const float gq = 2.f * err_gamma(64) * sqrtf(qtmax2);
    int* hcnt = amb + bh;
    const size_t BHs = gridDim.x / G_h;
    int* hids = amb + BHs + (size_t)bh * N;
    float* hbest = reinterpret_cast<float*>(amb + BHs + BHs * N) + (size_t)bh * N;
    for (int it = grp; it < ntiles; it += kGroups) {
      const int st = it % kQStages, r = it / kGroups;
      if (ok && !mbar_wait(&s.q_full[st], (it / kQStages) & 1)) ok = false;
      const int n = (c0 + it * G_h) * 128 + row;
      const bool live = ok && n < N;
      // the query's error bound first, while the scores are computed
      float twoE = 0.f;
      if (live) {
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
        twoE = gq * sqrtf((a0 + a1) + (a2 + a3));
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.q_empty[st]);   // this warp is done with the query tile
      RowTop top;
      for (int ch = 0; ch < nch; ++ch) {
        const int u = r * nch + ch;
        if (ok && !mbar_wait(&s.s_full[grp], u & 1)) ok = false;
        tc_fence_after();
        // W columns in pieces of 64: load, then two 32-score blocks
#pragma unroll
        for (int p = 0; p < kMaxW / 64; ++p) {
          if (p * 64 < W) {
            // the two 32-score blocks of this piece, each with its maximum
            float v[64];
            float bmx[2] = {-INFINITY, -INFINITY};
            if (ok) {
              bmx[0] = tmem_ld32_max(tb + p * 64, v);
              if (W - p * 64 >= 64) bmx[1] = tmem_ld32_max(tb + p * 64 + 32, v + 32);
              tmem_ld_wait();
              tmem_fence_regs<64>(v);
              tmem_fence_regs<2>(bmx);
            }
            if (p * 64 + 64 >= W) {                  // the buffer may be overwritten now
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&s.s_empty[grp]);
            }
            if (ok) {
#pragma unroll
              for (int cc = 0; cc < 64; cc += 32) {
                const int i0 = ch * W + p * 64 + cc;
                if (p * 64 + cc < W && i0 < m)
                  top_block(top, v + cc, bmx[cc / 32], i0, min(m - i0, 32), bb, sw);
              }
            }
          }
        }
      }
      const Cand c = finish_top(top, bb, sw);
      const bool ambiguous = live && !(c.v1 - c.v2 > twoE);
      if (live) {
        route[(size_t)bh * N + n] = c.i1;
        // the bucket stage's count of (expert, chunk of 4096 queries); an ambiguous
        // query is counted by the fix-up, under its exact route
        if (hist && !ambiguous && c.i1 >= 0 && c.i1 < m)
          atomicAdd(&hist[((size_t)bh * m + c.i1) * ((N + kBucketChunk - 1) / kBucketChunk) +
                          n / kBucketChunk], 1);
      }
      // append ambiguous queries to the head's list (one reservation per warp)
      const unsigned am = __ballot_sync(0xffffffffu, ambiguous);
      if (am) {
        int base = 0;
        if (lane == 0) base = atomicAdd(hcnt, __popc(am));
        base = __shfl_sync(0xffffffffu, base, 0);
        if (ambiguous) {
          const int pos = base + __popc(am & ((1u << lane) - 1u));
          hids[pos] = n;
          hbest[pos] = c.v1;
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
// within 2E of the routing kernel's fp32 best can win), re-score the
// survivors with exact-product arithmetic and reduce (score desc, index asc).
constexpr int kFixRow = 72;            // bf16 per padded landmark row

__global__ void __launch_bounds__(256)
route_fixup_kernel(const bf16* __restrict__ q, const bf16* __restrict__ q_tilde, int N, int m,
                   int per_head, const int* __restrict__ amb, int32_t* __restrict__ route,
                   int* __restrict__ hist) {
  griddep_wait();
  extern __shared__ __align__(16) unsigned char fix_raw[];
  bf16* qt = reinterpret_cast<bf16*>(fix_raw);       // [m][kFixRow]
  __shared__ float red[8];
  const int bh = blockIdx.x / per_head, part = blockIdx.x % per_head;
  const int count = amb[bh];
  const size_t BHs = gridDim.x / per_head;
  const int* hids = amb + BHs + (size_t)bh * N;
  const float* hbest = reinterpret_cast<const float*>(amb + BHs + BHs * N) + (size_t)bh * N;
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
    const int n = hids[w];
    if (n < 0 || n >= N) continue;
    float qr[64];
    load_row<bf16, 64>(q + ((size_t)bh * N + n) * 64, qr);
    float qn2 = 0.f;
#pragma unroll
    for (int l = 0; l < 64; ++l) qn2 = fmaf(qr[l], qr[l], qn2);
    // the tensor-core fp32 best v1 is within E of the exact score of the landmark it
    // came from, so the exact maximum is >= v1 - E and its fp32 dot here >= v1 - 2E
    const float best = hbest[w];
    const float twoE = 2.f * err_gamma(64) * sqrtf(qn2) * sqrtf(qt2);
    // exact re-scoring of the landmarks whose fp32 dot is within 2E of it (the landmark
    // loop stays rolled: unrolled copies of its body overflow the instruction cache)
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
    if (lane == 0) {
      route[(size_t)bh * N + n] = bi;
      if (hist && bi >= 0 && bi < m)   // the routing kernel left this query uncounted
        atomicAdd(&hist[((size_t)bh * m + bi) * ((N + kBucketChunk - 1) / kBucketChunk) +
                        n / kBucketChunk], 1);
    }
  }
}

// Exact top-s (s >= 2) re-routing of the queries route_shared_tc left ambiguous (its
// fp32 route list had a gap within 2E).  Same staging as route_fixup_kernel; the stored
// reference is the fp32 score of the s-th route, so every landmark of the exact top-s has
// its fp32 dot here within 2E of it.  Each lane keeps the best s of its survivors (exact
// products, ranked by (score desc, index asc)); s rounds of a warp-wide best-of-heads merge
// give the list, best first.
constexpr int kFixMaxS = 8;

__device__ __forceinline__ void fix_insert(F2 (&lv)[kFixMaxS], int (&li)[kFixMaxS], int s, F2 x,
                                           int j) {
#pragma unroll
  for (int t = kFixMaxS - 1; t > 0; --t) {
    if (t < s) {
      if (ranks_before(x, j, lv[t - 1], li[t - 1])) { lv[t] = lv[t - 1]; li[t] = li[t - 1]; }
      else if (ranks_before(x, j, lv[t], li[t])) { lv[t] = x; li[t] = j; }
    }
  }
  if (ranks_before(x, j, lv[0], li[0])) { lv[0] = x; li[0] = j; }
}

__global__ void __launch_bounds__(256)
route_fixup_top_kernel(const bf16* __restrict__ q, const bf16* __restrict__ q_tilde, int N, int m,
                       int s, int per_head, const int* __restrict__ amb,
                       int32_t* __restrict__ route, int* __restrict__ hist) {
  griddep_wait();
  extern __shared__ __align__(16) unsigned char fix_raw[];
  bf16* qt = reinterpret_cast<bf16*>(fix_raw);       // [m][kFixRow]
  __shared__ float red[8];
  const int bh = blockIdx.x / per_head, part = blockIdx.x % per_head;
  const int count = amb[bh];
  const size_t BHs = gridDim.x / per_head;
  const int* hids = amb + BHs + (size_t)bh * N;
  const float* hkeep = reinterpret_cast<const float*>(amb + BHs + BHs * N) + (size_t)bh * N;
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
    const int n = hids[w];
    if (n < 0 || n >= N) continue;
    float qr[64];
    load_row<bf16, 64>(q + ((size_t)bh * N + n) * 64, qr);
    float qn2 = 0.f;
#pragma unroll
    for (int l = 0; l < 64; ++l) qn2 = fmaf(qr[l], qr[l], qn2);
    const float keep = hkeep[w];
    const float twoE = 2.f * err_gamma(64) * sqrtf(qn2) * sqrtf(qt2);
    F2 lv[kFixMaxS];
    int li[kFixMaxS];
#pragma unroll
    for (int t = 0; t < kFixMaxS; ++t) { lv[t] = F2{-INFINITY, 0.f}; li[t] = 0x7fffffff; }
#pragma unroll 1
    for (int i = lane; i < m; i += 32) {
      float r[64];
      load_row<bf16, 64>(qt + i * kFixRow, r);
      float a = 0.f;
#pragma unroll
      for (int l = 0; l < 64; ++l) a = fmaf(qr[l], r[l], a);
      if (a >= keep - twoE) fix_insert(lv, li, s, dot_f2<64, 64>(qr, r), i);
    }
    // s rounds: the best head over the lanes, which its lane then pops
    for (int r = 0; r < s; ++r) {
      F2 bv = lv[0];
      int bi = li[0];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const F2 ov{__shfl_xor_sync(0xffffffffu, bv.hi, o), __shfl_xor_sync(0xffffffffu, bv.lo, o)};
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ranks_before(ov, oi, bv, bi)) { bv = ov; bi = oi; }
      }
      if (lane == 0) {
        route[((size_t)bh * N + n) * s + r] = bi;
        if (hist && bi >= 0 && bi < m)   // the routing kernel left this query uncounted
          atomicAdd(&hist[((size_t)bh * m + bi) * (((long long)N * s + kBucketChunk - 1) / kBucketChunk) +
                          ((long long)n * s + r) / kBucketChunk], 1);
      }
      if (li[0] == bi) {
#pragma unroll
        for (int t = 0; t < kFixMaxS - 1; ++t) { lv[t] = lv[t + 1]; li[t] = li[t + 1]; }
        lv[kFixMaxS - 1] = F2{-INFINITY, 0.f};
        li[kFixMaxS - 1] = 0x7fffffff;
      }
    }
  }
}

}  // namespace

size_t route_tc_smem_bytes() { return sizeof(RouteSmem) + 1024; }

bool route_tc_supported(int d, int m) { return d == 64 && m >= 1 && m <= kMaxM; }

cudaError_t launch_route_tc(const bf16* q, const bf16* q_tilde, int BH, int N, int m,
                            int num_sms, int32_t* route, int* amb, int* status, int* hist,
                            cudaStream_t st, bool prezeroed) {
  // chunk width: 32, 64 or 128 landmarks (a power of two, so the four group
  // buffers fill a power-of-two tensor-memory allocation)
  int W = 32;
  while (W < kMaxW && W < m) W <<= 1;
  const int nch = (m + W - 1) / W;
  const uint32_t cols = (uint32_t)(kGroups * W);
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
  if (!prezeroed && (e = cudaMemsetAsync(amb, 0, (size_t)BH * sizeof(int), st)) != cudaSuccess)
    return e;
  if (hist && !prezeroed) {
    const size_t nh = (size_t)BH * m * ((N + kBucketChunk - 1) / kBucketChunk);
    if ((e = cudaMemsetAsync(hist, 0, nh * sizeof(int), st)) != cudaSuccess) return e;
  }
  e = launch_pdl(route_tc_kernel, dim3((unsigned)(BH * G_h)), dim3(kThreads), smem, st, mq, mqt, N,
                 m, W, nch, G_h, cols, route, amb, status, hist);
  count_launch();
  if (e != cudaSuccess) return e;
  return launch_route_fixup(q, q_tilde, BH, N, m, num_sms, route, amb, hist, st);
}

cudaError_t launch_route_fixup_top(const bf16* q, const bf16* q_tilde, int BH, int N, int m,
                                   int s, int num_sms, int32_t* route, const int* amb, int* hist,
                                   cudaStream_t st) {
  if (s < 2 || s > kFixMaxS || s > m) return cudaErrorInvalidValue;
  const int per_head = std::max(1, std::max(num_sms, 1) / BH);
  const size_t fsm = (size_t)m * kFixRow * 2;
  cudaError_t e = cudaFuncSetAttribute(route_fixup_top_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)fsm);
  if (e != cudaSuccess) return e;
  e = launch_pdl(route_fixup_top_kernel, dim3((unsigned)(BH * per_head)), dim3(256), fsm, st, q,
                 q_tilde, N, m, s, per_head, amb, route, hist);
  count_launch();
  return e;
}

cudaError_t launch_route_fixup(const bf16* q, const bf16* q_tilde, int BH, int N, int m,
                               int num_sms, int32_t* route, const int* amb, int* hist,
                               cudaStream_t st) {
  cudaError_t e;
  const int per_head = std::max(1, std::max(num_sms, 1) / BH);
  const size_t fsm = (size_t)m * kFixRow * 2;
  e = cudaFuncSetAttribute(route_fixup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)fsm);
  if (e != cudaSuccess) return e;
  e = launch_pdl(route_fixup_kernel, dim3((unsigned)(BH * per_head)), dim3(256), fsm, st, q, q_tilde,
                 N, m, per_head, amb, route, hist);
  count_launch();
  return e;
}

}  // namespace mita
