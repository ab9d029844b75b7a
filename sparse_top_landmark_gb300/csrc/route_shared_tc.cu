// Step 4 on the tensor cores together with the shared branch of step 6 (bf16,
// d = 64; s = 1 with m <= 512, s = 2 with m <= 256): each query's best landmark
// (or best two) AND the partial result of its m shared pairs, from one set of
// query-landmark logits.
//
// MiTA tutorial (iwxt.cn), ch. 4 step 4 (paper eq. 10): the logits q . q~_i
// choose the expert (argmax, no gate); ch. 6 counts the same dot product once
// for routing and for the shared logits (N(2m + sk) scores per head), and the
// bit.fan article's expert-construction section reuses the query-to-landmark
// scores for routing.  Ch. 4 (branch merge): the joint softmax over [shared;
// raw] equals (Z1 o1 + Z2 o2) / (Z1 + Z2), so the shared pairs' part can be
// finished here as (log-sum-exp, normalised output) and merged by the expert
// stage, which then attends over the k raw pairs only.
//
// CTA = (head, slice of 128-query tiles); q~ and v~ of the head stay resident in
// shared memory (TMA for q~; v~ converted from fp32 to bf16 by the softmax warps).
//   warp 0       TMA: q~ once, then the query tiles into a kQStages ring;
//   warps 1-2    MMA issuers of tile slot 0 / 1 (the slot's tiles alternate):
//                S = Q . q~_c^T per chunk c of 128 landmarks, the next S as soon
//                as the softmax has copied S out, O += P . v~_c with P read from
//                tensor memory;
//   warps 4-7 / 8-11   one query row per thread: per chunk the running best
//                over 32-score blocks (with a shared-memory copy of the block
//                holding it) and the online softmax of the shared logits (lazy
//                O rescaling); at the tile's end the route (exact argmax, or the
//                query goes on the head's ambiguous list when the best and the
//                runner-up are within 2E), the bucket histogram count, and once
//                the tile's last P . V is done, lse and O / l.
// The exact argmax follows route_tc.cu's rules; route_fixup_kernel (same file
// there) re-routes the ambiguous queries.  Routing only needs the logits, so the
// shared branch's partial does not depend on the fix-up.
// s = 2 (tutorial ch. 4 step 4, eq. 10: the top-s landmarks): each thread keeps
// the three best 32-score blocks of its row, ranked by (block maximum desc,
// position asc), each copied to shared memory.  A score outside those blocks
// has three block maxima ranking ahead of it (a tie between maxima goes to the
// earlier block, whose tied score has the lower index), hence three scores
// ahead of it; so the row's best three scores, and the route (best two, ranked)
// with its gap test, come from the copies alone.  The route is exact when both
// gaps (first to second, second to third) exceed 2E; otherwise the query goes
// to the exact top-s fix-up.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"

namespace mita {
namespace {
using namespace sm100;

constexpr int BN = 128;             // landmarks per chunk
constexpr int kThreads = 384;       // producer, two issuers, one idle warp, 8 softmax warps
constexpr int kSoftThreads = 256;
constexpr float kLazy = 8.0f;

// per route count s: landmark limit, query-tile ring depth, 32-score block copies per thread
template <int kS> struct RsCfg;
template <> struct RsCfg<1> { static constexpr int kMaxM = 512, kQStages = 4, kBlocks = 1; };
template <> struct RsCfg<2> { static constexpr int kMaxM = 256, kQStages = 2, kBlocks = 3; };

template <int kS>
struct alignas(1024) RsSmem {
  using C = RsCfg<kS>;
  bf16 qt[C::kMaxM * 64];                 // landmark rows (128B-swizzled, TMA)
  bf16 vt[C::kMaxM * 64];                 // shared values, bf16 (128B-swizzled, written here)
  bf16 q[C::kQStages][128 * 64];          // query tiles
  float4 bbuf[C::kBlocks][kSoftThreads][8];   // per softmax thread: copies of 32-score blocks
  uint64_t q_full[C::kQStages], q_empty[C::kQStages];
  uint64_t res_full;                      // q~ loaded and v~ converted
  uint64_t s_full[2], s_free[2], p_full[2], pv_done[2], drain[2];
  float red[8];
  uint32_t tmem;
};

__device__ __forceinline__ void soft_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(kSoftThreads) : "memory");
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {   // a in the low half
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %2, %1;" : "=r"(r) : "f"(a), "f"(b));
  return r;
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

// Running best over blocks of 32 scores (as in route_tc.cu): per block only its maximum;
// the block holding the running best is copied to shared memory, every other block gives
// its maximum (mb, read by the loading instruction) to v2c.  Returns mb.
struct RowTop {
  float v1 = -INFINITY, v2c = -INFINITY;
  int bb0 = 0;
};
__device__ __forceinline__ float top_block(RowTop& t, const float* v, float mb, int i0,
                                           float4* bb, int sw) {
  const bool up = mb > t.v1;
  t.v2c = fmaxf(t.v2c, up ? t.v1 : mb);
  t.v1 = up ? mb : t.v1;
  if (up) {
#pragma unroll
    for (int c = 0; c < 8; ++c)
      bb[c ^ sw] = make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
    t.bb0 = i0;
  }
  return mb;
}
struct Cand {
  float v1, v2;
  int i1;
};
// (best, runner-up, lowest index of the best) of a finished row, from the best block's copy.
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

// ---- s = 2: the three best 32-score blocks, ranked by (maximum desc, position asc) -------
__device__ __forceinline__ float block_max32(const float* v) {
  float a[11];
#pragma unroll
  for (int i = 0; i < 10; ++i) a[i] = max3f(v[3 * i], v[3 * i + 1], v[3 * i + 2]);
  a[10] = fmaxf(v[30], v[31]);
  return fmaxf(max3f(max3f(a[0], a[1], a[2]), max3f(a[3], a[4], a[5]), max3f(a[6], a[7], a[8])),
               fmaxf(a[9], a[10]));
}
struct Top3Blocks {
  float bv[3] = {-INFINITY, -INFINITY, -INFINITY};   // block maxima, best first
  int b0[3] = {0, 0, 0};                             // first landmark index of each block
  int slot[3] = {0, 1, 2};                           // its copy's shared-memory slot
};
// bb: this thread's slot-0 copy; slot t lies t * slot_stride float4s further
__device__ __forceinline__ void top3_block(Top3Blocks& t, const float* v, float mb, int i0,
                                           float4* bb, int slot_stride, int sw) {
  // blocks already kept with an equal maximum come earlier, so they stay ahead
  const int p = (t.bv[0] >= mb ? 1 : 0) + (t.bv[1] >= mb ? 1 : 0) + (t.bv[2] >= mb ? 1 : 0);
  if (p < 3) {
    const int fs = t.slot[2];              // the third block's copy is dropped
    if (p <= 1) { t.bv[2] = t.bv[1]; t.b0[2] = t.b0[1]; t.slot[2] = t.slot[1]; }
    if (p == 0) { t.bv[1] = t.bv[0]; t.b0[1] = t.b0[0]; t.slot[1] = t.slot[0]; }
    if (p == 0) { t.bv[0] = mb; t.b0[0] = i0; t.slot[0] = fs; }
    else if (p == 1) { t.bv[1] = mb; t.b0[1] = i0; t.slot[1] = fs; }
    else { t.bv[2] = mb; t.b0[2] = i0; t.slot[2] = fs; }
    float4* dst = bb + fs * slot_stride;
#pragma unroll
    for (int c = 0; c < 8; ++c)
      dst[c ^ sw] = make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
  }
}
struct Top3 {
  float v[3];
  int i[3];
};
// the row's three best (score, index) pairs, ranked by (score desc, index asc), from the
// kept blocks' copies: three rounds of (best current block maximum, the lowest index holding
// it among the blocks that reach it, removal from its block and that block's new maximum)
__device__ __forceinline__ Top3 finish_top3(const Top3Blocks& t, const float4* bb,
                                            int slot_stride, int sw) {
  float x[3][32];
#pragma unroll
  for (int b = 0; b < 3; ++b) {
    const bool kept = t.bv[b] > -INFINITY;
    const float4* src = bb + t.slot[b] * slot_stride;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      float4 y = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      if (kept) y = src[q ^ sw];
      x[b][4 * q] = y.x; x[b][4 * q + 1] = y.y; x[b][4 * q + 2] = y.z; x[b][4 * q + 3] = y.w;
    }
  }
  float cm[3] = {t.bv[0], t.bv[1], t.bv[2]};   // each block's current maximum
  Top3 r;
#pragma unroll
  for (int e = 0; e < 3; ++e) {
    const float mx = fmaxf(fmaxf(cm[0], cm[1]), cm[2]);
    int best = 0x7fffffff, bsel = -1, isel = 0;
#pragma unroll
    for (int b = 0; b < 3; ++b) {
      if (cm[b] == mx && t.bv[b] > -INFINITY) {
        uint32_t eq[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int i = 0; i < 32; ++i) eq[i & 3] |= (x[b][i] == mx ? 1u : 0u) << i;
        const uint32_t msk = (eq[0] | eq[1]) | (eq[2] | eq[3]);
        const int i = __ffs(msk) - 1;
        if (msk && t.b0[b] + i < best) { best = t.b0[b] + i; bsel = b; isel = i; }
      }
    }
    r.v[e] = mx;
    r.i[e] = best;
    if (e < 2) {
#pragma unroll
      for (int b = 0; b < 3; ++b) {
        if (b == bsel) {
#pragma unroll
          for (int i = 0; i < 32; ++i) x[b][i] = (i == isel) ? -INFINITY : x[b][i];
          cm[b] = block_max32(x[b]);
        }
      }
    }
  }
  return r;
}

template <int kS>
__global__ void __launch_bounds__(kThreads, 1)
route_shared_tc_kernel(const __grid_constant__ CUtensorMap map_q,
                       const __grid_constant__ CUtensorMap map_qt,
                       const float* __restrict__ v_tilde, int N, int m, int nch, int G_h,
                       float cs_shared, int o_bf16, int32_t* __restrict__ route,
                       float* __restrict__ shared_lse, void* __restrict__ shared_o,
                       int* __restrict__ amb, int* status, int* __restrict__ hist) {
  griddep_wait();
  // amb: the heads' counts at amb[0, BH), then head bh's query ids at amb + BH + bh * N,
  // then (as floats) their fp32 best scores at amb + BH + BH * N + bh * N
  extern __shared__ unsigned char smem_raw[];
  using Cfg = RsCfg<kS>;
  constexpr int kQStages = Cfg::kQStages;
  RsSmem<kS>& s = *reinterpret_cast<RsSmem<kS>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.x / G_h, c0 = blockIdx.x % G_h;
  const int nqt = (N + 127) / 128;
  const int ntiles = (c0 < nqt) ? (nqt - c0 + G_h - 1) / G_h : 0;   // this CTA's tiles

  if (threadIdx.x == 0) {
    for (int i = 0; i < kQStages; ++i) {
      mbar_init(&s.q_full[i], 1);
      mbar_init(&s.q_empty[i], 1 + 4);   // the tile's last S commit + its four softmax warps
    }
    mbar_init(&s.res_full, 1 + kSoftThreads / 32);   // the q~ copy + the v~ converters
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.s_full[i], 1);
      mbar_init(&s.s_free[i], 4);
      mbar_init(&s.p_full[i], 4);
      mbar_init(&s.pv_done[i], 1);
      mbar_init(&s.drain[i], 1);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&s.tmem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = s.tmem;
  // tensor memory, slot t at 256 * t: S (128 columns), P (64, bf16 pairs), O (64)
  // registers: the launch grants 384 x 168; warps 0-3 keep 40 each, the softmax warps take
  // 232 (128 * 40 + 256 * 232 = 384 * 168)

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 40;\n" ::: "memory");
    if (warp == 0) {
      // ------------------------------------------------------------ producer
      bool ok = true;
      if (elect_one()) {
        prefetch_tmap(&map_q);
        prefetch_tmap(&map_qt);
        mbar_expect_tx(&s.res_full, (uint32_t)(nch * BN * 128));
        for (int ch = 0; ch < nch; ++ch)
          tma_load_3d(s.qt + ch * BN * 64, &map_qt, &s.res_full, 0, ch * BN, bh);
      }
      __syncwarp();
      for (int j = 0; j < ntiles; ++j) {
        const int st = j % kQStages;
        if (!mbar_wait_warp(&s.q_empty[st], ((j / kQStages) & 1) ^ 1)) { ok = false; break; }
        if (elect_one()) {
          mbar_expect_tx(&s.q_full[st], 128 * 128);
          tma_load_3d(s.q[st], &map_q, &s.q_full[st], 0, (c0 + j * G_h) * 128, bh);
        }
        __syncwarp();
      }
      if (!ok && lane == 0) flag_error(status, kDevErrTimeout);
    } else if (warp == 1 || warp == 2) {
      // ---------------------------------------------------------- MMA issuer of one slot
      const int slot = warp - 1;
      const int my_tiles = ntiles > slot ? (ntiles - slot + 1) / 2 : 0;
      const int G = my_tiles * nch;
      const uint32_t id_s = idesc_f16(128, BN, false);
      const uint32_t id_pv = idesc_f16(128, 64, true);
      const uint32_t tS = tbase + slot * 256, tP = tS + 128, tO = tS + 192;
      const uint32_t qtb = smem_u32(s.qt), vtb = smem_u32(s.vt);
      bool ok = mbar_wait_warp(&s.res_full, 0);
      auto issue_s = [&](int g) -> bool {
        const int it = g / nch, c = g % nch;
        const int j = slot + 2 * it, st = j % kQStages;
        if (c == 0 && !mbar_wait_warp(&s.q_full[st], (j / kQStages) & 1)) return false;
        tc_fence_after();
        const uint32_t qa = smem_u32(s.q[st]), kb = qtb + c * BN * 128;
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ss(tS, smem_desc_sw128(qa + kk * 32, 1024), smem_desc_sw128(kb + kk * 32, 1024),
                   id_s, kk > 0);
          mma_commit(&s.s_full[slot]);
          if (c == nch - 1) mma_commit(&s.q_empty[st]);
        }
        __syncwarp();
        return true;
      };
      if (ok && G > 0) ok = issue_s(0);
      for (int g = 0; g < G && ok; ++g) {
        const int c = g % nch;
        if (g + 1 < G) {
          if (!mbar_wait_warp(&s.s_free[slot], g & 1)) { ok = false; break; }
          if (!issue_s(g + 1)) { ok = false; break; }
        }
        if (!mbar_wait_warp(&s.p_full[slot], g & 1)) { ok = false; break; }
        tc_fence_after();
        const uint32_t vb = vtb + c * BN * 128;
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            mma_ts(tO, tP + kk * 8, smem_desc_sw128(vb + kk * 2048, 1024), id_pv, c > 0 || kk > 0);
          mma_commit(&s.pv_done[slot]);
        }
        __syncwarp();
      }
      if (elect_one()) mma_commit(&s.drain[slot]);
      __syncwarp();
      if (!mbar_wait_warp(&s.drain[slot], 0)) ok = false;
      if (!ok && lane == 0) flag_error(status, kDevErrTimeout);
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 232;\n" ::: "memory");
    // ------------------------------------------------------------ softmax
    const int et = threadIdx.x - 128;           // 0..255
    const int slot = (warp - 4) >> 2;
    const int quad = warp & 3;                  // tensor-memory lanes this warp may access
    const int row = quad * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t tS = tbase + lane_off + slot * 256, tP = tS + 128, tO = tS + 192;
    float4* bb = s.bbuf[0][et];
    constexpr int kSlotStride = kSoftThreads * 8;   // float4s from one block copy slot to the next
    const int sw = et & 7;
    bool ok = true;
    // v~ (fp32 in global memory) -> bf16 rows in the MMA's 128B-swizzled layout; rows from m
    // up to the last chunk's end are zero (their P is zero, but 0 * NaN would not be)
    {
      const int rows = nch * BN;
      for (int t = et; t < rows * 8; t += kSoftThreads) {
        const int r = t >> 3, c = t & 7;
        uint4 o = make_uint4(0u, 0u, 0u, 0u);
        if (r < m) {
          const float4* src = reinterpret_cast<const float4*>(v_tilde + ((size_t)bh * m + r) * 64 + c * 8);
          const float4 a = src[0], b = src[1];
          o.x = pack_bf16(a.x, a.y);
          o.y = pack_bf16(a.z, a.w);
          o.z = pack_bf16(b.x, b.y);
          o.w = pack_bf16(b.z, b.w);
        }
        *reinterpret_cast<uint4*>(reinterpret_cast<char*>(s.vt) + sw128_offset(r, c)) = o;
      }
      fence_proxy_async_smem();   // the tensor cores read what these threads wrote
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.res_full);
    }
    if (!mbar_wait(&s.res_full, 0)) ok = false;
    // largest landmark norm of the head (error bound of the fp32 logits)
    float n2max = 0.f;
    if (ok) {
      for (int i = et; i < m; i += kSoftThreads) {
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
    soft_bar();
    float qtmax2 = 0.f;
#pragma unroll
    for (int i = 0; i < kSoftThreads / 32; ++i) qtmax2 = fmaxf(qtmax2, s.red[i]);
    const float gq = 2.f * err_gamma(64) * sqrtf(qtmax2);
    const float cs = cs_shared;
    int* hcnt = amb + bh;
    const size_t BHs = gridDim.x / G_h;
    int* hids = amb + BHs + (size_t)bh * N;
    float* hbest = reinterpret_cast<float*>(amb + BHs + BHs * N) + (size_t)bh * N;
    // the finished tile's partial leaves once its last P . V is done
    // (the tensor-memory loads are warp-collective: every lane takes part, whether or not
    // its row is written)
    auto write_partial = [&](int n, float l, float mr) {
      const bool wr = ok && n >= 0;
      const float inv = 1.f / l;
      const size_t qi = (size_t)bh * N + (wr ? n : 0);
      if (wr) shared_lse[qi] = (mr + log2f(l)) * 0.6931471805599453f;   // natural log
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float o[32];
        tmem_ld32(tO + half * 32, o);
        tmem_ld_wait();
        tmem_fence_regs<32>(o);
        if (!wr) continue;
        if (o_bf16) {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<bf16*>(shared_o) + qi * 64 + half * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_uint4(pack_bf16(o[8 * i] * inv, o[8 * i + 1] * inv),
                                pack_bf16(o[8 * i + 2] * inv, o[8 * i + 3] * inv),
                                pack_bf16(o[8 * i + 4] * inv, o[8 * i + 5] * inv),
                                pack_bf16(o[8 * i + 6] * inv, o[8 * i + 7] * inv));
        } else {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(shared_o) + qi * 64 + half * 32);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(o[4 * i] * inv, o[4 * i + 1] * inv, o[4 * i + 2] * inv,
                                 o[4 * i + 3] * inv);
        }
      }
    };
    // the second slot's group starts half a chunk late (the two then take turns on the
    // exponential unit instead of competing for it in lockstep)
    if (slot == 1) __nanosleep(500);
    const int my_tiles = ntiles > slot ? (ntiles - slot + 1) / 2 : 0;
    int g = 0;
    int prev_n = -1;
    float prev_l = 1.f, prev_m = 0.f;
    bool pending = false;
    for (int it = 0; it < my_tiles; ++it) {
      const int j = slot + 2 * it, st = j % kQStages;
      const int n = (c0 + j * G_h) * 128 + row;
      if (ok && !mbar_wait(&s.q_full[st], (j / kQStages) & 1)) ok = false;
      // the query's error bound, before the tile is released
      float twoE = 0.f;
      if (ok && n < N) {
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
      if (lane == 0) mbar_arrive(&s.q_empty[st]);   // this warp is done with the tile
      const bool live = ok && n < N;
      RowTop top;
      Top3Blocks top3;
      float mref = -INFINITY, lsum = 0.f;
      for (int c = 0; c < nch; ++c, ++g) {
        if (ok && !mbar_wait(&s.s_full[slot], g & 1)) ok = false;
        tc_fence_after();
        const int nvalid = min(BN, m - c * BN);
        // warp-collective loads (no lane may skip them), with each 32-column block's maximum
        float v[BN];
        float q4[4];
#pragma unroll
        for (int b = 0; b < 4; ++b) q4[b] = tmem_ld32_max(tS + 32 * b, v + 32 * b);
        tmem_ld_wait();
        tmem_fence_regs<BN>(v);
        tmem_fence_regs<4>(q4);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.s_free[slot]);   // the next S may overwrite these columns
        if (nvalid < BN) {           // a ragged chunk: its blocks' maxima over valid entries
#pragma unroll
          for (int i = 0; i < BN; ++i) v[i] = i < nvalid ? v[i] : -INFINITY;
#pragma unroll
          for (int b = 0; b < 4; ++b) q4[b] = block_max32(v + 32 * b);
        }
        // the running best over 32-score blocks (s = 2: the three best blocks); the chunk
        // maximum is the blocks' maximum
        float tm = -INFINITY;
#pragma unroll
        for (int b = 0; b < BN / 32; ++b) {
          if (b * 32 < nvalid) {
            if constexpr (kS == 1) {
              tm = fmaxf(tm, top_block(top, v + 32 * b, q4[b], c * BN + b * 32, bb, sw));
            } else {
              tm = fmaxf(tm, q4[b]);
              top3_block(top3, v + 32 * b, q4[b], c * BN + b * 32, bb, kSlotStride, sw);
            }
          }
        }
        const float xm = tm * cs;
        const bool need = (c == 0) || (xm > mref + kLazy);
        const float f = (c > 0 && need) ? ex2(mref - xm) : 1.f;
        if (need) {
          lsum *= f;
          mref = xm;
        }
        const unsigned long long c2 = f2pack(cs, cs), nm2 = f2pack(-mref, -mref);
        unsigned long long lsa = f2pack(0.f, 0.f), lsb = lsa;
        auto exp_half = [&](int base, uint32_t* pk) {
#pragma unroll
          for (int i = 0; i < BN / 2; i += 2) {
            float x0, x1;
            f2unpack(fma2(f2pack(v[base + i], v[base + i + 1]), c2, nm2), x0, x1);
            const float p0 = ex2(x0), p1 = ex2(x1);
            if ((i >> 1) & 1) lsb = add2(lsb, f2pack(p0, p1));
            else lsa = add2(lsa, f2pack(p0, p1));
            pk[i / 2] = pack_bf16(p0, p1);
          }
        };
        uint32_t pk0[BN / 4];
        exp_half(0, pk0);
        // the previous P . V must have read P and finished with O
        if (g > 0 && ok && !mbar_wait(&s.pv_done[slot], (g - 1) & 1)) ok = false;
        tc_fence_after();
        tmem_st16(tP, pk0);
        tmem_st16(tP + 16, pk0 + 16);
        if (pending) {
          write_partial(prev_n, prev_l, prev_m);
          pending = false;
        }
        uint32_t pk1[BN / 4];
        exp_half(BN / 2, pk1);
        tmem_st16(tP + 32, pk1);
        tmem_st16(tP + 48, pk1 + 16);
        float la0, la1, lb0, lb1;
        f2unpack(lsa, la0, la1);
        f2unpack(lsb, lb0, lb1);
        lsum += (la0 + la1) + (lb0 + lb1);
        if (c > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            float o[16];
            tmem_ld16(tO + h * 16, o);
            tmem_ld_wait();
            tmem_fence_regs<16>(o);
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] *= f;
            tmem_st16(tO + h * 16, reinterpret_cast<uint32_t*>(o));
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.p_full[slot]);
      }
      // the route: exact when the best beats the runner-up by more than 2E (s = 2: when
      // both the first and the second gap exceed 2E); `keep` is the fp32 score of the
      // s-th route, the fix-up's screening reference
      bool ambiguous;
      float keep;
      if constexpr (kS == 1) {
        const Cand cd = finish_top(top, bb, sw);
        ambiguous = live && !(cd.v1 - cd.v2 > twoE);
        keep = cd.v1;
        if (live) {
          route[(size_t)bh * N + n] = cd.i1;
          if (hist && !ambiguous && cd.i1 >= 0 && cd.i1 < m)
            atomicAdd(&hist[((size_t)bh * m + cd.i1) * ((N + kBucketChunk - 1) / kBucketChunk) +
                            n / kBucketChunk], 1);
        }
      } else {
        const Top3 t3 = finish_top3(top3, bb, kSlotStride, sw);
        ambiguous = live && !(t3.v[0] - t3.v[1] > twoE && t3.v[1] - t3.v[2] > twoE);
        keep = t3.v[1];
        if (live) {
          route[((size_t)bh * N + n) * 2] = t3.i[0];
          route[((size_t)bh * N + n) * 2 + 1] = t3.i[1];
          // the bucket stage's counts of its N * 2 entries (entry 2n + r)
          if (hist && !ambiguous) {
            const long long nck = ((long long)N * 2 + kBucketChunk - 1) / kBucketChunk;
#pragma unroll
            for (int r = 0; r < 2; ++r) {
              const int e = t3.i[r];
              if (e >= 0 && e < m)
                atomicAdd(&hist[((size_t)bh * m + e) * nck + (2LL * n + r) / kBucketChunk], 1);
            }
          }
        }
      }
      const unsigned am = __ballot_sync(0xffffffffu, ambiguous);
      if (am) {
        int base = 0;
        if (lane == 0) base = atomicAdd(hcnt, __popc(am));
        base = __shfl_sync(0xffffffffu, base, 0);
        if (ambiguous) {
          const int pos = base + __popc(am & ((1u << lane) - 1u));
          hids[pos] = n;
          hbest[pos] = keep;
        }
      }
      prev_n = live ? n : -1;
      prev_l = lsum;
      prev_m = mref;
      pending = true;
    }
    if (pending) {
      if (ok && g > 0 && !mbar_wait(&s.pv_done[slot], (g - 1) & 1)) ok = false;
      tc_fence_after();
      write_partial(prev_n, prev_l, prev_m);
    }
    tc_fence_before();
    if (!ok) flag_error(status, kDevErrTimeout);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, 512);
}

}  // namespace

bool route_shared_tc_supported(int d, int m, int s) {
  if (d != 64 || m < 1 || m < s) return false;
  if (s == 1) return m <= RsCfg<1>::kMaxM;
  if (s == 2) return m <= RsCfg<2>::kMaxM;
  return false;
}

cudaError_t launch_route_shared_tc(const bf16* q, const bf16* q_tilde, const float* v_tilde,
                                   int BH, int N, int m, int num_sms, int shared_temp,
                                   int o_bf16, int32_t* route, float* shared_lse, void* shared_o,
                                   int* amb, int* status, int* hist, cudaStream_t st,
                                   bool prezeroed, int s) {
  if (!route_shared_tc_supported(64, m, s)) return cudaErrorInvalidValue;
  const int nch = (m + BN - 1) / BN;
  CUtensorMap mq, mqt;
  if (!make_tmap_rows64(&mq, q, (uint64_t)N, (uint64_t)BH, 128) ||
      !make_tmap_rows64(&mqt, q_tilde, (uint64_t)m, (uint64_t)BH, BN))
    return cudaErrorInvalidValue;
  const int nqt = (N + 127) / 128;
  int G_h = std::max(1, (num_sms + BH - 1) / BH);
  G_h = std::min(G_h, nqt);
  const size_t smem = (s == 1 ? sizeof(RsSmem<1>) : sizeof(RsSmem<2>)) + 1024;
  auto kern = s == 1 ? route_shared_tc_kernel<1> : route_shared_tc_kernel<2>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (!prezeroed && (e = cudaMemsetAsync(amb, 0, (size_t)BH * sizeof(int), st)) != cudaSuccess)
    return e;
  if (hist && !prezeroed) {
    const size_t nh = (size_t)BH * m * (((size_t)N * s + kBucketChunk - 1) / kBucketChunk);
    if ((e = cudaMemsetAsync(hist, 0, nh * sizeof(int), st)) != cudaSuccess) return e;
  }
  // shared logits in log2 units: log2(e) / sqrt(64), or log2(e) / 64 (the official code's)
  const float cs = shared_temp ? 0.022542110013890052f : 0.18033688011112042f;
  e = launch_pdl(kern, dim3((unsigned)(BH * G_h)), dim3(kThreads), smem, st, mq, mqt, v_tilde, N,
                 m, nch, G_h, cs, o_bf16, route, shared_lse, shared_o, amb, status, hist);
  count_launch();
  if (e != cudaSuccess) return e;
  if (s == 1) return launch_route_fixup(q, q_tilde, BH, N, m, num_sms, route, amb, hist, st);
  return launch_route_fixup_top(q, q_tilde, BH, N, m, s, num_sms, route, amb, hist, st);
}

}  // namespace mita
