// Steps 2-3 on the tensor cores (bf16, d = 64): shared landmark values and
// the per-landmark top-k key sets, for long sequences.
//
// MiTA tutorial (iwxt.cn), ch. 4 step 2 (paper eq. 6-7): landmark i scores
// all N keys with q~_i . k_j / sqrt(d) and keeps its top-k rows as expert i;
// ch. 4 step 3 (eq. 8-9): softmax over all N of the same scores weights V
// into v~_i.  The m x N score matrix never reaches HBM.
//
// Two sweeps over the keys, each split over CTAs (flash-decoding style):
//
// sweep (pass 1), CTA = (head, 128 landmarks, key split):
//   warp 0       TMA: K tiles of 128 keys into an 8-deep ring (a slot is freed
//                as soon as S is computed);
//   warps 1-2    MMA, one issuing warp per softmax group: S = q~ K^T into the
//                group's tensor memory, the group's next S as soon as the
//                softmax has copied S out, then O += P V with P read from
//                tensor memory;
//   warp 3       TMA: V tiles into a 4-deep ring (a slot is freed once P V is
//                done), so K runs ahead of V by the softmax latency; and the
//                largest |k| element of the split's keys, a bound on |k|^2
//                for the error bound of the fp32 scores (the split's nrt
//                row-block CTAs scan every nrt-th tile each; the threshold
//                kernel takes the maximum);
//   warps 4-7,   two softmax warpgroups that take alternate key tiles, each
//   warps 8-11   with its own online-softmax state (max, sum) and its own O
//                accumulator, so one computes while the other's MMAs run.
//                Rescaling of O is lazy (only when the max grows by more than
//                2^8).  Each also writes every key tile's largest raw score
//                per landmark row to a tile-maximum table (bm).
// threshold, CTA = one landmark: merges the softmax partials into v~
//   (tutorial ch. 4: (Z1 o1 + Z2 o2) / (Z1 + Z2)) and takes tau_L, a lower
//   bound of the row's k-th largest tile maximum (the lower edge of the
//   histogram bin where the count from the top reaches k).  k distinct tiles
//   reach tau_L, so at least k
//   keys score >= tau_L: every top-k key scores >= tau_L - E (exactly) and
//   >= tau_L - 2E in fp32 (E bounds the fp32 error).  Collection uses
//   tau_L - 4E, which stays valid even if pass 2's fp32 scores differ from
//   pass 1's by up to 2E.
// collect (pass 2): S = q~ K^T again; keys at or above the threshold are
//   appended to the row's candidate list (typically k plus a few).
// The exact selection over the candidates is landmark_select_kernel.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"

namespace mita {
namespace {
using namespace sm100;

constexpr int BN = 128;          // keys per tile
constexpr int kKRing = 8;        // sweep: K ring depth (K is freed as soon as S is computed)
constexpr int kVRing = 4;        // sweep: V ring depth (V is held until P . V is done)
constexpr int kThreads = 384;    // 12 warps
constexpr float kLazy = 8.0f;    // rescale O only when the max grows by > 2^8

__device__ __forceinline__ float softmax_c() { return 0.18033688011112042f; }  // log2(e)/8

struct alignas(1024) SweepSmem {
  bf16 qt[128 * 64];
  bf16 k[kKRing][BN * 64];
  bf16 v[kVRing][BN * 64];
  uint64_t k_full[kKRing], k_empty[kKRing], v_full[kVRing], v_empty[kVRing];
  uint64_t qt_full, drain[2];
  uint64_t s_full[2], s_free[2], p_full[2], pv_done[2];
  float nred;
  uint32_t tmem;
};

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Single MUFU 2^x (flushes subnormal results to zero; P is bf16 anyway).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
// max of |x| over the 64 bf16 values of a 128-byte row group: bf16 magnitudes
// (sign cleared) order like their 15-bit integer patterns.
__device__ __forceinline__ uint32_t umax16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// -------------------------------------------------------------------------------------------
// pass 1
// -------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 1)
lm_sweep_kernel(const __grid_constant__ CUtensorMap map_qt, const __grid_constant__ CUtensorMap map_k,
                const __grid_constant__ CUtensorMap map_v, int N, int m, int S, int split_len,
                LandmarkWs ws, int* status) {
  griddep_wait();
  extern __shared__ unsigned char smem_raw[];
  SweepSmem& s = *reinterpret_cast<SweepSmem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nrt = (m + 127) / 128;
  int b = blockIdx.x;                 // row tiles of one key split are adjacent (L2 reuse)
  const int rt = b % nrt; b /= nrt;
  const int sp = b % S;
  const int bh = b / S;
  const int j0 = sp * split_len;
  const int j1 = min(N, j0 + split_len);
  const int ntl = (j1 - j0 + BN - 1) / BN;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kKRing; ++i) {
      mbar_init(&s.k_full[i], 1);
      mbar_init(&s.k_empty[i], 2);         // the tile's S commit + the norm warp
    }
    for (int i = 0; i < kVRing; ++i) {
      mbar_init(&s.v_full[i], 1);
      mbar_init(&s.v_empty[i], 1);         // the tile's P . V commit
    }
    mbar_init(&s.qt_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.drain[i], 1);
      mbar_init(&s.s_full[i], 1);
      mbar_init(&s.s_free[i], 4);          // one arrival per softmax warp
      mbar_init(&s.p_full[i], 4);
      mbar_init(&s.pv_done[i], 1);
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
  // tensor memory, softmax group (slot) g at 256*g: S (128 columns), P (64, bf16 pairs), O (64).
  // registers: the launch grants 384 x 168; warps 0-3 keep 56 each, the two softmax
  // warpgroups take 224 each (128*56 + 2*128*224 = 384*168).

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 56;\n" ::: "memory");
    if (warp == 0) {
      bool ok = true;
      if (elect_one()) {
        prefetch_tmap(&map_qt);
        prefetch_tmap(&map_k);
        prefetch_tmap(&map_v);
        mbar_expect_tx(&s.qt_full, 128 * 128);
        tma_load_3d(s.qt, &map_qt, &s.qt_full, 0, rt * 128, bh);
      }
      __syncwarp();
      for (int j = 0; j < ntl; ++j) {
        const int st = j % kKRing;
        if (!mbar_wait_warp(&s.k_empty[st], ((j / kKRing) & 1) ^ 1)) { ok = false; break; }
        if (elect_one()) {
          mbar_expect_tx(&s.k_full[st], BN * 128);
          tma_load_3d(s.k[st], &map_k, &s.k_full[st], 0, j0 + j * BN, bh);
        }
        __syncwarp();
      }
      if (!ok && lane == 0) flag_error(status, kDevErrTimeout);
    } else if (warp == 1 || warp == 2) {
      // MMA issuer of softmax group `slot` (tiles j = slot, slot + 2, ...): whole warp,
      // one elected lane issues
      const int slot = warp - 1;
      const uint32_t id_s = idesc_f16(128, BN, false);
      const uint32_t id_pv = idesc_f16(128, 64, true);
      const uint32_t tS = tbase + slot * 256, tP = tS + 128, tO = tS + 192;
      const uint32_t qa = smem_u32(s.qt);
      bool ok = mbar_wait_warp(&s.qt_full, 0);
      auto issue_s = [&](int j) -> bool {
        const int st = j % kKRing;
        if (!mbar_wait_warp(&s.k_full[st], (j / kKRing) & 1)) return false;
        tc_fence_after();
        const uint32_t kb = smem_u32(s.k[st]);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ss(tS, smem_desc_sw128(qa + kk * 32, 1024), smem_desc_sw128(kb + kk * 32, 1024),
                   id_s, kk > 0);
          mma_commit(&s.s_full[slot]);
          mma_commit(&s.k_empty[st]);
        }
        __syncwarp();
        return true;
      };
      if (ok && slot < ntl) ok = issue_s(slot);
      int t = 0;
      for (int j = slot; j < ntl && ok; j += 2, ++t) {
        const int st = j % kVRing;
        if (j + 2 < ntl) {
          if (!mbar_wait_warp(&s.s_free[slot], t & 1)) { ok = false; break; }
          if (!issue_s(j + 2)) { ok = false; break; }
        }
        if (!mbar_wait_warp(&s.p_full[slot], t & 1)) { ok = false; break; }
        if (!mbar_wait_warp(&s.v_full[st], (j / kVRing) & 1)) { ok = false; break; }
        tc_fence_after();
        const uint32_t vb = smem_u32(s.v[st]);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            mma_ts(tO, tP + kk * 8, smem_desc_sw128(vb + kk * 2048, 1024), id_pv, t > 0 || kk > 0);
          mma_commit(&s.v_empty[st]);
          mma_commit(&s.pv_done[slot]);
        }
        __syncwarp();
      }
      if (elect_one()) mma_commit(&s.drain[slot]);
      __syncwarp();
      if (!mbar_wait_warp(&s.drain[slot], 0)) ok = false;
      if (!ok && lane == 0) flag_error(status, kDevErrTimeout);
    } else {
      // V producer (tile j into the V ring as soon as its slot is free), and the
      // largest |k| element of the split (bounds every key norm by 8 max|k|);
      // zero-filled rows past N are harmless.  The nrt CTAs of a key split (one per
      // 128-landmark block) share that maximum: each reads every nrt-th K tile (the
      // reads compete with the MMAs for shared-memory bandwidth), and the threshold
      // pass takes the maximum of their nrt partial maxima.
      uint32_t mx = 0u;
      bool ok = true;
      int vj = 0;                       // next V tile to request
      auto issue_v = [&](int upto) {
        for (; vj < upto && vj < ntl && ok; ++vj) {
          const int vs = vj % kVRing;
          if (!mbar_wait_warp(&s.v_empty[vs], ((vj / kVRing) & 1) ^ 1)) { ok = false; break; }
          if (elect_one()) {
            mbar_expect_tx(&s.v_full[vs], BN * 128);
            tma_load_3d(s.v[vs], &map_v, &s.v_full[vs], 0, j0 + vj * BN, bh);
          }
          __syncwarp();
        }
      };
      issue_v(kVRing);
      for (int j = 0; j < ntl; ++j) {
        const int st = j % kKRing;
        if (ok && !mbar_wait(&s.k_full[st], (j / kKRing) & 1)) ok = false;
        if (ok && j % nrt == rt) {
          const uint4* src = reinterpret_cast<const uint4*>(s.k[st]);
#pragma unroll 8
          for (int i = lane; i < 1024; i += 32) {
            const uint4 x = src[i];
            mx = umax16x2(mx, x.x & 0x7fff7fffu);
            mx = umax16x2(mx, x.y & 0x7fff7fffu);
            mx = umax16x2(mx, x.z & 0x7fff7fffu);
            mx = umax16x2(mx, x.w & 0x7fff7fffu);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.k_empty[st]);
        issue_v(j + kVRing + 1);
      }
      issue_v(ntl);
      const float a = fmaxf(__uint_as_float(mx << 16), __uint_as_float(mx & 0xffff0000u));
      const float km = warp_max(a);
      if (lane == 0) s.nred = 64.f * km * km;   // bound on |k|^2
      if (!ok && lane == 0) flag_error(status, kDevErrTimeout);
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 224;\n" ::: "memory");
    // ------------------------------------------------------------ softmax
    const int slot = (warp - 4) >> 2;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const int grow = rt * 128 + row;                // landmark index
    const bool live_row = grow < m;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t tS = tbase + lane_off + slot * 256, tP = tS + 128, tO = tS + 192;
    const float c = softmax_c();
    float mref = -INFINITY, lsum = 0.f;
    bool ok = true;
    int t = 0;
    const size_t rf = (size_t)bh * m + grow;
    float* tmax = ws.bm + rf * (size_t)((N + BN - 1) / BN) + j0 / BN;   // this split's tiles
    // the second group starts half a tile late, so the two take turns on the
    // exponential unit instead of competing for it in lockstep
    if (slot == 1) __nanosleep(500);
    for (int j = slot; j < ntl; j += 2, ++t) {
      if (ok && !mbar_wait(&s.s_full[slot], t & 1)) ok = false;
      tc_fence_after();
      const int kbase = j0 + j * BN;
      const int nvalid = min(BN, j1 - kbase);
      const bool full = nvalid == BN;
      // the tile's scores, with the maximum of each 32-column block from the reducing load
      float v[BN];
      float q4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      if (ok) {
#pragma unroll
        for (int b = 0; b < 4; ++b) q4[b] = tmem_ld32_max(tS + 32 * b, v + 32 * b);
        tmem_ld_wait();
        tmem_fence_regs<BN>(v);
        tmem_fence_regs<4>(q4);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.s_free[slot]);   // the next S may overwrite these columns
      // the tile's largest raw score (a ragged tile: over its valid keys only)
      float tm = fmaxf(fmaxf(q4[0], q4[1]), fmaxf(q4[2], q4[3]));
      if (!full) {
#pragma unroll
        for (int i = 0; i < BN; ++i) v[i] = i < nvalid ? v[i] : -INFINITY;
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};   // four independent chains
#pragma unroll
        for (int i = 0; i < BN; i += 8)
#pragma unroll
          for (int a = 0; a < 4; ++a) m4[a] = max3(m4[a], v[i + 2 * a], v[i + 2 * a + 1]);
        tm = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      }
      // every tile's maximum raw score goes out; the threshold pass takes the
      // k-th largest of the row's
      if (live_row) tmax[j] = tm;
      const float xm = tm * c;
      const bool need = (t == 0) || (xm > mref + kLazy);
      const float f = (t > 0 && need) ? ex2(mref - xm) : 1.f;
      if (need) {
        lsum *= f;
        mref = xm;
      }
      // P = exp2(s * c - mref) as bf16 pairs; the first half before waiting for the
      // previous P . V of this slot (which still reads P and accumulates O)
      const unsigned long long c2 = f2pack(c, c), nm2 = f2pack(-mref, -mref);
      unsigned long long ls2 = f2pack(0.f, 0.f), ls3 = ls2;   // two independent sum chains
      uint32_t pk[BN / 2];
#pragma unroll
      for (int i = 0; i < BN / 2; i += 2) {
        float x0, x1;
        f2unpack(fma2(f2pack(v[i], v[i + 1]), c2, nm2), x0, x1);
        const float p0 = ex2(x0), p1 = ex2(x1);
        if ((i >> 1) & 1) ls3 = add2(ls3, f2pack(p0, p1));
        else ls2 = add2(ls2, f2pack(p0, p1));
        pk[i / 2] = pack_bf16x2(p0, p1);
      }
      if (t > 0 && ok && !mbar_wait(&s.pv_done[slot], (t - 1) & 1)) ok = false;
      tc_fence_after();
      tmem_st16(tP, pk);
      tmem_st16(tP + 16, pk + 16);
#pragma unroll
      for (int i = BN / 2; i < BN; i += 2) {
        float x0, x1;
        f2unpack(fma2(f2pack(v[i], v[i + 1]), c2, nm2), x0, x1);
        const float p0 = ex2(x0), p1 = ex2(x1);
        if ((i >> 1) & 1) ls3 = add2(ls3, f2pack(p0, p1));
        else ls2 = add2(ls2, f2pack(p0, p1));
        pk[i / 2] = pack_bf16x2(p0, p1);
      }
      tmem_st16(tP + 32, pk + 32);
      tmem_st16(tP + 48, pk + 48);
      float ls_a, ls_b, ls_c, ls_d;
      f2unpack(ls2, ls_a, ls_b);
      f2unpack(ls3, ls_c, ls_d);
      lsum += (ls_a + ls_b) + (ls_c + ls_d);
      if (t > 0 && __any_sync(0xffffffffu, need)) {
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
    // final O of this slot
    float o[64];
    if (t > 0) {
      if (ok && !mbar_wait(&s.pv_done[slot], (t - 1) & 1)) ok = false;
      tc_fence_after();
      tmem_ld32(tO, o);
      tmem_ld32(tO + 32, o + 32);
      tmem_ld_wait();
      tmem_fence_regs<64>(o);
    } else {
#pragma unroll
      for (int i = 0; i < 64; ++i) o[i] = 0.f;
    }
    if (live_row) {
      const size_t pidx = ((size_t)bh * m + grow) * (2 * S) + sp * 2 + slot;
      ws.M[pidx] = mref;
      ws.L[pidx] = lsum;
      float4* dst = reinterpret_cast<float4*>(ws.A + pidx * 64);
#pragma unroll
      for (int i = 0; i < 16; ++i) dst[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
    }
    if (!ok) flag_error(status, kDevErrTimeout);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) ws.kmax2[((size_t)bh * S + sp) * nrt + rt] = s.nred;
  if (warp == 1) tmem_dealloc(tbase, 512);
}

// -------------------------------------------------------------------------------------------
// threshold, one CTA per landmark: v~ from the partials; tau_L = the topk-th
// largest of the row's tile maxima (each is the maximum of a distinct tile, so
// at least topk keys score >= tau_L)
// -------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
lm_threshold_kernel(const bf16* __restrict__ q_tilde, int m, int topk, int S2, int S,
                    int ntiles, LandmarkWs ws, float* __restrict__ v_tilde) {
  griddep_wait();
  __shared__ float red[8][5];
  __shared__ int hist[8 * 256];               // one histogram per warp
  __shared__ float vnum[4][64], vden[4];
  const long long rf = blockIdx.x;
  const long long bh = rf / m;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const size_t base = (size_t)rf * S2;
  const float* tm = ws.bm + (size_t)rf * ntiles;
  const bool vec = (ntiles & 3) == 0;         // rows start on 16 bytes
  // ---- one pass of reductions: the partials' maximum, the largest |k|^2, |q~|^2 and the
  // range of the tile maxima
  float mx = -INFINITY, km = 0.f, qn2 = 0.f, hi = -INFINITY, lo = INFINITY;
  for (int q = tid; q < S2; q += 256) mx = fmaxf(mx, ws.M[base + q]);
  for (int q = tid; q < S; q += 256) km = fmaxf(km, ws.kmax2[(size_t)bh * S + q]);
  if (tid < 64) {
    const float x = __bfloat162float(q_tilde[rf * 64 + tid]);
    qn2 = x * x;
  }
  auto range = [&](float v) {
    hi = fmaxf(hi, v);
    if (v > -INFINITY) lo = fminf(lo, v);
  };
  if (vec) {
    for (int t = tid; t < ntiles / 4; t += 256) {
      const float4 x = reinterpret_cast<const float4*>(tm)[t];
      range(x.x); range(x.y); range(x.z); range(x.w);
    }
  } else {
    for (int t = tid; t < ntiles; t += 256) range(tm[t]);
  }
  mx = warp_max(mx);
  km = warp_max(km);
  qn2 = warp_sum(qn2);
  hi = warp_max(hi);
  lo = -warp_max(-lo);
  if (lane == 0) {
    red[w][0] = mx; red[w][1] = km; red[w][2] = qn2; red[w][3] = hi; red[w][4] = lo;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) hist[i * 256 + tid] = 0;
  __syncthreads();
  mx = red[0][0]; km = red[0][1]; qn2 = red[0][2]; hi = red[0][3]; lo = red[0][4];
#pragma unroll
  for (int i = 1; i < 8; ++i) {
    mx = fmaxf(mx, red[i][0]);
    km = fmaxf(km, red[i][1]);
    qn2 += red[i][2];
    hi = fmaxf(hi, red[i][3]);
    lo = fminf(lo, red[i][4]);
  }
  // ---- v~: the tutorial's (Z1 o1 + Z2 o2) / (Z1 + Z2) merge of the split partials,
  // four groups of 64 threads over interleaved partials
  {
    const int g = tid >> 6, l = tid & 63;
    float num = 0.f, den = 0.f;
    for (int q = g; q < S2; q += 4) {
      const float wq = exp2f(ws.M[base + q] - mx);
      den = fmaf(wq, ws.L[base + q], den);
      num = fmaf(wq, ws.A[(base + q) * 64 + l], num);
    }
    vnum[g][l] = num;
    if (l == 0) vden[g] = den;
  }
  // ---- tau_L: 256 bins between the smallest and largest finite tile maximum
  const bool binned = ntiles >= topk && hi > lo;
  const float scale = binned ? 256.f / (hi - lo) : 0.f;
  if (binned) {
    int* hw = hist + w * 256;
    auto bin = [&](float v) {
      if (v > -INFINITY) atomicAdd(&hw[min(255, (int)((v - lo) * scale))], 1);
    };
    if (vec) {
      for (int t = tid; t < ntiles / 4; t += 256) {
        const float4 x = reinterpret_cast<const float4*>(tm)[t];
        bin(x.x); bin(x.y); bin(x.z); bin(x.w);
      }
    } else {
      for (int t = tid; t < ntiles; t += 256) bin(tm[t]);
    }
  }
  __syncthreads();
  if (binned) {
    int c = 0;
#pragma unroll
    for (int u = 0; u < 8; ++u) c += hist[u * 256 + tid];
    hist[tid] = c;                            // column tid is this thread's alone
  }
  if (tid < 64) {
    const float num = (vnum[0][tid] + vnum[1][tid]) + (vnum[2][tid] + vnum[3][tid]);
    const float den = (vden[0] + vden[1]) + (vden[2] + vden[3]);
    v_tilde[rf * 64 + tid] = num / den;
    // the row's softmax normaliser (M in log2 units of the scaled scores)
    if (tid == 0 && ws.lse_out) ws.lse_out[rf] = (mx + log2f(den)) * 0.6931471805599453f;
  }
  __syncthreads();
  if (w == 0) {
    // lane l owns bins 255-8l .. 248-8l (high to low); the highest bin from which the count
    // of tile maxima at or above reaches topk.  Its lower edge, one bin lower to absorb the
    // rounding of the bin index, has at least topk tile maxima at or above it.
    float tauL = -INFINITY;
    if (binned) {
      int cnt[8], tot = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        cnt[j] = hist[255 - 8 * lane - j];
        tot += cnt[j];
      }
      const int inc = warp_incl_scan(tot);
      const unsigned hit = __ballot_sync(0xffffffffu, inc >= topk);
      int b = -1;
      if (hit) {
        const int src = __ffs(hit) - 1;
        int cum = inc - tot, dg = -1;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (dg < 0) {
            if (cum + cnt[j] >= topk) dg = 255 - 8 * lane - j;
            else cum += cnt[j];
          }
        }
        b = __shfl_sync(0xffffffffu, dg, src);
      }
      if (b >= 0) tauL = b > 0 ? lo + (float)(b - 1) / scale : lo;
    }
    if (lane == 0) {
      const float E = err_gamma(64) * sqrtf(qn2) * sqrtf(km);
      ws.E[rf] = E;
      ws.thr[rf] = tauL - 4.f * E;
      ws.cnt[rf] = 0;
    }
  }
}

// -------------------------------------------------------------------------------------------
// pass 2: collect the keys at or above the threshold
// -------------------------------------------------------------------------------------------
constexpr int kKStages = 8;
constexpr int kCSlots = 4;                  // tile groups in flight (tensor-memory buffers)
constexpr int kCThreads = (4 + 4 * kCSlots) * 32;
constexpr int kLocalCand = 64;   // candidates per row buffered in shared memory

struct alignas(1024) CollectSmem {
  bf16 qt[128 * 64];
  bf16 k[kKStages][BN * 64];
  float cs[kLocalCand][128];      // [slot][row]: lanes never share a bank
  int ci[kLocalCand][128];
  int cn[128];
  uint64_t k_full[kKStages], k_empty[kKStages];
  uint64_t qt_full, drain;
  uint64_t s_full[kCSlots], s_free[kCSlots];
  uint32_t tmem;
};

// pass 2, CTA = (head, 128 landmarks, key split): warp 0 streams K tiles by TMA,
// warp 1 issues S = q~ K^T for tile j into tensor-memory buffer j % 4, and four
// epilogue warpgroups (one per buffer, one landmark row per thread) compare the
// scores with the row's threshold and keep the keys at or above it.
__global__ void __launch_bounds__(kCThreads, 1)
lm_collect_kernel(const __grid_constant__ CUtensorMap map_qt, const __grid_constant__ CUtensorMap map_k,
                  int N, int m, int S, int split_len, int cap, LandmarkWs ws, int* status) {
  griddep_wait();
  extern __shared__ unsigned char smem_raw[];
  CollectSmem& s = *reinterpret_cast<CollectSmem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nrt = (m + 127) / 128;
  int b = blockIdx.x;                 // row tiles of one key split are adjacent (L2 reuse)
  const int rt = b % nrt; b /= nrt;
  const int sp = b % S;
  const int bh = b / S;
  const int j0 = sp * split_len;
  const int j1 = min(N, j0 + split_len);
  const int ntl = (j1 - j0 + BN - 1) / BN;

  if (threadIdx.x < 128) s.cn[threadIdx.x] = 0;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(&s.k_full[i], 1);
      mbar_init(&s.k_empty[i], 1);
    }
    mbar_init(&s.qt_full, 1);
    mbar_init(&s.drain, 1);
    for (int i = 0; i < kCSlots; ++i) {
      mbar_init(&s.s_full[i], 1);
      mbar_init(&s.s_free[i], 4);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&s.tmem, 128 * kCSlots);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = s.tmem;
  // registers: the launch grants 640 x 96; warps 0-3 keep 40 each, the four epilogue
  // warpgroups take 104 each (128*40 + 4*128*104 = 58368 <= 640*96)

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 40;\n" ::: "memory");
    if (warp == 0) {
      bool ok = true;
      if (elect_one()) {
        prefetch_tmap(&map_qt);
        prefetch_tmap(&map_k);
        mbar_expect_tx(&s.qt_full, 128 * 128);
        tma_load_3d(s.qt, &map_qt, &s.qt_full, 0, rt * 128, bh);
      }
      __syncwarp();
      for (int j = 0; j < ntl; ++j) {
        const int st = j % kKStages;
        if (!mbar_wait_warp(&s.k_empty[st], ((j / kKStages) & 1) ^ 1)) { ok = false; break; }
        if (elect_one()) {
          mbar_expect_tx(&s.k_full[st], BN * 128);
          tma_load_3d(s.k[st], &map_k, &s.k_full[st], 0, j0 + j * BN, bh);
        }
        __syncwarp();
      }
      if (!ok && lane == 0) flag_error(status, kDevErrTimeout);
    } else if (warp == 1) {
      // MMA issuer: whole warp, one elected lane issues
      const uint32_t id_s = idesc_f16(128, BN, false);
      const uint32_t qa = smem_u32(s.qt);
      bool ok = mbar_wait_warp(&s.qt_full, 0);
      for (int j = 0; j < ntl && ok; ++j) {
        const int st = j % kKStages, slot = j % kCSlots, t = j / kCSlots;
        if (!mbar_wait_warp(&s.k_full[st], (j / kKStages) & 1)) { ok = false; break; }
        if (!mbar_wait_warp(&s.s_free[slot], (t & 1) ^ 1)) { ok = false; break; }
        tc_fence_after();
        const uint32_t kb = smem_u32(s.k[st]);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ss(tbase + slot * 128, smem_desc_sw128(qa + kk * 32, 1024),
                   smem_desc_sw128(kb + kk * 32, 1024), id_s, kk > 0);
          mma_commit(&s.s_full[slot]);
          mma_commit(&s.k_empty[st]);
        }
        __syncwarp();
      }
      if (elect_one()) mma_commit(&s.drain);
      __syncwarp();
      if (!mbar_wait_warp(&s.drain, 0)) ok = false;
      if (!ok && lane == 0) flag_error(status, kDevErrTimeout);
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 104;\n" ::: "memory");
    const int slot = (warp - 4) >> 2;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const int grow = rt * 128 + row;
    const bool live_row = grow < m;
    const size_t rf = (size_t)bh * m + grow;
    const float thr = live_row ? ws.thr[rf] : INFINITY;
    const uint32_t tS = tbase + ((uint32_t)(quad * 32) << 16) + slot * 128;
    bool ok = true;
    int t = 0;
    for (int j = slot; j < ntl; j += kCSlots, ++t) {
      if (ok && !mbar_wait(&s.s_full[slot], t & 1)) ok = false;
      tc_fence_after();
      const int kbase = j0 + j * BN;
      const int nvalid = min(BN, j1 - kbase);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        // two 32-score blocks, each with its maximum from the reducing load
        float v[64];
        float bmx[2] = {-INFINITY, -INFINITY};
        if (ok) {
          bmx[0] = tmem_ld32_max(tS + h * 64, v);
          bmx[1] = tmem_ld32_max(tS + h * 64 + 32, v + 32);
          tmem_ld_wait();
          tmem_fence_regs<64>(v);
          tmem_fence_regs<2>(bmx);
        }
        if (h == 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&s.s_free[slot]);   // the next S may overwrite these columns
        }
        if (!ok) continue;
#pragma unroll
        for (int cc = 0; cc < 64; cc += 32) {
          const float* vv = v + cc;
          const int c0 = h * 64 + cc;
          // most blocks of 32 hold no candidate for any row of the warp: screen with
          // the block maximum (from the load itself; past the split's end it may count
          // keys outside it, which the mask below drops) before building the mask
          const float bmax = bmx[cc / 32];
          if (!__any_sync(0xffffffffu, bmax >= thr)) continue;
          // bitmask of the scores at or above the threshold (branch-free), then
          // visit only its set bits
          uint32_t msk = 0u;
#pragma unroll
          for (int i = 0; i < 32; ++i) msk |= (vv[i] >= thr ? 1u : 0u) << i;
          if (nvalid - c0 < 32) msk &= (nvalid - c0 <= 0) ? 0u : (0xffffffffu >> (32 - (nvalid - c0)));
          while (msk) {
            const int i = __ffs(msk) - 1;
            msk &= msk - 1;
            float x = vv[0];
#pragma unroll
            for (int u = 1; u < 32; ++u) x = (u == i) ? vv[u] : x;
            const int pos = atomicAdd(&s.cn[row], 1);
            if (pos < kLocalCand) {
              s.cs[pos][row] = x;
              s.ci[pos][row] = kbase + c0 + i;
            } else {
              const int gpos = atomicAdd(ws.cnt + rf, 1);
              if (gpos < cap) {
                ws.cand_s[rf * cap + gpos] = x;
                ws.cand_i[rf * cap + gpos] = kbase + c0 + i;
              }
            }
          }
        }
      }
    }
    if (!ok) flag_error(status, kDevErrTimeout);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, 128 * kCSlots);
  // flush the shared-memory candidate lists, one global reservation per row
  if (warp >= 4 && warp < 8) {
    const int row = (warp & 3) * 32 + lane;
    const int grow = rt * 128 + row;
    if (grow < m) {
      const size_t rf = (size_t)bh * m + grow;
      const int n = min(s.cn[row], kLocalCand);
      if (n > 0) {
        const int base = atomicAdd(ws.cnt + rf, n);
        for (int i = 0; i < n && base + i < cap; ++i) {
          ws.cand_s[rf * cap + base + i] = s.cs[i][row];
          ws.cand_i[rf * cap + base + i] = s.ci[i][row];
        }
      }
    }
  }
}

}  // namespace

bool landmark_tc_eligible(int d, int N, int topk) {
  // the threshold pass holds one row's tile maxima in shared memory (<= 192 KB)
  const long long ntiles = ((long long)N + BN - 1) / BN;
  return d == 64 && ntiles >= 2LL * topk && ntiles <= 49152;
}


void plan_landmark_tc(LandmarkPlan& p, int BH, int N, int m, int topk, int num_sms) {
  p.tc = true;
  p.RT = 128;
  p.nrt = (m + 127) / 128;
  const int ctas_per_split = BH * p.nrt;
  int S = std::max(1, (num_sms + ctas_per_split - 1) / ctas_per_split);
  S = std::min(S, (N + BN - 1) / BN);
  p.split_len = ((N + S - 1) / S + BN - 1) / BN * BN;
  p.S = (N + p.split_len - 1) / p.split_len;
  p.ntiles = (N + BN - 1) / BN;
  p.cap = std::min(8192, next_pow2(std::max(1024, 2 * topk + 256)));
  p.P = p.cap;
  p.Tcap = 0;
}

cudaError_t launch_landmark_tc_passes(const bf16* q_tilde, const bf16* k, const bf16* v, int BH,
                                      int N, int m, int topk, const LandmarkPlan& p,
                                      const LandmarkWs& ws, float* v_tilde, int* status,
                                      cudaStream_t st) {
  CUtensorMap mqt, mk, mv;
  if (!make_tmap_rows64(&mqt, q_tilde, (uint64_t)m, (uint64_t)BH, 128) ||
      !make_tmap_rows64(&mk, k, (uint64_t)N, (uint64_t)BH, BN) ||
      !make_tmap_rows64(&mv, v, (uint64_t)N, (uint64_t)BH, BN))
    return cudaErrorInvalidValue;
  const unsigned blocks = (unsigned)(BH * p.nrt * p.S);
  const size_t sm1 = sizeof(SweepSmem) + 1024;
  cudaError_t e = cudaFuncSetAttribute(lm_sweep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)sm1);
  if (e != cudaSuccess) return e;
  e = launch_pdl(lm_sweep_kernel, dim3(blocks), dim3(kThreads), sm1, st, mqt, mk, mv, N, m, p.S,
                 p.split_len, ws, status);
  count_launch();
  if (e != cudaSuccess) return e;
  // (kmax2 holds nrt partial maxima per key split: S * nrt per head)
  e = launch_pdl(lm_threshold_kernel, dim3((unsigned)((long long)BH * m)), dim3(256), 0, st,
                 q_tilde, m, topk, 2 * p.S, p.S * p.nrt, p.ntiles, ws, v_tilde);
  count_launch();
  if (e != cudaSuccess) return e;
  const size_t sm2 = sizeof(CollectSmem) + 1024;
  e = cudaFuncSetAttribute(lm_collect_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm2);
  if (e != cudaSuccess) return e;
  e = launch_pdl(lm_collect_kernel, dim3(blocks), dim3(kCThreads), sm2, st, mqt, mk, N, m, p.S,
                 p.split_len, p.cap, ws, status);
  count_launch();
  return e;
}

}  // namespace mita
