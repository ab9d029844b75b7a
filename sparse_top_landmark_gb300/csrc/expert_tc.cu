// Step 6 on the tensor cores (bf16, d = 64): for every query, one joint
// softmax over the m shared pairs (q~_i, v~_i) and the k raw pairs of its
// routed expert, computed expert by expert.
//
// MiTA tutorial (iwxt.cn), ch. 4 steps 5-6 (paper eq. 11-12): the m + s*k
// logits, all scaled by 1/sqrt(d), share one softmax over [v~; V(e)].  The
// bit.fan article: queries are grouped by expert and an online softmax runs
// over the concatenated entries; each expert's k KV rows are gathered once.
//
// Three launches:
//   expert_gather_kernel  the k K / V rows of every (head, expert), copied once
//                         into contiguous [head*m + expert][k][64] blocks;
//   expert_prep_kernel    the work-unit table (unit = (head, expert, up to 256
//                         of its queries)) and v~ in fp16;
//   expert_tc_kernel      persistent CTAs, each over a contiguous run of units
//                         (units of one expert follow each other, so its
//                         gathered rows are re-read from L2):
//     warp 0     TMA: the unit's query rows (tile::gather4 of scattered rows),
//                then the entries in chunks of 128 -- the expert's gathered
//                K / V block first, then the q~ / v~ blocks -- as tiled loads
//                into a 4-stage ring shared by the two query tiles;
//     warp 1     MMA: S = Q . B^T per tile into tensor memory; O += P . V with
//                P read from tensor memory (shared chunks as fp16 x fp16, v~
//                kept in fp16; raw chunks bf16 x bf16).  Three S buffers
//                rotate over the sequence (chunk, tile), P overwriting its own
//                S, so the next score tile is computed while both softmax
//                groups are busy;
//     warps 2-5 / 6-9    online softmax of query tile 0 / 1 (one query row per
//                thread, lazy O rescaling), then O / l to the output rows.
#include <algorithm>

#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"

namespace mita {
namespace {
using namespace sm100;

constexpr int BN = 128;          // entries per chunk
constexpr int kStages = 4;
constexpr int kThreads = 320;   // 10 warps: producer, MMA, 8 softmax
constexpr int kSBuf = 3;         // S / P buffers in tensor memory, shared by the two tiles
constexpr int kUnitQ = 256;      // queries per work unit (two MMA tiles)
constexpr float kLazy = 8.0f;
constexpr int kGatherThreads = 256;

struct alignas(1024) ExpertSmem {
  bf16 q[2][2][128 * 64];          // [unit buffer][query tile]
  bf16 kb[kStages][BN * 64];       // q~ block or the expert's K rows
  bf16 vb[kStages][BN * 64];       // v~ block (fp16) or the expert's V rows
  uint64_t kv_full[kStages], kv_empty[kStages];
  uint64_t q_full[2], q_empty[2];
  uint64_t s_full[3], p_full[3], pv_done[2];
  uint64_t drain;
  uint32_t tmem;
};

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
__device__ __forceinline__ uint32_t pack_pair(float a, float b, bool fp16) {
  if (fp16) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

struct ExpertTcWs {
  __half* vt16;      // [BH*m][64]
  int* unit_start;   // [BH*m + 1]
  int4* unit;        // [max units]: (head*m + expert, first bucket slot, count, 0)
  bf16* kg;          // [BH*m][topk][64]
  bf16* vg;
};

size_t max_units(int BH, int N, int m) {
  return (size_t)BH * ((N + kUnitQ - 1) / kUnitQ + m);
}

ExpertTcWs carve(void* ws, int BH, int N, int m, int topk) {
  char* p = static_cast<char*>(ws);
  auto take = [&](size_t bytes) {
    char* r = p;
    p += (bytes + 255) / 256 * 256;
    return r;
  };
  ExpertTcWs w;
  w.vt16 = reinterpret_cast<__half*>(take((size_t)BH * m * 64 * 2));
  w.unit_start = reinterpret_cast<int*>(take(((size_t)BH * m + 1) * 4));
  w.unit = reinterpret_cast<int4*>(take(max_units(BH, N, m) * 16));
  w.kg = reinterpret_cast<bf16*>(take((size_t)BH * m * topk * 128));
  w.vg = reinterpret_cast<bf16*>(take((size_t)BH * m * topk * 128));
  return w;
}

// -------------------------------------------------------------------------------------------
// gather: row j of expert (head, e) -> kg / vg[(head*m + e)*topk + j]; eight lanes per row,
// 16 bytes each, four rows per warp step
// -------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(kGatherThreads)
expert_gather_kernel(const bf16* __restrict__ k, const bf16* __restrict__ v,
                     const int32_t* __restrict__ topk_idx, long long rows, int N, int m, int topk,
                     bf16* __restrict__ kg, bf16* __restrict__ vg, int* status) {
  constexpr int UNR = 4;
  const int piece = threadIdx.x & 7;
  const long long lane_row = (long long)blockIdx.x * (kGatherThreads / 8) + (threadIdx.x >> 3);
  const long long stride = (long long)gridDim.x * (kGatherThreads / 8);
  for (long long r0 = lane_row; r0 < rows; r0 += stride * UNR) {
    uint4 kr[UNR], vr[UNR];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const long long r = r0 + u * stride;
      kr[u] = vr[u] = make_uint4(0u, 0u, 0u, 0u);
      if (r < rows) {
        const long long bh = r / ((long long)m * topk);
        const int j = topk_idx[r];
        if (j >= 0 && j < N) {
          const size_t src = ((size_t)bh * N + j) * 64 + piece * 8;
          kr[u] = *reinterpret_cast<const uint4*>(k + src);
          vr[u] = *reinterpret_cast<const uint4*>(v + src);
        } else if (piece == 0) {
          flag_error(status, kDevErrBadIndex);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const long long r = r0 + u * stride;
      if (r < rows) {
        *reinterpret_cast<uint4*>(kg + (size_t)r * 64 + piece * 8) = kr[u];
        *reinterpret_cast<uint4*>(vg + (size_t)r * 64 + piece * 8) = vr[u];
      }
    }
  }
}

// -------------------------------------------------------------------------------------------
// prep: unit table (units per (head, expert) = ceil(count / 256), exclusive scan,
// then one entry per unit) and v~ in fp16
// -------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(1024)
expert_prep_kernel(const int32_t* __restrict__ bucket_off, const float* __restrict__ v_tilde,
                   int BH, int N, int m, ExpertTcWs w, int* status) {
  __shared__ int red[33];
  const int total = BH * m;
  int carry = 0;
  for (int i0 = 0; i0 < total; i0 += 1024) {
    const int i = i0 + threadIdx.x;
    int units = 0, a = 0, cnt = 0;
    if (i < total) {
      const int bh = i / m, e = i % m;
      a = bucket_off[(size_t)bh * (m + 1) + e];
      const int b = bucket_off[(size_t)bh * (m + 1) + e + 1];
      if (a < 0 || b > N || b < a) flag_error(status, kDevErrBadBucket);
      else { cnt = b - a; units = (cnt + kUnitQ - 1) / kUnitQ; }
    }
    int tot;
    const int ex = block_excl_scan(units, red, &tot);
    if (i < total) {
      w.unit_start[i] = carry + ex;
      for (int j = 0; j < units; ++j)
        w.unit[carry + ex + j] = make_int4(i, a + j * kUnitQ, min(kUnitQ, cnt - j * kUnitQ), 0);
    }
    carry += tot;
    __syncthreads();
  }
  if (threadIdx.x == 0) w.unit_start[total] = carry;
  for (size_t t = threadIdx.x; t < (size_t)total * 64; t += 1024)
    w.vt16[t] = __float2half_rn(v_tilde[t]);
}

// -------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 1)
expert_tc_kernel(const __grid_constant__ CUtensorMap map_qg, const __grid_constant__ CUtensorMap map_kg,
                 const __grid_constant__ CUtensorMap map_vg, const __grid_constant__ CUtensorMap map_qt,
                 const __grid_constant__ CUtensorMap map_vt, const int32_t* __restrict__ bucket_qidx,
                 const int* __restrict__ unit_count, const int4* __restrict__ unit_tab, int BH,
                 int N, int m, int topk, bf16* __restrict__ out, int* status) {
  extern __shared__ unsigned char smem_raw[];
  ExpertSmem& s = *reinterpret_cast<ExpertSmem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int U = *unit_count;
  const int per = (U + gridDim.x - 1) / gridDim.x;          // contiguous units per CTA
  const int ubase = blockIdx.x * per;
  const int units = max(0, min(per, U - ubase));
  const int nsc = (m + BN - 1) / BN, nrc = (topk + BN - 1) / BN, nc = nsc + nrc;
  const int G = units * nc;
  const int null_row = BH * N;   // out of range: TMA fills zeros

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&s.kv_full[i], 1);
      mbar_init(&s.kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.q_full[i], 1);
      mbar_init(&s.q_empty[i], 1);
      mbar_init(&s.pv_done[i], 1);
    }
    for (int i = 0; i < kSBuf; ++i) {
      mbar_init(&s.s_full[i], 1);
      mbar_init(&s.p_full[i], 4);
    }
    mbar_init(&s.drain, 1);
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
  // tensor memory: three S buffers at 0 / 128 / 256 (P written over the first half of its S),
  // O of query tile t at 384 + 64*t.  Tile sequence j = 2*chunk + query tile, buffer j % 3.

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    bool ok = true;
    if (lane == 0) {
      prefetch_tmap(&map_qg);
      prefetch_tmap(&map_kg);
      prefetch_tmap(&map_vg);
      prefetch_tmap(&map_qt);
      prefetch_tmap(&map_vt);
    }
    int gi = 0;
    int4 nxt = units > 0 ? unit_tab[ubase] : make_int4(0, 0, 0, 0);
    for (int it = 0; it < units && ok; ++it) {
      const int4 cur = nxt;
      if (it + 1 < units) nxt = unit_tab[ubase + it + 1];
      const int idx = cur.x, bh = idx / m, qbase = cur.y, qcnt = cur.z;
      const int qb = it & 1;
      // ---- the unit's query rows (two tiles): lane l owns rows 8l .. 8l+7
      int rows[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int r = 8 * lane + j;
        rows[j] = null_row;
        if (r < qcnt) {
          const int qi = bucket_qidx[(size_t)bh * N + qbase + r];
          if (qi >= 0 && qi < N) rows[j] = bh * N + qi;
          else flag_error(status, kDevErrBadBucket);
        }
      }
      if (lane == 0 && !mbar_wait(&s.q_empty[qb], ((it >> 1) & 1) ^ 1)) ok = false;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      if (lane == 0) mbar_expect_tx(&s.q_full[qb], 2 * 128 * 128);
      __syncwarp();
      {
        const int r = 8 * lane;
        bf16* dst = &s.q[qb][r >> 7][(r & 127) * 64];
        tma_gather4(dst, &map_qg, &s.q_full[qb], 0, rows[0], rows[1], rows[2], rows[3]);
        tma_gather4(dst + 4 * 64, &map_qg, &s.q_full[qb], 0, rows[4], rows[5], rows[6], rows[7]);
      }
      // ---- the entries: the expert's gathered rows, then the shared blocks
      for (int c = 0; c < nc; ++c, ++gi) {
        const int st = gi % kStages;
        if (lane == 0) {
          if (!mbar_wait(&s.kv_empty[st], ((gi / kStages) & 1) ^ 1)) {
            ok = false;
          } else {
            mbar_expect_tx(&s.kv_full[st], 2 * BN * 128);
            if (c < nrc) {
              tma_load_3d(s.kb[st], &map_kg, &s.kv_full[st], 0, c * BN, idx);
              tma_load_3d(s.vb[st], &map_vg, &s.kv_full[st], 0, c * BN, idx);
            } else {
              tma_load_3d(s.kb[st], &map_qt, &s.kv_full[st], 0, (c - nrc) * BN, bh);
              tma_load_3d(s.vb[st], &map_vt, &s.kv_full[st], 0, (c - nrc) * BN, bh);
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
      }
    }
    if (!ok && lane == 0) flag_error(status, kDevErrTimeout);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id_s = idesc_f16(128, BN, false);
      const uint32_t id_pv_raw = idesc_f16(128, 64, true, false);
      const uint32_t id_pv_sh = idesc_f16(128, 64, true, true);
      const int T = 2 * G;
      bool ok = true;
      // S(j) = Q_tile . B(chunk)^T into buffer j % 3
      auto issue_s = [&](int j) -> bool {
        const int g = j >> 1, slot = j & 1;
        const int it = g / nc, c = g % nc, qb = it & 1, st = g % kStages;
        if (slot == 0) {
          if (c == 0 && !mbar_wait(&s.q_full[qb], (it >> 1) & 1)) return false;
          if (!mbar_wait(&s.kv_full[st], (g / kStages) & 1)) return false;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t da = smem_desc_sw128(smem_u32(s.q[qb][slot]) + kk * 32, 1024);
          const uint64_t db = smem_desc_sw128(smem_u32(s.kb[st]) + kk * 32, 1024);
          mma_ss(tbase + (j % kSBuf) * 128, da, db, id_s, kk > 0);
        }
        mma_commit(&s.s_full[j % kSBuf]);
        if (slot == 1 && c == nc - 1) mma_commit(&s.q_empty[qb]);
        return true;
      };
      for (int j = 0; j < kSBuf && j < T && ok; ++j) ok = issue_s(j);
      for (int j = 0; j < T && ok; ++j) {
        const int g = j >> 1, slot = j & 1, c = g % nc, st = g % kStages, b = j % kSBuf;
        if (!mbar_wait(&s.p_full[b], (j / kSBuf) & 1)) { ok = false; break; }
        tc_fence_after();
        const uint32_t id_pv = c < nrc ? id_pv_raw : id_pv_sh;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          const uint64_t dv = smem_desc_sw128(smem_u32(s.vb[st]) + kk * 2048, 1024);
          mma_ts(tbase + 384 + slot * 64, tbase + b * 128 + kk * 8, dv, id_pv, c > 0 || kk > 0);
        }
        mma_commit(&s.pv_done[slot]);
        if (slot == 1) mma_commit(&s.kv_empty[st]);
        // the buffer is rewritten only after this product has read P (in-order pipe)
        if (j + kSBuf < T) ok = issue_s(j + kSBuf);
      }
      if (!ok) flag_error(status, kDevErrTimeout);
      mma_commit(&s.drain);
      mbar_wait(&s.drain, 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int slot = (warp - 2) >> 2;
    const int quad = warp & 3;             // tensor-memory lanes this warp may access
    const int row = quad * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t tO = tbase + lane_off + 384 + slot * 64;
    const float cs = 0.18033688011112042f;   // log2(e) / sqrt(64)
    bool ok = true;
    int g = 0;
    for (int it = 0; it < units; ++it) {
      const int4 cur = unit_tab[ubase + it];
      const int bh = cur.x / m;
      const int qr = slot * 128 + row;
      int qi = -1;
      if (qr < cur.z) {
        qi = bucket_qidx[(size_t)bh * N + cur.y + qr];
        if (qi < 0 || qi >= N) qi = -1;
      }
      float mref = -INFINITY, lsum = 0.f;
      for (int c = 0; c < nc; ++c, ++g) {
        const int j = 2 * g + slot;
        const uint32_t tS = tbase + lane_off + (j % kSBuf) * 128;
        if (ok && !mbar_wait(&s.s_full[j % kSBuf], (j / kSBuf) & 1)) ok = false;
        tc_fence_after();
        const int nvalid = c < nrc ? min(BN, topk - c * BN) : min(BN, m - (c - nrc) * BN);
        const bool full = nvalid == BN;
        float tm = -INFINITY;
        if (ok) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float v[64];
            tmem_ld32(tS + h * 64, v);
            tmem_ld32(tS + h * 64 + 32, v + 32);
            tmem_ld_wait();
            if (!full) {
#pragma unroll
              for (int i = 0; i < 64; ++i) v[i] = (h * 64 + i < nvalid) ? v[i] : -INFINITY;
            }
#pragma unroll
            for (int i = 0; i < 64; i += 2) tm = max3(tm, v[i], v[i + 1]);
          }
        }
        const float xm = tm * cs;
        if (c > 0 && ok && !mbar_wait(&s.pv_done[slot], (g - 1) & 1)) ok = false;
        tc_fence_after();
        const bool need = (c == 0) || (xm > mref + kLazy);
        if (c > 0 && __any_sync(0xffffffffu, need)) {
          const float f = need ? ex2(mref - xm) : 1.f;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float o[32];
            tmem_ld32(tO + h * 32, o);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= f;
            tmem_st16(tO + h * 32, reinterpret_cast<uint32_t*>(o));
            tmem_st16(tO + h * 32 + 16, reinterpret_cast<uint32_t*>(o + 16));
          }
          tmem_st_wait();
        }
        if (need) {
          if (c > 0) lsum *= ex2(mref - xm);
          mref = xm;
        }
        const bool fp16 = c >= nrc;
        const float nm = -mref;
        float ls = 0.f;
        if (ok) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float v[64];
            tmem_ld32(tS + h * 64, v);
            tmem_ld32(tS + h * 64 + 32, v + 32);
            tmem_ld_wait();
            uint32_t pk[32];
#pragma unroll
            for (int i = 0; i < 64; i += 2) {
              float p0 = ex2(fmaf(v[i], cs, nm)), p1 = ex2(fmaf(v[i + 1], cs, nm));
              if (!full) {
                p0 = (h * 64 + i < nvalid) ? p0 : 0.f;
                p1 = (h * 64 + i + 1 < nvalid) ? p1 : 0.f;
              }
              ls += p0 + p1;
              pk[i / 2] = pack_pair(p0, p1, fp16);
            }
            // P columns h*32 .. h*32+31 lie below the S columns already read
            tmem_st16(tS + h * 32, pk);
            tmem_st16(tS + h * 32 + 16, pk + 16);
          }
        }
        lsum += ls;
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.p_full[j % kSBuf]);
      }
      // ---- output row: O / l
      if (ok && !mbar_wait(&s.pv_done[slot], (g - 1) & 1)) ok = false;
      tc_fence_after();
      float o[64];
      tmem_ld32(tO, o);
      tmem_ld32(tO + 32, o + 32);
      tmem_ld_wait();
      tc_fence_before();
      if (ok && qi >= 0) {
        const float inv = 1.f / lsum;
        uint4* dst = reinterpret_cast<uint4*>(out + ((size_t)bh * N + qi) * 64);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          uint4 w;
          w.x = pack_pair(o[8 * i] * inv, o[8 * i + 1] * inv, false);
          w.y = pack_pair(o[8 * i + 2] * inv, o[8 * i + 3] * inv, false);
          w.z = pack_pair(o[8 * i + 4] * inv, o[8 * i + 5] * inv, false);
          w.w = pack_pair(o[8 * i + 6] * inv, o[8 * i + 7] * inv, false);
          dst[i] = w;
        }
      }
    }
    if (!ok) flag_error(status, kDevErrTimeout);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, 512);
}

}  // namespace

bool expert_tc_supported(int d, int m, int topk) { return d == 64 && m >= 1 && topk >= 1; }

size_t expert_tc_ws_bytes(int BH, int N, int m, int topk) {
  auto r = [](size_t b) { return (b + 255) / 256 * 256; };
  return r((size_t)BH * m * 64 * 2) + r(((size_t)BH * m + 1) * 4) + r(max_units(BH, N, m) * 16) +
         2 * r((size_t)BH * m * topk * 128);
}

cudaError_t launch_expert_tc(const bf16* q, const bf16* k, const bf16* v, const bf16* q_tilde,
                             const float* v_tilde, const int32_t* topk_idx,
                             const int32_t* bucket_off, const int32_t* bucket_qidx, int BH, int N,
                             int m, int topk, int num_sms, void* ws, bf16* out, int* status,
                             cudaStream_t st) {
  const ExpertTcWs w = carve(ws, BH, N, m, topk);
  const long long rows = (long long)BH * m * topk;
  const long long gblocks = std::min<long long>((rows + kGatherThreads / 8 - 1) / (kGatherThreads / 8),
                                                (long long)std::max(num_sms, 1) * 8);
  expert_gather_kernel<<<(unsigned)gblocks, kGatherThreads, 0, st>>>(k, v, topk_idx, rows, N, m,
                                                                      topk, w.kg, w.vg, status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  expert_prep_kernel<<<1, 1024, 0, st>>>(bucket_off, v_tilde, BH, N, m, w, status);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  CUtensorMap mqg, mkg, mvg, mqt, mvt;
  if (!make_tmap_gather64(&mqg, q, (uint64_t)BH * N) ||
      !make_tmap_rows64(&mkg, w.kg, (uint64_t)topk, (uint64_t)BH * m, BN) ||
      !make_tmap_rows64(&mvg, w.vg, (uint64_t)topk, (uint64_t)BH * m, BN) ||
      !make_tmap_rows64(&mqt, q_tilde, (uint64_t)m, (uint64_t)BH, BN) ||
      !make_tmap_rows64(&mvt, w.vt16, (uint64_t)m, (uint64_t)BH, BN, true))
    return cudaErrorInvalidValue;
  const size_t smem = sizeof(ExpertSmem) + 1024;
  e = cudaFuncSetAttribute(expert_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  expert_tc_kernel<<<(unsigned)std::max(num_sms, 1), kThreads, smem, st>>>(
      mqg, mkg, mvg, mqt, mvt, bucket_qidx, w.unit_start + (size_t)BH * m, w.unit, BH, N, m, topk,
      out, status);
  return cudaGetLastError();
}

}  // namespace mita
