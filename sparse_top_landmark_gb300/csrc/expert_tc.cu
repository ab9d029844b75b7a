// Step 6 on the tensor cores (bf16, d = 64): for every query, one joint
// softmax over the m shared pairs (q~_i, v~_i) and the k raw pairs of its
// routed expert, computed expert by expert.
//
// MiTA tutorial (iwxt.cn), ch. 4 steps 5-6 (paper eq. 11-12): the m + s*k
// logits, all scaled by 1/sqrt(d), share one softmax over [v~; V(e)].  The
// bit.fan article: queries are grouped by expert and an online softmax runs
// over the concatenated entries.
//
// Work unit = (head, expert, two tiles of 128 of its queries).  Persistent
// CTAs walk the units (table built by expert_prep_kernel):
//   warp 0      TMA: the unit's query rows (tile::gather4 of scattered rows),
//               then the entries in chunks of 128: q~ / v~ blocks (tiled
//               loads) and the expert's K / V rows (gather4); 3-stage ring
//               shared by both query tiles;
//   warp 1      MMA: S = Q . B^T per tile into tensor memory, then
//               O += P . V (P read from tensor memory; the shared branch runs
//               as an fp16 x fp16 product, v~ kept in fp16, the raw branch as
//               bf16 x bf16);
//   warps 4-7 / 8-11   online softmax of query tile 0 / 1 (one query row per
//               thread, lazy O rescaling), then O / l to the output rows.
#include <algorithm>

#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"

namespace mita {
namespace {
using namespace sm100;

constexpr int BN = 128;          // entries per chunk
constexpr int kStages = 3;
constexpr int kThreads = 384;
constexpr int kUnitQ = 256;      // queries per work unit (two MMA tiles)
constexpr float kLazy = 8.0f;

struct alignas(1024) ExpertSmem {
  bf16 q[2][2][128 * 64];          // [unit buffer][query tile]
  bf16 kb[kStages][BN * 64];       // q~ block or the expert's K rows
  bf16 vb[kStages][BN * 64];       // v~ block (fp16) or the expert's V rows
  uint64_t kv_full[kStages], kv_empty[kStages];
  uint64_t q_full[2], q_empty[2];
  uint64_t s_full[2], p_full[2], pv_done[2];
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

// unit u -> flat (head, expert) index: last i with start[i] <= u
__device__ __forceinline__ int find_unit(const int* start, int n, int u) {
  int lo = 0, hi = n;   // start[lo] <= u < start[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (start[mid] <= u) lo = mid; else hi = mid;
  }
  return lo;
}

// -------------------------------------------------------------------------------------------
// prep: unit table (units per (head, expert) = ceil(count / 256), exclusive scan)
// and v~ in fp16
// -------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(1024)
expert_prep_kernel(const int32_t* __restrict__ bucket_off, const float* __restrict__ v_tilde,
                   int BH, int N, int m, int* __restrict__ unit_start, __half* __restrict__ vt16,
                   int* status) {
  __shared__ int red[33];
  const int total = BH * m;
  int carry = 0;
  for (int i0 = 0; i0 < total; i0 += 1024) {
    const int i = i0 + threadIdx.x;
    int units = 0;
    if (i < total) {
      const int bh = i / m, e = i % m;
      const int a = bucket_off[(size_t)bh * (m + 1) + e], b = bucket_off[(size_t)bh * (m + 1) + e + 1];
      if (a < 0 || b > N || b < a) flag_error(status, kDevErrBadBucket);
      else units = (b - a + kUnitQ - 1) / kUnitQ;
    }
    int tot;
    const int ex = block_excl_scan(units, red, &tot);
    if (i < total) unit_start[i] = carry + ex;
    carry += tot;
    __syncthreads();
  }
  if (threadIdx.x == 0) unit_start[total] = carry;
  for (size_t t = threadIdx.x; t < (size_t)total * 64; t += 1024) vt16[t] = __float2half_rn(v_tilde[t]);
}

// -------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 1)
expert_tc_kernel(const __grid_constant__ CUtensorMap map_qg, const __grid_constant__ CUtensorMap map_kg,
                 const __grid_constant__ CUtensorMap map_vg, const __grid_constant__ CUtensorMap map_qt,
                 const __grid_constant__ CUtensorMap map_vt, const int32_t* __restrict__ topk_idx,
                 const int32_t* __restrict__ bucket_off, const int32_t* __restrict__ bucket_qidx,
                 const int* __restrict__ unit_start, int BH, int N, int m, int topk,
                 bf16* __restrict__ out, int* status) {
  extern __shared__ unsigned char smem_raw[];
  ExpertSmem& s = *reinterpret_cast<ExpertSmem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nidx = BH * m;
  const int U = unit_start[nidx];
  const int units = (blockIdx.x < U) ? (U - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
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
      mbar_init(&s.s_full[i], 1);
      mbar_init(&s.p_full[i], 4);
      mbar_init(&s.pv_done[i], 1);
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
  // tensor memory: S_slot at 128*slot, P_slot at 256 + 64*slot, O_slot at 384 + 64*slot

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
    for (int it = 0; it < units && ok; ++it) {
      const int u = blockIdx.x + it * gridDim.x;
      const int idx = find_unit(unit_start, nidx, u);
      const int bh = idx / m, e = idx % m;
      const int off0 = bucket_off[(size_t)bh * (m + 1) + e];
      const int off1 = bucket_off[(size_t)bh * (m + 1) + e + 1];
      const int qbase = off0 + (u - unit_start[idx]) * kUnitQ;
      const int qcnt = min(kUnitQ, off1 - qbase);
      const int qb = it & 1;
      // ---- the unit's query rows (two tiles)
      if (lane == 0 && !mbar_wait(&s.q_empty[qb], ((it >> 1) & 1) ^ 1)) ok = false;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      if (lane == 0) mbar_expect_tx(&s.q_full[qb], 2 * 128 * 128);
      for (int r0 = 0; r0 < kUnitQ; r0 += 32) {
        int row = null_row;
        if (r0 + lane < qcnt) {
          const int qi = bucket_qidx[(size_t)bh * N + qbase + r0 + lane];
          if (qi >= 0 && qi < N) row = bh * N + qi;
          else flag_error(status, kDevErrBadBucket);
        }
#pragma unroll
        for (int g4 = 0; g4 < 8; ++g4) {
          const int a = __shfl_sync(0xffffffffu, row, 4 * g4), b = __shfl_sync(0xffffffffu, row, 4 * g4 + 1);
          const int c = __shfl_sync(0xffffffffu, row, 4 * g4 + 2), d = __shfl_sync(0xffffffffu, row, 4 * g4 + 3);
          const int r = r0 + 4 * g4;
          if (lane == 0) tma_gather4(&s.q[qb][r >> 7][(r & 127) * 64], &map_qg, &s.q_full[qb], 0, a, b, c, d);
        }
      }
      // ---- the entries: shared blocks, then the expert's raw rows
      const int32_t* eidx = topk_idx + (size_t)idx * topk;
      for (int c = 0; c < nc; ++c, ++gi) {
        const int st = gi % kStages;
        if (lane == 0 && !mbar_wait(&s.kv_empty[st], ((gi / kStages) & 1) ^ 1)) ok = false;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        if (lane == 0) mbar_expect_tx(&s.kv_full[st], 2 * BN * 128);
        if (c < nsc) {
          if (lane == 0) {
            tma_load_3d(s.kb[st], &map_qt, &s.kv_full[st], 0, c * BN, bh);
            tma_load_3d(s.vb[st], &map_vt, &s.kv_full[st], 0, c * BN, bh);
          }
        } else {
          const int cr = (c - nsc) * BN;
          for (int r0 = 0; r0 < BN; r0 += 32) {
            int row = null_row;
            if (cr + r0 + lane < topk) {
              const int j = eidx[cr + r0 + lane];
              if (j >= 0 && j < N) row = bh * N + j;
              else flag_error(status, kDevErrBadIndex);
            }
#pragma unroll
            for (int g4 = 0; g4 < 8; ++g4) {
              const int a = __shfl_sync(0xffffffffu, row, 4 * g4), b = __shfl_sync(0xffffffffu, row, 4 * g4 + 1);
              const int cc = __shfl_sync(0xffffffffu, row, 4 * g4 + 2), d = __shfl_sync(0xffffffffu, row, 4 * g4 + 3);
              const int r = r0 + 4 * g4;
              if (lane == 0) {
                tma_gather4(&s.kb[st][r * 64], &map_kg, &s.kv_full[st], 0, a, b, cc, d);
                tma_gather4(&s.vb[st][r * 64], &map_vg, &s.kv_full[st], 0, a, b, cc, d);
              }
            }
          }
        }
      }
    }
    if (!ok && lane == 0) flag_error(status, kDevErrTimeout);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id_s = idesc_f16(128, BN, false);
      const uint32_t id_pv_raw = idesc_f16(128, 64, true, false);
      const uint32_t id_pv_sh = idesc_f16(128, 64, true, true);
      bool ok = true;
      auto issue_s = [&](int g, int slot) -> bool {
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
          mma_ss(tbase + slot * 128, da, db, id_s, kk > 0);
        }
        mma_commit(&s.s_full[slot]);
        if (slot == 1 && c == nc - 1) mma_commit(&s.q_empty[qb]);
        return true;
      };
      if (G > 0) ok = issue_s(0, 0) && issue_s(0, 1);
      for (int g = 0; g < G && ok; ++g) {
        const int c = g % nc, st = g % kStages;
        const uint32_t id_pv = c < nsc ? id_pv_sh : id_pv_raw;
        for (int slot = 0; slot < 2 && ok; ++slot) {
          if (!mbar_wait(&s.p_full[slot], g & 1)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            const uint64_t dv = smem_desc_sw128(smem_u32(s.vb[st]) + kk * 2048, 1024);
            mma_ts(tbase + 384 + slot * 64, tbase + 256 + slot * 64 + kk * 8, dv, id_pv,
                   c > 0 || kk > 0);
          }
          mma_commit(&s.pv_done[slot]);
          if (slot == 1) mma_commit(&s.kv_empty[st]);
          if (g + 1 < G) ok = issue_s(g + 1, slot);
        }
      }
      if (!ok) flag_error(status, kDevErrTimeout);
      mma_commit(&s.drain);
      mbar_wait(&s.drain, 0);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int slot = (warp - 4) >> 2;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t tS = tbase + lane_off + slot * 128;
    const uint32_t tP = tbase + lane_off + 256 + slot * 64;
    const uint32_t tO = tbase + lane_off + 384 + slot * 64;
    const float cs = 0.18033688011112042f;   // log2(e) / sqrt(64)
    bool ok = true;
    int g = 0;
    for (int it = 0; it < units; ++it) {
      const int u = blockIdx.x + it * gridDim.x;
      const int idx = find_unit(unit_start, nidx, u);
      const int bh = idx / m, e = idx % m;
      const int off0 = bucket_off[(size_t)bh * (m + 1) + e];
      const int off1 = bucket_off[(size_t)bh * (m + 1) + e + 1];
      const int qbase = off0 + (u - unit_start[idx]) * kUnitQ;
      const int qr = slot * 128 + row;
      int qi = -1;
      if (qbase + qr < off1) {
        qi = bucket_qidx[(size_t)bh * N + qbase + qr];
        if (qi < 0 || qi >= N) qi = -1;
      }
      float mref = -INFINITY, lsum = 0.f;
      for (int c = 0; c < nc; ++c, ++g) {
        if (ok && !mbar_wait(&s.s_full[slot], g & 1)) ok = false;
        tc_fence_after();
        const int nvalid = c < nsc ? min(BN, m - c * BN) : min(BN, topk - (c - nsc) * BN);
        const bool full = nvalid == BN;
        float tm = -INFINITY;
        if (ok) {
#pragma unroll
          for (int cc = 0; cc < BN / 32; ++cc) {
            float v[32];
            tmem_ld32(tS + cc * 32, v);
            tmem_ld_wait();
            if (!full) {
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = (cc * 32 + i < nvalid) ? v[i] : -INFINITY;
            }
#pragma unroll
            for (int i = 0; i < 32; i += 2) tm = max3(tm, v[i], v[i + 1]);
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
        const bool fp16 = c < nsc;
        const float nm = -mref;
        float ls = 0.f;
#pragma unroll
        for (int cc = 0; cc < BN / 32; ++cc) {
          float v[32];
          tmem_ld32(tS + cc * 32, v);
          tmem_ld_wait();
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            float p0 = ex2(fmaf(v[i], cs, nm)), p1 = ex2(fmaf(v[i + 1], cs, nm));
            if (!full) {
              p0 = (cc * 32 + i < nvalid) ? p0 : 0.f;
              p1 = (cc * 32 + i + 1 < nvalid) ? p1 : 0.f;
            }
            ls += p0 + p1;
            pk[i / 2] = pack_pair(p0, p1, fp16);
          }
          tmem_st16(tP + cc * 16, pk);
        }
        lsum += ls;
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.p_full[slot]);
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

size_t expert_tc_ws_bytes(int BH, int m) {
  return ((size_t)BH * m * 64 * 2 + 255) / 256 * 256 + ((size_t)BH * m + 1) * 4;
}

cudaError_t launch_expert_tc(const bf16* q, const bf16* k, const bf16* v, const bf16* q_tilde,
                             const float* v_tilde, const int32_t* topk_idx,
                             const int32_t* bucket_off, const int32_t* bucket_qidx, int BH, int N,
                             int m, int topk, int num_sms, void* ws, bf16* out, int* status,
                             cudaStream_t st) {
  __half* vt16 = static_cast<__half*>(ws);
  int* unit_start = reinterpret_cast<int*>(static_cast<char*>(ws) +
                                           ((size_t)BH * m * 64 * 2 + 255) / 256 * 256);
  expert_prep_kernel<<<1, 1024, 0, st>>>(bucket_off, v_tilde, BH, N, m, unit_start, vt16, status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  CUtensorMap mqg, mkg, mvg, mqt, mvt;
  const uint64_t rows = (uint64_t)BH * N;
  if (!make_tmap_gather64(&mqg, q, rows) || !make_tmap_gather64(&mkg, k, rows) ||
      !make_tmap_gather64(&mvg, v, rows) ||
      !make_tmap_rows64(&mqt, q_tilde, (uint64_t)m, (uint64_t)BH, BN) ||
      !make_tmap_rows64(&mvt, vt16, (uint64_t)m, (uint64_t)BH, BN, true))
    return cudaErrorInvalidValue;
  const size_t smem = sizeof(ExpertSmem) + 1024;
  e = cudaFuncSetAttribute(expert_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  expert_tc_kernel<<<(unsigned)std::max(num_sms, 1), kThreads, smem, st>>>(
      mqg, mkg, mvg, mqt, mvt, topk_idx, bucket_off, bucket_qidx, unit_start, BH, N, m, topk, out,
      status);
  return cudaGetLastError();
}

}  // namespace mita
