// Step 6 on the tensor cores (bf16, d = 64): for every query, one joint
// softmax over the m shared pairs (q~_i, v~_i) and the k raw pairs of its
// routed expert, computed expert by expert.
//
// MiTA tutorial (iwxt.cn), ch. 4 steps 5-6 (paper eq. 11-12): the m + s*k
// logits, all scaled by 1/sqrt(d), share one softmax over [v~; V(e)] (on
// request the shared logits take 1/d, the official code's temperature read in
// tutorial ch. 8 caveat 3).  The
// bit.fan article: queries are grouped by expert and an online softmax runs
// over the concatenated entries; each expert's k KV rows are gathered once.
//
// Two launches (grouped form):
//   expert_gather_kernel  the k K / V rows of every (head, expert), copied once
//                         into contiguous [head*m + expert][k][64] blocks; one
//                         more CTA builds the work-unit table (unit = (head,
//                         expert, up to 256 of its queries)); v~ to bf16;
//   expert_tc_kernel      persistent CTAs, each over a contiguous run of units
//                         (units of one expert follow each other, so its
//                         gathered rows are re-read from L2):
//     warps 0, 3 TMA: the unit's query rows (tile::gather4 of scattered rows;
//                warp 0 tile 0, warp 3 tile 1); warp 0 then the entries in
//                chunks of 128 -- the expert's gathered
//                K / V block first, then the q~ / v~ blocks -- as tiled loads
//                into a 4-stage ring shared by the two query tiles;
//     warps 1-2  MMA, one issuing thread per query tile (one thread issues a
//                tcgen05.mma only every ~130 cycles, so the two tiles get an
//                issuer each): S = Q . B^T into the tile's S columns, and as
//                soon as the softmax has copied S out, the next chunk's S;
//                then O += P . V with P read from tensor memory (bf16 x bf16
//                for both kinds of chunk: v~ is kept in bf16, fp32's range);
//     warps 4-7 / 8-11   online softmax of query tile 0 / 1 (one query row per
//                thread, lazy O rescaling; half of a chunk's exponentials are
//                computed before waiting for the previous P . V), then O / l to
//                the output rows.  One code path for every chunk: a second,
//                fp16 copy of the unrolled exponential loop (for an fp16 v~)
//                cost ~8 % of the forward's time, measured.
// Two more forms of expert_tc_kernel (template flags):
//   carried  the shared branch arrives as a partial (log-sum-exp and output
//            over the m shared pairs, from the route stage); only raw chunks
//            run, and the partial joins each row at write-out by the
//            branch-merge identity (Z1 o1 + Z2 o2) / (Z1 + Z2);
//   masked   short sequences: a unit is a tile of a head's consecutive
//            queries and its raw entries are all N keys of the head, each
//            masked per query to its routed expert's top-k set (membership bit
//            masks from expert_mask_kernel) -- fewer chunks than grouping
//            when N is small;
//   partial  top-s routing (s > 1; tutorial ch. 4 step 4, eq. 10-12): the
//            buckets hold N * s (query, expert) entries; each entry runs the
//            raw chunks of its expert and leaves its partial (natural
//            log-sum-exp and O / l in fp32, with its bucket position) in one of
//            its query's s slots; expert_merge_kernel joins the shared partial
//            and the s raw ones by the branch-merge identity.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"

namespace mita {
namespace {
using namespace sm100;

constexpr int BN = 128;          // entries per chunk
constexpr int kStages = 4;
constexpr int kThreads = 384;   // producer, two MMA issuers, second gatherer, 8 softmax warps
constexpr int kUnitQ = 256;      // queries per work unit (two MMA tiles)
constexpr float kLazy = 8.0f;
constexpr int kGatherThreads = 256;

struct alignas(1024) ExpertSmem {
  bf16 q[2][2][128 * 64];          // [unit buffer][query tile]
  bf16 kb[kStages][BN * 64];       // q~ block or the expert's K rows
  bf16 vb[kStages][BN * 64];       // v~ block (bf16) or the expert's V rows
  uint64_t kv_full[kStages], kv_empty[kStages];
  uint64_t q_full[2], q_empty[2];
  uint64_t s_full[2], s_free[2], p_full[2], pv_done[2];
  uint64_t drain[2];               // one per MMA issuer
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
// two floats to a bf16 pair (a in the low half), round to nearest even
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %2, %1;" : "=r"(r) : "f"(a), "f"(b));
  return r;
}

struct ExpertTcWs {
  bf16* vtb;         // [BH*m][64]: v~ in bf16
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
  w.vtb = reinterpret_cast<bf16*>(take((size_t)BH * m * 64 * 2));
  w.unit_start = reinterpret_cast<int*>(take(((size_t)BH * m + 1) * 4));
  w.unit = reinterpret_cast<int4*>(take(max_units(BH, N, m) * 16));
  w.kg = reinterpret_cast<bf16*>(take((size_t)BH * m * topk * 128));
  w.vg = reinterpret_cast<bf16*>(take((size_t)BH * m * topk * 128));
  return w;
}

// -------------------------------------------------------------------------------------------
// Preparation, one launch: the last CTA builds the work-unit table (unit = (head*m + e, first
// bucket slot, count <= 256); unit_start[head*m + e] = the expert's first unit, then one
// entry per unit); every CTA converts a slice of v~ to bf16, and the other CTAs gather the
// experts' rows: row j of expert (head, e) -> kg / vg[(head*m + e)*topk + j], eight lanes per
// row, 16 bytes each, four rows per warp step.
// -------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(kGatherThreads)
expert_gather_kernel(const bf16* __restrict__ k, const bf16* __restrict__ v,
                     const int32_t* __restrict__ topk_idx, long long rows, int N, int m, int topk,
                     const int32_t* __restrict__ bucket_off, const float* __restrict__ v_tilde,
                     int BH, ExpertTcWs w, int* status, int nent) {
  griddep_wait();
  // v~ in bf16, four values per thread step (not needed, and possibly absent, when the
  // kernel runs no shared chunks)
  if (v_tilde != nullptr) {
    const long long n4 = (long long)BH * m * 16;
    for (long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x; t < n4;
         t += (long long)gridDim.x * blockDim.x) {
      const float4 x = reinterpret_cast<const float4*>(v_tilde)[t];
      uint2 o;
      o.x = pack_bf16(x.x, x.y);
      o.y = pack_bf16(x.z, x.w);
      reinterpret_cast<uint2*>(w.vtb)[t] = o;
    }
  }
  if (blockIdx.x == gridDim.x - 1) {
    // the unit table: an exclusive scan of the experts' unit counts
    __shared__ int red[kGatherThreads / 32 + 1];
    const int total = BH * m;
    int carry = 0;
    for (int i0 = 0; i0 < total; i0 += kGatherThreads) {
      const int i = i0 + threadIdx.x;
      int units = 0, a = 0, cnt = 0;
      if (i < total) {
        const int bh = i / m, e = i % m;
        a = bucket_off[(size_t)bh * (m + 1) + e];
        const int b = bucket_off[(size_t)bh * (m + 1) + e + 1];
        if (a < 0 || b > nent || b < a) flag_error(status, kDevErrBadBucket);
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
    return;
  }
  constexpr int UNR = 4;
  const int piece = threadIdx.x & 7;
  const long long lane_row = (long long)blockIdx.x * (kGatherThreads / 8) + (threadIdx.x >> 3);
  const long long stride = (long long)(gridDim.x - 1) * (kGatherThreads / 8);
  // the key indices of the next step are loaded while this step's rows are in flight
  int jn[UNR];
#pragma unroll
  for (int u = 0; u < UNR; ++u) {
    const long long r = lane_row + u * stride;
    jn[u] = r < rows ? topk_idx[r] : 0;
  }
  for (long long r0 = lane_row; r0 < rows; r0 += stride * UNR) {
    uint4 kr[UNR], vr[UNR];
    int jc[UNR];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      jc[u] = jn[u];
      const long long rn = r0 + stride * UNR + u * stride;
      jn[u] = rn < rows ? topk_idx[rn] : 0;
    }
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const long long r = r0 + u * stride;
      kr[u] = vr[u] = make_uint4(0u, 0u, 0u, 0u);
      if (r < rows) {
        const long long bh = r / ((long long)m * topk);
        const int j = jc[u];
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
        *reinterpret_cast<uint4*>(w.kg + (size_t)r * 64 + piece * 8) = kr[u];
        *reinterpret_cast<uint4*>(w.vg + (size_t)r * 64 + piece * 8) = vr[u];
      }
    }
  }
}

// -------------------------------------------------------------------------------------------
// kMasked: the short-sequence form -- units are tiles of a head's consecutive queries, the
// raw chunks are all of the head's keys in place (K / V maps over [BH, N, 64]), and each
// query keeps only the keys of its routed expert's top-k set (bit mask kmask[bh][e][words],
// the expert from qroute), so one softmax still spans the m shared pairs and exactly the k
// raw pairs of eq. 11-12.
template <bool kCarried, bool kMasked, bool kPartial = false>
__global__ void __launch_bounds__(kThreads, 1)
expert_tc_kernel(const __grid_constant__ CUtensorMap map_qg, const __grid_constant__ CUtensorMap map_kg,
                 const __grid_constant__ CUtensorMap map_vg, const __grid_constant__ CUtensorMap map_qt,
                 const __grid_constant__ CUtensorMap map_vt, const int32_t* __restrict__ bucket_qidx,
                 const int* __restrict__ unit_count, const int4* __restrict__ unit_tab, int BH,
                 int N, int m, int topk, float cs_shared, int use_shared,
                 const float* __restrict__ sh_lse, const void* __restrict__ sh_o, int o_bf16,
                 const uint32_t* __restrict__ kmask, int mwords, const int32_t* __restrict__ qroute,
                 bf16* __restrict__ out, int* status, int nent, int nroutes, ExpertPartials part) {
  griddep_wait();
  extern __shared__ unsigned char smem_raw[];
  ExpertSmem& s = *reinterpret_cast<ExpertSmem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int U = *unit_count;
  const int per = (U + gridDim.x - 1) / gridDim.x;          // contiguous units per CTA
  const int ubase = blockIdx.x * per;
  const int units = max(0, min(per, U - ubase));
  // shared chunks (none for the routing-only ablation and for dense attention)
  const int nsc = use_shared ? (m + BN - 1) / BN : 0;
  const int nrc = (topk + BN - 1) / BN, nc = nsc + nrc;
  const int G = units * nc;
  const int null_row = BH * N;   // out of range: TMA fills zeros

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&s.kv_full[i], 1);
      mbar_init(&s.kv_empty[i], 2);     // both tiles' P . V
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.q_full[i], 2);       // the two gathering warps, one tile each
      mbar_init(&s.q_empty[i], 2);      // both tiles' last S
      mbar_init(&s.s_full[i], 1);
      mbar_init(&s.s_free[i], 4);
      mbar_init(&s.p_full[i], 4);
      mbar_init(&s.pv_done[i], 1);
    }
    mbar_init(&s.drain[0], 1);
    mbar_init(&s.drain[1], 1);
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
  // tensor memory, query tile t at 256*t: S (128 columns), P (64, bf16 / fp16 pairs), O (64)

  // registers: the launch grants 384 x 168; warps 0-3 keep 40 each, the two softmax
  // warpgroups take 232 each (128*40 + 2*128*232 = 384*168), via setmaxnreg in each role

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 40;\n" ::: "memory");
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
        // ---- query tile 0 of the unit (warp 3 gathers tile 1): lane l owns rows 4l .. 4l+3
        int rows[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int r = 4 * lane + j;
          rows[j] = null_row;
          if (r < qcnt) {
            const int qi = bucket_qidx[(size_t)bh * nent + qbase + r];
            if (qi >= 0 && qi < N) rows[j] = bh * N + qi;
            else flag_error(status, kDevErrBadBucket);
          }
        }
        if (!mbar_wait_warp(&s.q_empty[qb], ((it >> 1) & 1) ^ 1)) { ok = false; break; }
        if (lane == 0) mbar_expect_tx(&s.q_full[qb], 128 * 128);
        __syncwarp();
        tma_gather4(&s.q[qb][0][4 * lane * 64], &map_qg, &s.q_full[qb], 0, rows[0], rows[1], rows[2],
                    rows[3]);
        // ---- the entries: the expert's gathered rows, then the shared blocks
        for (int c = 0; c < nc; ++c, ++gi) {
          const int st = gi % kStages;
          if (!mbar_wait_warp(&s.kv_empty[st], ((gi / kStages) & 1) ^ 1)) { ok = false; break; }
          if (elect_one()) {
            mbar_expect_tx(&s.kv_full[st], 2 * BN * 128);
            if (c < nrc) {
              const int rawb = kMasked ? bh : idx;   // the head's keys, or the expert's block
              tma_load_3d(s.kb[st], &map_kg, &s.kv_full[st], 0, c * BN, rawb);
              tma_load_3d(s.vb[st], &map_vg, &s.kv_full[st], 0, c * BN, rawb);
            } else {
              tma_load_3d(s.kb[st], &map_qt, &s.kv_full[st], 0, (c - nrc) * BN, bh);
              tma_load_3d(s.vb[st], &map_vt, &s.kv_full[st], 0, (c - nrc) * BN, bh);
            }
          }
          __syncwarp();
        }
      }
      if (!ok && lane == 0) flag_error(status, kDevErrTimeout);
    } else if (warp == 1 || warp == 2) {
      // ---------------------------------------------------------- MMA issuer of one tile
      // the whole warp walks the schedule (waits without loops on the fast path);
      // one elected lane issues each batch of MMAs and its commits
      const int slot = warp - 1;
      const uint32_t id_s = idesc_f16(128, BN, false);
      const uint32_t id_pv = idesc_f16(128, 64, true);
      const uint32_t tS = tbase + slot * 256, tP = tS + 128, tO = tS + 192;
      bool ok = true;
      // S(g) = Q_slot . B(g)^T
      auto issue_s = [&](int g) -> bool {
        const int it = g / nc, c = g % nc, qb = it & 1, st = g % kStages;
        if (c == 0 && !mbar_wait_warp(&s.q_full[qb], (it >> 1) & 1)) return false;
        if (!mbar_wait_warp(&s.kv_full[st], (g / kStages) & 1)) return false;
        tc_fence_after();
        const uint32_t qa = smem_u32(s.q[qb][slot]), kb = smem_u32(s.kb[st]);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ss(tS, smem_desc_sw128(qa + kk * 32, 1024), smem_desc_sw128(kb + kk * 32, 1024),
                   id_s, kk > 0);
          mma_commit(&s.s_full[slot]);
          if (c == nc - 1) mma_commit(&s.q_empty[qb]);
        }
        __syncwarp();
        return true;
      };
      if (G > 0) ok = issue_s(0);
      for (int g = 0; g < G && ok; ++g) {
        const int c = g % nc, st = g % kStages;
        if (g + 1 < G) {
          if (!mbar_wait_warp(&s.s_free[slot], g & 1)) { ok = false; break; }
          if (!issue_s(g + 1)) { ok = false; break; }
        }
        if (!mbar_wait_warp(&s.p_full[slot], g & 1)) { ok = false; break; }
        tc_fence_after();
        const uint32_t vb = smem_u32(s.vb[st]);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            mma_ts(tO, tP + kk * 8, smem_desc_sw128(vb + kk * 2048, 1024), id_pv, c > 0 || kk > 0);
          mma_commit(&s.pv_done[slot]);
          mma_commit(&s.kv_empty[st]);
        }
        __syncwarp();
      }
      if (elect_one()) mma_commit(&s.drain[slot]);
      __syncwarp();
      if (!mbar_wait_warp(&s.drain[slot], 0)) ok = false;
      if (!ok && lane == 0) flag_error(status, kDevErrTimeout);
    } else {
      // ------------------------------------------------------------ query tile 1
      // of every unit, gathered alongside the producer's tile 0: one warp issues a
      // four-row TMA gather only every ~130 cycles, so two warps share the 64 per unit
      bool ok = true;
      for (int it = 0; it < units && ok; ++it) {
        const int4 cur = unit_tab[ubase + it];
        const int bh = cur.x / m, qbase = cur.y, qcnt = cur.z, qb = it & 1;
        int rows[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int r = 128 + 4 * lane + j;
          rows[j] = null_row;
          if (r < qcnt) {
            const int qi = bucket_qidx[(size_t)bh * nent + qbase + r];
            if (qi >= 0 && qi < N) rows[j] = bh * N + qi;
            else flag_error(status, kDevErrBadBucket);
          }
        }
        if (!mbar_wait_warp(&s.q_empty[qb], ((it >> 1) & 1) ^ 1)) { ok = false; break; }
        if (lane == 0) mbar_expect_tx(&s.q_full[qb], 128 * 128);
        __syncwarp();
        tma_gather4(&s.q[qb][1][4 * lane * 64], &map_qg, &s.q_full[qb], 0, rows[0], rows[1],
                    rows[2], rows[3]);
      }
      if (!ok && lane == 0) flag_error(status, kDevErrTimeout);
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 232;\n" ::: "memory");
    // ------------------------------------------------------------ softmax
    const int slot = (warp - 4) >> 2;
    const int quad = warp & 3;             // tensor-memory lanes this warp may access
    const int row = quad * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t tS = tbase + lane_off + slot * 256, tP = tS + 128, tO = tS + 192;
    const float cs = 0.18033688011112042f;   // log2(e) / sqrt(64)
    bool ok = true;
    const int qr = slot * 128 + row;
    // query id of this thread's row in unit u (-1: padding row)
    auto row_query = [&](const int4& u) -> int {
      if (qr >= u.z) return -1;
      const int qi = bucket_qidx[(size_t)(u.x / m) * nent + u.y + qr];
      return (qi >= 0 && qi < N) ? qi : -1;
    };
    // O / l of the finished unit to its query's output row
    // With a carried shared partial (sh_lse, sh_o: the route stage's log-sum-exp and
    // normalised output of the m shared pairs) this unit attended over the raw pairs only,
    // and the two partials merge here: tutorial ch. 4, (Z1 o1 + Z2 o2) / (Z1 + Z2).
    constexpr bool carried = kCarried;
    auto write_row = [&](int bh, int qi, float lsum, float mr, float l1, int pos) {
      bool wr = ok && qi >= 0;
      const size_t rowi = (size_t)bh * N + (wr ? qi : 0);
      size_t pi = 0;
      if (kPartial && wr) {
        // this (query, expert) entry's slot among the query's s partials
        const int ps = atomicAdd(&part.cnt[rowi], 1);
        if (ps >= nroutes) {
          flag_error(status, kDevErrBadBucket);
          wr = false;
        } else {
          pi = rowi * nroutes + ps;
          part.lse[pi] = (mr + log2f(lsum)) * 0.6931471805599453f;   // natural log
          part.pos[pi] = pos;
        }
      }
      float w1 = 0.f, w2 = 1.f / lsum;
      if (carried) {
        const float L1 = l1 * 1.4426950408889634f, L2 = mr + log2f(lsum);   // log2 units
        const float M = fmaxf(L1, L2);
        const float a1 = ex2(L1 - M), a2 = ex2(L2 - M);
        const float inv = 1.f / (a1 + a2);
        w1 = a1 * inv;
        w2 = a2 * inv / lsum;
      }
      bf16* dst = out + rowi * 64;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float o[32];
        tmem_ld32(tO + half * 32, o);   // warp-collective: every lane takes part
        tmem_ld_wait();
        tmem_fence_regs<32>(o);
        if (!wr) continue;
        if (kPartial) {
          const float inv = 1.f / lsum;
          float4* dp = reinterpret_cast<float4*>(part.o + pi * 64 + half * 32);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dp[i] = make_float4(o[4 * i] * inv, o[4 * i + 1] * inv, o[4 * i + 2] * inv,
                                o[4 * i + 3] * inv);
          continue;
        }
        if (carried) {
          float o1[32];
          if (o_bf16) {
            const uint4* src = reinterpret_cast<const uint4*>(static_cast<const bf16*>(sh_o) + rowi * 64 + half * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint4 x = src[i];
              const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                o1[8 * i + 2 * e] = __uint_as_float(w[e] << 16);
                o1[8 * i + 2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
              }
            }
          } else {
            const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(sh_o) + rowi * 64 + half * 32);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float4 x = src[i];
              o1[4 * i] = x.x; o1[4 * i + 1] = x.y; o1[4 * i + 2] = x.z; o1[4 * i + 3] = x.w;
            }
          }
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = fmaf(w1, o1[i], w2 * o[i]);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= w2;
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {   // 32-byte stores
          uint32_t w[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) w[e] = pack_bf16(o[16 * i + 2 * e], o[16 * i + 2 * e + 1]);
          asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst + 32 * half + 16 * i),
                       "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]),
                       "r"(w[7])
                       : "memory");
        }
      }
    };
    // start the second tile's group half a chunk late: the two groups then take turns on
    // the exponential unit instead of competing for it in lockstep
    if (slot == 1) __nanosleep(500);
    int4 cur = units > 0 ? unit_tab[ubase] : make_int4(0, 0, 0, 0);
    int4 nxt = units > 1 ? unit_tab[ubase + 1] : cur;
    int qi = units > 0 ? row_query(cur) : -1;
    // the carried shared log-sum-exp of this thread's query in the current unit
    // (and the carried output row is prefetched into L2 now: it is read only when the unit
    // is written out, a unit of chunks later)
    auto row_lse = [&](const int4& u, int q) -> float {
      if (!(carried && q >= 0)) return 0.f;
      const size_t r = (size_t)(u.x / m) * N + q;
      const char* p = o_bf16 ? reinterpret_cast<const char*>(static_cast<const bf16*>(sh_o) + r * 64)
                             : reinterpret_cast<const char*>(static_cast<const float*>(sh_o) + r * 64);
      asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
      if (!o_bf16) asm volatile("prefetch.global.L2 [%0];" ::"l"(p + 128));
      return sh_lse[r];
    };
    float l1 = units > 0 ? row_lse(cur, qi) : 0.f;
    // masked form: the routed expert of this thread's query (-1: a padding row)
    auto row_expert = [&](const int4& u, int q) -> int {
      if (!kMasked || q < 0) return -1;
      const int e = qroute[(size_t)(u.x / m) * N + q];
      return (e >= 0 && e < m) ? e : -1;
    };
    int eq = units > 0 ? row_expert(cur, qi) : -1;
    int it = 0, c = 0;
    int prev_bh = 0, prev_qi = -1, prev_pos = 0;
    float prev_lsum = 1.f, prev_mref = 0.f, prev_l1 = 0.f;
    bool pending = false;          // a finished unit's O still waits in tensor memory
    float mref = -INFINITY, lsum = 0.f;
    for (int g = 0; g < G; ++g, ++c) {
      if (c == nc) {
        // next unit; the finished one is written out inside this chunk, once its
        // last P . V is done
        prev_bh = cur.x / m;
        prev_qi = qi;
        prev_pos = cur.y + qr;
        prev_lsum = lsum;
        prev_mref = mref;
        prev_l1 = l1;
        pending = true;
        ++it;
        c = 0;
        cur = nxt;
        if (it + 1 < units) nxt = unit_tab[ubase + it + 1];
        qi = row_query(cur);
        l1 = row_lse(cur, qi);
        eq = row_expert(cur, qi);
        mref = -INFINITY;
        lsum = 0.f;
      }
      if (ok && !mbar_wait(&s.s_full[slot], g & 1)) ok = false;
      tc_fence_after();
      const int nvalid = c < nrc ? min(BN, topk - c * BN) : min(BN, m - (c - nrc) * BN);
      // the chunk's scores, with the maximum of each 32-column block from the reducing load
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
      if (nvalid < BN) {
#pragma unroll
        for (int i = 0; i < BN; ++i) v[i] = i < nvalid ? v[i] : -INFINITY;
      }
      if (kMasked && c < nrc) {
        // only the keys of the query's expert (a padding row keeps none)
        const uint32_t* mw = kmask + ((size_t)(cur.x / m) * m + (eq >= 0 ? eq : 0)) * mwords;
#pragma unroll
        for (int w4 = 0; w4 < 4; ++w4) {
          const int wi = c * 4 + w4;
          const uint32_t bits = (eq >= 0 && wi < mwords) ? mw[wi] : 0u;
#pragma unroll
          for (int i = 0; i < 32; ++i) v[32 * w4 + i] = ((bits >> i) & 1u) ? v[32 * w4 + i] : -INFINITY;
        }
      }
      // row maximum: the loads' block maxima, or (a ragged chunk, or keys masked out) four
      // independent chains over the valid entries
      float tm = fmaxf(fmaxf(q4[0], q4[1]), fmaxf(q4[2], q4[3]));
      if (kMasked || nvalid < BN) {
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int i = 0; i < BN; i += 8)
#pragma unroll
          for (int a = 0; a < 4; ++a) m4[a] = max3(m4[a], v[i + 2 * a], v[i + 2 * a + 1]);
        tm = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      }
      const float csc = c >= nrc ? cs_shared : cs;  // the chunk's logit scale, log2 units
      const float xm = tm * csc;
      const bool need = (c == 0) || (xm > mref + kLazy);
      const float f = (c > 0 && need) ? ex2(mref - xm) : 1.f;
      if (need) {
        lsum *= f;
        mref = xm;
      }
      // P = 2^(s * csc - mref) in fp32 pairs, packed to bf16 pairs; the row sum in two
      // pair chains (from the unrounded values).  (Masked form: a row with no key of its
      // expert so far keeps mref = -inf; its P is 0, not inf - inf.)
      const float mr_off = (kMasked && mref == -INFINITY) ? 0.f : mref;
      const unsigned long long c2 = f2pack(csc, csc), nm2 = f2pack(-mr_off, -mr_off);
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
      // first half of P while the previous P . V may still run
      uint32_t pk0[BN / 4];
      exp_half(0, pk0);
      // the previous P . V must have read P and finished with O
      if (g > 0 && ok && !mbar_wait(&s.pv_done[slot], (g - 1) & 1)) ok = false;
      tc_fence_after();
      tmem_st16(tP, pk0);
      tmem_st16(tP + 16, pk0 + 16);
      if (pending) {
        write_row(prev_bh, prev_qi, prev_lsum, prev_mref, prev_l1, prev_pos);
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
    if (G > 0) {
      if (ok && !mbar_wait(&s.pv_done[slot], (G - 1) & 1)) ok = false;
      tc_fence_after();
      write_row(cur.x / m, qi, lsum, mref, l1, cur.y + qr);
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

bool expert_tc_supported(int d, int m, int topk) { return d == 64 && m >= 1 && topk >= 1; }

size_t expert_tc_ws_bytes(int BH, int N, int m, int topk) {
  auto r = [](size_t b) { return (b + 255) / 256 * 256; };
  return r((size_t)BH * m * 64 * 2) + r(((size_t)BH * m + 1) * 4) +
         r(max_units(BH, N, m) * 16) + 2 * r((size_t)BH * m * topk * 128);
}

cudaError_t launch_expert_tc(const bf16* q, const bf16* k, const bf16* v, const bf16* q_tilde,
                             const float* v_tilde, const int32_t* topk_idx,
                             const int32_t* bucket_off, const int32_t* bucket_qidx, int BH, int N,
                             int m, int topk, int num_sms, void* ws, bf16* out, int* status,
                             cudaStream_t st, int shared_temp, int routed_only,
                             const float* shared_lse, const void* shared_o, int o_bf16) {
  const ExpertTcWs w = carve(ws, BH, N, m, topk);
  // log2(e) / sqrt(64), or log2(e) / 64 for the shared logits at the official code's temperature
  const float cs_shared = shared_temp ? 0.022542110013890052f : 0.18033688011112042f;
  const long long rows = (long long)BH * m * topk;
  const long long gblocks = std::min<long long>((rows + kGatherThreads / 8 - 1) / (kGatherThreads / 8),
                                                (long long)std::max(num_sms, 1) * 8);
  // gblocks gathering CTAs plus the one that builds the unit table
  // shared chunks run in the kernel unless the routing-only ablation drops the branch or the
  // route stage carried its partial
  const bool shared_chunks = !(routed_only || shared_lse);
  cudaError_t e = launch_pdl(expert_gather_kernel, dim3((unsigned)gblocks + 1), dim3(kGatherThreads),
                             0, st, k, v, topk_idx, rows, N, m, topk, bucket_off,
                             shared_chunks ? v_tilde : static_cast<const float*>(nullptr), BH, w,
                             status, N);
  count_launch();
  if (e != cudaSuccess) return e;
  CUtensorMap mqg, mkg, mvg, mqt, mvt;
  if (!make_tmap_gather64(&mqg, q, (uint64_t)BH * N) ||
      !make_tmap_rows64(&mkg, w.kg, (uint64_t)topk, (uint64_t)BH * m, BN) ||
      !make_tmap_rows64(&mvg, w.vg, (uint64_t)topk, (uint64_t)BH * m, BN) ||
      // (without shared chunks these two maps are never loaded: any valid map will do)
      !make_tmap_rows64(&mqt, shared_chunks ? static_cast<const void*>(q_tilde) : w.kg,
                        (uint64_t)(shared_chunks ? m : topk), (uint64_t)(shared_chunks ? BH : BH * m), BN) ||
      !make_tmap_rows64(&mvt, shared_chunks ? static_cast<const void*>(w.vtb) : w.vg,
                        (uint64_t)(shared_chunks ? m : topk), (uint64_t)(shared_chunks ? BH : BH * m), BN))
    return cudaErrorInvalidValue;
  const size_t smem = sizeof(ExpertSmem) + 1024;
  e = cudaFuncSetAttribute(expert_tc_kernel<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(expert_tc_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(shared_lse ? expert_tc_kernel<true, false> : expert_tc_kernel<false, false>,
                 dim3((unsigned)std::max(num_sms, 1)), dim3(kThreads), smem, st,
                 mqg, mkg, mvg, mqt, mvt, bucket_qidx,
                 static_cast<const int*>(w.unit_start + (size_t)BH * m),
                 static_cast<const int4*>(w.unit), BH, N, m, topk, cs_shared, shared_chunks ? 1 : 0,
                 shared_lse, shared_o, o_bf16, static_cast<const uint32_t*>(nullptr), 0,
                 static_cast<const int32_t*>(nullptr), out, status, N, 1, ExpertPartials{});
  count_launch();
  return e;
}

// Top-s partials (s > 1): the raw pairs of every (query, expert) entry of the N * s-entry
// buckets, one partial per entry into `part` (cleared slot counters: the caller merges).
size_t expert_tc_partials_ws_bytes(int BH, int N, int m, int topk, int s) {
  return expert_tc_ws_bytes(BH, N * s, m, topk);
}

cudaError_t launch_expert_tc_partials(const bf16* q, const bf16* k, const bf16* v,
                                      const int32_t* topk_idx, const int32_t* bucket_off,
                                      const int32_t* bucket_qidx, int BH, int N, int m, int topk,
                                      int s, int num_sms, void* ws, ExpertPartials part,
                                      int* status, cudaStream_t st) {
  if (s < 1 || (long long)N * s >= (1LL << 31)) return cudaErrorInvalidValue;
  const int nent = N * s;
  const ExpertTcWs w = carve(ws, BH, nent, m, topk);
  const long long rows = (long long)BH * m * topk;
  const long long gblocks = std::min<long long>((rows + kGatherThreads / 8 - 1) / (kGatherThreads / 8),
                                                (long long)std::max(num_sms, 1) * 8);
  cudaError_t e = cudaMemsetAsync(part.cnt, 0, (size_t)BH * N * sizeof(int), st);
  if (e != cudaSuccess) return e;
  e = launch_pdl(expert_gather_kernel, dim3((unsigned)gblocks + 1), dim3(kGatherThreads), 0, st, k,
                 v, topk_idx, rows, N, m, topk, bucket_off, static_cast<const float*>(nullptr), BH,
                 w, status, nent);
  count_launch();
  if (e != cudaSuccess) return e;
  CUtensorMap mqg, mkg, mvg;
  if (!make_tmap_gather64(&mqg, q, (uint64_t)BH * N) ||
      !make_tmap_rows64(&mkg, w.kg, (uint64_t)topk, (uint64_t)BH * m, BN) ||
      !make_tmap_rows64(&mvg, w.vg, (uint64_t)topk, (uint64_t)BH * m, BN))
    return cudaErrorInvalidValue;
  const size_t smem = sizeof(ExpertSmem) + 1024;
  auto kern = expert_tc_kernel<false, false, true>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // no shared chunks: the q~ / v~ maps are never loaded (the expert block maps stand in)
  e = launch_pdl(kern, dim3((unsigned)std::max(num_sms, 1)), dim3(kThreads), smem, st, mqg, mkg,
                 mvg, mkg, mvg, bucket_qidx,
                 static_cast<const int*>(w.unit_start + (size_t)BH * m),
                 static_cast<const int4*>(w.unit), BH, N, m, topk, 0.18033688011112042f, 0,
                 static_cast<const float*>(nullptr), static_cast<const void*>(nullptr), 0,
                 static_cast<const uint32_t*>(nullptr), 0, static_cast<const int32_t*>(nullptr),
                 static_cast<bf16*>(nullptr), status, nent, s, part);
  count_launch();
  return e;
}

// ---------------------------------------------------------------------------------------------
// Dense softmax attention on the same kernel: one "expert" per head holding all N keys in
// order (K and V are read in place, no gather), no shared chunks, queries in natural order.
// ---------------------------------------------------------------------------------------------
namespace {
__global__ void __launch_bounds__(256)
dense_units_kernel(int BH, int N, int4* __restrict__ unit, int* __restrict__ unit_count,
                   int32_t* __restrict__ qidx) {
  griddep_wait();
  const long long per = (N + kUnitQ - 1) / kUnitQ;
  const long long nu = (long long)BH * per, nq = (long long)BH * N;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x; t < nu || t < nq;
       t += stride) {
    if (t < nu) {
      const int bh = (int)(t / per), j = (int)(t % per);
      unit[t] = make_int4(bh, j * kUnitQ, min(kUnitQ, N - j * kUnitQ), 0);
    }
    if (t < nq) qidx[t] = (int32_t)(t % N);
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) *unit_count = (int)nu;
}
}  // namespace

size_t dense_tc_ws_bytes(int BH, int N) {
  auto r = [](size_t b) { return (b + 255) / 256 * 256; };
  const size_t nu = (size_t)BH * ((N + kUnitQ - 1) / kUnitQ);
  return r(nu * 16) + r(4) + r((size_t)BH * N * 4);
}

cudaError_t launch_dense_tc(const bf16* q, const bf16* k, const bf16* v, int BH, int N,
                            int num_sms, void* ws, bf16* out, int* status, cudaStream_t st) {
  auto r = [](size_t b) { return (b + 255) / 256 * 256; };
  const size_t nu = (size_t)BH * ((N + kUnitQ - 1) / kUnitQ);
  char* p = static_cast<char*>(ws);
  int4* unit = reinterpret_cast<int4*>(p);
  int* ucount = reinterpret_cast<int*>(p + r(nu * 16));
  int32_t* qidx = reinterpret_cast<int32_t*>(p + r(nu * 16) + r(4));
  const long long work = std::max<long long>((long long)nu, (long long)BH * N);
  const unsigned blocks =
      (unsigned)std::min<long long>((work + 255) / 256, (long long)std::max(num_sms, 1) * 8);
  cudaError_t e = launch_pdl(dense_units_kernel, dim3(blocks), dim3(256), 0, st, BH, N, unit,
                             ucount, qidx);
  count_launch();
  if (e != cudaSuccess) return e;
  CUtensorMap mqg, mkg, mvg, mqt, mvt;
  // the shared-block maps are never loaded (no shared chunks); any valid map will do
  if (!make_tmap_gather64(&mqg, q, (uint64_t)BH * N) ||
      !make_tmap_rows64(&mkg, k, (uint64_t)N, (uint64_t)BH, BN) ||
      !make_tmap_rows64(&mvg, v, (uint64_t)N, (uint64_t)BH, BN) ||
      !make_tmap_rows64(&mqt, k, (uint64_t)N, (uint64_t)BH, BN) ||
      !make_tmap_rows64(&mvt, v, (uint64_t)N, (uint64_t)BH, BN))
    return cudaErrorInvalidValue;
  const size_t smem = sizeof(ExpertSmem) + 1024;
  e = cudaFuncSetAttribute(expert_tc_kernel<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(expert_tc_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(expert_tc_kernel<false, false>, dim3((unsigned)std::max(num_sms, 1)), dim3(kThreads), smem, st,
                 mqg, mkg, mvg, mqt, mvt, static_cast<const int32_t*>(qidx),
                 static_cast<const int*>(ucount), static_cast<const int4*>(unit), BH, N, 1, N,
                 0.18033688011112042f, 0, static_cast<const float*>(nullptr),
                 static_cast<const void*>(nullptr), 0, static_cast<const uint32_t*>(nullptr), 0,
                 static_cast<const int32_t*>(nullptr), out, status, N, 1, ExpertPartials{});
  count_launch();
  return e;
}

}  // namespace mita

// ---------------------------------------------------------------------------------------------
// Short sequences (N <= 1024): tiles of a head's consecutive queries attend over the m shared
// pairs and all N keys, each query's raw keys masked to its routed expert's top-k set
// (expert_tc_kernel<false, true>).  When experts hold only a handful of queries each (ViT-S:
// ~8 of 196), this replaces ~m mostly empty 256-query units per head by ceil(N / 256) full
// ones and needs neither the bucket stage nor the gathered K / V blocks.
// ---------------------------------------------------------------------------------------------
namespace mita {
namespace {

// One launch: each CTA takes (head, expert) rows in turn and builds the expert's key bit mask
// (32 keys per word) in shared memory; the grid also writes the unit table (unit = (head * m,
// first query, count <= 256)), the identity query list and v~ in bf16.
__global__ void __launch_bounds__(256)
expert_mask_kernel(const int32_t* __restrict__ topk_idx, const float* __restrict__ v_tilde,
                   int BH, int N, int m, int topk, int mwords, uint32_t* __restrict__ kmask,
                   bf16* __restrict__ vtb, int4* __restrict__ unit, int* __restrict__ ucount,
                   int32_t* __restrict__ qidx, int* status) {
  griddep_wait();
  extern __shared__ uint32_t words[];       // [mwords]
  const long long stride = (long long)gridDim.x * blockDim.x;
  const long long t0 = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (v_tilde != nullptr) {
    const long long n4 = (long long)BH * m * 16;
    for (long long t = t0; t < n4; t += stride) {
      const float4 x = reinterpret_cast<const float4*>(v_tilde)[t];
      uint2 o;
      o.x = pack_bf16(x.x, x.y);
      o.y = pack_bf16(x.z, x.w);
      reinterpret_cast<uint2*>(vtb)[t] = o;
    }
  }
  const long long per = (N + kUnitQ - 1) / kUnitQ, nu = (long long)BH * per;
  const long long nq = (long long)BH * N;
  for (long long t = t0; t < nu || t < nq; t += stride) {
    if (t < nu) {
      const int bh = (int)(t / per), j = (int)(t % per);
      unit[t] = make_int4(bh * m, j * kUnitQ, min(kUnitQ, N - j * kUnitQ), 0);
    }
    if (t < nq) qidx[t] = (int32_t)(t % N);
  }
  if (t0 == 0) *ucount = (int)nu;
  const long long rows = (long long)BH * m;
  for (long long r = blockIdx.x; r < rows; r += gridDim.x) {
    for (int w = threadIdx.x; w < mwords; w += blockDim.x) words[w] = 0u;
    __syncthreads();
    for (int t = threadIdx.x; t < topk; t += blockDim.x) {
      const int j = topk_idx[r * topk + t];
      if (j >= 0 && j < N) atomicOr(&words[j >> 5], 1u << (j & 31));
      else flag_error(status, kDevErrBadIndex);
    }
    __syncthreads();
    for (int w = threadIdx.x; w < mwords; w += blockDim.x) kmask[r * mwords + w] = words[w];
    __syncthreads();
  }
}

struct MaskedWs {
  int4* unit;
  int* ucount;
  int32_t* qidx;
  bf16* vtb;
  uint32_t* kmask;
};

MaskedWs carve_masked(void* ws, int BH, int N, int m) {
  auto r = [](size_t b) { return (b + 255) / 256 * 256; };
  const size_t nu = (size_t)BH * ((N + kUnitQ - 1) / kUnitQ);
  const int mwords = (N + 31) / 32;
  char* p = static_cast<char*>(ws);
  MaskedWs w;
  w.unit = reinterpret_cast<int4*>(p); p += r(nu * 16);
  w.ucount = reinterpret_cast<int*>(p); p += r(4);
  w.qidx = reinterpret_cast<int32_t*>(p); p += r((size_t)BH * N * 4);
  w.vtb = reinterpret_cast<bf16*>(p); p += r((size_t)BH * m * 64 * 2);
  w.kmask = reinterpret_cast<uint32_t*>(p);
  (void)mwords;
  return w;
}

}  // namespace

bool expert_masked_preferred(int N, int m, int topk, int routed_only) {
  if (N > 1024 || N < 1) return false;
  const long long nsc = routed_only ? 0 : (m + BN - 1) / BN;
  const long long tiles = (N + kUnitQ - 1) / kUnitQ;
  // MMA chunks per head: masked tiles over all keys, against ~one unit per expert (plus the
  // ragged ones) over the expert's keys
  const long long masked = tiles * ((N + BN - 1) / BN + nsc);
  const long long grouped = ((long long)m + tiles) * ((topk + BN - 1) / BN + nsc);
  return masked < grouped;
}

size_t expert_masked_ws_bytes(int BH, int N, int m) {
  auto r = [](size_t b) { return (b + 255) / 256 * 256; };
  const size_t nu = (size_t)BH * ((N + kUnitQ - 1) / kUnitQ);
  const size_t mwords = (size_t)(N + 31) / 32;
  return r(nu * 16) + r(4) + r((size_t)BH * N * 4) + r((size_t)BH * m * 64 * 2) +
         r((size_t)BH * m * mwords * 4);
}

cudaError_t launch_expert_masked_tc(const bf16* q, const bf16* k, const bf16* v,
                                    const bf16* q_tilde, const float* v_tilde,
                                    const int32_t* topk_idx, const int32_t* route, int BH, int N,
                                    int m, int topk, int num_sms, void* ws, bf16* out,
                                    int* status, cudaStream_t st, int shared_temp,
                                    int routed_only) {
  const MaskedWs w = carve_masked(ws, BH, N, m);
  const int mwords = (N + 31) / 32;
  const bool shared_chunks = !routed_only;
  const float cs_shared = shared_temp ? 0.022542110013890052f : 0.18033688011112042f;
  const long long work = std::max<long long>((long long)BH * m, (long long)BH * N / 256 + 1);
  const unsigned blocks = (unsigned)std::min<long long>(work, (long long)std::max(num_sms, 1) * 8);
  cudaError_t e = launch_pdl(expert_mask_kernel, dim3(blocks), dim3(256), (size_t)mwords * 4, st,
                             topk_idx, shared_chunks ? v_tilde : static_cast<const float*>(nullptr),
                             BH, N, m, topk, mwords, w.kmask, w.vtb, w.unit, w.ucount, w.qidx,
                             status);
  count_launch();
  if (e != cudaSuccess) return e;
  CUtensorMap mqg, mkg, mvg, mqt, mvt;
  if (!make_tmap_gather64(&mqg, q, (uint64_t)BH * N) ||
      !make_tmap_rows64(&mkg, k, (uint64_t)N, (uint64_t)BH, BN) ||
      !make_tmap_rows64(&mvg, v, (uint64_t)N, (uint64_t)BH, BN) ||
      // (without shared chunks these two maps are never loaded: any valid map will do)
      !make_tmap_rows64(&mqt, shared_chunks ? static_cast<const void*>(q_tilde) : k,
                        (uint64_t)(shared_chunks ? m : N), (uint64_t)BH, BN) ||
      !make_tmap_rows64(&mvt, shared_chunks ? static_cast<const void*>(w.vtb) : v,
                        (uint64_t)(shared_chunks ? m : N), (uint64_t)BH, BN))
    return cudaErrorInvalidValue;
  const size_t smem = sizeof(ExpertSmem) + 1024;
  e = cudaFuncSetAttribute(expert_tc_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem);
  if (e != cudaSuccess) return e;
  // the raw "entries" of a unit are all N keys of its head (topk = N for the chunk count)
  e = launch_pdl(expert_tc_kernel<false, true>, dim3((unsigned)std::max(num_sms, 1)), dim3(kThreads),
                 smem, st, mqg, mkg, mvg, mqt, mvt, static_cast<const int32_t*>(w.qidx),
                 static_cast<const int*>(w.ucount), static_cast<const int4*>(w.unit), BH, N, m, N,
                 cs_shared, shared_chunks ? 1 : 0, static_cast<const float*>(nullptr),
                 static_cast<const void*>(nullptr), 0, static_cast<const uint32_t*>(w.kmask),
                 mwords, route, out, status, N, 1, ExpertPartials{});
  count_launch();
  return e;
}

}  // namespace mita
