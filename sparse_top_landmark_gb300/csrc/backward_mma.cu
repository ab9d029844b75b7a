// Gradient passes of the backward on the warp-level tensor cores (bf16 operands, d = 64).
//
// The backward (selections held constant; the formulas are in backward.cu) consists of
// three passes of one shape: a set of query rows (q, with upstream rows g, a log-sum-exp L
// and D = g . o per row) against a set of key rows (k, with value rows v) under one logit
// scale c:
//   P = exp(c q.k - L),  dS = P (g.v - D),
//   dq += c dS k,   dk += c dS^T q,   dv += P^T g.
//   raw pass     queries = the bucket entries of one expert, keys = its top-k rows
//                (MiTA tutorial ch. 4 steps 5-6: the routed pairs of the joint softmax);
//   shared pass  queries = all N queries, keys = the m landmarks (q~, v~), c = c_sh
//                (the shared pairs of the joint softmax);
//   v~ pass      queries = the m landmarks (q~, dv~, the landmark softmax normaliser,
//                dv~ . v~), keys = all N keys (tutorial ch. 4 step 3, v~ = softmax(q~ K^T c) V).
// Each pass runs two or three launches of bwd_mma_kernel (with s = 1 one joint launch does
// the routed and shared passes' row sums and dq together: a query's whole joint softmax is
// its expert's top-k rows and the head's landmarks, swept once for D and once for dq):
//   row sums     query-major, D = sum over the pass's keys of P dP added to each query's D
//                (the forward's outputs, recomputed with bf16 operands, would give a D that
//                does not match these P and dP; the gradient of q sums dS = P (dP - D) k
//                over keys whose dS cancel, so every error in D is amplified there);
//   query-major  a CTA owns 64 query rows (16 per warp) and streams key rows in chunks of 64:
//                S = q k^T and dP = g v^T as m16n8k16 MMAs, P and dS in registers, then
//                dq += dS k with dS re-used in place as the A operand, split into a bf16 part
//                and a bf16 remainder (the same cancellation); dq is added to memory once
//                per owned element at the end;
//   key-major    a CTA owns 64 key rows and streams query chunks: S^T and dP^T, then
//                dv += P^T g and dk += dS^T q, added once per owned element at the end.
// Both recompute S and dP, three extra products per pair, but every accumulator stays in
// the registers of the warp that owns its row: no cross-warp reduction and no per-chunk
// atomics.  Streams longer than kSplitRows are split over CTAs (the v~ pass's N keys, the
// shared pass's N queries), whose results meet in the final atomic adds (16 bytes each);
// a launch that is the first and only writer of its owned rows (BwdPass::first: one
// segment per row and an unsplit stream) stores them instead, so they need no clearing.
// Operands: bf16 rows staged by cp.async (double-buffered, zero-filled past the end) into
// shared memory with a 144-byte row stride, so the eight rows of an ldmatrix hit distinct
// banks; P and dS are rounded to bf16 for the second products; accumulation is fp32.
#include "common.cuh"
#include "kernels.h"

namespace mita {
namespace {

constexpr int kRows = 64;          // owned rows per CTA and streamed rows per chunk
constexpr int kPad = 72;           // shared-memory row stride in bf16 elements (144 B)
constexpr int kSplitRows = kBwdSplitRows;   // streamed rows per CTA
constexpr int kThreads = 128;      // four warps, 16 owned rows each
constexpr float kLog2e = 1.4426950408889634f;
constexpr bool kSplitDs = true;    // dq += (dS_hi + dS_lo) k
enum { kQueryMajor = 0, kKeyMajor = 1, kRowSums = 2, kJoint = 3 };

struct MmaSmem {
  bf16 own[2][kRows][kPad];        // owned rows: (q, g) or (k, v)
  bf16 st[2][2][kRows][kPad];      // [buffer][matrix][row]: streamed (k, v) or (q, g)
  float sa[2][kRows];              // per streamed row: key bias (0 / -inf), or the query's L
  float sb[2][kRows];              // per streamed query row: D
  long long own_row[kRows];        // global row of each owned row, -1 past the end
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// 16-byte copy, zero-filled when src_bytes is 0 (nothing is read then)
__device__ __forceinline__ void cp16(void* dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(src_bytes)
               : "memory");
}
// 4-byte copy, zero-filled when src_bytes is 0
__device__ __forceinline__ void cp4(void* dst, const void* src, int src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void ldsm4(uint32_t* r, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm4t(uint32_t* r, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
// c += a (16x16, row) * b (16x8, col), bf16 in, fp32 accumulate
__device__ __forceinline__ void mma(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// two fp32 values as a bf16 pair, `lo` in the low half
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// the remainders of (lo, hi) after their bf16 pair h
__device__ __forceinline__ uint32_t pack2_rest(float lo, float hi, uint32_t h) {
  return pack2(lo - __uint_as_float(h << 16), hi - __uint_as_float(h & 0xffff0000u));
}
__device__ __forceinline__ float exp2a(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The rows of one side of a segment: row p (0 <= p < cnt) is global row
// base + (list ? list[p] : p); list values outside [0, lim) are flagged and skipped.
struct Side {
  const int32_t* list;
  long long base;
  int cnt, lim;
};
// A thread stages four rows of a 64-row block, rows (tid >> 3) + 16 j, 16 bytes (piece
// tid & 7) of each.  side_fetch reads their list values (kPastEnd past the end); the kernel
// fetches them one block ahead, so a block's copies never wait on its index loads.
constexpr int kPastEnd = -2147483647 - 1;
__device__ __forceinline__ void side_fetch(const Side& s, int p0, int* x) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int p = p0 + (threadIdx.x >> 3) + 16 * j;
    x[j] = p < s.cnt ? (s.list ? s.list[p] : p) : kPastEnd;
  }
}
// Copies the two 64-wide bf16 rows of each of the thread's four rows, zero-filled past the
// end and for invalid list values (flagged); gr[j] = the global row, or -1.
__device__ __forceinline__ void stage4(bf16 (*d0)[kPad], bf16 (*d1)[kPad], const bf16* s0,
                                       const bf16* s1, const Side& sd, const int* x, int* status,
                                       long long* gr) {
  const int piece = threadIdx.x & 7;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int r = (threadIdx.x >> 3) + 16 * j;
    long long g = -1;
    if (x[j] >= 0 && x[j] < sd.lim) g = sd.base + x[j];
    else if (x[j] != kPastEnd && piece == 0) flag_error(status, kDevErrBadIndex);
    gr[j] = g;
    const size_t o = (g < 0 ? 0 : (size_t)g * 64) + piece * 8;
    cp16(d0[r] + piece * 8, s0 + o, g < 0 ? 0 : 16);
    cp16(d1[r] + piece * 8, s1 + o, g < 0 ? 0 : 16);
  }
}

// Work items of one segment: (owned 64-row block, split of the stream).
__device__ __forceinline__ int seg_items(int own_cnt, int st_cnt) {
  if (own_cnt <= 0 || st_cnt <= 0) return 0;
  return ((own_cnt + kRows - 1) / kRows) * ((st_cnt + kSplitRows - 1) / kSplitRows);
}

template <int kMode>
__global__ void __launch_bounds__(kThreads, 3)   // three CTAs (twelve warps) per SM
bwd_mma_kernel(BwdPass a) {
  constexpr bool kKM = kMode == kKeyMajor, kRS = kMode == kRowSums, kJ = kMode == kJoint;
  extern __shared__ __align__(128) unsigned char smraw[];
  MmaSmem& sm = *reinterpret_cast<MmaSmem*>(smraw);
  __shared__ int s_e, s_w;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const long long bh = blockIdx.x / a.items;
  const int item = blockIdx.x % a.items;
  const bool raw = a.bucket_off != nullptr;

  // ---- the segment and the (owned block, stream split) of this CTA
  Side qs, ks;
  int w = item;
  if (raw) {
    const int32_t* off = a.bucket_off + (size_t)bh * (a.m + 1);
    if (warp == 0) {
      int run = 0, fe = -1, fw = 0;
      for (int e0 = 0; e0 < a.m && fe < 0; e0 += 32) {
        const int e = e0 + lane;
        int cnt = 0;
        if (e < a.m) {
          const int x0 = off[e], x1 = off[e + 1];
          if (x0 < 0 || x1 > a.NS || x1 < x0) flag_error(a.status, kDevErrBadBucket);
          else cnt = x1 - x0;
        }
        const int W = kKM ? seg_items(a.topk, cnt) : kJ ? seg_items(cnt, 1) : seg_items(cnt, a.topk);
        const int inc = warp_incl_scan(W);
        const int tot = __shfl_sync(0xffffffffu, inc, 31);
        if (item < run + tot) {
          const unsigned hit = __ballot_sync(0xffffffffu, run + inc > item);
          const int f = __ffs(hit) - 1;
          fe = e0 + f;
          fw = item - (run + __shfl_sync(0xffffffffu, inc - W, f));
        }
        run += tot;
      }
      if (lane == 0) { s_e = fe; s_w = fw; }
    }
    __syncthreads();
    const int e = s_e;
    if (e < 0) return;
    w = s_w;
    const int x0 = off[e];
    qs = Side{a.bucket_qidx + (size_t)bh * a.NS + x0, bh * (long long)a.N, off[e + 1] - x0, a.N};
    ks = Side{a.topk_idx + ((size_t)bh * a.m + e) * a.topk, bh * (long long)a.N, a.topk, a.N};
  } else {
    qs = Side{nullptr, bh * (long long)a.nq, a.nq, a.nq};
    ks = Side{nullptr, bh * (long long)a.nk, a.nk, a.nk};
    if (w >= (kKM ? seg_items(a.nk, a.nq) : seg_items(a.nq, a.nk))) return;
  }
  const Side& os = kKM ? ks : qs;   // owned side
  const Side& ss = kKM ? qs : ks;   // streamed side
  const int splits = kJ ? 1 : (ss.cnt + kSplitRows - 1) / kSplitRows;
  const int o0 = (w / splits) * kRows;
  const int s0 = (w % splits) * kSplitRows;
  // joint: the expert's top-k rows, then the head's n2 rows of (k2, v2), each swept twice
  const Side sb2{nullptr, bh * (long long)a.n2, a.n2, a.n2};
  const int ncA = kJ ? (ss.cnt + kRows - 1) / kRows
                     : (min(ss.cnt - s0, kSplitRows) + kRows - 1) / kRows;
  const int nch = kJ ? ncA + (a.n2 + kRows - 1) / kRows : ncA;
  const int nv = kJ ? 2 * nch : nch;
  // virtual block v: (second side?, its first row)
  auto block_of = [&](int v, int& p0) {
    const int c = kJ ? v % nch : v;
    const bool b2 = kJ && c >= ncA;
    p0 = b2 ? (c - ncA) * kRows : s0 + c * kRows;
    return b2;
  };

  const bf16* own0 = kKM ? a.k : a.q;
  const bf16* own1 = kKM ? a.v : a.g;
  const bf16* st0 = kKM ? a.q : a.k;
  const bf16* st1 = kKM ? a.g : a.v;

  const bool piece0 = (tid & 7) == 0;
  {
    int xo[4];
    long long go[4];
    side_fetch(os, o0, xo);
    stage4(sm.own[0], sm.own[1], own0, own1, os, xo, a.status, go);
    if (piece0)
#pragma unroll
      for (int j = 0; j < 4; ++j) sm.own_row[(tid >> 3) + 16 * j] = go[j];
  }
  cp_commit();
  // A streamed block from its fetched list values.  Per row: key-major copies L and D
  // (zero for a missing query row, whose q and g rows are zero too, so its P = 1 meets
  // zero rows and adds nothing); query-major writes the key's bias (-inf: no key).
  auto stage_stream = [&](int buf, const int* x, bool b2) {
    long long gs[4];
    stage4(sm.st[buf][0], sm.st[buf][1], b2 ? a.k2 : st0, b2 ? a.v2 : st1, b2 ? sb2 : ss, x,
           a.status, gs);
    if (piece0) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = (tid >> 3) + 16 * j;
        if constexpr (kKM) {
          cp4(&sm.sa[buf][r], a.L + (gs[j] < 0 ? 0 : gs[j]), gs[j] < 0 ? 0 : 4);
          cp4(&sm.sb[buf][r], a.D + (gs[j] < 0 ? 0 : gs[j]), gs[j] < 0 ? 0 : 4);
        } else {
          sm.sa[buf][r] = gs[j] < 0 ? -INFINITY : 0.f;
        }
      }
    }
  };
  int xs[4], p0;
  bool xb = block_of(0, p0);
  side_fetch(xb ? sb2 : ss, p0, xs);
  stage_stream(0, xs, xb);
  cp_commit();
  if (nv > 1) {
    xb = block_of(1, p0);
    side_fetch(xb ? sb2 : ss, p0, xs);
  }
  cp_wait<1>();
  __syncthreads();

  // ---- owned fragments: rows 16 warp .. +15, as A operands over d (four k-steps)
  uint32_t fa[4][4], fb[4][4];
  {
    const int r = 16 * warp + (lane & 7) + ((lane >> 3) & 1) * 8, c = (lane >> 4) * 8;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      ldsm4(fa[kk], &sm.own[0][r][16 * kk + c]);
      ldsm4(fb[kk], &sm.own[1][r][16 * kk + c]);
    }
  }
  const long long row_g = sm.own_row[16 * warp + g], row_g8 = sm.own_row[16 * warp + g + 8];
  // query-major: the owned rows' L log2e and D
  float Lr[2] = {0.f, 0.f}, Dr[2] = {0.f, 0.f}, rs[2] = {0.f, 0.f};
  if constexpr (!kKM) {
    if (row_g >= 0) { Lr[0] = a.L[row_g] * kLog2e; if (!kRS && !kJ) Dr[0] = a.D[row_g]; }
    if (row_g8 >= 0) { Lr[1] = a.L[row_g8] * kLog2e; if (!kRS && !kJ) Dr[1] = a.D[row_g8]; }
  }
  float cl2 = a.c * kLog2e;
  float acc0[8][4], acc1[8][4];    // dq (query-major); dk and dv (key-major)
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) { acc0[i][j] = 0.f; acc1[i][j] = 0.f; }

  // lane addresses of the streamed-operand loads within a 16-row group
  const int rb = (lane & 7) + (lane >> 4) * 8, cb = ((lane >> 3) & 1) * 8;    // B, n = rows
  const int rt = (lane & 7) + ((lane >> 3) & 1) * 8, ct = (lane >> 4) * 8;     // B, k = rows

  for (int c = 0; c < nv; ++c) {
    const int buf = c & 1;
    if (c + 1 < nv) {
      stage_stream(buf ^ 1, xs, xb);              // fetched one block ago
      cp_commit();
      if (c + 2 < nv) {
        xb = block_of(c + 2, p0);
        side_fetch(xb ? sb2 : ss, p0, xs);
      }
      cp_wait<1>();
    } else {
      cp_wait<0>();
    }
    __syncthreads();
    // joint: the block's scale, and after the first sweep each row's D from its sums
    bool grad = !kRS;
    float cs = 1.f;
    if constexpr (kJ) {
      int pz;
      cs = block_of(c, pz) ? a.c2 : a.c;
      cl2 = cs * kLog2e;
      grad = c >= nch;
      if (c == nch) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          rs[i] += __shfl_xor_sync(0xffffffffu, rs[i], 1);
          rs[i] += __shfl_xor_sync(0xffffffffu, rs[i], 2);
          Dr[i] = rs[i];
        }
        if (t == 0) {
          if (row_g >= 0) a.Dacc[row_g] = Dr[0];
          if (row_g8 >= 0) a.Dacc[row_g8] = Dr[1];
        }
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {          // 32 streamed rows at a time
      float s[4][4], dp[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) { s[i][j] = 0.f; dp[i][j] = 0.f; }
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
        for (int np = 0; np < 2; ++np) {
          uint32_t b[4];
          ldsm4(b, &sm.st[buf][0][32 * h + 16 * np + rb][16 * kk + cb]);
          mma(s[2 * np], fa[kk], b[0], b[1]);
          mma(s[2 * np + 1], fa[kk], b[2], b[3]);
          ldsm4(b, &sm.st[buf][1][32 * h + 16 * np + rb][16 * kk + cb]);
          mma(dp[2 * np], fb[kk], b[0], b[1]);
          mma(dp[2 * np + 1], fb[kk], b[2], b[3]);
        }
      }
      // P and dS in place of S and dP.  Fragment entry j of n-tile nt: row g + 8 (j >> 1),
      // streamed row 32 h + 8 nt + 2 t + (j & 1).
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const int col = 32 * h + 8 * nt + 2 * t;
        if constexpr (kKM) {
          const float2 L2 = *reinterpret_cast<const float2*>(&sm.sa[buf][col]);
          const float2 D2 = *reinterpret_cast<const float2*>(&sm.sb[buf][col]);
          const float nl0 = -L2.x * kLog2e, nl1 = -L2.y * kLog2e;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float p = exp2a(fmaf(s[nt][j], cl2, (j & 1) ? nl1 : nl0));
            dp[nt][j] = p * (dp[nt][j] - ((j & 1) ? D2.y : D2.x));
            s[nt][j] = p;
          }
        } else {
          const float2 B2 = *reinterpret_cast<const float2*>(&sm.sa[buf][col]);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float p = exp2a(fmaf(s[nt][j], cl2, -Lr[j >> 1]) + ((j & 1) ? B2.y : B2.x));
            if (!grad) rs[j >> 1] = fmaf(p, dp[nt][j], rs[j >> 1]);
            else dp[nt][j] = (kJ ? cs * p : p) * (dp[nt][j] - Dr[j >> 1]);   // joint: c dS
          }
        }
      }
      // second products over these 32 streamed rows (two k-steps), d as eight n-tiles
#pragma unroll
      for (int ksx = 0; ksx < 2 && grad; ++ksx) {
        const uint32_t ad[4] = {pack2(dp[2 * ksx][0], dp[2 * ksx][1]),
                                pack2(dp[2 * ksx][2], dp[2 * ksx][3]),
                                pack2(dp[2 * ksx + 1][0], dp[2 * ksx + 1][1]),
                                pack2(dp[2 * ksx + 1][2], dp[2 * ksx + 1][3])};
        const int r = 32 * h + 16 * ksx + rt;
        if constexpr (kKM) {
          const uint32_t ap[4] = {pack2(s[2 * ksx][0], s[2 * ksx][1]),
                                  pack2(s[2 * ksx][2], s[2 * ksx][3]),
                                  pack2(s[2 * ksx + 1][0], s[2 * ksx + 1][1]),
                                  pack2(s[2 * ksx + 1][2], s[2 * ksx + 1][3])};
#pragma unroll
          for (int dq = 0; dq < 4; ++dq) {
            uint32_t b[4];
            ldsm4t(b, &sm.st[buf][0][r][16 * dq + ct]);     // q rows: dk += dS^T q
            mma(acc0[2 * dq], ad, b[0], b[1]);
            mma(acc0[2 * dq + 1], ad, b[2], b[3]);
            ldsm4t(b, &sm.st[buf][1][r][16 * dq + ct]);     // g rows: dv += P^T g
            mma(acc1[2 * dq], ap, b[0], b[1]);
            mma(acc1[2 * dq + 1], ap, b[2], b[3]);
          }
        } else {
          uint32_t al[4] = {0u, 0u, 0u, 0u};
          if constexpr (kSplitDs) {
            al[0] = pack2_rest(dp[2 * ksx][0], dp[2 * ksx][1], ad[0]);
            al[1] = pack2_rest(dp[2 * ksx][2], dp[2 * ksx][3], ad[1]);
            al[2] = pack2_rest(dp[2 * ksx + 1][0], dp[2 * ksx + 1][1], ad[2]);
            al[3] = pack2_rest(dp[2 * ksx + 1][2], dp[2 * ksx + 1][3], ad[3]);
          }
#pragma unroll
          for (int dq = 0; dq < 4; ++dq) {
            uint32_t b[4];
            ldsm4t(b, &sm.st[buf][0][r][16 * dq + ct]);     // k rows: dq += dS k
            mma(acc0[2 * dq], ad, b[0], b[1]);
            mma(acc0[2 * dq + 1], ad, b[2], b[3]);
            if constexpr (kSplitDs) {
              mma(acc0[2 * dq], al, b[0], b[1]);
              mma(acc0[2 * dq + 1], al, b[2], b[3]);
            }
          }
        }
      }
    }
    __syncthreads();
  }

  if constexpr (kRS) {   // each row's sum over the quad's columns, added to D
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      rs[i] += __shfl_xor_sync(0xffffffffu, rs[i], 1);
      rs[i] += __shfl_xor_sync(0xffffffffu, rs[i], 2);
    }
    if (t == 0) {
      if (a.first) {
        if (row_g >= 0) a.Dacc[row_g] = rs[0];
        if (row_g8 >= 0) a.Dacc[row_g8] = rs[1];
      } else {
        if (row_g >= 0) atomicAdd(a.Dacc + row_g, rs[0]);
        if (row_g8 >= 0) atomicAdd(a.Dacc + row_g8, rs[1]);
      }
    }
    return;
  }
  // ---- one 16-byte atomic add per lane and n-tile: lanes t and t ^ 1 swap halves, so an
  // even t adds row g's columns 8 nt + 2 t .. +3 and an odd t row g + 8's columns
  // 8 nt + 2 t - 2 .. +1
  const bool ev = (t & 1) == 0;
  const long long row = ev ? row_g : row_g8;
  auto flush = [&](float* out, float (*acc)[4], float scale) {
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const float r0 = __shfl_xor_sync(0xffffffffu, ev ? acc[nt][2] : acc[nt][0], 1);
      const float r1 = __shfl_xor_sync(0xffffffffu, ev ? acc[nt][3] : acc[nt][1], 1);
      const float4 v = ev ? make_float4(acc[nt][0], acc[nt][1], r0, r1)
                          : make_float4(r0, r1, acc[nt][2], acc[nt][3]);
      if (row < 0) continue;
      float4* o = reinterpret_cast<float4*>(out + (size_t)row * 64 + 8 * nt + 2 * t - (ev ? 0 : 2));
      const float4 x = make_float4(scale * v.x, scale * v.y, scale * v.z, scale * v.w);
      if (a.first) *o = x;
      else atomicAdd(o, x);
    }
  };
  if constexpr (kKM) {
    if (a.dk) flush(a.dk, acc0, a.c);
    if (a.dv) flush(a.dv, acc1, 1.f);
  } else {
    if (a.dq) flush(a.dq, acc0, kJ ? 1.f : a.c);   // joint: the scale is in dS already
  }
}

}  // namespace

cudaError_t launch_bwd_pass_mma(BwdPass p, int kind, cudaStream_t st) {
  const bool key_major = kind == 1;
  const bool raw = p.bucket_off != nullptr;
  auto ceil_div = [](long long x, long long y) { return (x + y - 1) / y; };
  long long items;
  if (kind == 3) {   // joint: routed segments, every query row once, streams not split
    if (!raw || !p.first || p.n2 < 0) return cudaErrorInvalidValue;
    items = ceil_div(p.NS, kRows) + p.m;
  } else if (raw) {
    // upper bound: sum over experts of ceil(cnt_e / 64) <= NS / 64 + m (and likewise for splits)
    items = key_major ? ceil_div(p.topk, kRows) * (ceil_div(p.NS, kSplitRows) + p.m)
                      : (ceil_div(p.NS, kRows) + p.m) * ceil_div(p.topk, kSplitRows);
  } else {
    items = key_major ? ceil_div(p.nk, kRows) * ceil_div(p.nq, kSplitRows)
                      : ceil_div(p.nq, kRows) * ceil_div(p.nk, kSplitRows);
  }
  if (items <= 0) return cudaSuccess;
  if (items * p.BH >= (1LL << 31)) return cudaErrorInvalidValue;
  // a first writer must own each of its rows in one CTA: one segment per owned row (the
  // caller's promise) and a stream short enough not to be split
  if (kind != 3 && p.first &&
      (raw ? (key_major ? p.NS : p.topk) : (key_major ? p.nq : p.nk)) > kSplitRows)
    return cudaErrorInvalidValue;
  p.items = (int)items;
  for (const float* x : {p.dq, p.dk, p.dv})   // the 16-byte atomic adds
    if (reinterpret_cast<uintptr_t>(x) % 16 != 0) return cudaErrorMisalignedAddress;
  const size_t smem = sizeof(MmaSmem);
  auto kern = kind == 1   ? bwd_mma_kernel<kKeyMajor>
              : kind == 2 ? bwd_mma_kernel<kRowSums>
              : kind == 3 ? bwd_mma_kernel<kJoint>
                          : bwd_mma_kernel<kQueryMajor>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)(items * p.BH), kThreads, smem, st>>>(p);
  count_launch();
  return cudaGetLastError();
}

}  // namespace mita
