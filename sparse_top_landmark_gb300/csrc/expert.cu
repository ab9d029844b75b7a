// Step 6: one joint softmax per query over the m shared pairs and the k raw
// pairs of its routed expert, computed expert by expert.
//
// MiTA tutorial (iwxt.cn), ch. 4 steps 5-6 (paper eq. 11-12): all queries
// see the m shared pairs (q~_i, v~_i); each adds the s*k raw pairs of its
// chosen experts; the m + s*k logits (all scaled by 1/sqrt(d); on request the
// shared ones by 1/d, the official code's temperature) share one
// softmax.  The bit.fan article: queries are processed grouped by expert with
// an online softmax.  Tutorial ch. 4 also states the merge rule used when the
// shared part arrives as a partial: (Z1 o1 + Z2 o2) / (Z1 + Z2).
//
// One CTA handles one tile of (up to kQTile) queries of one expert; the tile
// is found from bucket_off (tiles of all experts of a head, in expert order).
// The expert's K/V rows are gathered once per tile into shared memory.
//
// s > 1: a query sits in s buckets.  Each (query, expert) pair then yields a
// partial over that expert's k raw pairs only -- its log-sum-exp and
// normalised output -- in one of the query's s partial slots (taken with an
// atomic counter; the slot records the bucket position).  A second kernel
// merges, per query, the shared branch's partial and the s raw partials with
// the tutorial's rule, in ascending bucket position (= ascending expert), so
// the result does not depend on which CTA took which slot.  Overlapping
// experts thus contribute duplicated rows, the literal concatenation.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace mita {
namespace {

constexpr int kQTile = 64;   // queries per CTA (one per thread)
constexpr int kRows = 32;    // KV rows staged per chunk
constexpr int kMergeWarps = 8;

__device__ __forceinline__ void put(float* p, float x) { *p = x; }
__device__ __forceinline__ void put(bf16* p, float x) { *p = __float2bfloat16_rn(x); }

using Partials = ExpertPartials;   // partial mode when .o is set

template <typename T, int D>
__global__ void __launch_bounds__(kQTile)
expert_attn_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                   const T* __restrict__ q_tilde, const float* __restrict__ v_tilde,
                   const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ bucket_off,
                   const int32_t* __restrict__ bucket_qidx, const float* __restrict__ shared_lse,
                   const float* __restrict__ shared_o, int N, int m, int topk, int s,
                   float c_shared, int routed_only, int tiles_per_bh, T* __restrict__ out,
                   Partials part, int* status) {
  __shared__ __align__(16) float ks[kRows][D];
  __shared__ __align__(16) float vs[kRows][D];
  __shared__ int rowid[kRows];
  __shared__ int s_e, s_t;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long bh = blockIdx.x / tiles_per_bh;
  const int t = blockIdx.x % tiles_per_bh;
  const int32_t* off = bucket_off + (size_t)bh * (m + 1);
  const int NS = N * s;   // bucket entries per head

  // ---- locate (expert, tile within expert) for this CTA ---------------------
  if (warp == 0) {
    int run = 0, fe = -1, ft = 0;
    for (int e0 = 0; e0 < m && fe < 0; e0 += 32) {
      const int e = e0 + lane;
      int cnt = 0;
      if (e < m) {
        const int a = off[e], b = off[e + 1];
        if (a < 0 || b > NS || b < a) flag_error(status, kDevErrBadBucket);
        else cnt = b - a;
      }
      const int nt = (cnt + kQTile - 1) / kQTile;
      const int inc = warp_incl_scan(nt);
      const int tot = __shfl_sync(0xffffffffu, inc, 31);
      if (t < run + tot) {
        const unsigned hit = __ballot_sync(0xffffffffu, run + inc > t);
        const int f = __ffs(hit) - 1;
        const int before = __shfl_sync(0xffffffffu, inc - nt, f);
        fe = e0 + f;
        ft = t - (run + before);
      }
      run += tot;
    }
    if (lane == 0) { s_e = fe; s_t = ft; }
  }
  __syncthreads();
  const int e = s_e;
  if (e < 0) return;
  const int slot = off[e] + s_t * kQTile + tid;
  bool live = slot < off[e + 1];
  int n = 0;
  if (live) {
    n = bucket_qidx[(size_t)bh * NS + slot];
    if (n < 0 || n >= N) { flag_error(status, kDevErrBadBucket); live = false; }
  }

  float qr[D];
  if (live) load_row<T, D>(q + ((size_t)bh * N + n) * D, qr);
  else {
#pragma unroll
    for (int l = 0; l < D; ++l) qr[l] = 0.f;
  }
  const float c = (float)(1.4426950408889634 / sqrt((double)D));
  float mrun = -INFINITY, lsum = 0.f;
  float acc[D];
#pragma unroll
  for (int l = 0; l < D; ++l) acc[l] = 0.f;

  auto absorb = [&](float x, const float* vr) {
    if (x > mrun) {
      const float sc = exp2f(mrun - x);
      lsum *= sc;
#pragma unroll
      for (int l = 0; l < D; ++l) acc[l] *= sc;
      mrun = x;
    }
    const float p = exp2f(x - mrun);
    lsum += p;
#pragma unroll
    for (int l = 0; l < D; ++l) acc[l] = fmaf(p, vr[l], acc[l]);
  };

  // ---- shared branch: the m pairs (q~_i, v~_i) -------------------------------
  const bool partial = part.o != nullptr;
  if (partial || routed_only) {
    // partials: merged per query afterwards; routing only: no shared pairs
  } else if (shared_o != nullptr) {
    if (live) {
      const size_t qi = (size_t)bh * N + n;
      mrun = shared_lse[qi] * 1.4426950408889634f;  // natural -> log2 units
      lsum = 1.f;
#pragma unroll
      for (int l = 0; l < D; ++l) acc[l] = shared_o[qi * D + l];
    }
  } else {
    const T* qtb = q_tilde + (size_t)bh * m * D;
    const float* vtb = v_tilde + (size_t)bh * m * D;
    for (int i0 = 0; i0 < m; i0 += kRows) {
      const int nc = min(kRows, m - i0);
      __syncthreads();
      for (int x = tid; x < nc * D; x += kQTile) {
        const int r = x / D, l = x % D;
        ks[r][l] = to_f(qtb[(size_t)(i0 + r) * D + l]);
        vs[r][l] = vtb[(size_t)(i0 + r) * D + l];
      }
      __syncthreads();
      if (!live) continue;
      for (int r = 0; r < nc; ++r) {
        float s = 0.f;
#pragma unroll
        for (int l = 0; l < D; ++l) s = fmaf(qr[l], ks[r][l], s);
        absorb(s * c_shared, vs[r]);
      }
    }
  }

  // ---- routed branch: the expert's k raw pairs ------------------------------
  const int32_t* idx = topk_idx + ((size_t)bh * m + e) * topk;
  const T* kb = k + (size_t)bh * N * D;
  const T* vb = v + (size_t)bh * N * D;
  constexpr int VEC = Vec<T>::N;
  for (int j0 = 0; j0 < topk; j0 += kRows) {
    const int nc = min(kRows, topk - j0);
    __syncthreads();
    if (tid < nc) {
      int j = idx[j0 + tid];
      if (j < 0 || j >= N) { flag_error(status, kDevErrBadIndex); j = -1; }
      rowid[tid] = j;
    }
    __syncthreads();
    for (int x = tid; x < nc * (D / VEC); x += kQTile) {
      const int r = x / (D / VEC), part = (x % (D / VEC)) * VEC;
      const int j = rowid[r];
      float xk[VEC], xv[VEC];
      if (j >= 0) {
        Vec<T>::load(kb + (size_t)j * D + part, xk);
        Vec<T>::load(vb + (size_t)j * D + part, xv);
      } else {
#pragma unroll
        for (int u = 0; u < VEC; ++u) { xk[u] = 0.f; xv[u] = 0.f; }
      }
#pragma unroll
      for (int u = 0; u < VEC; ++u) { ks[r][part + u] = xk[u]; vs[r][part + u] = xv[u]; }
    }
    __syncthreads();
    if (!live) continue;
    for (int r = 0; r < nc; ++r) {
      if (rowid[r] < 0) continue;
      float s = 0.f;
#pragma unroll
      for (int l = 0; l < D; ++l) s = fmaf(qr[l], ks[r][l], s);
      absorb(s * c, vs[r]);
    }
  }
  if (!live) return;
  const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
#pragma unroll
  for (int l = 0; l < D; ++l) acc[l] *= inv;
  const size_t qi = (size_t)bh * N + n;
  if (!partial) {
    store_row<T, D>(out + qi * D, acc);
    return;
  }
  const int ps = atomicAdd(&part.cnt[qi], 1);   // this pair's partial slot
  if (ps >= s) {
    flag_error(status, kDevErrBadBucket);
    return;
  }
  const size_t pi = qi * s + ps;
  part.lse[pi] = lsum > 0.f ? (mrun + log2f(lsum)) * 0.6931471805599453f : -INFINITY;
  part.pos[pi] = slot;
#pragma unroll
  for (int l = 0; l < D; l += 4)
    *reinterpret_cast<float4*>(part.o + pi * D + l) = make_float4(acc[l], acc[l + 1], acc[l + 2], acc[l + 3]);
}

// s > 1: out = (Z_sh o_sh + sum_t Z_t o_t) / (Z_sh + sum_t Z_t), Z = exp(lse) (the
// tutorial's branch merge).  D / 4 lanes per query, four dimensions each (16-byte loads; the
// shared output may come in bf16); every load of a query is issued before its arithmetic, and KS >= s
// slots are read, so a small KS keeps registers (and more queries in flight) for small s.
// The s partials are added in ascending bucket position (their slots were taken by atomics),
// so the result does not depend on which CTA wrote which slot.
__device__ __forceinline__ float4 load4f(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}
__device__ __forceinline__ float4 load4f(const bf16* p) {
  const uint2 w = *reinterpret_cast<const uint2*>(p);
  return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                     __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
}
__device__ __forceinline__ void store4(float* out, const float* a) {
  *reinterpret_cast<float4*>(out) = make_float4(a[0], a[1], a[2], a[3]);
}
__device__ __forceinline__ void store4(bf16* out, const float* a) {
  __nv_bfloat162 h0 = __floats2bfloat162_rn(a[0], a[1]), h1 = __floats2bfloat162_rn(a[2], a[3]);
  uint2 w;
  w.x = *reinterpret_cast<uint32_t*>(&h0);
  w.y = *reinterpret_cast<uint32_t*>(&h1);
  *reinterpret_cast<uint2*>(out) = w;
}

template <typename T, int D, int KS>
__global__ void __launch_bounds__(kMergeWarps * 32)
expert_merge_kernel(const float* __restrict__ shared_lse, const void* __restrict__ shared_o,
                    int so_bf16, Partials part, long long BHN, int s, T* __restrict__ out,
                    int* status) {
  constexpr int LPQ = D / 4;                 // lanes per query
  constexpr int QPB = kMergeWarps * 32 / LPQ;
  const int c = threadIdx.x % LPQ;
  const long long qi = (long long)blockIdx.x * QPB + threadIdx.x / LPQ;
  if (qi >= BHN) return;                     // whole query groups
  const bool sh = shared_lse != nullptr;     // routing only: no shared partial
  const int cnt = part.cnt[qi];
  float pl[KS];
  int pp[KS];
  float4 po[KS];
#pragma unroll
  for (int t = 0; t < KS; ++t) {
    pl[t] = -INFINITY;
    pp[t] = 0x7fffffff;
    po[t] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (t < s) {
      pl[t] = part.lse[qi * s + t];
      pp[t] = part.pos[qi * s + t];
      const size_t off = ((size_t)qi * s + t) * D + 4 * c;
      po[t] = load4f(part.o + off);
    }
  }
  const float lsh = sh ? shared_lse[qi] : -INFINITY;
  float4 osh = make_float4(0.f, 0.f, 0.f, 0.f);
  if (sh) {
    const size_t off = (size_t)qi * D + 4 * c;
    osh = so_bf16 ? load4f(static_cast<const bf16*>(shared_o) + off)
                  : load4f(static_cast<const float*>(shared_o) + off);
  }
  if (cnt != s) {
    if (c == 0) flag_error(status, kDevErrBadBucket);
    return;
  }
  float M = lsh;
#pragma unroll
  for (int t = 0; t < KS; ++t) M = fmaxf(M, pl[t]);
  constexpr float kL2e = 1.4426950408889634f;
  const float wsh = sh ? exp2f((lsh - M) * kL2e) : 0.f;
  float z = wsh;
  float acc[4] = {wsh * osh.x, wsh * osh.y, wsh * osh.z, wsh * osh.w};
  // rank r: the slot holding the r-th smallest bucket position
#pragma unroll
  for (int r = 0; r < KS; ++r) {
    if (r >= s) break;
    int src = -1;
#pragma unroll
    for (int t = 0; t < KS; ++t) {
      int rank = 0;
#pragma unroll
      for (int u = 0; u < KS; ++u) rank += (u < s && pp[u] < pp[t]) ? 1 : 0;
      if (t < s && rank == r) src = t;
    }
    if (src < 0) {                           // two partials claim one bucket position
      if (c == 0) flag_error(status, kDevErrBadBucket);
      return;
    }
    float wl = -INFINITY;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int t = 0; t < KS; ++t)
      if (t == src) { wl = pl[t]; o = po[t]; }
    const float w = exp2f((wl - M) * kL2e);
    z += w;
    acc[0] = fmaf(w, o.x, acc[0]);
    acc[1] = fmaf(w, o.y, acc[1]);
    acc[2] = fmaf(w, o.z, acc[2]);
    acc[3] = fmaf(w, o.w, acc[3]);
  }
  const float inv = 1.f / z;
#pragma unroll
  for (int e = 0; e < 4; ++e) acc[e] *= inv;
  store4(out + (size_t)qi * D + 4 * c, acc);
}

template <typename T, int D>
cudaError_t launch_merge_d(const float* shared_lse, const void* shared_o, int so_bf16,
                           Partials part, long long BHN, int s, T* out, int* status,
                           cudaStream_t st) {
  constexpr long long QPB = kMergeWarps * 32 / (D / 4);
  const unsigned grid = (unsigned)((BHN + QPB - 1) / QPB);
  if (s <= 2)
    expert_merge_kernel<T, D, 2><<<grid, kMergeWarps * 32, 0, st>>>(shared_lse, shared_o, so_bf16,
                                                                    part, BHN, s, out, status);
  else if (s <= 4)
    expert_merge_kernel<T, D, 4><<<grid, kMergeWarps * 32, 0, st>>>(shared_lse, shared_o, so_bf16,
                                                                    part, BHN, s, out, status);
  else
    expert_merge_kernel<T, D, kMaxRouteS><<<grid, kMergeWarps * 32, 0, st>>>(
        shared_lse, shared_o, so_bf16, part, BHN, s, out, status);
  count_launch();
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t run(const T* q, const T* k, const T* v, const T* qt, const float* vt,
                const int32_t* ti, const int32_t* off, const int32_t* qidx, const float* lse,
                const float* so, int BH, int N, int m, int topk, int s, int temp, int routed,
                void* pws, T* out, int* status, cudaStream_t st) {
  const float c_shared = (float)(1.4426950408889634 / (temp ? (double)D : sqrt((double)D)));
  const int tiles = (int)(((long long)N * s + kQTile - 1) / kQTile) + m;
  const long long blocks = (long long)BH * tiles;
  Partials part{};
  const long long BHN = (long long)BH * N;
  if (s > 1) {
    char* p = static_cast<char*>(pws);
    part.o = reinterpret_cast<float*>(p);
    p += (size_t)BHN * s * D * sizeof(float);
    part.lse = reinterpret_cast<float*>(p);
    p += (size_t)BHN * s * sizeof(float);
    part.pos = reinterpret_cast<int*>(p);
    p += (size_t)BHN * s * sizeof(int);
    part.cnt = reinterpret_cast<int*>(p);
    const cudaError_t e = cudaMemsetAsync(part.cnt, 0, (size_t)BHN * sizeof(int), st);
    if (e != cudaSuccess) return e;
  }
  expert_attn_kernel<T, D><<<(unsigned)blocks, kQTile, 0, st>>>(
      q, k, v, qt, vt, ti, off, qidx, lse, so, N, m, topk, s, c_shared, routed, tiles, out, part,
      status);
  count_launch();
  if (s > 1) {
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_merge_d<T, D>(routed ? nullptr : lse, routed ? nullptr : so, 0, part, BHN, s,
                                out, status, st);
  }
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t run_partials(const T* q, const T* k, const T* v, const int32_t* ti, const int32_t* off,
                         const int32_t* qidx, int BH, int N, int m, int topk, int s,
                         ExpertPartials part, int* status, cudaStream_t st) {
  const int tiles = (int)(((long long)N * s + kQTile - 1) / kQTile) + m;
  const cudaError_t e = cudaMemsetAsync(part.cnt, 0, (size_t)BH * N * sizeof(int), st);
  if (e != cudaSuccess) return e;
  expert_attn_kernel<T, D><<<(unsigned)((long long)BH * tiles), kQTile, 0, st>>>(
      q, k, v, q, nullptr, ti, off, qidx, nullptr, nullptr, N, m, topk, s, 0.f, 1, tiles,
      nullptr, part, status);
  count_launch();
  return cudaGetLastError();
}

}  // namespace

template <typename T>
cudaError_t launch_expert_partials(const T* q, const T* k, const T* v, const int32_t* topk_idx,
                                   const int32_t* bucket_off, const int32_t* bucket_qidx, int BH,
                                   int N, int d, int m, int topk, int s, ExpertPartials part,
                                   int* status, cudaStream_t st) {
  switch (d) {
    case 16: return run_partials<T, 16>(q, k, v, topk_idx, bucket_off, bucket_qidx, BH, N, m, topk, s, part, status, st);
    case 32: return run_partials<T, 32>(q, k, v, topk_idx, bucket_off, bucket_qidx, BH, N, m, topk, s, part, status, st);
    case 64: return run_partials<T, 64>(q, k, v, topk_idx, bucket_off, bucket_qidx, BH, N, m, topk, s, part, status, st);
    case 128: return run_partials<T, 128>(q, k, v, topk_idx, bucket_off, bucket_qidx, BH, N, m, topk, s, part, status, st);
    default: return cudaErrorInvalidValue;
  }
}
template cudaError_t launch_expert_partials<float>(const float*, const float*, const float*,
                                                   const int32_t*, const int32_t*, const int32_t*,
                                                   int, int, int, int, int, int, ExpertPartials,
                                                   int*, cudaStream_t);
template cudaError_t launch_expert_partials<bf16>(const bf16*, const bf16*, const bf16*,
                                                  const int32_t*, const int32_t*, const int32_t*,
                                                  int, int, int, int, int, int, ExpertPartials,
                                                  int*, cudaStream_t);

size_t expert_partials_ws_bytes(int BH, int N, int d, int s) {
  if (s <= 0) return 0;
  const size_t r = (size_t)BH * N;
  return r * s * d * sizeof(float) + 2 * r * s * sizeof(float) + r * sizeof(int);
}

ExpertPartials carve_expert_partials(void* ws, int BH, int N, int d, int s) {
  const size_t r = (size_t)BH * N;
  char* p = static_cast<char*>(ws);
  ExpertPartials part{};
  part.o = reinterpret_cast<float*>(p);
  p += r * s * d * sizeof(float);
  part.lse = reinterpret_cast<float*>(p);
  p += r * s * sizeof(float);
  part.pos = reinterpret_cast<int*>(p);
  p += r * s * sizeof(int);
  part.cnt = reinterpret_cast<int*>(p);
  return part;
}

template <typename T>
cudaError_t launch_expert_merge(const float* shared_lse, const void* shared_o, int so_bf16,
                                ExpertPartials part, int BH, int N, int d, int s, T* out,
                                int* status, cudaStream_t st) {
  const long long BHN = (long long)BH * N;
  switch (d) {
    case 16: return launch_merge_d<T, 16>(shared_lse, shared_o, so_bf16, part, BHN, s, out, status, st);
    case 32: return launch_merge_d<T, 32>(shared_lse, shared_o, so_bf16, part, BHN, s, out, status, st);
    case 64: return launch_merge_d<T, 64>(shared_lse, shared_o, so_bf16, part, BHN, s, out, status, st);
    case 128: return launch_merge_d<T, 128>(shared_lse, shared_o, so_bf16, part, BHN, s, out, status, st);
    default: return cudaErrorInvalidValue;
  }
}
template cudaError_t launch_expert_merge<float>(const float*, const void*, int, ExpertPartials,
                                                int, int, int, int, float*, int*, cudaStream_t);
template cudaError_t launch_expert_merge<bf16>(const float*, const void*, int, ExpertPartials,
                                               int, int, int, int, bf16*, int*, cudaStream_t);

template <typename T>
cudaError_t launch_expert_attn(const T* q, const T* k, const T* v, const T* q_tilde,
                               const float* v_tilde, const int32_t* topk_idx,
                               const int32_t* bucket_off, const int32_t* bucket_qidx,
                               const float* shared_lse, const float* shared_o, int BH, int N,
                               int d, int m, int topk, int s, void* ws, T* out, int* status,
                               cudaStream_t st, int shared_temp, int routed_only) {
  if (s < 1 || (s > 1 && (ws == nullptr ||
                          (!routed_only && (shared_lse == nullptr || shared_o == nullptr)))))
    return cudaErrorInvalidValue;
#define MITA_EXPERT_CASE(DD)                                                                 \
  case DD:                                                                                   \
    return run<T, DD>(q, k, v, q_tilde, v_tilde, topk_idx, bucket_off, bucket_qidx,          \
                      shared_lse, shared_o, BH, N, m, topk, s, shared_temp, routed_only, ws,   \
                      out, status, st);
  switch (d) {
    MITA_EXPERT_CASE(16)
    MITA_EXPERT_CASE(32)
    MITA_EXPERT_CASE(64)
    MITA_EXPERT_CASE(128)
    default: return cudaErrorInvalidValue;
  }
#undef MITA_EXPERT_CASE
}

template cudaError_t launch_expert_attn<float>(const float*, const float*, const float*,
                                               const float*, const float*, const int32_t*,
                                               const int32_t*, const int32_t*, const float*,
                                               const float*, int, int, int, int, int, int, void*,
                                               float*, int*, cudaStream_t, int, int);
template cudaError_t launch_expert_attn<bf16>(const bf16*, const bf16*, const bf16*, const bf16*,
                                              const float*, const int32_t*, const int32_t*,
                                              const int32_t*, const float*, const float*, int,
                                              int, int, int, int, int, void*, bf16*, int*,
                                              cudaStream_t, int, int);

// Dense softmax attention through the same kernel: per head one expert holding every key
// (identity index list), every query in its bucket, no shared pairs.
namespace {
__global__ void __launch_bounds__(256)
dense_index_kernel(int BH, int N, int32_t* __restrict__ idx, int32_t* __restrict__ off) {
  const long long nq = (long long)BH * N;
  for (long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x; t < nq;
       t += (long long)gridDim.x * blockDim.x) {
    idx[t] = (int32_t)(t % N);
    if (t % N == 0) {
      off[2 * (t / N)] = 0;
      off[2 * (t / N) + 1] = N;
    }
  }
}
}  // namespace

size_t dense_simt_ws_bytes(int BH, int N) {
  return ((size_t)BH * N * 4 + 255) / 256 * 256 + (size_t)BH * 2 * 4;
}

template <typename T>
cudaError_t launch_dense_attn(const T* q, const T* k, const T* v, int BH, int N, int d, void* ws,
                              T* out, int* status, cudaStream_t st) {
  int32_t* idx = static_cast<int32_t*>(ws);
  int32_t* off = reinterpret_cast<int32_t*>(static_cast<char*>(ws) +
                                            ((size_t)BH * N * 4 + 255) / 256 * 256);
  const long long nq = (long long)BH * N;
  dense_index_kernel<<<(unsigned)std::min<long long>((nq + 255) / 256, 4096), 256, 0, st>>>(
      BH, N, idx, off);
  count_launch();
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // the identity list is both the expert's key list ([BH, 1, N]) and the bucket ([BH, N])
  return launch_expert_attn<T>(q, k, v, q, nullptr, idx, off, idx, nullptr, nullptr, BH, N, d, 1,
                               N, 1, nullptr, out, status, st, 0, 1);
}

template cudaError_t launch_dense_attn<float>(const float*, const float*, const float*, int, int,
                                              int, void*, float*, int*, cudaStream_t);
template cudaError_t launch_dense_attn<bf16>(const bf16*, const bf16*, const bf16*, int, int, int,
                                             void*, bf16*, int*, cudaStream_t);

}  // namespace mita
