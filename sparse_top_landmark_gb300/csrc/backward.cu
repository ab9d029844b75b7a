// Backward pass of the MiTA forward with the selections held constant.
//
// The pages train MiTA end to end (MiTA tutorial ch. 7 table 5, LRA; the
// bit.fan article's LRA section) but give no gradient through the selections.
// Reading: every landmark's top-k key set and every query's top-s landmarks are
// constants (top-k and argmax are piecewise constant) and q~'s rounding to the
// input dtype passes the gradient straight through.  With
//   q~ = pool(Q);  A = softmax(q~ K^T c);  v~ = A V            (tutorial ch. 4 steps 1-3)
//   l_n = [q_n.q~_i c_sh]_i ++ [q_n.k_j c]_j;  o_n = softmax(l_n) . [v~; V_rows]  (steps 5-6)
// (c = 1/sqrt(d), c_sh = c or 1/d) and dO the upstream gradient:
//   D_n = dO_n . o_n;  for each entry e of query n:  p = exp(l - lse_n),
//   ds = p (dO_n . val_e - D_n);  dq_n += ds key_e c_e;  dkey_e += ds q_n c_e;  dval_e += p dO_n
// and through v~ = A V, with dv~ from the shared entries:
//   dv_j += sum_i A_ij dv~_i;  dS_ij = A_ij (dv~_i . v_j - dv~_i . v~_i);
//   dk_j += sum_i dS_ij q~_i c;  dq~_i += sum_j dS_ij k_j c;  dq_t += dq~_i / |window_i|.
//
// bf16 inputs with d = 64 run the three gradient passes (raw, shared, through v~) on the
// tensor cores (backward_mma.cu: row-sum, query-major and key-major launches per pass,
// after bwd_lse_kernel, which forms lse_n alone: those passes sum D_n as P dP themselves);
// every other shape runs these SIMT kernels (fp32, gradients accumulated with atomics into
// fp32 buffers):
//   bwd_stats_kernel     per query: lse_n and D_n from the shared partial and the s raw
//                        partials (the forward's own kernels recompute those);
//   (each landmark's softmax normaliser ln sum_j exp(q~_i . k_j c) comes from the
//    landmark stage, which forms it while merging v~);
//   bwd_raw_kernel       per 64 bucket entries of one expert (its k rows staged 32 at a
//                        time): dq, and the chunk's dK / dV as dS^T Q and P^T dO;
//   bwd_shared_kernel    per 64 queries (landmarks staged 32 at a time): dq, dq~, dv~;
//   bwd_vtilde_kernel    per 64 keys (landmarks staged 32 at a time): dk, dv, dq~;
//   bwd_pool_gather_kernel  per token: the sum of dq~ / |window| over the windows holding it
//                        (bwd_pool_kernel, per landmark with atomics, for grids whose window
//                        arithmetic would not fit 32 bits).
#include <algorithm>
#include <cmath>
#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace mita {
namespace {

constexpr int kT = 64;       // rows (queries or keys) per CTA, one per thread
constexpr int kC = 32;       // staged rows per chunk
constexpr float kL2e = 1.4426950408889634f;

// ---- per-query statistics of the joint softmax -----------------------------------------
template <int D>
__global__ void __launch_bounds__(256)
bwd_stats_kernel(const float* __restrict__ sh_lse, const float* __restrict__ sh_o,
                 ExpertPartials part, long long BHN, int s, const void* __restrict__ dout,
                 int dout_bf16, float* __restrict__ lse, float* __restrict__ Dn, int* status) {
  const int lane = threadIdx.x & 31;
  const long long qi = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (qi >= BHN) return;
  if (part.cnt[qi] != s) {
    if (lane == 0) flag_error(status, kDevErrBadBucket);
    return;
  }
  float pl = -INFINITY;
  if (lane < s) pl = part.lse[qi * s + lane];
  const bool sh = sh_lse != nullptr;
  float M = sh ? sh_lse[qi] : -INFINITY;
  for (int t = 0; t < s; ++t) M = fmaxf(M, __shfl_sync(0xffffffffu, pl, t));
  constexpr int PER = (D + 31) / 32;
  const float wsh = sh ? exp2f((sh_lse[qi] - M) * kL2e) : 0.f;
  float z = wsh, acc[PER];
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int l = lane + 32 * j;
    acc[j] = (sh && l < D) ? wsh * sh_o[qi * D + l] : 0.f;
  }
  for (int t = 0; t < s; ++t) {
    const float w = exp2f((__shfl_sync(0xffffffffu, pl, t) - M) * kL2e);
    z += w;
    const float* o = part.o + ((size_t)qi * s + t) * D;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int l = lane + 32 * j;
      if (l < D) acc[j] = fmaf(w, o[l], acc[j]);
    }
  }
  float dd = 0.f;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int l = lane + 32 * j;
    if (l < D) {
      const float g = dout_bf16 ? to_f(static_cast<const bf16*>(dout)[qi * D + l])
                                : static_cast<const float*>(dout)[qi * D + l];
      dd = fmaf(g, acc[j] / z, dd);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) dd += __shfl_xor_sync(0xffffffffu, dd, o);
  if (lane == 0) {
    lse[qi] = M + logf(z);
    Dn[qi] = dd;
  }
}

// per query (one thread each): lse_n only, for the tensor-core passes that sum D themselves
__global__ void __launch_bounds__(256)
bwd_lse_kernel(const float* __restrict__ sh_lse, ExpertPartials part, long long BHN, int s,
               float* __restrict__ lse, int* status) {
  const long long qi = (long long)blockIdx.x * 256 + threadIdx.x;
  if (qi >= BHN) return;
  if (part.cnt[qi] != s) {
    flag_error(status, kDevErrBadBucket);
    return;
  }
  float M = sh_lse ? sh_lse[qi] : -INFINITY;
  for (int t = 0; t < s; ++t) M = fmaxf(M, part.lse[qi * s + t]);
  float z = sh_lse ? exp2f((sh_lse[qi] - M) * kL2e) : 0.f;
  for (int t = 0; t < s; ++t) z += exp2f((part.lse[qi * s + t] - M) * kL2e);
  lse[qi] = M + logf(z);
}

// Shared-memory tiles of one CTA: its kT rows (q or k, and dO or v), and kC staged rows.
template <int D>
struct BwdSmem {
  float a[kT][D + 1];     // this CTA's rows: q (raw / shared) or k (v~ pass)
  float g[kT][D + 1];     // dO (raw / shared) or v (v~ pass)
  float ck[kC][D + 1];    // staged keys: k rows, q~ rows, or q~ rows
  float cv[kC][D + 1];    // staged values: v rows, v~ rows, or dv~ rows
  float P[kT][kC + 1];    // softmax weights of the chunk
  float S[kT][kC + 1];    // their logit gradients
  int rowid[kC];
};

// After a chunk's P and S are in shared memory: d(keys) = c * S^T A and d(values) = P^T G
// for the kC staged rows, added with atomics at rows dst_k / dst_v (row r -> base + id*D).
template <int D>
__device__ __forceinline__ void chunk_outer(BwdSmem<D>& sm, int nc, float c, float* dkey_base,
                                           float* dval_base, int tid) {
  for (int x = tid; x < nc * D; x += kT) {
    const int r = x / D, l = x % D;
    const int id = sm.rowid[r];
    float dk = 0.f, dv = 0.f;
#pragma unroll 8
    for (int n = 0; n < kT; ++n) {
      dk = fmaf(sm.S[n][r], sm.a[n][l], dk);
      dv = fmaf(sm.P[n][r], sm.g[n][l], dv);
    }
    if (id >= 0) {
      if (dkey_base) atomicAdd(dkey_base + (size_t)id * D + l, dk * c);
      if (dval_base) atomicAdd(dval_base + (size_t)id * D + l, dv);
    }
  }
}

// ---- raw entries, expert-grouped -----------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(kT)
bwd_raw_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
               const T* __restrict__ dout, const int32_t* __restrict__ topk_idx,
               const int32_t* __restrict__ bucket_off, const int32_t* __restrict__ bucket_qidx,
               const float* __restrict__ lse, const float* __restrict__ Dn, int N, int m, int topk,
               int s, int tiles_per_bh, float* __restrict__ dq, float* __restrict__ dk,
               float* __restrict__ dv, int* status) {
  extern __shared__ __align__(16) unsigned char smraw[];
  BwdSmem<D>& sm = *reinterpret_cast<BwdSmem<D>*>(smraw);
  __shared__ int s_e, s_t;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long bh = blockIdx.x / tiles_per_bh;
  const int t = blockIdx.x % tiles_per_bh;
  const int32_t* off = bucket_off + (size_t)bh * (m + 1);
  const int NS = N * s;
  if (warp == 0) {   // locate (expert, tile of the expert)
    int run = 0, fe = -1, ft = 0;
    for (int e0 = 0; e0 < m && fe < 0; e0 += 32) {
      const int e = e0 + lane;
      int cnt = 0;
      if (e < m) {
        const int a = off[e], b = off[e + 1];
        if (a < 0 || b > NS || b < a) flag_error(status, kDevErrBadBucket);
        else cnt = b - a;
      }
      const int nt = (cnt + kT - 1) / kT;
      const int inc = warp_incl_scan(nt);
      const int tot = __shfl_sync(0xffffffffu, inc, 31);
      if (t < run + tot) {
        const unsigned hit = __ballot_sync(0xffffffffu, run + inc > t);
        const int f = __ffs(hit) - 1;
        fe = e0 + f;
        ft = t - (run + __shfl_sync(0xffffffffu, inc - nt, f));
      }
      run += tot;
    }
    if (lane == 0) { s_e = fe; s_t = ft; }
  }
  __syncthreads();
  const int e = s_e;
  if (e < 0) return;
  const int slot = off[e] + s_t * kT + tid;
  bool live = slot < off[e + 1];
  int n = 0;
  if (live) {
    n = bucket_qidx[(size_t)bh * NS + slot];
    if (n < 0 || n >= N) { flag_error(status, kDevErrBadBucket); live = false; }
  }
  const size_t qi = (size_t)bh * N + n;
  float L = 0.f, Dq = 0.f;
  if (live) {
    float x[D];
    load_row<T, D>(q + qi * D, x);
#pragma unroll
    for (int l = 0; l < D; ++l) sm.a[tid][l] = x[l];
    load_row<T, D>(dout + qi * D, x);
#pragma unroll
    for (int l = 0; l < D; ++l) sm.g[tid][l] = x[l];
    L = lse[qi];
    Dq = Dn[qi];
  } else {
    for (int l = 0; l < D; ++l) { sm.a[tid][l] = 0.f; sm.g[tid][l] = 0.f; }
  }
  const float c = rsqrtf((float)D);
  float dqa[D];
#pragma unroll
  for (int l = 0; l < D; ++l) dqa[l] = 0.f;
  const int32_t* idx = topk_idx + ((size_t)bh * m + e) * topk;
  const T* kb = k + (size_t)bh * N * D;
  const T* vb = v + (size_t)bh * N * D;
  for (int j0 = 0; j0 < topk; j0 += kC) {
    const int nc = min(kC, topk - j0);
    __syncthreads();
    if (tid < kC) {
      int j = -1;
      if (tid < nc) {
        j = idx[j0 + tid];
        if (j < 0 || j >= N) { flag_error(status, kDevErrBadIndex); j = -1; }
      }
      sm.rowid[tid] = j;
    }
    __syncthreads();
    for (int x = tid; x < nc * D; x += kT) {
      const int r = x / D, l = x % D;
      const int j = sm.rowid[r];
      sm.ck[r][l] = j >= 0 ? to_f(kb[(size_t)j * D + l]) : 0.f;
      sm.cv[r][l] = j >= 0 ? to_f(vb[(size_t)j * D + l]) : 0.f;
    }
    __syncthreads();
    for (int r = 0; r < kC; ++r) {
      float p = 0.f, ds = 0.f;
      if (live && r < nc && sm.rowid[r] >= 0) {
        float a = 0.f, b = 0.f;
#pragma unroll
        for (int l = 0; l < D; ++l) {
          a = fmaf(sm.a[tid][l], sm.ck[r][l], a);
          b = fmaf(sm.g[tid][l], sm.cv[r][l], b);
        }
        p = __expf(a * c - L);
        ds = p * (b - Dq);
#pragma unroll
        for (int l = 0; l < D; ++l) dqa[l] = fmaf(ds * c, sm.ck[r][l], dqa[l]);
      }
      sm.P[tid][r] = p;
      sm.S[tid][r] = ds;
    }
    __syncthreads();
    chunk_outer<D>(sm, nc, c, dk + (size_t)bh * N * D, dv + (size_t)bh * N * D, tid);
  }
  if (live) {
#pragma unroll
    for (int l = 0; l < D; ++l) atomicAdd(dq + qi * D + l, dqa[l]);
  }
}

// ---- shared entries, query-major ------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(kT)
bwd_shared_kernel(const T* __restrict__ q, const T* __restrict__ dout,
                  const T* __restrict__ q_tilde, const float* __restrict__ v_tilde,
                  const float* __restrict__ lse, const float* __restrict__ Dn, int N, int m,
                  float c_sh, int tiles_per_bh, float* __restrict__ dq, float* __restrict__ dqt,
                  float* __restrict__ dvt) {
  extern __shared__ __align__(16) unsigned char smraw[];
  BwdSmem<D>& sm = *reinterpret_cast<BwdSmem<D>*>(smraw);
  const int tid = threadIdx.x;
  const long long bh = blockIdx.x / tiles_per_bh;
  const int n = (blockIdx.x % tiles_per_bh) * kT + tid;
  const bool live = n < N;
  const size_t qi = (size_t)bh * N + n;
  float L = 0.f, Dq = 0.f;
  if (live) {
    float x[D];
    load_row<T, D>(q + qi * D, x);
#pragma unroll
    for (int l = 0; l < D; ++l) sm.a[tid][l] = x[l];
    load_row<T, D>(dout + qi * D, x);
#pragma unroll
    for (int l = 0; l < D; ++l) sm.g[tid][l] = x[l];
    L = lse[qi];
    Dq = Dn[qi];
  } else {
    for (int l = 0; l < D; ++l) { sm.a[tid][l] = 0.f; sm.g[tid][l] = 0.f; }
  }
  float dqa[D];
#pragma unroll
  for (int l = 0; l < D; ++l) dqa[l] = 0.f;
  for (int i0 = 0; i0 < m; i0 += kC) {
    const int nc = min(kC, m - i0);
    __syncthreads();
    if (tid < kC) sm.rowid[tid] = tid < nc ? i0 + tid : -1;
    for (int x = tid; x < nc * D; x += kT) {
      const int r = x / D, l = x % D;
      sm.ck[r][l] = to_f(q_tilde[((size_t)bh * m + i0 + r) * D + l]);
      sm.cv[r][l] = v_tilde[((size_t)bh * m + i0 + r) * D + l];
    }
    __syncthreads();
    for (int r = 0; r < kC; ++r) {
      float p = 0.f, ds = 0.f;
      if (live && r < nc) {
        float a = 0.f, b = 0.f;
#pragma unroll
        for (int l = 0; l < D; ++l) {
          a = fmaf(sm.a[tid][l], sm.ck[r][l], a);
          b = fmaf(sm.g[tid][l], sm.cv[r][l], b);
        }
        p = __expf(a * c_sh - L);
        ds = p * (b - Dq);
#pragma unroll
        for (int l = 0; l < D; ++l) dqa[l] = fmaf(ds * c_sh, sm.ck[r][l], dqa[l]);
      }
      sm.P[tid][r] = p;
      sm.S[tid][r] = ds;
    }
    __syncthreads();
    chunk_outer<D>(sm, nc, c_sh, dqt + (size_t)bh * m * D, dvt + (size_t)bh * m * D, tid);
  }
  if (live) {
#pragma unroll
    for (int l = 0; l < D; ++l) atomicAdd(dq + qi * D + l, dqa[l]);
  }
}

// ---- through v~ = A V, key-major ------------------------------------------------------------
// per landmark: cvt_i = dv~_i . v~_i
__global__ void __launch_bounds__(256)
bwd_vt_dot_kernel(const float* __restrict__ dvt, const float* __restrict__ v_tilde, long long rows,
                  int D, float* __restrict__ cvt) {
  const int lane = threadIdx.x & 31;
  const long long r = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (r >= rows) return;
  float a = 0.f;
  for (int l = lane; l < D; l += 32) a = fmaf(dvt[r * D + l], v_tilde[r * D + l], a);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
  if (lane == 0) cvt[r] = a;
}

template <typename T, int D>
__global__ void __launch_bounds__(kT)
bwd_vtilde_kernel(const T* __restrict__ k, const T* __restrict__ v, const T* __restrict__ q_tilde,
                  const float* __restrict__ dvt, const float* __restrict__ lseA,
                  const float* __restrict__ cvt, int N, int m, int tiles_per_bh,
                  float* __restrict__ dk, float* __restrict__ dv, float* __restrict__ dqt) {
  extern __shared__ __align__(16) unsigned char smraw[];
  BwdSmem<D>& sm = *reinterpret_cast<BwdSmem<D>*>(smraw);
  __shared__ float s_lse[kC], s_c[kC];
  const int tid = threadIdx.x;
  const long long bh = blockIdx.x / tiles_per_bh;
  const int j = (blockIdx.x % tiles_per_bh) * kT + tid;
  const bool live = j < N;
  const size_t kj = (size_t)bh * N + j;
  if (live) {
    float x[D];
    load_row<T, D>(k + kj * D, x);
#pragma unroll
    for (int l = 0; l < D; ++l) sm.a[tid][l] = x[l];
    load_row<T, D>(v + kj * D, x);
#pragma unroll
    for (int l = 0; l < D; ++l) sm.g[tid][l] = x[l];
  } else {
    for (int l = 0; l < D; ++l) { sm.a[tid][l] = 0.f; sm.g[tid][l] = 0.f; }
  }
  const float c = rsqrtf((float)D);
  float dka[D], dva[D];
#pragma unroll
  for (int l = 0; l < D; ++l) { dka[l] = 0.f; dva[l] = 0.f; }
  for (int i0 = 0; i0 < m; i0 += kC) {
    const int nc = min(kC, m - i0);
    __syncthreads();
    if (tid < kC) {
      sm.rowid[tid] = tid < nc ? i0 + tid : -1;
      s_lse[tid] = tid < nc ? lseA[(size_t)bh * m + i0 + tid] : 0.f;
      s_c[tid] = tid < nc ? cvt[(size_t)bh * m + i0 + tid] : 0.f;
    }
    for (int x = tid; x < nc * D; x += kT) {
      const int r = x / D, l = x % D;
      sm.ck[r][l] = to_f(q_tilde[((size_t)bh * m + i0 + r) * D + l]);
      sm.cv[r][l] = dvt[((size_t)bh * m + i0 + r) * D + l];
    }
    __syncthreads();
    for (int r = 0; r < kC; ++r) {
      float ds = 0.f;
      if (live && r < nc) {
        float a = 0.f, b = 0.f;
#pragma unroll
        for (int l = 0; l < D; ++l) {
          a = fmaf(sm.a[tid][l], sm.ck[r][l], a);   // k_j . q~_i
          b = fmaf(sm.g[tid][l], sm.cv[r][l], b);   // v_j . dv~_i
        }
        const float aw = __expf(a * c - s_lse[r]);   // A_ij
        ds = aw * (b - s_c[r]);
#pragma unroll
        for (int l = 0; l < D; ++l) {
          dva[l] = fmaf(aw, sm.cv[r][l], dva[l]);
          dka[l] = fmaf(ds * c, sm.ck[r][l], dka[l]);
        }
      }
      sm.S[tid][r] = ds;
      sm.P[tid][r] = 0.f;
    }
    __syncthreads();
    // dq~_i += c * sum_j dS_ij k_j   (no value-side term here)
    chunk_outer<D>(sm, nc, c, dqt + (size_t)bh * m * D, nullptr, tid);
  }
  if (live) {
#pragma unroll
    for (int l = 0; l < D; ++l) {
      atomicAdd(dk + kj * D + l, dka[l]);
      atomicAdd(dv + kj * D + l, dva[l]);
    }
  }
}

// ---- pooling: dq_t += dq~_i / |window_i| ---------------------------------------------------
__global__ void __launch_bounds__(128)
bwd_pool_kernel(const float* __restrict__ dqt, int N, int D, int grid_h, int grid_w, int mh,
                int mw, float* __restrict__ dq) {
  const int m = mh * mw;
  const long long flat = blockIdx.x;
  const int i = (int)(flat % m);
  const long long bh = flat / m;
  int r0, r1, c0, c1;
  adaptive_window(i / mw, grid_h, mh, &r0, &r1);
  adaptive_window(i % mw, grid_w, mw, &c0, &c1);
  const int nc = c1 - c0, cnt = (r1 - r0) * nc;
  const float inv = 1.f / (float)cnt;
  for (int x = threadIdx.x; x < cnt * D; x += blockDim.x) {
    const int t = x / D, l = x % D;
    const size_t tok = (size_t)(r0 + t / nc) * grid_w + c0 + t % nc;
    atomicAdd(dq + ((size_t)bh * N + tok) * D + l, dqt[flat * D + l] * inv);
  }
}

// The same as a gather: per (token, 4 columns), the sum over the windows holding the token,
// added to dq with one read-modify-write (no other launch writes dq then).  kEven: every
// window along an axis has in / out tokens, so token r lies in window r / (in / out) alone;
// else adaptive windows, which along each axis start at window floor(r * out / in) and
// overlap by at most one token (32-bit index arithmetic; the host checks it fits).
template <bool kEven>
__global__ void __launch_bounds__(256)
bwd_pool_gather_kernel(const float* __restrict__ dqt, long long BH, int N, int D, int grid_h,
                       int grid_w, int mh, int mw, float* __restrict__ dq) {
  const int D4 = D / 4;
  const long long x = (long long)blockIdx.x * 256 + threadIdx.x;
  if (x >= BH * N * D4) return;
  const long long tok = x / D4;
  const int c4 = (int)(x % D4);
  const long long bh = tok / N;
  const unsigned n = (unsigned)(tok - bh * N), r = n / (unsigned)grid_w, cc = n - r * grid_w;
  const float* base = dqt + (size_t)bh * mh * mw * D;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  auto add = [&](unsigned i, unsigned j, float inv) {
    const float4 gq = reinterpret_cast<const float4*>(base + ((size_t)i * mw + j) * D)[c4];
    acc.x = fmaf(gq.x, inv, acc.x); acc.y = fmaf(gq.y, inv, acc.y);
    acc.z = fmaf(gq.z, inv, acc.z); acc.w = fmaf(gq.w, inv, acc.w);
  };
  if constexpr (kEven) {
    const unsigned wh = (unsigned)(grid_h / mh), ww = (unsigned)(grid_w / mw);
    add(r / wh, cc / ww, 1.f / (float)(wh * ww));
  } else {
    const unsigned uh = grid_h, uw = grid_w, umh = mh, umw = mw;
    for (unsigned i = r * umh / uh; i < umh; ++i) {
      const unsigned r0 = i * uh / umh, r1 = ((i + 1) * uh + umh - 1) / umh;
      if (r0 > r) break;
      if (r >= r1) continue;
      for (unsigned j = cc * umw / uw; j < umw; ++j) {
        const unsigned c0 = j * uw / umw, c1 = ((j + 1) * uw + umw - 1) / umw;
        if (c0 > cc) break;
        if (cc >= c1) continue;
        add(i, j, 1.f / (float)((r1 - r0) * (c1 - c0)));
      }
    }
  }
  float4* o = reinterpret_cast<float4*>(dq + (size_t)tok * D) + c4;
  float4 v = *o;
  v.x += acc.x; v.y += acc.y; v.z += acc.z; v.w += acc.w;
  *o = v;
}
void launch_pool_grad(const float* dqt, int BH, int N, int D, int gh, int gw, int mh, int mw,
                      float* dq, cudaStream_t st) {
  // the adaptive form's products (index + 1) * extent stay below 2^32; dq is 16-byte aligned
  // (the entry point checks every buffer)
  const bool fits = ((long long)gh + 1) * (mh + 1) < (1LL << 32) &&
                    ((long long)gw + 1) * (mw + 1) < (1LL << 32);
  const bool even = gh % mh == 0 && gw % mw == 0;
  if (even || fits) {
    const long long n = (long long)BH * N * (D / 4);
    auto kern = even ? bwd_pool_gather_kernel<true> : bwd_pool_gather_kernel<false>;
    kern<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(dqt, BH, N, D, gh, gw, mh, mw, dq);
  } else {
    bwd_pool_kernel<<<(unsigned)((long long)BH * mh * mw), 128, 0, st>>>(dqt, N, D, gh, gw, mh, mw,
                                                                       dq);
  }
  count_launch();
}

template <int D>
size_t smem_bytes() { return sizeof(BwdSmem<D>); }

__global__ void __launch_bounds__(256)
to_bf16_kernel(const float* __restrict__ x, long long n, bf16* __restrict__ y) {
  for (long long i = (long long)blockIdx.x * 256 + threadIdx.x; i < n; i += (long long)gridDim.x * 256)
    y[i] = __float2bfloat16_rn(x[i]);
}
cudaError_t to_bf16(const float* x, long long n, bf16* y, cudaStream_t st) {
  const long long blocks = std::min<long long>((n + 255) / 256, 4096);
  to_bf16_kernel<<<(unsigned)std::max<long long>(blocks, 1), 256, 0, st>>>(x, n, y);
  count_launch();
  return cudaGetLastError();
}

// The gradient passes on the tensor cores (bf16, d = 64), after bwd_lse.  Each query's D
// (and each landmark's dv~ . v~) is summed as P dP over the same bf16 operands the gradient
// launches use (launch kind 2), so the dS of a row sum to zero up to fp32 rounding.
// Order: routed and shared row sums, dq (routed, shared) -- with s = 1 one joint launch for
// these four -- dq~ / dv~ (shared key-major), the pass through v~ (its row sums, dq~, then
// dk / dv), the routed dk / dv last, the pooling gradient.  A launch that is the first writer of rows it alone owns stores them (`first`),
// which saves clearing dq (the routed query-major launch with s = 1 and an unsplit top-k
// list), dk and dv (the v~ pass's key-major launch, before the routed one adds to them) and
// D (the routed row sums).
cudaError_t run_mma(const BwdArgs<bf16>& A, cudaStream_t st) {
  const float c = 0.125f;   // 1 / sqrt(64)
  const long long rows = (long long)A.BH * A.m;
  const size_t gbytes = (size_t)A.BH * A.N * 64 * sizeof(float);
  const bool joint = A.s == 1 && !A.routed;                    // a query's whole softmax per CTA
  const bool q_first = joint || (A.s == 1 && A.topk <= kBwdSplitRows);   // one routed segment
  const bool kv_first = !A.routed && A.m <= kBwdSplitRows;     // the v~ pass owns every key once
  cudaError_t e;
  if (!q_first && (e = cudaMemsetAsync(A.dq, 0, gbytes, st)) != cudaSuccess) return e;
  if (!kv_first) {
    if ((e = cudaMemsetAsync(A.dk, 0, gbytes, st)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(A.dv, 0, gbytes, st)) != cudaSuccess) return e;
  }
  if (!q_first &&
      (e = cudaMemsetAsync(A.Dn, 0, (size_t)A.BH * A.N * sizeof(float), st)) != cudaSuccess)
    return e;
  // routed pairs: each expert's bucket entries against its top-k rows
  BwdPass p{};
  p.q = A.q; p.g = A.dout; p.k = A.k; p.v = A.v; p.L = A.lse; p.D = A.Dn; p.Dacc = A.Dn;
  p.dq = A.dq; p.dk = A.dk; p.dv = A.dv; p.c = c; p.BH = A.BH;
  p.bucket_off = A.bucket_off; p.bucket_qidx = A.bucket_qidx; p.topk_idx = A.topk_idx;
  p.N = A.N; p.m = A.m; p.topk = A.topk; p.NS = A.N * A.s; p.status = A.status;
  // shared pairs: every query against the m landmarks (q~, v~) -> dq, dq~, dv~
  BwdPass sp{};
  sp.q = A.q; sp.g = A.dout; sp.k = A.q_tilde; sp.v = A.vt16; sp.L = A.lse; sp.D = A.Dn;
  sp.Dacc = A.Dn; sp.dq = A.dq; sp.dk = A.dqt; sp.dv = A.dvt; sp.c = A.c_sh; sp.BH = A.BH;
  sp.nq = A.N; sp.nk = A.m; sp.status = A.status;
  if (!A.routed && (e = to_bf16(A.v_tilde, rows * 64, A.vt16, st)) != cudaSuccess) return e;
  if (joint) {   // both passes' D and dq in one launch
    BwdPass jp = p;
    jp.k2 = A.q_tilde; jp.v2 = A.vt16; jp.c2 = A.c_sh; jp.n2 = A.m; jp.first = 1;
    if ((e = launch_bwd_pass_mma(jp, 3, st)) != cudaSuccess) return e;
  } else {
    p.first = q_first;
    if ((e = launch_bwd_pass_mma(p, 2, st)) != cudaSuccess) return e;
    if (!A.routed && (e = launch_bwd_pass_mma(sp, 2, st)) != cudaSuccess) return e;
    if ((e = launch_bwd_pass_mma(p, 0, st)) != cudaSuccess) return e;
    p.first = 0;
  }
  if (!A.routed) {
    if (!joint && (e = launch_bwd_pass_mma(sp, 0, st)) != cudaSuccess) return e;
    if ((e = launch_bwd_pass_mma(sp, 1, st)) != cudaSuccess) return e;
    // through v~ = A V: the landmarks (q~, dv~, normaliser, dv~.v~) against every key
    if ((e = to_bf16(A.dvt, rows * 64, A.dvt16, st)) != cudaSuccess) return e;
    BwdPass vp{};
    vp.q = A.q_tilde; vp.g = A.dvt16; vp.k = A.k; vp.v = A.v; vp.L = A.lseA; vp.D = A.cvt;
    vp.Dacc = A.cvt; vp.dq = A.dqt; vp.dk = A.dk; vp.dv = A.dv; vp.c = c; vp.BH = A.BH;
    vp.nq = A.m; vp.nk = A.N; vp.status = A.status;
    if ((e = cudaMemsetAsync(A.cvt, 0, (size_t)rows * sizeof(float), st)) != cudaSuccess) return e;
    if ((e = launch_bwd_pass_mma(vp, 2, st)) != cudaSuccess) return e;
    if ((e = launch_bwd_pass_mma(vp, 0, st)) != cudaSuccess) return e;
    vp.first = kv_first;
    if ((e = launch_bwd_pass_mma(vp, 1, st)) != cudaSuccess) return e;
  }
  if ((e = launch_bwd_pass_mma(p, 1, st)) != cudaSuccess) return e;   // adds to dk, dv
  if (!A.routed)
    launch_pool_grad(A.dqt, A.BH, A.N, 64, A.grid_h, A.grid_w, A.mh, A.mw, A.dq, st);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t run(const BwdArgs<T>& A, cudaStream_t st) {
  const int BH = A.BH, N = A.N, m = A.m;
  const long long BHN = (long long)BH * N;
  const size_t sm = smem_bytes<D>();
  cudaError_t e;
  for (const void* f : {(const void*)bwd_raw_kernel<T, D>, (const void*)bwd_shared_kernel<T, D>,
                        (const void*)bwd_vtilde_kernel<T, D>}) {
    e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
  }
  bool mma = false;
  if constexpr (std::is_same<T, bf16>::value && D == 64) mma = A.vt16 && A.dvt16;
  if (!mma) {   // the SIMT kernels add into cleared gradients (run_mma clears what it must)
    const size_t gbytes = (size_t)BHN * D * sizeof(float);
    float* const grads[3] = {A.dq, A.dk, A.dv};
    for (int i = 0; i < 3; ++i) {
      e = cudaMemsetAsync(grads[i], 0, gbytes, st);
      if (e != cudaSuccess) return e;
    }
  }
  if (mma) {
    bwd_lse_kernel<<<(unsigned)((BHN + 255) / 256), 256, 0, st>>>(
        A.routed ? nullptr : A.sh_lse, A.part, BHN, A.s, A.lse, A.status);
  } else {
    bwd_stats_kernel<D><<<(unsigned)((BHN + 7) / 8), 256, 0, st>>>(
        A.routed ? nullptr : A.sh_lse, A.routed ? nullptr : A.sh_o, A.part, BHN, A.s, A.dout,
        std::is_same<T, bf16>::value ? 1 : 0, A.lse, A.Dn, A.status);
  }
  count_launch();
  if constexpr (std::is_same<T, bf16>::value && D == 64) {
    if (mma) return run_mma(A, st);
  }
  const int qtiles = (N + kT - 1) / kT;
  const int rtiles = (int)(((long long)N * A.s + kT - 1) / kT) + m;
  bwd_raw_kernel<T, D><<<(unsigned)((long long)BH * rtiles), kT, sm, st>>>(
      A.q, A.k, A.v, A.dout, A.topk_idx, A.bucket_off, A.bucket_qidx, A.lse, A.Dn, N, m, A.topk,
      A.s, rtiles, A.dq, A.dk, A.dv, A.status);
  count_launch();
  if (!A.routed) {
    bwd_shared_kernel<T, D><<<(unsigned)((long long)BH * qtiles), kT, sm, st>>>(
        A.q, A.dout, A.q_tilde, A.v_tilde, A.lse, A.Dn, N, m, A.c_sh, qtiles, A.dq, A.dqt, A.dvt);
    count_launch();
    const long long rows = (long long)BH * m;
    bwd_vt_dot_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, st>>>(A.dvt, A.v_tilde, rows, D,
                                                                  A.cvt);
    count_launch();
    bwd_vtilde_kernel<T, D><<<(unsigned)((long long)BH * qtiles), kT, sm, st>>>(
        A.k, A.v, A.q_tilde, A.dvt, A.lseA, A.cvt, N, m, qtiles, A.dk, A.dv, A.dqt);
    count_launch();
    launch_pool_grad(A.dqt, BH, N, D, A.grid_h, A.grid_w, A.mh, A.mw, A.dq, st);
  }
  return cudaGetLastError();
}

}  // namespace

template <typename T>
cudaError_t launch_backward(const BwdArgs<T>& a, int d, cudaStream_t st) {
  switch (d) {
    case 16: return run<T, 16>(a, st);
    case 32: return run<T, 32>(a, st);
    case 64: return run<T, 64>(a, st);
    case 128: return run<T, 128>(a, st);
    default: return cudaErrorInvalidValue;
  }
}
template cudaError_t launch_backward<float>(const BwdArgs<float>&, int, cudaStream_t);
template cudaError_t launch_backward<bf16>(const BwdArgs<bf16>&, int, cudaStream_t);

}  // namespace mita
