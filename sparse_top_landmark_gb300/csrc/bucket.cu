// Step 5: group queries by their routed expert.
//
// The bit.fan article on MiTA describes Algorithm 1 as first building the
// experts, then grouping the queries by routing result so that each expert's
// KV rows are gathered once for all of its queries.  The grouping here is a
// stable counting sort in three launches (phases meet at kernel boundaries,
// no inter-CTA waiting), with the queries of a head cut into chunks of
// kBucketChunk:
//   count   -- one CTA per chunk: shared-memory histogram of its experts,
//              written as hist[bh][e][chunk];
//   scan    -- one warp per (head, expert): the expert's total, and for every
//              chunk the chunk's first slot relative to the expert's bucket;
//   scatter -- one CTA per chunk: the exclusive prefix of the expert totals
//              (bucket_off, written by the head's first chunk), then eight
//              warps on consecutive sub-chunks: a per-expert prefix across the
//              warps, then each warp places its queries in order (warp match +
//              popcount ranks equal experts in a batch of 32), so every bucket
//              lists its queries ascending.
// Experts beyond kSmemExperts use the same passes with global counters.
//
// With s > 1 the grouped list is the flat [N, s] route array (entry n * s + t
// is query n's t-th expert), so every bucket still lists its queries in
// ascending order, each query once per chosen expert; the stored value is the
// query index n = entry / s.
#include "common.cuh"
#include "kernels.h"

namespace mita {
namespace {

constexpr int kWarps = 8;
constexpr int kSub = kBucketChunk / kWarps;     // queries per warp in the scatter
constexpr int kSmemExperts = 2048;               // 8 x 2048 ints = 64 KB of shared memory

__device__ __forceinline__ int load_route(const int32_t* route, long long bh, int N, int n,
                                          int m, int* status) {
  if (n >= N) return -1;
  const int e = route[(size_t)bh * N + n];
  if (e < 0 || e >= m) {
    flag_error(status, kDevErrRoute);
    return -1;
  }
  return e;
}

__global__ void __launch_bounds__(256)
bucket_count_kernel(const int32_t* __restrict__ route, int N, int m, int nchunks,
                    int* __restrict__ hist, int* status) {
  griddep_wait();
  extern __shared__ int h[];                     // [m] when m <= kSmemExperts
  const long long bh = blockIdx.x / nchunks;
  const int chunk = blockIdx.x % nchunks;
  const bool smem = m <= kSmemExperts;
  int* hg = hist + (size_t)bh * m * nchunks;      // [e][chunk]
  if (smem) {
    for (int e = threadIdx.x; e < m; e += 256) h[e] = 0;
    __syncthreads();
  }
  const int n0 = chunk * kBucketChunk;
#pragma unroll 4
  for (int t = threadIdx.x; t < kBucketChunk; t += 256) {
    const int e = load_route(route, bh, N, n0 + t, m, status);
    if (e >= 0) {
      if (smem) atomicAdd(&h[e], 1);
      else atomicAdd(&hg[(size_t)e * nchunks + chunk], 1);
    }
  }
  if (smem) {
    __syncthreads();
    for (int e = threadIdx.x; e < m; e += 256) hg[(size_t)e * nchunks + chunk] = h[e];
  }
}

__global__ void __launch_bounds__(256)
bucket_scan_kernel(long long BHm, int nchunks, int* __restrict__ hist, int* __restrict__ total) {
  griddep_wait();
  const long long be = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5);   // bh * m + e
  const int lane = threadIdx.x & 31;
  if (be >= BHm) return;
  int* h = hist + (size_t)be * nchunks;
  int run = 0;
  for (int c0 = 0; c0 < nchunks; c0 += 32) {
    const int c = c0 + lane;
    const int x = c < nchunks ? h[c] : 0;
    const int inc = warp_incl_scan(x);
    if (c < nchunks) h[c] = run + inc - x;
    run += __shfl_sync(0xffffffffu, inc, 31);
  }
  if (lane == 0) total[be] = run;
}

// exclusive prefix of the head's expert totals into off[0..m] (shared or global)
__device__ void expert_offsets(const int* __restrict__ tot, int m, int* off, int* red) {
  __shared__ int carry_s;
  if (threadIdx.x == 0) carry_s = 0;
  __syncthreads();
  for (int e0 = 0; e0 < m; e0 += 256) {
    const int e = e0 + threadIdx.x;
    const int cnt = e < m ? tot[e] : 0;
    int t;
    const int ex = block_excl_scan(cnt, red, &t);
    const int base = carry_s;
    __syncthreads();
    if (e < m) off[e] = base + ex;
    if (threadIdx.x == 0) carry_s = base + t;
    __syncthreads();
  }
  if (threadIdx.x == 0) off[m] = carry_s;
  __syncthreads();
}

// many experts: one CTA per head writes bucket_off before the scatter
__global__ void __launch_bounds__(256)
bucket_offsets_kernel(const int* __restrict__ total, int m, int32_t* __restrict__ bucket_off) {
  griddep_wait();
  __shared__ int red[33];
  const long long bh = blockIdx.x;
  expert_offsets(total + (size_t)bh * m, m, bucket_off + (size_t)bh * (m + 1), red);
}

__global__ void __launch_bounds__(256)
bucket_scatter_kernel(const int32_t* __restrict__ route, int N, int m, int s, int nchunks,
                      int* __restrict__ hist, const int* __restrict__ total,
                      int32_t* __restrict__ bucket_off, int32_t* __restrict__ bucket_qidx,
                      int* status) {
  griddep_wait();
  extern __shared__ int hw[];                    // [kWarps][m] + off[m + 1] when m <= kSmemExperts
  __shared__ int red[33];
  const long long bh = blockIdx.x / nchunks;
  const int chunk = blockIdx.x % nchunks;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int* hg = hist + (size_t)bh * m * nchunks;
  int32_t* out = bucket_qidx + (size_t)bh * N;
  int32_t* boff = bucket_off + (size_t)bh * (m + 1);
  const int n0 = chunk * kBucketChunk + warp * kSub;
  const unsigned lt = (1u << lane) - 1u;
  if (m <= kSmemExperts) {
    int* off = hw + kWarps * m;
    expert_offsets(total + (size_t)bh * m, m, off, red);
    if (chunk == 0)
      for (int e = threadIdx.x; e <= m; e += 256) boff[e] = off[e];
    for (int i = threadIdx.x; i < kWarps * m; i += 256) hw[i] = 0;
    __syncthreads();
    // per-warp counts of its sub-chunk
    for (int it = 0; it < kSub; it += 32) {
      const int e = load_route(route, bh, N, n0 + it + lane, m, nullptr);
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      if (e >= 0 && lane == __ffs(peers) - 1) hw[warp * m + e] += __popc(peers);
      __syncwarp();
    }
    __syncthreads();
    // exclusive prefix across the warps, starting at the chunk's slot
    for (int e = threadIdx.x; e < m; e += 256) {
      int run = off[e] + hg[(size_t)e * nchunks + chunk];
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const int t = hw[w * m + e];
        hw[w * m + e] = run;
        run += t;
      }
    }
    __syncthreads();
    int* my = hw + warp * m;
    for (int it = 0; it < kSub; it += 32) {
      const int n = n0 + it + lane;
      const int e = load_route(route, bh, N, n, m, nullptr);
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      int base = 0;
      if (e >= 0) base = my[e];
      __syncwarp();
      if (e >= 0) {
        const int pos = base + __popc(peers & lt);
        if (pos >= 0 && pos < N) out[pos] = s == 1 ? n : n / s;
        else flag_error(status, kDevErrBadBucket);
        if (lane == __ffs(peers) - 1) my[e] = base + __popc(peers);
      }
      __syncwarp();
    }
  } else if (warp == 0) {
    // many experts (bucket_off written by bucket_offsets_kernel): one warp
    // walks the chunk in order with global counters
    int* hgw = hg;
    for (int it = 0; it < kBucketChunk; it += 32) {
      const int n = chunk * kBucketChunk + it + lane;
      const int e = load_route(route, bh, N, n, m, nullptr);
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      int base = 0;
      if (e >= 0) base = boff[e] + hgw[(size_t)e * nchunks + chunk];
      __syncwarp();
      if (e >= 0) {
        const int pos = base + __popc(peers & lt);
        if (pos >= 0 && pos < N) out[pos] = s == 1 ? n : n / s;
        else flag_error(status, kDevErrBadBucket);
        if (lane == __ffs(peers) - 1) hgw[(size_t)e * nchunks + chunk] = base - boff[e] + __popc(peers);
      }
      __syncwarp();
    }
  }
}

}  // namespace

size_t bucket_ws_bytes(int BH, int entries, int m) {
  const size_t nchunks = ((size_t)entries + kBucketChunk - 1) / kBucketChunk;
  return (size_t)BH * (nchunks + 1) * m * sizeof(int);
}

cudaError_t launch_bucket(const int32_t* route_idx, int BH, int N, int m, void* ws,
                          int32_t* bucket_off, int32_t* bucket_qidx, int* status,
                          cudaStream_t st, bool counted, int s) {
  if (s < 1 || (long long)N * s >= (1LL << 31)) return cudaErrorInvalidValue;
  N *= s;   // entries of the flat route list per head
  const int nchunks = (N + kBucketChunk - 1) / kBucketChunk;
  int* hist = static_cast<int*>(ws);                       // [BH][m][nchunks]
  int* total = hist + (size_t)BH * m * nchunks;             // [BH][m]
  const bool smem = m <= kSmemExperts;
  cudaError_t e;
  if (!smem && !counted) {
    e = cudaMemsetAsync(hist, 0, (size_t)BH * m * nchunks * sizeof(int), st);
    if (e != cudaSuccess) return e;
  }
  const unsigned blocks = (unsigned)((long long)BH * nchunks);
  const size_t s1 = smem ? (size_t)m * 4 : 0, s3 = smem ? ((size_t)kWarps * m + m + 1) * 4 : 0;
  if (s3 > 48 * 1024) {
    e = cudaFuncSetAttribute(bucket_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)s3);
    if (e != cudaSuccess) return e;
  }
  if (!counted) {
    e = launch_pdl(bucket_count_kernel, dim3(blocks), dim3(256), s1, st, route_idx, N, m, nchunks,
                   hist, status);
    count_launch();
    if (e != cudaSuccess) return e;
  }
  const long long BHm = (long long)BH * m;
  e = launch_pdl(bucket_scan_kernel, dim3((unsigned)((BHm + kWarps - 1) / kWarps)), dim3(256), 0, st,
                 BHm, nchunks, hist, total);
  count_launch();
  if (e != cudaSuccess) return e;
  if (!smem) {
    e = launch_pdl(bucket_offsets_kernel, dim3(BH), dim3(256), 0, st, total, m, bucket_off);
    count_launch();
    if (e != cudaSuccess) return e;
  }
  e = launch_pdl(bucket_scatter_kernel, dim3(blocks), dim3(256), s3, st, route_idx, N, m, s,
                 nchunks, hist, total, bucket_off, bucket_qidx, status);
  count_launch();
  return e;
}

}  // namespace mita
