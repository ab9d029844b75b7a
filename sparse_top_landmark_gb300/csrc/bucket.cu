// Step 5: group queries by their routed expert.
//
// The bit.fan article on MiTA describes Algorithm 1 as first building the
// experts, then grouping the queries by routing result so that each expert's
// KV rows are gathered once for all of its queries.  The grouping here is a
// stable counting sort in three launches (phases meet at kernel boundaries,
// no inter-CTA waiting):
//   count   -- one warp per chunk of kBucketChunk queries adds its per-expert
//              counts into hist[bh][chunk][e];
//   scan    -- one CTA per head: bucket_off = exclusive prefix of the counts,
//              and hist[bh][chunk][e] becomes the chunk's first slot in e;
//   scatter -- the same warps walk their chunk in query order and place each
//              query at its slot (warp match + popcount gives the rank among
//              equal experts in a batch of 32), so every bucket lists its
//              queries in ascending order.
#include "common.cuh"
#include "kernels.h"

namespace mita {
namespace {

constexpr int kWarpsPerBlock = 8;

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

__global__ void __launch_bounds__(kWarpsPerBlock * 32)
bucket_count_kernel(const int32_t* __restrict__ route, int N, int m, int nchunks, int cpb,
                    int* __restrict__ hist, int* status) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long long bh = blockIdx.x / cpb;
  const int chunk = (blockIdx.x % cpb) * kWarpsPerBlock + warp;
  if (chunk >= nchunks) return;
  int* h = hist + ((size_t)bh * nchunks + chunk) * m;
  const int n0 = chunk * kBucketChunk;
  for (int it = 0; it < kBucketChunk; it += 32) {
    const int e = load_route(route, bh, N, n0 + it + lane, m, status);
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int leader = __ffs(peers) - 1;
    if (e >= 0 && lane == leader) atomicAdd(h + e, __popc(peers));
  }
}

__global__ void __launch_bounds__(1024)
bucket_scan_kernel(int N, int m, int nchunks, int* __restrict__ hist,
                   int32_t* __restrict__ bucket_off) {
  __shared__ int red[33];
  const long long bh = blockIdx.x;
  int* hb = hist + (size_t)bh * nchunks * m;
  int32_t* off = bucket_off + (size_t)bh * (m + 1);
  int carry = 0;
  for (int e0 = 0; e0 < m; e0 += blockDim.x) {
    const int e = e0 + threadIdx.x;
    int cnt = 0;
    if (e < m)
      for (int c = 0; c < nchunks; ++c) cnt += hb[(size_t)c * m + e];
    int tot;
    const int excl = block_excl_scan(cnt, red, &tot);
    if (e < m) {
      int run = carry + excl;
      off[e] = run;
      for (int c = 0; c < nchunks; ++c) {
        const int t = hb[(size_t)c * m + e];
        hb[(size_t)c * m + e] = run;
        run += t;
      }
    }
    carry += tot;
  }
  if (threadIdx.x == 0) off[m] = carry;
  (void)N;
}

__global__ void __launch_bounds__(kWarpsPerBlock * 32)
bucket_scatter_kernel(const int32_t* __restrict__ route, int N, int m, int nchunks, int cpb,
                      int* __restrict__ hist, int32_t* __restrict__ bucket_qidx, int* status) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long long bh = blockIdx.x / cpb;
  const int chunk = (blockIdx.x % cpb) * kWarpsPerBlock + warp;
  if (chunk >= nchunks) return;
  int* h = hist + ((size_t)bh * nchunks + chunk) * m;
  int32_t* out = bucket_qidx + (size_t)bh * N;
  const int n0 = chunk * kBucketChunk;
  const unsigned lt = (1u << lane) - 1u;
  for (int it = 0; it < kBucketChunk; it += 32) {
    const int n = n0 + it + lane;
    const int e = load_route(route, bh, N, n, m, nullptr);
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int leader = __ffs(peers) - 1;
    int base = 0;
    if (e >= 0) base = h[e];
    __syncwarp();
    if (e >= 0) {
      const int pos = base + __popc(peers & lt);
      if (pos >= 0 && pos < N) out[pos] = n;
      else flag_error(status, kDevErrBadBucket);
      if (lane == leader) h[e] = base + __popc(peers);
    }
    __syncwarp();
  }
}

}  // namespace

size_t bucket_ws_bytes(int BH, int N, int m) {
  const size_t nchunks = (N + kBucketChunk - 1) / kBucketChunk;
  return (size_t)BH * nchunks * m * sizeof(int);
}

cudaError_t launch_bucket(const int32_t* route_idx, int BH, int N, int m, void* ws,
                          int32_t* bucket_off, int32_t* bucket_qidx, int* status,
                          cudaStream_t st) {
  const int nchunks = (N + kBucketChunk - 1) / kBucketChunk;
  const int cpb = (nchunks + kWarpsPerBlock - 1) / kWarpsPerBlock;
  int* hist = static_cast<int*>(ws);
  cudaError_t e = cudaMemsetAsync(hist, 0, bucket_ws_bytes(BH, N, m), st);
  if (e != cudaSuccess) return e;
  const unsigned blocks = (unsigned)((long long)BH * cpb);
  bucket_count_kernel<<<blocks, kWarpsPerBlock * 32, 0, st>>>(route_idx, N, m, nchunks, cpb,
                                                               hist, status);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  bucket_scan_kernel<<<BH, 1024, 0, st>>>(N, m, nchunks, hist, bucket_off);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  bucket_scatter_kernel<<<blocks, kWarpsPerBlock * 32, 0, st>>>(route_idx, N, m, nchunks, cpb,
                                                                 hist, bucket_qidx, status);
  return cudaGetLastError();
}

}  // namespace mita
