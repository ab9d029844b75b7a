// Internal helpers shared by the MiTA CUDA kernels (not part of the C-ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cfloat>
#include <cstdint>

namespace mita {

using bf16 = __nv_bfloat16;

// ---------------------------------------------------------------------------
// Limits of this build (checked on the host before any launch).
// ---------------------------------------------------------------------------
constexpr int kMaxTopk = 4096;   // experts keep at most this many KV rows
constexpr int kMaxRouteS = 8;    // experts a query may be routed to (s)
constexpr int kTcapMax = 64;     // per-split candidates kept by the landmark sweep
constexpr int kBandCap = 1024;   // near-boundary candidates re-scored exactly
constexpr int kKeyTile = 32;     // keys staged per shared-memory tile (SIMT path)
constexpr int kExactCtas = 8;    // CTAs (and scratch rows) of the exact fallback

// ---------------------------------------------------------------------------
// Programmatic dependent launch: the forward's kernels are launched so that a
// kernel's grid becomes resident while the previous kernel's last CTAs still
// run; each such kernel starts with griddep_wait(), which returns once the
// previous grid has completed and its memory writes are visible (a no-op for a
// kernel launched the ordinary way).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Bits of the per-device status word (read by mita_get_last_device_error).
enum : int {
  kDevErrBadIndex = 1,    // an expert index outside [0, N)
  kDevErrBadBucket = 2,   // bucket offsets / query ids inconsistent
  kDevErrRoute = 4,       // a routed landmark outside [0, m)
  kDevErrTimeout = 8,     // a bounded wait inside a kernel gave up
};

// Relative bound on |fp32 dot - exact dot| per unit of |a|_2 |b|_2 for a
// length-D dot product accumulated in fp32 (sequential FMA or tensor-core
// fp32 accumulation).  Rounding every partial sum gives at most
// D * 2^-24 * sum|a_l b_l|, truncating it at most twice that; this takes
// twice the truncation bound, which also covers the fp32 norms used to
// evaluate it (sum|a_l b_l| <= |a|_2 |b|_2).
__host__ __device__ constexpr float err_gamma(int D) { return (float)D * 2.384185791015625e-07f; }  // D * 2^-22

// ---------------------------------------------------------------------------
// Element access
// ---------------------------------------------------------------------------
__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(bf16 x) { return __bfloat162float(x); }

template <typename T> struct Vec;
template <> struct Vec<float> {
  static constexpr int N = 4;
  __device__ __forceinline__ static void load(const float* p, float* o) {
    float4 x = *reinterpret_cast<const float4*>(p);
    o[0] = x.x; o[1] = x.y; o[2] = x.z; o[3] = x.w;
  }
  __device__ __forceinline__ static void store(float* p, const float* o) {
    *reinterpret_cast<float4*>(p) = make_float4(o[0], o[1], o[2], o[3]);
  }
};
template <> struct Vec<bf16> {
  static constexpr int N = 8;
  __device__ __forceinline__ static void load(const bf16* p, float* o) {
    uint4 x = *reinterpret_cast<const uint4*>(p);
    uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      o[2 * i] = __uint_as_float(w[i] << 16);
      o[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  __device__ __forceinline__ static void store(bf16* p, const float* o) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 h = __floats2bfloat162_rn(o[2 * i], o[2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
  }
};

// Load a full D-element row as floats (row start must be 16-byte aligned).
template <typename T, int D>
__device__ __forceinline__ void load_row(const T* p, float* o) {
#pragma unroll
  for (int i = 0; i < D; i += Vec<T>::N) Vec<T>::load(p + i, o + i);
}
template <typename T, int D>
__device__ __forceinline__ void store_row(T* p, const float* o) {
#pragma unroll
  for (int i = 0; i < D; i += Vec<T>::N) Vec<T>::store(p + i, o + i);
}

// double -> T with one rounding to nearest (ties to even).
template <typename T> __device__ T round_double(double x);
template <> __device__ __forceinline__ float round_double<float>(double x) {
  return __double2float_rn(x);
}
// Round to odd into float (24 bits), then to nearest into bf16 (8 bits): the
// 16 spare bits make the two-step rounding equal to one direct rounding.
template <> __device__ __forceinline__ bf16 round_double<bf16>(double x) {
  float f = __double2float_rz(x);
  if ((double)f != x) f = __uint_as_float(__float_as_uint(f) | 1u);
  return __float2bfloat16_rn(f);
}

// Error-free accumulation: after any sequence of calls, s + c equals the sum
// of the inputs up to the (second-order) rounding of c.  The _rn intrinsics
// keep the compiler from contracting or reassociating the two-sum.
__device__ __forceinline__ void two_sum_acc(float& s, float& c, float x) {
  const float t = __fadd_rn(s, x);
  const float bp = __fsub_rn(t, s);
  const float e = __fadd_rn(__fsub_rn(s, __fsub_rn(t, bp)), __fsub_rn(x, bp));
  s = t;
  c = __fadd_rn(c, e);
}

// A value carried as an unevaluated sum hi + lo (|lo| <= ulp(hi) / 2).
struct F2 {
  float hi, lo;
};
__device__ __forceinline__ F2 f2_normalize(float s, float c) {
  const float hi = __fadd_rn(s, c);
  return {hi, __fsub_rn(c, __fsub_rn(hi, s))};
}
__device__ __forceinline__ bool f2_greater(F2 x, F2 y) {
  return x.hi > y.hi || (x.hi == y.hi && x.lo > y.lo);
}
__device__ __forceinline__ bool ranks_before(F2 a, int ia, F2 b, int ib) {
  return f2_greater(a, b) || (a.hi == b.hi && a.lo == b.lo && ia < ib);
}

// Dot product with every product split exactly (two-product via FMA) and
// every sum error-free (two-sum): hi + lo is the exact dot up to ~n * 2^-48
// relative -- exact enough to order candidates whose exact scores differ by
// far less than the 1e-6 relative gap the parity rule allows.  fp32 only:
// fp64 runs at a small fraction of the fp32 rate on this part.
template <int D, int UNROLL = 8>
__device__ __forceinline__ F2 dot_f2(const float* a, const float* b) {
  float s = 0.f, c = 0.f;
#pragma unroll UNROLL
  for (int l = 0; l < D; ++l) {
    const float p = __fmul_rn(a[l], b[l]);
    const float e = fmaf(a[l], b[l], -p);
    two_sum_acc(s, c, p);
    c = __fadd_rn(c, e);
  }
  return f2_normalize(s, c);
}


// Lexicographic order of (score, index): higher score first, then lower index.
__device__ __forceinline__ bool ranks_before(float sa, int ia, float sb, int ib) {
  return sa > sb || (sa == sb && ia < ib);
}
__device__ __forceinline__ bool ranks_before(double sa, int ia, double sb, int ib) {
  return sa > sb || (sa == sb && ia < ib);
}

// Paired fp32 arithmetic (two values per instruction).
__device__ __forceinline__ unsigned long long f2pack(float a, float b) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2unpack(unsigned long long v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b,
                                                   unsigned long long c) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ unsigned long long add2(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// Monotone map float -> uint32 (larger float -> larger key) and back.
__device__ __forceinline__ uint32_t fkey(float x) {
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float fkey_inv(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Monotone map double -> uint64 (larger double -> larger key).
__device__ __forceinline__ unsigned long long order_key(double x) {
  if (x == 0.0) x = 0.0;  // fold -0 onto +0
  unsigned long long u = (unsigned long long)__double_as_longlong(x);
  return (u & 0x8000000000000000ull) ? ~u : (u | 0x8000000000000000ull);
}

// Exact (fp64) dot product of a T row with a double row.  Products of two
// bf16 (or fp32) values are exact in fp64 and, for the value ranges of
// attention inputs, so are the sums.
template <typename T, int D>
__device__ __forceinline__ double dot_exact(const double* a, const T* b) {
  double acc = 0.0;
#pragma unroll 8
  for (int l = 0; l < D; ++l) acc = fma(a[l], (double)to_f(b[l]), acc);
  return acc;
}

// ---------------------------------------------------------------------------
// Warp / block helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ int warp_incl_scan(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  return v;
}

// Block-wide max of one float per thread; `red` needs blockDim/32 floats.
__device__ __forceinline__ float block_max(float v, float* red) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_max(v);
  __syncthreads();
  if (lane == 0) red[w] = v;
  __syncthreads();
  float r = -INFINITY;
  for (int i = 0; i < nw; ++i) r = fmaxf(r, red[i]);
  return r;
}
__device__ __forceinline__ float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[w] = v;
  __syncthreads();
  float r = 0.f;
  for (int i = 0; i < nw; ++i) r += red[i];
  return r;
}

// Exclusive block scan of one int per thread; returns the block total in
// *total.  `red` needs blockDim/32 + 1 ints.
__device__ __forceinline__ int block_excl_scan(int v, int* red, int* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int inc = warp_incl_scan(v);
  __syncthreads();
  if (lane == 31) red[w] = inc;
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0;
    for (int i = 0; i < nw; ++i) { int t = red[i]; red[i] = run; run += t; }
    red[nw] = run;
  }
  __syncthreads();
  *total = red[nw];
  return red[w] + inc - v;
}

// Bitonic sort in shared memory of P (power of two) (key, index) pairs into
// ranks_before order (best first).  Called by the whole block.
template <typename K>
__device__ void bitonic_sort_desc(K* key, int* idx, int P) {
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      __syncthreads();
      for (int i = threadIdx.x; i < (P >> 1); i += blockDim.x) {
        int lo = 2 * i - (i & (stride - 1));
        int hi = lo + stride;
        bool up = (lo & size) == 0;
        K klo = key[lo], khi = key[hi];
        int ilo = idx[lo], ihi = idx[hi];
        bool swap = up ? ranks_before(khi, ihi, klo, ilo) : ranks_before(klo, ilo, khi, ihi);
        if (swap) { key[lo] = khi; key[hi] = klo; idx[lo] = ihi; idx[hi] = ilo; }
      }
    }
  }
  __syncthreads();
}

// Bitonic sort of P ints ascending.
__device__ inline void bitonic_sort_int_asc(int* a, int P) {
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      __syncthreads();
      for (int i = threadIdx.x; i < (P >> 1); i += blockDim.x) {
        int lo = 2 * i - (i & (stride - 1));
        int hi = lo + stride;
        bool up = (lo & size) == 0;
        int x = a[lo], y = a[hi];
        if (up ? (y < x) : (x < y)) { a[lo] = y; a[hi] = x; }
      }
    }
  }
  __syncthreads();
}

__host__ __device__ __forceinline__ int next_pow2(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

__device__ __forceinline__ void flag_error(int* status, int bit) {
  if (status) atomicOr(status, bit);
}

// Half-open adaptive window [floor(i*in/out), ceil((i+1)*in/out)).
__host__ __device__ __forceinline__ void adaptive_window(long long i, long long in,
                                                         long long out, int* lo, int* hi) {
  *lo = (int)((i * in) / out);
  *hi = (int)(((i + 1) * in + out - 1) / out);
}

}  // namespace mita
