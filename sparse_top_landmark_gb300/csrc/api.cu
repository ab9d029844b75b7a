// C ABI of libmita.so: argument validation, workspace cache, stage
// orchestration.  Every arithmetic step runs in the kernels of this library.
#include "mita.h"

#include <algorithm>
#include <cmath>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <map>
#include <mutex>
#include <string>
#include <type_traits>
#include <utility>

#include "common.cuh"
#include "kernels.h"

namespace mita {
namespace {

thread_local std::string g_msg;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_msg = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* where) {
  return fail(MITA_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

struct DevState {
  int* status = nullptr;
  int num_sms = 0;
};

std::mutex g_mu;
std::map<int, DevState> g_dev;
struct WsEntry {
  void* ptr = nullptr;
  size_t bytes = 0;
};
std::map<std::pair<int, cudaStream_t>, WsEntry> g_ws;
std::map<std::pair<int, cudaStream_t>, WsEntry> g_stage;
// Bytes one cached buffer may grow to (0: no limit).  A growth beyond it fails exactly as a
// failed cudaMallocAsync does, before the allocator is called: the host-side way to make the
// allocation failure path run without exhausting a GPU.
std::atomic<unsigned long long> g_ws_limit{0};

int device_state(DevState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lk(g_mu);
  DevState& s = g_dev[dev];
  if (s.status == nullptr) {
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    int* p = nullptr;
    e = cudaMalloc(&p, sizeof(int));
    if (e != cudaSuccess) return fail(MITA_ERR_OOM, "status word: %s", cudaGetErrorString(e));
    e = cudaMemset(p, 0, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemset");
    s.status = p;
    s.num_sms = sms;
  }
  *out = &s;
  return MITA_OK;
}

// One buffer per (device, stream) in `cache`, grown (stream-ordered) when a
// call needs more.
int cached_buffer(std::map<std::pair<int, cudaStream_t>, WsEntry>& cache, const char* what,
                  size_t bytes, cudaStream_t st, void** out) {
  *out = nullptr;
  if (bytes == 0) return MITA_OK;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lk(g_mu);
  WsEntry& w = cache[{dev, st}];
  if (w.bytes >= bytes) {
    *out = w.ptr;
    return MITA_OK;
  }
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  e = cudaStreamIsCapturing(st, &cs);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
  if (cs != cudaStreamCaptureStatusNone)
    return fail(MITA_ERR_UNSUPPORTED,
                "%s must grow to %zu bytes while the stream is capturing; make one "
                "call of this size outside capture first", what, bytes);
  if (w.ptr) {
    e = cudaFreeAsync(w.ptr, st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFreeAsync");
    w.ptr = nullptr;
    w.bytes = 0;
  }
  const size_t want = bytes + bytes / 8;
  const unsigned long long limit = g_ws_limit.load();
  if (limit != 0 && want > limit)
    return fail(MITA_ERR_OOM, "%s of %zu bytes: above the workspace limit of %llu bytes", what,
                want, limit);
  void* p = nullptr;
  e = cudaMallocAsync(&p, want, st);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(MITA_ERR_OOM, "%s of %zu bytes: %s", what, want, cudaGetErrorString(e));
  }
  w.ptr = p;
  w.bytes = want;
  *out = p;
  return MITA_OK;
}

int workspace(size_t bytes, cudaStream_t st, void** out) {
  return cached_buffer(g_ws, "workspace", bytes, st, out);
}

// device copies of the host-buffer forward's inputs and output
int staging(size_t bytes, cudaStream_t st, void** out) {
  return cached_buffer(g_stage, "staging buffer", bytes, st, out);
}

// ---------------------------------------------------------------------------
// Validation
// ---------------------------------------------------------------------------
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_ptrs(std::initializer_list<std::pair<const void*, const char*>> ps) {
  for (auto& p : ps) {
    if (p.first == nullptr) return fail(MITA_ERR_INVALID_ARG, "%s is NULL", p.second);
    if (!aligned16(p.first))
      return fail(MITA_ERR_INVALID_ARG, "%s is not 16-byte aligned", p.second);
  }
  return MITA_OK;
}

int check_shape(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1)
    return fail(MITA_ERR_INVALID_ARG, "B, H, N must be >= 1 (got %d, %d, %d)", B, H, N);
  if (d != 16 && d != 32 && d != 64 && d != 128)
    return fail(MITA_ERR_UNSUPPORTED, "head dim d=%d not in {16, 32, 64, 128}", d);
  if ((long long)B * H * N >= (1LL << 31))
    return fail(MITA_ERR_UNSUPPORTED, "B*H*N must be < 2^31");
  return MITA_OK;
}

int check_m(int N, int m) {
  if (m < 1 || m > N) return fail(MITA_ERR_INVALID_ARG, "need 1 <= m <= N (m=%d, N=%d)", m, N);
  return MITA_OK;
}

int check_topk(int N, int topk) {
  if (topk < 1 || topk > N)
    return fail(MITA_ERR_INVALID_ARG, "need 1 <= topk <= N (topk=%d, N=%d)", topk, N);
  if (topk > kMaxTopk)
    return fail(MITA_ERR_UNSUPPORTED, "topk=%d above this build's limit %d", topk, kMaxTopk);
  return MITA_OK;
}

int check_s(int m, int s) {
  if (s < 1 || s > m) return fail(MITA_ERR_INVALID_ARG, "need 1 <= s <= m (s=%d)", s);
  if (s > kMaxRouteS)
    return fail(MITA_ERR_UNSUPPORTED, "s=%d above this build's limit %d", s, kMaxRouteS);
  return MITA_OK;
}

// B*H*N*s route entries must stay below 2^31
int check_entries(int B, int H, int N, int s) {
  if ((long long)B * H * N * s >= (1LL << 31))
    return fail(MITA_ERR_UNSUPPORTED, "B*H*N*s must be < 2^31");
  return MITA_OK;
}

// The landmark grid: lm_h x lm_w when given (both > 0), else 1 x m for a 1D
// sequence (grid_h = 1) and sqrt(m) x sqrt(m) for a 2D grid.
int check_grid(int N, int grid_h, int grid_w, int m, int lm_h = 0, int lm_w = 0,
               int* mh = nullptr, int* mw = nullptr) {
  if (grid_h < 1 || grid_w < 1 || (long long)grid_h * grid_w != N)
    return fail(MITA_ERR_INVALID_ARG, "grid %dx%d does not hold N=%d tokens", grid_h, grid_w, N);
  int h = 1, w = m;
  if (lm_h != 0 || lm_w != 0) {
    if (lm_h < 1 || lm_w < 1 || (long long)lm_h * lm_w != m)
      return fail(MITA_ERR_INVALID_ARG, "landmark grid %dx%d does not hold m=%d landmarks", lm_h,
                  lm_w, m);
    if (grid_h == 1 && lm_h != 1)
      return fail(MITA_ERR_INVALID_ARG, "a 1D sequence pools onto 1 x m landmarks");
    h = lm_h;
    w = lm_w;
  } else if (grid_h != 1) {
    int r = 1;
    while ((r + 1) * (r + 1) <= m) ++r;
    if (r * r != m)
      return fail(MITA_ERR_INVALID_ARG,
                  "2D pooling needs a square m (got %d) or an explicit landmark grid", m);
    h = w = r;
  }
  if (mh) *mh = h;
  if (mw) *mw = w;
  return MITA_OK;
}

int check_options(const mita_options* o) {
  if (o == nullptr) return MITA_OK;
  if (o->shared_temperature != MITA_SHARED_SQRT_D && o->shared_temperature != MITA_SHARED_D)
    return fail(MITA_ERR_INVALID_ARG, "unknown shared_temperature %d", o->shared_temperature);
  if (o->branches != MITA_BRANCHES_BOTH && o->branches != MITA_BRANCHES_ROUTED)
    return fail(MITA_ERR_INVALID_ARG, "unknown branches %d", o->branches);
  return MITA_OK;
}

#define MITA_TRY(x)                  \
  do {                               \
    int rc_ = (x);                   \
    if (rc_ != MITA_OK) return rc_;  \
  } while (0)

#define MITA_CUDA(x, where)                            \
  do {                                                 \
    cudaError_t e_ = (x);                              \
    if (e_ != cudaSuccess) return cuda_fail(e_, where); \
  } while (0)

size_t align256(size_t n) { return (n + 255) / 256 * 256; }

// ---------------------------------------------------------------------------
// Stage implementations (T = float or bf16)
// ---------------------------------------------------------------------------
template <typename T>
int pool_impl(const T* q, int B, int H, int N, int d, int gh, int gw, int m, T* qt,
              cudaStream_t st, int lm_h = 0, int lm_w = 0) {
  MITA_TRY(check_shape(B, H, N, d));
  MITA_TRY(check_m(N, m));
  int mh = 0, mw = 0;
  MITA_TRY(check_grid(N, gh, gw, m, lm_h, lm_w, &mh, &mw));
  MITA_TRY(check_ptrs({{q, "q"}, {qt, "q_tilde"}}));
  MITA_CUDA(launch_pool<T>(q, B * H, N, d, gh, gw, mh, mw, qt, st), "pool launch");
  return MITA_OK;
}

template <typename T>
int landmark_impl(const T* qt, const T* k, const T* v, int B, int H, int N, int d, int m,
                  int topk, int32_t* ti, float* vt, cudaStream_t st) {
  MITA_TRY(check_shape(B, H, N, d));
  MITA_TRY(check_m(N, m));
  MITA_TRY(check_topk(N, topk));
  MITA_TRY(check_ptrs({{qt, "q_tilde"}, {k, "k"}, {v, "v"}, {ti, "topk_idx"}, {vt, "v_tilde"}}));
  DevState* ds = nullptr;
  MITA_TRY(device_state(&ds));
  const LandmarkPlan plan =
      plan_landmark(B * H, N, d, m, topk, ds->num_sms, std::is_same<T, bf16>::value);
  void* ws = nullptr;
  MITA_TRY(workspace(landmark_ws_bytes(plan, B * H, N, d, m), st, &ws));
  const LandmarkWs lw = carve_landmark_ws(ws, plan, B * H, N, d, m);
  MITA_CUDA(launch_landmark<T>(qt, k, v, B * H, N, d, m, topk, plan, lw, ti, vt, ds->status, st),
            "landmark launch");
  return MITA_OK;
}

// Tensor-core route for bf16 / d = 64 / m <= 512 when no shared partial is
// requested; the SIMT kernel otherwise.
// per head: a count, then the ambiguous query ids and their fp32 best scores
size_t route_ws_bytes(int BH, int N) { return (size_t)BH * (2 * (size_t)N + 1) * sizeof(int); }

template <typename T>
bool route_uses_tc(int d, int m, int s, const float* lse, const float* so) {
  return std::is_same<T, bf16>::value && s == 1 && !lse && !so && route_tc_supported(d, m);
}
// the shared branch's partial requested (both outputs), s = 1 or 2: the tensor-core kernel
// that reuses the routing logits as the shared logits
template <typename T>
bool route_shared_uses_tc(int d, int m, int s, const float* lse, const float* so) {
  return std::is_same<T, bf16>::value && lse && so && route_shared_tc_supported(d, m, s);
}

template <typename T>
cudaError_t route_dispatch(const T* q, const T* qt, const float* vt, int BH, int N, int d, int m,
                           int s, int32_t* route, float* lse, float* so, DevState* ds, void* ws,
                           cudaStream_t st, int* hist = nullptr, bool* counted = nullptr,
                           bool prezeroed = false, int temp = 0) {
  if constexpr (std::is_same<T, bf16>::value) {
    if (route_uses_tc<T>(d, m, s, lse, so)) {
      if (counted) *counted = hist != nullptr;
      return launch_route_tc(q, qt, BH, N, m, ds->num_sms, route, static_cast<int*>(ws),
                             ds->status, hist, st, prezeroed);
    }
    if (route_shared_uses_tc<T>(d, m, s, lse, so)) {
      if (counted) *counted = hist != nullptr;
      return launch_route_shared_tc(q, qt, vt, BH, N, m, ds->num_sms, temp, 0, route, lse, so,
                                    static_cast<int*>(ws), ds->status, hist, st, prezeroed, s);
    }
  }
  return launch_route<T>(q, qt, vt, BH, N, d, m, s, route, lse, so, st, temp);
}

template <typename T>
int route_impl(const T* q, const T* qt, const float* vt, int B, int H, int N, int d, int m,
               int s, int32_t* route, float* lse, float* so, cudaStream_t st) {
  MITA_TRY(check_shape(B, H, N, d));
  MITA_TRY(check_m(N, m));
  MITA_TRY(check_s(m, s));
  MITA_TRY(check_entries(B, H, N, s));
  MITA_TRY(check_ptrs({{q, "q"}, {qt, "q_tilde"}, {route, "route_idx"}}));
  if (lse || so) MITA_TRY(check_ptrs({{vt, "v_tilde"}}));
  if (so) MITA_TRY(check_ptrs({{so, "shared_o"}}));
  DevState* ds = nullptr;
  MITA_TRY(device_state(&ds));
  void* ws = nullptr;
  if (route_uses_tc<T>(d, m, s, lse, so) || route_shared_uses_tc<T>(d, m, s, lse, so))
    MITA_TRY(workspace(route_ws_bytes(B * H, N), st, &ws));
  MITA_CUDA(route_dispatch<T>(q, qt, vt, B * H, N, d, m, s, route, lse, so, ds, ws, st),
            "route launch");
  return MITA_OK;
}

int bucket_impl(const int32_t* route, int B, int H, int N, int m, int s, int32_t* off,
                int32_t* qidx, cudaStream_t st) {
  if (B < 1 || H < 1 || N < 1) return fail(MITA_ERR_INVALID_ARG, "B, H, N must be >= 1");
  if ((long long)B * H * N >= (1LL << 31)) return fail(MITA_ERR_UNSUPPORTED, "B*H*N >= 2^31");
  MITA_TRY(check_m(N, m));
  MITA_TRY(check_s(m, s));
  MITA_TRY(check_entries(B, H, N, s));
  if (!route || !off || !qidx) return fail(MITA_ERR_INVALID_ARG, "NULL bucket argument");
  DevState* ds = nullptr;
  MITA_TRY(device_state(&ds));
  void* ws = nullptr;
  MITA_TRY(workspace(bucket_ws_bytes(B * H, N * s, m), st, &ws));
  MITA_CUDA(launch_bucket(route, B * H, N, m, ws, off, qidx, ds->status, st, false, s),
            "bucket launch");
  return MITA_OK;
}

template <typename T>
int expert_impl(const T* q, const T* k, const T* v, const T* qt, const float* vt,
                const int32_t* ti, const int32_t* off, const int32_t* qidx, const float* lse,
                const float* so, int B, int H, int N, int d, int m, int topk, int s, T* out,
                cudaStream_t st) {
  MITA_TRY(check_shape(B, H, N, d));
  MITA_TRY(check_m(N, m));
  MITA_TRY(check_topk(N, topk));
  MITA_TRY(check_s(m, s));
  MITA_TRY(check_entries(B, H, N, s));
  MITA_TRY(check_ptrs({{q, "q"}, {k, "k"}, {v, "v"}, {out, "out"}}));
  if (!ti || !off || !qidx) return fail(MITA_ERR_INVALID_ARG, "NULL index argument");
  if ((lse == nullptr) != (so == nullptr))
    return fail(MITA_ERR_INVALID_ARG, "shared_lse and shared_o must be both set or both NULL");
  if (so == nullptr) MITA_TRY(check_ptrs({{qt, "q_tilde"}, {vt, "v_tilde"}}));
  DevState* ds = nullptr;
  MITA_TRY(device_state(&ds));
  if (s > 1) {
    // per-expert partials, merged per query with the shared branch's partial; without a
    // caller-supplied shared partial it is computed here (the SIMT route, s = 1, into scratch)
    const int BH = B * H;
    const size_t pb = align256(expert_partials_ws_bytes(BH, N, d, s));
    const size_t rb = align256((size_t)BH * N * 4), lb = align256((size_t)BH * N * 4);
    const size_t ob = align256((size_t)BH * N * d * 4);
    const bool tc = std::is_same<T, bf16>::value && expert_tc_supported(d, m, topk);
    const size_t tb = tc ? align256(expert_tc_partials_ws_bytes(BH, N, m, topk, s)) : 0;
    void* wsv = nullptr;
    MITA_TRY(workspace(pb + tb + (so ? 0 : rb + lb + ob), st, &wsv));
    char* ws = static_cast<char*>(wsv);
    if (so == nullptr) {
      int32_t* r1 = reinterpret_cast<int32_t*>(ws + pb + tb);
      float* l1 = reinterpret_cast<float*>(ws + pb + tb + rb);
      float* o1 = reinterpret_cast<float*>(ws + pb + tb + rb + lb);
      MITA_CUDA(launch_route<T>(q, qt, vt, BH, N, d, m, 1, r1, l1, o1, st), "shared partial");
      lse = l1;
      so = o1;
    }
    if constexpr (std::is_same<T, bf16>::value) {
      if (tc) {
        const ExpertPartials part = carve_expert_partials(ws, BH, N, d, s);
        MITA_CUDA(launch_expert_tc_partials(q, k, v, ti, off, qidx, BH, N, m, topk, s,
                                            ds->num_sms, ws + pb, part, ds->status, st),
                  "expert launch");
        MITA_CUDA(launch_expert_merge<T>(lse, so, 0, part, BH, N, d, s, out, ds->status, st),
                  "merge launch");
        return MITA_OK;
      }
    }
    MITA_CUDA(launch_expert_attn<T>(q, k, v, qt, vt, ti, off, qidx, lse, so, BH, N, d, m, topk, s,
                                    ws, out, ds->status, st),
              "expert launch");
    return MITA_OK;
  }
  if constexpr (std::is_same<T, bf16>::value) {
    if (expert_tc_supported(d, m, topk)) {
      // with a carried shared partial the kernel attends over the raw pairs only and merges
      void* ws = nullptr;
      MITA_TRY(workspace(expert_tc_ws_bytes(B * H, N, m, topk), st, &ws));
      MITA_CUDA(launch_expert_tc(q, k, v, qt, vt, ti, off, qidx, B * H, N, m, topk, ds->num_sms,
                                 ws, out, ds->status, st, 0, 0, lse, so, 0),
                "expert launch");
      return MITA_OK;
    }
  }
  MITA_CUDA(launch_expert_attn<T>(q, k, v, qt, vt, ti, off, qidx, lse, so, B * H, N, d, m, topk,
                                  1, nullptr, out, ds->status, st),
            "expert launch");
  return MITA_OK;
}

struct ForwardLayout {
  size_t qt, vt, ti, route, off, qidx, lm, bk, ex, rt, lse, so, total;
  LandmarkPlan plan;
};

ForwardLayout forward_layout(int BH, int N, int d, int m, int topk, int s, size_t esize, int sms) {
  ForwardLayout L{};
  L.plan = plan_landmark(BH, N, d, m, topk, sms, esize == 2);
  const size_t NS = (size_t)N * s;
  size_t o = 0;
  L.qt = o; o += align256((size_t)BH * m * d * esize);
  L.vt = o; o += align256((size_t)BH * m * d * 4);
  L.ti = o; o += align256((size_t)BH * m * topk * 4);
  L.route = o; o += align256((size_t)BH * NS * 4);
  L.off = o; o += align256((size_t)BH * (m + 1) * 4);
  L.qidx = o; o += align256((size_t)BH * NS * 4);
  L.lm = o; o += align256(landmark_ws_bytes(L.plan, BH, N, d, m));
  L.bk = o; o += align256(bucket_ws_bytes(BH, (int)NS, m));
  L.ex = o;
  if (s > 1) {
    o += align256(expert_partials_ws_bytes(BH, N, d, s));
    if (esize == 2 && expert_tc_supported(d, m, topk))
      o += align256(expert_tc_partials_ws_bytes(BH, N, m, topk, s));
  }
  else if (esize == 2 && expert_tc_supported(d, m, topk))
    o += align256(std::max(expert_tc_ws_bytes(BH, N, m, topk),
                           N <= 1024 ? expert_masked_ws_bytes(BH, N, m) : size_t(0)));
  L.rt = o; o += align256(route_ws_bytes(BH, N));
  // s > 1: the shared branch's partial, emitted by the route kernel
  L.lse = o; if (s > 1) o += align256((size_t)BH * N * 4);
  L.so = o; if (s > 1) o += align256((size_t)BH * N * d * 4);
  L.total = o;
  return L;
}

// The forward's counters, cleared by one kernel at its start (a memset between two
// kernels would hold back the next kernel's early launch): the landmark stage's
// slow-row count, the heads' ambiguous-query counts and the bucket histogram.
__global__ void __launch_bounds__(256)
forward_zero_kernel(int* a, long long na, int* b, long long nb, int* c, long long nc) {
  griddep_wait();
  const long long t0 = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long t = t0; t < na; t += stride) a[t] = 0;
  for (long long t = t0; t < nb; t += stride) b[t] = 0;
  for (long long t = t0; t < nc; t += stride) c[t] = 0;
}

template <typename T>
int forward_impl(const T* q, const T* k, const T* v, int B, int H, int N, int d, int gh, int gw,
                 int m, int topk, int s, T* out, cudaStream_t st,
                 const mita_options* opt = nullptr) {
  MITA_TRY(check_shape(B, H, N, d));
  MITA_TRY(check_m(N, m));
  MITA_TRY(check_options(opt));
  const int temp = opt ? opt->shared_temperature : MITA_SHARED_SQRT_D;
  const int routed = opt ? (opt->branches == MITA_BRANCHES_ROUTED) : 0;
  int mh = 0, mw = 0;
  MITA_TRY(check_grid(N, gh, gw, m, opt ? opt->landmark_grid_h : 0,
                      opt ? opt->landmark_grid_w : 0, &mh, &mw));
  MITA_TRY(check_topk(N, topk));
  MITA_TRY(check_s(m, s));
  MITA_TRY(check_entries(B, H, N, s));
  MITA_TRY(check_ptrs({{q, "q"}, {k, "k"}, {v, "v"}, {out, "out"}}));
  DevState* ds = nullptr;
  MITA_TRY(device_state(&ds));
  const int BH = B * H;
  const ForwardLayout L = forward_layout(BH, N, d, m, topk, s, sizeof(T), ds->num_sms);
  void* wsv = nullptr;
  MITA_TRY(workspace(L.total, st, &wsv));
  char* ws = static_cast<char*>(wsv);
  T* qt = reinterpret_cast<T*>(ws + L.qt);
  float* vt = reinterpret_cast<float*>(ws + L.vt);
  int32_t* ti = reinterpret_cast<int32_t*>(ws + L.ti);
  int32_t* route = reinterpret_cast<int32_t*>(ws + L.route);
  int32_t* off = reinterpret_cast<int32_t*>(ws + L.off);
  int32_t* qidx = reinterpret_cast<int32_t*>(ws + L.qidx);
  const LandmarkWs lw = carve_landmark_ws(ws + L.lm, L.plan, BH, N, d, m);
  {
    const long long nh = (long long)BH * m * (((long long)N * s + kBucketChunk - 1) / kBucketChunk);
    MITA_CUDA(launch_pdl(forward_zero_kernel, dim3((unsigned)std::min<long long>(
                             (nh + 255) / 256 + 1, (long long)ds->num_sms * 4)),
                         dim3(256), 0, st, lw.nslow, 1LL, reinterpret_cast<int*>(ws + L.rt),
                         (long long)BH, reinterpret_cast<int*>(ws + L.bk), nh),
              "counter clearing");
    count_launch();
  }
  MITA_CUDA(launch_pool<T>(q, BH, N, d, gh, gw, mh, mw, qt, st), "pool launch");
  MITA_CUDA(launch_landmark<T>(qt, k, v, BH, N, d, m, topk, L.plan, lw, ti, vt, ds->status, st,
                               true),
            "landmark launch");
  if (s > 1) {
    // top-s routing with the shared branch's partial, grouping of the N*s (query, expert)
    // entries, per-expert partials and their merge
    float* lse = reinterpret_cast<float*>(ws + L.lse);
    float* so = reinterpret_cast<float*>(ws + L.so);
    // routing only: no shared partial (the SIMT route then lists the routes alone); with the
    // shared branch, s = 2 and m <= 256 route on the tensor cores, the shared partial's output
    // in bf16
    int so_bf16 = 0;
    bool counted = false;       // the tensor-core route counts the bucket histogram too
    if constexpr (std::is_same<T, bf16>::value) {
      if (!routed && route_shared_tc_supported(d, m, s)) {
        so_bf16 = 1;
        counted = true;
        MITA_CUDA(launch_route_shared_tc(q, qt, vt, BH, N, m, ds->num_sms, temp, 1, route, lse, so,
                                         reinterpret_cast<int*>(ws + L.rt), ds->status,
                                         reinterpret_cast<int*>(ws + L.bk), st, true, s),
                  "route launch");
      }
    }
    if (!so_bf16)
      MITA_CUDA(route_dispatch<T>(q, qt, vt, BH, N, d, m, s, route, routed ? nullptr : lse,
                                  routed ? nullptr : so, ds, ws + L.rt, st, nullptr, nullptr, true,
                                  temp),
                "route launch");
    MITA_CUDA(launch_bucket(route, BH, N, m, ws + L.bk, off, qidx, ds->status, st, counted, s),
              "bucket launch");
    if constexpr (std::is_same<T, bf16>::value) {
      if (expert_tc_supported(d, m, topk)) {
        // every (query, expert) entry's raw-pair partial on the tensor cores (fp32 outputs:
        // bf16 partials measured beyond the output tolerance), then the merge
        const ExpertPartials part = carve_expert_partials(ws + L.ex, BH, N, d, s);
        void* tws = ws + L.ex + align256(expert_partials_ws_bytes(BH, N, d, s));
        MITA_CUDA(launch_expert_tc_partials(q, k, v, ti, off, qidx, BH, N, m, topk, s,
                                            ds->num_sms, tws, part, ds->status, st),
                  "expert launch");
        MITA_CUDA(launch_expert_merge<T>(routed ? nullptr : lse, routed ? nullptr : so, so_bf16,
                                         part, BH, N, d, s, out, ds->status, st),
                  "merge launch");
        return MITA_OK;
      }
    }
    MITA_CUDA(launch_expert_attn<T>(q, k, v, qt, vt, ti, off, qidx, lse, so, BH, N, d, m, topk, s,
                                    ws + L.ex, out, ds->status, st, temp, routed),
              "expert launch");
    return MITA_OK;
  }
  if constexpr (std::is_same<T, bf16>::value) {
    if (expert_tc_supported(d, m, topk) && expert_masked_preferred(N, m, topk, routed)) {
      // short sequences: each query's expert from the route, then per-head query tiles over
      // all keys masked to that expert's set -- no grouping needed
      MITA_CUDA(route_dispatch<T>(q, qt, vt, BH, N, d, m, 1, route, nullptr, nullptr, ds,
                                  ws + L.rt, st, nullptr, nullptr, true),
                "route launch");
      MITA_CUDA(launch_expert_masked_tc(q, k, v, qt, vt, ti, route, BH, N, m, topk, ds->num_sms,
                                        ws + L.ex, out, ds->status, st, temp, routed),
                "expert launch");
      return MITA_OK;
    }
  }
  // s = 1: the expert kernel recomputes the shared logits q . q~ on the tensor cores rather
  // than taking them from the route stage as a carried partial (measured: the carried split,
  // route_shared_tc + raw-pairs-only expert, is slower at both long workloads)
  // the tensor-core route also counts the bucket stage's (expert, chunk) histogram
  bool counted = false;
  MITA_CUDA(route_dispatch<T>(q, qt, vt, BH, N, d, m, 1, route, nullptr, nullptr, ds, ws + L.rt,
                              st, reinterpret_cast<int*>(ws + L.bk), &counted, true),
            "route launch");
  MITA_CUDA(launch_bucket(route, BH, N, m, ws + L.bk, off, qidx, ds->status, st, counted),
            "bucket launch");
  if constexpr (std::is_same<T, bf16>::value) {
    if (expert_tc_supported(d, m, topk)) {
      MITA_CUDA(launch_expert_tc(q, k, v, qt, vt, ti, off, qidx, BH, N, m, topk, ds->num_sms,
                                 ws + L.ex, out, ds->status, st, temp, routed),
                "expert launch");
      return MITA_OK;
    }
  }
  MITA_CUDA(launch_expert_attn<T>(q, k, v, qt, vt, ti, off, qidx, nullptr, nullptr, BH, N, d, m,
                                  topk, 1, nullptr, out, ds->status, st, temp, routed),
            "expert launch");
  return MITA_OK;
}

template <typename T>
int dense_impl(const T* q, const T* k, const T* v, int B, int H, int N, int d, T* out,
               cudaStream_t st) {
  MITA_TRY(check_shape(B, H, N, d));
  MITA_TRY(check_ptrs({{q, "q"}, {k, "k"}, {v, "v"}, {out, "out"}}));
  DevState* ds = nullptr;
  MITA_TRY(device_state(&ds));
  const int BH = B * H;
  void* ws = nullptr;
  if constexpr (std::is_same<T, bf16>::value) {
    if (d == 64) {
      MITA_TRY(workspace(dense_tc_ws_bytes(BH, N), st, &ws));
      MITA_CUDA(launch_dense_tc(q, k, v, BH, N, ds->num_sms, ws, out, ds->status, st),
                "dense launch");
      return MITA_OK;
    }
  }
  MITA_TRY(workspace(dense_simt_ws_bytes(BH, N), st, &ws));
  MITA_CUDA(launch_dense_attn<T>(q, k, v, BH, N, d, ws, out, ds->status, st), "dense launch");
  return MITA_OK;
}

// The backward with the selections held constant: the forward's selections and partials
// recomputed by the forward's own kernels, then the gradient kernels (backward.cu).
template <typename T>
int backward_impl(const T* q, const T* k, const T* v, const T* dout, int B, int H, int N, int d,
                  int gh, int gw, int m, int topk, int s, const mita_options* opt, float* dq,
                  float* dk, float* dv, cudaStream_t st) {
  MITA_TRY(check_shape(B, H, N, d));
  MITA_TRY(check_m(N, m));
  MITA_TRY(check_options(opt));
  int mh = 0, mw = 0;
  MITA_TRY(check_grid(N, gh, gw, m, opt ? opt->landmark_grid_h : 0,
                      opt ? opt->landmark_grid_w : 0, &mh, &mw));
  MITA_TRY(check_topk(N, topk));
  MITA_TRY(check_s(m, s));
  MITA_TRY(check_entries(B, H, N, s));
  MITA_TRY(check_ptrs({{q, "q"}, {k, "k"}, {v, "v"}, {dout, "dout"}, {dq, "dq"}, {dk, "dk"},
                       {dv, "dv"}}));
  const int temp = opt ? opt->shared_temperature : MITA_SHARED_SQRT_D;
  const int routed = opt ? (opt->branches == MITA_BRANCHES_ROUTED) : 0;
  DevState* ds = nullptr;
  MITA_TRY(device_state(&ds));
  const int BH = B * H;
  const size_t BHN = (size_t)BH * N, NS = (size_t)N * s;
  const LandmarkPlan plan = plan_landmark(BH, N, d, m, topk, ds->num_sms, sizeof(T) == 2);
  size_t o = 0;
  auto take = [&](size_t bytes) { const size_t at = o; o += align256(bytes); return at; };
  const size_t o_qt = take((size_t)BH * m * d * sizeof(T)), o_vt = take((size_t)BH * m * d * 4);
  const size_t o_ti = take((size_t)BH * m * topk * 4), o_r = take((size_t)BH * NS * 4);
  const size_t o_off = take((size_t)BH * (m + 1) * 4), o_qi = take((size_t)BH * NS * 4);
  const size_t o_lm = take(landmark_ws_bytes(plan, BH, N, d, m));
  const size_t o_bk = take(bucket_ws_bytes(BH, (int)NS, m));
  const size_t o_sl = take(BHN * 4), o_so = take(BHN * d * 4);
  const size_t o_pt = take(expert_partials_ws_bytes(BH, N, d, s));
  const size_t o_lse = take(BHN * 4), o_dn = take(BHN * 4);
  const size_t o_la = take((size_t)BH * m * 4), o_cv = take((size_t)BH * m * 4);
  const size_t o_dqt = take((size_t)BH * m * d * 4), o_dvt = take((size_t)BH * m * d * 4);
  // bf16 with d = 64: the selections are recomputed by the tensor-core route and expert
  // kernels where they apply, and the gradient passes run on the tensor cores
  const bool mma = std::is_same<T, bf16>::value && d == 64;
  const bool tc_expert = mma && expert_tc_supported(d, m, topk);
  const bool tc_route = std::is_same<T, bf16>::value &&
                        (routed ? s == 1 && route_tc_supported(d, m) : route_shared_tc_supported(d, m, s));
  const size_t o_v16 = mma ? take((size_t)BH * m * 64 * 2) : 0;
  const size_t o_dv16 = mma ? take((size_t)BH * m * 64 * 2) : 0;
  const size_t o_rws = tc_route ? take(route_ws_bytes(BH, N)) : 0;
  const size_t o_tcx = tc_expert ? take(expert_tc_partials_ws_bytes(BH, N, m, topk, s)) : 0;
  void* wsv = nullptr;
  MITA_TRY(workspace(o, st, &wsv));
  char* ws = static_cast<char*>(wsv);
  T* qt = reinterpret_cast<T*>(ws + o_qt);
  float* vt = reinterpret_cast<float*>(ws + o_vt);
  int32_t* ti = reinterpret_cast<int32_t*>(ws + o_ti);
  int32_t* route = reinterpret_cast<int32_t*>(ws + o_r);
  int32_t* off = reinterpret_cast<int32_t*>(ws + o_off);
  int32_t* qidx = reinterpret_cast<int32_t*>(ws + o_qi);
  float* sl = reinterpret_cast<float*>(ws + o_sl);
  float* so = reinterpret_cast<float*>(ws + o_so);
  ExpertPartials part;
  part.o = reinterpret_cast<float*>(ws + o_pt);
  part.lse = part.o + BHN * s * d;
  part.pos = reinterpret_cast<int*>(part.lse + BHN * s);
  part.cnt = part.pos + BHN * s;
  // dq, dk, dv are cleared by the gradient launcher where its kernels add rather than store
  MITA_CUDA(cudaMemsetAsync(ws + o_dqt, 0, (o_dvt - o_dqt) + (size_t)BH * m * d * 4, st),
            "clearing scratch");
  MITA_CUDA(launch_pool<T>(q, BH, N, d, gh, gw, mh, mw, qt, st), "pool launch");
  LandmarkWs lw = carve_landmark_ws(ws + o_lm, plan, BH, N, d, m);
  lw.lse_out = reinterpret_cast<float*>(ws + o_la);   // each landmark's softmax normaliser
  MITA_CUDA(launch_landmark<T>(qt, k, v, BH, N, d, m, topk, plan, lw, ti, vt, ds->status, st),
            "landmark launch");
  MITA_CUDA(route_dispatch<T>(q, qt, vt, BH, N, d, m, s, route, routed ? nullptr : sl,
                              routed ? nullptr : so, ds, tc_route ? ws + o_rws : nullptr, st,
                              nullptr, nullptr, false, temp),
            "route launch");
  MITA_CUDA(launch_bucket(route, BH, N, m, ws + o_bk, off, qidx, ds->status, st, false, s),
            "bucket launch");
  if constexpr (std::is_same<T, bf16>::value) {
    if (tc_expert)
      MITA_CUDA(launch_expert_tc_partials(q, k, v, ti, off, qidx, BH, N, m, topk, s,
                                          ds->num_sms, ws + o_tcx, part, ds->status, st),
                "expert partials");
  }
  if (!tc_expert)
    MITA_CUDA(launch_expert_partials<T>(q, k, v, ti, off, qidx, BH, N, d, m, topk, s, part,
                                        ds->status, st),
              "expert partials");
  BwdArgs<T> a{};
  a.q = q; a.k = k; a.v = v; a.dout = dout; a.q_tilde = qt; a.v_tilde = vt;
  a.topk_idx = ti; a.bucket_off = off; a.bucket_qidx = qidx;
  a.sh_lse = routed ? nullptr : sl; a.sh_o = routed ? nullptr : so; a.part = part;
  a.BH = BH; a.N = N; a.m = m; a.topk = topk; a.s = s; a.routed = routed;
  a.c_sh = (float)(temp == MITA_SHARED_D ? 1.0 / d : 1.0 / std::sqrt((double)d));
  a.grid_h = gh; a.grid_w = gw; a.mh = mh; a.mw = mw;
  a.lse = reinterpret_cast<float*>(ws + o_lse); a.Dn = reinterpret_cast<float*>(ws + o_dn);
  a.lseA = reinterpret_cast<float*>(ws + o_la); a.cvt = reinterpret_cast<float*>(ws + o_cv);
  a.dqt = reinterpret_cast<float*>(ws + o_dqt); a.dvt = reinterpret_cast<float*>(ws + o_dvt);
  a.dq = dq; a.dk = dk; a.dv = dv; a.status = ds->status;
  if (mma) {
    a.vt16 = reinterpret_cast<bf16*>(ws + o_v16);
    a.dvt16 = reinterpret_cast<bf16*>(ws + o_dv16);
  }
  MITA_CUDA(launch_backward<T>(a, d, st), "backward launch");
  return MITA_OK;
}

// The forward on host buffers.  The host link, not the GPU, bounds this call (H2D and D2H
// each run at about 200 GB/s on this part, whether a copy engine or the SMs drive them), so
// the heads are split into up to kHostGroups groups that pipeline: a copy stream brings in
// group g + 1's q, k, v while `st` runs group g's forward, and a second copy stream takes
// group g's output back meanwhile (the link is full duplex).  Returns after `st` is
// synchronised.
constexpr int kHostGroups = 4;
struct HostPipe {
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t ev[2 + 2 * kHostGroups] = {};
  std::mutex mu;   // one host-buffer forward at a time per device uses these
};
std::map<int, HostPipe*> g_pipe;

int host_pipe(HostPipe** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lk(g_mu);
  HostPipe*& p = g_pipe[dev];
  if (p == nullptr) {
    HostPipe* np = new HostPipe();
    e = cudaStreamCreateWithFlags(&np->h2d, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&np->d2h, cudaStreamNonBlocking);
    for (auto& ev : np->ev)
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
    if (e != cudaSuccess) {
      delete np;   // (any stream or event created so far is left to the context's teardown)
      return cuda_fail(e, "copy streams");
    }
    p = np;
  }
  *out = p;
  return MITA_OK;
}

template <typename T>
int forward_host_impl(const T* q, const T* k, const T* v, int B, int H, int N, int d, int gh,
                      int gw, int m, int topk, int s, T* out, cudaStream_t st) {
  MITA_TRY(check_shape(B, H, N, d));
  MITA_TRY(check_m(N, m));
  MITA_TRY(check_grid(N, gh, gw, m));
  MITA_TRY(check_topk(N, topk));
  MITA_TRY(check_s(m, s));
  if (!q || !k || !v || !out) return fail(MITA_ERR_INVALID_ARG, "null host pointer");
  const size_t n = (size_t)B * H * N * d;
  const size_t bytes = align256(n * sizeof(T));
  HostPipe* hp = nullptr;
  MITA_TRY(host_pipe(&hp));
  // Held before the staging buffer is looked up: a call that grows (frees and reallocates)
  // the buffer must not do so while another host-buffer forward is still copying into it.
  std::lock_guard<std::mutex> lk(hp->mu);
  void* sv = nullptr;
  MITA_TRY(staging(4 * bytes, st, &sv));
  char* sb = static_cast<char*>(sv);
  T* dq = reinterpret_cast<T*>(sb);
  T* dk = reinterpret_cast<T*>(sb + bytes);
  T* dv = reinterpret_cast<T*>(sb + 2 * bytes);
  T* dout = reinterpret_cast<T*>(sb + 3 * bytes);
  // On an error return, wait for every copy already queued: they read and write the caller's
  // host buffers, which the caller may free as soon as this call returns.
  struct Drain {
    HostPipe* hp;
    cudaStream_t st;
    bool armed = true;
    ~Drain() {
      if (!armed) return;
      cudaStreamSynchronize(hp->h2d);
      cudaStreamSynchronize(hp->d2h);
      cudaStreamSynchronize(st);
    }
  } drain{hp, st};
  const int BH = B * H;
  const int per = (BH + std::min(BH, kHostGroups) - 1) / std::min(BH, kHostGroups);
  const int G = (BH + per - 1) / per;   // groups of `per` heads (the last may be smaller)
  const size_t head = (size_t)N * d;    // elements per head
  cudaEvent_t ev_start = hp->ev[0], ev_done = hp->ev[1];
  MITA_CUDA(cudaEventRecord(ev_start, st), "event");
  MITA_CUDA(cudaStreamWaitEvent(hp->h2d, ev_start, 0), "event wait");
  MITA_CUDA(cudaStreamWaitEvent(hp->d2h, ev_start, 0), "event wait");
  for (int g = 0; g < G; ++g) {
    const size_t o = (size_t)g * per * head, c = (size_t)std::min(per, BH - g * per) * head;
    MITA_CUDA(cudaMemcpyAsync(dq + o, q + o, c * sizeof(T), cudaMemcpyHostToDevice, hp->h2d),
              "copy of q");
    MITA_CUDA(cudaMemcpyAsync(dk + o, k + o, c * sizeof(T), cudaMemcpyHostToDevice, hp->h2d),
              "copy of k");
    MITA_CUDA(cudaMemcpyAsync(dv + o, v + o, c * sizeof(T), cudaMemcpyHostToDevice, hp->h2d),
              "copy of v");
    MITA_CUDA(cudaEventRecord(hp->ev[2 + g], hp->h2d), "event");
  }
  for (int g = 0; g < G; ++g) {
    const int hg = std::min(per, BH - g * per);
    const size_t o = (size_t)g * per * head, c = (size_t)hg * head;
    MITA_CUDA(cudaStreamWaitEvent(st, hp->ev[2 + g], 0), "event wait");
    // the heads are independent: a group runs as one batch of hg heads
    MITA_TRY(forward_impl<T>(dq + o, dk + o, dv + o, 1, hg, N, d, gh, gw, m, topk, s, dout + o,
                             st));
    MITA_CUDA(cudaEventRecord(hp->ev[2 + kHostGroups + g], st), "event");
    MITA_CUDA(cudaStreamWaitEvent(hp->d2h, hp->ev[2 + kHostGroups + g], 0), "event wait");
    MITA_CUDA(cudaMemcpyAsync(out + o, dout + o, c * sizeof(T), cudaMemcpyDeviceToHost, hp->d2h),
              "copy of out");
  }
  MITA_CUDA(cudaEventRecord(ev_done, hp->d2h), "event");
  MITA_CUDA(cudaStreamWaitEvent(st, ev_done, 0), "event wait");
  MITA_CUDA(cudaStreamSynchronize(st), "synchronisation");
  drain.armed = false;   // every stream is idle: st waited for the last copy out
  return MITA_OK;
}

}  // namespace

int report_error(int code, const char* text) { return fail(code, "%s", text); }

}  // namespace mita

using mita::bf16;

namespace mita {
std::atomic<unsigned long long> g_launches{0};
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
}  // namespace mita

extern "C" {

int mita_pool(const void* q, int B, int H, int N, int d, int grid_h, int grid_w, int m,
              void* q_tilde, mita_stream_t stream) {
  return mita::pool_impl<bf16>(static_cast<const bf16*>(q), B, H, N, d, grid_h, grid_w, m,
                               static_cast<bf16*>(q_tilde), stream);
}
int mita_pool_grid(const void* q, int B, int H, int N, int d, int grid_h, int grid_w,
                   int landmark_grid_h, int landmark_grid_w, void* q_tilde, mita_stream_t stream) {
  return mita::pool_impl<bf16>(static_cast<const bf16*>(q), B, H, N, d, grid_h, grid_w,
                               landmark_grid_h * landmark_grid_w, static_cast<bf16*>(q_tilde),
                               stream, landmark_grid_h, landmark_grid_w);
}
int mita_pool_grid_f32(const float* q, int B, int H, int N, int d, int grid_h, int grid_w,
                       int landmark_grid_h, int landmark_grid_w, float* q_tilde,
                       mita_stream_t stream) {
  return mita::pool_impl<float>(q, B, H, N, d, grid_h, grid_w, landmark_grid_h * landmark_grid_w,
                                q_tilde, stream, landmark_grid_h, landmark_grid_w);
}
int mita_pool_f32(const float* q, int B, int H, int N, int d, int grid_h, int grid_w, int m,
                  float* q_tilde, mita_stream_t stream) {
  return mita::pool_impl<float>(q, B, H, N, d, grid_h, grid_w, m, q_tilde, stream);
}

int mita_landmark_topk_shared(const void* q_tilde, const void* k, const void* v, int B, int H,
                              int N, int d, int m, int topk, int32_t* topk_idx, float* v_tilde,
                              mita_stream_t stream) {
  return mita::landmark_impl<bf16>(static_cast<const bf16*>(q_tilde),
                                   static_cast<const bf16*>(k), static_cast<const bf16*>(v), B,
                                   H, N, d, m, topk, topk_idx, v_tilde, stream);
}
int mita_landmark_topk_shared_f32(const float* q_tilde, const float* k, const float* v, int B,
                                  int H, int N, int d, int m, int topk, int32_t* topk_idx,
                                  float* v_tilde, mita_stream_t stream) {
  return mita::landmark_impl<float>(q_tilde, k, v, B, H, N, d, m, topk, topk_idx, v_tilde,
                                    stream);
}

int mita_route(const void* q, const void* q_tilde, const float* v_tilde, int B, int H, int N,
               int d, int m, int s, int32_t* route_idx, float* shared_lse, float* shared_o,
               mita_stream_t stream) {
  return mita::route_impl<bf16>(static_cast<const bf16*>(q), static_cast<const bf16*>(q_tilde),
                                v_tilde, B, H, N, d, m, s, route_idx, shared_lse, shared_o,
                                stream);
}
int mita_route_f32(const float* q, const float* q_tilde, const float* v_tilde, int B, int H,
                   int N, int d, int m, int s, int32_t* route_idx, float* shared_lse,
                   float* shared_o, mita_stream_t stream) {
  return mita::route_impl<float>(q, q_tilde, v_tilde, B, H, N, d, m, s, route_idx, shared_lse,
                                 shared_o, stream);
}

int mita_bucket(const int32_t* route_idx, int B, int H, int N, int m, int s,
                int32_t* bucket_off, int32_t* bucket_qidx, mita_stream_t stream) {
  return mita::bucket_impl(route_idx, B, H, N, m, s, bucket_off, bucket_qidx, stream);
}

int mita_expert_attn(const void* q, const void* k, const void* v, const void* q_tilde,
                     const float* v_tilde, const int32_t* topk_idx, const int32_t* bucket_off,
                     const int32_t* bucket_qidx, const float* shared_lse, const float* shared_o,
                     int B, int H, int N, int d, int m, int topk, int s, void* out,
                     mita_stream_t stream) {
  return mita::expert_impl<bf16>(
      static_cast<const bf16*>(q), static_cast<const bf16*>(k), static_cast<const bf16*>(v),
      static_cast<const bf16*>(q_tilde), v_tilde, topk_idx, bucket_off, bucket_qidx, shared_lse,
      shared_o, B, H, N, d, m, topk, s, static_cast<bf16*>(out), stream);
}
int mita_expert_attn_f32(const float* q, const float* k, const float* v, const float* q_tilde,
                         const float* v_tilde, const int32_t* topk_idx,
                         const int32_t* bucket_off, const int32_t* bucket_qidx,
                         const float* shared_lse, const float* shared_o, int B, int H, int N,
                         int d, int m, int topk, int s, float* out, mita_stream_t stream) {
  return mita::expert_impl<float>(q, k, v, q_tilde, v_tilde, topk_idx, bucket_off, bucket_qidx,
                                  shared_lse, shared_o, B, H, N, d, m, topk, s, out, stream);
}

int mita_forward(const void* q, const void* k, const void* v, int B, int H, int N, int d,
                 int grid_h, int grid_w, int m, int topk, int s, void* out,
                 mita_stream_t stream) {
  return mita::forward_impl<bf16>(static_cast<const bf16*>(q), static_cast<const bf16*>(k),
                                  static_cast<const bf16*>(v), B, H, N, d, grid_h, grid_w, m,
                                  topk, s, static_cast<bf16*>(out), stream);
}
int mita_forward_f32(const float* q, const float* k, const float* v, int B, int H, int N, int d,
                     int grid_h, int grid_w, int m, int topk, int s, float* out,
                     mita_stream_t stream) {
  return mita::forward_impl<float>(q, k, v, B, H, N, d, grid_h, grid_w, m, topk, s, out, stream);
}

int mita_forward_ex(const void* q, const void* k, const void* v, int B, int H, int N, int d,
                    int grid_h, int grid_w, int m, int topk, int s, const mita_options* options,
                    void* out, mita_stream_t stream) {
  return mita::forward_impl<bf16>(static_cast<const bf16*>(q), static_cast<const bf16*>(k),
                                  static_cast<const bf16*>(v), B, H, N, d, grid_h, grid_w, m, topk,
                                  s, static_cast<bf16*>(out), stream, options);
}
int mita_forward_ex_f32(const float* q, const float* k, const float* v, int B, int H, int N,
                        int d, int grid_h, int grid_w, int m, int topk, int s,
                        const mita_options* options, float* out, mita_stream_t stream) {
  return mita::forward_impl<float>(q, k, v, B, H, N, d, grid_h, grid_w, m, topk, s, out, stream,
                                   options);
}

int mita_dense_attn(const void* q, const void* k, const void* v, int B, int H, int N, int d,
                    void* out, mita_stream_t stream) {
  return mita::dense_impl<bf16>(static_cast<const bf16*>(q), static_cast<const bf16*>(k),
                                static_cast<const bf16*>(v), B, H, N, d, static_cast<bf16*>(out),
                                stream);
}
int mita_dense_attn_f32(const float* q, const float* k, const float* v, int B, int H, int N,
                        int d, float* out, mita_stream_t stream) {
  return mita::dense_impl<float>(q, k, v, B, H, N, d, out, stream);
}

int mita_backward(const void* q, const void* k, const void* v, const void* dout, int B, int H,
                  int N, int d, int grid_h, int grid_w, int m, int topk, int s,
                  const mita_options* options, float* dq, float* dk, float* dv,
                  mita_stream_t stream) {
  return mita::backward_impl<bf16>(static_cast<const bf16*>(q), static_cast<const bf16*>(k),
                                   static_cast<const bf16*>(v), static_cast<const bf16*>(dout), B,
                                   H, N, d, grid_h, grid_w, m, topk, s, options, dq, dk, dv,
                                   stream);
}
int mita_backward_f32(const float* q, const float* k, const float* v, const float* dout, int B,
                      int H, int N, int d, int grid_h, int grid_w, int m, int topk, int s,
                      const mita_options* options, float* dq, float* dk, float* dv,
                      mita_stream_t stream) {
  return mita::backward_impl<float>(q, k, v, dout, B, H, N, d, grid_h, grid_w, m, topk, s,
                                    options, dq, dk, dv, stream);
}

int mita_forward_host(const void* q, const void* k, const void* v, int B, int H, int N, int d,
                      int grid_h, int grid_w, int m, int topk, int s, void* out,
                      mita_stream_t stream) {
  return mita::forward_host_impl<bf16>(static_cast<const bf16*>(q), static_cast<const bf16*>(k),
                                       static_cast<const bf16*>(v), B, H, N, d, grid_h, grid_w,
                                       m, topk, s, static_cast<bf16*>(out), stream);
}
int mita_forward_host_f32(const float* q, const float* k, const float* v, int B, int H, int N,
                          int d, int grid_h, int grid_w, int m, int topk, int s, float* out,
                          mita_stream_t stream) {
  return mita::forward_host_impl<float>(q, k, v, B, H, N, d, grid_h, grid_w, m, topk, s, out,
                                        stream);
}

uint64_t mita_forward_workspace_bytes(int B, int H, int N, int d, int m, int topk, int s,
                                      int is_f32) {
  if (mita::check_shape(B, H, N, d) || mita::check_m(N, m) || mita::check_topk(N, topk) ||
      mita::check_s(m, s) || mita::check_entries(B, H, N, s))
    return 0;
  int sms = 152;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaGetLastError();
  return mita::forward_layout(B * H, N, d, m, topk, s, is_f32 ? 4 : 2, sms).total;
}

const char* mita_status_string(int status) {
  switch (status) {
    case MITA_OK: return "ok";
    case MITA_ERR_INVALID_ARG: return "invalid argument";
    case MITA_ERR_UNSUPPORTED: return "unsupported by this build";
    case MITA_ERR_CUDA: return "CUDA error";
    case MITA_ERR_OOM: return "out of device memory";
    case MITA_ERR_DEVICE_CHECK: return "a kernel flagged inconsistent input data";
    default: return "unknown status";
  }
}

const char* mita_last_error_message(void) { return mita::g_msg.c_str(); }

int mita_get_last_device_error(mita_stream_t stream, int* bits) {
  if (bits) *bits = 0;
  mita::DevState* ds = nullptr;
  int rc = mita::device_state(&ds);
  if (rc != MITA_OK) return rc;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return mita::cuda_fail(e, "cudaStreamSynchronize");
  int v = 0;
  e = cudaMemcpy(&v, ds->status, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return mita::cuda_fail(e, "cudaMemcpy");
  e = cudaMemset(ds->status, 0, sizeof(int));
  if (e != cudaSuccess) return mita::cuda_fail(e, "cudaMemset");
  if (bits) *bits = v;
  return v ? mita::fail(MITA_ERR_DEVICE_CHECK, "device status bits 0x%x", v) : MITA_OK;
}

uint64_t mita_kernel_launches(void) { return mita::g_launches.load(std::memory_order_relaxed); }

int mita_check_bounded_wait(int* gave_up, mita_stream_t stream) {
  if (!gave_up) return mita::fail(MITA_ERR_INVALID_ARG, "mita_check_bounded_wait: NULL gave_up");
  mita::DevState* ds = nullptr;
  int rc = mita::device_state(&ds);
  if (rc != MITA_OK) return rc;
  const cudaError_t e = mita::launch_bounded_wait_probe(ds->status, gave_up, stream);
  return e == cudaSuccess ? MITA_OK : mita::cuda_fail(e, "mita_check_bounded_wait launch");
}

uint64_t mita_workspace_set_limit(uint64_t bytes) {
  return mita::g_ws_limit.exchange(bytes);
}

int mita_workspace_release(void) {
  std::lock_guard<std::mutex> lk(mita::g_mu);
  int prev = 0;
  cudaGetDevice(&prev);
  for (auto* cache : {&mita::g_ws, &mita::g_stage}) {
    for (auto& kv : *cache) {
      if (kv.second.ptr) {
        cudaSetDevice(kv.first.first);
        cudaDeviceSynchronize();
        cudaFree(kv.second.ptr);
      }
    }
    cache->clear();
  }
  cudaSetDevice(prev);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? MITA_OK : mita::cuda_fail(e, "workspace release");
}

}  // extern "C"
