/*
 * mita.h -- C ABI of libmita.so: the MiTA (Mixture-of-Top-k Attention)
 * forward pass on NVIDIA GB300 (sm_103a).
 *
 * Method (cited per entry point below):
 *   MiTA tutorial, iwxt.cn/tutorials/mita-attention, ch. 4 (paper Sec. 3.2,
 *   eq. 5-12) and ch. 8; gist.science summary of arXiv 2602.01219, Sec. 2.2-2.3
 *   (Algorithm 1); bit.fan news article on MiTA (expert construction,
 *   grouping by expert with online softmax).
 *
 * Conventions (all entry points):
 *   - Tensors are dense, row-major.  Q, K, V and the output are [B, H, N, d]:
 *     head (b, h) owns N consecutive rows of d elements.  For a 2D token grid
 *     (grid_h > 1) token t sits at row t / grid_w, column t % grid_w.
 *   - Unsuffixed entry points take bfloat16 data (`const void*` holding
 *     __nv_bfloat16); the `_f32` twins take float with the same parameters.
 *     Landmark values v~ and the optional shared-branch partial are float.
 *     Index outputs are int32.
 *   - Every pointer is a DEVICE pointer owned by the caller (except the data
 *     pointers of mita_forward_host*, which are host pointers); the library
 *     never frees or retains it.  Element arrays must start on a 16-byte boundary.
 *   - Calls are asynchronous on `stream` (NULL = legacy default stream) and
 *     never synchronise the host.  Arguments are validated on the host before
 *     any launch; an invalid call launches nothing and returns non-zero.
 *   - Launch failures return MITA_ERR_CUDA.  Faults during execution surface
 *     at the caller's next synchronisation.  Data-dependent problems the
 *     kernels detect (an index out of range in caller-supplied arrays) set a
 *     per-device status word read by mita_get_last_device_error(); the
 *     offending entry is skipped, never dereferenced.
 *   - Stages that need scratch memory (landmark, bucket, forward) draw it from
 *     a library-owned, stream-ordered cache (cudaMallocAsync on `stream`),
 *     one buffer per (device, stream), grown when a call needs more.  Growing
 *     is refused (MITA_ERR_UNSUPPORTED) while `stream` is being captured into
 *     a CUDA graph: make one call of the same size outside capture first.
 *     mita_workspace_release() frees the cache.
 *   - Supported: d in {16, 32, 64, 128}; 1 <= topk <= min(N, 4096);
 *     1 <= m <= N; 1 <= s <= min(m, 8) (s = 1 is the setting of every
 *     experiment on the pages and the one with the tensor-core path; s > 1
 *     runs SIMT kernels); B*H*N*s < 2^31.
 */
#ifndef MITA_H_
#define MITA_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* mita_stream_t;

/*
 * Options of mita_forward_ex (a zeroed struct, or NULL, gives mita_forward).
 *   shared_temperature  MITA_SHARED_SQRT_D: every joint-softmax logit is
 *                       divided by sqrt(d) (tutorial ch. 4, eq. 11-12).
 *                       MITA_SHARED_D: the m shared logits are q . q~_i / d,
 *                       the temperature tutorial ch. 8 caveat 3 reads out of
 *                       the official code (shared key pre-scaled by d^-1/2,
 *                       then the mixed attention's d^-1/2); the raw logits
 *                       stay q . k_j / sqrt(d) and v~ is unchanged.
 *   landmark_grid_h,    2D pooling onto this landmark grid (row-major landmark
 *   landmark_grid_w     index; landmark_grid_h * landmark_grid_w == m), e.g. a
 *                       non-square grid; 0, 0: 1 x m for a 1D sequence,
 *                       sqrt(m) x sqrt(m) for a 2D grid.
 *   branches            MITA_BRANCHES_BOTH: the m shared pairs and the s*k raw
 *                       pairs.  MITA_BRANCHES_ROUTED: the routing-only model
 *                       the bit.fan article's LRA ablation compares against at
 *                       an equal entry count (no shared branch: one softmax
 *                       over the s*k raw pairs; choose topk for the count).
 */
enum { MITA_SHARED_SQRT_D = 0, MITA_SHARED_D = 1 };
enum { MITA_BRANCHES_BOTH = 0, MITA_BRANCHES_ROUTED = 1 };
typedef struct mita_options {
  int shared_temperature;
  int landmark_grid_h;
  int landmark_grid_w;
  int branches;
} mita_options;

enum mita_status {
  MITA_OK = 0,
  MITA_ERR_INVALID_ARG = 1,   /* bad shape, null or misaligned pointer      */
  MITA_ERR_UNSUPPORTED = 2,   /* valid but outside this build's limits       */
  MITA_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed        */
  MITA_ERR_OOM = 4,           /* workspace allocation failed                 */
  MITA_ERR_DEVICE_CHECK = 5   /* a kernel flagged inconsistent input data    */
};

/*
 * mita_pool -- landmark queries by local average pooling of Q.
 * Tutorial ch. 4 step 1 (paper eq. 5): each landmark query q~_i is the mean of
 * a group of queries; the bit.fan article calls it local average pooling.
 *   q        [B,H,N,d]  input queries.
 *   grid_h, grid_w      token grid, grid_h * grid_w == N.  grid_h == 1: 1D,
 *                       m windows of the sequence; else m must be a perfect
 *                       square and the grid is pooled to sqrt(m) x sqrt(m).
 *                       Window i covers [floor(i*in/out), ceil((i+1)*in/out))
 *                       along each axis (adaptive average pooling).
 *   q_tilde  [B,H,m,d]  output, the exact window mean rounded once to the
 *                       element type (round to nearest even).
 */
int mita_pool(const void* q, int B, int H, int N, int d, int grid_h, int grid_w, int m,
              void* q_tilde, mita_stream_t stream);
/*
 * mita_pool_grid -- mita_pool onto an explicit landmark_grid_h x
 * landmark_grid_w grid (m = their product; a 1D sequence needs
 * landmark_grid_h == 1).  q_tilde [B,H,m,d], landmark i = row i / landmark_grid_w,
 * column i % landmark_grid_w; same window rule and rounding as mita_pool.
 */
int mita_pool_grid(const void* q, int B, int H, int N, int d, int grid_h, int grid_w,
                   int landmark_grid_h, int landmark_grid_w, void* q_tilde, mita_stream_t stream);
int mita_pool_grid_f32(const float* q, int B, int H, int N, int d, int grid_h, int grid_w,
                       int landmark_grid_h, int landmark_grid_w, float* q_tilde,
                       mita_stream_t stream);
int mita_pool_f32(const float* q, int B, int H, int N, int d, int grid_h, int grid_w, int m,
                  float* q_tilde, mita_stream_t stream);

/*
 * mita_landmark_topk_shared -- routed experts and shared landmark values.
 * Tutorial ch. 4 step 2 (eq. 6-7): s_ij = q~_i . k_j / sqrt(d) over all N
 * keys; expert i is the top-k keys of row i.  Step 3 (eq. 8-9): the same
 * scores, softmax over all N, weight all of V: v~_i.
 *   q_tilde  [B,H,m,d], k, v [B,H,N,d]   inputs.
 *   topk_idx [B,H,m,topk] int32  output: the topk key indices of each
 *            landmark in ascending index order.  The set is the one exact
 *            scores select, ties broken toward the lowest key index.
 *   v_tilde  [B,H,m,d] float     output.
 * Uses the workspace cache.
 */
int mita_landmark_topk_shared(const void* q_tilde, const void* k, const void* v, int B, int H,
                              int N, int d, int m, int topk, int32_t* topk_idx, float* v_tilde,
                              mita_stream_t stream);
int mita_landmark_topk_shared_f32(const float* q_tilde, const float* k, const float* v, int B,
                                  int H, int N, int d, int m, int topk, int32_t* topk_idx,
                                  float* v_tilde, mita_stream_t stream);

/*
 * mita_route -- route each query to its best landmark.
 * Tutorial ch. 4 step 4 (eq. 10): compare q . q~_i and keep the top-s; the
 * scores select, no gate.  The bit.fan article: those logits are reused for
 * the shared branch.
 *   q [B,H,N,d], q_tilde [B,H,m,d]  inputs.
 *   v_tilde [B,H,m,d] float          input, read only when a shared output is
 *                                    requested (may be NULL otherwise).
 *   route_idx [B,H,N,s] int32        output: the s landmarks with the largest
 *                                    q . q~_i, best first (exact; ties to the
 *                                    lowest landmark index).
 *   shared_lse [B,H,N] float or NULL output: ln sum_i exp(q . q~_i / sqrt(d)).
 *   shared_o [B,H,N,d] float or NULL output: softmax-weighted sum of v~ over
 *                                    the m shared pairs.
 */
int mita_route(const void* q, const void* q_tilde, const float* v_tilde, int B, int H, int N,
               int d, int m, int s, int32_t* route_idx, float* shared_lse, float* shared_o,
               mita_stream_t stream);
int mita_route_f32(const float* q, const float* q_tilde, const float* v_tilde, int B, int H,
                   int N, int d, int m, int s, int32_t* route_idx, float* shared_lse,
                   float* shared_o, mita_stream_t stream);

/*
 * mita_bucket -- group queries by routed expert (Algorithm 1, bit.fan
 * article: queries are grouped by routing result).
 *   route_idx [B,H,N,s] int32          input, values in [0, m).
 *   bucket_off [B,H,m+1] int32         output: exclusive prefix of the
 *                                      per-expert query counts.
 *   bucket_qidx [B,H,N*s] int32        output: for expert e, the query
 *                                      indices bucket_qidx[off[e]:off[e+1]]
 *                                      in ascending order (a stable sort;
 *                                      with s > 1 a query is listed once in
 *                                      each of its s buckets).
 * Values outside [0, m) are skipped and flag MITA_ERR_DEVICE_CHECK.  Uses the
 * workspace cache.
 */
int mita_bucket(const int32_t* route_idx, int B, int H, int N, int m, int s,
                int32_t* bucket_off, int32_t* bucket_qidx, mita_stream_t stream);

/*
 * mita_bucket_noalloc -- mita_bucket for callers that cannot allocate device
 * memory.  The paper has no counterpart: this is an engineering variant.
 * Callers that own every byte of device memory through their own allocator,
 * or that forbid allocation after start-up (real-time loops), cannot let the
 * library grow its workspace cache.  This entry point computes exactly what
 * mita_bucket computes but keeps its counters in a fixed 4 MiB device array
 * compiled into the library (held by every GPU that loads it until exit), so
 * it calls no allocator at all.
 *   Same arguments and outputs as mita_bucket.
 *   Limit: B*H*(ceil(N*s/4096)+1)*m <= 1048576, else MITA_ERR_UNSUPPORTED and
 *   nothing runs.
 *   The array is shared by every call and keeps the last call's contents;
 *   each call clears what it uses first.  Calls that overlap on the GPU
 *   (unordered streams) race on it: order them.
 *   The first call in each CUDA context (normally the device's primary
 *   context) looks up the array's address in that context and caches it; make
 *   it before any stream capture starts.  After cudaDeviceReset, or in another
 *   context the caller makes current, the next call looks it up again, so
 *   that call too belongs before any capture.
 *   Out-of-range route values are skipped but not recorded in the status word
 *   of mita_get_last_device_error.
 */
int mita_bucket_noalloc(const int32_t* route_idx, int B, int H, int N, int m, int s,
                        int32_t* bucket_off, int32_t* bucket_qidx, mita_stream_t stream);

/*
 * mita_expert_attn -- joint softmax over the shared pairs and the routed
 * expert's raw pairs, computed expert by expert.
 * Tutorial ch. 4 steps 5-6 (eq. 11-12): logits [q . q~_i / sqrt(d)]_{i<m}
 * followed by [q . k_j / sqrt(d)]_{j in expert}, one softmax, values
 * [v~_i] then [v_j].  With a precomputed shared partial the two branches are
 * merged by (Z1 o1 + Z2 o2) / (Z1 + Z2) (tutorial ch. 4).  With s > 1 each
 * query gets m + s*k logits: the raw pairs of all s of its experts (rows two
 * experts share count twice); every (query, expert) pair yields a partial and
 * the partials are merged per query by the same rule.
 *   q, k, v [B,H,N,d]; q_tilde [B,H,m,d]; v_tilde [B,H,m,d] float;
 *   topk_idx [B,H,m,topk]; bucket_off [B,H,m+1]; bucket_qidx [B,H,N*s]  inputs.
 *   shared_lse, shared_o   the partial from mita_route, or both NULL to
 *                          recompute the shared branch here.
 *   out [B,H,N,d]          output (every query appearing in bucket_qidx; with
 *                          s > 1 every query must appear in exactly s buckets,
 *                          else MITA_ERR_DEVICE_CHECK).
 * Indices outside their range are skipped and flag MITA_ERR_DEVICE_CHECK.
 */
int mita_expert_attn(const void* q, const void* k, const void* v, const void* q_tilde,
                     const float* v_tilde, const int32_t* topk_idx, const int32_t* bucket_off,
                     const int32_t* bucket_qidx, const float* shared_lse, const float* shared_o,
                     int B, int H, int N, int d, int m, int topk, int s, void* out,
                     mita_stream_t stream);
int mita_expert_attn_f32(const float* q, const float* k, const float* v, const float* q_tilde,
                         const float* v_tilde, const int32_t* topk_idx,
                         const int32_t* bucket_off, const int32_t* bucket_qidx,
                         const float* shared_lse, const float* shared_o, int B, int H, int N,
                         int d, int m, int topk, int s, float* out, mita_stream_t stream);

/*
 * mita_forward -- the whole MiTA forward pass (pool, landmark experts and
 * shared values, route, bucket, expert attention), gist.science summary
 * Sec. 2.3 Algorithm 1, tutorial ch. 4 eq. 5-12.
 *   q, k, v [B,H,N,d] inputs; out [B,H,N,d] output.  Intermediates live in
 *   the workspace cache.
 */
int mita_forward(const void* q, const void* k, const void* v, int B, int H, int N, int d,
                 int grid_h, int grid_w, int m, int topk, int s, void* out,
                 mita_stream_t stream);
int mita_forward_f32(const float* q, const float* k, const float* v, int B, int H, int N, int d,
                     int grid_h, int grid_w, int m, int topk, int s, float* out,
                     mita_stream_t stream);

/*
 * mita_forward_ex -- mita_forward with options (see mita_options; NULL gives
 * mita_forward).  Unknown option values return MITA_ERR_INVALID_ARG.
 */
int mita_forward_ex(const void* q, const void* k, const void* v, int B, int H, int N, int d,
                    int grid_h, int grid_w, int m, int topk, int s, const mita_options* options,
                    void* out, mita_stream_t stream);
int mita_forward_ex_f32(const float* q, const float* k, const float* v, int B, int H, int N,
                        int d, int grid_h, int grid_w, int m, int topk, int s,
                        const mita_options* options, float* out, mita_stream_t stream);

/*
 * mita_dense_attn -- dense softmax attention, out = softmax(q k^T / sqrt(d)) v
 * over all N keys of each (batch, head): the baseline of the long-sequence
 * throughput comparison (tutorial ch. 7, figure 5; bit.fan article,
 * throughput section).  q, k, v, out [B,H,N,d] device pointers; bf16 with
 * d = 64 runs on the tensor cores (the expert-attention kernel with one
 * expert of all keys per head), other shapes on SIMT cores.  Uses the
 * workspace cache.
 */
int mita_dense_attn(const void* q, const void* k, const void* v, int B, int H, int N, int d,
                    void* out, mita_stream_t stream);
int mita_dense_attn_f32(const float* q, const float* k, const float* v, int B, int H, int N,
                        int d, float* out, mita_stream_t stream);

/*
 * mita_backward -- gradients of mita_forward_ex's output with respect to q, k
 * and v.  The pages give no gradient through the selections; reading taken:
 * every landmark's top-k key set and every query's top-s landmarks are held
 * constant (top-k and argmax are piecewise constant) and q~'s rounding to the
 * input dtype passes the gradient straight through.  The gradient then flows
 * through the joint softmax (tutorial ch. 4 steps 5-6), the shared values
 * v~ = softmax(q~ K^T / sqrt(d)) V (steps 2-3) and the pooling (step 1).
 *   q, k, v, dout [B,H,N,d]  inputs (device, bf16 or fp32); dout = dL/dout.
 *   dq, dk, dv [B,H,N,d]     outputs, fp32 (device, 16-byte aligned like every
 *                            buffer here; cleared, then accumulated).
 *   options                  as for mita_forward_ex (NULL: the defaults).
 * Recomputes the forward's selections and partials with the forward's kernels,
 * then runs the gradient kernels: bf16 with d = 64 on the tensor cores (warp-
 * level MMAs; per pass, each query's D = sum of P dP over the same operands,
 * then dq query-major and dk / dv key-major), other shapes on SIMT cores.
 * Gradients are added with fp32 atomics, so results vary in the last bits
 * between runs.  Uses the workspace cache.
 */
int mita_backward(const void* q, const void* k, const void* v, const void* dout, int B, int H,
                  int N, int d, int grid_h, int grid_w, int m, int topk, int s,
                  const mita_options* options, float* dq, float* dk, float* dv,
                  mita_stream_t stream);
int mita_backward_f32(const float* q, const float* k, const float* v, const float* dout, int B,
                      int H, int N, int d, int grid_h, int grid_w, int m, int topk, int s,
                      const mita_options* options, float* dq, float* dk, float* dv,
                      mita_stream_t stream);

/*
 * mita_forward_host -- mita_forward on HOST buffers (same method and
 * parameters).  q, k, v [B,H,N,d] and out [B,H,N,d] are host pointers owned
 * by the caller; page-locked memory (cudaHostAlloc) copies at full speed,
 * pageable memory works but copies slower.  The call copies q, k, v to the
 * current device (a library-owned staging cache, one per (device, stream),
 * freed by mita_workspace_release), runs the forward on `stream`, copies the
 * output back into `out` and synchronises `stream` before returning: `out`
 * holds the result when the call returns MITA_OK.  The heads are split into
 * up to four groups that pipeline (copies in, forward, copies out on two
 * library-owned copy streams), and each group runs as its own batch, so the
 * result can differ in the last bits from one mita_forward over all heads.  Arguments are validated
 * before any copy; on an error `out` is left unspecified.
 */
int mita_forward_host(const void* q, const void* k, const void* v, int B, int H, int N, int d,
                      int grid_h, int grid_w, int m, int topk, int s, void* out,
                      mita_stream_t stream);
int mita_forward_host_f32(const float* q, const float* k, const float* v, int B, int H, int N,
                          int d, int grid_h, int grid_w, int m, int topk, int s, float* out,
                          mita_stream_t stream);

/* Bytes of workspace mita_forward needs for this shape (0 if invalid). */
uint64_t mita_forward_workspace_bytes(int B, int H, int N, int d, int m, int topk, int s,
                                      int is_f32);

/* Text for a status code (static storage). */
const char* mita_status_string(int status);

/* Detail of the last non-zero status returned on this host thread. */
const char* mita_last_error_message(void);

/*
 * Synchronises `stream`, reads and clears the current device's status word.
 * Returns MITA_OK if no kernel flagged bad input data since the last call,
 * MITA_ERR_DEVICE_CHECK otherwise (the flag bits go to *bits if non-NULL),
 * MITA_ERR_CUDA if the synchronisation itself failed.
 */
int mita_get_last_device_error(mita_stream_t stream, int* bits);

/* Frees every cached workspace (synchronises each owning device first). */
int mita_workspace_release(void);

/*
 * Caps the size one cached buffer (workspace or staging) may grow to; 0 removes
 * the cap.  A call that would grow a buffer past it returns MITA_ERR_OOM before
 * any allocation, exactly as when cudaMallocAsync fails, so callers can test
 * their out-of-memory handling without exhausting a GPU.  Buffers already
 * larger are kept.  Returns the previous cap.  Thread-safe.
 */
uint64_t mita_workspace_set_limit(uint64_t bytes);

/*
 * mita_check_bounded_wait -- exercises the failure path of the kernels' waits.
 * Not a step of the paper's method: a diagnostic.  Every wait inside this
 * library's kernels gives up after about one second (2^31 SM cycles), sets
 * the timeout bit (8) of the device status word and lets its kernel return, so
 * a lost arrival can never hang the GPU.  This call launches one small kernel
 * that waits, with the same two wait routines the kernels use, on an mbarrier
 * that nothing ever arrives on.
 *   gave_up  device int[2]: 1 where the whole-warp (index 0) and the
 *            single-thread (index 1) wait gave up, 0 where it completed.
 * Asynchronous on `stream`; about one second later the kernel has returned,
 * and mita_get_last_device_error reports bit 8.  Other work on the device is
 * unaffected.  Returns MITA_ERR_INVALID_ARG for a NULL gave_up.
 */
int mita_check_bounded_wait(int* gave_up, mita_stream_t stream);

/*
 * Number of kernel launches this library has issued in this process so far
 * (all devices, all threads; a launch counts when it is enqueued).  The
 * difference of two readings around a section of host code is the number of
 * library kernels that section launched.  Never fails.
 */
uint64_t mita_kernel_launches(void);

#ifdef __cplusplus
}
#endif

#endif /* MITA_H_ */
