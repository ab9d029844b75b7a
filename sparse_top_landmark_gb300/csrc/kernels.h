// Host-side launchers of the MiTA kernels (internal; the C-ABI is in mita.h).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace mita {

// ---- step 1: landmark pooling --------------------------------------------
// onto an mh x mw landmark grid (m = mh * mw; 1D: mh = 1)
template <typename T>
cudaError_t launch_pool(const T* q, int BH, int N, int d, int grid_h, int grid_w,
                        int mh, int mw, T* q_tilde, cudaStream_t st);

// ---- steps 2-3: landmark top-k experts + shared values --------------------
struct LandmarkPlan {
  bool tc;        // tensor-core two-pass path (bf16, d = 64, long N)
  int RT;         // landmark rows per CTA (32, 64 or 128)
  int nrt;        // row tiles per head
  int Tcap;       // candidates kept per (row, split)          (SIMT path)
  int S;          // key splits per head
  int split_len;  // keys per split (last one may be shorter)
  int P;          // padded candidate count per row in the merge (power of 2)
  int ntiles;     // 128-key tiles per head                      (tc path)
  int cap;        // candidate capacity per row                  (tc and small paths)
  bool small = false;   // N <= 1024 without the tc path: every key is a candidate
};

struct LandmarkWs {
  float* M;        // [BH, m, S]      running max (log2 domain, scaled)
  float* L;        // [BH, m, S]      softmax denominator at that max
  float* A;        // [BH, m, S, d]   unnormalised numerator
  float* cs;       // [BH, m, S, Tcap] candidate scores (unscaled fp32 dots)
  int* ci;         // [BH, m, S, Tcap] candidate key indices
  int* cn;         // [BH, m, S]       candidates kept
  float* theta;    // [BH, m, S]       worst kept score if the split dropped keys, else -inf
  float* kmax2;    // [BH, S(, nrt)]   max squared key norm per split (tensor-core path: a
                   // partial maximum per 128-landmark block of the split)
  int* nslow;      // [1]              rows routed to the exact fallback
  int* slow_rows;  // [BH * m]
  double* exact;   // [kExactCtas, N]  fp64 score scratch of the fallback
  // tensor-core path (M/L/A then hold 2 partials per split: one per softmax slot)
  float* bm;       // [BH*m, ntiles]  every key tile's maximum raw score per landmark
  float* thr;      // [BH, m]          collection threshold tau_L - 4E
  float* E;        // [BH, m]          fp32 score error bound
  int* cnt;        // [BH, m]          candidates collected
  float* cand_s;   // [BH, m, cap]
  int* cand_i;     // [BH, m, cap]
  float* lse_out;  // [BH, m] or null: ln sum_j exp(q~_i . k_j / sqrt(d)) of every landmark
                   // (the softmax normaliser behind v~; the backward reads it)
};

LandmarkPlan plan_landmark(int BH, int N, int d, int m, int topk, int num_sms, bool bf16_input);
size_t landmark_ws_bytes(const LandmarkPlan& p, int BH, int N, int d, int m);
LandmarkWs carve_landmark_ws(void* base, const LandmarkPlan& p, int BH, int N, int d, int m);

template <typename T>
cudaError_t launch_landmark(const T* q_tilde, const T* k, const T* v, int BH, int N, int d,
                            int m, int topk, const LandmarkPlan& plan, const LandmarkWs& ws,
                            int32_t* topk_idx, float* v_tilde, int* status, cudaStream_t st,
                            bool prezeroed = false);   // ws.nslow already cleared on the stream

bool landmark_tc_eligible(int d, int N, int topk);
void plan_landmark_tc(LandmarkPlan& p, int BH, int N, int m, int topk, int num_sms);
cudaError_t launch_landmark_tc_passes(const __nv_bfloat16* q_tilde, const __nv_bfloat16* k,
                                      const __nv_bfloat16* v, int BH, int N, int m, int topk,
                                      const LandmarkPlan& p, const LandmarkWs& ws, float* v_tilde,
                                      int* status, cudaStream_t st);

// ---- step 4: routing (optionally emitting the shared-branch partial) ------
// route_idx: [BH, N, s], each query's s landmarks best first (1 <= s <= kMaxRouteS).
// shared_temp: the shared partial's logits are q . q~ / sqrt(d) (0) or q . q~ / d (1).
template <typename T>
cudaError_t launch_route(const T* q, const T* q_tilde, const float* v_tilde, int BH, int N,
                         int d, int m, int s, int32_t* route_idx, float* shared_lse,
                         float* shared_o, cudaStream_t st, int shared_temp = 0);

// ---- step 5: stable grouping of queries by expert -------------------------
constexpr int kBucketChunk = 4096;   // route entries per chunk
// `entries` = N * s route entries per head
size_t bucket_ws_bytes(int BH, int entries, int m);
// ws: [BH][m][nchunks] per-chunk counts, then [BH][m] totals.  counted = the counts are
// already in ws (left by launch_route_tc's histogram).  route_idx is [BH, N, s];
// bucket_qidx receives [BH, N * s] query indices.
cudaError_t launch_bucket(const int32_t* route_idx, int BH, int N, int m, void* ws,
                          int32_t* bucket_off, int32_t* bucket_qidx, int* status,
                          cudaStream_t st, bool counted = false, int s = 1);

// ---- step 6: expert-grouped joint attention -------------------------------
// Per (query, expert) partials over the expert's raw pairs: slot t < s of query qi.
struct ExpertPartials {
  float* lse;   // [BH*N, s]     natural log-sum-exp
  float* o;     // [BH*N, s, d]  softmax-weighted mean of the expert's V rows
  int* pos;     // [BH*N, s]     bucket position of the (query, expert) entry
  int* cnt;     // [BH*N]        slots taken (cleared by the launcher)
};
// the raw-pair partials only (no shared pairs, no merge), for any s >= 1
template <typename T>
cudaError_t launch_expert_partials(const T* q, const T* k, const T* v, const int32_t* topk_idx,
                                   const int32_t* bucket_off, const int32_t* bucket_qidx, int BH,
                                   int N, int d, int m, int topk, int s, ExpertPartials part,
                                   int* status, cudaStream_t st);
// s > 1 needs the shared partial (shared_lse, shared_o) and `ws` of
// expert_partials_ws_bytes(BH, N, d, s) bytes for the per-expert partials.
size_t expert_partials_ws_bytes(int BH, int N, int d, int s);
// the partial arrays inside such a workspace (lse, o, pos, then the slot counters)
ExpertPartials carve_expert_partials(void* ws, int BH, int N, int d, int s);
// out = the branch-merge of the shared partial (none when shared_lse is null) and each
// query's s raw partials, taken in ascending bucket position
// (shared_o in bf16 when so_bf16, else fp32)
template <typename T>
cudaError_t launch_expert_merge(const float* shared_lse, const void* shared_o, int so_bf16,
                                ExpertPartials part, int BH, int N, int d, int s, T* out,
                                int* status, cudaStream_t st);
template <typename T>
cudaError_t launch_expert_attn(const T* q, const T* k, const T* v, const T* q_tilde,
                               const float* v_tilde, const int32_t* topk_idx,
                               const int32_t* bucket_off, const int32_t* bucket_qidx,
                               const float* shared_lse, const float* shared_o, int BH,
                               int N, int d, int m, int topk, int s, void* ws, T* out,
                               int* status, cudaStream_t st, int shared_temp = 0,
                               int routed_only = 0);
// dense softmax attention (SIMT, any supported d): scratch of dense_simt_ws_bytes
size_t dense_simt_ws_bytes(int BH, int N);
template <typename T>
cudaError_t launch_dense_attn(const T* q, const T* k, const T* v, int BH, int N, int d, void* ws,
                              T* out, int* status, cudaStream_t st);

// ---- tensor-core (tcgen05) kernels: bf16, d = 64 ---------------------------
// TMA map over a [batches, rows, 64] bf16 array, boxes of box_rows rows.
bool make_tmap_rows64(CUtensorMap* map, const void* base, uint64_t rows, uint64_t batches,
                      uint32_t box_rows, bool fp16 = false);
// TMA map over a [rows, 64] bf16 array for tile::gather4 (four scattered rows).
bool make_tmap_gather64(CUtensorMap* map, const void* base, uint64_t rows);
bool route_tc_supported(int d, int m);
// `amb` is scratch of BH*(2N+1) words: the heads' counts, then per head the ambiguous
// query ids and their fp32 best scores.  `hist`, if not null, receives the bucket
// stage's per-chunk expert counts ([BH][m][ceil(N / kBucketChunk)], cleared here), so
// that launch_bucket(..., counted = true) can skip its counting pass.
cudaError_t launch_route_tc(const __nv_bfloat16* q, const __nv_bfloat16* q_tilde, int BH, int N,
                            int m, int num_sms, int32_t* route, int* amb, int* status, int* hist,
                            cudaStream_t st, bool prezeroed = false);   // amb counts, hist cleared

// exact re-routing of the queries route_tc / route_shared_tc left on the heads'
// ambiguous lists in `amb` (counted into `hist` under their exact route, if not null)
cudaError_t launch_route_fixup(const __nv_bfloat16* q, const __nv_bfloat16* q_tilde, int BH,
                               int N, int m, int num_sms, int32_t* route, const int* amb,
                               int* hist, cudaStream_t st);
// exact top-s re-routing (2 <= s <= 8) of the queries route_shared_tc (s = 2) left on the
// ambiguous lists in `amb`; route is [BH*N][s]; their N*s entries counted into `hist`
// ([BH][m][ceil(N*s / kBucketChunk)]) if not null
cudaError_t launch_route_fixup_top(const __nv_bfloat16* q, const __nv_bfloat16* q_tilde, int BH,
                                   int N, int m, int s, int num_sms, int32_t* route,
                                   const int* amb, int* hist, cudaStream_t st);
// Routing (s = 1, or the best two with s = 2) together with the shared branch's partial from
// the same logits: per query the route ([BH*N][s], best first), shared_lse (natural
// log-sum-exp of the scaled shared logits) and shared_o = the normalised shared output,
// [BH*N][64] in bf16 (o_bf16 = 1) or fp32.  `amb` and `hist` as for launch_route_tc (the
// fix-up runs inside; with s = 2 `hist` counts the N*s entries, [BH][m][ceil(2N / chunk)]).
bool route_shared_tc_supported(int d, int m, int s = 1);
cudaError_t launch_route_shared_tc(const __nv_bfloat16* q, const __nv_bfloat16* q_tilde,
                                   const float* v_tilde, int BH, int N, int m, int num_sms,
                                   int shared_temp, int o_bf16, int32_t* route,
                                   float* shared_lse, void* shared_o, int* amb, int* status,
                                   int* hist, cudaStream_t st, bool prezeroed = false,
                                   int s = 1);

bool expert_tc_supported(int d, int m, int topk);
size_t expert_tc_ws_bytes(int BH, int N, int m, int topk);
// top-s (s > 1) raw-pair partials on the tensor cores: one per (query, expert) entry of the
// N*s-entry buckets, into `part` (its slot counters are cleared here); ws of
// expert_tc_partials_ws_bytes bytes
size_t expert_tc_partials_ws_bytes(int BH, int N, int m, int topk, int s);
cudaError_t launch_expert_tc_partials(const __nv_bfloat16* q, const __nv_bfloat16* k,
                                      const __nv_bfloat16* v, const int32_t* topk_idx,
                                      const int32_t* bucket_off, const int32_t* bucket_qidx,
                                      int BH, int N, int m, int topk, int s, int num_sms,
                                      void* ws, ExpertPartials part, int* status,
                                      cudaStream_t st);
cudaError_t launch_expert_tc(const __nv_bfloat16* q, const __nv_bfloat16* k,
                             const __nv_bfloat16* v, const __nv_bfloat16* q_tilde,
                             const float* v_tilde, const int32_t* topk_idx,
                             const int32_t* bucket_off, const int32_t* bucket_qidx, int BH, int N,
                             int m, int topk, int num_sms, void* ws, __nv_bfloat16* out,
                             int* status, cudaStream_t st, int shared_temp = 0,
                             int routed_only = 0, const float* shared_lse = nullptr,
                             const void* shared_o = nullptr, int o_bf16 = 0);
// Short sequences (N <= 1024): per-head query tiles over the shared pairs and all N keys,
// each query's raw keys masked to its routed expert's top-k set; no bucket stage (route is
// [BH, N] s = 1).  expert_masked_preferred: fewer MMA chunks than the grouped form.
bool expert_masked_preferred(int N, int m, int topk, int routed_only);
size_t expert_masked_ws_bytes(int BH, int N, int m);
cudaError_t launch_expert_masked_tc(const __nv_bfloat16* q, const __nv_bfloat16* k,
                                    const __nv_bfloat16* v, const __nv_bfloat16* q_tilde,
                                    const float* v_tilde, const int32_t* topk_idx,
                                    const int32_t* route, int BH, int N, int m, int topk,
                                    int num_sms, void* ws, __nv_bfloat16* out, int* status,
                                    cudaStream_t st, int shared_temp, int routed_only);
// dense softmax attention of every query over all N keys of its head (bf16, d = 64)
size_t dense_tc_ws_bytes(int BH, int N);
cudaError_t launch_dense_tc(const __nv_bfloat16* q, const __nv_bfloat16* k,
                            const __nv_bfloat16* v, int BH, int N, int num_sms, void* ws,
                            __nv_bfloat16* out, int* status, cudaStream_t st);

// ---- backward (selections held constant) ------------------------------------
template <typename T>
struct BwdArgs {
  const T *q, *k, *v, *dout, *q_tilde;    // inputs, upstream gradient, the forward's q~
  const float* v_tilde;                   // the forward's v~
  const int32_t *topk_idx, *bucket_off, *bucket_qidx;
  const float *sh_lse, *sh_o;             // the shared branch's partial (null: routing only)
  ExpertPartials part;                    // the raw partials of every (query, expert)
  int BH, N, m, topk, s, routed;
  float c_sh;                             // shared-logit scale (1/sqrt(d) or 1/d)
  int grid_h, grid_w, mh, mw;             // token grid and landmark grid
  float *lse, *Dn;                        // [BH*N] scratch
  float *lseA, *cvt;                      // [BH*m] scratch
  float *dqt, *dvt;                       // [BH*m*d] scratch, cleared
  float *dq, *dk, *dv;                    // [BH*N*d] outputs, cleared
  int* status;
  // bf16 with d = 64: [BH*m*64] scratch for bf16 copies of v~ and dv~; when both are set the
  // gradient passes run on the tensor cores (backward_mma.cu), else on SIMT cores
  __nv_bfloat16 *vt16, *dvt16;
};
template <typename T>
cudaError_t launch_backward(const BwdArgs<T>& a, int d, cudaStream_t st);

// One gradient pass of the backward on the tensor cores (bf16 rows of 64, fp32 results):
// queries (q, g, L, D) against keys (k, v) under logit scale c, P = exp(c q.k - L),
// dS = P (g.v - D); kind 0 (query-major) adds c dS k to dq; kind 1 (key-major) adds
// c dS^T q to dk and P^T g to dv (a null output is skipped); kind 2 (query-major) adds
// each query's sum of P (g.v) over the pass's keys to Dacc; kind 3 (joint, routed segments,
// each query in one segment: s = 1) streams each expert's top-k rows and then the head's n2
// rows of (k2, v2) under scale c2 twice -- first to sum D, stored to Dacc, then for dq,
// stored (`first` must be set).  Segments: with bucket_off set, one per (head, expert)
// -- queries n = bucket_qidx[bh][off[e] ..] and keys j = topk_idx[bh][e][0 .. topk), rows
// bh*N + n and bh*N + j -- else one per head with nq query rows at bh*nq and nk key rows at
// bh*nk.  Outputs 16-byte aligned.  `first`: no earlier launch wrote the outputs and each
// owned row lies in one segment, so the results are stored, not added (the launcher refuses
// it when the stream would be split over CTAs: longer than kBwdSplitRows rows).  `items` is
// set by the launcher.
struct BwdPass {
  const __nv_bfloat16 *q, *g, *k, *v;
  const float *L, *D;
  float *dq, *dk, *dv, *Dacc;
  float c;
  const __nv_bfloat16 *k2, *v2;   // joint: the second key set (rows bh*n2 ..), scale c2
  float c2;
  int n2;
  int BH, nq, nk;
  const int32_t *bucket_off, *bucket_qidx, *topk_idx;
  int N, m, topk, NS, items, first;
  int* status;
};
constexpr int kBwdSplitRows = 1024;   // streamed rows per CTA of the tensor-core passes
cudaError_t launch_bwd_pass_mma(BwdPass p, int kind, cudaStream_t st);

int num_sms_of_current_device();

// Records one kernel launch by this library (process-wide counter behind
// mita_kernel_launches()).
void count_launch();

// Records `text` as the message mita_last_error_message() returns on this
// thread and returns `code`.
int report_error(int code, const char* text);

// A one-CTA kernel whose two bounded waits (whole-warp and single-thread) run out on an
// mbarrier nothing arrives on: each flags kDevErrTimeout in *status and writes 1 to
// gave_up[0] / gave_up[1] (device memory) when it gave up.
cudaError_t launch_bounded_wait_probe(int* status, int* gave_up, cudaStream_t st);

}  // namespace mita
