/*
 * ls.h -- C ABI of the response-replay attention library (libls).
 *
 * The operator: exact response-replay attention for GRPO post-training with a
 * shared, detached long prompt.  The prompt is run once without gradients and
 * its full-attention K/V are kept as compact pages (the capture step of the
 * LongStraw DeepRead summary, section Method).  Each group member's short
 * response is then replayed on its own: its queries attend over every prompt
 * key through the page table and causally over the response's own keys,
 * partial results are recombined exactly by log-sum-exp (the Qwen path's
 * global merge in the same section; the LongStraw abstract on exact attention
 * composition), and the backward treats the prompt K/V as constants (the
 * stored prompt state is stop-gradient, DeepRead summary, Method, last
 * paragraph; the review's mind map, node on equations 1-3: the
 * d(loss)/d(z_P) d(z_P)/d(theta) term is omitted).
 *
 * Conventions shared by every call
 * --------------------------------
 *  Shapes: Hq query heads, Hkv KV heads (Hq % Hkv == 0), head dim d, page
 *  size S_p; query head h reads KV head h / (Hq/Hkv).  R = response length,
 *  P = prompt length.  Response row i sees all P prompt keys and response keys
 *  j <= i.  The softmax scale is a parameter (normally 1/sqrt(d)).
 *  Layouts (all row-major, contiguous, device memory unless stated):
 *    prompt pools   k_pool, v_pool : [pool_pages][Hkv][S_p][d]   element dtype
 *    page table                    : int32 [num_pages], logical page -> slot
 *    q, d_o, o, dq                 : [R][Hq][d]                  element dtype
 *    k_resp, v_resp, dk, dv        : [R][Hkv][d]                 element dtype
 *    lse, delta                    : float32 [R][Hq]; lse is the natural log
 *                                    of the softmax denominator, scale included
 *  Element dtype is uniform per call (LS_DTYPE_F32 or LS_DTYPE_BF16);
 *  accumulation is always float32.
 *
 *  Ownership: the caller allocates every buffer and keeps each one alive
 *  until the work that reads it has finished on its stream; the structs
 *  (ls_prompt_kv, ls_member) only hold pointers.  The library never allocates
 *  or frees device memory.  It keeps a small host-side cache (tensor-map
 *  descriptors) and per-process trace counters, nothing else.  The prompt
 *  pools are read-only for every replay call.
 *
 *  Workspace: one caller-owned device buffer of ls_replay_workspace_size()
 *  bytes, sized for the longest response, reused by every member (the
 *  workspace does not grow with the group size).  Its first 256 bytes hold a
 *  device status word that kernels set on device-side errors.
 *
 *  Errors: every call validates its arguments on the host before any launch
 *  and returns a status; nothing aborts.  Device-side problems set bits in
 *  the workspace status word: a page-table entry outside the pool (that page
 *  is then treated as holding no keys: nothing is read from it and it adds
 *  nothing to the softmax), or a bounded wait that ran out (the affected work
 *  is skipped).  The call itself has already returned LS_OK by then, so read
 *  them with ls_read_device_status().
 *  ls_last_error() gives a one-line reason for the last failing call on the
 *  calling thread.
 *
 *  Streams: every compute call is asynchronous on the given stream
 *  (a cudaStream_t passed as void*; NULL = legacy default stream).  Calls are
 *  thread-safe when they use distinct workspaces.
 */
#ifndef LS_H_
#define LS_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define LS_API __attribute__((visibility("default")))
#else
#define LS_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LS_OK = 0,
  LS_ERR_INVALID_ARGUMENT = 1,   /* null pointer, bad size, misaligned buffer */
  LS_ERR_UNSUPPORTED = 2,        /* valid but unsupported shape or dtype */
  LS_ERR_WORKSPACE_TOO_SMALL = 3,
  LS_ERR_CUDA = 4,               /* a CUDA runtime/driver call failed */
  LS_ERR_DEVICE_BOUNDS = 5,      /* device saw a page id outside the pool */
  LS_ERR_DEVICE_TIMEOUT = 6      /* a device-side bounded wait ran out */
} ls_status;

typedef enum { LS_DTYPE_F32 = 0, LS_DTYPE_BF16 = 1 } ls_dtype;

/* Shape and numerics of one attention layer.
 * dtype: ls_dtype of every element buffer.  head_dim in {64, 128, 256};
 * page_size >= 1.  softmax_scale > 0 and finite. */
typedef struct {
  int32_t dtype;
  int32_t hq;
  int32_t hkv;
  int32_t head_dim;
  int32_t page_size;
  float softmax_scale;
} ls_attn_desc;

/* The captured prompt of one layer: pools plus page table (device pointers).
 * Logical prompt position t lives in slot page_table[t / page_size] at row
 * t % page_size.  Requires num_pages * page_size >= prompt_len; rows of the
 * last page beyond prompt_len are never read as keys (they may hold anything,
 * NaN included). */
typedef struct {
  const void* k_pool;
  const void* v_pool;
  int64_t pool_pages;
  const int32_t* page_table;
  int64_t num_pages;
  int64_t prompt_len;
} ls_prompt_kv;

/* One group member for ls_replay_group.  Inputs q, k, v, d_o; outputs o, lse,
 * delta (rowsum(dO*O), written as a by-product), dq, dk, dv. */
typedef struct {
  const void* q;
  const void* k;
  const void* v;
  const void* d_o;
  int32_t resp_len;
  int32_t reserved;
  void* o;
  float* lse;
  float* delta;
  void* dq;
  void* dk;
  void* dv;
} ls_member;

/* A1. Capture-side page write (DeepRead summary, Method, the capture step;
 * review section 二.2: the full-attention layers keep their K/V in pages).
 * Scatters token t of k, v ([n_tok][Hkv][d]) to
 *   pool[page_table[(start_pos+t)/S_p]][kv][(start_pos+t)%S_p][:].
 * page_table holds num_pages entries; requires start_pos + n_tok <=
 * num_pages * S_p.  Entries outside [0, pool_pages) are skipped on the device
 * and, if ws is non-NULL, reported through its status word.  Bit-exact copy.
 * ws may be NULL (then ws_bytes is ignored). */
LS_API ls_status ls_kv_page_write(const ls_attn_desc* desc, void* k_pool, void* v_pool,
                           int64_t pool_pages, const int32_t* page_table,
                           int64_t num_pages, int64_t start_pos, int64_t n_tok,
                           const void* k, const void* v, void* ws, size_t ws_bytes,
                           void* stream);

/* Workspace bytes needed by ls_replay_fwd / ls_replay_bwd / ls_replay_group
 * for responses of up to max_resp_len tokens against this prompt on the
 * current device.  Host-only; does not touch the device. */
LS_API ls_status ls_replay_workspace_size(const ls_attn_desc* desc, const ls_prompt_kv* prompt,
                                   int32_t max_resp_len, size_t* bytes);

/* A2+A3+A4. Replay forward: O [R][Hq][d] (element dtype) and LSE [R][Hq]
 * (float32, natural log, scale included) of softmax attention over all prompt
 * keys plus the causal response keys.  The prompt part runs split over page
 * ranges into float32 partials held in ws, the response part adds one more
 * partial, and an exact LSE merge writes o and lse (DeepRead summary,
 * Method, Qwen path).  resp_len == 0 is a no-op. */
LS_API ls_status ls_replay_fwd(const ls_attn_desc* desc, const ls_prompt_kv* prompt,
                        const void* q, const void* k_resp, const void* v_resp,
                        int32_t resp_len, void* o, float* lse, void* ws, size_t ws_bytes,
                        void* stream);

/* A4. Exact log-sum-exp merge of partial attention results (the global
 * LSE and output merge of the DeepRead summary, Method):
 *   L[n] = log sum_s exp(Lp[s][n]);  O[n] = sum_s exp(Lp[s][n] - L[n]) Op[s][n].
 * o_parts float32 [n_parts][n_rows][head_dim], lse_parts float32
 * [n_parts][n_rows], natural log; a part with Lp = -inf contributes nothing;
 * a row whose parts are all -inf gets O = 0, L = -inf.  o is written in
 * out_dtype, lse as float32 (lse may be NULL).  head_dim % 4 == 0. */
LS_API ls_status ls_lse_merge(int32_t n_parts, int64_t n_rows, int32_t head_dim,
                       const float* o_parts, const float* lse_parts, int32_t out_dtype,
                       void* o, float* lse, void* stream);

/* A5. Backward preprocess: delta[r][h] = sum_c dO[r][h][c] * O[r][h][c]
 * (float32 accumulation of the element-dtype inputs). */
LS_API ls_status ls_replay_bwd_preprocess(const ls_attn_desc* desc, const void* o, const void* d_o,
                                   int32_t resp_len, float* delta, void* stream);

/* A6+A7. Replay backward with the prompt state detached (DeepRead summary,
 * Method: stored prompt state is stop-gradient; review section 二, last
 * paragraph: on the Qwen path only the query gradient crosses ranks).
 * Recomputes P = exp(s - LSE) from the stored lse (no score matrix is kept),
 * dS = P * (dO.v - delta), and returns
 *   dq      [R][Hq][d]  = scale * sum over prompt and visible response keys of dS k
 *   dk_resp [R][Hkv][d] = scale * sum over the group's heads, rows i >= j of dS q
 *   dv_resp [R][Hkv][d] = sum over the group's heads, rows i >= j of P dO
 * No gradient is produced for prompt K/V.  lse and delta come from
 * ls_replay_fwd and ls_replay_bwd_preprocess. */
LS_API ls_status ls_replay_bwd(const ls_attn_desc* desc, const ls_prompt_kv* prompt,
                        const void* q, const void* k_resp, const void* v_resp,
                        const void* d_o, const float* lse, const float* delta,
                        int32_t resp_len, void* dq, void* dk_resp, void* dv_resp,
                        void* ws, size_t ws_bytes, void* stream);

/* A8. Serial replay of a group's response suffixes (DeepRead summary, Method;
 * abstract: one response at a time is rebuilt under autograd and
 * backpropagated, back to the prompt boundary).  For each member in order:
 * forward, preprocess, backward, all on one stream and into the one workspace,
 * so only one member's intermediates are live and the workspace does not grow
 * with n_members.  Each member's results equal a standalone replay of it. */
LS_API ls_status ls_replay_group(const ls_attn_desc* desc, const ls_prompt_kv* prompt,
                          int32_t n_members, const ls_member* members, void* ws,
                          size_t ws_bytes, void* stream);

/* Context parallelism, one rank's share (DeepRead summary, Method, Qwen path:
 * the prompt pages are sharded over ranks and the partial results are merged
 * globally by LSE; review section 二: the query gradient is what crosses
 * ranks).  `prompt` holds the pages this rank owns, in any order: attention
 * over a set of keys does not depend on their order.  Every rank holds the
 * whole response (q, k_resp, v_resp, d_o).  Exactly one rank passes
 * with_response != 0 and adds the causal response keys.
 *
 * ls_replay_fwd_part writes the rank's exact partial in float32: o_part
 * [R][Hq][d], normalised over the rank's keys, and lse_part [R][Hq].  A rank
 * with no visible key gets O = 0 and LSE = -inf.  The global O, LSE is
 * ls_lse_merge over all ranks' partials (an all-gather, then the merge).
 *
 * ls_replay_bwd_part writes dq_part float32 [R][Hq][d], the rank's share of
 * dQ with the scale applied.  The global dQ is the sum over ranks (an
 * all-reduce).  lse and delta must be the global ones (from the merged
 * forward).  dk_resp and dv_resp are written only with_response, and may be
 * NULL otherwise.  Workspace: ls_replay_workspace_size for the rank's prompt.
 * The interface is this library's; the pages describe the split, not a call. */
LS_API ls_status ls_replay_fwd_part(const ls_attn_desc* desc, const ls_prompt_kv* prompt,
                                    const void* q, const void* k_resp, const void* v_resp,
                                    int32_t resp_len, int32_t with_response, float* o_part,
                                    float* lse_part, void* ws, size_t ws_bytes, void* stream);
LS_API ls_status ls_replay_bwd_part(const ls_attn_desc* desc, const ls_prompt_kv* prompt,
                                    const void* q, const void* k_resp, const void* v_resp,
                                    const void* d_o, const float* lse, const float* delta,
                                    int32_t resp_len, int32_t with_response, float* dq_part,
                                    void* dk_resp, void* dv_resp, void* ws, size_t ws_bytes,
                                    void* stream);

/* Sum of float32 partials: out[i] = sum_s parts[s][i] (float32
 * accumulation, in part order), written in out_dtype.  parts float32
 * [n_parts][n_elems], 16-byte aligned; n_elems % 4 == 0; n_parts == 0 writes
 * zeros.  The dQ reduction of A6 as a call of its own, for callers that hold
 * several dQ shares (context-parallel ranks without a collective, or prompt
 * pages streamed from host memory in chunks). */
LS_API ls_status ls_sum_parts(int32_t n_parts, int64_t n_elems, const float* parts,
                              int32_t out_dtype, void* out, void* stream);

/* Staging of prompt pages kept outside HBM (the GLM path of the DeepRead
 * summary, Method, keeps its prompt state in CPU memory and stages it per
 * layer; on GB300 the Grace memory sits behind the coherent CPU-GPU link).
 * Copies logical pages first_page .. first_page + n_pages - 1 of a prompt,
 * K and V, from source pools [src_pages][Hkv][S_p][d] into staging pools
 * [n_pages][Hkv][S_p][d], in logical order:
 *   k_dst[i] = k_src[page_table[first_page + i]], likewise v.
 * The GPU reads the sources directly (one kernel, no copy-engine calls), so
 * they must be device memory or pinned host memory (pageable host memory is
 * refused with LS_ERR_INVALID_ARGUMENT).  page_table is device memory and
 * holds at least first_page + n_pages entries; the staging pools hold
 * n_pages pages.  An entry outside [0, src_pages) zeroes its staging page and
 * is reported through the status word of ws (ws may be NULL).  Pages are
 * copied bit for bit.  0 <= n_pages <= 65535.  The interface is this
 * library's. */
LS_API ls_status ls_stage_pages(const ls_attn_desc* desc, const void* k_src, const void* v_src,
                                int64_t src_pages, const int32_t* page_table, int64_t first_page,
                                int32_t n_pages, void* k_dst, void* v_dst, void* ws,
                                size_t ws_bytes, void* stream);

/* Gated-DeltaNet state replay (the Qwen model's recurrent layers keep a
 * fixed-size state for the prompt and replay each response from it with that
 * state detached: DeepRead summary, Method, Qwen path; review sections 二,
 * 三).  The pages name the layer but not its recurrence.  This library takes
 * the published gated delta rule, per member and head, with S [dv][dk] and
 * S_0 the captured state:
 *   a_t = exp(g_t);  S_t = a_t S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T;
 *   o_t = S_t q_t.
 * A call replays `batch` members of one group, all of resp_len tokens, from
 * one shared S_0.  float32 throughout, row-major, device memory:
 *   s0 [H][dv][dk] (shared);  s_final [B][H][dv][dk];
 *   q, k [B][R][H][dk];  v, o [B][R][H][dv];  g, beta [B][R][H].
 * Supported: dk = dv = 128.  s0 and the token buffers are read only.
 * ls_gdn_replay_fwd writes o and, if s_final is non-NULL, the state after the
 * last token.  ls_gdn_replay_bwd returns the gradient of sum(d_o * o) for q,
 * k, v, g and beta (same shapes); none is formed for s0 (the detached prompt
 * state).  The backward, and the forward with LS_GDN_TENSOR_CORE, need
 * ls_gdn_workspace_size() bytes of workspace (256-byte aligned, owned by the
 * caller; the forward with LS_GDN_EXACT takes ws = NULL, ws_bytes = 0, and
 * ignores a workspace it is given).  The workspace starts with the same
 * 256-byte device status word as the attention workspace: a bounded device
 * wait that ran out in the tensor-core path sets it, and
 * ls_read_device_status(ws) reports it (the outputs of that call are then
 * not to be used).  resp_len == 0 or batch == 0 is a no-op (the forward still
 * copies s0 to s_final when R = 0).
 *
 * precision selects the kernels (a zeroed desc selects the exact path):
 *   LS_GDN_EXACT        float32 recurrence, one token at a time; about 1e-7
 *                       relative error, held to 1e-5 against the float64
 *                       oracle.
 *   LS_GDN_TENSOR_CORE  the chunk-parallel forward and backward (chunks of
 *                       128 tokens) on tcgen05 tensor cores with bf16
 *                       operands and float32 accumulation; about 5e-3
 *                       relative error, held to 2e-2 (the bf16 bar).  s0, q,
 *                       k, v, d_o and the outputs must be 16-byte aligned
 *                       (else LS_ERR_CUDA).
 * Float32 callers that need the 1e-5 result keep LS_GDN_EXACT.
 * Errors: LS_ERR_UNSUPPORTED for other dk/dv, LS_ERR_INVALID_ARGUMENT for
 * NULL buffers, negative sizes, an unknown precision or unknown flags,
 * LS_ERR_WORKSPACE_TOO_SMALL; all before any launch. */
typedef enum { LS_GDN_EXACT = 0, LS_GDN_TENSOR_CORE = 1 } ls_gdn_precision;

/* flags (0 by default):
 *   LS_GDN_BWD_REUSES_FORWARD  with LS_GDN_TENSOR_CORE, the backward takes the
 *       forward's per-chunk terms and states from ws instead of forming them
 *       again: the caller promises that ws was last written by
 *       ls_gdn_replay_fwd with the same desc precision, buffers and resp_len
 *       (the inputs unchanged since).  The results are then the ones the
 *       backward forms without the flag, bit for bit; if the promise is
 *       broken they are wrong (every access still stays inside ws).  Ignored
 *       by LS_GDN_EXACT. */
enum { LS_GDN_BWD_REUSES_FORWARD = 1 };

typedef struct {
  int32_t batch;
  int32_t heads;
  int32_t dk;
  int32_t dv;
  int32_t precision; /* ls_gdn_precision */
  int32_t flags;     /* LS_GDN_BWD_REUSES_FORWARD or 0 */
} ls_gdn_desc;

LS_API ls_status ls_gdn_workspace_size(const ls_gdn_desc* desc, int32_t resp_len, size_t* bytes);
LS_API ls_status ls_gdn_replay_fwd(const ls_gdn_desc* desc, const float* s0, const float* q,
                                   const float* k, const float* v, const float* g,
                                   const float* beta, int32_t resp_len, float* o, float* s_final,
                                   void* ws, size_t ws_bytes, void* stream);
LS_API ls_status ls_gdn_replay_bwd(const ls_gdn_desc* desc, const float* s0, const float* q,
                                   const float* k, const float* v, const float* g,
                                   const float* beta, const float* d_o, int32_t resp_len,
                                   float* dq, float* dk, float* dv, float* dg, float* dbeta,
                                   void* ws, size_t ws_bytes, void* stream);

/* Prompt prefill with capture (the capture step of the DeepRead summary,
 * Method: the shared prompt is run once without gradients and its
 * full-attention K/V are kept as pages; the summary's Key Results put most
 * of the wall time in this no-gradient prefill).  Two steps on one stream:
 *   1. page write, as ls_kv_page_write with start_pos 0: token t of k, v
 *      ([n_tok][Hkv][d]) goes to pool[page_table[t/S_p]][kv][t%S_p][:];
 *   2. causal self-attention of the prompt: o [n_tok][Hq][d] (element dtype)
 *      and lse float32 [n_tok][Hq] (natural log, scale included), row t over
 *      keys 0..t of k, v (read from the contiguous k, v, not the pages).
 * Step 2 is the replay forward with an empty prompt and the prompt in the
 * response's place, so it runs on the same kernels.  ws must hold
 * ls_prompt_prefill_workspace_size() bytes (float32 partials of n_tok rows);
 * a page-table entry outside the pool is skipped and reported through the
 * workspace status word.  n_tok == 0 is a no-op.  No counterpart in the pages
 * beyond the step itself: the interface is this library's. */
LS_API ls_status ls_prompt_prefill(const ls_attn_desc* desc, const void* q, const void* k,
                                   const void* v, int32_t n_tok, void* o, float* lse,
                                   void* k_pool, void* v_pool, int64_t pool_pages,
                                   const int32_t* page_table, int64_t num_pages, void* ws,
                                   size_t ws_bytes, void* stream);

/* Workspace bytes ls_prompt_prefill needs for n_tok tokens.  Host-only. */
LS_API ls_status ls_prompt_prefill_workspace_size(const ls_attn_desc* desc, int32_t n_tok,
                                                  size_t* bytes);

/* Replay forward (same arguments and results as ls_replay_fwd) for callers
 * that cannot allocate device memory: no workspace argument; the library's
 * own fixed 64 MiB device scratch (held by every GPU that loads the library
 * until exit) takes the workspace's place.  The pages have no counterpart to
 * this call; it exists for embedders that own every allocation.
 * The first call on each device looks up the scratch's device address with
 * that device current; make it before any stream capture.  All calls share
 * the one scratch, so calls that overlap on the GPU race.  A call that would
 * need more scratch than 64 MiB returns LS_ERR_WORKSPACE_TOO_SMALL.  Device
 * status bits set by this call are not reported (the status word lives in
 * the scratch). */
LS_API ls_status ls_replay_fwd_noalloc(const ls_attn_desc* desc, const ls_prompt_kv* prompt,
                                       const void* q, const void* k_resp, const void* v_resp,
                                       int32_t resp_len, void* o, float* lse, void* stream);

/* Bytes of the fixed scratch ls_replay_fwd_noalloc uses (64 MiB). */
LS_API size_t ls_replay_fwd_noalloc_scratch_bytes(void);

/* Synchronises the stream, then reports the device status word of ws
 * (LS_OK, LS_ERR_DEVICE_BOUNDS or LS_ERR_DEVICE_TIMEOUT) and clears it. */
LS_API ls_status ls_read_device_status(void* ws, size_t ws_bytes, void* stream);

/* Zeroes the workspace status word (asynchronous on the stream). */
LS_API ls_status ls_clear_device_status(void* ws, size_t ws_bytes, void* stream);

LS_API const char* ls_status_string(ls_status status);
/* One-line reason for the last non-OK status returned on this thread. */
LS_API const char* ls_last_error(void);

/* Tracing.  When enabled, every kernel launch is bracketed by CUDA events on
 * its own stream and accumulated per kernel id; ls_trace_read synchronises
 * those events and reports launches and total milliseconds since the last
 * reset.  ls_launch_count counts every kernel this library launched in this
 * process (traced or not). */
LS_API ls_status ls_trace_enable(int32_t on);
LS_API ls_status ls_trace_reset(void);
LS_API ls_status ls_trace_read(int32_t kernel_id, int64_t* launches, double* total_ms);
LS_API int32_t ls_num_kernel_ids(void);
LS_API const char* ls_kernel_name(int32_t kernel_id);
LS_API int64_t ls_launch_count(void);

/* Which prompt-attention implementation the current device and desc select:
 * 1 = tcgen05/TMEM tensor-core kernels, 0 = CUDA-core kernels. */
LS_API int32_t ls_uses_tensor_cores(const ls_attn_desc* desc);

#ifdef __cplusplus
}
#endif

#endif /* LS_H_ */
