// Internal declarations shared by the libls translation units (not installed).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ls.h"

namespace ls {

// Bits of the device status word (first 4 bytes of the workspace).  The
// next word records the first bounded wait that gave up: kernel id << 16 | line.
enum : uint32_t {
  kStatusBadPage = 1u,   // a page-table entry pointed outside the pool
  kStatusTimeout = 2u,   // a bounded device wait gave up
};

// Bytes at the head of the workspace reserved for the status word.
constexpr size_t kWsHeader = 256;

// Runs every host-side check ls_replay_fwd makes (descriptor, prompt,
// pointers, alignment) without launching anything, and gives the workspace
// bytes the call needs on the current device.
ls_status replay_fwd_validate(const ls_attn_desc* desc, const ls_prompt_kv* prompt, const void* q,
                              const void* k_resp, const void* v_resp, int32_t resp_len,
                              const void* o, const float* lse, size_t* ws_need);

// Kernel ids used by tracing (ls_trace_read / ls_kernel_name).
enum KernelId : int32_t {
  kKPageWrite = 0,
  kKSimtFwd,
  kKTcFwd,
  kKLseMerge,
  kKBwdPre,
  kKSimtBwdDq,
  kKTcBwdDq,
  kKSimtDkDv,
  kKTcDkDv,
  kKDqReduce,
  kKGdnFwd,
  kKGdnBwd,
  kKStagePages,
  kNumKernelIds
};

// Launch bookkeeping (ls_api.cu): count every launch, optionally bracket it
// with events on its stream.
struct LaunchScope {
  LaunchScope(int32_t kid, cudaStream_t s);
  ~LaunchScope();
  // A scope counts as one kernel launch; a launcher that runs n kernels
  // under one scope (one trace entry) adds the other n - 1 here.
  void more_kernels(int n);
  int32_t kid;
  cudaStream_t stream;
  void* ev0;
  void* ev1;
};

// Rows of one KV group are numbered t = hh * R + r (hh = head within group).
// Output row index is n = r * Hq + h with h = g * Gq + hh.

// Common geometry of the attention kernels.
struct AttnGeom {
  int32_t hq, hkv, gq, d, page_size;
  int32_t R;             // response length
  int64_t P;             // prompt length
  int64_t pool_pages;
  float scale;           // softmax scale
  float scale_log2;      // scale * log2(e)
  int32_t ns;            // prompt splits (part ns is the response part)
  int64_t split_span;    // prompt keys per split (a multiple of every key tile)
  bool resp_part;        // compute part ns; false on a context-parallel rank
                         // that does not hold the response (parts 0..ns-1 only)
};

// Parts a forward/backward launch covers: the ns prompt splits plus the
// causal response part when it is wanted.
inline int launch_parts(const AttnGeom& g) { return g.ns + (g.resp_part ? 1 : 0); }

struct FwdParams {
  AttnGeom g;
  const void* q;
  const void* k_pool;
  const void* v_pool;
  const int32_t* page_table;
  const void* k_resp;
  const void* v_resp;
  float* o_parts;    // [n_parts][R*Hq][d]
  float* lse_parts;  // [n_parts][R*Hq]
  uint32_t* status;
};

struct BwdParams {
  AttnGeom g;
  const void* q;
  const void* d_o;
  const float* lse;    // [R][Hq]
  const float* delta;  // [R][Hq]
  const void* k_pool;
  const void* v_pool;
  const int32_t* page_table;
  const void* k_resp;
  const void* v_resp;
  float* dq_parts;     // [n_parts][R*Hq][d], unscaled
  void* dk;            // [R][Hkv][d] element dtype
  void* dv;
  uint32_t* status;
};

// CUDA-core kernels (ls_simt.cu)
cudaError_t launch_page_write(int dtype, int hkv, int d, int page_size, void* k_pool,
                              void* v_pool, int64_t pool_pages, const int32_t* pt,
                              int64_t start_pos, int64_t n_tok, const void* k,
                              const void* v, uint32_t* status, cudaStream_t s);
cudaError_t launch_simt_fwd(int dtype, const FwdParams& p, cudaStream_t s);
cudaError_t launch_simt_fwd_resp(int dtype, const FwdParams& p, cudaStream_t s);
// Whole pages of a device-readable source pool into a staging pool (ls_stage_pages).
cudaError_t launch_stage_pages(int64_t page_bytes, const void* k_src, const void* v_src,
                               int64_t src_pages, const int32_t* pt, int64_t first, int n_pages,
                               void* k_dst, void* v_dst, uint32_t* status, cudaStream_t s);
cudaError_t launch_lse_merge(int n_parts, int64_t n_rows, int d, const float* o_parts,
                             const float* lse_parts, int out_dtype, void* o, float* lse,
                             cudaStream_t s);
cudaError_t launch_bwd_preprocess(int dtype, int64_t n_rows, int d, const void* o,
                                  const void* d_o, float* delta, cudaStream_t s);
cudaError_t launch_simt_bwd_dq(int dtype, const BwdParams& p, cudaStream_t s);
cudaError_t launch_simt_bwd_dq_resp(int dtype, const BwdParams& p, cudaStream_t s);
cudaError_t launch_simt_dkdv(int dtype, const BwdParams& p, cudaStream_t s);
cudaError_t launch_dq_reduce(int n_parts, int64_t n_rows, int d, float scale,
                             const float* parts, int out_dtype, void* dq, cudaStream_t s);

// Tensor-core kernels (ls_tc_fwd.cu, ls_tc_bwd.cu): bf16, d = 256,
// page_size % 128 == 0, sm_100-family device.  Query tiles are 128 rows;
// split spans are multiples of kTcSpanQuantum keys.
constexpr int kTcRows = 128;
constexpr int kTcSpanQuantum = 128;
cudaError_t launch_tc_fwd(const FwdParams& p, cudaStream_t s);
cudaError_t launch_tc_bwd_dq(const BwdParams& p, cudaStream_t s);

// 2-D TMA map over a bf16 matrix [rows][256] with [box_rows x 64] boxes and
// the 128-byte swizzle (ls_api.cu; cuTensorMapEncodeTiled resolved once
// through the runtime, no -lcuda).
// Sets the message ls_last_error() returns on this thread.
void set_last_error(const char* msg);

bool encode_pool_map(CUtensorMap* m, const void* base, int64_t rows, int box_rows);
// 3-D TMA map over a bf16 tensor [rows][heads][256] with [box_rows x 1 x 64]
// boxes and the 128-byte swizzle (response K/V, Q, dO); rows past the end
// read as zeros.
bool encode_rows_map(CUtensorMap* m, const void* base, int heads, int64_t rows, int box_rows);
// One-instruction [box_rows x 64*box_blocks] tiles landing as box_blocks
// swizzled [box_rows x 64] column boxes (pool rows; token-major rows).
bool encode_pool_tile_map(CUtensorMap* m, const void* base, int64_t rows, int box_rows,
                          int box_blocks = 4);
bool encode_rows_tile_map(CUtensorMap* m, const void* base, int heads, int64_t rows, int box_rows,
                          int box_blocks = 4);
cudaError_t launch_tc_dkdv(const BwdParams& p, cudaStream_t s);
// Gated-DeltaNet replay (ls_gdn.cu): dk = dv = 128, one CTA per (head, member).
bool gdn_supported(int dk, int dv);
size_t gdn_workspace_bytes(int B, int H, int R);
cudaError_t launch_gdn_fwd(int B, int H, int R, const float* s0, const float* q, const float* k,
                           const float* v, const float* g, const float* beta, float* o,
                           float* s_final, cudaStream_t st);
// Chunk-parallel tensor-core forward and backward (ls_gdn_cp.cu), precision
// LS_GDN_TENSOR_CORE; both use gdn_cp_workspace_bytes of scratch.
size_t gdn_cp_workspace_bytes(int B, int H, int R);
// status: the workspace status word a wait that gives up sets.
cudaError_t launch_gdn_cp_fwd(int B, int H, int R, const float* s0, const float* q, const float* k,
                              const float* v, const float* g, const float* beta, float* o,
                              float* s_final, float* ws, uint32_t* status, cudaStream_t st);
// reuse_forward: ws holds the scratch of launch_gdn_cp_fwd on the same inputs.
cudaError_t launch_gdn_cp_bwd(int B, int H, int R, const float* s0, const float* q, const float* k,
                              const float* v, const float* g, const float* beta, const float* d_o,
                              float* dq, float* dk, float* dv, float* dg, float* dbeta, float* ws,
                              bool reuse_forward, uint32_t* status, cudaStream_t st);
cudaError_t launch_gdn_bwd(int B, int H, int R, const float* s0, const float* q, const float* k,
                           const float* v, const float* g, const float* beta, const float* d_o,
                           float* dq, float* dk, float* dv, float* dg, float* dbeta, float* ws,
                           cudaStream_t st);

}  // namespace ls
