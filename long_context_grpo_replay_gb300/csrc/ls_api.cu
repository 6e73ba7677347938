// Host side of libls: argument validation, split planning, workspace layout,
// kernel dispatch, launch tracing and the device status word.  Every entry
// point of include/ls.h is defined here.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdarg>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "ls_internal.h"

namespace ls {
namespace {

thread_local char g_err[512] = "";

ls_status fail(ls_status st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
ls_status fail(ls_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return st;
}

ls_status cuda_fail(cudaError_t e, const char* what) {
  return fail(LS_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ------------------------------------------------------------------ tracing
struct Pending {
  int32_t kid;
  cudaEvent_t e0, e1;
};
std::mutex g_trace_mu;
bool g_trace_on = false;
std::vector<Pending> g_pending;
std::vector<cudaEvent_t> g_event_pool;
double g_total_ms[kNumKernelIds];
int64_t g_launches[kNumKernelIds];
std::atomic<int64_t> g_launch_count{0};

cudaEvent_t take_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

const char* kKernelNames[kNumKernelIds] = {
    "page_write",  "simt_fwd",   "tc_fwd",     "lse_merge", "bwd_preprocess",
    "simt_bwd_dq", "tc_bwd_dq",  "simt_dkdv",  "tc_dkdv",   "dq_reduce",
    "gdn_fwd",     "gdn_bwd",    "stage_pages"};

// ------------------------------------------------------------------ devices
int device_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return 152;
  return sms;
}

bool device_is_sm100_family() {
  int dev = 0, major = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
    return false;
  return major == 10;
}

bool force_simt() {
  static int v = [] {
    const char* e = getenv("LS_FORCE_SIMT");
    return e ? atoi(e) : 0;
  }();
  return v != 0;
}

bool tc_shape(const ls_attn_desc& d) {
  return d.dtype == LS_DTYPE_BF16 && d.head_dim == 256 && d.page_size % kTcSpanQuantum == 0;
}

// ------------------------------------------------------------------ planning
struct Plan {
  bool tc;
  int ns;            // prompt splits
  int64_t span;      // keys per split
  int n_parts;       // ns + 1 (the response part)
  size_t o_bytes;    // partial O / dQ region
  size_t lse_bytes;  // partial LSE region
  size_t ws_bytes;
};

Plan make_plan(const ls_attn_desc& d, int64_t P, int64_t R, int sms, bool tc) {
  Plan pl{};
  pl.tc = tc;
  if (P <= 0) {
    pl.ns = 0;
    pl.span = 0;
  } else if (tc) {
    // Balance whole waves of 1-CTA-per-SM units against per-unit set-up cost
    // (Q/dO tile load and epilogue, worth about 8 key tiles of 64).
    const int64_t n_mt = (d.hq / d.hkv * R + kTcRows - 1) / kTcRows;
    const int64_t units = (int64_t)d.hkv * n_mt;
    const int64_t quanta = (P + kTcSpanQuantum - 1) / kTcSpanQuantum;
    const int64_t max_ns = quanta < 64 ? quanta : 64;
    double best = 1e300;
    int best_ns = 1;
    for (int64_t ns = 1; ns <= max_ns; ++ns) {
      const int64_t span_q = (quanta + ns - 1) / ns;
      const int64_t real_ns = (quanta + span_q - 1) / span_q;
      const int64_t waves = (units * real_ns + sms - 1) / sms;
      const double cost = (double)waves * ((double)span_q * 2.0 + 8.0);
      if (cost < best * 0.999) {
        best = cost;
        best_ns = (int)real_ns;
      }
    }
    const int64_t span_q = (quanta + best_ns - 1) / best_ns;
    pl.span = span_q * kTcSpanQuantum;
    pl.ns = (int)((P + pl.span - 1) / pl.span);
  } else {
    const int64_t ctas = (int64_t)d.hkv * ((d.hq / d.hkv * R + 7) / 8);
    const int64_t target = (int64_t)sms * 16;
    const int64_t chunks = (P + 31) / 32;
    int64_t ns = (target + ctas - 1) / ctas;
    if (ns > 64) ns = 64;
    if (ns > chunks) ns = chunks;
    if (ns < 1) ns = 1;
    const int64_t span_c = (chunks + ns - 1) / ns;
    pl.span = span_c * 32;
    pl.ns = (int)((P + pl.span - 1) / pl.span);
  }
  pl.n_parts = pl.ns + 1;
  const size_t rows = (size_t)R * d.hq;
  pl.o_bytes = round_up((size_t)pl.n_parts * rows * d.head_dim * sizeof(float), 256);
  pl.lse_bytes = round_up((size_t)pl.n_parts * rows * sizeof(float), 256);
  pl.ws_bytes = kWsHeader + pl.o_bytes + pl.lse_bytes;
  return pl;
}

bool use_tc(const ls_attn_desc& d) {
  return !force_simt() && tc_shape(d) && device_is_sm100_family();
}

// ------------------------------------------------------------------ validation
ls_status check_desc(const ls_attn_desc* d) {
  if (!d) return fail(LS_ERR_INVALID_ARGUMENT, "desc is NULL");
  if (d->dtype != LS_DTYPE_F32 && d->dtype != LS_DTYPE_BF16)
    return fail(LS_ERR_INVALID_ARGUMENT, "dtype %d is not LS_DTYPE_F32 or LS_DTYPE_BF16", d->dtype);
  if (d->hq <= 0 || d->hkv <= 0 || d->hq % d->hkv != 0)
    return fail(LS_ERR_INVALID_ARGUMENT, "hq=%d hkv=%d: need hq, hkv > 0 and hq %% hkv == 0", d->hq,
                d->hkv);
  if (d->head_dim != 64 && d->head_dim != 128 && d->head_dim != 256)
    return fail(LS_ERR_UNSUPPORTED, "head_dim=%d: supported are 64, 128, 256", d->head_dim);
  if (d->page_size < 1) return fail(LS_ERR_INVALID_ARGUMENT, "page_size=%d < 1", d->page_size);
  if (!(d->softmax_scale > 0.f) || !std::isfinite(d->softmax_scale))
    return fail(LS_ERR_INVALID_ARGUMENT, "softmax_scale must be finite and > 0");
  return LS_OK;
}

ls_status check_prompt(const ls_attn_desc* d, const ls_prompt_kv* p) {
  if (!p) return fail(LS_ERR_INVALID_ARGUMENT, "prompt is NULL");
  if (p->prompt_len < 0) return fail(LS_ERR_INVALID_ARGUMENT, "prompt_len < 0");
  if (p->prompt_len == 0) return LS_OK;
  if (!p->k_pool || !p->v_pool || !p->page_table)
    return fail(LS_ERR_INVALID_ARGUMENT, "prompt pools and page table must be non-NULL");
  if (p->pool_pages < 1) return fail(LS_ERR_INVALID_ARGUMENT, "pool_pages < 1");
  if (p->num_pages < 1 || p->num_pages * (int64_t)d->page_size < p->prompt_len)
    return fail(LS_ERR_INVALID_ARGUMENT, "num_pages*page_size=%lld < prompt_len=%lld",
                (long long)(p->num_pages * (int64_t)d->page_size), (long long)p->prompt_len);
  if (!aligned(p->k_pool, 16) || !aligned(p->v_pool, 16) || !aligned(p->page_table, 4))
    return fail(LS_ERR_INVALID_ARGUMENT, "pools must be 16-byte aligned, page table 4-byte");
  const int64_t rows = p->pool_pages * d->hkv * (int64_t)d->page_size;
  if (rows >= (int64_t)INT32_MAX)
    return fail(LS_ERR_UNSUPPORTED, "pool of %lld rows exceeds 2^31-1", (long long)rows);
  return LS_OK;
}

ls_status check_ws(const void* ws, size_t ws_bytes, size_t need) {
  if (!ws) return fail(LS_ERR_INVALID_ARGUMENT, "workspace is NULL");
  if (!aligned(ws, 256)) return fail(LS_ERR_INVALID_ARGUMENT, "workspace must be 256-byte aligned");
  if (ws_bytes < need)
    return fail(LS_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes < %zu needed", ws_bytes, need);
  return LS_OK;
}

#define LS_CHECK(expr)               \
  do {                               \
    const ls_status _st = (expr);    \
    if (_st != LS_OK) return _st;    \
  } while (0)

#define LS_CUDA(expr, what)                          \
  do {                                               \
    const cudaError_t _e = (expr);                   \
    if (_e != cudaSuccess) return cuda_fail(_e, what); \
  } while (0)

AttnGeom make_geom(const ls_attn_desc& d, const ls_prompt_kv& p, int32_t R, const Plan& pl) {
  AttnGeom g{};
  g.hq = d.hq;
  g.hkv = d.hkv;
  g.gq = d.hq / d.hkv;
  g.d = d.head_dim;
  g.page_size = d.page_size;
  g.R = R;
  g.P = p.prompt_len;
  g.pool_pages = p.pool_pages;
  g.scale = d.softmax_scale;
  g.scale_log2 = d.softmax_scale * 1.4426950408889634f;
  g.ns = pl.ns;
  g.split_span = pl.span;
  g.resp_part = true;
  return g;
}

// with_resp == false leaves the response keys out: the causal part (the
// last of the ns+1) is neither computed nor merged; out_dtype is the dtype o
// is written in.
// The host-side checks of a replay forward (nothing is launched).
ls_status fwd_check(const ls_attn_desc* desc, const ls_prompt_kv* prompt, const void* q,
                    const void* k_resp, const void* v_resp, int32_t R, const void* o,
                    const float* lse) {
  LS_CHECK(check_desc(desc));
  LS_CHECK(check_prompt(desc, prompt));
  if (R < 0) return fail(LS_ERR_INVALID_ARGUMENT, "resp_len < 0");
  if (R == 0) return LS_OK;
  if (!q || !k_resp || !v_resp || !o || !lse)
    return fail(LS_ERR_INVALID_ARGUMENT, "q, k_resp, v_resp, o, lse must be non-NULL");
  if (!aligned(q, 16) || !aligned(k_resp, 16) || !aligned(v_resp, 16) || !aligned(o, 16) ||
      !aligned(lse, 4))
    return fail(LS_ERR_INVALID_ARGUMENT, "element buffers must be 16-byte aligned");
  return LS_OK;
}

ls_status fwd_impl(const ls_attn_desc* desc, const ls_prompt_kv* prompt, const void* q,
                   const void* k_resp, const void* v_resp, int32_t R, void* o, float* lse,
                   void* ws, size_t ws_bytes, cudaStream_t s, bool with_resp = true,
                   int out_dtype = -1) {
  LS_CHECK(fwd_check(desc, prompt, q, k_resp, v_resp, R, o, lse));
  if (R == 0) return LS_OK;
  const bool tc = use_tc(*desc);
  const Plan pl = make_plan(*desc, prompt->prompt_len, R, device_sms(), tc);
  LS_CHECK(check_ws(ws, ws_bytes, pl.ws_bytes));
  FwdParams fp{};
  fp.g = make_geom(*desc, *prompt, R, pl);
  fp.g.resp_part = with_resp;
  fp.q = q;
  fp.k_pool = prompt->k_pool;
  fp.v_pool = prompt->v_pool;
  fp.page_table = prompt->page_table;
  fp.k_resp = k_resp;
  fp.v_resp = v_resp;
  fp.status = reinterpret_cast<uint32_t*>(ws);
  fp.o_parts = reinterpret_cast<float*>(static_cast<char*>(ws) + kWsHeader);
  fp.lse_parts = reinterpret_cast<float*>(static_cast<char*>(ws) + kWsHeader + pl.o_bytes);
  if (tc) {
    LS_CUDA(launch_tc_fwd(fp, s), "tensor-core forward launch");
  } else {
    LS_CUDA(launch_simt_fwd(desc->dtype, fp, s), "forward launch");
  }
  LS_CUDA(launch_lse_merge(with_resp ? pl.n_parts : pl.n_parts - 1, (int64_t)R * desc->hq,
                           desc->head_dim, fp.o_parts, fp.lse_parts,
                           out_dtype < 0 ? desc->dtype : out_dtype, o, lse, s),
          "LSE merge launch");
  return LS_OK;
}

// with_resp == false computes and sums dQ over the prompt parts only and
// skips the response dK/dV (dk, dv may then be NULL); dq_dtype is the dtype
// dq is written in.
ls_status bwd_impl(const ls_attn_desc* desc, const ls_prompt_kv* prompt, const void* q,
                   const void* k_resp, const void* v_resp, const void* d_o, const float* lse,
                   const float* delta, int32_t R, void* dq, void* dk, void* dv, void* ws,
                   size_t ws_bytes, cudaStream_t s, bool with_resp = true, int dq_dtype = -1) {
  LS_CHECK(check_desc(desc));
  LS_CHECK(check_prompt(desc, prompt));
  if (R < 0) return fail(LS_ERR_INVALID_ARGUMENT, "resp_len < 0");
  if (R == 0) return LS_OK;
  if (!q || !k_resp || !v_resp || !d_o || !lse || !delta || !dq || (with_resp && (!dk || !dv)))
    return fail(LS_ERR_INVALID_ARGUMENT, "backward buffers must be non-NULL");
  if (!aligned(q, 16) || !aligned(k_resp, 16) || !aligned(v_resp, 16) || !aligned(d_o, 16) ||
      !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) || !aligned(lse, 4) ||
      !aligned(delta, 4))
    return fail(LS_ERR_INVALID_ARGUMENT, "element buffers must be 16-byte aligned");
  const bool tc = use_tc(*desc);
  const Plan pl = make_plan(*desc, prompt->prompt_len, R, device_sms(), tc);
  LS_CHECK(check_ws(ws, ws_bytes, pl.ws_bytes));
  BwdParams bp{};
  bp.g = make_geom(*desc, *prompt, R, pl);
  bp.g.resp_part = with_resp;
  bp.q = q;
  bp.d_o = d_o;
  bp.lse = lse;
  bp.delta = delta;
  bp.k_pool = prompt->k_pool;
  bp.v_pool = prompt->v_pool;
  bp.page_table = prompt->page_table;
  bp.k_resp = k_resp;
  bp.v_resp = v_resp;
  bp.dq_parts = reinterpret_cast<float*>(static_cast<char*>(ws) + kWsHeader);
  bp.dk = dk;
  bp.dv = dv;
  bp.status = reinterpret_cast<uint32_t*>(ws);
  if (tc) {
    LS_CUDA(launch_tc_bwd_dq(bp, s), "tensor-core backward launch");
  } else {
    LS_CUDA(launch_simt_bwd_dq(desc->dtype, bp, s), "backward launch");
  }
  LS_CUDA(launch_dq_reduce(with_resp ? pl.n_parts : pl.n_parts - 1, (int64_t)R * desc->hq,
                           desc->head_dim, desc->softmax_scale, bp.dq_parts,
                           dq_dtype < 0 ? desc->dtype : dq_dtype, dq, s),
          "dQ reduce launch");
  if (!with_resp) return LS_OK;
  if (tc) {
    LS_CUDA(launch_tc_dkdv(bp, s), "tensor-core response dK/dV launch");
  } else {
    LS_CUDA(launch_simt_dkdv(desc->dtype, bp, s), "response dK/dV launch");
  }
  return LS_OK;
}

}  // namespace

ls_status replay_fwd_validate(const ls_attn_desc* desc, const ls_prompt_kv* prompt, const void* q,
                              const void* k_resp, const void* v_resp, int32_t R, const void* o,
                              const float* lse, size_t* ws_need) {
  LS_CHECK(fwd_check(desc, prompt, q, k_resp, v_resp, R, o, lse));
  *ws_need = R == 0 ? 0
                    : make_plan(*desc, prompt->prompt_len, R, device_sms(), use_tc(*desc)).ws_bytes;
  return LS_OK;
}

// ------------------------------------------------------------------ LaunchScope
LaunchScope::LaunchScope(int32_t k, cudaStream_t s) : kid(k), stream(s), ev0(nullptr), ev1(nullptr) {
  g_launch_count.fetch_add(1, std::memory_order_relaxed);
  std::lock_guard<std::mutex> lk(g_trace_mu);
  if (!g_trace_on) return;
  cudaEvent_t e = take_event();
  if (e && cudaEventRecord(e, s) == cudaSuccess) ev0 = e;
}

void LaunchScope::more_kernels(int n) { g_launch_count.fetch_add(n, std::memory_order_relaxed); }

namespace {
// LS_DEBUG_SYNC=1: synchronise after every launch and log it to stderr, so
// that a stall or an error names its kernel.
bool debug_sync() {
  static int v = [] {
    const char* e = getenv("LS_DEBUG_SYNC");
    return e ? atoi(e) : 0;
  }();
  return v != 0;
}
}  // namespace

LaunchScope::~LaunchScope() {
  if (debug_sync()) {
    fprintf(stderr, "[libls] %s launched\n", kKernelNames[kid]);
    const cudaError_t e = cudaStreamSynchronize(stream);
    fprintf(stderr, "[libls] %s done: %s\n", kKernelNames[kid], cudaGetErrorString(e));
  }
  if (!ev0) return;
  std::lock_guard<std::mutex> lk(g_trace_mu);
  cudaEvent_t e = take_event();
  if (!e || cudaEventRecord(e, stream) != cudaSuccess) {
    g_event_pool.push_back(static_cast<cudaEvent_t>(ev0));
    if (e) g_event_pool.push_back(e);
    return;
  }
  g_pending.push_back({kid, static_cast<cudaEvent_t>(ev0), e});
}

void set_last_error(const char* msg) { snprintf(g_err, sizeof(g_err), "%s", msg); }

// ------------------------------------------------------------------ TMA maps
namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encoder() {
  static EncodeTiledFn enc = []() -> EncodeTiledFn {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(fn);
  }();
  return enc;
}
}  // namespace

bool encode_pool_map(CUtensorMap* m, const void* base, int64_t rows, int box_rows) {
  EncodeTiledFn enc = encoder();
  if (!enc) return false;
  cuuint64_t gdim[2] = {256u, (cuuint64_t)rows};
  cuuint64_t gstr[1] = {256u * 2u};
  cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1u, 1u};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim, gstr, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_rows_map(CUtensorMap* m, const void* base, int heads, int64_t rows, int box_rows) {
  EncodeTiledFn enc = encoder();
  if (!enc) return false;
  cuuint64_t gdim[3] = {256u, (cuuint64_t)heads, (cuuint64_t)rows};
  cuuint64_t gstr[2] = {256u * 2u, (cuuint64_t)heads * 256u * 2u};
  cuuint32_t box[3] = {64u, 1u, (cuuint32_t)box_rows};
  cuuint32_t es[3] = {1u, 1u, 1u};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), gdim, gstr, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Whole-tile maps: one TMA instruction moves a [box_rows x 64*box_blocks]
// bf16 tile and lands it as box_blocks 128B-swizzled [box_rows x 64] column
// boxes, one after the other (the layout the MMA descriptors address).  The 256 columns of a row
// are viewed as (64 columns) x (4 column blocks): dim 0 = column in block,
// dim 1 = row, dim 2 = column block (stride 128 bytes).
bool encode_pool_tile_map(CUtensorMap* m, const void* base, int64_t rows, int box_rows,
                          int box_blocks) {
  EncodeTiledFn enc = encoder();
  if (!enc) return false;
  cuuint64_t gdim[3] = {64u, (cuuint64_t)rows, 4u};
  cuuint64_t gstr[2] = {256u * 2u, 64u * 2u};
  cuuint32_t box[3] = {64u, (cuuint32_t)box_rows, (cuuint32_t)box_blocks};
  cuuint32_t es[3] = {1u, 1u, 1u};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), gdim, gstr, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The same over token-major [rows][heads][256] data: dim 1 = token (stride
// heads*512 bytes), dim 3 = head; rows past the end read as zero.
bool encode_rows_tile_map(CUtensorMap* m, const void* base, int heads, int64_t rows, int box_rows,
                          int box_blocks) {
  EncodeTiledFn enc = encoder();
  if (!enc) return false;
  cuuint64_t gdim[4] = {64u, (cuuint64_t)rows, 4u, (cuuint64_t)heads};
  cuuint64_t gstr[3] = {(cuuint64_t)heads * 256u * 2u, 64u * 2u, 256u * 2u};
  cuuint32_t box[4] = {64u, (cuuint32_t)box_rows, (cuuint32_t)box_blocks, 1u};
  cuuint32_t es[4] = {1u, 1u, 1u, 1u};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), gdim, gstr, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace ls

using namespace ls;

extern "C" {

ls_status ls_kv_page_write(const ls_attn_desc* desc, void* k_pool, void* v_pool,
                           int64_t pool_pages, const int32_t* page_table, int64_t num_pages,
                           int64_t start_pos, int64_t n_tok, const void* k, const void* v,
                           void* ws, size_t ws_bytes, void* stream) {
  LS_CHECK(check_desc(desc));
  if (n_tok < 0 || start_pos < 0) return fail(LS_ERR_INVALID_ARGUMENT, "n_tok/start_pos < 0");
  if (n_tok == 0) return LS_OK;
  if (!k_pool || !v_pool || !page_table || !k || !v)
    return fail(LS_ERR_INVALID_ARGUMENT, "pools, page table, k and v must be non-NULL");
  if (pool_pages < 1) return fail(LS_ERR_INVALID_ARGUMENT, "pool_pages < 1");
  if (start_pos + n_tok > num_pages * (int64_t)desc->page_size)
    return fail(LS_ERR_INVALID_ARGUMENT, "start_pos + n_tok exceeds num_pages * page_size");
  if (!aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(k, 16) || !aligned(v, 16) ||
      !aligned(page_table, 4))
    return fail(LS_ERR_INVALID_ARGUMENT, "buffers must be 16-byte aligned");
  uint32_t* status = nullptr;
  if (ws) {
    LS_CHECK(check_ws(ws, ws_bytes, kWsHeader));
    status = reinterpret_cast<uint32_t*>(ws);
  }
  LS_CUDA(launch_page_write(desc->dtype, desc->hkv, desc->head_dim, desc->page_size, k_pool,
                            v_pool, pool_pages, page_table, start_pos, n_tok, k, v, status,
                            static_cast<cudaStream_t>(stream)),
          "page write launch");
  return LS_OK;
}

ls_status ls_replay_workspace_size(const ls_attn_desc* desc, const ls_prompt_kv* prompt,
                                   int32_t max_resp_len, size_t* bytes) {
  LS_CHECK(check_desc(desc));
  LS_CHECK(check_prompt(desc, prompt));
  if (!bytes) return fail(LS_ERR_INVALID_ARGUMENT, "bytes is NULL");
  if (max_resp_len < 0) return fail(LS_ERR_INVALID_ARGUMENT, "max_resp_len < 0");
  const bool tc = tc_shape(*desc) && !force_simt();
  const int sms = device_sms();
  size_t need = kWsHeader;
  // The split count depends on R, so take the largest need over 1..max_resp_len.
  for (int32_t R = 1; R <= max_resp_len; ++R) {
    const Plan a = make_plan(*desc, prompt->prompt_len, R, sms, tc);
    const Plan b = make_plan(*desc, prompt->prompt_len, R, sms, false);
    if (a.ws_bytes > need) need = a.ws_bytes;
    if (b.ws_bytes > need) need = b.ws_bytes;
  }
  *bytes = need;
  return LS_OK;
}

ls_status ls_replay_fwd(const ls_attn_desc* desc, const ls_prompt_kv* prompt, const void* q,
                        const void* k_resp, const void* v_resp, int32_t resp_len, void* o,
                        float* lse, void* ws, size_t ws_bytes, void* stream) {
  return fwd_impl(desc, prompt, q, k_resp, v_resp, resp_len, o, lse, ws, ws_bytes,
                  static_cast<cudaStream_t>(stream));
}

ls_status ls_prompt_prefill_workspace_size(const ls_attn_desc* desc, int32_t n_tok, size_t* bytes) {
  LS_CHECK(check_desc(desc));
  if (!bytes) return fail(LS_ERR_INVALID_ARGUMENT, "bytes is NULL");
  if (n_tok < 0) return fail(LS_ERR_INVALID_ARGUMENT, "n_tok < 0");
  // an empty prompt: one part (the causal one) whatever the route
  *bytes = make_plan(*desc, 0, n_tok, device_sms(), false).ws_bytes;
  return LS_OK;
}

ls_status ls_prompt_prefill(const ls_attn_desc* desc, const void* q, const void* k, const void* v,
                            int32_t n_tok, void* o, float* lse, void* k_pool, void* v_pool,
                            int64_t pool_pages, const int32_t* page_table, int64_t num_pages,
                            void* ws, size_t ws_bytes, void* stream) {
  LS_CHECK(check_desc(desc));
  if (n_tok < 0) return fail(LS_ERR_INVALID_ARGUMENT, "n_tok < 0");
  if (n_tok == 0) return LS_OK;
  size_t need = 0;
  LS_CHECK(ls_prompt_prefill_workspace_size(desc, n_tok, &need));
  LS_CHECK(check_ws(ws, ws_bytes, need));
  LS_CHECK(ls_kv_page_write(desc, k_pool, v_pool, pool_pages, page_table, num_pages, 0, n_tok, k, v,
                            ws, ws_bytes, stream));
  ls_prompt_kv empty{};
  empty.prompt_len = 0;
  return fwd_impl(desc, &empty, q, k, v, n_tok, o, lse, ws, ws_bytes,
                  static_cast<cudaStream_t>(stream));
}

ls_status ls_replay_fwd_part(const ls_attn_desc* desc, const ls_prompt_kv* prompt, const void* q,
                             const void* k_resp, const void* v_resp, int32_t resp_len,
                             int32_t with_response, float* o_part, float* lse_part, void* ws,
                             size_t ws_bytes, void* stream) {
  return fwd_impl(desc, prompt, q, k_resp, v_resp, resp_len, o_part, lse_part, ws, ws_bytes,
                  static_cast<cudaStream_t>(stream), with_response != 0, LS_DTYPE_F32);
}

ls_status ls_replay_bwd_part(const ls_attn_desc* desc, const ls_prompt_kv* prompt, const void* q,
                             const void* k_resp, const void* v_resp, const void* d_o,
                             const float* lse, const float* delta, int32_t resp_len,
                             int32_t with_response, float* dq_part, void* dk_resp, void* dv_resp,
                             void* ws, size_t ws_bytes, void* stream) {
  return bwd_impl(desc, prompt, q, k_resp, v_resp, d_o, lse, delta, resp_len, dq_part, dk_resp,
                  dv_resp, ws, ws_bytes, static_cast<cudaStream_t>(stream), with_response != 0,
                  LS_DTYPE_F32);
}

ls_status ls_sum_parts(int32_t n_parts, int64_t n_elems, const float* parts, int32_t out_dtype,
                       void* out, void* stream) {
  if (n_parts < 0 || n_elems < 0 || n_elems % 4 != 0)
    return fail(LS_ERR_INVALID_ARGUMENT, "need n_parts >= 0 and n_elems a multiple of 4");
  if (out_dtype != LS_DTYPE_F32 && out_dtype != LS_DTYPE_BF16)
    return fail(LS_ERR_INVALID_ARGUMENT, "bad out_dtype");
  if (n_elems == 0) return LS_OK;
  if ((n_parts > 0 && !parts) || !out)
    return fail(LS_ERR_INVALID_ARGUMENT, "parts and out must be non-NULL");
  if (!aligned(parts, 16) || !aligned(out, out_dtype == LS_DTYPE_F32 ? 4 : 2))
    return fail(LS_ERR_INVALID_ARGUMENT, "parts must be 16-byte aligned");
  // the dQ partial-sum kernel over rows of 4 elements, scale 1
  LS_CUDA(launch_dq_reduce(n_parts, n_elems / 4, 4, 1.0f, parts, out_dtype, out,
                           static_cast<cudaStream_t>(stream)),
          "partial sum launch");
  return LS_OK;
}

namespace {
ls_status check_gdn(const ls_gdn_desc* d) {
  if (!d) return fail(LS_ERR_INVALID_ARGUMENT, "desc is NULL");
  if (d->heads < 0 || d->batch < 0) return fail(LS_ERR_INVALID_ARGUMENT, "heads or batch < 0");
  if (d->batch > 65535) return fail(LS_ERR_UNSUPPORTED, "batch %d > 65535", d->batch);
  if (d->precision != LS_GDN_EXACT && d->precision != LS_GDN_TENSOR_CORE)
    return fail(LS_ERR_INVALID_ARGUMENT, "precision %d is not LS_GDN_EXACT or LS_GDN_TENSOR_CORE",
                d->precision);
  if (d->flags & ~LS_GDN_BWD_REUSES_FORWARD)
    return fail(LS_ERR_INVALID_ARGUMENT, "unknown flags 0x%x", (unsigned)d->flags);
  if (!gdn_supported(d->dk, d->dv))
    return fail(LS_ERR_UNSUPPORTED, "dk=%d dv=%d: supported is dk = dv = 128", d->dk, d->dv);
  return LS_OK;
}

// Backward workspace: the status header, then the kernels' scratch.
size_t gdn_ws_need(const ls_gdn_desc& d, int32_t R) {
  return kWsHeader + (d.precision == LS_GDN_TENSOR_CORE ? gdn_cp_workspace_bytes(d.batch, d.heads, R)
                                                        : gdn_workspace_bytes(d.batch, d.heads, R));
}
}  // namespace

ls_status ls_gdn_workspace_size(const ls_gdn_desc* desc, int32_t resp_len, size_t* bytes) {
  LS_CHECK(check_gdn(desc));
  if (!bytes) return fail(LS_ERR_INVALID_ARGUMENT, "bytes is NULL");
  if (resp_len < 0) return fail(LS_ERR_INVALID_ARGUMENT, "resp_len < 0");
  *bytes = gdn_ws_need(*desc, resp_len);
  return LS_OK;
}

ls_status ls_gdn_replay_fwd(const ls_gdn_desc* desc, const float* s0, const float* q,
                            const float* k, const float* v, const float* g, const float* beta,
                            int32_t resp_len, float* o, float* s_final, void* ws, size_t ws_bytes,
                            void* stream) {
  LS_CHECK(check_gdn(desc));
  if (resp_len < 0) return fail(LS_ERR_INVALID_ARGUMENT, "resp_len < 0");
  if (desc->batch == 0 || desc->heads == 0 || (resp_len == 0 && !s_final)) return LS_OK;
  if (!s0 || (resp_len > 0 && (!q || !k || !v || !g || !beta || !o)))
    return fail(LS_ERR_INVALID_ARGUMENT, "state and token buffers must be non-NULL");
  const bool tc = desc->precision == LS_GDN_TENSOR_CORE && resp_len > 0;
  if (tc) LS_CHECK(check_ws(ws, ws_bytes, gdn_ws_need(*desc, resp_len)));
  if (tc)
    LS_CUDA(launch_gdn_cp_fwd(desc->batch, desc->heads, resp_len, s0, q, k, v, g, beta, o, s_final,
                              reinterpret_cast<float*>(static_cast<char*>(ws) + kWsHeader),
                              static_cast<uint32_t*>(ws), static_cast<cudaStream_t>(stream)),
            "GDN chunk-parallel forward launch");
  else
    LS_CUDA(launch_gdn_fwd(desc->batch, desc->heads, resp_len, s0, q, k, v, g, beta, o, s_final,
                           static_cast<cudaStream_t>(stream)),
            "GDN forward launch");
  return LS_OK;
}

ls_status ls_gdn_replay_bwd(const ls_gdn_desc* desc, const float* s0, const float* q,
                            const float* k, const float* v, const float* g, const float* beta,
                            const float* d_o, int32_t resp_len, float* dq, float* dk, float* dv,
                            float* dg, float* dbeta, void* ws, size_t ws_bytes, void* stream) {
  LS_CHECK(check_gdn(desc));
  if (resp_len < 0) return fail(LS_ERR_INVALID_ARGUMENT, "resp_len < 0");
  if (desc->batch == 0 || desc->heads == 0 || resp_len == 0) return LS_OK;
  if (!s0 || !q || !k || !v || !g || !beta || !d_o || !dq || !dk || !dv || !dg || !dbeta)
    return fail(LS_ERR_INVALID_ARGUMENT, "backward buffers must be non-NULL");
  LS_CHECK(check_ws(ws, ws_bytes, gdn_ws_need(*desc, resp_len)));
  uint32_t* status = static_cast<uint32_t*>(ws);
  float* scratch = reinterpret_cast<float*>(static_cast<char*>(ws) + kWsHeader);
  if (desc->precision == LS_GDN_TENSOR_CORE)
    LS_CUDA(launch_gdn_cp_bwd(desc->batch, desc->heads, resp_len, s0, q, k, v, g, beta, d_o, dq, dk,
                              dv, dg, dbeta, scratch, (desc->flags & LS_GDN_BWD_REUSES_FORWARD) != 0,
                              status, static_cast<cudaStream_t>(stream)),
            "GDN chunk-parallel backward launch");
  else
    LS_CUDA(launch_gdn_bwd(desc->batch, desc->heads, resp_len, s0, q, k, v, g, beta, d_o, dq, dk,
                           dv, dg, dbeta, scratch, static_cast<cudaStream_t>(stream)),
            "GDN backward launch");
  return LS_OK;
}

namespace {
// A device-readable address for p: device or managed memory as is, pinned
// host memory through its device mapping; NULL for memory the GPU cannot
// read (pageable host memory), which is refused before any launch.
const void* device_readable(const void* p) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();  // clear the sticky-free error of an unknown pointer
    return nullptr;
  }
  switch (a.type) {
    case cudaMemoryTypeDevice:
    case cudaMemoryTypeManaged: return p;
    case cudaMemoryTypeHost: return a.devicePointer;
    default: return nullptr;
  }
}
}  // namespace

ls_status ls_stage_pages(const ls_attn_desc* desc, const void* k_src, const void* v_src,
                         int64_t src_pages, const int32_t* page_table, int64_t first_page,
                         int32_t n_pages, void* k_dst, void* v_dst, void* ws, size_t ws_bytes,
                         void* stream) {
  LS_CHECK(check_desc(desc));
  if (n_pages < 0 || n_pages > 65535 || first_page < 0 || src_pages < 1)
    return fail(LS_ERR_INVALID_ARGUMENT,
                "need 0 <= n_pages <= 65535, first_page >= 0 and src_pages >= 1");
  if (n_pages == 0) return LS_OK;
  if (!k_src || !v_src || !page_table || !k_dst || !v_dst)
    return fail(LS_ERR_INVALID_ARGUMENT, "pools, page table and staging buffers must be non-NULL");
  if (!aligned(k_src, 16) || !aligned(v_src, 16) || !aligned(k_dst, 16) || !aligned(v_dst, 16) ||
      !aligned(page_table, 4))
    return fail(LS_ERR_INVALID_ARGUMENT, "pools and staging buffers must be 16-byte aligned");
  const void* ks = device_readable(k_src);
  const void* vs = device_readable(v_src);
  if (!ks || !vs)
    return fail(LS_ERR_INVALID_ARGUMENT,
                "source pools must be device memory or pinned host memory (the GPU cannot read "
                "pageable host memory)");
  uint32_t* status = nullptr;
  if (ws) {
    LS_CHECK(check_ws(ws, ws_bytes, kWsHeader));
    status = reinterpret_cast<uint32_t*>(ws);
  }
  const int64_t page_bytes = (int64_t)desc->hkv * desc->page_size * desc->head_dim *
                             (desc->dtype == LS_DTYPE_F32 ? 4 : 2);
  LS_CUDA(launch_stage_pages(page_bytes, ks, vs, src_pages, page_table, first_page, n_pages, k_dst,
                             v_dst, status, static_cast<cudaStream_t>(stream)),
          "page staging launch");
  return LS_OK;
}

ls_status ls_lse_merge(int32_t n_parts, int64_t n_rows, int32_t head_dim, const float* o_parts,
                       const float* lse_parts, int32_t out_dtype, void* o, float* lse,
                       void* stream) {
  if (n_parts < 1 || n_rows < 0) return fail(LS_ERR_INVALID_ARGUMENT, "n_parts < 1 or n_rows < 0");
  if (head_dim <= 0 || head_dim % 4 != 0)
    return fail(LS_ERR_INVALID_ARGUMENT, "head_dim must be a positive multiple of 4");
  if (out_dtype != LS_DTYPE_F32 && out_dtype != LS_DTYPE_BF16)
    return fail(LS_ERR_INVALID_ARGUMENT, "bad out_dtype");
  if (n_rows == 0) return LS_OK;
  if (!o_parts || !lse_parts || !o)
    return fail(LS_ERR_INVALID_ARGUMENT, "o_parts, lse_parts, o must be non-NULL");
  if (!aligned(o_parts, 16) || !aligned(o, out_dtype == LS_DTYPE_F32 ? 4 : 2))
    return fail(LS_ERR_INVALID_ARGUMENT, "o_parts must be 16-byte aligned");
  LS_CUDA(launch_lse_merge(n_parts, n_rows, head_dim, o_parts, lse_parts, out_dtype, o, lse,
                           static_cast<cudaStream_t>(stream)),
          "LSE merge launch");
  return LS_OK;
}

ls_status ls_replay_bwd_preprocess(const ls_attn_desc* desc, const void* o, const void* d_o,
                                   int32_t resp_len, float* delta, void* stream) {
  LS_CHECK(check_desc(desc));
  if (resp_len < 0) return fail(LS_ERR_INVALID_ARGUMENT, "resp_len < 0");
  if (resp_len == 0) return LS_OK;
  if (!o || !d_o || !delta) return fail(LS_ERR_INVALID_ARGUMENT, "o, d_o, delta must be non-NULL");
  LS_CUDA(launch_bwd_preprocess(desc->dtype, (int64_t)resp_len * desc->hq, desc->head_dim, o, d_o,
                                delta, static_cast<cudaStream_t>(stream)),
          "preprocess launch");
  return LS_OK;
}

ls_status ls_replay_bwd(const ls_attn_desc* desc, const ls_prompt_kv* prompt, const void* q,
                        const void* k_resp, const void* v_resp, const void* d_o,
                        const float* lse, const float* delta, int32_t resp_len, void* dq,
                        void* dk_resp, void* dv_resp, void* ws, size_t ws_bytes, void* stream) {
  return bwd_impl(desc, prompt, q, k_resp, v_resp, d_o, lse, delta, resp_len, dq, dk_resp,
                  dv_resp, ws, ws_bytes, static_cast<cudaStream_t>(stream));
}

ls_status ls_replay_group(const ls_attn_desc* desc, const ls_prompt_kv* prompt, int32_t n_members,
                          const ls_member* members, void* ws, size_t ws_bytes, void* stream) {
  LS_CHECK(check_desc(desc));
  LS_CHECK(check_prompt(desc, prompt));
  if (n_members < 0) return fail(LS_ERR_INVALID_ARGUMENT, "n_members < 0");
  if (n_members > 0 && !members) return fail(LS_ERR_INVALID_ARGUMENT, "members is NULL");
  for (int32_t g = 0; g < n_members; ++g) {
    const ls_member& m = members[g];
    if (m.resp_len > 0 && !m.delta)
      return fail(LS_ERR_INVALID_ARGUMENT, "member %d: delta is NULL", g);
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  for (int32_t g = 0; g < n_members; ++g) {
    const ls_member& m = members[g];
    LS_CHECK(fwd_impl(desc, prompt, m.q, m.k, m.v, m.resp_len, m.o, m.lse, ws, ws_bytes, s));
    LS_CHECK(ls_replay_bwd_preprocess(desc, m.o, m.d_o, m.resp_len, m.delta, stream));
    LS_CHECK(bwd_impl(desc, prompt, m.q, m.k, m.v, m.d_o, m.lse, m.delta, m.resp_len, m.dq, m.dk,
                      m.dv, ws, ws_bytes, s));
  }
  return LS_OK;
}

ls_status ls_read_device_status(void* ws, size_t ws_bytes, void* stream) {
  LS_CHECK(check_ws(ws, ws_bytes, kWsHeader));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t words[2] = {0u, 0u};
  LS_CUDA(cudaStreamSynchronize(s), "stream synchronize");
  LS_CUDA(cudaMemcpy(words, ws, sizeof(words), cudaMemcpyDeviceToHost), "status read");
  LS_CUDA(cudaMemset(ws, 0, sizeof(words)), "status clear");
  const uint32_t word = words[0];
  if (word & kStatusTimeout) {
    const int kid = (int)(words[1] >> 16);
    return fail(LS_ERR_DEVICE_TIMEOUT,
                "a device-side bounded wait ran out in %s at source line %u (status 0x%x)",
                (kid >= 0 && kid < kNumKernelIds) ? kKernelNames[kid] : "?", words[1] & 0xFFFFu,
                word);
  }
  if (word & kStatusBadPage)
    return fail(LS_ERR_DEVICE_BOUNDS, "a page-table entry was outside the pool (status 0x%x)",
                word);
  return LS_OK;
}

ls_status ls_clear_device_status(void* ws, size_t ws_bytes, void* stream) {
  LS_CHECK(check_ws(ws, ws_bytes, kWsHeader));
  LS_CUDA(cudaMemsetAsync(ws, 0, kWsHeader, static_cast<cudaStream_t>(stream)), "status clear");
  return LS_OK;
}

const char* ls_status_string(ls_status st) {
  switch (st) {
    case LS_OK: return "LS_OK";
    case LS_ERR_INVALID_ARGUMENT: return "LS_ERR_INVALID_ARGUMENT";
    case LS_ERR_UNSUPPORTED: return "LS_ERR_UNSUPPORTED";
    case LS_ERR_WORKSPACE_TOO_SMALL: return "LS_ERR_WORKSPACE_TOO_SMALL";
    case LS_ERR_CUDA: return "LS_ERR_CUDA";
    case LS_ERR_DEVICE_BOUNDS: return "LS_ERR_DEVICE_BOUNDS";
    case LS_ERR_DEVICE_TIMEOUT: return "LS_ERR_DEVICE_TIMEOUT";
  }
  return "LS_ERR_UNKNOWN";
}

const char* ls_last_error(void) { return g_err; }

ls_status ls_trace_enable(int32_t on) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  g_trace_on = on != 0;
  return LS_OK;
}

ls_status ls_trace_reset(void) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  for (auto& p : g_pending) {
    cudaEventSynchronize(p.e1);
    g_event_pool.push_back(p.e0);
    g_event_pool.push_back(p.e1);
  }
  g_pending.clear();
  for (int i = 0; i < kNumKernelIds; ++i) {
    g_total_ms[i] = 0.0;
    g_launches[i] = 0;
  }
  return LS_OK;
}

ls_status ls_trace_read(int32_t kernel_id, int64_t* launches, double* total_ms) {
  if (kernel_id < 0 || kernel_id >= kNumKernelIds)
    return fail(LS_ERR_INVALID_ARGUMENT, "kernel_id out of range");
  std::lock_guard<std::mutex> lk(g_trace_mu);
  for (auto& p : g_pending) {
    float ms = 0.f;
    if (cudaEventSynchronize(p.e1) == cudaSuccess &&
        cudaEventElapsedTime(&ms, p.e0, p.e1) == cudaSuccess) {
      g_total_ms[p.kid] += ms;
      g_launches[p.kid] += 1;
    }
    g_event_pool.push_back(p.e0);
    g_event_pool.push_back(p.e1);
  }
  g_pending.clear();
  if (launches) *launches = g_launches[kernel_id];
  if (total_ms) *total_ms = g_total_ms[kernel_id];
  return LS_OK;
}

int32_t ls_num_kernel_ids(void) { return kNumKernelIds; }

const char* ls_kernel_name(int32_t kernel_id) {
  if (kernel_id < 0 || kernel_id >= kNumKernelIds) return "";
  return kKernelNames[kernel_id];
}

int64_t ls_launch_count(void) { return g_launch_count.load(); }

int32_t ls_uses_tensor_cores(const ls_attn_desc* desc) {
  if (!desc || check_desc(desc) != LS_OK) return 0;
  return use_tc(*desc) ? 1 : 0;
}

}  // extern "C"
