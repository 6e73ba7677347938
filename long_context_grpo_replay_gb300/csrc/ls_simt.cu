// CUDA-core kernels of libls: page write, LSE merge, backward preprocess,
// dQ reduction, and the generic (any dtype / head dim / page size) attention
// kernels.  The tensor-core kernels for the bf16 d=256 shape live in
// ls_tc_fwd.cu and ls_tc_bwd.cu; these kernels also compute the response
// parts that those kernels leave out.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "ls_internal.h"

namespace ls {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float ldf(const float* p) { return *p; }
__device__ __forceinline__ float ldf(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void stf(float* p, float v) { *p = v; }
__device__ __forceinline__ void stf(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

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

// ---------------------------------------------------------------------------
// A1 page write: one warp copies one (token, kv head) row of d elements,
// 16 bytes per lane, from the token-major source to its pool slot.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) page_write_kernel(
    int row_bytes, int hkv, int page_size, char* __restrict__ k_pool,
    char* __restrict__ v_pool, int64_t pool_pages, const int32_t* __restrict__ pt,
    int64_t start_pos, int64_t n_tok, const char* __restrict__ k,
    const char* __restrict__ v, uint32_t* status) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int64_t rows = n_tok * hkv;
  const int chunks = row_bytes >> 4;
  for (int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < rows;
       row += nwarps) {
    const int64_t t = row / hkv;
    const int kv = (int)(row - t * hkv);
    const int64_t pos = start_pos + t;
    const int32_t slot = __ldg(pt + pos / page_size);
    if (slot < 0 || slot >= pool_pages) {
      if (lane == 0 && status) atomicOr(status, kStatusBadPage);
      continue;
    }
    const int64_t dst = (((int64_t)slot * hkv + kv) * page_size + pos % page_size) * row_bytes;
    const int64_t src = row * (int64_t)row_bytes;
    for (int c = lane; c < chunks; c += 32) {
      const uint4 kk = __ldcs(reinterpret_cast<const uint4*>(k + src) + c);
      const uint4 vv = __ldcs(reinterpret_cast<const uint4*>(v + src) + c);
      __stcs(reinterpret_cast<uint4*>(k_pool + dst) + c, kk);
      __stcs(reinterpret_cast<uint4*>(v_pool + dst) + c, vv);
    }
  }
}

// ---------------------------------------------------------------------------
// Staging of whole pages from a (host-resident, device-mapped) pool into a
// compact staging pool: dst page i <- src page page_table[first + i], K and
// V.  A small grid (kStageBlocks blocks) walks all 16-byte pieces of the
// chunk with a grid-stride loop, each thread keeping four loads in flight:
// about 0.6 MB in flight, enough for the microseconds of latency of the
// CPU-GPU link at the 40-70 GB/s it gives under load, while the replay
// kernels that run beside it on another stream keep the other SMs to
// themselves (measured at the 2M prefix: 38 blocks slow them by about 4 %,
// two blocks per SM by about 9 %).  A page id outside the source pool zeroes the destination
// page and sets the status word.
__global__ void __launch_bounds__(256) stage_pages_kernel(
    int64_t page_bytes, const char* __restrict__ k_src, const char* __restrict__ v_src,
    int64_t src_pages, const int32_t* __restrict__ pt, int64_t first, int n_pages,
    char* __restrict__ k_dst, char* __restrict__ v_dst, uint32_t* status) {
  const int64_t n16 = page_bytes >> 4;       // pieces per page
  const int64_t total = 2 * n_pages * n16;   // K pages, then V pages
  const int64_t step = (int64_t)gridDim.x * blockDim.x;
  for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < total; c += 4 * step) {
    uint4 v[4];
    int64_t dsti[4];
    char* dstb[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t g = c + u * step;
      dstb[u] = nullptr;
      v[u] = make_uint4(0u, 0u, 0u, 0u);
      if (g < total) {
        const bool isv = g >= n_pages * n16;
        const int64_t gg = isv ? g - n_pages * n16 : g;
        const int64_t i = gg / n16, piece = gg - i * n16;
        const int32_t slot = __ldg(pt + first + i);
        const bool ok = slot >= 0 && slot < src_pages;
        if (!ok && piece == 0 && !isv && status) atomicOr(status, kStatusBadPage);
        if (ok)
          v[u] = __ldcs(reinterpret_cast<const uint4*>((isv ? v_src : k_src) + (int64_t)slot * page_bytes) + piece);
        dstb[u] = isv ? v_dst : k_dst;
        dsti[u] = gg;
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (dstb[u]) __stcs(reinterpret_cast<uint4*>(dstb[u]) + dsti[u], v[u]);
  }
}

// ---------------------------------------------------------------------------
// A4 exact LSE merge: one thread per (row, 4 columns).
// ---------------------------------------------------------------------------
template <typename TO>
__global__ void __launch_bounds__(256) lse_merge_kernel(int n_parts, int64_t n_rows, int d,
                                                        const float* __restrict__ o_parts,
                                                        const float* __restrict__ lse_parts,
                                                        TO* __restrict__ o, float* lse) {
  const int q4 = d >> 2;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= n_rows * q4) return;
  const int64_t row = idx / q4;
  const int c = (int)(idx - row * q4) * 4;
  float m = -CUDART_INF_F;
  for (int s = 0; s < n_parts; ++s) m = fmaxf(m, __ldg(lse_parts + (int64_t)s * n_rows + row));
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  float L = -CUDART_INF_F;
  if (m != -CUDART_INF_F) {
    float tot = 0.f;
    for (int s = 0; s < n_parts; ++s) tot += expf(__ldg(lse_parts + (int64_t)s * n_rows + row) - m);
    L = m + logf(tot);
    for (int s = 0; s < n_parts; ++s) {
      const float ls = __ldg(lse_parts + (int64_t)s * n_rows + row);
      if (ls == -CUDART_INF_F) continue;
      const float w = expf(ls - L);
      const float4 v = __ldg(reinterpret_cast<const float4*>(o_parts + ((int64_t)s * n_rows + row) * d + c));
      acc[0] += w * v.x;
      acc[1] += w * v.y;
      acc[2] += w * v.z;
      acc[3] += w * v.w;
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) stf(o + row * d + c + i, acc[i]);
  if (c == 0 && lse) lse[row] = L;
}

// ---------------------------------------------------------------------------
// A5 preprocess: delta = rowsum(dO * O), one warp per row.
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(int64_t n_rows, int d,
                                                             const T* __restrict__ o,
                                                             const T* __restrict__ d_o,
                                                             float* __restrict__ delta) {
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= n_rows) return;
  float acc = 0.f;
  for (int c = lane; c < d; c += 32) acc += ldf(o + row * d + c) * ldf(d_o + row * d + c);
  acc = warp_sum(acc);
  if (lane == 0) delta[row] = acc;
}

// ---------------------------------------------------------------------------
// dQ = scale * sum of the per-part float32 accumulators, in the output dtype.
// ---------------------------------------------------------------------------
template <typename TO>
__global__ void __launch_bounds__(256) dq_reduce_kernel(int n_parts, int64_t n_elems, float scale,
                                                        const float* __restrict__ parts,
                                                        TO* __restrict__ dq) {
  const int64_t i4 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (i4 >= n_elems) return;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s = 0; s < n_parts; ++s) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(parts + (int64_t)s * n_elems + i4));
    acc.x += v.x;
    acc.y += v.y;
    acc.z += v.z;
    acc.w += v.w;
  }
  stf(dq + i4 + 0, scale * acc.x);
  stf(dq + i4 + 1, scale * acc.y);
  stf(dq + i4 + 2, scale * acc.z);
  stf(dq + i4 + 3, scale * acc.w);
}

// ---------------------------------------------------------------------------
// Generic attention kernels.  A CTA holds 8 query rows of one KV group (rows
// numbered t = hh*R + r within the group) and walks a key range in chunks of
// 32 keys staged in shared memory as float32; lane j of a warp scores key j,
// and each lane accumulates d/32 output columns.
// ---------------------------------------------------------------------------
constexpr int kNW = 8;   // warps (query rows) per CTA
constexpr int kKC = 32;  // keys per chunk

// Key range of part `part` for a CTA whose rows are t0..t1 (inclusive).
__device__ __forceinline__ void part_range(const AttnGeom& g, int part, int64_t t0, int64_t t1,
                                           bool* resp, int64_t* kb, int64_t* ke) {
  if (part < g.ns) {
    *resp = false;
    const int64_t span = g.split_span;
    *kb = (int64_t)part * span;
    *ke = min(g.P, *kb + span);
  } else {
    *resp = true;
    *kb = 0;
    const bool same_head = (t0 / g.R) == (t1 / g.R);
    *ke = same_head ? (t1 % g.R) + 1 : g.R;
  }
}

// Whether prompt key `key` (< prompt_len) lies on a page inside the pool; a
// key on a page outside it is no key at all (its page was skipped and the
// status word flagged).
__device__ __forceinline__ bool prompt_key_ok(const AttnGeom& g, const int32_t* pt, int64_t key) {
  const int32_t slot = __ldg(pt + key / g.page_size);
  return slot >= 0 && slot < g.pool_pages;
}

// Stage keys kb..kb+31 of the range into sK/sV ([kKC][D+1] float32).
template <typename T, int D>
__device__ __forceinline__ void stage_keys(const AttnGeom& g, bool resp, int kvh, int64_t kb,
                                           int64_t ke, const T* k_pool, const T* v_pool,
                                           const int32_t* pt, const T* k_resp, const T* v_resp,
                                           float* sK, float* sV, uint32_t* status) {
  constexpr int DP = D + 1;
  for (int idx = threadIdx.x; idx < kKC * D; idx += blockDim.x) {
    const int j = idx / D;
    const int x = idx - j * D;
    const int64_t key = kb + j;
    float kv = 0.f, vv = 0.f;
    if (key < ke) {
      if (!resp) {
        const int32_t slot = __ldg(pt + key / g.page_size);
        if (slot >= 0 && slot < g.pool_pages) {
          const int64_t off =
              (((int64_t)slot * g.hkv + kvh) * g.page_size + key % g.page_size) * D + x;
          kv = ldf(k_pool + off);
          vv = ldf(v_pool + off);
        } else if (x == 0) {
          atomicOr(status, kStatusBadPage);
        }
      } else {
        const int64_t off = (key * g.hkv + kvh) * D + x;
        kv = ldf(k_resp + off);
        vv = ldf(v_resp + off);
      }
    }
    sK[j * DP + x] = kv;
    sV[j * DP + x] = vv;
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(kNW * 32) simt_fwd_kernel(FwdParams p, int part0) {
  constexpr int DP = D + 1, VPL = D / 32;
  extern __shared__ float smem[];
  float* sK = smem;
  float* sV = sK + kKC * DP;
  float* sQ = sV + kKC * DP;
  const AttnGeom& g = p.g;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kvh = blockIdx.y;
  const int part = part0 + blockIdx.z;
  const int64_t rows_g = (int64_t)g.gq * g.R;
  const int64_t t0 = (int64_t)blockIdx.x * kNW;
  const int64_t t1 = min(rows_g, t0 + kNW) - 1;
  const int64_t t = t0 + warp;
  const bool active = t < rows_g;
  const int hh = active ? (int)(t / g.R) : 0;
  const int r = active ? (int)(t % g.R) : 0;
  const int h = kvh * g.gq + hh;
  const T* qrow = reinterpret_cast<const T*>(p.q) + ((int64_t)r * g.hq + h) * D;
  for (int x = lane; x < D; x += 32) sQ[warp * D + x] = active ? ldf(qrow + x) : 0.f;
  bool resp;
  int64_t kb0, ke;
  part_range(g, part, t0, t1, &resp, &kb0, &ke);
  float m = -CUDART_INF_F, l = 0.f, o[VPL];
#pragma unroll
  for (int c = 0; c < VPL; ++c) o[c] = 0.f;
  for (int64_t kb = kb0; kb < ke; kb += kKC) {
    __syncthreads();
    stage_keys<T, D>(g, resp, kvh, kb, ke, reinterpret_cast<const T*>(p.k_pool),
                     reinterpret_cast<const T*>(p.v_pool), p.page_table,
                     reinterpret_cast<const T*>(p.k_resp), reinterpret_cast<const T*>(p.v_resp),
                     sK, sV, p.status);
    __syncthreads();
    if (!active) continue;
    float s = 0.f;
#pragma unroll 8
    for (int x = 0; x < D; ++x) s = fmaf(sQ[warp * D + x], sK[lane * DP + x], s);
    const int64_t key = kb + lane;
    const bool valid = key < ke && (resp ? key <= r : prompt_key_ok(g, p.page_table, key));
    const float s2 = valid ? s * g.scale_log2 : -CUDART_INF_F;
    const float m_new = fmaxf(m, warp_max(s2));
    if (m_new == -CUDART_INF_F) continue;
    const float alpha = exp2f(m - m_new);
    const float pj = valid ? exp2f(s2 - m_new) : 0.f;
    l = l * alpha + warp_sum(pj);
#pragma unroll
    for (int c = 0; c < VPL; ++c) o[c] *= alpha;
    for (int j = 0; j < kKC; ++j) {
      const float pjj = __shfl_sync(0xffffffffu, pj, j);
#pragma unroll
      for (int c = 0; c < VPL; ++c) o[c] = fmaf(pjj, sV[j * DP + lane + 32 * c], o[c]);
    }
    m = m_new;
  }
  if (!active) return;
  const int64_t n = (int64_t)r * g.hq + h;
  const int64_t nrows = (int64_t)g.R * g.hq;
  float* orow = p.o_parts + ((int64_t)part * nrows + n) * D;
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int c = 0; c < VPL; ++c) orow[lane + 32 * c] = o[c] * inv;
  if (lane == 0) p.lse_parts[(int64_t)part * nrows + n] = l > 0.f ? (m + log2f(l)) * kLn2 : -CUDART_INF_F;
}

template <typename T, int D>
__global__ void __launch_bounds__(kNW * 32) simt_bwd_dq_kernel(BwdParams p, int part0) {
  constexpr int DP = D + 1, VPL = D / 32;
  extern __shared__ float smem[];
  float* sK = smem;
  float* sV = sK + kKC * DP;
  float* sQ = sV + kKC * DP;
  float* sO = sQ + kNW * D;  // dO rows
  const AttnGeom& g = p.g;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kvh = blockIdx.y;
  const int part = part0 + blockIdx.z;
  const int64_t rows_g = (int64_t)g.gq * g.R;
  const int64_t t0 = (int64_t)blockIdx.x * kNW;
  const int64_t t1 = min(rows_g, t0 + kNW) - 1;
  const int64_t t = t0 + warp;
  const bool active = t < rows_g;
  const int hh = active ? (int)(t / g.R) : 0;
  const int r = active ? (int)(t % g.R) : 0;
  const int h = kvh * g.gq + hh;
  const int64_t n = (int64_t)r * g.hq + h;
  const T* qrow = reinterpret_cast<const T*>(p.q) + n * D;
  const T* dorow = reinterpret_cast<const T*>(p.d_o) + n * D;
  for (int x = lane; x < D; x += 32) {
    sQ[warp * D + x] = active ? ldf(qrow + x) : 0.f;
    sO[warp * D + x] = active ? ldf(dorow + x) : 0.f;
  }
  const float lse2 = active ? p.lse[n] * kLog2e : 0.f;
  const float dl = active ? p.delta[n] : 0.f;
  bool resp;
  int64_t kb0, ke;
  part_range(g, part, t0, t1, &resp, &kb0, &ke);
  float dq[VPL];
#pragma unroll
  for (int c = 0; c < VPL; ++c) dq[c] = 0.f;
  for (int64_t kb = kb0; kb < ke; kb += kKC) {
    __syncthreads();
    stage_keys<T, D>(g, resp, kvh, kb, ke, reinterpret_cast<const T*>(p.k_pool),
                     reinterpret_cast<const T*>(p.v_pool), p.page_table,
                     reinterpret_cast<const T*>(p.k_resp), reinterpret_cast<const T*>(p.v_resp),
                     sK, sV, p.status);
    __syncthreads();
    if (!active) continue;
    float s = 0.f, dp = 0.f;
#pragma unroll 8
    for (int x = 0; x < D; ++x) {
      s = fmaf(sQ[warp * D + x], sK[lane * DP + x], s);
      dp = fmaf(sO[warp * D + x], sV[lane * DP + x], dp);
    }
    const int64_t key = kb + lane;
    const bool valid = key < ke && (resp ? key <= r : prompt_key_ok(g, p.page_table, key));
    const float pj = valid ? exp2f(s * g.scale_log2 - lse2) : 0.f;
    const float ds = pj * (dp - dl);
    for (int j = 0; j < kKC; ++j) {
      const float dsj = __shfl_sync(0xffffffffu, ds, j);
#pragma unroll
      for (int c = 0; c < VPL; ++c) dq[c] = fmaf(dsj, sK[j * DP + lane + 32 * c], dq[c]);
    }
  }
  if (!active) return;
  const int64_t nrows = (int64_t)g.R * g.hq;
  float* out = p.dq_parts + ((int64_t)part * nrows + n) * D;
#pragma unroll
  for (int c = 0; c < VPL; ++c) out[lane + 32 * c] = dq[c];
}

// dK/dV of the response keys: one warp per key row j of one KV head; the CTA
// walks the query rows i >= j of every head of the group in chunks of 32.
template <typename T, int D>
__global__ void __launch_bounds__(kNW * 32) simt_dkdv_kernel(BwdParams p) {
  constexpr int DP = D + 1, VPL = D / 32, QC = 32;
  extern __shared__ float smem[];
  float* sQ = smem;              // [QC][DP]
  float* sO = sQ + QC * DP;      // [QC][DP] dO
  float* sKj = sO + QC * DP;     // [kNW][D]
  float* sVj = sKj + kNW * D;    // [kNW][D]
  float* sL = sVj + kNW * D;     // [QC] lse * log2e
  float* sDl = sL + QC;          // [QC] delta
  const AttnGeom& g = p.g;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kvh = blockIdx.y;
  const int j0 = blockIdx.x * kNW;
  const int j = j0 + warp;
  const bool active = j < g.R;
  const T* krow = reinterpret_cast<const T*>(p.k_resp) + ((int64_t)j * g.hkv + kvh) * D;
  const T* vrow = reinterpret_cast<const T*>(p.v_resp) + ((int64_t)j * g.hkv + kvh) * D;
  for (int x = lane; x < D; x += 32) {
    sKj[warp * D + x] = active ? ldf(krow + x) : 0.f;
    sVj[warp * D + x] = active ? ldf(vrow + x) : 0.f;
  }
  float dk[VPL], dv[VPL];
#pragma unroll
  for (int c = 0; c < VPL; ++c) dk[c] = dv[c] = 0.f;
  for (int hh = 0; hh < g.gq; ++hh) {
    const int h = kvh * g.gq + hh;
    for (int r0 = j0; r0 < g.R; r0 += QC) {
      __syncthreads();
      for (int idx = threadIdx.x; idx < QC * D; idx += blockDim.x) {
        const int i = idx / D, x = idx - (idx / D) * D;
        const int ri = r0 + i;
        float qv = 0.f, ov = 0.f;
        if (ri < g.R) {
          const int64_t off = ((int64_t)ri * g.hq + h) * D + x;
          qv = ldf(reinterpret_cast<const T*>(p.q) + off);
          ov = ldf(reinterpret_cast<const T*>(p.d_o) + off);
        }
        sQ[i * DP + x] = qv;
        sO[i * DP + x] = ov;
      }
      if (threadIdx.x < QC) {
        const int ri = r0 + threadIdx.x;
        sL[threadIdx.x] = ri < g.R ? p.lse[(int64_t)ri * g.hq + h] * kLog2e : 0.f;
        sDl[threadIdx.x] = ri < g.R ? p.delta[(int64_t)ri * g.hq + h] : 0.f;
      }
      __syncthreads();
      if (!active) continue;
      const int ri = r0 + lane;
      float s = 0.f, dp = 0.f;
#pragma unroll 8
      for (int x = 0; x < D; ++x) {
        s = fmaf(sQ[lane * DP + x], sKj[warp * D + x], s);
        dp = fmaf(sO[lane * DP + x], sVj[warp * D + x], dp);
      }
      const bool valid = ri < g.R && ri >= j;
      const float pi = valid ? exp2f(s * g.scale_log2 - sL[lane]) : 0.f;
      const float dsi = pi * (dp - sDl[lane]);
      for (int i = 0; i < QC; ++i) {
        const float pp = __shfl_sync(0xffffffffu, pi, i);
        const float dd = __shfl_sync(0xffffffffu, dsi, i);
#pragma unroll
        for (int c = 0; c < VPL; ++c) {
          dv[c] = fmaf(pp, sO[i * DP + lane + 32 * c], dv[c]);
          dk[c] = fmaf(dd, sQ[i * DP + lane + 32 * c], dk[c]);
        }
      }
    }
  }
  if (!active) return;
  T* dko = reinterpret_cast<T*>(p.dk) + ((int64_t)j * g.hkv + kvh) * D;
  T* dvo = reinterpret_cast<T*>(p.dv) + ((int64_t)j * g.hkv + kvh) * D;
#pragma unroll
  for (int c = 0; c < VPL; ++c) {
    stf(dko + lane + 32 * c, g.scale * dk[c]);
    stf(dvo + lane + 32 * c, dv[c]);
  }
}

template <typename T, int D>
size_t fwd_smem() { return sizeof(float) * (2 * kKC * (D + 1) + kNW * D); }
template <typename T, int D>
size_t bwd_smem() { return sizeof(float) * (2 * kKC * (D + 1) + 2 * kNW * D); }
template <typename T, int D>
size_t dkdv_smem() { return sizeof(float) * (2 * 32 * (D + 1) + 2 * kNW * D + 64); }

template <typename T, int D>
cudaError_t fwd_impl(const FwdParams& p, int part0, int nparts, cudaStream_t s) {
  if (nparts <= 0) return cudaSuccess;
  const size_t sm = fwd_smem<T, D>();
  cudaError_t e = cudaFuncSetAttribute(simt_fwd_kernel<T, D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  const int64_t rows_g = (int64_t)p.g.gq * p.g.R;
  dim3 grid((unsigned)((rows_g + kNW - 1) / kNW), p.g.hkv, nparts);
  LaunchScope ls(kKSimtFwd, s);
  simt_fwd_kernel<T, D><<<grid, kNW * 32, sm, s>>>(p, part0);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t bwd_impl(const BwdParams& p, int part0, int nparts, cudaStream_t s) {
  if (nparts <= 0) return cudaSuccess;
  const size_t sm = bwd_smem<T, D>();
  cudaError_t e = cudaFuncSetAttribute(simt_bwd_dq_kernel<T, D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  const int64_t rows_g = (int64_t)p.g.gq * p.g.R;
  dim3 grid((unsigned)((rows_g + kNW - 1) / kNW), p.g.hkv, nparts);
  LaunchScope ls(kKSimtBwdDq, s);
  simt_bwd_dq_kernel<T, D><<<grid, kNW * 32, sm, s>>>(p, part0);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t dkdv_impl(const BwdParams& p, cudaStream_t s) {
  const size_t sm = dkdv_smem<T, D>();
  cudaError_t e = cudaFuncSetAttribute(simt_dkdv_kernel<T, D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((p.g.R + kNW - 1) / kNW), p.g.hkv, 1);
  LaunchScope ls(kKSimtDkDv, s);
  simt_dkdv_kernel<T, D><<<grid, kNW * 32, sm, s>>>(p);
  return cudaGetLastError();
}

template <template <typename, int> class F, typename... A>
cudaError_t dispatch(int dtype, int d, A&&... a);

#define LS_DISPATCH(FN, dtype, d, ...)                                              \
  do {                                                                              \
    if ((dtype) == LS_DTYPE_F32) {                                                  \
      if ((d) == 64) return FN<float, 64>(__VA_ARGS__);                             \
      if ((d) == 128) return FN<float, 128>(__VA_ARGS__);                           \
      if ((d) == 256) return FN<float, 256>(__VA_ARGS__);                           \
    } else {                                                                        \
      if ((d) == 64) return FN<__nv_bfloat16, 64>(__VA_ARGS__);                     \
      if ((d) == 128) return FN<__nv_bfloat16, 128>(__VA_ARGS__);                   \
      if ((d) == 256) return FN<__nv_bfloat16, 256>(__VA_ARGS__);                   \
    }                                                                               \
    return cudaErrorInvalidValue;                                                   \
  } while (0)

}  // namespace

cudaError_t launch_page_write(int dtype, int hkv, int d, int page_size, void* k_pool,
                              void* v_pool, int64_t pool_pages, const int32_t* pt,
                              int64_t start_pos, int64_t n_tok, const void* k,
                              const void* v, uint32_t* status, cudaStream_t s) {
  if (n_tok == 0) return cudaSuccess;
  const int esize = dtype == LS_DTYPE_F32 ? 4 : 2;
  const int64_t rows = n_tok * hkv;
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t want = (rows + 7) / 8;
  const unsigned grid = (unsigned)(want < (int64_t)sms * 8 ? want : (int64_t)sms * 8);
  LaunchScope ls(kKPageWrite, s);
  page_write_kernel<<<grid, 256, 0, s>>>(d * esize, hkv, page_size,
                                         reinterpret_cast<char*>(k_pool),
                                         reinterpret_cast<char*>(v_pool), pool_pages, pt,
                                         start_pos, n_tok, reinterpret_cast<const char*>(k),
                                         reinterpret_cast<const char*>(v), status);
  return cudaGetLastError();
}

cudaError_t launch_stage_pages(int64_t page_bytes, const void* k_src, const void* v_src,
                               int64_t src_pages, const int32_t* pt, int64_t first, int n_pages,
                               void* k_dst, void* v_dst, uint32_t* status, cudaStream_t s) {
  if (n_pages == 0) return cudaSuccess;
  constexpr int64_t kStageBlocks = 38;
  const int64_t pieces = 2 * (int64_t)n_pages * (page_bytes >> 4);
  const int64_t want = (pieces + 4 * 256 - 1) / (4 * 256);
  const unsigned grid = (unsigned)(want < kStageBlocks ? want : kStageBlocks);
  LaunchScope ls(kKStagePages, s);
  stage_pages_kernel<<<grid, 256, 0, s>>>(page_bytes, reinterpret_cast<const char*>(k_src),
                                          reinterpret_cast<const char*>(v_src), src_pages, pt, first,
                                          n_pages, reinterpret_cast<char*>(k_dst),
                                          reinterpret_cast<char*>(v_dst), status);
  return cudaGetLastError();
}

cudaError_t launch_lse_merge(int n_parts, int64_t n_rows, int d, const float* o_parts,
                             const float* lse_parts, int out_dtype, void* o, float* lse,
                             cudaStream_t s) {
  const int64_t threads = n_rows * (d / 4);
  if (threads == 0) return cudaSuccess;
  const unsigned grid = (unsigned)((threads + 255) / 256);
  LaunchScope ls(kKLseMerge, s);
  if (out_dtype == LS_DTYPE_F32)
    lse_merge_kernel<float><<<grid, 256, 0, s>>>(n_parts, n_rows, d, o_parts, lse_parts,
                                                 reinterpret_cast<float*>(o), lse);
  else
    lse_merge_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(
        n_parts, n_rows, d, o_parts, lse_parts, reinterpret_cast<__nv_bfloat16*>(o), lse);
  return cudaGetLastError();
}

cudaError_t launch_bwd_preprocess(int dtype, int64_t n_rows, int d, const void* o,
                                  const void* d_o, float* delta, cudaStream_t s) {
  if (n_rows == 0) return cudaSuccess;
  const unsigned grid = (unsigned)((n_rows + 7) / 8);
  LaunchScope ls(kKBwdPre, s);
  if (dtype == LS_DTYPE_F32)
    bwd_preprocess_kernel<float><<<grid, 256, 0, s>>>(n_rows, d, reinterpret_cast<const float*>(o),
                                                      reinterpret_cast<const float*>(d_o), delta);
  else
    bwd_preprocess_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(
        n_rows, d, reinterpret_cast<const __nv_bfloat16*>(o),
        reinterpret_cast<const __nv_bfloat16*>(d_o), delta);
  return cudaGetLastError();
}

cudaError_t launch_dq_reduce(int n_parts, int64_t n_rows, int d, float scale,
                             const float* parts, int out_dtype, void* dq, cudaStream_t s) {
  const int64_t n_elems = n_rows * d;
  if (n_elems == 0) return cudaSuccess;
  const unsigned grid = (unsigned)((n_elems / 4 + 255) / 256);
  LaunchScope ls(kKDqReduce, s);
  if (out_dtype == LS_DTYPE_F32)
    dq_reduce_kernel<float><<<grid, 256, 0, s>>>(n_parts, n_elems, scale, parts,
                                                 reinterpret_cast<float*>(dq));
  else
    dq_reduce_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(n_parts, n_elems, scale, parts,
                                                         reinterpret_cast<__nv_bfloat16*>(dq));
  return cudaGetLastError();
}

cudaError_t launch_simt_fwd(int dtype, const FwdParams& p, cudaStream_t s) {
  LS_DISPATCH(fwd_impl, dtype, p.g.d, p, 0, launch_parts(p.g), s);
}
cudaError_t launch_simt_fwd_resp(int dtype, const FwdParams& p, cudaStream_t s) {
  LS_DISPATCH(fwd_impl, dtype, p.g.d, p, p.g.ns, 1, s);
}
cudaError_t launch_simt_bwd_dq(int dtype, const BwdParams& p, cudaStream_t s) {
  LS_DISPATCH(bwd_impl, dtype, p.g.d, p, 0, launch_parts(p.g), s);
}
cudaError_t launch_simt_bwd_dq_resp(int dtype, const BwdParams& p, cudaStream_t s) {
  LS_DISPATCH(bwd_impl, dtype, p.g.d, p, p.g.ns, 1, s);
}
cudaError_t launch_simt_dkdv(int dtype, const BwdParams& p, cudaStream_t s) {
  LS_DISPATCH(dkdv_impl, dtype, p.g.d, p, s);
}

}  // namespace ls
