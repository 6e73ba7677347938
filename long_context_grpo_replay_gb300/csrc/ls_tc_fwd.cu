// Tensor-core (tcgen05/TMEM) prompt-attention forward for bf16, head dim 256.
//
// One CTA owns a work unit (KV head g, 128-row query tile, key part):
//   rows  : t = hh*R + r over the Gq query heads of KV head g (so the K/V tile
//           staged in shared memory serves all Gq heads of the group),
//   keys  : part s < ns: a contiguous range of logical prompt positions,
//           streamed page by page through the page table with TMA (a key tile
//           never crosses a page); part ns: the response keys with the causal
//           mask, read through a 4-D map over [R][Hkv][256].
// Output: float32 partial O (normalised) and partial LSE (natural log) for
// the part, merged exactly afterwards by the LSE-merge kernel (the global
// LSE and output merge of the LongStraw DeepRead summary, section Method).
//
// tc_fwd_ring_kernel streams K and V through a ring of 32 KB chunks.  Warp
// roles (384 threads):
//   warp 0        : TMA producer for K and V (one instruction per chunk)
//   warp 1 lane 0 : MMA issuer: S[b] = Q K^T (SS), O += P V (P from tensor
//                   memory, V as an N-major B operand)
//   warp 2        : tensor-memory allocation / release
//   warps 4-11    : softmax, two threads per query row (TMEM lane): read S,
//                   mask, keep the running max/sum in the log2 domain with
//                   lazy rescaling (the running max only moves when the tile
//                   max exceeds it by more than 8, so exp2 stays below 256),
//                   write P as bf16 and finally normalise O.
// Tensor memory: O in columns [0,256), S double-buffered at 256 + b*128.
#include <cuda.h>
#include <cuda_bf16.h>
#include <math_constants.h>

#include <cstdlib>
#include <cstring>

#include "ls_internal.h"
#include "ls_tc.cuh"

namespace ls {
namespace {
using namespace tc;

constexpr int kD = 256;
constexpr int kBM = 128;
constexpr int kThreads = 256;
constexpr float kLn2f = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct FwdKParams {
  int32_t hq, hkv, gq, R;
  int64_t P;
  int64_t pool_rows;        // pool_pages * hkv * page_size
  int64_t pool_pages;
  int32_t page_size;
  int32_t ns;
  int64_t split_span;
  int32_t n_mt;             // query tiles per KV head
  float scale_log2;
  const __nv_bfloat16* q;
  const int32_t* page_table;
  float* o_parts;
  float* lse_parts;
  uint32_t* status;
};

// ===========================================================================
// Chunk-ring forward (default), 128-key tiles.  K and V stream through one
// ring of five 32 KB shared-memory chunks.  A "unit" is one K tile (two
// chunks: columns 0-127 and 128-255 of 128 keys) or one V tile (two chunks:
// keys 0-63 and 64-127, all 256 columns); the producer loads units in the
// order the MMA thread consumes them,
//   K_0, K_1, V_0, K_2, V_1, ..., K_{n-1}, V_{n-2}, V_{n-1},
// and a chunk slot is reloaded as soon as the MMAs that read its previous
// chunk are done: each half of a unit is released on its own, half a group
// before the unit ends, which is what lets K_{j+1} and V_j land before S_{j+1}
// and PV_j need them with only five chunks.  Per tile the MMA thread waits
// three times (K unit, P_j, V unit) and commits six (S ready, four chunks
// done, O updated).
// Softmax: eight warps, two threads per query row, each taking half of the
// tile's keys and half of O's columns.  Both threads of a row read all 128
// S columns for the row maximum (so they agree on it without exchanging
// anything) and meet on an mbarrier before the P stores that overwrite S.
// ===========================================================================
struct FwdRingLayout {
  static constexpr int BN = 128, NC = 5, NU = 4, NCD = 8;
  static constexpr uint32_t kQBytes = kBM * kD * 2;  // 64 KB
  static constexpr uint32_t kQBox = kBM * 128;       // 16 KB
  static constexpr uint32_t kChunk = 32768;
  static constexpr uint32_t kKBox = BN * 128;        // K chunk: 2 boxes [128 x 64]
  static constexpr uint32_t kVBox = (BN / 2) * 128;  // V chunk: 4 boxes [64 x 64]
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kRing = kQ + kQBytes;
  static constexpr uint32_t kEnd = kRing + NC * kChunk;
  static constexpr uint32_t kSmem = kEnd + 1024;
  static constexpr uint32_t kTmemS = 256;
  static_assert(kTmemS + 2 * BN <= 512, "tensor memory budget");
  static_assert(kSmem <= 227 * 1024 - 512, "shared memory budget");
  // a unit's full barrier is reused by unit u+NU, which can only load after
  // unit u+1 is done; a chunk's done barrier is reused by chunk c+NCD, which
  // can only load after chunk c+NCD-NC is done
  static_assert(NU >= 3 && NCD > NC, "barrier rings");
};

// Position of K_j / V_j in the unit sequence of a part with n tiles.
__device__ __forceinline__ int unit_of_k(int j) { return j == 0 ? 0 : 2 * j - 1; }
__device__ __forceinline__ int unit_of_v(int j, int n) { return j < n - 1 ? 2 * j + 2 : 2 * n - 1; }

__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

constexpr int kThreadsRing = 384;  // 4 control warps + 8 softmax warps

__global__ void __launch_bounds__(kThreadsRing, 1)
    tc_fwd_ring_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ CUtensorMap tmKr, const __grid_constant__ CUtensorMap tmVr,
                       const FwdKParams p) {
  using L = FwdRingLayout;
  constexpr int BN = L::BN, NC = L::NC, NU = L::NU, NCD = L::NCD;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_q, bar_uf[NU], bar_cd[NCD], bar_sf[2], bar_pf[2], bar_sr, bar_od, bar_ofin,
      bar_drain;
  __shared__ uint32_t tmem_base_s;
  __shared__ uint32_t abort_s;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQ = sbase + L::kQ, sRing = sbase + L::kRing;

  const int mt = blockIdx.x % p.n_mt;
  const int kvh = (blockIdx.x / p.n_mt) % p.hkv;
  const int part = blockIdx.x / (p.n_mt * p.hkv);
  const bool resp = part == p.ns;
  const int64_t rows_g = (int64_t)p.gq * p.R;
  int64_t kb, ke;
  if (!resp) {
    kb = (int64_t)part * p.split_span;
    ke = kb + p.split_span < p.P ? kb + p.split_span : p.P;
  } else {
    const int64_t t0 = (int64_t)mt * kBM;
    const int64_t t1 = (t0 + kBM < rows_g ? t0 + kBM : rows_g) - 1;
    kb = 0;
    ke = (t0 / p.R == t1 / p.R) ? (t1 % p.R) + 1 : p.R;
  }
  const int ntiles = ke > kb ? (int)((ke - kb + BN - 1) / BN) : 0;
  const int nunits = 2 * ntiles;

  if (tid == 0) {
    abort_s = 0;
    mbar_init(smem_u32(&bar_q), 256);
    mbar_init(smem_u32(&bar_sr), 256);
    for (int u = 0; u < NU; ++u) mbar_init(smem_u32(&bar_uf[u]), 1);
    for (int c = 0; c < NCD; ++c) mbar_init(smem_u32(&bar_cd[c]), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&bar_sf[b]), 1);
      mbar_init(smem_u32(&bar_pf[b]), 256);
    }
    mbar_init(smem_u32(&bar_od), 1);
    mbar_init(smem_u32(&bar_ofin), 1);
    mbar_init(smem_u32(&bar_drain), 1);
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(&tmem_base_s), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base_s;
  const volatile uint32_t* abortp = &abort_s;
  auto fail = [&](int line) {
    atomicOr(p.status, kStatusTimeout);
    atomicCAS(p.status + 1, 0u, ((uint32_t)kKTcFwd << 16) | (uint32_t)line);
    abort_s = 1;
  };
  auto chunk_addr = [&](int c) -> uint32_t { return sRing + (uint32_t)(c % NC) * L::kChunk; };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (ntiles > 0) {
      if (lane == 0) {
        prefetch_tmap(resp ? &tmKr : &tmK);
        prefetch_tmap(resp ? &tmVr : &tmV);
      }
      // Page ids are fetched one K tile ahead, so the page-table load latency
      // is not on the issue path; a K tile's row is kept until its V tile.
      auto page_of = [&](int j) -> int32_t {
        return resp ? 0 : __ldg(p.page_table + (kb + (int64_t)j * BN) / p.page_size);
      };
      auto row_of = [&](int32_t slot, int j) -> int32_t {
        if (resp) return 0;
        if (slot < 0 || slot >= p.pool_pages) {
          if (lane == 0) atomicOr(p.status, kStatusBadPage);
          return (int32_t)p.pool_rows;  // out of range: the load reads zeros
        }
        return (int32_t)(((int64_t)slot * p.hkv + kvh) * p.page_size + (kb + (int64_t)j * BN) % p.page_size);
      };
      int32_t pf_slot = page_of(0);
      int32_t rk = 0, rk_prev = 0;  // rows of the last K tile issued (jk) and of jk-1
      int jk = -1;
      int issued = 0;
      bool ok = true;
      for (int u = 0; ok && u < nunits; ++u) {
        // which tile and operand this unit carries
        bool isK;
        int j;
        if (u == 0) {
          isK = true, j = 0;
        } else if (u & 1) {
          j = (u + 1) / 2;
          isK = j < ntiles;
          if (!isK) j = ntiles - 1;
        } else {
          isK = false, j = (u - 2) / 2;
        }
        const int64_t key0 = kb + (int64_t)j * BN;
        int32_t row;
        if (isK) {
          rk_prev = rk;
          rk = row_of(pf_slot, j);
          jk = j;
          if (j + 1 < ntiles) pf_slot = page_of(j + 1);
          row = rk;
        } else {
          row = j == jk ? rk : rk_prev;  // V_j follows K_{j+1}, or K_j for the last tile
        }
        const uint32_t fb = smem_u32(&bar_uf[u % NU]);
        for (int h = 0; h < 2; ++h) {
          const int c = 2 * u + h;
          if (c >= NC) {  // the slot's previous chunk, c-NC, must be done
            const int v = c - NC;
            if (!mbar_wait_warp(smem_u32(&bar_cd[v % NCD]), (v / NCD) & 1, abortp)) {
              if (lane == 0) fail(__LINE__);
              ok = false;
              break;
            }
          }
          if (h == 0 && lane == 0) mbar_expect_tx(fb, 2 * L::kChunk);
          __syncwarp();
          if (lane == 0) {
            const uint32_t dst = chunk_addr(c);
            if (isK) {
              if (resp) tma_load_4d(dst, &tmKr, fb, 0, (int32_t)key0, 2 * h, kvh);
              else      tma_load_3d(dst, &tmK, fb, 0, row, 2 * h);
            } else {
              if (resp) tma_load_4d(dst, &tmVr, fb, 0, (int32_t)(key0 + 64 * h), 0, kvh);
              else      tma_load_3d(dst, &tmV, fb, 0, row + 64 * h, 0);
            }
          }
          __syncwarp();
        }
        if (ok) issued = u + 1;
      }
      // no copy may still be landing in shared memory when the CTA ends
      for (int u = issued - NU < 0 ? 0 : issued - NU; u < issued; ++u)
        mbar_wait(smem_u32(&bar_uf[u % NU]), (u / NU) & 1, abortp);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && ntiles > 0) {
      constexpr uint32_t idesc_qk = idesc_bf16(kBM, BN, false);
      constexpr uint32_t idesc_pv = idesc_bf16(kBM, kD, true);
      auto issue_s = [&](int j) -> bool {  // S[b] = Q K_j^T
        const int u = unit_of_k(j);
        if (!mbar_wait(smem_u32(&bar_uf[u % NU]), (u / NU) & 1, abortp)) { fail(__LINE__); return false; }
        tc_fence_after();
        const uint32_t dS = tbase + L::kTmemS + (j & 1) * BN;
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t kc = chunk_addr(2 * u + (kk >> 3));
          mma_ss(dS, sdesc_sw128(sQ + (kk >> 2) * L::kQBox + (kk & 3) * 32, 16, 1024),
                 sdesc_sw128(kc + ((kk >> 2) & 1) * L::kKBox + (kk & 3) * 32, 16, 1024), idesc_qk,
                 kk > 0 ? 1u : 0u);
          if (kk == 7) mma_commit(smem_u32(&bar_cd[(2 * u) % NCD]));  // columns 0-127 read
        }
        mma_commit(smem_u32(&bar_sf[j & 1]));
        mma_commit(smem_u32(&bar_cd[(2 * u + 1) % NCD]));
        return true;
      };
      bool ok = mbar_wait(smem_u32(&bar_q), 0, abortp);
      if (!ok) fail(__LINE__);
      tc_fence_after();
      if (ok) ok = issue_s(0);
      for (int j = 0; ok && j < ntiles; ++j) {
        // S_{j+1} goes into the other S buffer; its previous contents (P_{j-1})
        // were read by PV_{j-1}, issued before this
        if (j + 1 < ntiles && !issue_s(j + 1)) break;
        const int b = j & 1;
        const int u = unit_of_v(j, ntiles);
        if (!mbar_wait(smem_u32(&bar_pf[b]), (j >> 1) & 1, abortp) ||
            !mbar_wait(smem_u32(&bar_uf[u % NU]), (u / NU) & 1, abortp)) {
          fail(__LINE__);
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          const uint32_t vc = chunk_addr(2 * u + (kk >> 2));
          mma_ts(tbase, tbase + L::kTmemS + b * BN + kk * 8,
                 sdesc_sw128(vc + (kk & 3) * 16 * 128, L::kVBox, 1024), idesc_pv,
                 (j > 0 || kk > 0) ? 1u : 0u);
          if (kk == 3) mma_commit(smem_u32(&bar_cd[(2 * u) % NCD]));  // keys 0-63 read
        }
        mma_commit(smem_u32(&bar_cd[(2 * u + 1) % NCD]));
        mma_commit(smem_u32(&bar_od));
        if (j == ntiles - 1) mma_commit(smem_u32(&bar_ofin));
      }
      mma_commit(smem_u32(&bar_drain));
      mbar_wait(smem_u32(&bar_drain), 0, abortp);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    // Eight warps, two threads per query row: warp 4+q and warp 8+q both
    // reach tensor-memory lanes 32q..32q+31; half hf = 0 / 1 owns keys
    // 0-63 / 64-127 of each tile and O columns 0-127 / 128-255.
    const int sw = warp - 4, q4 = sw & 3, hf = sw >> 2;
    const int i = q4 * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const int64_t t = (int64_t)mt * kBM + i;
    const bool row_ok = t < rows_g;
    const int hh = row_ok ? (int)(t / p.R) : 0;
    const int r = row_ok ? (int)(t % p.R) : 0;
    const int64_t n = (int64_t)r * p.hq + (int64_t)kvh * p.gq + hh;
    {
      for (int rr = 0; rr < 16; ++rr) {
        const int row = sw * 16 + rr;
        const int64_t tt = (int64_t)mt * kBM + row;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (tt < rows_g) {
          const int hh2 = (int)(tt / p.R), r2 = (int)(tt % p.R);
          const int64_t n2 = (int64_t)r2 * p.hq + (int64_t)kvh * p.gq + hh2;
          v = __ldg(reinterpret_cast<const uint4*>(p.q + n2 * kD) + lane);
        }
        st_shared_v4(sQ + (lane >> 3) * L::kQBox + sw128_offset(row, lane & 7), v);
      }
      fence_proxy_async_smem();
      mbar_arrive(smem_u32(&bar_q));
    }

    float m_run = -CUDART_INF_F, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      const int b = j & 1;
      const int64_t tkey0 = kb + (int64_t)j * BN;
      // a tile whose page id lies outside the pool holds no keys (the
      // producer loaded zeros for it and flagged the status word); the id is
      // read before the wait so that its latency hides behind it
      const int32_t tslot = resp ? 0 : __ldg(p.page_table + tkey0 / p.page_size);
      if (!mbar_wait_warp(smem_u32(&bar_sf[b]), (j >> 1) & 1, abortp)) { fail(__LINE__); ok = false; break; }
      tc_fence_after();
      const int64_t lim = resp ? (int64_t)r + 1 : (tslot >= 0 && tslot < p.pool_pages ? ke : tkey0);
      // visible keys of this row in the tile, and in each half
      const int nv_row = (int)(lim - tkey0 < 0 ? 0 : (lim - tkey0 < BN ? lim - tkey0 : BN));
      const bool full = !resp && nv_row == BN;  // the common case skips the masks
      // Row maximum over all 128 keys: first the other half's columns (read
      // only for the maximum), then this half's, which are kept.  Both
      // threads of a row see the same values, so they agree on the maximum.
      float mq[4];
      {
        uint32_t r0[32], r1[32];
        const int oh = 1 - hf;
        const uint32_t sa = tbase + lane_off + L::kTmemS + b * BN + oh * 64;
        tmem_ld32(sa, r0);
        tmem_ld32(sa + 32, r1);
        tmem_wait_ld_r(r0);
        reg_dep(r1);
        const int nvo = nv_row - oh * 64;
#pragma unroll
        for (int q = 0; q < 4; ++q) mq[q] = -CUDART_INF_F;
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          const float a0 = full || c < nvo ? __uint_as_float(r0[c]) : -CUDART_INF_F;
          const float a1 = full || c + 1 < nvo ? __uint_as_float(r0[c + 1]) : -CUDART_INF_F;
          const float b0 = full || c + 32 < nvo ? __uint_as_float(r1[c]) : -CUDART_INF_F;
          const float b1 = full || c + 33 < nvo ? __uint_as_float(r1[c + 1]) : -CUDART_INF_F;
          mq[(c >> 1) & 1] = max3f(mq[(c >> 1) & 1], a0, a1);
          mq[2 + ((c >> 1) & 1)] = max3f(mq[2 + ((c >> 1) & 1)], b0, b1);
        }
      }
      float s[64];
      {
        uint32_t r0[32], r1[32];
        const uint32_t sa = tbase + lane_off + L::kTmemS + b * BN + hf * 64;
        tmem_ld32(sa, r0);
        tmem_ld32(sa + 32, r1);
        tmem_wait_ld_r(r0);
        reg_dep(r1);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          s[c] = __uint_as_float(r0[c]);
          s[32 + c] = __uint_as_float(r1[c]);
        }
      }
      // S reads of this tile are done: the P stores below overwrite S
      // columns the other half reads, so both halves meet first
      tc_fence_before();
      mbar_arrive(smem_u32(&bar_sr));
      if (!full) {
        const int nv = nv_row - hf * 64;
#pragma unroll
        for (int c = 0; c < 64; ++c) s[c] = c < nv ? s[c] : -CUDART_INF_F;
      }
#pragma unroll
      for (int c = 0; c < 64; c += 4) {
        mq[(c >> 2) & 3] = max3f(mq[(c >> 2) & 3], s[c], s[c + 1]);
        mq[(c >> 2) & 3] = max3f(mq[(c >> 2) & 3], s[c + 2], s[c + 3]);
      }
      const float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])) * p.scale_log2;
      // lazy rescale, identical in both halves of a row (same maximum)
      float alpha = 1.f;
      bool rescale_o = false;
      if (mx > m_run + kRescaleThreshold) {
        if (m_run != -CUDART_INF_F) {
          alpha = ex2(m_run - mx);
          rescale_o = true;
        }
        l_run *= alpha;
        m_run = mx;
      }
      if (__any_sync(0xffffffffu, rescale_o)) {
        // O holds PV_0..PV_{j-1}; S_j complete implies PV_{j-2} complete, so
        // bar_od has completed j-1 or j phases and the parity is unambiguous
        if (!mbar_wait_warp(smem_u32(&bar_od), (j - 1) & 1, abortp)) { fail(__LINE__); ok = false; break; }
        tc_fence_after();
#pragma unroll 1
        for (int c0 = hf * 128; c0 < hf * 128 + 128; c0 += 32) {
          uint32_t rr[32];
          tmem_ld32(tbase + lane_off + c0, rr);
          tmem_wait_ld_r(rr);
#pragma unroll
          for (int c = 0; c < 32; ++c) rr[c] = __float_as_uint(__uint_as_float(rr[c]) * alpha);
          tmem_st32(tbase + lane_off + c0, rr);
        }
        tmem_wait_st();
      }
      uint32_t pk[32];
      float ps[4] = {0.f, 0.f, 0.f, 0.f};
      if (m_run != -CUDART_INF_F) {
        // the exponents' arguments and the row sums two keys per packed
        // instruction
        const uint64_t sc2 = f2(p.scale_log2, p.scale_log2), nm2 = f2(-m_run, -m_run);
        uint64_t acc[2] = {f2(0.f, 0.f), f2(0.f, 0.f)};
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          float x0, x1;
          f2_split(f2_fma(f2(s[c], s[c + 1]), sc2, nm2), x0, x1);
          const float p0 = ex2(x0), p1 = ex2(x1);
          acc[(c >> 1) & 1] = f2_add(acc[(c >> 1) & 1], f2(p0, p1));
          pk[c >> 1] = pack_bf16x2(p0, p1);
        }
        f2_split(acc[0], ps[0], ps[1]);
        f2_split(acc[1], ps[2], ps[3]);
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) pk[c] = 0u;
      }
      l_run += (ps[0] + ps[1]) + (ps[2] + ps[3]);
      if (!mbar_wait_warp(smem_u32(&bar_sr), j & 1, abortp)) { fail(__LINE__); ok = false; break; }
      tc_fence_after();
      // P (bf16 pairs) of keys 64hf.. goes to columns 32hf.. of the S buffer
#pragma unroll
      for (int c0 = 0; c0 < 32; c0 += 16)
        tmem_st16(tbase + lane_off + L::kTmemS + b * BN + hf * 32 + c0, pk + c0);
      tmem_wait_st();
      const int nvalid_tile = (int)(ke - (kb + (int64_t)j * BN) < BN ? ke - (kb + (int64_t)j * BN) : BN);
      if (!resp && nvalid_tile < BN) {
        // partial last prompt tile: rows past the prompt end may hold anything
        // (NaN included); zero them in V so that P = 0 times V stays 0
        const int u = unit_of_v(j, ntiles);
        if (!mbar_wait_warp(smem_u32(&bar_uf[u % NU]), (u / NU) & 1, abortp)) { fail(__LINE__); ok = false; break; }
        const int nz = (BN - nvalid_tile) * 4 * 8;  // 16-byte pieces
        for (int z = sw * 32 + lane; z < nz; z += 256) {
          const int key = nvalid_tile + z / 32;
          const int box = (z / 8) & 3;
          const uint32_t vc = chunk_addr(2 * u + (key >> 6));
          st_shared_v4(vc + box * L::kVBox + (key & 63) * 128 + (z & 7) * 16, make_uint4(0u, 0u, 0u, 0u));
        }
        fence_proxy_async_smem();
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&bar_pf[b]));
    }

    // ---- epilogue: the row sum of both halves (exchanged through two
    // tensor-memory columns of the idle S buffer once every PV is done), then
    // the normalised O columns of this half and (half 0) the LSE
    if (ok && ntiles > 0) {
      if (!mbar_wait_warp(smem_u32(&bar_ofin), 0, abortp)) { fail(__LINE__); ok = false; }
      tc_fence_after();
      if (ok) {
        tmem_st1(tbase + lane_off + L::kTmemS + hf, __float_as_uint(l_run));
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(smem_u32(&bar_sr));
        if (!mbar_wait_warp(smem_u32(&bar_sr), ntiles & 1, abortp)) { fail(__LINE__); ok = false; }
        tc_fence_after();
      }
      if (ok) {
        uint32_t l0, l1;
        tmem_ld1x2(tbase + lane_off + L::kTmemS, tbase + lane_off + L::kTmemS + 1, l0, l1);
        l_run = __uint_as_float(l0) + __uint_as_float(l1);
      }
    }
    const int64_t nrows = (int64_t)p.R * p.hq;
    float* orow = p.o_parts + ((int64_t)part * nrows + n) * kD;
    const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll 1
    for (int c0 = hf * 128; c0 < hf * 128 + 128; c0 += 32) {
      uint32_t rr[32];
      __syncwarp();
      if (ok && ntiles > 0) {
        tmem_ld32(tbase + lane_off + c0, rr);
        tmem_wait_ld_r(rr);
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) rr[c] = 0u;
      }
      if (row_ok) {
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
          float4 v = make_float4(__uint_as_float(rr[c]) * inv, __uint_as_float(rr[c + 1]) * inv,
                                 __uint_as_float(rr[c + 2]) * inv, __uint_as_float(rr[c + 3]) * inv);
          *reinterpret_cast<float4*>(orow + c0 + c) = v;
        }
      }
    }
    if (row_ok && hf == 0)
      p.lse_parts[(int64_t)part * nrows + n] =
          (ok && l_run > 0.f) ? (m_run + __log2f(l_run)) * kLn2f : -CUDART_INF_F;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

cudaError_t fwd_ring(const FwdParams& a, cudaStream_t s) {
  using L = FwdRingLayout;
  const AttnGeom& g = a.g;
  FwdKParams p;
  p.hq = g.hq;
  p.hkv = g.hkv;
  p.gq = g.gq;
  p.R = g.R;
  p.P = g.P;
  p.pool_pages = g.pool_pages;
  p.pool_rows = g.pool_pages * g.hkv * g.page_size;
  p.page_size = g.page_size;
  p.ns = g.ns;
  p.split_span = g.split_span;
  p.n_mt = (int)(((int64_t)g.gq * g.R + kBM - 1) / kBM);
  p.scale_log2 = g.scale_log2;
  p.q = reinterpret_cast<const __nv_bfloat16*>(a.q);
  p.page_table = a.page_table;
  p.o_parts = a.o_parts;
  p.lse_parts = a.lse_parts;
  p.status = a.status;
  CUtensorMap tk, tv, tkr, tvr;
  memset(&tk, 0, sizeof(tk));
  memset(&tv, 0, sizeof(tv));
  // K units: [128 keys x 128 columns] (two column blocks); V units: [64 keys x 256 columns]
  if (g.P > 0 && (!encode_pool_tile_map(&tk, a.k_pool, p.pool_rows, L::BN, 2) ||
                  !encode_pool_tile_map(&tv, a.v_pool, p.pool_rows, L::BN / 2, 4)))
    return cudaErrorInvalidValue;
  if (!encode_rows_tile_map(&tkr, a.k_resp, g.hkv, g.R, L::BN, 2) ||
      !encode_rows_tile_map(&tvr, a.v_resp, g.hkv, g.R, L::BN / 2, 4))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(tc_fwd_ring_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)L::kSmem);
  if (e != cudaSuccess) return e;
  const int64_t units = (int64_t)launch_parts(g) * g.hkv * p.n_mt;
  if (units == 0) return cudaSuccess;
  LaunchScope ls(kKTcFwd, s);
  tc_fwd_ring_kernel<<<(unsigned)units, kThreadsRing, L::kSmem, s>>>(tk, tv, tkr, tvr, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tc_fwd(const FwdParams& a, cudaStream_t s) { return fwd_ring(a, s); }

}  // namespace ls
