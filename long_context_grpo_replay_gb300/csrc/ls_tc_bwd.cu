// Tensor-core (tcgen05/TMEM) prompt-attention backward for bf16, head dim 256:
// the query gradient only.  The prompt K/V are stop-gradient (LongStraw
// DeepRead summary, section Method, last paragraph; the review's mind map,
// node on equations 1-3), so no dK/dV is formed for prompt keys and the kernel is
// query-stationary: a CTA keeps its 128 query rows (Q and dO tiles) in shared
// memory, streams the part's key pages, recomputes P from the stored LSE and
// accumulates dQ in tensor memory.  No score matrix is kept between tiles.
//
// Per key tile j (128 keys), with dO held in tensor memory as the A operand
// of dP = dO V^T:
//   S_j  = Q K_j^T            (tcgen05, SS)        -> TMEM X
//   dP_j = dO V_j^T           (tcgen05, TS)        -> TMEM X (after S_j is read)
//   softmax warps: P = exp2(S*scale*log2e - LSE*log2e), dS = P * (dP - delta),
//                  dS (bf16) written back over X
//   dQ  += dS_j K_j           (tcgen05, A from TMEM, K as N-major B operand)
// (details and the shared-memory ring below, at the kernel).
// Output: unscaled float32 dQ partial of the part; the reduction kernel sums
// parts and applies the softmax scale.
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
constexpr float kLog2ef = 1.4426950408889634f;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct BwdKParams {
  int32_t hq, hkv, gq, R;
  int64_t P;
  int64_t pool_rows;
  int64_t pool_pages;
  int32_t page_size;
  int32_t ns;
  int64_t split_span;
  int32_t n_mt;
  float scale_log2;
  const __nv_bfloat16* q;
  const __nv_bfloat16* d_o;
  const float* lse;
  const float* delta;
  const int32_t* page_table;
  float* dq_parts;
  uint32_t* status;
};

// ===========================================================================
// Backward with 128-key tiles at the tensor pipe's full rate.
//
// The dQ accumulator (256 columns) and dO (128 columns of bf16 pairs) leave
// one 128-column tensor-memory area X, which S_j, dP_j and dS_j share in
// turn, so S and dP are N=128 MMAs (an N=64 MMA costs as much as an N=128
// one).  Per key tile j the MMA thread issues
//   S_j  = Q K_j^T   into X            (16 x N=128, SS)   commit s_full
//   dP_j = dO V_j^T  into X            (16 x N=128, TS)   commit dp_full
//   dQ  += dS_j K_j  (dS_j from X)     (2 halves x 8 x N=128, TS) commit dq_done
// and waits between them for the softmax warps: s_free (S_j read into
// registers) before dP_j, ds_full (dS_j written over X) before dQ_j.  S_{j+1}
// overwrites X after dQ_j, which read dS_j, was issued before it.
// K and V stream through a ring of five 32 KB chunks ([128 keys x 128
// columns], two swizzled [128 x 64] boxes).  Chunk n = 4j + {0, 1, 2, 3}
// holds columns 0-127 / 128-255 of K_j / V_j; a V chunk is free once dP of
// its tile is done (dp_full), a K chunk once dQ of its tile is done
// (dq_done).  Chunk n reuses the slot of chunk n-7 (n = 0, 3 mod 4) or n-3
// (n = 1, 2 mod 4): the slot freed earliest that keeps every load about a
// thousand cycles ahead of its first MMA.  That rule is periodic in 20
// chunks (five tiles), so the slot of chunk n is a table entry.  The two
// chunks of one K or V tile land on one full barrier, so the MMA thread
// tests two barriers per tile for its operands.
// Softmax: sixteen warps, four threads per query row (two warps per
// scheduler leave the dS arithmetic, which sits on the critical path,
// latency-bound); quarter qq owns keys 32qq..32qq+31 of each tile and writes
// their dS (bf16 pairs) over the first half of its own dP columns.
// ===========================================================================
struct BwdRingLayout {
  static constexpr int BN = 128, NC = 5, NF = 4;  // NF: full barriers, one per chunk pair
  static constexpr uint32_t kRowBox = kBM * 128;  // Q box [128 rows x 64 columns], 16 KB
  static constexpr uint32_t kBox = BN * 128;      // K/V box [128 keys x 64 columns], 16 KB
  static constexpr uint32_t kChunk = 2 * kBox;    // 32 KB
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kRing = kQ + 4 * kRowBox;
  static constexpr uint32_t kEnd = kRing + NC * kChunk;
  static constexpr uint32_t kSmem = kEnd + 1024;
  static constexpr uint32_t kTmemO = 256, kTmemX = 384;
  static_assert(kSmem <= 227 * 1024 - 512, "shared memory budget");
};

// The slot rule above, run for 40 chunks: slots of chunks 0-19, 3 bits each.
constexpr int ring_pred(int n) { return (n % 4 == 0 || n % 4 == 3) ? n - 7 : n - 3; }
constexpr uint64_t ring_table() {
  int h[40] = {};
  for (int n = 0; n < 40; ++n) h[n] = n < 5 ? n : h[ring_pred(n)];
  uint64_t t = 0;
  for (int n = 0; n < 20; ++n) t |= (uint64_t)h[n] << (3 * n);
  return t;
}
constexpr bool ring_table_is_periodic() {
  int h[80] = {};
  for (int n = 0; n < 80; ++n) h[n] = n < 5 ? n : h[ring_pred(n)];
  for (int n = 20; n < 80; ++n)
    if (h[n] != h[n - 20] || h[n] > 4) return false;
  return true;
}
static_assert(ring_table_is_periodic(), "chunk slots repeat every 20 chunks");
constexpr uint64_t kRingTable = ring_table();
__device__ __forceinline__ uint32_t ring_slot(int n) {
  return (uint32_t)(kRingTable >> (3 * (n % 20))) & 7u;
}

constexpr int kThreadsRing = 640;  // 4 control warps + 16 softmax warps
constexpr int kSoftWarps = 16;

__global__ void __launch_bounds__(kThreadsRing, 1)
    tc_bwd_dq_ring_kernel(const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV,
                          const __grid_constant__ CUtensorMap tmKr,
                          const __grid_constant__ CUtensorMap tmVr, const BwdKParams p) {
  using L = BwdRingLayout;
  constexpr int BN = L::BN, NF = L::NF;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_q, bar_full[NF], bar_sf, bar_sfree, bar_dpf, bar_dsf, bar_dqd, bar_fin,
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

  if (tid == 0) {
    abort_s = 0;
    mbar_init(smem_u32(&bar_q), kSoftWarps);
    for (int f = 0; f < NF; ++f) mbar_init(smem_u32(&bar_full[f]), 1);
    mbar_init(smem_u32(&bar_sf), 1);
    mbar_init(smem_u32(&bar_sfree), kSoftWarps);
    mbar_init(smem_u32(&bar_dpf), 1);
    mbar_init(smem_u32(&bar_dsf), kSoftWarps);
    mbar_init(smem_u32(&bar_dqd), 1);
    mbar_init(smem_u32(&bar_fin), 1);
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
    atomicCAS(p.status + 1, 0u, ((uint32_t)kKTcBwdDq << 16) | (uint32_t)line);
    abort_s = 1;
  };
  auto chunk_addr = [&](int n) -> uint32_t { return sRing + ring_slot(n) * L::kChunk; };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // whole warp waits; lane 0 posts the bytes and issues one TMA per chunk
    if (ntiles > 0) {
      if (lane == 0) {
        prefetch_tmap(resp ? &tmKr : &tmK);
        prefetch_tmap(resp ? &tmVr : &tmV);
      }
      const int nch = 4 * ntiles;
      int dp_seen = -1, dq_seen = -1;  // last tile whose dP / dQ completion was awaited
      int32_t row = 0;
      int issued = 0;
      bool failed = false;
      for (int n = 0; n < nch; ++n) {
        const int j = n >> 2, kind = n & 3;
        // after a wait gave up, only the second chunk of a pair already begun
        // is still loaded, so that its full barrier completes and the drain
        // below can account for every copy in flight
        if (failed && (n & 1) == 0) break;
        if (n >= 5 && !failed) {
          // the slot's previous chunk must be done with: a V chunk after dP
          // of its tile, a K chunk after dQ of its tile
          const int pr = ring_pred(n), t = pr >> 2;
          bool ok = true;
          if ((pr & 3) < 2) {
            if (t > dq_seen) ok = mbar_wait_warp(smem_u32(&bar_dqd), t & 1, abortp), dq_seen = t;
          } else {
            if (t > dp_seen) ok = mbar_wait_warp(smem_u32(&bar_dpf), t & 1, abortp), dp_seen = t;
          }
          if (!ok) {
            if (lane == 0) fail(__LINE__);
            failed = true;
            if ((n & 1) == 0) break;
          }
        }
        const int64_t key0 = kb + (int64_t)j * BN;
        if (kind == 0 && !resp) {
          const int32_t slot = __ldg(p.page_table + key0 / p.page_size);
          if (slot < 0 || slot >= p.pool_pages) {
            if (lane == 0) atomicOr(p.status, kStatusBadPage);
            row = (int32_t)p.pool_rows;  // out of range: the load reads zeros
          } else {
            row = (int32_t)(((int64_t)slot * p.hkv + kvh) * p.page_size + key0 % p.page_size);
          }
        }
        if (lane == 0) {
          // chunks 2g and 2g+1 (the two column halves of one K or V tile)
          // land on full barrier g: armed for both with the first
          const int g = n >> 1;
          const uint32_t fb = smem_u32(&bar_full[g % NF]);
          if ((n & 1) == 0) mbar_expect_tx(fb, 2 * L::kChunk);
          const uint32_t dst = chunk_addr(n);
          if (resp)
            tma_load_4d(dst, kind < 2 ? &tmKr : &tmVr, fb, 0, (int32_t)key0, 2 * (kind & 1), kvh);
          else
            tma_load_3d(dst, kind < 2 ? &tmK : &tmV, fb, 0, row, 2 * (kind & 1));
        }
        __syncwarp();
        issued = n + 1;
      }
      // no copy may still be landing in shared memory when the CTA ends
      // (issued is even: pairs are always completed)
      const int gend = issued >> 1;
      for (int g = gend - NF < 0 ? 0 : gend - NF; g < gend; ++g)
        mbar_wait(smem_u32(&bar_full[g % NF]), (g / NF) & 1, abortp);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && ntiles > 0) {
      constexpr uint32_t idesc_s = idesc_bf16(kBM, BN, false);  // S, dP: K-major B
      constexpr uint32_t idesc_q = idesc_bf16(kBM, 128, true);  // dQ halves: N-major B
      auto wait_full = [&](int g) {  // chunk pair g: K_j is pair 2j, V_j pair 2j+1
        return mbar_wait(smem_u32(&bar_full[g % NF]), (g / NF) & 1, abortp);
      };
      bool ok = mbar_wait(smem_u32(&bar_q), 0, abortp);
      if (!ok) fail(__LINE__);
      tc_fence_after();
      for (int j = 0; ok && j < ntiles; ++j) {
        const int n0 = 4 * j;
        // S_j = Q K_j^T into X (X last held dS_{j-1}, read by dQ_{j-1} before)
        if (!wait_full(2 * j)) { fail(__LINE__); break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t kc = chunk_addr(n0 + (kk >> 3));
          mma_ss(tbase + L::kTmemX, sdesc_sw128(sQ + (kk >> 2) * L::kRowBox + (kk & 3) * 32, 16, 1024),
                 sdesc_sw128(kc + ((kk >> 2) & 1) * L::kBox + (kk & 3) * 32, 16, 1024), idesc_s,
                 kk > 0 ? 1u : 0u);
        }
        mma_commit(smem_u32(&bar_sf));
        // dP_j = dO V_j^T into X, once the softmax warps have read S_j
        if (!mbar_wait(smem_u32(&bar_sfree), j & 1, abortp) || !wait_full(2 * j + 1)) {
          fail(__LINE__);
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t vc = chunk_addr(n0 + 2 + (kk >> 3));
          mma_ts(tbase + L::kTmemX, tbase + L::kTmemO + kk * 8,
                 sdesc_sw128(vc + ((kk >> 2) & 1) * L::kBox + (kk & 3) * 32, 16, 1024), idesc_s,
                 kk > 0 ? 1u : 0u);
        }
        mma_commit(smem_u32(&bar_dpf));  // dP_j ready; V_j's chunks free
        // dQ += dS_j K_j; dS of keys 32q..32q+31 in X columns 32q..32q+15
        if (!mbar_wait(smem_u32(&bar_dsf), j & 1, abortp)) { fail(__LINE__); break; }
        tc_fence_after();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t kc = chunk_addr(n0 + h);
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            mma_ts(tbase + h * 128, tbase + L::kTmemX + 32 * (kk >> 1) + 8 * (kk & 1),
                   sdesc_sw128(kc + kk * 16 * 128, L::kBox, 1024), idesc_q,
                   (j > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(smem_u32(&bar_dqd));  // dQ_j done; K_j's chunks free
        if (j == ntiles - 1) mma_commit(smem_u32(&bar_fin));
      }
      mma_commit(smem_u32(&bar_drain));
      mbar_wait(smem_u32(&bar_drain), 0, abortp);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    // Sixteen warps, four threads per query row: warp 4 + 4qq + q reaches
    // tensor-memory lanes 32q..32q+31 (its rows) and owns quarter qq of every
    // key tile (keys 32qq..32qq+31), dO columns 64qq..64qq+63 and dQ columns
    // 64qq..64qq+63.  Each quarter writes its dS (bf16 pairs) over the first
    // half of its own dP columns, so quarters never touch each other's data.
    // One lane per warp arrives on the MMA thread's barriers.
    const int sw = warp - 4, q4 = sw & 3, qq = sw >> 2;
    const int i = q4 * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const uint32_t tX = tbase + lane_off + L::kTmemX + qq * 32;
    const int64_t t = (int64_t)mt * kBM + i;
    const bool row_ok = t < rows_g;
    const int hh = row_ok ? (int)(t / p.R) : 0;
    const int r = row_ok ? (int)(t % p.R) : 0;
    const int64_t n = (int64_t)r * p.hq + (int64_t)kvh * p.gq + hh;
    const float lse2 = row_ok ? __ldg(p.lse + n) * kLog2ef : 0.f;
    const float dl = row_ok ? __ldg(p.delta + n) : 0.f;
    auto warp_arrive = [&](uint32_t bar) {  // after each lane's own ordering
      __syncwarp();
      if (lane == 0) mbar_arrive(bar);
    };
    {
      // Q tile into shared memory (8 rows per warp, swizzled) ...
      for (int rr = 0; rr < 8; ++rr) {
        const int row = sw * 8 + rr;
        const int64_t tt = (int64_t)mt * kBM + row;
        uint4 vq = make_uint4(0u, 0u, 0u, 0u);
        if (tt < rows_g) {
          const int hh2 = (int)(tt / p.R), r2 = (int)(tt % p.R);
          const int64_t n2 = (int64_t)r2 * p.hq + (int64_t)kvh * p.gq + hh2;
          vq = __ldg(reinterpret_cast<const uint4*>(p.q + n2 * kD) + lane);
        }
        st_shared_v4(sQ + (lane >> 3) * L::kRowBox + sw128_offset(row, lane & 7), vq);
      }
      fence_proxy_async_smem();
      // ... and this quarter of the row's dO into tensor memory (bf16 pairs)
      const uint4* orow = reinterpret_cast<const uint4*>(p.d_o + n * kD) + qq * 8;
      uint32_t rr[32];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint4 v = row_ok ? __ldg(orow + u) : make_uint4(0u, 0u, 0u, 0u);
        rr[4 * u] = v.x;
        rr[4 * u + 1] = v.y;
        rr[4 * u + 2] = v.z;
        rr[4 * u + 3] = v.w;
      }
      tmem_st32(tbase + lane_off + L::kTmemO + qq * 32, rr);
      tmem_wait_st();
      tc_fence_before();
      warp_arrive(smem_u32(&bar_q));
    }

    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      const int64_t key0 = kb + (int64_t)j * BN;
      // a tile whose page id lies outside the pool holds no keys (zeros were
      // loaded for it and the status word flagged); read before the wait
      const int32_t tslot = resp ? 0 : __ldg(p.page_table + key0 / p.page_size);
      if (!mbar_wait_warp(smem_u32(&bar_sf), j & 1, abortp)) { fail(__LINE__); ok = false; break; }
      tc_fence_after();
      const int64_t lim = resp ? (int64_t)r + 1 : (tslot >= 0 && tslot < p.pool_pages ? ke : key0);
      const int64_t nvq = lim - key0 - qq * 32;
      const int nv = (int)(nvq < 0 ? 0 : (nvq < 32 ? nvq : 32));  // visible keys of this quarter
      const bool full = nv == 32;  // every key visible: no masks
      const int nvalid_tile = (int)(ke - key0 < BN ? ke - key0 : BN);
      float pv[32];
      {
        uint32_t r0[32];
        tmem_ld32(tX, r0);
        tmem_wait_ld_r(r0);
#pragma unroll
        for (int c = 0; c < 32; ++c) pv[c] = __uint_as_float(r0[c]);
      }
      tc_fence_before();
      warp_arrive(smem_u32(&bar_sfree));  // dP_j may now overwrite X
      if (full) {
        const uint64_t sc2 = f2(p.scale_log2, p.scale_log2), nl2 = f2(-lse2, -lse2);
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          float x0, x1;
          f2_split(f2_fma(f2(pv[c], pv[c + 1]), sc2, nl2), x0, x1);
          pv[c] = ex2(x0);
          pv[c + 1] = ex2(x1);
        }
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) pv[c] = c < nv ? ex2(fmaf(pv[c], p.scale_log2, -lse2)) : 0.f;
      }
      if (!mbar_wait_warp(smem_u32(&bar_dpf), j & 1, abortp)) { fail(__LINE__); ok = false; break; }
      tc_fence_after();
      uint32_t ds_pk[16];
      {
        uint32_t rp[32];
        tmem_ld32(tX, rp);
        tmem_wait_ld_r(rp);
        if (full) {
          // dS = P (dP - D), two keys per packed instruction
          const uint64_t nd2 = f2(-dl, -dl);
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            float d0, d1;
            f2_split(f2_mul(f2(pv[c], pv[c + 1]),
                            f2_add(f2(__uint_as_float(rp[c]), __uint_as_float(rp[c + 1])), nd2)),
                     d0, d1);
            ds_pk[c >> 1] = pack_bf16x2(d0, d1);
          }
        } else {
          // masked keys give dS = 0 exactly, whatever dP holds (NaN included)
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            const float d0 = c < nv ? pv[c] * (__uint_as_float(rp[c]) - dl) : 0.f;
            const float d1 = c + 1 < nv ? pv[c + 1] * (__uint_as_float(rp[c + 1]) - dl) : 0.f;
            ds_pk[c >> 1] = pack_bf16x2(d0, d1);
          }
        }
      }
      // every dP column of this quarter has been read: its dS goes over the
      // first half of those columns
      tmem_st16(tX, ds_pk);
      tmem_wait_st();
      if (!resp && nvalid_tile < BN) {
        // partial last prompt tile: rows past the prompt end may hold anything
        // (NaN included); zero them in both K chunks so that dS = 0 times K
        // stays 0 in dQ += dS K
        const int nz = (BN - nvalid_tile) * 32;  // 16-byte pieces: 2 chunks x 2 boxes x 8
        for (int z = sw * 32 + lane; z < nz; z += 32 * kSoftWarps) {
          const int row = nvalid_tile + z / 32;
          const int rem = z & 31;
          st_shared_v4(chunk_addr(4 * j + (rem >> 4)) + ((rem >> 3) & 1) * L::kBox + row * 128 +
                           (rem & 7) * 16,
                       make_uint4(0u, 0u, 0u, 0u));
        }
        fence_proxy_async_smem();
      }
      tc_fence_before();
      warp_arrive(smem_u32(&bar_dsf));
    }

    if (ok && ntiles > 0) {
      if (!mbar_wait_warp(smem_u32(&bar_fin), 0, abortp)) { fail(__LINE__); ok = false; }
      tc_fence_after();
    }
    const int64_t nrows = (int64_t)p.R * p.hq;
    float* out = p.dq_parts + ((int64_t)part * nrows + n) * kD;
#pragma unroll 1
    for (int c0 = qq * 64; c0 < qq * 64 + 64; c0 += 32) {
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
        for (int c = 0; c < 32; c += 4)
          *reinterpret_cast<float4*>(out + c0 + c) =
              make_float4(__uint_as_float(rr[c]), __uint_as_float(rr[c + 1]),
                          __uint_as_float(rr[c + 2]), __uint_as_float(rr[c + 3]));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

cudaError_t bwd_ring(const BwdParams& a, cudaStream_t s) {
  using L = BwdRingLayout;
  const AttnGeom& g = a.g;
  BwdKParams p;
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
  p.d_o = reinterpret_cast<const __nv_bfloat16*>(a.d_o);
  p.lse = a.lse;
  p.delta = a.delta;
  p.page_table = a.page_table;
  p.dq_parts = a.dq_parts;
  p.status = a.status;
  CUtensorMap tk, tv, tkr, tvr;
  memset(&tk, 0, sizeof(tk));
  memset(&tv, 0, sizeof(tv));
  // K and V chunks alike: [128 keys x 128 columns] (two column blocks)
  if (g.P > 0 && (!encode_pool_tile_map(&tk, a.k_pool, p.pool_rows, L::BN, 2) ||
                  !encode_pool_tile_map(&tv, a.v_pool, p.pool_rows, L::BN, 2)))
    return cudaErrorInvalidValue;
  if (!encode_rows_tile_map(&tkr, a.k_resp, g.hkv, g.R, L::BN, 2) ||
      !encode_rows_tile_map(&tvr, a.v_resp, g.hkv, g.R, L::BN, 2))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(tc_bwd_dq_ring_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::kSmem);
  if (e != cudaSuccess) return e;
  const int64_t units = (int64_t)launch_parts(g) * g.hkv * p.n_mt;
  if (units == 0) return cudaSuccess;
  LaunchScope ls(kKTcBwdDq, s);
  tc_bwd_dq_ring_kernel<<<(unsigned)units, kThreadsRing, L::kSmem, s>>>(tk, tv, tkr, tvr, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tc_bwd_dq(const BwdParams& a, cudaStream_t s) { return bwd_ring(a, s); }

}  // namespace ls
