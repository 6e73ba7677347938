// Tensor-core (tcgen05/TMEM) response dK/dV for bf16, head dim 256.
//
// Only response keys get K/V gradients; prompt K/V are stop-gradient
// (LongStraw DeepRead summary, section Method, last paragraph).  The kernel
// is key-stationary: a CTA owns (KV head g, a tile of 128 response keys j0..,
// one half of the head dimension) and walks the query rows that see those
// keys (rows r >= j0 of the Gq query heads of g), 64 rows at a time.
//
// With TMEM lanes = keys:
//   S^T  = K Q^T                      (SS)  -> TMEM
//   dP^T = V dO^T                     (SS)  -> TMEM
//   softmax warps: P^T = exp2(S^T*scale*log2e - LSE*log2e) and
//                  dS^T = P^T (dP^T - delta), both written back as bf16
//   dV[:, half] += P^T  dO[:, half]   (A from TMEM, dO as N-major B)
//   dK[:, half] += dS^T Q[:, half]    (A from TMEM, Q as N-major B)
// The two halves of d run in different CTAs so that dK, dV (128 columns each)
// and S^T, dP^T fit in tensor memory; S^T/dP^T are recomputed per half, which
// costs 1.5x the minimal flops on a part that is a small fraction of the
// replay.  dK is scaled by the softmax scale in the epilogue.
#include <cuda.h>
#include <cuda_bf16.h>
#include <math_constants.h>

#include <cstring>

#include "ls_internal.h"
#include "ls_tc.cuh"

namespace ls {
namespace {
using namespace tc;

constexpr int kD = 256;
constexpr int kBK = 128;  // keys per CTA (TMEM lanes)
constexpr int kBR = 64;   // query rows per step
constexpr int kThreads = 256;
constexpr float kLog2ef = 1.4426950408889634f;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct Layout {
  static constexpr uint32_t kKBox = kBK * 128;   // [128 x 64] box, 16 KB
  static constexpr uint32_t kRBox = kBR * 128;   // [64 x 64] box, 8 KB
  static constexpr uint32_t kK = 0;
  static constexpr uint32_t kV = kK + 4 * kKBox;
  static constexpr uint32_t kQ = kV + 4 * kKBox;
  static constexpr uint32_t kO = kQ + 4 * kRBox;
  static constexpr uint32_t kEnd = kO + 4 * kRBox;
  static constexpr uint32_t kSmem = kEnd + 1024;
  static constexpr uint32_t kTmemDK = 0, kTmemDV = 128, kTmemS = 256, kTmemP = 320;
};

struct DkdvKParams {
  int32_t hq, hkv, gq, R;
  int32_t n_kt;
  float scale, scale_log2;
  const float* lse;
  const float* delta;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  uint32_t* status;
};

__global__ void __launch_bounds__(kThreads, 1)
    tc_dkdv_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmO,
                   const DkdvKParams p) {
  using L = Layout;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_kv, bar_qf, bar_qe, bar_sd, bar_ds, bar_fin, bar_drain, bar_st[2];
  __shared__ uint32_t tmem_base_s, abort_s;
  __shared__ float s_lse[2][kBR], s_dl[2][kBR];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sK = sbase + L::kK, sV = sbase + L::kV, sQ = sbase + L::kQ, sO = sbase + L::kO;

  const int hf = blockIdx.x & 1;
  const int kt = (blockIdx.x >> 1) % p.n_kt;
  const int g = (blockIdx.x >> 1) / p.n_kt;
  const int j0 = kt * kBK;
  const int nrt = (p.R - j0 + kBR - 1) / kBR;  // row tiles per head (rows >= j0)
  const int nit = p.gq * nrt;

  if (tid == 0) {
    abort_s = 0;
    mbar_init(smem_u32(&bar_kv), 1);
    mbar_init(smem_u32(&bar_qf), 1);
    mbar_init(smem_u32(&bar_qe), 1);
    mbar_init(smem_u32(&bar_sd), 1);
    mbar_init(smem_u32(&bar_ds), 128);
    mbar_init(smem_u32(&bar_fin), 1);
    mbar_init(smem_u32(&bar_drain), 1);
    mbar_init(smem_u32(&bar_st[0]), 128);
    mbar_init(smem_u32(&bar_st[1]), 128);
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
  // a wait that gives up records its kernel and source line in status[1]
  auto fail = [&](int line) {
    atomicOr(p.status, kStatusTimeout);
    atomicCAS(p.status + 1, 0u, ((uint32_t)kKTcDkDv << 16) | (uint32_t)line);
    abort_s = 1;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && nit > 0) {
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmQ);
      const uint32_t bkv = smem_u32(&bar_kv);
      mbar_expect_tx(bkv, 8 * L::kKBox);
      for (int c = 0; c < 4; ++c) {
        tma_load_3d(sK + c * L::kKBox, &tmK, bkv, c * 64, g, j0);
        tma_load_3d(sV + c * L::kKBox, &tmV, bkv, c * 64, g, j0);
      }
      int issued = 0;
      for (int it = 0; it < nit; ++it) {
        if (it > 0 && !mbar_wait(smem_u32(&bar_qe), (it - 1) & 1, abortp)) { fail(__LINE__); break; }
        const int h = g * p.gq + it / nrt;
        const int r0 = j0 + (it % nrt) * kBR;
        const uint32_t bq = smem_u32(&bar_qf);
        mbar_expect_tx(bq, 8 * L::kRBox);
        for (int c = 0; c < 4; ++c) {
          tma_load_3d(sQ + c * L::kRBox, &tmQ, bq, c * 64, h, r0);
          tma_load_3d(sO + c * L::kRBox, &tmO, bq, c * 64, h, r0);
        }
        issued = it + 1;
      }
      // no copy may still be landing in shared memory when the CTA ends
      mbar_wait(bkv, 0, abortp);
      if (issued > 0) mbar_wait(smem_u32(&bar_qf), (issued - 1) & 1, abortp);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && nit > 0) {
      constexpr uint32_t idesc_s = idesc_bf16(kBK, kBR, false);
      constexpr uint32_t idesc_g = idesc_bf16(kBK, 128, true);
      bool ok = mbar_wait(smem_u32(&bar_kv), 0, abortp);
      if (!ok) fail(__LINE__);
      for (int it = 0; ok && it < nit; ++it) {
        if (!mbar_wait(smem_u32(&bar_qf), it & 1, abortp)) { fail(__LINE__); break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t ko = (kk >> 2) * L::kKBox + (kk & 3) * 32;
          const uint32_t ro = (kk >> 2) * L::kRBox + (kk & 3) * 32;
          mma_ss(tbase + L::kTmemS, sdesc_sw128(sK + ko, 16, 1024), sdesc_sw128(sQ + ro, 16, 1024),
                 idesc_s, kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t ko = (kk >> 2) * L::kKBox + (kk & 3) * 32;
          const uint32_t ro = (kk >> 2) * L::kRBox + (kk & 3) * 32;
          mma_ss(tbase + L::kTmemP, sdesc_sw128(sV + ko, 16, 1024), sdesc_sw128(sO + ro, 16, 1024),
                 idesc_s, kk > 0 ? 1u : 0u);
        }
        mma_commit(smem_u32(&bar_sd));
        if (!mbar_wait(smem_u32(&bar_ds), it & 1, abortp)) { fail(__LINE__); break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kBR / 16; ++kk) {
          const uint32_t acc = (it > 0 || kk > 0) ? 1u : 0u;
          const uint32_t bo = (2 * hf) * L::kRBox + kk * 16 * 128;
          mma_ts(tbase + L::kTmemDV, tbase + L::kTmemS + kk * 8,
                 sdesc_sw128(sO + bo, L::kRBox, 1024), idesc_g, acc);
          mma_ts(tbase + L::kTmemDK, tbase + L::kTmemP + kk * 8,
                 sdesc_sw128(sQ + bo, L::kRBox, 1024), idesc_g, acc);
        }
        mma_commit(smem_u32(&bar_qe));
        if (it == nit - 1) mma_commit(smem_u32(&bar_fin));
      }
      mma_commit(smem_u32(&bar_drain));
      mbar_wait(smem_u32(&bar_drain), 0, abortp);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int i = tid - 128;  // key in the tile == TMEM lane
    const int j = j0 + i;
    const uint32_t lane_off = (uint32_t)((warp - 4) * 32) << 16;
    bool ok = true;
    for (int it = 0; it < nit; ++it) {
      const int h = g * p.gq + it / nrt;
      const int r0 = j0 + (it % nrt) * kBR;
      const int b = it & 1;
      // stage LSE*log2e and delta of the step's rows (double-buffered; buffer
      // b is rewritten two steps later, after every thread arrived at the
      // step in between, i.e. after every thread finished reading it)
      if (i < kBR) {
        const int r = r0 + i;
        s_lse[b][i] = r < p.R ? __ldg(p.lse + (int64_t)r * p.hq + h) * kLog2ef : 0.f;
      } else {
        const int r = r0 + i - kBR;
        s_dl[b][i - kBR] = r < p.R ? __ldg(p.delta + (int64_t)r * p.hq + h) : 0.f;
      }
      mbar_arrive(smem_u32(&bar_st[b]));
      if (!mbar_wait_warp(smem_u32(&bar_st[b]), (it >> 1) & 1, abortp)) { fail(__LINE__); ok = false; break; }
      if (!mbar_wait_warp(smem_u32(&bar_sd), it & 1, abortp)) { fail(__LINE__); ok = false; break; }
      tc_fence_after();
      uint32_t pk[kBR / 2], dk[kBR / 2];
#pragma unroll
      for (int c0 = 0; c0 < kBR; c0 += 32) {
        uint32_t rs[32], rp[32];
        tmem_ld32(tbase + lane_off + L::kTmemS + c0, rs);
        tmem_ld32(tbase + lane_off + L::kTmemP + c0, rp);
        tmem_wait_ld_r(rs);
        reg_dep(rp);
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          float pv[2], dv[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int col = c0 + c + u;
            const int r = r0 + col;
            const bool valid = r < p.R && r >= j;
            const float e = ex2(__uint_as_float(rs[c + u]) * p.scale_log2 - s_lse[b][col]);
            pv[u] = valid ? e : 0.f;
            dv[u] = valid ? e * (__uint_as_float(rp[c + u]) - s_dl[b][col]) : 0.f;
          }
          pk[(c0 + c) >> 1] = pack_bf16x2(pv[0], pv[1]);
          dk[(c0 + c) >> 1] = pack_bf16x2(dv[0], dv[1]);
        }
      }
      tmem_st32(tbase + lane_off + L::kTmemS, pk);
      tmem_st32(tbase + lane_off + L::kTmemP, dk);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(smem_u32(&bar_ds));
    }
    // ---- epilogue: rows j < R of dK (scaled) and dV, columns of this half
    if (ok && nit > 0) {
      if (!mbar_wait_warp(smem_u32(&bar_fin), 0, abortp)) { fail(__LINE__); ok = false; }
      tc_fence_after();
    }
    // ok is warp-uniform here; the tensor-memory loads run on the whole warp
    // and only the stores are limited to keys j < R
    if (ok && nit > 0) {
      __nv_bfloat16* dko = p.dk + ((int64_t)j * p.hkv + g) * kD + hf * 128;
      __nv_bfloat16* dvo = p.dv + ((int64_t)j * p.hkv + g) * kD + hf * 128;
#pragma unroll 1
      for (int c0 = 0; c0 < 128; c0 += 32) {
        uint32_t rk[32], rv[32];
        __syncwarp();  // the j < R stores of the previous chunk diverge
        tmem_ld32(tbase + lane_off + L::kTmemDK + c0, rk);
        tmem_ld32(tbase + lane_off + L::kTmemDV + c0, rv);
        tmem_wait_ld_r(rk);
        reg_dep(rv);
        if (j >= p.R) continue;
#pragma unroll
        for (int c = 0; c < 32; c += 8) {
          uint4 vk, vv;
          vk.x = pack_bf16x2(p.scale * __uint_as_float(rk[c]), p.scale * __uint_as_float(rk[c + 1]));
          vk.y = pack_bf16x2(p.scale * __uint_as_float(rk[c + 2]), p.scale * __uint_as_float(rk[c + 3]));
          vk.z = pack_bf16x2(p.scale * __uint_as_float(rk[c + 4]), p.scale * __uint_as_float(rk[c + 5]));
          vk.w = pack_bf16x2(p.scale * __uint_as_float(rk[c + 6]), p.scale * __uint_as_float(rk[c + 7]));
          vv.x = pack_bf16x2(__uint_as_float(rv[c]), __uint_as_float(rv[c + 1]));
          vv.y = pack_bf16x2(__uint_as_float(rv[c + 2]), __uint_as_float(rv[c + 3]));
          vv.z = pack_bf16x2(__uint_as_float(rv[c + 4]), __uint_as_float(rv[c + 5]));
          vv.w = pack_bf16x2(__uint_as_float(rv[c + 6]), __uint_as_float(rv[c + 7]));
          *reinterpret_cast<uint4*>(dko + c0 + c) = vk;
          *reinterpret_cast<uint4*>(dvo + c0 + c) = vv;
        }
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

}  // namespace

cudaError_t launch_tc_dkdv(const BwdParams& a, cudaStream_t s) {
  const AttnGeom& g = a.g;
  if (g.R == 0) return cudaSuccess;
  DkdvKParams p;
  p.hq = g.hq;
  p.hkv = g.hkv;
  p.gq = g.gq;
  p.R = g.R;
  p.n_kt = (g.R + kBK - 1) / kBK;
  p.scale = g.scale;
  p.scale_log2 = g.scale_log2;
  p.lse = a.lse;
  p.delta = a.delta;
  p.dk = reinterpret_cast<__nv_bfloat16*>(a.dk);
  p.dv = reinterpret_cast<__nv_bfloat16*>(a.dv);
  p.status = a.status;
  CUtensorMap tk, tv, tq, to;
  if (!encode_rows_map(&tk, a.k_resp, g.hkv, g.R, kBK) ||
      !encode_rows_map(&tv, a.v_resp, g.hkv, g.R, kBK) ||
      !encode_rows_map(&tq, a.q, g.hq, g.R, kBR) || !encode_rows_map(&to, a.d_o, g.hq, g.R, kBR))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(tc_dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)Layout::kSmem);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)(g.hkv * p.n_kt * 2);
  LaunchScope ls(kKTcDkDv, s);
  tc_dkdv_kernel<<<grid, kThreads, Layout::kSmem, s>>>(tk, tv, tq, to, p);
  return cudaGetLastError();
}

}  // namespace ls
