// Gated-DeltaNet replay forward in chunkwise form on the tensor cores.
//
// The recurrence (see ls_gdn.cu) is rewritten per chunk of C = 128 tokens.
// With c_t the running sum of the log-decays inside the chunk, gamma_t =
// exp(c_t), Gamma_ts = exp(c_t - c_s) and S the state at the chunk's start:
//   A = strict_lower(diag(b) (Gamma . K K^T))        [C x C]
//   U = diag(b) (V - diag(gamma) K S^T)             [C x dv]
//   E = (I + A)^-1 U                                 (unit lower-triangular solve)
//   O = diag(gamma) Q S^T + (lower(Gamma) . Q K^T) E
//   S <- gamma_C S + E^T diag(gamma_C / gamma) K
// which is the same rule, exactly, up to rounding.  K K^T, Q K^T, K S^T,
// Q S^T, P E and E^T W are 128 x 128 x 128 products on tcgen05.mma (bf16
// operands, fp32 accumulators in tensor memory); the solve runs on the CUDA
// cores, one thread per column of E.  The state stays in fp32 registers (one
// row per thread) and is rounded to bf16 only as an MMA operand, so this path
// carries bf16-operand rounding: about 4e-3 relative on o and on the final
// state at 4096 tokens.  The per-element decay factors use the fast __expf (a few
// ulp).
//
// One CTA of 128 threads per (head, member).  Thread r is token row r of the
// chunk (tensor-memory lane r) in the epilogues, state row r for the state,
// and column r of E in the solve.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>

#include "ls_internal.h"
#include "ls_tc.cuh"

namespace ls {
namespace {
using namespace tc;

constexpr int kC = 128;    // tokens per chunk: the MMAs' M
constexpr int kD = 128;    // dk = dv
constexpr int kThr = 128;
constexpr uint32_t kBox = kC * 128;   // [128 rows x 64 bf16] 128B-swizzled box
constexpr uint32_t kTile = 2 * kBox;  // [128 x 128] bf16 tile, K-major, two boxes
constexpr uint32_t kOffK = 0, kOffQ = kTile, kOffS = 2 * kTile, kOffP = 3 * kTile;
constexpr uint32_t kOffEt = 4 * kTile, kOffA = 5 * kTile;
constexpr uint32_t kOffU = kOffQ;  // fp32 [128 x 128] over the Q and S tiles once read
constexpr uint32_t kOffMisc = 6 * kTile;
constexpr uint32_t kSmemBytes = kOffMisc + 2048 + 1024;  // + scalars, barriers, alignment
// tensor-memory columns (fp32, lane = row)
constexpr uint32_t kTmKK = 0, kTmQK = 128, kTmKS = 256, kTmQS = 384;
constexpr uint32_t kTmPE = 0, kTmDS = 128;  // reuse KK and QK once read

__device__ __forceinline__ uint64_t kdesc(uint32_t tile, int kk) {  // K-major, K step kk
  return sdesc_sw128(tile + (kk >> 2) * kBox + (kk & 3) * 32, 16, 1024);
}
__device__ __forceinline__ uint64_t mndesc(uint32_t tile, int kk) {  // N-major B, K rows 16kk..
  return sdesc_sw128(tile + kk * 16 * 128, kBox, 1024);
}
// 16-byte group gq (columns 8gq .. 8gq+7) of row r of a [128 x 128] bf16 tile
__device__ __forceinline__ uint32_t tile_off(int r, int gq) {
  return (gq >> 3) * kBox + sw128_offset(r, gq & 7);
}
// fp32 U / E buffer: row t, column j, columns XOR-swizzled by the row so that
// row writes (one thread per row) and column reads (one thread per column)
// are both free of bank conflicts
__device__ __forceinline__ int u_at(int t, int j) { return t * kD + (j ^ (t & 31)); }
// packed strict lower triangle of A
__device__ __forceinline__ int a_at(int t, int s) { return t * (t - 1) / 2 + s; }

__device__ __forceinline__ uint4 pack8(const float* x) {
  return make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]),
                    pack_bf16x2(x[6], x[7]));
}

__global__ void __launch_bounds__(kThr, 1)
    gdn_chunk_fwd_kernel(int H, int R, const float* __restrict__ s0, const float* __restrict__ q,
                         const float* __restrict__ k, const float* __restrict__ v,
                         const float* __restrict__ g, const float* __restrict__ beta,
                         float* __restrict__ o, float* __restrict__ s_final,
                         uint32_t* __restrict__ fault) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(sm);
  float* sA = reinterpret_cast<float*>(sm + kOffA);
  float* sU = reinterpret_cast<float*>(sm + kOffU);
  float* sc = reinterpret_cast<float*>(sm + kOffMisc);  // c_t
  float* sbt = sc + kC;                                  // b_t
  float* swt = sbt + kC;                                 // per-warp totals of the scan
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffMisc + 1536);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 3);
  uint32_t* abort_s = tslot + 1;

  const int h = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  {  // member blockIdx.y
    const int64_t tok = (int64_t)blockIdx.y * R * H;
    q += tok * kD, k += tok * kD, v += tok * kD, o += tok * kD, g += tok, beta += tok;
    if (s_final) s_final += (int64_t)blockIdx.y * H * kD * kD;
  }
  if (tid == 0) {
    for (int i = 0; i < 3; ++i) mbar_init(smem_u32(&bars[i]), 1);
    *abort_s = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tslot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = *tslot;
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
  const volatile uint32_t* abortp = abort_s;

  float S[kD];  // state row tid, fp32
  {
    const float* src = s0 + ((int64_t)h * kD + tid) * kD;
#pragma unroll
    for (int c = 0; c < kD; ++c) S[c] = src[c];
  }

  const int nch = (R + kC - 1) / kC;
  bool ok = true;
  uint32_t issued = 0;  // MMA groups committed by thread 0
  for (int ch = 0; ch < nch; ++ch) {
    const int t0 = ch * kC, nt = R - t0 < kC ? R - t0 : kC;
    // ---- stage K and Q (bf16, zero rows past the response), S (bf16), b, c
#pragma unroll 4
    for (int it = 0; it < 16; ++it) {
      const int item = tid + kThr * it, r = item >> 4, gq = item & 15;
      uint4 kb = make_uint4(0, 0, 0, 0), qb = kb;
      if (r < nt) {
        const int64_t e = ((int64_t)(t0 + r) * H + h) * kD + gq * 8;
        const float4 k0 = *reinterpret_cast<const float4*>(k + e);
        const float4 k1 = *reinterpret_cast<const float4*>(k + e + 4);
        const float4 q0 = *reinterpret_cast<const float4*>(q + e);
        const float4 q1 = *reinterpret_cast<const float4*>(q + e + 4);
        const float kf[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
        const float qf[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        kb = pack8(kf);
        qb = pack8(qf);
      }
      st_shared_v4(sb + kOffK + tile_off(r, gq), kb);
      st_shared_v4(sb + kOffQ + tile_off(r, gq), qb);
    }
#pragma unroll
    for (int gq = 0; gq < 16; ++gq) st_shared_v4(sb + kOffS + tile_off(tid, gq), pack8(&S[8 * gq]));
    float x = 0.f;
    if (tid < nt) {
      x = g[(int64_t)(t0 + tid) * H + h];
      sbt[tid] = beta[(int64_t)(t0 + tid) * H + h];
    } else {
      sbt[tid] = 0.f;
    }
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += y;
    }
    if (lane == 31) swt[warp] = x;
    __syncthreads();
    for (int w = 0; w < warp; ++w) x += swt[w];
    sc[tid] = x;
    fence_proxy_async_smem();
    __syncthreads();

    // ---- K K^T, Q K^T, K S^T, Q S^T
    if (tid == 0) {
      tc_fence_after();
      constexpr uint32_t id = idesc_bf16(128, 128, false);
#pragma unroll
      for (int kk = 0; kk < kD / 16; ++kk) {
        const uint32_t acc = kk > 0 ? 1u : 0u;
        mma_ss(tb + kTmKK, kdesc(sb + kOffK, kk), kdesc(sb + kOffK, kk), id, acc);
        mma_ss(tb + kTmQK, kdesc(sb + kOffQ, kk), kdesc(sb + kOffK, kk), id, acc);
        mma_ss(tb + kTmKS, kdesc(sb + kOffK, kk), kdesc(sb + kOffS, kk), id, acc);
        mma_ss(tb + kTmQS, kdesc(sb + kOffQ, kk), kdesc(sb + kOffS, kk), id, acc);
      }
      mma_commit(smem_u32(&bars[0]));
      ++issued;
    }
    if (!mbar_wait_warp(smem_u32(&bars[0]), ch & 1, abortp)) ok = false;
    if (__syncthreads_or(!ok)) {
      ok = false;
      break;
    }
    tc_fence_after();

    // ---- epilogue 1, thread r = token row r: A, P, U
    const int r = tid;
    const float cr = sc[r], br = sbt[r], gr = expf(cr);
#pragma unroll 1
    for (int cb = 0; cb < 4; ++cb) {
      uint32_t t32[32];  // one 32-column block at a time keeps the state in registers
      tmem_ld32(tb + lane_off + kTmKK + cb * 32, t32);
      tmem_wait_ld_r(t32);
#pragma unroll
      for (int xx = 0; xx < 32; ++xx) {
        const int s = cb * 32 + xx;
        if (s < r) sA[a_at(r, s)] = br * __expf(cr - sc[s]) * __uint_as_float(t32[xx]);
      }
      tmem_ld32(tb + lane_off + kTmQK + cb * 32, t32);
      tmem_wait_ld_r(t32);
      float pv[32];
#pragma unroll
      for (int xx = 0; xx < 32; ++xx) {
        const int s = cb * 32 + xx;
        pv[xx] = s <= r ? __expf(cr - sc[s]) * __uint_as_float(t32[xx]) : 0.f;
      }
#pragma unroll
      for (int gg = 0; gg < 4; ++gg)
        st_shared_v4(sb + kOffP + tile_off(r, cb * 4 + gg), pack8(&pv[8 * gg]));
      float vr[32];
      if (r < nt) {
        const float4* vp =
            reinterpret_cast<const float4*>(v + ((int64_t)(t0 + r) * H + h) * kD + cb * 32);
#pragma unroll
        for (int i4 = 0; i4 < 8; ++i4) {
          const float4 a = vp[i4];
          vr[4 * i4] = a.x, vr[4 * i4 + 1] = a.y, vr[4 * i4 + 2] = a.z, vr[4 * i4 + 3] = a.w;
        }
      } else {
#pragma unroll
        for (int xx = 0; xx < 32; ++xx) vr[xx] = 0.f;
      }
      tmem_ld32(tb + lane_off + kTmKS + cb * 32, t32);
      tmem_wait_ld_r(t32);
#pragma unroll
      for (int xx = 0; xx < 32; ++xx)
        sU[u_at(r, cb * 32 + xx)] = br * (vr[xx] - gr * __uint_as_float(t32[xx]));
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- solve (I + A) E = U, thread j = column j, eight rows at a time
    {
      const int j = tid, nt8 = (nt + 7) & ~7;
      for (int t8 = 0; t8 < nt8; t8 += 8) {
        float acc[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) acc[u] = sU[u_at(t8 + u, j)];
        for (int s = 0; s < t8; ++s) {
          const float e = sU[u_at(s, j)];
#pragma unroll
          for (int u = 0; u < 8; ++u) acc[u] = fmaf(-sA[a_at(t8 + u, s)], e, acc[u]);
        }
#pragma unroll
        for (int u = 1; u < 8; ++u)
#pragma unroll
          for (int u2 = 0; u2 < u; ++u2) acc[u] = fmaf(-sA[a_at(t8 + u, t8 + u2)], acc[u2], acc[u]);
#pragma unroll
        for (int u = 0; u < 8; ++u) sU[u_at(t8 + u, j)] = acc[u];
      }
      // E^T row j (K-major over tokens): B operand of P E and A operand of E^T W
#pragma unroll 4
      for (int gq = 0; gq < 16; ++gq) {
        float e8[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) e8[u] = sU[u_at(8 * gq + u, j)];
        st_shared_v4(sb + kOffEt + tile_off(j, gq), pack8(e8));
      }
      // W = diag(gamma_C / gamma) K, token row j scaled in place
      const float wj = expf(sc[kC - 1] - sc[j]);
#pragma unroll 4
      for (int gq = 0; gq < 16; ++gq) {
        const uint32_t ad = sb + kOffK + tile_off(j, gq);
        const uint4 kb = ld_shared_v4(ad);
        const uint32_t w4[4] = {kb.x, kb.y, kb.z, kb.w};
        float f8[8];
#pragma unroll
        for (int i2 = 0; i2 < 4; ++i2) {
          const float2 f = unpack_bf16x2(w4[i2]);
          f8[2 * i2] = f.x * wj, f8[2 * i2 + 1] = f.y * wj;
        }
        st_shared_v4(ad, pack8(f8));
      }
    }
    fence_proxy_async_smem();
    __syncthreads();

    // ---- P E and E^T W
    if (tid == 0) {
      tc_fence_after();
      constexpr uint32_t id_k = idesc_bf16(128, 128, false);
      constexpr uint32_t id_mn = idesc_bf16(128, 128, true);
#pragma unroll
      for (int kk = 0; kk < kC / 16; ++kk) {
        const uint32_t acc = kk > 0 ? 1u : 0u;
        mma_ss(tb + kTmPE, kdesc(sb + kOffP, kk), kdesc(sb + kOffEt, kk), id_k, acc);
        mma_ss(tb + kTmDS, kdesc(sb + kOffEt, kk), mndesc(sb + kOffK, kk), id_mn, acc);
      }
      mma_commit(smem_u32(&bars[1]));
      ++issued;
    }
    if (!mbar_wait_warp(smem_u32(&bars[1]), ch & 1, abortp)) ok = false;
    if (__syncthreads_or(!ok)) {
      ok = false;
      break;
    }
    tc_fence_after();

    // ---- epilogue 2: o rows, and the state S <- gamma_C S + E^T W (row tid)
    const float gl = expf(sc[kC - 1]);
#pragma unroll
    for (int cb = 0; cb < 4; ++cb) {
      uint32_t a32[32], b32[32];
      tmem_ld32(tb + lane_off + kTmQS + cb * 32, a32);
      tmem_ld32(tb + lane_off + kTmPE + cb * 32, b32);
      tmem_wait_ld_r(a32);
      reg_dep(b32);
      if (r < nt) {
        float4* op = reinterpret_cast<float4*>(o + ((int64_t)(t0 + r) * H + h) * kD + cb * 32);
#pragma unroll
        for (int i4 = 0; i4 < 8; ++i4)
          op[i4] = make_float4(fmaf(gr, __uint_as_float(a32[4 * i4]), __uint_as_float(b32[4 * i4])),
                               fmaf(gr, __uint_as_float(a32[4 * i4 + 1]), __uint_as_float(b32[4 * i4 + 1])),
                               fmaf(gr, __uint_as_float(a32[4 * i4 + 2]), __uint_as_float(b32[4 * i4 + 2])),
                               fmaf(gr, __uint_as_float(a32[4 * i4 + 3]), __uint_as_float(b32[4 * i4 + 3])));
      }
      tmem_ld32(tb + lane_off + kTmDS + cb * 32, a32);
      tmem_wait_ld_r(a32);
#pragma unroll
      for (int xx = 0; xx < 32; ++xx) S[cb * 32 + xx] = fmaf(gl, S[cb * 32 + xx], __uint_as_float(a32[xx]));
    }
    tc_fence_before();
    __syncthreads();
  }

  if (!ok) {  // a wait gave up: mark the results so that no caller takes them for data
    if (tid == 0 && fault) atomicExch(fault, 1u);
    for (int t = 0; t < R; ++t) o[((int64_t)t * H + h) * kD + tid] = __int_as_float(0x7fc00000);
    if (s_final)
      for (int c = 0; c < kD; ++c) s_final[((int64_t)h * kD + tid) * kD + c] = __int_as_float(0x7fc00000);
  } else if (s_final) {
    float* dst = s_final + ((int64_t)h * kD + tid) * kD;
#pragma unroll
    for (int c = 0; c < kD; ++c) dst[c] = S[c];
  }
  // drain: every MMA issued above is complete before tensor memory is freed
  if (tid == 0 && issued > 0) {
    mma_commit(smem_u32(&bars[2]));
    mbar_wait(smem_u32(&bars[2]), 0, abortp);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tb, 512);
  }
}

}  // namespace

cudaError_t launch_gdn_chunk_fwd(int B, int H, int R, const float* s0, const float* q,
                                 const float* k, const float* v, const float* g, const float* beta,
                                 float* o, float* s_final, cudaStream_t st) {
  if (B == 0 || H == 0) return cudaSuccess;
  for (const void* p : {(const void*)q, (const void*)k, (const void*)v, (const void*)o})
    if (R > 0 && (reinterpret_cast<uintptr_t>(p) & 15u)) return cudaErrorMisalignedAddress;
  cudaError_t e = cudaFuncSetAttribute(gdn_chunk_fwd_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  LaunchScope ls(kKGdnFwd, st);
  gdn_chunk_fwd_kernel<<<dim3(H, B), kThr, kSmemBytes, st>>>(H, R, s0, q, k, v, g, beta, o, s_final,
                                                             nullptr);
  return cudaGetLastError();
}

}  // namespace ls
