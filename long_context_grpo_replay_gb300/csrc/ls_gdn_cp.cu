// Gated-DeltaNet replay in chunk-parallel form (forward and backward): the
// recurrent layers of the Qwen path replayed from the captured prompt state
// (LongStraw DeepRead summary, section Method), the gated delta rule of
// ls_gdn.cu rewritten over chunks.
//
// With chunks of C = 128 tokens, per chunk: c_t the running sum of the
// log-decays, gamma_t = exp(c_t), Gamma_ts = exp(c_t - c_s), w_t = gamma_C /
// gamma_t, GK = strict_lower(Gamma . K K^T), A = diag(b) GK, T = (I + A)^-1,
// P = lower(Gamma . Q K^T), W = diag(w) K.  The replay is three stages:
//   prep  (all chunks at once): E0 = T diag(b) V, ZK = T diag(b gamma) K,
//         dU0 = T^T P^T dO, ZW = T^T W         (the only triangular solves)
//   chain (per head and member, over the chunks):
//         state forward   E = E0 - ZK S^T,  S <- gamma_C S + E^T W
//         dL/dS backward  dU = dU0 + ZW G^T, G <- gamma_C G + (gamma dO)^T Q - (gamma b dU)^T K
//   out   (all chunks at once): o = diag(gamma) Q S^T + P E and the gradients
//         of q, k, v, g, b from S, G, E and dU of the chunk.
// The chains carry only two 128 x 128 products per chunk; everything else is
// parallel over chunks.  Products are tcgen05.mma on bf16 operands with fp32
// accumulators; solves and states are fp32.  The per-element decay
// factors exp(c_t - c_s) use the fast __expf (a few ulp), far below the
// bf16 rounding of the products' operands.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ls_gdn_tiles.cuh"
#include "ls_internal.h"

namespace ls {
namespace {
using namespace gdn;

// float32 scratch per (member, head, chunk): the [128 x 128] blocks below,
// then the packed GK.
enum : int { kE0 = 0, kZK, kDU0, kZW, kEblk, kDUblk, kSstart, kGend, kGKblk, kScrBlocks };
constexpr int64_t kScrFloats = (int64_t)kScrBlocks * kTileElems;

__device__ __forceinline__ float* scratch_of(float* scr, int H, int nch, int m, int h, int ch) {
  return scr + (((int64_t)m * H + h) * nch + ch) * kScrFloats;
}

// Cumulative log-decay and write strength of the chunk's tokens into sc[],
// sbt[] (zero past the response); swt[4] is scan scratch.  Called by all
// threads of the block; threads past the chunk's 128 only meet the barrier.
__device__ __forceinline__ void stage_gates(const float* g, const float* beta, int64_t t0, int nt,
                                            int H, int h, float* sc, float* sbt, float* swt) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid >= kThr) {
    __syncthreads();
    return;
  }
  float x = 0.f;
  if (tid < nt) {
    x = g[(t0 + tid) * H + h];
    sbt[tid] = beta[(t0 + tid) * H + h];
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
}

// fp32 [128 x 128] buffer of T with rows of 129 floats: a column read by
// consecutive threads and a row read by a whole warp are both free of bank
// conflicts, with no index arithmetic beyond the row base.
constexpr int kTStride = kC + 1;
__device__ __forceinline__ int b_at(int t, int x) { return t * kTStride + x; }

// Column x of the inverse of the unit lower-triangular diagonal block of
// (I + diag(b) GK) on rows and columns r0 .. r0+63, by forward substitution
// eight rows at a time, into buf (column x, rows r0 .. r0+63; the rows above
// x come out zero).  x lies inside the block.
__device__ __forceinline__ void invert_block64(float* buf, const float* gk, const float* sbt, int r0,
                                               int x) {
  for (int t8 = r0; t8 < r0 + 64; t8 += 8) {
    float sum[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int s = r0; s < t8; ++s) {
      const float e = buf[b_at(s, x)];
#pragma unroll
      for (int u = 0; u < 8; ++u) sum[u] = fmaf(gk[a_at(t8 + u, s)], e, sum[u]);
    }
    float ev[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
#pragma unroll
      for (int u2 = 0; u2 < u; ++u2) sum[u] = fmaf(gk[a_at(t8 + u, t8 + u2)], ev[u2], sum[u]);
      ev[u] = fmaf(-sbt[t8 + u], sum[u], t8 + u == x ? 1.f : 0.f);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) buf[b_at(t8 + u, x)] = ev[u];
  }
}

// ---------------------------------------------------------------- prep
// One CTA per (chunk, head, member), 256 threads in two groups of 128.
// T = (I + diag(b) GK)^-1 is formed explicitly in fp32 by blocks of 64
// rows: each diagonal block by forward substitution (group A, one column per
// thread), the off-diagonal block as T21 = -T22 (diag(b) GK21) T11 by two
// products on the CUDA cores.  The four right-hand sides are then tensor-core
// products with T as the A operand, split into bf16 hi + lo parts (their sum
// is T to about 2^-17):
//   E0 = T (b V), ZK = T (b gamma K)      (the T tile read M-major)
//   dU0 = T^T dE0, ZW = T^T (w K)         (the same tile read K-major)
// Group B stages the right-hand sides while group A forms T.
// Shared memory: R0 K -> b V, R1 Q -> P^T -> b gamma K, R2 dO -> w K,
// R3 GK (packed fp32) -> dE0, R4 + R5 (and 512 bytes more) T (fp32) -> T hi (R4),
// T lo (R5).
constexpr uint32_t kPrepR0 = 0, kPrepR1 = kTile, kPrepR2 = 2 * kTile, kPrepR3 = 3 * kTile;
constexpr uint32_t kPrepR4 = 4 * kTile, kPrepR5 = 5 * kTile;
// T in fp32 (rows of 129 floats) runs 512 bytes past R5
constexpr uint32_t kPrepMisc = 6 * kTile + 1024;
constexpr uint32_t kPrepSmem = kPrepMisc + 3072 + 1024;
static_assert(kPrepR4 + kC * kTStride * 4 <= kPrepMisc, "T buffer overlaps the misc area");
constexpr int kPrepThr = 2 * kThr;

__global__ void __launch_bounds__(kPrepThr, 1)
    gdn_cp_prep_kernel(int H, int R, int nch, const float* __restrict__ q,
                       const float* __restrict__ k, const float* __restrict__ v,
                       const float* __restrict__ g, const float* __restrict__ beta,
                       const float* __restrict__ d_o, float* __restrict__ scr,
                       uint32_t* __restrict__ status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(sm);
  float* gk = reinterpret_cast<float*>(sm + kPrepR3);
  float* buf = reinterpret_cast<float*>(sm + kPrepR4);
  float* sc = reinterpret_cast<float*>(sm + kPrepMisc);
  float* sbt = sc + kC;    // b
  float* sbg = sbt + kC;   // b gamma
  float* swk = sbg + kC;   // w (zero past the response)
  float* swt = swk + kC;   // 8 floats of scan scratch
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kPrepMisc + 2560);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 4);
  uint32_t* abort_s = tslot + 1;

  const int ch = blockIdx.x, h = blockIdx.y, m = blockIdx.z, tid = threadIdx.x, warp = tid >> 5;
  const bool grpA = tid < kThr;
  const int gt = tid & (kThr - 1);  // index within the group: row / column
  const int64_t t0 = (int64_t)ch * kC;
  const int nt = R - t0 < kC ? (int)(R - t0) : kC;
  {
    const int64_t tok = (int64_t)m * R * H;
    q += tok * kD, k += tok * kD, v += tok * kD, d_o += tok * kD, g += tok, beta += tok;
  }
  float* out = scratch_of(scr, H, nch, m, h, ch);
  if (tid == 0) {
    for (int i = 0; i < 4; ++i) mbar_init(smem_u32(&bars[i]), 1);
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
  const uint32_t tb = *tslot, lane_off = (uint32_t)((warp & 3) * 32) << 16;
  const volatile uint32_t* abortp = abort_s;
  const int64_t rs = (int64_t)H * kD;  // token stride of q, k, v, d_o
  const int64_t row0 = (t0 * H + h) * kD;

  if (grpA) {
    stage_rows<4>(sb + kPrepR0, k + row0, rs, nt, nullptr, gt);
    stage_rows<4>(sb + kPrepR1, q + row0, rs, nt, nullptr, gt);
  } else {
    stage_rows<4>(sb + kPrepR2, d_o + row0, rs, nt, nullptr, gt);
  }
  stage_gates(g, beta, t0, nt, H, h, sc, sbt, swt);
  fence_proxy_async_smem();
  __syncthreads();
  if (!grpA) {  // the right-hand sides' row scales (read after the next block barrier)
    const float ct = sc[gt], clast = sc[kC - 1];
    sbg[gt] = sbt[gt] * __expf(ct);
    swk[gt] = gt < nt ? __expf(clast - ct) : 0.f;
  }

  if (tid == 0) {  // K K^T -> cols 0..127, K Q^T -> 128..255
    tc_fence_after();
    mma_group(tb + 0, sb + kPrepR0, sb + kPrepR0, false, false);
    mma_group(tb + 128, sb + kPrepR0, sb + kPrepR1, false, false);
    mma_commit(smem_u32(&bars[0]));
  }
  bool ok = mbar_wait_warp(smem_u32(&bars[0]), 0, abortp);
  if (!__syncthreads_or(!ok)) {
    tc_fence_after();
    if (grpA) {
      // thread r: GK row r (s < r); P^T row r: P^T[r][t] = [t >= r] Gamma_tr (K_r . Q_t)
      const int r = gt;
      const float cr = sc[r];
      float* gko = out + (int64_t)kGKblk * kTileElems;
#pragma unroll 1
      for (int cb = 0; cb < 4; ++cb) {
        uint32_t t32[32];
        tmem_ld32(tb + lane_off + 0 + cb * 32, t32);
        tmem_wait_ld_r(t32);
#pragma unroll
        for (int xx = 0; xx < 32; ++xx) {
          const int s = cb * 32 + xx;
          if (s < r) {
            const float val = __expf(cr - sc[s]) * __uint_as_float(t32[xx]);
            gk[a_at(r, s)] = val;
            gko[a_at(r, s)] = val;
          }
        }
        tmem_ld32(tb + lane_off + 128 + cb * 32, t32);
        tmem_wait_ld_r(t32);
        float pv[32];
#pragma unroll
        for (int xx = 0; xx < 32; ++xx) {
          const int t = cb * 32 + xx;
          pv[xx] = t >= r ? __expf(sc[t] - cr) * __uint_as_float(t32[xx]) : 0.f;
        }
#pragma unroll
        for (int gg = 0; gg < 4; ++gg) st_shared_v4(sb + kPrepR1 + tile_off(r, cb * 4 + gg), pack8(&pv[8 * gg]));
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {  // dE0 = P^T dO -> cols 256..383 (dO as an N-major B)
      tc_fence_after();
      mma_group(tb + 256, sb + kPrepR1, sb + kPrepR2, true, false);
      mma_commit(smem_u32(&bars[1]));
    }
    if (grpA) {
      // ---- T by blocks of 64 rows.  Column x: T11 (x < 64) or T22 (x >= 64)
      // by substitution; the rest of the column zero.
      const int x = gt, r0 = x & 64;
      for (int t = 0; t < kC; ++t)
        if (t < r0 || t >= r0 + 64) buf[b_at(t, x)] = 0.f;
      invert_block64(buf, gk, sbt, r0, x);
      named_bar_sync(1, kThr);
      // thread (xc, hf) owns column xc of the off-diagonal block, rows
      // 64 + 32 hf .. 64 + 32 hf + 31
      const int xc = x & 63, hf = x >> 6;
      {  // Y = diag(b) GK21 T11 into the block's place (T11 does not read it)
        float tcol[64];
#pragma unroll
        for (int s = 0; s < 64; ++s) tcol[s] = buf[b_at(s, xc)];
#pragma unroll 1
        for (int j = 0; j < 32; ++j) {
          const int t = 64 + 32 * hf + j;
          const float* gr = gk + a_at(t, 0);
          float p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
#pragma unroll
          for (int s = 0; s < 64; s += 4) {
            p0 = fmaf(gr[s], tcol[s], p0);
            p1 = fmaf(gr[s + 1], tcol[s + 1], p1);
            p2 = fmaf(gr[s + 2], tcol[s + 2], p2);
            p3 = fmaf(gr[s + 3], tcol[s + 3], p3);
          }
          buf[b_at(t, xc)] = sbt[t] * ((p0 + p1) + (p2 + p3));
        }
      }
      named_bar_sync(1, kThr);
      {  // T21 = -T22 Y (T22 stored with its zero upper triangle and unit diagonal)
        float ycol[64];
#pragma unroll
        for (int s = 0; s < 64; ++s) ycol[s] = buf[b_at(64 + s, xc)];
        named_bar_sync(1, kThr);  // Y read everywhere before T21 overwrites it
#pragma unroll 1
        for (int j = 0; j < 32; ++j) {
          const int t = 64 + 32 * hf + j;
          const float* tr = buf + b_at(t, 64);
          float p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
#pragma unroll
          for (int s = 0; s < 64; s += 4) {
            p0 = fmaf(tr[s], ycol[s], p0);
            p1 = fmaf(tr[s + 1], ycol[s + 1], p1);
            p2 = fmaf(tr[s + 2], ycol[s + 2], p2);
            p3 = fmaf(tr[s + 3], ycol[s + 3], p3);
          }
          buf[b_at(t, xc)] = -((p0 + p1) + (p2 + p3));
        }
      }
    } else {
      // ---- group B: the right-hand sides, once P^T dO has read R1 and R2
      ok = mbar_wait_warp(smem_u32(&bars[1]), 0, abortp);
      if (ok) {
        stage_rows<4>(sb + kPrepR0, v + row0, rs, nt, sbt, gt);  // b V
        stage_rows<4>(sb + kPrepR1, k + row0, rs, nt, sbg, gt);  // b gamma K
        stage_rows<4>(sb + kPrepR2, k + row0, rs, nt, swk, gt);  // w K
      }
    }
    if (!__syncthreads_or(!ok)) {
      float tcol[kC];
      if (grpA) {
#pragma unroll
        for (int t = 0; t < kC; ++t) tcol[t] = buf[b_at(t, gt)];
      } else {
        // dE0 rows (bf16) over GK, which the substitution no longer needs
        tc_fence_after();
#pragma unroll 1
        for (int cb = 0; cb < 4; ++cb) {
          uint32_t t32[32];
          tmem_ld32(tb + lane_off + 256 + cb * 32, t32);
          tmem_wait_ld_r(t32);
          float f32[32];
#pragma unroll
          for (int xx = 0; xx < 32; ++xx) f32[xx] = __uint_as_float(t32[xx]);
#pragma unroll
          for (int gg = 0; gg < 4; ++gg) st_shared_v4(sb + kPrepR3 + tile_off(gt, cb * 4 + gg), pack8(&f32[8 * gg]));
        }
      }
      __syncthreads();  // T read from R4 / R5 before its bf16 halves overwrite them
      if (grpA) {  // row x of the hi and lo tiles = column x of T
#pragma unroll
        for (int gq = 0; gq < 16; ++gq) {
          float hi[8], lo[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const uint16_t hb = bf16_of(tcol[8 * gq + u]);
            hi[u] = __uint_as_float((uint32_t)hb << 16);
            lo[u] = tcol[8 * gq + u] - hi[u];
          }
          st_shared_v4(sb + kPrepR4 + tile_off(gt, gq), pack8(hi));
          st_shared_v4(sb + kPrepR5 + tile_off(gt, gq), pack8(lo));
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();
      if (tid == 0) {
        tc_fence_after();
        const uint32_t th = sb + kPrepR4, tl = sb + kPrepR5;
        mma_group_amn(tb + 0, th, sb + kPrepR0, true, false);    // E0 = T (b V)
        mma_group_amn(tb + 0, tl, sb + kPrepR0, true, true);
        mma_group_amn(tb + 128, th, sb + kPrepR1, true, false);  // ZK = T (b gamma K)
        mma_group_amn(tb + 128, tl, sb + kPrepR1, true, true);
        mma_group(tb + 256, th, sb + kPrepR3, true, false);      // dU0 = T^T dE0
        mma_group(tb + 256, tl, sb + kPrepR3, true, true);
        mma_group(tb + 384, th, sb + kPrepR2, true, false);      // ZW = T^T (w K)
        mma_group(tb + 384, tl, sb + kPrepR2, true, true);
        mma_commit(smem_u32(&bars[2]));
      }
      ok = mbar_wait_warp(smem_u32(&bars[2]), 0, abortp);
      if (!__syncthreads_or(!ok)) {
        // warps 0-3: E0 and ZK (columns 0..255); warps 4-7: dU0 and ZW
        tc_fence_after();
        float* wscr = reinterpret_cast<float*>(sm + kPrepR0) + warp * 32 * 33;
        const int r0w = (warp & 3) * 32;
#pragma unroll 1
        for (int bi = 0; bi < 2; ++bi) {
          const int blkid = grpA ? (bi == 0 ? kE0 : kZK) : (bi == 0 ? kDU0 : kZW);
          const uint32_t col = (grpA ? 0 : 256) + bi * 128;
          float* dst = out + (int64_t)blkid * kTileElems + r0w * kD;
#pragma unroll 1
          for (int cb = 0; cb < 4; ++cb) {
            uint32_t t32[32];
            tmem_ld32(tb + lane_off + col + cb * 32, t32);
            tmem_wait_ld_r(t32);
            float f32[32];
#pragma unroll
            for (int xx = 0; xx < 32; ++xx) f32[xx] = __uint_as_float(t32[xx]);
            rows_store32(f32, dst + cb * 32, kD, 32, wscr);
          }
        }
      }
    }
  }
  if (__syncthreads_or(!ok) && tid == 0 && status) atomicOr(status, kStatusTimeout);
  if (tid == 0) {  // drain before tensor memory is freed
    mma_commit(smem_u32(&bars[3]));
    mbar_wait(smem_u32(&bars[3]), 0, abortp);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tb, 512);
  }
}

// ---------------------------------------------------------------- chain
// One CTA per (head, member), sequential over the chunks: the state forward,
// then dL/dS backward.  Per chunk it writes S at the chunk's start, G at its
// end, E and dU into the scratch.
constexpr uint32_t kChT0 = 0, kChT1 = kTile, kChT2 = 2 * kTile, kChT3 = 3 * kTile;
constexpr uint32_t kChT4 = 4 * kTile, kChT5 = 5 * kTile, kChMisc = 6 * kTile;
constexpr uint32_t kChainSmem = kChMisc + 2048 + 1024;

__global__ void __launch_bounds__(kThr, 1)
    gdn_cp_chain_kernel(int H, int R, int nch, const float* __restrict__ s0,
                        const float* __restrict__ q, const float* __restrict__ k,
                        const float* __restrict__ g, const float* __restrict__ beta,
                        const float* __restrict__ d_o, float* __restrict__ scr,
                        float* __restrict__ s_final, uint32_t* __restrict__ status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(sm);
  float* sc = reinterpret_cast<float*>(sm + kChMisc);
  float* sbt = sc + kC;
  float* swt = sbt + kC;
  float* sw = swt + 4;  // w_t (state pass) or gamma_t (gradient pass), zero past the response
  // the barriers sit past sw (which ends at byte 1552 of the misc area)
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kChMisc + 1600);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 3);
  uint32_t* abort_s = tslot + 1;

  const int h = blockIdx.x, m = blockIdx.y, tid = threadIdx.x, warp = tid >> 5;
  {
    const int64_t tok = (int64_t)m * R * H;
    q += tok * kD, k += tok * kD, d_o += tok * kD, g += tok, beta += tok;
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
  const uint32_t tb = *tslot, lane_off = (uint32_t)(warp * 32) << 16;
  const volatile uint32_t* abortp = abort_s;
  const int64_t rs = (int64_t)H * kD;
  const int x = tid;  // state row i / token row t / column, by phase
  uint32_t n0 = 0, n1 = 0;  // completed phases of bars[0], bars[1]
  bool ok = true;

  float st[kD];  // S (state pass), then G (gradient pass): row x, fp32
  {
    const float4* src = reinterpret_cast<const float4*>(s0 + ((int64_t)h * kD + x) * kD);
#pragma unroll
    for (int c = 0; c < kD / 4; ++c) {
      const float4 a4 = src[c];
      st[4 * c] = a4.x, st[4 * c + 1] = a4.y, st[4 * c + 2] = a4.z, st[4 * c + 3] = a4.w;
    }
  }
  // ---- state forward
  for (int ch = 0; ok && ch < nch; ++ch) {
    const int64_t t0 = (int64_t)ch * kC;
    const int nt = R - t0 < kC ? (int)(R - t0) : kC;
    float* blk = scratch_of(scr, H, nch, m, h, ch);
    {
      // each thread's own row, in 16-byte pieces: the stores are not waited
      // on, and this sequential kernel runs faster with them than with a
      // staged transpose
      float4* dst = reinterpret_cast<float4*>(blk + (int64_t)kSstart * kTileElems + x * kD);
#pragma unroll
      for (int c = 0; c < kD / 4; ++c) dst[c] = make_float4(st[4 * c], st[4 * c + 1], st[4 * c + 2], st[4 * c + 3]);
    }
    stage_gates(g, beta, t0, nt, H, h, sc, sbt, swt);
    __syncthreads();
    sw[x] = x < nt ? expf(sc[kC - 1] - sc[x]) : 0.f;
    __syncthreads();
    stage_row_regs(sb + kChT0, x, st);                                         // S (bf16)
    stage_rows<4>(sb + kChT1, blk + (int64_t)kZK * kTileElems, kD, kC, nullptr);  // ZK
    stage_rows<4>(sb + kChT2, k + (t0 * H + h) * kD, rs, nt, sw);                 // W = diag(w) K
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {  // ZK S^T -> cols 0..127
      tc_fence_after();
      mma_group(tb + 0, sb + kChT1, sb + kChT0, false, false);
      mma_commit(smem_u32(&bars[0]));
    }
    ok = mbar_wait_warp(smem_u32(&bars[0]), n0++ & 1, abortp);
    if (__syncthreads_or(!ok)) break;
    tc_fence_after();
    {  // E row x = E0 row x - (ZK S^T) row x; E^T column x as bf16
      const float4* e0 = reinterpret_cast<const float4*>(blk + (int64_t)kE0 * kTileElems + x * kD);
      float4* eo = reinterpret_cast<float4*>(blk + (int64_t)kEblk * kTileElems + x * kD);
#pragma unroll 1
      for (int cb = 0; cb < 4; ++cb) {
        uint32_t t32[32];
        float e[32];
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) {
          const float4 a4 = e0[cb * 8 + q4];
          e[4 * q4] = a4.x, e[4 * q4 + 1] = a4.y, e[4 * q4 + 2] = a4.z, e[4 * q4 + 3] = a4.w;
        }
        tmem_ld32(tb + lane_off + cb * 32, t32);
        tmem_wait_ld_r(t32);
#pragma unroll
        for (int xx = 0; xx < 32; ++xx) {
          e[xx] -= __uint_as_float(t32[xx]);
          st_shared_u16(sb + kChT3 + elem_off(cb * 32 + xx, x), bf16_of(e[xx]));
        }
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4)
          eo[cb * 8 + q4] = make_float4(e[4 * q4], e[4 * q4 + 1], e[4 * q4 + 2], e[4 * q4 + 3]);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {  // E^T W -> cols 128..255 (W as an N-major B)
      tc_fence_after();
      mma_group(tb + 128, sb + kChT3, sb + kChT2, true, false);
      mma_commit(smem_u32(&bars[1]));
    }
    ok = mbar_wait_warp(smem_u32(&bars[1]), n1++ & 1, abortp);
    if (__syncthreads_or(!ok)) break;
    tc_fence_after();
    {
      const float gl = expf(sc[kC - 1]);
#pragma unroll
      for (int cb = 0; cb < 4; ++cb) {
        uint32_t t32[32];
        tmem_ld32(tb + lane_off + 128 + cb * 32, t32);
        tmem_wait_ld_r(t32);
#pragma unroll
        for (int xx = 0; xx < 32; ++xx) st[cb * 32 + xx] = fmaf(gl, st[cb * 32 + xx], __uint_as_float(t32[xx]));
      }
    }
    tc_fence_before();
    __syncthreads();
  }
  if (ok && s_final) {
    float4* dst = reinterpret_cast<float4*>(s_final + (((int64_t)m * H + h) * kD + x) * kD);
#pragma unroll
    for (int c = 0; c < kD / 4; ++c) dst[c] = make_float4(st[4 * c], st[4 * c + 1], st[4 * c + 2], st[4 * c + 3]);
  }
  // ---- dL/dS backward
#pragma unroll
  for (int c = 0; c < kD; ++c) st[c] = 0.f;
  for (int ch = nch - 1; ok && ch >= 0; --ch) {
    const int64_t t0 = (int64_t)ch * kC;
    const int nt = R - t0 < kC ? (int)(R - t0) : kC;
    float* blk = scratch_of(scr, H, nch, m, h, ch);
    {
      float4* dst = reinterpret_cast<float4*>(blk + (int64_t)kGend * kTileElems + x * kD);
#pragma unroll
      for (int c = 0; c < kD / 4; ++c) dst[c] = make_float4(st[4 * c], st[4 * c + 1], st[4 * c + 2], st[4 * c + 3]);
    }
    stage_gates(g, beta, t0, nt, H, h, sc, sbt, swt);
    __syncthreads();
    sw[x] = expf(sc[x]);
    __syncthreads();
    stage_row_regs(sb + kChT0, x, st);                                         // G (bf16)
    stage_rows<4>(sb + kChT1, blk + (int64_t)kZW * kTileElems, kD, kC, nullptr);  // ZW
    stage_rows<4>(sb + kChT2, q + (t0 * H + h) * kD, rs, nt, nullptr);            // Q
    stage_rows<4>(sb + kChT3, k + (t0 * H + h) * kD, rs, nt, nullptr);            // K
#pragma unroll 4
    for (int gq = 0; gq < 16; ++gq) {  // (gamma dO)^T row x (tokens along K)
      float f8[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int t = 8 * gq + u;
        f8[u] = t < nt ? sw[t] * d_o[(t0 + t) * rs + h * kD + x] : 0.f;
      }
      st_shared_v4(sb + kChT4 + tile_off(x, gq), pack8(f8));
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {  // ZW G^T -> cols 0..127
      tc_fence_after();
      mma_group(tb + 0, sb + kChT1, sb + kChT0, false, false);
      mma_commit(smem_u32(&bars[0]));
    }
    ok = mbar_wait_warp(smem_u32(&bars[0]), n0++ & 1, abortp);
    if (__syncthreads_or(!ok)) break;
    tc_fence_after();
    {  // dU row x = dU0 row x + (ZW G^T) row x; -(gamma b dU)^T column x as bf16
      const float4* u0 = reinterpret_cast<const float4*>(blk + (int64_t)kDU0 * kTileElems + x * kD);
      float4* uo = reinterpret_cast<float4*>(blk + (int64_t)kDUblk * kTileElems + x * kD);
      const float f = -sw[x] * sbt[x];
#pragma unroll 1
      for (int cb = 0; cb < 4; ++cb) {
        uint32_t t32[32];
        float du[32];
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) {
          const float4 a4 = u0[cb * 8 + q4];
          du[4 * q4] = a4.x, du[4 * q4 + 1] = a4.y, du[4 * q4 + 2] = a4.z, du[4 * q4 + 3] = a4.w;
        }
        tmem_ld32(tb + lane_off + cb * 32, t32);
        tmem_wait_ld_r(t32);
#pragma unroll
        for (int xx = 0; xx < 32; ++xx) {
          du[xx] += __uint_as_float(t32[xx]);
          st_shared_u16(sb + kChT5 + elem_off(cb * 32 + xx, x), bf16_of(f * du[xx]));
        }
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4)
          uo[cb * 8 + q4] = make_float4(du[4 * q4], du[4 * q4 + 1], du[4 * q4 + 2], du[4 * q4 + 3]);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {  // (gamma dO)^T Q - (gamma b dU)^T K -> cols 128..255
      tc_fence_after();
      mma_group(tb + 128, sb + kChT4, sb + kChT2, true, false);
      mma_group(tb + 128, sb + kChT5, sb + kChT3, true, true);
      mma_commit(smem_u32(&bars[1]));
    }
    ok = mbar_wait_warp(smem_u32(&bars[1]), n1++ & 1, abortp);
    if (__syncthreads_or(!ok)) break;
    tc_fence_after();
    {
      const float gl = expf(sc[kC - 1]);
#pragma unroll
      for (int cb = 0; cb < 4; ++cb) {
        uint32_t t32[32];
        tmem_ld32(tb + lane_off + 128 + cb * 32, t32);
        tmem_wait_ld_r(t32);
#pragma unroll
        for (int xx = 0; xx < 32; ++xx) st[cb * 32 + xx] = fmaf(gl, st[cb * 32 + xx], __uint_as_float(t32[xx]));
      }
    }
    tc_fence_before();
    __syncthreads();
  }
  if (!ok && tid == 0 && status) atomicOr(status, kStatusTimeout);
  if (tid == 0) {
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

// ---------------------------------------------------------------- out
// One CTA per (chunk, head, member): the output o and the gradients of the
// chunk's q, k, v, g, b from S (start), G (end), E and dU of the chunk.
//   o   = diag(gamma) Q S^T + P E
//   dQ  = diag(gamma) dO S + LdP K,            LdP = lower(Gamma . dP), dP = dO E^T
//   dK  = LdP^T Q + Msym K - diag(gamma b) dU S + diag(w) E G,
//         Msym = M + M^T, M = strict_lower(dA . b . Gamma), dA = -strict_lower(dU E^T)
//   dV  = diag(b) dU
//   db  = rowsum(dA . GK) + rowsum(dU . X),    X = V - diag(gamma) K S^T
//   dg  = reverse cumulative sum of dc, with r = dP . P + dA . b . GK,
//         dc = dgamma . gamma + rowsum(r) - colsum(r) - rw, rw = w . rowsum(E G . K),
//         dgamma = rowsum(dO . Q S^T) - rowsum(b . dU . K S^T),
//         and dc_last += sum(rw) + gamma_C <G, S>.
constexpr uint32_t kOutMisc = 6 * kTile;
constexpr uint32_t kOutRowScr = kOutMisc + 4096;  // per-warp row scratch (rows_load32 / rows_store32)
constexpr uint32_t kOutSmem = kOutRowScr + kRowScrFloats * 4 + 1024;

__global__ void __launch_bounds__(kThr, 1)
    gdn_cp_out_kernel(int H, int R, int nch, const float* __restrict__ q,
                      const float* __restrict__ k, const float* __restrict__ v,
                      const float* __restrict__ g, const float* __restrict__ beta,
                      const float* __restrict__ d_o, float* __restrict__ scr,
                      float* __restrict__ o, float* __restrict__ dq, float* __restrict__ dk,
                      float* __restrict__ dv, float* __restrict__ dg, float* __restrict__ dbeta,
                      uint32_t* __restrict__ status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(sm);
  const uint32_t S0 = sb, S1 = sb + kTile, S2 = sb + 2 * kTile, S3 = sb + 3 * kTile,
                 S4 = sb + 4 * kTile, S5 = sb + 5 * kTile;
  float* sc = reinterpret_cast<float*>(sm + kOutMisc);
  float* sbt = sc + kC;
  float* sgam = sbt + kC;
  float* sw = sgam + kC;
  float* rcol = sw + kC;
  float* swt = rcol + kC;  // 8 floats of scan and reduction scratch
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOutMisc + 3584);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 5);
  uint32_t* abort_s = tslot + 1;

  const int ch = blockIdx.x, h = blockIdx.y, m = blockIdx.z, tid = threadIdx.x, warp = tid >> 5;
  const int lane = tid & 31;
  float* wscr = reinterpret_cast<float*>(sm + kOutRowScr) + warp * 32 * 33;
  const int64_t t0 = (int64_t)ch * kC;
  const int nt = R - t0 < kC ? (int)(R - t0) : kC;
  {
    const int64_t tok = (int64_t)m * R * H;
    q += tok * kD, k += tok * kD, v += tok * kD, d_o += tok * kD, g += tok, beta += tok;
    if (o) o += tok * kD;
    dq += tok * kD, dk += tok * kD, dv += tok * kD, dg += tok, dbeta += tok;
  }
  float* blk = scratch_of(scr, H, nch, m, h, ch);
  const float* Sst = blk + (int64_t)kSstart * kTileElems;
  const float* Gen = blk + (int64_t)kGend * kTileElems;
  const float* Eb = blk + (int64_t)kEblk * kTileElems;
  const float* dUb = blk + (int64_t)kDUblk * kTileElems;
  const float* gkb = blk + (int64_t)kGKblk * kTileElems;
  if (tid == 0) {
    for (int i = 0; i < 5; ++i) mbar_init(smem_u32(&bars[i]), 1);
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
  const uint32_t tb = *tslot, lane_off = (uint32_t)(warp * 32) << 16;
  const volatile uint32_t* abortp = abort_s;
  const int64_t rs = (int64_t)H * kD;
  const int t = tid;  // token row in the epilogues
  const bool live = t < nt;
  const int r0 = warp * 32;          // first row of this warp's 32
  const int nvw = nt - r0;           // rows of the warp inside the response
  const int64_t wrow = ((t0 + r0) * H + h) * kD;  // row r0 of q, k, v, d_o, o, dq, dk, dv
  bool ok = true;

  // ---- round 1: Q K^T -> T0, Q S^T -> T1, K S^T -> T2
  stage_rows(S0, q + (t0 * H + h) * kD, rs, nt, nullptr);
  stage_rows(S1, k + (t0 * H + h) * kD, rs, nt, nullptr);
  stage_rows(S2, Sst, kD, kD, nullptr);
  stage_rows(S3, Eb, kD, kC, nullptr);
  stage_rows(S4, d_o + (t0 * H + h) * kD, rs, nt, nullptr);
  stage_gates(g, beta, t0, nt, H, h, sc, sbt, swt);
  __syncthreads();
  sgam[t] = expf(sc[t]);
  sw[t] = live ? expf(sc[kC - 1] - sc[t]) : 0.f;
  rcol[t] = 0.f;
  fence_proxy_async_smem();
  __syncthreads();
  if (tid == 0) {
    tc_fence_after();
    mma_group(tb + 0, S0, S1, false, false);
    mma_group(tb + 128, S0, S2, false, false);
    mma_group(tb + 256, S1, S2, false, false);
    mma_commit(smem_u32(&bars[0]));
  }
  ok = mbar_wait_warp(smem_u32(&bars[0]), 0, abortp);
  float dgam = 0.f, dbt = 0.f, rrow = 0.f, rw = 0.f;
  if (!__syncthreads_or(!ok)) {
    tc_fence_after();
    const float ct = sc[t], gt = sgam[t], bt = sbt[t];
#pragma unroll 1
    for (int cb = 0; cb < 4; ++cb) {
      uint32_t t32[32];
      float f32[32], ra[32], rb[32];
      // P row t (bf16 tile S5: the A operand of P E, and read back for r)
      tmem_ld32(tb + lane_off + 0 + cb * 32, t32);
      tmem_wait_ld_r(t32);
#pragma unroll
      for (int xx = 0; xx < 32; ++xx) {
        const int s = cb * 32 + xx;
        f32[xx] = s <= t ? __expf(ct - sc[s]) * __uint_as_float(t32[xx]) : 0.f;
      }
#pragma unroll
      for (int gg = 0; gg < 4; ++gg) st_shared_v4(S5 + tile_off(t, cb * 4 + gg), pack8(&f32[8 * gg]));
      // Q S^T row t: dgamma, and T1 scaled by gamma_t for o = gamma Q S^T + P E
      rows_load32(ra, d_o + wrow + cb * 32, rs, nvw, wscr);
      tmem_ld32(tb + lane_off + 128 + cb * 32, t32);
      tmem_wait_ld_r(t32);
#pragma unroll
      for (int xx = 0; xx < 32; ++xx) {
        const float qs = __uint_as_float(t32[xx]);
        dgam = fmaf(ra[xx], qs, dgam);  // 0 past the response
        t32[xx] = __float_as_uint(gt * qs);
      }
      tmem_st32(tb + lane_off + 128 + cb * 32, t32);
      // K S^T row t: db (dU . X) and dgamma (- b dU . K S^T)
      rows_load32(ra, dUb + r0 * kD + cb * 32, kD, 32, wscr);
      rows_load32(rb, v + wrow + cb * 32, rs, nvw, wscr);
      tmem_ld32(tb + lane_off + 256 + cb * 32, t32);
      tmem_wait_ld_r(t32);
      if (live) {
#pragma unroll
        for (int xx = 0; xx < 32; ++xx) {
          const float ks = __uint_as_float(t32[xx]), du = ra[xx];
          dbt = fmaf(du, rb[xx] - gt * ks, dbt);
          dgam = fmaf(-bt * du, ks, dgam);
        }
      }
    }
    tmem_wait_st();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    // ---- round 2: P E -> T1 (onto gamma Q S^T), dO E^T -> T0, dU E^T -> T2, E G -> T3
    stage_rows(S0, dUb, kD, kC, nullptr);
    stage_rows(S1, Gen, kD, kD, nullptr);
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      mma_group(tb + 128, S5, S3, true, true);
      mma_group(tb + 0, S4, S3, false, false);
      mma_group(tb + 256, S0, S3, false, false);
      mma_group(tb + 384, S3, S1, true, false);
      mma_commit(smem_u32(&bars[1]));
    }
    ok = mbar_wait_warp(smem_u32(&bars[1]), 0, abortp);
  }
  if (!__syncthreads_or(!ok)) {
    tc_fence_after();
    const float ct = sc[t], bt = sbt[t], gt = sgam[t], wt = sw[t];
#pragma unroll 1
    for (int cb = 0; cb < 4; ++cb) {
      uint32_t t32[32];
      float f32[32], rv[32];
      // o row t
      tmem_ld32(tb + lane_off + 128 + cb * 32, t32);
      tmem_wait_ld_r(t32);
      if (o) {
#pragma unroll
        for (int xx = 0; xx < 32; ++xx) f32[xx] = __uint_as_float(t32[xx]);
        rows_store32(f32, o + wrow + cb * 32, rs, nvw, wscr);
      }
      // P row t, back from the bf16 tile S5 (before LdP overwrites the row)
#pragma unroll
      for (int gg = 0; gg < 4; ++gg) {
        const uint4 pk = ld_shared_v4(S5 + tile_off(t, cb * 4 + gg));
        const uint32_t w4[4] = {pk.x, pk.y, pk.z, pk.w};
#pragma unroll
        for (int i2 = 0; i2 < 4; ++i2) {
          const float2 f = unpack_bf16x2(w4[i2]);
          rv[8 * gg + 2 * i2] = f.x, rv[8 * gg + 2 * i2 + 1] = f.y;
        }
      }
      // dP row t: LdP (tile S5, row t; and LdP^T column t into S0), r = dP . P
      tmem_ld32(tb + lane_off + 0 + cb * 32, t32);
      tmem_wait_ld_r(t32);
#pragma unroll
      for (int xx = 0; xx < 32; ++xx) {
        const int s = cb * 32 + xx;
        const float dp = __uint_as_float(t32[xx]);
        f32[xx] = s <= t ? __expf(ct - sc[s]) * dp : 0.f;
        rv[xx] *= dp;  // r = dP . P
        st_shared_u16(S0 + elem_off(s, t), bf16_of(f32[xx]));
      }
#pragma unroll
      for (int gg = 0; gg < 4; ++gg) st_shared_v4(S5 + tile_off(t, cb * 4 + gg), pack8(&f32[8 * gg]));
      // dA row t = -strict_lower(dU E^T): db, r, and Msym (both triangles) into S3
      tmem_ld32(tb + lane_off + 256 + cb * 32, t32);
      tmem_wait_ld_r(t32);
#pragma unroll
      for (int xx = 0; xx < 32; ++xx) {
        const int s = cb * 32 + xx;
        float mk = 0.f;
        if (s < t) {
          const float da = -__uint_as_float(t32[xx]);
          const float gkv = gkb[a_at(t, s)];
          dbt = fmaf(da, gkv, dbt);
          rv[xx] = fmaf(da * bt, gkv, rv[xx]);
          mk = da * bt * __expf(ct - sc[s]);
        }
        if (s <= t) {
          const uint16_t hb = bf16_of(mk);
          st_shared_u16(S3 + elem_off(t, s), hb);
          st_shared_u16(S3 + elem_off(s, t), hb);
        }
      }
      // row sums of r stay with the thread; column sums over the warp's rows
      // by a shuffle exchange, then one shared add per column and warp
#pragma unroll
      for (int xx = 0; xx < 32; ++xx) rrow += rv[xx];
      atomicAdd(&rcol[cb * 32 + lane], warp_colsum32(rv));
      // E G row t: rw = w . rowsum(E G . K)
      rows_load32(f32, k + wrow + cb * 32, rs, nvw, wscr);
      tmem_ld32(tb + lane_off + 384 + cb * 32, t32);
      tmem_wait_ld_r(t32);
#pragma unroll
      for (int xx = 0; xx < 32; ++xx) rw = fmaf(__uint_as_float(t32[xx]), f32[xx], rw);  // 0 past R
    }
    rw *= wt;
    // dO tile rows scaled by gamma for dQ; K back into S1; dV
    {
#pragma unroll
      for (int gq = 0; gq < 16; ++gq) {
        const uint32_t ad = S4 + tile_off(t, gq);
        const uint4 pk = ld_shared_v4(ad);
        const uint32_t w4[4] = {pk.x, pk.y, pk.z, pk.w};
        float f8[8];
#pragma unroll
        for (int i2 = 0; i2 < 4; ++i2) {
          const float2 f = unpack_bf16x2(w4[i2]);
          f8[2 * i2] = f.x * gt, f8[2 * i2 + 1] = f.y * gt;
        }
        st_shared_v4(ad, pack8(f8));
      }
#pragma unroll 1
      for (int cb = 0; cb < 4; ++cb) {
        float u[32];
        rows_load32(u, dUb + r0 * kD + cb * 32, kD, 32, wscr);
#pragma unroll
        for (int xx = 0; xx < 32; ++xx) u[xx] *= bt;
        rows_store32(u, dv + wrow + cb * 32, rs, nvw, wscr);
      }
    }
    __syncthreads();
    stage_rows(S1, k + (t0 * H + h) * kD, rs, nt, nullptr);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    // ---- round 3a: dQ = (gamma dO) S + LdP K -> T0
    if (tid == 0) {
      tc_fence_after();
      mma_group(tb + 0, S4, S2, true, false);
      mma_group(tb + 0, S5, S1, true, true);
      mma_commit(smem_u32(&bars[2]));
    }
    ok = mbar_wait_warp(smem_u32(&bars[2]), 0, abortp);
  }
  if (!__syncthreads_or(!ok)) {
    tc_fence_after();
#pragma unroll 1
    for (int cb = 0; cb < 4; ++cb) {
      uint32_t t32[32];
      float f32[32];
      tmem_ld32(tb + lane_off + 0 + cb * 32, t32);
      tmem_wait_ld_r(t32);
#pragma unroll
      for (int xx = 0; xx < 32; ++xx) f32[xx] = __uint_as_float(t32[xx]);
      rows_store32(f32, dq + wrow + cb * 32, rs, nvw, wscr);
    }
    // Q into S4, -(gamma b) dU into S5 for dK
    {
      const float f = -sgam[t] * sbt[t];
#pragma unroll 1
      for (int cb = 0; cb < 4; ++cb) {
        float u[32];
        rows_load32(u, dUb + r0 * kD + cb * 32, kD, 32, wscr);
#pragma unroll
        for (int xx = 0; xx < 32; ++xx) u[xx] *= f;
#pragma unroll
        for (int gg = 0; gg < 4; ++gg) st_shared_v4(S5 + tile_off(t, cb * 4 + gg), pack8(&u[8 * gg]));
      }
    }
    stage_rows(S4, q + (t0 * H + h) * kD, rs, nt, nullptr);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    // ---- round 3b: dK = LdP^T Q + Msym K - (gamma b dU) S -> T2 (+ w E G from T3)
    if (tid == 0) {
      tc_fence_after();
      mma_group(tb + 256, S0, S4, true, false);
      mma_group(tb + 256, S3, S1, true, true);
      mma_group(tb + 256, S5, S2, true, true);
      mma_commit(smem_u32(&bars[3]));
    }
    ok = mbar_wait_warp(smem_u32(&bars[3]), 0, abortp);
  }
  if (!__syncthreads_or(!ok)) {
    tc_fence_after();
    const float wt = sw[t];
#pragma unroll 1
    for (int cb = 0; cb < 4; ++cb) {
      uint32_t a32[32], b32[32];
      float f32[32];
      tmem_ld32(tb + lane_off + 256 + cb * 32, a32);
      tmem_ld32(tb + lane_off + 384 + cb * 32, b32);
      tmem_wait_ld_r(a32);
      reg_dep(b32);
#pragma unroll
      for (int xx = 0; xx < 32; ++xx) f32[xx] = fmaf(wt, __uint_as_float(b32[xx]), __uint_as_float(a32[xx]));
      rows_store32(f32, dk + wrow + cb * 32, rs, nvw, wscr);
    }
    // <G, S> over the block, then dc and its reverse cumulative sum
    float gs = 0.f;
#pragma unroll 1
    for (int cb = 0; cb < 4; ++cb) {
      float ga[32], sa[32];
      rows_load32(ga, Gen + r0 * kD + cb * 32, kD, 32, wscr);
      rows_load32(sa, Sst + r0 * kD + cb * 32, kD, 32, wscr);
#pragma unroll
      for (int xx = 0; xx < 32; ++xx) gs = fmaf(ga[xx], sa[xx], gs);
    }
    float rws = rw;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      gs += __shfl_xor_sync(0xffffffffu, gs, off);
      rws += __shfl_xor_sync(0xffffffffu, rws, off);
    }
    __syncthreads();
    if (lane == 0) {
      swt[warp] = gs;
      swt[4 + warp] = rws;
    }
    __syncthreads();
    float dc = dgam * sgam[t] + rrow - rcol[t] - rw;
    if (t == kC - 1)
      dc += (swt[4] + swt[5] + swt[6] + swt[7]) + sgam[kC - 1] * (swt[0] + swt[1] + swt[2] + swt[3]);
    float x = dc;  // suffix sum within the warp
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float y = __shfl_down_sync(0xffffffffu, x, off);
      if (lane + off < 32) x += y;
    }
    __syncthreads();
    if (lane == 0) swt[warp] = x;  // the warp's total
    __syncthreads();
    for (int w = warp + 1; w < 4; ++w) x += swt[w];
    if (live) {
      dg[(t0 + t) * H + h] = x;
      dbeta[(t0 + t) * H + h] = dbt;
    }
  }
  if (!ok && tid == 0 && status) atomicOr(status, kStatusTimeout);
  if (tid == 0) {
    mma_commit(smem_u32(&bars[4]));
    mbar_wait(smem_u32(&bars[4]), 0, abortp);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tb, 512);
  }
}

}  // namespace

size_t gdn_cp_workspace_bytes(int B, int H, int R) {
  const int64_t nch = (R + kC - 1) / kC;
  return (size_t)B * H * nch * kScrFloats * sizeof(float);
}

// The backward in chunk-parallel form: prep over all chunks, the two chains
// per (head, member), then the outputs over all chunks.  ws holds the
// scratch (gdn_cp_workspace_bytes); q, k, v and d_o must be 16-byte aligned.
cudaError_t launch_gdn_cp_bwd(int B, int H, int R, const float* s0, const float* q, const float* k,
                              const float* v, const float* g, const float* beta, const float* d_o,
                              float* dq, float* dk, float* dv, float* dg, float* dbeta, float* ws,
                              uint32_t* status, cudaStream_t st) {
  if (B == 0 || H == 0 || R == 0) return cudaSuccess;
  if (H > 65535 || B > 65535) return cudaErrorInvalidValue;  // grid y and z
  for (const void* p : {(const void*)s0, (const void*)q, (const void*)k, (const void*)v,
                        (const void*)d_o, (const void*)dq, (const void*)dk, (const void*)ws})
    if (reinterpret_cast<uintptr_t>(p) & 15u) return cudaErrorMisalignedAddress;
  const int nch = (R + kC - 1) / kC;
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(gdn_cp_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kPrepSmem)) != cudaSuccess ||
      (e = cudaFuncSetAttribute(gdn_cp_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kChainSmem)) != cudaSuccess ||
      (e = cudaFuncSetAttribute(gdn_cp_out_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kOutSmem)) != cudaSuccess)
    return e;
  LaunchScope ls(kKGdnBwd, st);
  gdn_cp_prep_kernel<<<dim3(nch, H, B), kPrepThr, kPrepSmem, st>>>(H, R, nch, q, k, v, g, beta, d_o, ws,
                                                              status);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  gdn_cp_chain_kernel<<<dim3(H, B), kThr, kChainSmem, st>>>(H, R, nch, s0, q, k, g, beta, d_o, ws,
                                                           nullptr, status);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  gdn_cp_out_kernel<<<dim3(nch, H, B), kThr, kOutSmem, st>>>(H, R, nch, q, k, v, g, beta, d_o, ws,
                                                            nullptr, dq, dk, dv, dg, dbeta, status);
  return cudaGetLastError();
}

}  // namespace ls
