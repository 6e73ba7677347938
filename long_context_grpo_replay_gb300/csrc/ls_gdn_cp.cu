// Gated-DeltaNet replay in chunk-parallel form (forward and backward): the
// recurrent layers of the Qwen path replayed from the captured prompt state
// (LongStraw DeepRead summary, section Method), the gated delta rule of
// ls_gdn.cu rewritten over chunks.
//
// With chunks of C = 128 tokens, per chunk: c_t the running sum of the
// log-decays, gamma_t = exp(c_t), Gamma_ts = exp(c_t - c_s), w_t = gamma_C /
// gamma_t, GK = strict_lower(Gamma . K K^T), A = diag(b) GK, T = (I + A)^-1,
// P = lower(Gamma . Q K^T), W = diag(w) K.  The replay is three stages:
//   prep  (all chunks at once): T, then E0 = T diag(b) V, ZK = T diag(b gamma) K,
//         dU0 = T^T P^T dO, ZW = T^T W, and the chains' per-chunk terms
//         M = ZK^T W, F = E0^T W, M' = ZW^T diag(gamma b) K,
//         F' = (gamma dO)^T Q - (gamma b dU0)^T K
//   chain (per head and member, over the chunks): the affine recurrences
//         state forward   S <- gamma_C S - S M + F     (S at each chunk's start)
//         dL/dS backward  G <- gamma_C G - G M' + F'   (G at each chunk's end)
//   out   (all chunks at once): E = E0 - ZK S^T, dU = dU0 + ZW G^T, then
//         o = diag(gamma) Q S^T + P E and the gradients of q, k, v, g, b from
//         S, G, E and dU of the chunk.
// (S M = (ZK S^T)^T W and G M' = (diag(gamma b) ZW G^T)^T K: the recurrences
// are the state and gradient updates S <- gamma_C S + E^T W and
// G <- gamma_C G + (gamma dO)^T Q - (gamma b dU)^T K with E and dU expanded.)
// The chains carry one 128 x 128 product group per chunk; everything else is
// parallel over chunks.  Products are tcgen05.mma on bf16 operands with fp32
// accumulators; where an operand carries the chain's state or its input term
// it is split into bf16 hi + lo parts, so the recurrences lose no more than
// one bf16 rounding of M, M' per chunk.  Solves and states are fp32.  The
// per-element decay factors exp(c_t - c_s) use the fast __expf (a few ulp),
// far below the bf16 rounding of the products' operands.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <initializer_list>

#include "ls_gdn_tiles.cuh"
#include "ls_internal.h"

namespace ls {
namespace {
using namespace gdn;

// float32 scratch per (member, head, chunk), in [128 x 128] blocks stored
// column-group interleaved (element (r, c) at ((c / 4) * 128 + r) * 4 + c % 4:
// the 32 threads of a warp, holding 32 consecutive rows, touch 512
// contiguous bytes with each 16-byte access):
//   kE0, kDU0       E0 and dU0 (prep)
//   kSstart         S at the chunk's start (chain)
//   kDUblk          dU (out, for its own later passes)
//   kGKblk          GK (prep; zero on and above the diagonal)
// then bf16 tile images of 32 KB in the swizzled shared-memory layout, so a
// plain copy lands them ready for the MMAs: ZK, ZW, -M, F hi, F lo, -M',
// F' hi, F' lo (rows as in the formulas above), T hi, T lo (row x = column x
// of T), and the tiles of K, Q, dO (token rows; prep), S at the chunk's start
// and G = dL/dS at its end (state rows; chain) for the output kernels; then
// 16 floats: gamma_C (prep), then <G, S> of G at the chunk's end and S at its
// start (the backward chain).
enum : int { kE0 = 0, kDU0, kSstart, kDUblk, kGKblk, kFloatBlocks };
enum : int {
  kImZK = 0, kImZW, kImM, kImFhi, kImFlo, kImMg, kImFghi, kImFglo, kImThi, kImTlo,
  kImK, kImQ, kImDO, kImS, kImG, kImages
};
constexpr int64_t kImgFloats = kTile / 4;
constexpr int64_t kGammaAt = (int64_t)kFloatBlocks * kTileElems + kImages * kImgFloats;
constexpr int64_t kGsAt = kGammaAt + 1;
constexpr int64_t kScrFloats = kGammaAt + 16;

__device__ __forceinline__ float* scratch_of(float* scr, int H, int nch, int m, int h, int ch) {
  return scr + (((int64_t)m * H + h) * nch + ch) * kScrFloats;
}
__device__ __forceinline__ float* image_of(float* blk, int i) {
  return blk + (int64_t)kFloatBlocks * kTileElems + i * kImgFloats;
}
// 16-byte groups gq0 .. gq0+ngq-1 of row r of a bf16 tile, from 8 ngq fp32
// values: into the shared-memory tile at `tile` when to_smem, and into the
// same place of a tile image in global memory when img is given.
__device__ __forceinline__ void put_tile_row(bool to_smem, uint32_t tile, float* img, int r, const float* x,
                                             int gq0, int ngq) {
  for (int gq = gq0; gq < gq0 + ngq; ++gq) {
    const uint4 pk = pack8(x + 8 * (gq - gq0));
    if (to_smem) st_shared_v4(tile + tile_off(r, gq), pk);
    if (img) *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(img) + tile_off(r, gq)) = pk;
  }
}
// bf16 hi and lo parts of 8 values: hi = bf16(x), lo = bf16(x - hi).
__device__ __forceinline__ void split8(const float* x, float* hi, float* lo) {
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    hi[u] = __uint_as_float((uint32_t)bf16_of(x[u]) << 16);
    lo[u] = x[u] - hi[u];
  }
}
// Bulk copies of n tile images into shared-memory tiles, completing on bar
// (thread 0 of the CTA; the tiles' previous readers must be done).
__device__ __forceinline__ void copy_tiles(uint32_t bar, int n, const uint32_t* dst, const float* const* src) {
  mbar_expect_tx(bar, (uint32_t)n * kTile);
  for (int i = 0; i < n; ++i) bulk_load(dst[i], src[i], kTile, bar);
}
// Row r, columns c0 .. c0+31 of an interleaved scratch block.
__device__ __forceinline__ float4* blk4(float* b, int r, int c4) {
  return reinterpret_cast<float4*>(b) + c4 * kC + r;
}
__device__ __forceinline__ const float4* blk4(const float* b, int r, int c4) {
  return reinterpret_cast<const float4*>(b) + c4 * kC + r;
}
__device__ __forceinline__ void blk_ld32(float* v, const float* b, int r, int c0) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 a = *blk4(b, r, c0 / 4 + i);
    v[4 * i] = a.x, v[4 * i + 1] = a.y, v[4 * i + 2] = a.z, v[4 * i + 3] = a.w;
  }
}
__device__ __forceinline__ void blk_st32(const float* v, float* b, int r, int c0) {
#pragma unroll
  for (int i = 0; i < 8; ++i) *blk4(b, r, c0 / 4 + i) = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
}
// Row r of an interleaved scratch block into row r of a bf16 tile.
__device__ __forceinline__ void stage_row_blk(uint32_t tile, const float* b, int r) {
#pragma unroll 1
  for (int c0 = 0; c0 < kD; c0 += 32) {
    float v[32];
    blk_ld32(v, b, r, c0);
#pragma unroll
    for (int gg = 0; gg < 4; ++gg) st_shared_v4(tile + tile_off(r, c0 / 8 + gg), pack8(&v[8 * gg]));
  }
}
// 32 consecutive floats of one row, 16-byte pieces (zeros when !valid).
__device__ __forceinline__ void row_ld32(float* v, const float* p, bool valid) {
  const float4* p4 = reinterpret_cast<const float4*>(p);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 a = valid ? p4[i] : make_float4(0.f, 0.f, 0.f, 0.f);
    v[4 * i] = a.x, v[4 * i + 1] = a.y, v[4 * i + 2] = a.z, v[4 * i + 3] = a.w;
  }
}
__device__ __forceinline__ void row_st32(const float* v, float* p, bool valid) {
  if (!valid) return;
  float4* p4 = reinterpret_cast<float4*>(p);
#pragma unroll
  for (int i = 0; i < 8; ++i) p4[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
}

// Cumulative log-decay and write strength of the chunk's tokens, in two
// steps so that the loads' latency hides behind other work: load_gates
// (threads 0..127: token tid's g and b, zero past the response) early, then
// scan_gates (every thread of the block, which meets one barrier inside; the
// threads past the chunk's 128 only meet it) into sc[] (running log-decay)
// and sbt[] (b); swt[4] is scan scratch.
struct Gates {
  float g, b;
};
__device__ __forceinline__ Gates load_gates(const float* g, const float* beta, int64_t t0, int nt, int H,
                                            int h) {
  const int tid = threadIdx.x;
  Gates x{0.f, 0.f};
  if (tid < kThr && tid < nt) {
    x.g = g[(t0 + tid) * H + h];
    x.b = beta[(t0 + tid) * H + h];
  }
  return x;
}
__device__ __forceinline__ void scan_gates(Gates x, float* sc, float* sbt, float* swt) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid >= kThr) {
    __syncthreads();
    return;
  }
  sbt[tid] = x.b;
  float c = x.g;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, c, off);
    if (lane >= off) c += y;
  }
  if (lane == 31) swt[warp] = c;
  __syncthreads();
  for (int w = 0; w < warp; ++w) c += swt[w];
  sc[tid] = c;
}

// fp32 [128 x 128] buffer of T with rows of 129 floats: a column read by
// consecutive threads and a row read by a whole warp are both free of bank
// conflicts, with no index arithmetic beyond the row base.
constexpr int kTStride = kC + 1;
__device__ __forceinline__ int b_at(int t, int x) { return t * kTStride + x; }

// GK in shared memory by blocks of eight rows: the part of rows 8j .. 8j+7
// left of column 8j at gk + 32 j (j - 1), element (8j + u, s) at s * 8 + u
// (one column's eight coefficients in two 16-byte loads); the strict lower
// triangles of the diagonal 8 x 8 blocks apart, in gkd, element
// (8j + u, 8j + u2) at j * 64 + u * 8 + u2.
__device__ __forceinline__ int gk_base(int j) { return 32 * j * (j - 1); }
constexpr int kGkFloats = 32 * 16 * 15;  // blocks 0 .. 15
constexpr int kGkdFloats = 16 * 64;

// Column x of the inverse of the unit lower-triangular diagonal block of
// (I + diag(b) GK) on rows and columns r0 .. r0+63, by forward substitution
// eight rows at a time, into buf (column x, rows r0 .. r0+63; the rows above
// x come out zero).  x lies inside the block.
__device__ __forceinline__ void invert_block64(float* buf, const float* gk, const float* gkd,
                                               const float* sbt, int r0, int x) {
  for (int t8 = r0; t8 < r0 + 64; t8 += 8) {
    const int j = t8 >> 3;
    const float* gb = gk + gk_base(j);
    // the eight rows' sums in packed pairs (rows u, u+1 per 64-bit register)
    uint64_t sp[4] = {f2(0.f, 0.f), f2(0.f, 0.f), f2(0.f, 0.f), f2(0.f, 0.f)};
    // eight columns s at a time (t8 - r0 is a multiple of 8): the inner loop
    // has a fixed length, so all of its 24 loads issue ahead of the FMAs
#pragma unroll 1
    for (int s8 = r0; s8 < t8; s8 += 8) {
      float e[8];
      float4 a[8], c[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        e[i] = buf[b_at(s8 + i, x)];
        a[i] = *reinterpret_cast<const float4*>(gb + (s8 + i) * 8);
        c[i] = *reinterpret_cast<const float4*>(gb + (s8 + i) * 8 + 4);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint64_t ee = f2(e[i], e[i]);
        sp[0] = f2_fma(f2(a[i].x, a[i].y), ee, sp[0]);
        sp[1] = f2_fma(f2(a[i].z, a[i].w), ee, sp[1]);
        sp[2] = f2_fma(f2(c[i].x, c[i].y), ee, sp[2]);
        sp[3] = f2_fma(f2(c[i].z, c[i].w), ee, sp[3]);
      }
    }
    float sum[8];
#pragma unroll
    for (int u = 0; u < 4; ++u) f2_split(sp[u], sum[2 * u], sum[2 * u + 1]);
    float ev[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
#pragma unroll
      for (int u2 = 0; u2 < u; ++u2) sum[u] = fmaf(gkd[j * 64 + u * 8 + u2], ev[u2], sum[u]);
      ev[u] = fmaf(-sbt[t8 + u], sum[u], t8 + u == x ? 1.f : 0.f);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) buf[b_at(t8 + u, x)] = ev[u];
  }
}

// ---------------------------------------------------------------- prep
// The forward's share of each chunk, one CTA per (chunk, head, member), 256
// threads in two groups of 128.  T = (I + diag(b) GK)^-1 is formed
// explicitly in fp32 by blocks of 64 rows: each diagonal block by forward
// substitution (group A, one column per thread), the off-diagonal block as
// T21 = -T22 (diag(b) GK21) T11 by two products on the CUDA cores, while
// group B stages the right-hand sides.  With T split into bf16 hi + lo parts
// (their sum is T to about 2^-17) as the A operand (its tile read M-major):
// E0 = T (b V), ZK = T (b gamma K); then the state chain's terms M = ZK^T W
// and F = E0^T W.  Written to the scratch: E0, GK, gamma_C, and the images of
// ZK, -M, F hi / lo and T hi / lo (the last for the backward's own terms).
// Shared memory: R0 K -> b V -> E0, R1 b gamma K, R2 w K, R3 GK (packed
// fp32) -> ZK, R4 + R5 (and 512 bytes more) T (fp32) -> T hi (R4), T lo (R5).
constexpr uint32_t kPrepR0 = 0, kPrepR1 = kTile, kPrepR2 = 2 * kTile, kPrepR3 = 3 * kTile;
constexpr uint32_t kPrepR4 = 4 * kTile, kPrepR5 = 5 * kTile;
// T in fp32 (rows of 129 floats) runs 512 bytes past R5
constexpr uint32_t kPrepMisc = 6 * kTile + 1024;
constexpr uint32_t kPrepGkd = kPrepMisc + 3072;  // GK's diagonal blocks
constexpr uint32_t kPrepSmem = kPrepGkd + kGkdFloats * 4 + 1024;
static_assert(kGkFloats * 4 <= kTile, "GK's blocks fit in R3");
static_assert(kPrepR4 + kC * kTStride * 4 <= kPrepMisc, "T buffer overlaps the misc area");
constexpr int kPrepThr = 2 * kThr;

__global__ void __launch_bounds__(kPrepThr, 1)
    gdn_cp_prep_kernel(int H, int R, int nch, const float* __restrict__ k,
                       const float* __restrict__ v, const float* __restrict__ g,
                       const float* __restrict__ beta, float* __restrict__ scr,
                       uint32_t* __restrict__ status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(sm);
  float* gk = reinterpret_cast<float*>(sm + kPrepR3);
  float* gkd = reinterpret_cast<float*>(sm + kPrepGkd);
  float* buf = reinterpret_cast<float*>(sm + kPrepR4);
  float* sc = reinterpret_cast<float*>(sm + kPrepMisc);
  float* sbt = sc + kC;    // b
  float* sbg = sbt + kC;   // b gamma
  float* swk = sbg + kC;   // w (zero past the response)
  float* sgm = swk + kC;   // gamma
  float* swt = sgm + kC;   // 8 floats of scan scratch
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kPrepMisc + 2624);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 6);
  uint32_t* abort_s = tslot + 1;

  const int ch = blockIdx.x, h = blockIdx.y, m = blockIdx.z, tid = threadIdx.x, warp = tid >> 5;
  const bool grpA = tid < kThr;
  const int gt = tid & (kThr - 1);  // index within the group: row / column
  const int64_t t0 = (int64_t)ch * kC;
  const int nt = R - t0 < kC ? (int)(R - t0) : kC;
  {
    const int64_t tok = (int64_t)m * R * H;
    k += tok * kD, v += tok * kD, g += tok, beta += tok;
  }
  const Gates gates = load_gates(g, beta, t0, nt, H, h);  // scanned later
  float* out = scratch_of(scr, H, nch, m, h, ch);
  if (tid == 0) {
    for (int i = 0; i < 6; ++i) mbar_init(smem_u32(&bars[i]), 1);
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
  if (gt < nt) prefetch_l2((grpA ? k : v) + row0 + gt * rs, kD * 4);  // the chunk's rows into L2

  if (grpA) stage_rows<16>(sb + kPrepR0, k + row0, rs, nt, nullptr, gt, image_of(out, kImK));
  scan_gates(gates, sc, sbt, swt);
  fence_proxy_async_smem();
  __syncthreads();
  if (!grpA) {  // the right-hand sides' row scales (read after the next block barrier)
    const float ct = sc[gt], clast = sc[kC - 1];
    sgm[gt] = __expf(ct);
    sbg[gt] = sbt[gt] * sgm[gt];
    swk[gt] = gt < nt ? __expf(clast - ct) : 0.f;
    if (gt == 0) out[kGammaAt] = expf(clast);  // gamma_C for the chains
  }

  if (tid == 0) {  // K K^T -> cols 0..127
    tc_fence_after();
    mma_group(tb + 0, sb + kPrepR0, sb + kPrepR0, false, false);
    mma_commit(smem_u32(&bars[0]));
  }
  bool ok = mbar_wait_warp(smem_u32(&bars[0]), 0, abortp);
  if (!__syncthreads_or(!ok)) {
    tc_fence_after();
    if (grpA) {
      // thread r: GK row r (s < r)
      const int r = gt;
      const float cr = sc[r];
      float* gko = out + (int64_t)kGKblk * kTileElems;
#pragma unroll 1
      for (int cb = 0; cb < 4; ++cb) {
        uint32_t t32[32];
        float row[32];
        tmem_ld32(tb + lane_off + 0 + cb * 32, t32);
        tmem_wait_ld_r(t32);
#pragma unroll
        for (int xx = 0; xx < 32; ++xx) {
          const int s = cb * 32 + xx;
          row[xx] = 0.f;
          if (s < r) {
            const float val = __expf(cr - sc[s]) * __uint_as_float(t32[xx]);
            if (s < (r & ~7))
              gk[gk_base(r >> 3) + s * 8 + (r & 7)] = val;
            else
              gkd[(r >> 3) * 64 + (r & 7) * 8 + (s & 7)] = val;
            row[xx] = val;
          }
        }
        blk_st32(row, gko, r, cb * 32);
      }
    }
    __syncthreads();
    if (grpA) {
      // ---- T by blocks of 64 rows.  Column x: T11 (x < 64) or T22 (x >= 64)
      // by substitution; the rest of the column zero.
      const int x = gt, r0 = x & 64;
      for (int t = 0; t < kC; ++t)
        if (t < r0 || t >= r0 + 64) buf[b_at(t, x)] = 0.f;
      invert_block64(buf, gk, gkd, sbt, r0, x);
      named_bar_sync(1, kThr);
      // thread (xc, rq) owns columns xc and xc + 32 of the off-diagonal block,
      // rows 64 + 16 rq .. 64 + 16 rq + 15: the 16 rows' coefficients of one
      // column are shared by the warp and serve two columns per thread
      const int xc = x & 31, rq = x >> 5, t0r = 64 + 16 * rq;
      // acc[i]: rows t0r + i of columns xc and xc + 32, as one packed pair
      uint64_t acc[16];
      {  // Y = diag(b) GK21 T11 into the block's place (T11 does not read it)
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] = f2(0.f, 0.f);
        const float* g0 = gk + gk_base(t0r >> 3);      // rows t0r .. t0r+7
        const float* g1 = gk + gk_base((t0r >> 3) + 1);  // rows t0r+8 .. t0r+15
#pragma unroll 4
        for (int s = 0; s < 64; ++s) {
          const uint64_t ee = f2(buf[b_at(s, xc)], buf[b_at(s, xc + 32)]);
          const float4 a0 = *reinterpret_cast<const float4*>(g0 + s * 8);
          const float4 a1 = *reinterpret_cast<const float4*>(g0 + s * 8 + 4);
          const float4 a2 = *reinterpret_cast<const float4*>(g1 + s * 8);
          const float4 a3 = *reinterpret_cast<const float4*>(g1 + s * 8 + 4);
          const float gcoef[16] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w,
                                   a2.x, a2.y, a2.z, a2.w, a3.x, a3.y, a3.z, a3.w};
#pragma unroll
          for (int i = 0; i < 16; ++i) acc[i] = f2_fma(f2(gcoef[i], gcoef[i]), ee, acc[i]);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float y0, y1;
          f2_split(acc[i], y0, y1);
          buf[b_at(t0r + i, xc)] = sbt[t0r + i] * y0;
          buf[b_at(t0r + i, xc + 32)] = sbt[t0r + i] * y1;
        }
      }
      named_bar_sync(1, kThr);
      {  // T21 = -T22 Y (T22 stored with its zero upper triangle and unit diagonal)
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] = f2(0.f, 0.f);
#pragma unroll 4
        for (int s = 0; s < 64; ++s) {
          const uint64_t yy = f2(buf[b_at(64 + s, xc)], buf[b_at(64 + s, xc + 32)]);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float tc = buf[b_at(t0r + i, 64 + s)];
            acc[i] = f2_fma(f2(tc, tc), yy, acc[i]);
          }
        }
        named_bar_sync(1, kThr);  // Y read everywhere before T21 overwrites it
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float t0v, t1v;
          f2_split(acc[i], t0v, t1v);
          buf[b_at(t0r + i, xc)] = -t0v;
          buf[b_at(t0r + i, xc + 32)] = -t1v;
        }
      }
    } else {
      // ---- group B: the right-hand sides (K K^T has read R0)
      stage_rows<16>(sb + kPrepR0, v + row0, rs, nt, sbt, gt);                   // b V
      stage_rows_pair<16>(sb + kPrepR1, sbg, sb + kPrepR2, swk, k + row0, rs, nt, gt);  // b gamma K, w K
    }
    if (!__syncthreads_or(!ok)) {
      float tcol[kC];
      if (grpA) {
#pragma unroll
        for (int t = 0; t < kC; ++t) tcol[t] = buf[b_at(t, gt)];
      }
      __syncthreads();  // T read from R4 / R5 before its bf16 halves overwrite them
      if (grpA) {  // row x of the hi and lo tiles = column x of T; also their images
        float* ih = image_of(out, kImThi);
        float* il = image_of(out, kImTlo);
#pragma unroll
        for (int gq = 0; gq < 16; ++gq) {
          float hi[8], lo[8];
          split8(&tcol[8 * gq], hi, lo);
          put_tile_row(true, sb + kPrepR4, ih, gt, hi, gq, 1);
          put_tile_row(true, sb + kPrepR5, il, gt, lo, gq, 1);
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
        mma_commit(smem_u32(&bars[2]));
      }
      ok = mbar_wait_warp(smem_u32(&bars[2]), 0, abortp);
      if (!__syncthreads_or(!ok)) {
        // ---- E0 and ZK (warps 0-3): E0 to the scratch in fp32; bf16 tiles of
        // E0 (R0) and ZK (R3) for M and F, ZK also as an image for out
        tc_fence_after();
        const int r = gt;  // row = token
        float* fdst = out + (int64_t)kE0 * kTileElems;
        float* img = image_of(out, kImZK);
#pragma unroll 1
        for (int cb = 0; grpA && cb < 4; ++cb) {
          uint32_t t32[32];
          float f[32];
          tmem_ld32(tb + lane_off + cb * 32, t32);
          tmem_wait_ld_r(t32);
#pragma unroll
          for (int xx = 0; xx < 32; ++xx) f[xx] = __uint_as_float(t32[xx]);
          blk_st32(f, fdst, r, cb * 32);
          put_tile_row(true, sb + kPrepR0, nullptr, r, f, cb * 4, 4);
          tmem_ld32(tb + lane_off + 128 + cb * 32, t32);
          tmem_wait_ld_r(t32);
#pragma unroll
          for (int xx = 0; xx < 32; ++xx) f[xx] = __uint_as_float(t32[xx]);
          put_tile_row(true, sb + kPrepR3, img, r, f, cb * 4, 4);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
          tc_fence_after();
          mma_group_amn(tb + 0, sb + kPrepR3, sb + kPrepR2, true, false);    // M = ZK^T W
          mma_group_amn(tb + 128, sb + kPrepR0, sb + kPrepR2, true, false);  // F = E0^T W
          mma_commit(smem_u32(&bars[3]));
        }
        ok = mbar_wait_warp(smem_u32(&bars[3]), 0, abortp);
        if (!__syncthreads_or(!ok)) {
          // -M and F hi / lo to their images (group A)
          tc_fence_after();
#pragma unroll 1
          for (int cb = 0; grpA && cb < 4; ++cb) {
            uint32_t t32[32];
            float f[32], hi[32], lo[32];
            tmem_ld32(tb + lane_off + cb * 32, t32);
            tmem_wait_ld_r(t32);
#pragma unroll
            for (int xx = 0; xx < 32; ++xx) f[xx] = -__uint_as_float(t32[xx]);
            put_tile_row(false, 0, image_of(out, kImM), r, f, cb * 4, 4);
            tmem_ld32(tb + lane_off + 128 + cb * 32, t32);
            tmem_wait_ld_r(t32);
#pragma unroll
            for (int xx = 0; xx < 32; ++xx) f[xx] = __uint_as_float(t32[xx]);
#pragma unroll
            for (int gg = 0; gg < 4; ++gg) split8(&f[8 * gg], &hi[8 * gg], &lo[8 * gg]);
            put_tile_row(false, 0, image_of(out, kImFhi), r, hi, cb * 4, 4);
            put_tile_row(false, 0, image_of(out, kImFlo), r, lo, cb * 4, 4);
          }
        }
      }
    }
  }
  if (__syncthreads_or(!ok) && tid == 0 && status) atomicOr(status, kStatusTimeout);
  if (tid == 0) {  // drain before tensor memory is freed
    mma_commit(smem_u32(&bars[5]));
    mbar_wait(smem_u32(&bars[5]), 0, abortp);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tb, 512);
  }
}

// ---------------------------------------------------------------- prep (backward's terms)
// The backward's own terms of each chunk from what the forward share left in
// the scratch (T as its hi and lo images and K's tile, brought in by bulk
// copy): one CTA per (chunk, head, member), 256 threads in two groups of 128.
//   dE0 = P^T dO (P^T from a K Q^T product), dU0 = T^T dE0, ZW = T^T W,
//   M' = (diag(gamma b) ZW)^T K, F' = dO^T (diag(gamma) Q) - (gamma b dU0)^T K.
// The row scales sit on tiles formed here (ZW's rows, Q's rows), so K and
// dO serve unscaled.  Written to the scratch: dU0, and the images of Q, dO,
// ZW, -M', F' hi / lo.
// Shared memory: G0 K, G1 Q -> P^T -> w K, G2 dO, G3 dE0 -> -gamma b dU0,
// G4 T hi -> gamma Q, G5 T lo -> gamma b ZW.
constexpr uint32_t kGr0 = 0, kGr1 = kTile, kGr2 = 2 * kTile, kGr3 = 3 * kTile, kGr4 = 4 * kTile,
                   kGr5 = 5 * kTile, kGrMisc = 6 * kTile;
constexpr uint32_t kGrSmem = kGrMisc + 3072 + 1024;

__global__ void __launch_bounds__(kPrepThr, 1)
    gdn_cp_prep_grad_kernel(int H, int R, int nch, const float* __restrict__ q,
                            const float* __restrict__ k, const float* __restrict__ g,
                            const float* __restrict__ beta, const float* __restrict__ d_o,
                            float* __restrict__ scr, uint32_t* __restrict__ status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(sm);
  float* sc = reinterpret_cast<float*>(sm + kGrMisc);
  float* sbt = sc + kC;    // b
  float* sbg = sbt + kC;   // b gamma
  float* swk = sbg + kC;   // w (zero past the response)
  float* sgm = swk + kC;   // gamma
  float* swt = sgm + kC;   // 8 floats of scan scratch
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kGrMisc + 2624);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 6);
  uint32_t* abort_s = tslot + 1;
  uint32_t* never_s = tslot + 2;  // stays 0: the drain's waits are bounded by time alone

  const int ch = blockIdx.x, h = blockIdx.y, m = blockIdx.z, tid = threadIdx.x, warp = tid >> 5;
  const bool grpA = tid < kThr;
  const int gt = tid & (kThr - 1);  // index within the group: row
  const int64_t t0 = (int64_t)ch * kC;
  const int nt = R - t0 < kC ? (int)(R - t0) : kC;
  {
    const int64_t tok = (int64_t)m * R * H;
    q += tok * kD, k += tok * kD, d_o += tok * kD, g += tok, beta += tok;
  }
  const Gates gates = load_gates(g, beta, t0, nt, H, h);  // scanned later
  float* out = scratch_of(scr, H, nch, m, h, ch);
  if (tid == 0) {
    for (int i = 0; i < 6; ++i) mbar_init(smem_u32(&bars[i]), 1);
    *abort_s = 0;
    *never_s = 0;
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
  const int64_t rs = (int64_t)H * kD;
  const int64_t row0 = (t0 * H + h) * kD;
  if (tid == 0) {  // K, T hi, T lo
    const uint32_t dst[3] = {sb + kGr0, sb + kGr4, sb + kGr5};
    const float* src[3] = {image_of(out, kImK), image_of(out, kImThi), image_of(out, kImTlo)};
    copy_tiles(smem_u32(&bars[2]), 3, dst, src);
  }
  if (gt < nt) prefetch_l2((grpA ? q : k) + row0 + gt * rs, kD * 4);  // q, k are read twice
  if (grpA)
    stage_rows<16>(sb + kGr1, q + row0, rs, nt, nullptr, gt, image_of(out, kImQ));
  else
    stage_rows<16>(sb + kGr2, d_o + row0, rs, nt, nullptr, gt, image_of(out, kImDO));
  scan_gates(gates, sc, sbt, swt);
  fence_proxy_async_smem();
  __syncthreads();
  if (!grpA) {  // row scales (read after the next block barrier)
    const float ct = sc[gt], clast = sc[kC - 1];
    sgm[gt] = __expf(ct);
    sbg[gt] = sbt[gt] * sgm[gt];
    swk[gt] = gt < nt ? __expf(clast - ct) : 0.f;
  }
  bool ok = true, copied = false;  // copied (thread 0): the copies were waited for
  if (warp == 0) {
    ok = mbar_wait_warp(smem_u32(&bars[2]), 0, abortp);  // K, T hi, T lo landed
    if (tid == 0) copied = ok;
  }
  if (!__syncthreads_or(!ok)) {
    if (tid == 0) {  // K Q^T -> cols 0..127
      tc_fence_after();
      mma_group(tb + 0, sb + kGr0, sb + kGr1, false, false);
      mma_commit(smem_u32(&bars[0]));
    }
    ok = mbar_wait_warp(smem_u32(&bars[0]), 0, abortp);
  }
  if (!__syncthreads_or(!ok)) {
    tc_fence_after();
    if (grpA) {  // P^T row r: P^T[r][t] = [t >= r] Gamma_tr (K_r . Q_t), over Q (G1)
      const int r = gt;
      const float cr = sc[r];
#pragma unroll 1
      for (int cb = 0; cb < 4; ++cb) {
        uint32_t t32[32];
        float pv[32];
        tmem_ld32(tb + lane_off + cb * 32, t32);
        tmem_wait_ld_r(t32);
#pragma unroll
        for (int xx = 0; xx < 32; ++xx) {
          const int t = cb * 32 + xx;
          pv[xx] = t >= r ? __expf(sc[t] - cr) * __uint_as_float(t32[xx]) : 0.f;
        }
        put_tile_row(true, sb + kGr1, nullptr, r, pv, cb * 4, 4);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {  // dE0 = P^T dO -> cols 128..255 (dO as an N-major B)
      tc_fence_after();
      mma_group(tb + 128, sb + kGr1, sb + kGr2, true, false);
      mma_commit(smem_u32(&bars[1]));
    }
    ok = mbar_wait_warp(smem_u32(&bars[1]), 0, abortp);
    if (!__syncthreads_or(!ok)) {
      tc_fence_after();
      if (grpA) {  // dE0 rows (bf16) into G3
#pragma unroll 1
        for (int cb = 0; cb < 4; ++cb) {
          uint32_t t32[32];
          float f[32];
          tmem_ld32(tb + lane_off + 128 + cb * 32, t32);
          tmem_wait_ld_r(t32);
#pragma unroll
          for (int xx = 0; xx < 32; ++xx) f[xx] = __uint_as_float(t32[xx]);
          put_tile_row(true, sb + kGr3, nullptr, gt, f, cb * 4, 4);
        }
      } else {  // w K over P^T (G1), which dE0 has read
        stage_rows<16>(sb + kGr1, k + row0, rs, nt, swk, gt);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();
      if (tid == 0) {
        tc_fence_after();
        mma_group(tb + 256, sb + kGr4, sb + kGr3, true, false);  // dU0 = T^T dE0
        mma_group(tb + 256, sb + kGr5, sb + kGr3, true, true);
        mma_group(tb + 384, sb + kGr4, sb + kGr1, true, false);  // ZW = T^T (w K)
        mma_group(tb + 384, sb + kGr5, sb + kGr1, true, true);
        mma_commit(smem_u32(&bars[3]));
      }
      ok = mbar_wait_warp(smem_u32(&bars[3]), 0, abortp);
      if (!__syncthreads_or(!ok)) {
        // group A: dU0 rows to the scratch (fp32) and -gamma b dU0 into G3,
        // then gamma Q into G4; group B: ZW rows to their image and, times
        // gamma b, into G5
        tc_fence_after();
        const int r = gt;
        if (grpA) {
          float* fdst = out + (int64_t)kDU0 * kTileElems;
          const float fa = -sbg[r];
#pragma unroll 1
          for (int cb = 0; cb < 4; ++cb) {
            uint32_t t32[32];
            float f[32];
            tmem_ld32(tb + lane_off + 256 + cb * 32, t32);
            tmem_wait_ld_r(t32);
#pragma unroll
            for (int xx = 0; xx < 32; ++xx) f[xx] = __uint_as_float(t32[xx]);
            blk_st32(f, fdst, r, cb * 32);
#pragma unroll
            for (int xx = 0; xx < 32; ++xx) f[xx] *= fa;
            put_tile_row(true, sb + kGr3, nullptr, r, f, cb * 4, 4);
          }
          stage_rows<16>(sb + kGr4, q + row0, rs, nt, sgm, gt);
        } else {
          float* img = image_of(out, kImZW);
          const float fb = sbg[r];
#pragma unroll 1
          for (int cb = 0; cb < 4; ++cb) {
            uint32_t t32[32];
            float f[32];
            tmem_ld32(tb + lane_off + 384 + cb * 32, t32);
            tmem_wait_ld_r(t32);
#pragma unroll
            for (int xx = 0; xx < 32; ++xx) f[xx] = __uint_as_float(t32[xx]);
            put_tile_row(false, 0, img, r, f, cb * 4, 4);
#pragma unroll
            for (int xx = 0; xx < 32; ++xx) f[xx] *= fb;
            put_tile_row(true, sb + kGr5, nullptr, r, f, cb * 4, 4);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
          tc_fence_after();
          mma_group_amn(tb + 0, sb + kGr5, sb + kGr0, true, false);    // M' = (gamma b ZW)^T K
          mma_group_amn(tb + 128, sb + kGr2, sb + kGr4, true, false);  // F' = dO^T (gamma Q)
          mma_group_amn(tb + 128, sb + kGr3, sb + kGr0, true, true);   //      - (gamma b dU0)^T K
          mma_commit(smem_u32(&bars[4]));
        }
        ok = mbar_wait_warp(smem_u32(&bars[4]), 0, abortp);
        if (!__syncthreads_or(!ok)) {
          // -M' (group A) and F' hi / lo (group B) to their images
          tc_fence_after();
#pragma unroll 1
          for (int cb = 0; cb < 4; ++cb) {
            uint32_t t32[32];
            float f[32], hi[32], lo[32];
            tmem_ld32(tb + lane_off + (grpA ? 0 : 128) + cb * 32, t32);
            tmem_wait_ld_r(t32);
            if (grpA) {
#pragma unroll
              for (int xx = 0; xx < 32; ++xx) f[xx] = -__uint_as_float(t32[xx]);
              put_tile_row(false, 0, image_of(out, kImMg), r, f, cb * 4, 4);
            } else {
#pragma unroll
              for (int xx = 0; xx < 32; ++xx) f[xx] = __uint_as_float(t32[xx]);
#pragma unroll
              for (int gg = 0; gg < 4; ++gg) split8(&f[8 * gg], &hi[8 * gg], &lo[8 * gg]);
              put_tile_row(false, 0, image_of(out, kImFghi), r, hi, cb * 4, 4);
              put_tile_row(false, 0, image_of(out, kImFglo), r, lo, cb * 4, 4);
            }
          }
        }
      }
    }
  }
  if (__syncthreads_or(!ok) && tid == 0 && status) atomicOr(status, kStatusTimeout);
  if (tid == 0) {  // drain: the products, and the copies if nobody waited for them
    mma_commit(smem_u32(&bars[5]));
    mbar_wait(smem_u32(&bars[5]), 0, never_s);
    if (!copied) mbar_wait(smem_u32(&bars[2]), 0, never_s);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tb, 512);
  }
}

// ---------------------------------------------------------------- chain
// One CTA per (head, member), sequential over the chunks: the state forward
// S <- gamma_C S + D (writing S at each chunk's start), then dL/dS backward
// G <- gamma_C G + D (writing G at each chunk's end), with one product group
// per chunk, D = S_hi (-M) + S_lo (-M) + I F_hi + I F_lo (S split into bf16
// hi + lo, the identity as A).  The chunk's three tiles come from prep's
// images by bulk copy; the next chunk's copies start as soon as the current
// chunk's products have read theirs.  256 threads: thread (x, half) keeps
// columns 64 half .. 64 half + 63 of state row x.  A backward step also
// forms <G, S> of the chunk (G at its end, S at its start, both fp32) while
// its products run, for the output kernel's dg; the eight warps' partial
// sums meet in a fixed order, so the sum does not depend on timing.
constexpr uint32_t kChI = 0, kChShi = kTile, kChSlo = 2 * kTile, kChM = 3 * kTile,
                   kChFhi = 4 * kTile, kChFlo = 5 * kTile, kChMisc = 6 * kTile;
constexpr uint32_t kChainSmem = kChMisc + 1024 + 1024;
constexpr int kChThr = 2 * kThr;

// Steps i0 .. i1-1 of the 2 nch steps (forward over the chunks, then backward):
// [0, nch) the replay's forward (writing s_final), [nch, 2 nch) the backward
// alone (the forward's S already in the scratch), [0, 2 nch) both.
__global__ void __launch_bounds__(kChThr, 1)
    gdn_cp_chain_kernel(int H, int nch, int i0, int i1, const float* __restrict__ s0,
                        float* __restrict__ scr, float* __restrict__ s_final,
                        uint32_t* __restrict__ status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(sm);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kChMisc);  // copies, products, drain
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 3);
  float* gsw = reinterpret_cast<float*>(sm + kChMisc + 64);  // <G, S>: one partial per warp
  uint32_t* abort_s = tslot + 1;
  uint32_t* never_s = tslot + 2;  // stays 0: the drain's waits are bounded by time alone

  const int h = blockIdx.x, m = blockIdx.y, tid = threadIdx.x, warp = tid >> 5;
  const int x = tid & (kThr - 1), half = tid >> 7, c0 = 64 * half, gq0 = 8 * half;
  if (tid == 0) {
    for (int i = 0; i < 3; ++i) mbar_init(smem_u32(&bars[i]), 1);
    *abort_s = 0;
    *never_s = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tslot), 128);
    tmem_relinquish();
  }
#pragma unroll 1
  for (int gq = gq0; gq < gq0 + 8; ++gq) {  // the identity, row x
    float e[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) e[u] = 8 * gq + u == x ? 1.f : 0.f;
    st_shared_v4(sb + kChI + tile_off(x, gq), pack8(e));
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = *tslot, lane_off = (uint32_t)((warp & 3) * 32) << 16;
  const volatile uint32_t* abortp = abort_s;
  uint32_t ncp = 0, nmm = 0;  // completed phases of the copy and product barriers
  int pend = -1;              // thread 0: parity of a copy phase given up on
  bool ok = true;

  // chunk visited at step i of the 2 nch steps: forward, then backward
  auto chunk_at = [&](int i) { return i < nch ? i : 2 * nch - 1 - i; };
  auto issue = [&](int i) {  // thread 0: the three tiles of step i
    float* blk = scratch_of(scr, H, nch, m, h, chunk_at(i));
    const bool bw = i >= nch;
    const uint32_t bar = smem_u32(&bars[0]);
    mbar_expect_tx(bar, 3 * kTile);
    bulk_load(sb + kChM, image_of(blk, bw ? kImMg : kImM), kTile, bar);
    bulk_load(sb + kChFhi, image_of(blk, bw ? kImFghi : kImFhi), kTile, bar);
    bulk_load(sb + kChFlo, image_of(blk, bw ? kImFglo : kImFlo), kTile, bar);
    if (bw) prefetch_l2(blk + (int64_t)kSstart * kTileElems, kTileElems * 4);  // for <G, S>
  };
  if (tid == 0 && i0 < i1) issue(i0);

  float st[64];  // S (forward), then G (backward): row x, columns c0 .. c0+63, fp32
  {
    const float4* src = reinterpret_cast<const float4*>(s0 + ((int64_t)h * kD + x) * kD + c0);
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const float4 a4 = i0 < nch ? src[c] : make_float4(0.f, 0.f, 0.f, 0.f);
      st[4 * c] = a4.x, st[4 * c + 1] = a4.y, st[4 * c + 2] = a4.z, st[4 * c + 3] = a4.w;
    }
  }
  const int steps = i1;
  for (int i = i0; ok && i <= steps; ++i) {
    const bool bw = i >= nch;
    if (i == nch && i0 < nch) {
      if (s_final) {
        float4* dst = reinterpret_cast<float4*>(s_final + (((int64_t)m * H + h) * kD + x) * kD + c0);
#pragma unroll
        for (int c = 0; c < 16; ++c) dst[c] = make_float4(st[4 * c], st[4 * c + 1], st[4 * c + 2], st[4 * c + 3]);
      }
#pragma unroll
      for (int c = 0; c < 64; ++c) st[c] = 0.f;
    }
    if (i == steps) break;
    float* blk = scratch_of(scr, H, nch, m, h, chunk_at(i));
    const float gc = blk[kGammaAt];
    float* sst = blk + (int64_t)kSstart * kTileElems;
    if (!bw) {  // S at the chunk's start, row x
#pragma unroll
      for (int c = 0; c < 16; ++c) *blk4(sst, x, c0 / 4 + c) = make_float4(st[4 * c], st[4 * c + 1], st[4 * c + 2], st[4 * c + 3]);
    }
    uint8_t* simg = reinterpret_cast<uint8_t*>(image_of(blk, bw ? kImG : kImS));  // bf16 S (or G) for the output kernels
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float hi[8], lo[8];
      split8(&st[8 * j], hi, lo);
      const uint4 ph = pack8(hi);
      st_shared_v4(sb + kChShi + tile_off(x, gq0 + j), ph);
      st_shared_v4(sb + kChSlo + tile_off(x, gq0 + j), pack8(lo));
      *reinterpret_cast<uint4*>(simg + tile_off(x, gq0 + j)) = ph;
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
      const bool got = mbar_wait_warp(smem_u32(&bars[0]), ncp & 1, abortp);
      if (tid == 0) {
        if (got) {
          tc_fence_after();
          mma_group(tb, sb + kChShi, sb + kChM, true, false);
          mma_group(tb, sb + kChSlo, sb + kChM, true, true);
          mma_group(tb, sb + kChI, sb + kChFhi, true, true);
          mma_group(tb, sb + kChI, sb + kChFlo, true, true);
          mma_commit(smem_u32(&bars[1]));
        } else {
          pend = (int)(ncp & 1);
          *abort_s = 1u;
        }
      }
    }
    ++ncp;
    if (bw) {  // <G, S> of this chunk, row x (S read back as this thread wrote it)
      float gs = 0.f;
#pragma unroll
      for (int c4 = 0; c4 < 16; c4 += 4) {
        float4 a4[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) a4[u] = *blk4(sst, x, c0 / 4 + c4 + u);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float* sv = &st[4 * (c4 + u)];
          gs = fmaf(sv[0], a4[u].x, fmaf(sv[1], a4[u].y, fmaf(sv[2], a4[u].z, fmaf(sv[3], a4[u].w, gs))));
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) gs += __shfl_xor_sync(0xffffffffu, gs, off);
      if ((tid & 31) == 0) gsw[warp] = gs;
    }
    ok = mbar_wait_warp(smem_u32(&bars[1]), nmm++ & 1, abortp);
    if (__syncthreads_or(!ok)) break;
    if (tid == 0 && i + 1 < steps) issue(i + 1);  // the products have read this step's tiles
    if (bw && tid == 32)  // the next step's partials come after its next barrier
      blk[kGsAt] = ((gsw[0] + gsw[1]) + (gsw[2] + gsw[3])) + ((gsw[4] + gsw[5]) + (gsw[6] + gsw[7]));
    tc_fence_after();
#pragma unroll
    for (int cb = 0; cb < 2; ++cb) {
      uint32_t t32[32];
      tmem_ld32(tb + lane_off + c0 + cb * 32, t32);
      tmem_wait_ld_r(t32);
#pragma unroll
      for (int xx = 0; xx < 32; ++xx) st[cb * 32 + xx] = fmaf(gc, st[cb * 32 + xx], __uint_as_float(t32[xx]));
    }
    tc_fence_before();
  }
  if (!ok && tid == 0 && status) atomicOr(status, kStatusTimeout);
  if (tid == 0) {  // drain the products, and a copy given up on, before the CTA ends
    mma_commit(smem_u32(&bars[2]));
    mbar_wait(smem_u32(&bars[2]), 0, never_s);
    if (pend >= 0) mbar_wait(smem_u32(&bars[0]), (uint32_t)pend, never_s);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tb, 128);
  }
}

// ---------------------------------------------------------------- out
// One CTA per (chunk, head, member): first E = E0 - ZK S^T and
// dU = dU0 + ZW G^T of the chunk (into the scratch), then the output o and
// the gradients of the chunk's q, k, v, g, b from S (start), G (end), E and
// dU.
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
constexpr uint32_t kOutSmem = kOutMisc + 8192 + 1024;
constexpr int kOutThr = 2 * kThr;

// 256 threads: thread (t, hf) owns token row t and the column half
// 64 hf .. 64 hf + 63 (column blocks cb = 2 hf, 2 hf + 1) in every epilogue;
// the row sums of the two halves meet in shared memory at the end.
__global__ void __launch_bounds__(kOutThr, 1)
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
  float* part = rcol + kC;     // [4][128] row sums of the second column half
  float* swt = part + 4 * kC;  // 8 floats of scan and reduction scratch
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOutMisc + 5184);
  float* colpart = reinterpret_cast<float*>(sm + kOutMisc + 5376);  // [4][128] column sums of r per row quarter
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 7);
  uint32_t* abort_s = tslot + 1;
  uint32_t* never_s = tslot + 2;  // stays 0: the drain's waits are bounded by time alone

  const int ch = blockIdx.x, h = blockIdx.y, m = blockIdx.z, tid = threadIdx.x, warp = tid >> 5;
  const int lane = tid & 31;
  const int t = tid & (kThr - 1), hf = tid >> 7, cb0 = 2 * hf;  // row, column half
  const int64_t t0 = (int64_t)ch * kC;
  const int nt = R - t0 < kC ? (int)(R - t0) : kC;
  {
    const int64_t tok = (int64_t)m * R * H;
    q += tok * kD, k += tok * kD, v += tok * kD, d_o += tok * kD, g += tok, beta += tok;
    if (o) o += tok * kD;
    dq += tok * kD, dk += tok * kD, dv += tok * kD, dg += tok, dbeta += tok;
  }
  const Gates gates = load_gates(g, beta, t0, nt, H, h);  // scanned later
  float* blk = scratch_of(scr, H, nch, m, h, ch);
  float* dUb = blk + (int64_t)kDUblk * kTileElems;
  const float* gkb = blk + (int64_t)kGKblk * kTileElems;
  if (tid == 0) {
    for (int i = 0; i < 7; ++i) mbar_init(smem_u32(&bars[i]), 1);
    *abort_s = 0;
    *never_s = 0;
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
  const uint32_t cbar = smem_u32(&bars[6]);  // the tile images' bulk copies, one phase per product step
  uint32_t ncp = 0, nwt = 0;  // copy phases issued, and waited for (every thread keeps both)
  int pend = -1;              // thread 0: parity of a copy phase whose wait gave up
  const bool live = t < nt;
  const int r0 = (warp & 3) * 32;  // first row of this warp's 32
  const int64_t rowt = ((t0 + t) * H + h) * kD;  // row t of q, k, v, d_o, o, dq, dk, dv
  bool ok = true;
  auto wait_copies = [&]() {  // every warp: the current copy phase has landed
    const bool got = mbar_wait_warp(cbar, nwt & 1, abortp);
    if (!got && tid == 0) pend = (int)(nwt & 1);
    ++nwt;
    return got;
  };

  // everything this CTA reads, asked into L2 up front: rows of v and dO (the
  // tiles come from images) and the chunk's scratch blocks
  if (live) prefetch_l2((hf ? v : d_o) + rowt, kD * 4);
  if (tid == 0) {
    prefetch_l2(blk, 2 * kTileElems * 4);                             // E0, dU0
    prefetch_l2(blk + (int64_t)kGKblk * kTileElems, kTileElems * 4);  // GK
    const uint32_t dst[4] = {S0, S1, S2, S3};  // ---- step 0 tiles: ZK, ZW, S, G
    const float* src[4] = {image_of(blk, kImZK), image_of(blk, kImZW), image_of(blk, kImS),
                           image_of(blk, kImG)};
    copy_tiles(cbar, 4, dst, src);
  }
  ++ncp;
  // the gates while the copies land
  scan_gates(gates, sc, sbt, swt);
  __syncthreads();
  if (hf == 0) {
    sgam[t] = expf(sc[t]);
    sw[t] = live ? expf(sc[kC - 1] - sc[t]) : 0.f;
  }
  // ---- step 0: ZK S^T -> T0, ZW G^T -> T1; E into S3 (bf16), dU rows into
  // the scratch, and dV = diag(b) dU
  ok = wait_copies();
  if (!__syncthreads_or(!ok)) {
    if (tid == 0) {
      tc_fence_after();
      mma_group(tb + 0, S0, S2, false, false);
      mma_group(tb + 128, S1, S3, false, false);
      mma_commit(smem_u32(&bars[5]));
    }
    ok = mbar_wait_warp(smem_u32(&bars[5]), 0, abortp);
  }
  if (!__syncthreads_or(!ok)) {
    if (tid == 0) {  // step 1 tiles: Q, K, dO (the step-0 products are done with S0, S1)
      const uint32_t dst[3] = {S0, S1, S4};
      const float* src[3] = {image_of(blk, kImQ), image_of(blk, kImK), image_of(blk, kImDO)};
      copy_tiles(cbar, 3, dst, src);
    }
    ++ncp;
    tc_fence_after();
    const float* e0b = blk + (int64_t)kE0 * kTileElems;
    const float* du0b = blk + (int64_t)kDU0 * kTileElems;
#pragma unroll 1
    for (int cb = cb0; cb < cb0 + 2; ++cb) {
      uint32_t t32[32];
      float f32[32];
      blk_ld32(f32, e0b, t, cb * 32);
      tmem_ld32(tb + lane_off + 0 + cb * 32, t32);
      tmem_wait_ld_r(t32);
#pragma unroll
      for (int xx = 0; xx < 32; ++xx) f32[xx] -= __uint_as_float(t32[xx]);
#pragma unroll
      for (int gg = 0; gg < 4; ++gg) st_shared_v4(S3 + tile_off(t, cb * 4 + gg), pack8(&f32[8 * gg]));
      blk_ld32(f32, du0b, t, cb * 32);
      tmem_ld32(tb + lane_off + 128 + cb * 32, t32);
      tmem_wait_ld_r(t32);
#pragma unroll
      for (int xx = 0; xx < 32; ++xx) f32[xx] += __uint_as_float(t32[xx]);
      blk_st32(f32, dUb, t, cb * 32);
      const float bt = sbt[t];
#pragma unroll
      for (int xx = 0; xx < 32; ++xx) f32[xx] *= bt;
      row_st32(f32, dv + rowt + cb * 32, live);
    }
  }
  tc_fence_before();
  __syncthreads();  // dU rows written before any thread reads them back

  // ---- step 1: Q K^T -> T0, Q S^T -> T1, K S^T -> T2
  if (ok) ok = wait_copies();
  fence_proxy_async_smem();
  if (__syncthreads_or(!ok)) ok = false;
  if (ok && tid == 0) {
    tc_fence_after();
    mma_group(tb + 0, S0, S1, false, false);
    mma_group(tb + 128, S0, S2, false, false);
    mma_group(tb + 256, S1, S2, false, false);
    mma_commit(smem_u32(&bars[0]));
  }
  if (ok) ok = mbar_wait_warp(smem_u32(&bars[0]), 0, abortp);
  float dgam = 0.f, dbt = 0.f, rrow = 0.f, rw = 0.f;  // this half's parts of the row sums
  if (!__syncthreads_or(!ok)) {
    if (tid == 0) {  // step 2's G (the step-1 products are done with S1)
      const uint32_t dst[1] = {S1};
      const float* src[1] = {image_of(blk, kImG)};
      copy_tiles(cbar, 1, dst, src);
    }
    ++ncp;
    tc_fence_after();
    const float ct = sc[t], gt = sgam[t], bt = sbt[t];
#pragma unroll 1
    for (int cb = cb0; cb < cb0 + 2; ++cb) {
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
      row_ld32(ra, d_o + rowt + cb * 32, live);
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
      blk_ld32(ra, dUb, t, cb * 32);
      row_ld32(rb, v + rowt + cb * 32, live);
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
    // ---- step 2: P E -> T1 (onto gamma Q S^T), dO E^T -> T0, dU E^T -> T2, E G -> T3
    if (hf == 0) stage_row_blk(S0, dUb, t);
    ok = wait_copies();
    fence_proxy_async_smem();
    if (__syncthreads_or(!ok)) ok = false;
    if (ok && tid == 0) {
      tc_fence_after();
      mma_group(tb + 128, S5, S3, true, true);
      mma_group(tb + 0, S4, S3, false, false);
      mma_group(tb + 256, S0, S3, false, false);
      mma_group(tb + 384, S3, S1, true, false);
      mma_commit(smem_u32(&bars[1]));
    }
    if (ok) ok = mbar_wait_warp(smem_u32(&bars[1]), 0, abortp);
  }
  if (!__syncthreads_or(!ok)) {
    if (tid == 0) {  // step 3a's K (the step-2 products are done with S1)
      const uint32_t dst[1] = {S1};
      const float* src[1] = {image_of(blk, kImK)};
      copy_tiles(cbar, 1, dst, src);
    }
    ++ncp;
    tc_fence_after();
    const float ct = sc[t], bt = sbt[t], gt = sgam[t], wt = sw[t];
#pragma unroll 1
    for (int cb = cb0; cb < cb0 + 2; ++cb) {
      uint32_t t32[32];
      float f32[32], rv[32];
      // o row t
      tmem_ld32(tb + lane_off + 128 + cb * 32, t32);
      tmem_wait_ld_r(t32);
      if (o) {
#pragma unroll
        for (int xx = 0; xx < 32; ++xx) f32[xx] = __uint_as_float(t32[xx]);
        row_st32(f32, o + rowt + cb * 32, live);
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
      // dP row t: LdP (tile S5, row t; LdP^T is the same tile read M-major),
      // r = dP . P
      tmem_ld32(tb + lane_off + 0 + cb * 32, t32);
      tmem_wait_ld_r(t32);
#pragma unroll
      for (int xx = 0; xx < 32; ++xx) {
        const int s = cb * 32 + xx;
        const float dp = __uint_as_float(t32[xx]);
        f32[xx] = s <= t ? __expf(ct - sc[s]) * dp : 0.f;
        rv[xx] *= dp;  // r = dP . P
      }
#pragma unroll
      for (int gg = 0; gg < 4; ++gg) st_shared_v4(S5 + tile_off(t, cb * 4 + gg), pack8(&f32[8 * gg]));
      // dA row t = -strict_lower(dU E^T): db, r, and M row t into S3 (Msym K is
      // M K plus the same tile read M-major)
      float gkr[32];  // GK row t, columns cb*32 ..
      if (cb * 32 < r0 + 32) blk_ld32(gkr, gkb, t, cb * 32);
      tmem_ld32(tb + lane_off + 256 + cb * 32, t32);
      tmem_wait_ld_r(t32);
#pragma unroll
      for (int gg = 0; gg < 4; ++gg) {
        float mk[8];  // M row t, columns 8 gg .. (zero on and right of the diagonal)
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int xx = 8 * gg + u, s = cb * 32 + xx;
          mk[u] = 0.f;
          if (s < t) {
            const float da = -__uint_as_float(t32[xx]);
            const float gkv = gkr[xx];
            dbt = fmaf(da, gkv, dbt);
            rv[xx] = fmaf(da * bt, gkv, rv[xx]);
            mk[u] = da * bt * __expf(ct - sc[s]);
          }
        }
        st_shared_v4(S3 + tile_off(t, cb * 4 + gg), pack8(mk));
      }
      // row sums of r stay with the thread; column sums over the warp's rows
      // by a shuffle exchange, one slot per (row quarter, column): summed in
      // a fixed order later, so the result does not depend on warp timing
#pragma unroll
      for (int xx = 0; xx < 32; ++xx) rrow += rv[xx];
      colpart[(warp & 3) * kC + cb * 32 + lane] = warp_colsum32(rv);
      // E G row t: rw = w . rowsum(E G . K)
      row_ld32(f32, k + rowt + cb * 32, live);
      tmem_ld32(tb + lane_off + 384 + cb * 32, t32);
      tmem_wait_ld_r(t32);
#pragma unroll
      for (int xx = 0; xx < 32; ++xx) rw = fmaf(__uint_as_float(t32[xx]), f32[xx], rw);  // 0 past R
    }
    rw *= wt;
    // dO tile rows scaled by gamma for dQ
#pragma unroll
    for (int gq = 8 * hf; gq < 8 * hf + 8; ++gq) {
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
    ok = wait_copies();  // K back in S1
    fence_proxy_async_smem();
    tc_fence_before();
    if (__syncthreads_or(!ok)) ok = false;
    // ---- step 3a: dQ = (gamma dO) S + LdP K -> T0
    if (ok && tid == 0) {
      tc_fence_after();
      mma_group(tb + 0, S4, S2, true, false);
      mma_group(tb + 0, S5, S1, true, true);
      mma_commit(smem_u32(&bars[2]));
    }
    if (ok) ok = mbar_wait_warp(smem_u32(&bars[2]), 0, abortp);
  }
  if (!__syncthreads_or(!ok)) {
    if (tid == 0) {  // step 3b's Q (the step-3a products are done with S4)
      const uint32_t dst[1] = {S4};
      const float* src[1] = {image_of(blk, kImQ)};
      copy_tiles(cbar, 1, dst, src);
    }
    ++ncp;
    tc_fence_after();
    const float f = -sgam[t] * sbt[t];
#pragma unroll 1
    for (int cb = cb0; cb < cb0 + 2; ++cb) {
      uint32_t t32[32];
      float f32[32];
      tmem_ld32(tb + lane_off + 0 + cb * 32, t32);
      tmem_wait_ld_r(t32);
#pragma unroll
      for (int xx = 0; xx < 32; ++xx) f32[xx] = __uint_as_float(t32[xx]);
      row_st32(f32, dq + rowt + cb * 32, live);
      // -(gamma b) dU into S0 for dK (LdP stays in S5)
      blk_ld32(f32, dUb, t, cb * 32);
#pragma unroll
      for (int xx = 0; xx < 32; ++xx) f32[xx] *= f;
#pragma unroll
      for (int gg = 0; gg < 4; ++gg) st_shared_v4(S0 + tile_off(t, cb * 4 + gg), pack8(&f32[8 * gg]));
    }
    ok = wait_copies();  // Q in S4
    fence_proxy_async_smem();
    tc_fence_before();
    if (__syncthreads_or(!ok)) ok = false;  // S0 rows of both halves written; dQ read out of T0
    // ---- step 3b: dK = LdP^T Q + (M + M^T) K - (gamma b dU) S -> T2 (+ w E G from T3)
    if (ok && tid == 0) {
      tc_fence_after();
      mma_group_amn(tb + 256, S5, S4, true, false);
      mma_group(tb + 256, S3, S1, true, true);
      mma_group_amn(tb + 256, S3, S1, true, true);
      mma_group(tb + 256, S0, S2, true, true);
      mma_commit(smem_u32(&bars[3]));
    }
    if (ok) ok = mbar_wait_warp(smem_u32(&bars[3]), 0, abortp);
  }
  if (!__syncthreads_or(!ok)) {
    tc_fence_after();
    const float wt = sw[t];
#pragma unroll 1
    for (int cb = cb0; cb < cb0 + 2; ++cb) {
      uint32_t a32[32], b32[32];
      float f32[32];
      tmem_ld32(tb + lane_off + 256 + cb * 32, a32);
      tmem_ld32(tb + lane_off + 384 + cb * 32, b32);
      tmem_wait_ld_r(a32);
      reg_dep(b32);
#pragma unroll
      for (int xx = 0; xx < 32; ++xx) f32[xx] = fmaf(wt, __uint_as_float(b32[xx]), __uint_as_float(a32[xx]));
      row_st32(f32, dk + rowt + cb * 32, live);
    }
    // the second half's row sums to the first; the column sums of r
    if (hf) {
      part[0 * kC + t] = dgam;
      part[1 * kC + t] = dbt;
      part[2 * kC + t] = rrow;
      part[3 * kC + t] = rw;
    }
    __syncthreads();
    float rws = 0.f;
    if (!hf) {
      rcol[t] = ((colpart[t] + colpart[kC + t]) + colpart[2 * kC + t]) + colpart[3 * kC + t];
      dgam += part[0 * kC + t];
      dbt += part[1 * kC + t];
      rrow += part[2 * kC + t];
      rw += part[3 * kC + t];
      rws = rw;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) rws += __shfl_xor_sync(0xffffffffu, rws, off);
      if (lane == 0) swt[4 + warp] = rws;
    }
    __syncthreads();
    // dc and its reverse cumulative sum over the chunk (first half: one thread per row)
    float x = 0.f;
    if (!hf) {
      float dc = dgam * sgam[t] + rrow - rcol[t] - rw;
      if (t == kC - 1)
        dc += (swt[4] + swt[5] + swt[6] + swt[7]) + sgam[kC - 1] * blk[kGsAt];
      x = dc;  // suffix sum within the warp
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_down_sync(0xffffffffu, x, off);
        if (lane + off < 32) x += y;
      }
    }
    __syncthreads();
    if (!hf && lane == 0) swt[warp] = x;  // the warp's total
    __syncthreads();
    if (!hf) {
      for (int w = warp + 1; w < 4; ++w) x += swt[w];
      if (live) {
        dg[(t0 + t) * H + h] = x;
        dbeta[(t0 + t) * H + h] = dbt;
      }
    }
  }
  if (!ok && tid == 0 && status) atomicOr(status, kStatusTimeout);
  if (tid == 0) {  // drain: the products, and a copy phase nobody waited for
    mma_commit(smem_u32(&bars[4]));
    mbar_wait(smem_u32(&bars[4]), 0, never_s);
    if (nwt < ncp) mbar_wait(cbar, (ncp - 1) & 1, never_s);
    else if (pend >= 0) mbar_wait(cbar, (uint32_t)pend, never_s);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tb, 512);
  }
}

// ---------------------------------------------------------------- forward out
// The replay's forward output, one CTA per (chunk, head, member), 256
// threads (row t, column half hf): E = E0 - ZK S^T, then
// o = diag(gamma) Q S^T + P E with P = lower(Gamma . Q K^T).
// Shared memory: F0 Q -> P, F1 K -> E, F2 S (start), F3 ZK.
constexpr uint32_t kFoMisc = 4 * kTile;
constexpr uint32_t kFoSmem = kFoMisc + 2048 + 1024;

__global__ void __launch_bounds__(kOutThr, 1)
    gdn_cp_fwd_out_kernel(int H, int R, int nch, const float* __restrict__ q,
                          const float* __restrict__ k, const float* __restrict__ g,
                          const float* __restrict__ beta, float* __restrict__ scr,
                          float* __restrict__ o, uint32_t* __restrict__ status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(sm);
  const uint32_t F0 = sb, F1 = sb + kTile, F2 = sb + 2 * kTile, F3 = sb + 3 * kTile;
  float* sc = reinterpret_cast<float*>(sm + kFoMisc);
  float* sbt = sc + kC;
  float* swt = sbt + kC;  // 8 floats of scan scratch
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kFoMisc + 1088);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 4);
  uint32_t* abort_s = tslot + 1;
  uint32_t* never_s = tslot + 2;  // stays 0: the drain's waits are bounded by time alone

  const int ch = blockIdx.x, h = blockIdx.y, m = blockIdx.z, tid = threadIdx.x, warp = tid >> 5;
  const int t = tid & (kThr - 1), hf = tid >> 7, cb0 = 2 * hf;
  const int64_t t0 = (int64_t)ch * kC;
  const int nt = R - t0 < kC ? (int)(R - t0) : kC;
  {
    const int64_t tok = (int64_t)m * R * H;
    q += tok * kD, k += tok * kD, g += tok, beta += tok, o += tok * kD;
  }
  const Gates gates = load_gates(g, beta, t0, nt, H, h);  // scanned later
  float* blk = scratch_of(scr, H, nch, m, h, ch);
  if (tid == 0) {
    for (int i = 0; i < 4; ++i) mbar_init(smem_u32(&bars[i]), 1);
    *abort_s = 0;
    *never_s = 0;
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
  const int64_t rs = (int64_t)H * kD;
  const bool live = t < nt;
  const int64_t row0 = (t0 * H + h) * kD, rowt = ((t0 + t) * H + h) * kD;
  if (tid == 0) prefetch_l2(blk + (int64_t)kE0 * kTileElems, kTileElems * 4);  // E0

  const uint32_t cbar = smem_u32(&bars[3]);
  if (tid == 0) {  // K, S and ZK from their images
    const uint32_t dst[3] = {F1, F2, F3};
    const float* src[3] = {image_of(blk, kImK), image_of(blk, kImS), image_of(blk, kImZK)};
    copy_tiles(cbar, 3, dst, src);
  }
  if (hf == 0) stage_rows<16>(F0, q + row0, rs, nt, nullptr, t);
  scan_gates(gates, sc, sbt, swt);
  bool ok = mbar_wait_warp(cbar, 0, abortp);
  const bool copied = ok;  // thread 0: the copies landed (else the drain waits for them)
  fence_proxy_async_smem();
  if (__syncthreads_or(!ok)) ok = false;
  if (ok && tid == 0) {  // Q K^T -> 0, Q S^T -> 128, ZK S^T -> 256
    tc_fence_after();
    mma_group(tb + 0, F0, F1, false, false);
    mma_group(tb + 128, F0, F2, false, false);
    mma_group(tb + 256, F3, F2, false, false);
    mma_commit(smem_u32(&bars[0]));
  }
  if (ok) ok = mbar_wait_warp(smem_u32(&bars[0]), 0, abortp);
  if (!__syncthreads_or(!ok)) {
    tc_fence_after();
    const float ct = sc[t], gt = expf(ct);
    const float* e0b = blk + (int64_t)kE0 * kTileElems;
#pragma unroll 1
    for (int cb = cb0; cb < cb0 + 2; ++cb) {
      uint32_t t32[32];
      float f32[32];
      // P row t over Q (F0)
      tmem_ld32(tb + lane_off + 0 + cb * 32, t32);
      tmem_wait_ld_r(t32);
#pragma unroll
      for (int xx = 0; xx < 32; ++xx) {
        const int s = cb * 32 + xx;
        f32[xx] = s <= t ? __expf(ct - sc[s]) * __uint_as_float(t32[xx]) : 0.f;
      }
#pragma unroll
      for (int gg = 0; gg < 4; ++gg) st_shared_v4(F0 + tile_off(t, cb * 4 + gg), pack8(&f32[8 * gg]));
      // E row t = E0 - ZK S^T over K (F1)
      blk_ld32(f32, e0b, t, cb * 32);
      tmem_ld32(tb + lane_off + 256 + cb * 32, t32);
      tmem_wait_ld_r(t32);
#pragma unroll
      for (int xx = 0; xx < 32; ++xx) f32[xx] -= __uint_as_float(t32[xx]);
#pragma unroll
      for (int gg = 0; gg < 4; ++gg) st_shared_v4(F1 + tile_off(t, cb * 4 + gg), pack8(&f32[8 * gg]));
      // gamma_t Q S^T, back into its columns for o = gamma Q S^T + P E
      tmem_ld32(tb + lane_off + 128 + cb * 32, t32);
      tmem_wait_ld_r(t32);
#pragma unroll
      for (int xx = 0; xx < 32; ++xx) t32[xx] = __float_as_uint(gt * __uint_as_float(t32[xx]));
      tmem_st32(tb + lane_off + 128 + cb * 32, t32);
    }
    tmem_wait_st();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {  // + P E -> 128 (E as an N-major B)
      tc_fence_after();
      mma_group(tb + 128, F0, F1, true, true);
      mma_commit(smem_u32(&bars[1]));
    }
    ok = mbar_wait_warp(smem_u32(&bars[1]), 0, abortp);
    if (!__syncthreads_or(!ok)) {
      tc_fence_after();
#pragma unroll 1
      for (int cb = cb0; cb < cb0 + 2; ++cb) {
        uint32_t t32[32];
        float f32[32];
        tmem_ld32(tb + lane_off + 128 + cb * 32, t32);
        tmem_wait_ld_r(t32);
#pragma unroll
        for (int xx = 0; xx < 32; ++xx) f32[xx] = __uint_as_float(t32[xx]);
        row_st32(f32, o + rowt + cb * 32, live);
      }
    }
  }
  if (!ok && tid == 0 && status) atomicOr(status, kStatusTimeout);
  if (tid == 0) {  // drain: the products, and the copies if their wait gave up
    mma_commit(smem_u32(&bars[2]));
    mbar_wait(smem_u32(&bars[2]), 0, never_s);
    if (!copied) mbar_wait(cbar, 0, never_s);
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

namespace {
cudaError_t set_smem_attributes() {
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(gdn_cp_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kPrepSmem)) != cudaSuccess ||
      (e = cudaFuncSetAttribute(gdn_cp_prep_grad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kGrSmem)) != cudaSuccess ||
      (e = cudaFuncSetAttribute(gdn_cp_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kChainSmem)) != cudaSuccess ||
      (e = cudaFuncSetAttribute(gdn_cp_out_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kOutSmem)) != cudaSuccess ||
      (e = cudaFuncSetAttribute(gdn_cp_fwd_out_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kFoSmem)) != cudaSuccess)
    return e;
  return cudaSuccess;
}
bool misaligned(std::initializer_list<const void*> ps) {
  for (const void* p : ps)
    if (reinterpret_cast<uintptr_t>(p) & 15u) return true;
  return false;
}
}  // namespace

// The forward in chunk-parallel form: the forward share of every chunk, the
// state chain per (head, member), then o over all chunks.  ws holds the
// scratch (gdn_cp_workspace_bytes); s0, q, k, v, o and s_final 16-byte aligned.
cudaError_t launch_gdn_cp_fwd(int B, int H, int R, const float* s0, const float* q, const float* k,
                              const float* v, const float* g, const float* beta, float* o,
                              float* s_final, float* ws, uint32_t* status, cudaStream_t st) {
  if (B == 0 || H == 0 || R == 0) return cudaSuccess;
  if (H > 65535 || B > 65535) return cudaErrorInvalidValue;  // grid y and z
  if (misaligned({s0, q, k, v, o, s_final, ws})) return cudaErrorMisalignedAddress;
  const int nch = (R + kC - 1) / kC;
  cudaError_t e;
  if ((e = set_smem_attributes()) != cudaSuccess) return e;
  LaunchScope ls(kKGdnFwd, st);
  gdn_cp_prep_kernel<<<dim3(nch, H, B), kPrepThr, kPrepSmem, st>>>(H, R, nch, k, v, g, beta, ws, status);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  gdn_cp_chain_kernel<<<dim3(H, B), kChThr, kChainSmem, st>>>(H, nch, 0, nch, s0, ws, s_final, status);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  gdn_cp_fwd_out_kernel<<<dim3(nch, H, B), kOutThr, kFoSmem, st>>>(H, R, nch, q, k, g, beta, ws, o,
                                                                  status);
  ls.more_kernels(2);
  return cudaGetLastError();
}

// The backward in chunk-parallel form: the forward share of every chunk
// (unless reuse_forward: the scratch already holds it, from the forward on
// the same inputs), the backward's own terms, the chains (the backward one
// alone under reuse_forward), then the outputs over all chunks.  ws holds
// the scratch; s0, q, k, v, d_o, dq, dk, dv 16-byte aligned.
cudaError_t launch_gdn_cp_bwd(int B, int H, int R, const float* s0, const float* q, const float* k,
                              const float* v, const float* g, const float* beta, const float* d_o,
                              float* dq, float* dk, float* dv, float* dg, float* dbeta, float* ws,
                              bool reuse_forward, uint32_t* status, cudaStream_t st) {
  if (B == 0 || H == 0 || R == 0) return cudaSuccess;
  if (H > 65535 || B > 65535) return cudaErrorInvalidValue;  // grid y and z
  if (misaligned({s0, q, k, v, d_o, dq, dk, dv, ws})) return cudaErrorMisalignedAddress;
  const int nch = (R + kC - 1) / kC;
  cudaError_t e;
  if ((e = set_smem_attributes()) != cudaSuccess) return e;
  LaunchScope ls(kKGdnBwd, st);
  if (!reuse_forward) {
    gdn_cp_prep_kernel<<<dim3(nch, H, B), kPrepThr, kPrepSmem, st>>>(H, R, nch, k, v, g, beta, ws,
                                                                    status);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  gdn_cp_prep_grad_kernel<<<dim3(nch, H, B), kPrepThr, kGrSmem, st>>>(H, R, nch, q, k, g, beta, d_o, ws,
                                                                     status);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  gdn_cp_chain_kernel<<<dim3(H, B), kChThr, kChainSmem, st>>>(H, nch, reuse_forward ? nch : 0, 2 * nch,
                                                             s0, ws, nullptr, status);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  gdn_cp_out_kernel<<<dim3(nch, H, B), kOutThr, kOutSmem, st>>>(H, R, nch, q, k, v, g, beta, d_o, ws,
                                                               nullptr, dq, dk, dv, dg, dbeta, status);
  ls.more_kernels(reuse_forward ? 2 : 3);
  return cudaGetLastError();
}

}  // namespace ls
