// Tile helpers of the chunkwise gated-DeltaNet kernels: [128 x 128] bf16
// operand tiles in the 128-byte-swizzled K-major layout (two [128 x 64]
// boxes), their shared-memory descriptors, staging from float32 rows, and
// 128 x 128 x 128 tcgen05.mma groups.  One CTA of 128 threads.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ls_tc.cuh"

namespace ls {
namespace gdn {
using namespace tc;

constexpr int kC = 128;   // tokens per chunk: the MMAs' M
constexpr int kD = 128;   // dk = dv
constexpr int kThr = 128;
constexpr uint32_t kBox = kC * 128;   // [128 rows x 64 bf16] box
constexpr uint32_t kTile = 2 * kBox;  // [128 x 128] tile
constexpr int kTileElems = kC * kD;   // also the float32 [128 x 128] block of a chunk

__device__ __forceinline__ uint64_t kdesc(uint32_t tile, int kk) {  // K-major, K step kk of 16
  return sdesc_sw128(tile + (kk >> 2) * kBox + (kk & 3) * 32, 16, 1024);
}
__device__ __forceinline__ uint64_t mndesc(uint32_t tile, int kk) {  // N-major B: K rows 16kk..
  return sdesc_sw128(tile + kk * 16 * 128, kBox, 1024);
}
// byte offset of the 16-byte group gq (columns 8gq .. 8gq+7) of row r
__device__ __forceinline__ uint32_t tile_off(int r, int gq) {
  return (gq >> 3) * kBox + sw128_offset(r, gq & 7);
}
// byte offset of element (r, c)
__device__ __forceinline__ uint32_t elem_off(int r, int c) { return tile_off(r, c >> 3) + (c & 7) * 2; }
__device__ __forceinline__ uint4 pack8(const float* x) {
  return make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]),
                    pack_bf16x2(x[6], x[7]));
}
__device__ __forceinline__ uint16_t bf16_of(float x) { return (uint16_t)(pack_bf16x2(x, 0.f) & 0xffffu); }

// Rows 0..nt-1 of a float32 matrix (row r at src + r * stride, 128 columns)
// into a tile, each row times scale[r] when scale is given; rows nt..127 zero.
// 128 threads.  The shared-memory stores are ordering points for the
// compiler, so each batch of kBatch row pieces is loaded into registers
// before any of it is stored: kBatch global loads in flight, not one.
// tid: the caller's index among the kWorkers threads that stage the tile.
// img, when given, receives the same bytes as the tile (a 32 KB image of it
// in global memory, 16-byte aligned), for a later bulk copy.
template <int kBatch = 8, int kWorkers = kThr>
__device__ __forceinline__ void stage_rows(uint32_t tile, const float* src, int64_t stride, int nt,
                                           const float* scale, int tid = threadIdx.x,
                                           void* img = nullptr) {
  constexpr int kPer = 2048 / kWorkers;  // 16-byte pieces per thread
  static_assert(kPer % kBatch == 0, "batch divides the pieces per thread");
#pragma unroll 1
  for (int it0 = 0; it0 < kPer; it0 += kBatch) {
    float4 a[kBatch], b[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int item = tid + kWorkers * (it0 + j), r = item >> 4, gq = item & 15;
      a[j] = b[j] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (r < nt) {
        const float4* p = reinterpret_cast<const float4*>(src + r * stride + gq * 8);
        a[j] = p[0], b[j] = p[1];
      }
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int item = tid + kWorkers * (it0 + j), r = item >> 4, gq = item & 15;
      const float f = (scale && r < nt) ? scale[r] : 1.f;
      const float x[8] = {a[j].x * f, a[j].y * f, a[j].z * f, a[j].w * f,
                          b[j].x * f, b[j].y * f, b[j].z * f, b[j].w * f};
      const uint4 pk = pack8(x);
      st_shared_v4(tile + tile_off(r, gq), pk);
      if (img) *reinterpret_cast<uint4*>(static_cast<uint8_t*>(img) + tile_off(r, gq)) = pk;
    }
  }
}
// The same rows staged into two tiles at once, row r times scale_a[r] into
// tile_a and times scale_b[r] into tile_b (both scales given): one pass of
// global loads for two scaled copies.
template <int kBatch = 8, int kWorkers = kThr>
__device__ __forceinline__ void stage_rows_pair(uint32_t tile_a, const float* scale_a, uint32_t tile_b,
                                                const float* scale_b, const float* src, int64_t stride,
                                                int nt, int tid = threadIdx.x) {
  constexpr int kPer = 2048 / kWorkers;  // 16-byte pieces per thread
  static_assert(kPer % kBatch == 0, "batch divides the pieces per thread");
#pragma unroll 1
  for (int it0 = 0; it0 < kPer; it0 += kBatch) {
    float4 a[kBatch], b[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int item = tid + kWorkers * (it0 + j), r = item >> 4, gq = item & 15;
      a[j] = b[j] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (r < nt) {
        const float4* p = reinterpret_cast<const float4*>(src + r * stride + gq * 8);
        a[j] = p[0], b[j] = p[1];
      }
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int item = tid + kWorkers * (it0 + j), r = item >> 4, gq = item & 15;
      const float fa = r < nt ? scale_a[r] : 0.f, fb = r < nt ? scale_b[r] : 0.f;
      const float xa[8] = {a[j].x * fa, a[j].y * fa, a[j].z * fa, a[j].w * fa,
                           b[j].x * fa, b[j].y * fa, b[j].z * fa, b[j].w * fa};
      const float xb[8] = {a[j].x * fb, a[j].y * fb, a[j].z * fb, a[j].w * fb,
                           b[j].x * fb, b[j].y * fb, b[j].z * fb, b[j].w * fb};
      st_shared_v4(tile_a + tile_off(r, gq), pack8(xa));
      st_shared_v4(tile_b + tile_off(r, gq), pack8(xb));
    }
  }
}
// D[tmem] (+)= A B^T over K = 128 (eight K steps); B K-major or N-major.
__device__ __forceinline__ void mma_group(uint32_t d, uint32_t a, uint32_t b, bool b_mn, bool acc) {
  const uint32_t id = idesc_bf16(128, 128, b_mn);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    mma_ss(d, kdesc(a, kk), b_mn ? mndesc(b, kk) : kdesc(b, kk), id, (acc || kk > 0) ? 1u : 0u);
}
// The same with A read M-major (a tile whose row s holds column s of A), so
// one tile serves as A in K-major form for one product and as A^T in M-major
// form for another.
__device__ __forceinline__ void mma_group_amn(uint32_t d, uint32_t a, uint32_t b, bool b_mn, bool acc) {
  const uint32_t id = idesc_bf16(128, 128, b_mn, true);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    mma_ss(d, mndesc(a, kk), b_mn ? mndesc(b, kk) : kdesc(b, kk), id, (acc || kk > 0) ? 1u : 0u);
}
// Column sums of a [32 x 32] block held one row per lane (v[c] = column c of
// the lane's row): after the five halving exchange rounds (31 shuffles) lane
// l holds the sum of column l over the warp's 32 rows.  v is overwritten.
__device__ __forceinline__ float warp_colsum32(float (&v)[32]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const bool upper = (lane & w) != 0;
#pragma unroll
    for (int c = 0; c < w; ++c) {
      const float send = upper ? v[c] : v[c + w];
      const float keep = upper ? v[c + w] : v[c];
      v[c] = keep + __shfl_xor_sync(0xffffffffu, send, w);
    }
  }
  return v[0];
}
}  // namespace gdn
}  // namespace ls
