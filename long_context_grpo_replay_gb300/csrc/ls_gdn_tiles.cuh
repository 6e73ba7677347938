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
// One row of a tile from 128 registers (thread = row).
__device__ __forceinline__ void stage_row_regs(uint32_t tile, int r, const float (&x)[kD]) {
#pragma unroll
  for (int gq = 0; gq < 16; ++gq) st_shared_v4(tile + tile_off(r, gq), pack8(&x[8 * gq]));
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
// ---- thread-per-row code and coalesced global rows.  The 32 threads of a
// warp own 32 consecutive rows; a [32 rows x 32 columns] float block moves
// between global memory and their registers through a padded [32 x 33]
// shared-memory scratch of the warp, so every global access is one 128-byte
// row segment (one row per warp instruction) instead of 32 rows' scattered
// words.  Rows at or past nvalid (relative to the block) read as 0 / are not
// written.  base points to the block's element (0, 0); row r at base + r * stride.
// v: 32 consecutive values of the thread's row (registers when the caller's
// indices are compile-time constants).
__device__ __forceinline__ void rows_load32(float* v, const float* base, int64_t stride, int nvalid,
                                            float* scr) {
  const int lane = threadIdx.x & 31;
  float tmp[32];  // all 32 loads issued before the first shared store
#pragma unroll
  for (int r = 0; r < 32; ++r) tmp[r] = r < nvalid ? base[r * stride + lane] : 0.f;
#pragma unroll
  for (int r = 0; r < 32; ++r) scr[r * 33 + lane] = tmp[r];
  __syncwarp();
#pragma unroll
  for (int c = 0; c < 32; ++c) v[c] = scr[lane * 33 + c];
  __syncwarp();
}
__device__ __forceinline__ void rows_store32(const float* v, float* base, int64_t stride, int nvalid,
                                             float* scr) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int c = 0; c < 32; ++c) scr[lane * 33 + c] = v[c];
  __syncwarp();
#pragma unroll 4
  for (int r = 0; r < 32; ++r)
    if (r < nvalid) base[r * stride + lane] = scr[r * 33 + lane];
  __syncwarp();
}
// The same for rows r0 .. r0+31 of a packed strict lower triangle (row t at
// t (t - 1) / 2), columns c0 .. c0+31: v[c] = element (r0 + lane, c0 + c).
// Entries on or above the diagonal come out as whatever the packing holds
// there (the caller masks them); every read stays below row 128's start.
__device__ __forceinline__ void rows_load32_packed(float* v, const float* packed, int r0, int c0,
                                                   float* scr) {
  const int lane = threadIdx.x & 31;
  float tmp[32];
#pragma unroll
  for (int r = 0; r < 32; ++r) tmp[r] = packed[(r0 + r) * (r0 + r - 1) / 2 + c0 + lane];
#pragma unroll
  for (int r = 0; r < 32; ++r) scr[r * 33 + lane] = tmp[r];
  __syncwarp();
#pragma unroll
  for (int c = 0; c < 32; ++c) v[c] = scr[lane * 33 + c];
  __syncwarp();
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
// Words of the per-warp row scratch (32 x 33 floats per warp, four warps).
constexpr int kRowScrFloats = 4 * 32 * 33;

// fp32 [128 x 128] shared buffer, columns XOR-swizzled by the row: row
// writes (thread = row) and column reads (thread = column) are both free of
// bank conflicts.
__device__ __forceinline__ int u_at(int t, int j) { return t * kD + (j ^ (t & 31)); }
// packed strict lower triangle
__device__ __forceinline__ int a_at(int t, int s) { return t * (t - 1) / 2 + s; }

}  // namespace gdn
}  // namespace ls
