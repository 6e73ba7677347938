// Host stand-in for the CUDA runtime header when a kernel's source is run
// on the CPU block emulator (emu_core.h): the qualifiers compile away
// (__shared__ objects become function statics, shared by the block's
// threads), the vector types are plain structs, and the block built-ins go
// to the emulator.  A kernel's "extern __shared__" array is declared by the
// test harness, which rewrites that line to "extern".
#pragma once
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "emu_core.h"

#define __global__
#define __device__
#define __host__
#define __forceinline__ inline
#define __restrict__
#define __shared__ static
#define __grid_constant__
#define __launch_bounds__(...)

struct dim3 {
  unsigned x = 0, y = 0, z = 0;
};
inline thread_local dim3 threadIdx, blockIdx;

struct alignas(8) float2 {
  float x, y;
};
struct alignas(16) float4 {
  float x, y, z, w;
};
struct alignas(16) uint4 {
  unsigned x, y, z, w;
};
inline float4 make_float4(float x, float y, float z, float w) { return {x, y, z, w}; }
inline uint4 make_uint4(unsigned x, unsigned y, unsigned z, unsigned w) { return {x, y, z, w}; }

inline float __uint_as_float(unsigned u) {
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}
inline float __int_as_float(int i) {
  float f;
  std::memcpy(&f, &i, 4);
  return f;
}
inline unsigned __float_as_uint(float f) {
  unsigned u;
  std::memcpy(&u, &f, 4);
  return u;
}
inline float __log2f(float x) { return std::log2(x); }
inline float __expf(float x) { return std::exp(x); }
template <class T>
inline T __ldg(const T* p) {
  return *p;
}
inline unsigned atomicExch(unsigned* p, unsigned v) {
  return std::atomic_ref<unsigned>(*p).exchange(v);
}
inline unsigned atomicOr(unsigned* p, unsigned v) { return std::atomic_ref<unsigned>(*p).fetch_or(v); }
inline unsigned atomicCAS(unsigned* p, unsigned cmp, unsigned v) {
  std::atomic_ref<unsigned>(*p).compare_exchange_strong(cmp, v);
  return cmp;
}
inline float atomicAdd(float* p, float v) { return std::atomic_ref<float>(*p).fetch_add(v); }
inline void __syncthreads() { emu::syncthreads(); }
inline int __syncthreads_or(int p) { return emu::syncthreads_or(p); }
inline void __syncwarp(unsigned = 0xffffffffu) { emu::syncwarp(); }
inline float __shfl_up_sync(unsigned, float x, int off) { return emu::shfl_up(x, off); }
inline float __shfl_xor_sync(unsigned, float x, int mask) { return emu::shfl_xor(x, mask); }
inline float __shfl_down_sync(unsigned, float x, int off) { return emu::shfl_down(x, off); }
inline int __all_sync(unsigned, int p) { return emu::all_sync(p); }
inline int __any_sync(unsigned, int p) { return emu::any_sync(p); }

typedef int cudaError_t;
typedef void* cudaStream_t;
enum { cudaSuccess = 0, cudaErrorInvalidValue = 1, cudaErrorMisalignedAddress = 74 };

namespace emu {
// Runs body() on every thread of one block of n threads.
template <class F>
void run_block(unsigned bx, unsigned by, int n, F body, unsigned seed = 1) {
  std::unique_ptr<Block> blk(new Block(n, seed));
  std::memset(blk->tmem, 0xff, sizeof(blk->tmem));  // poison: unwritten tensor memory shows
  g_block = blk.get();
  std::vector<std::thread> ts;
  for (int t = 0; t < n; ++t)
    ts.emplace_back([=, &body] {
      threadIdx.x = (unsigned)t;
      blockIdx.x = bx, blockIdx.y = by;
      t_tid = t;
      body();
    });
  for (auto& t : ts) t.join();
  if (blk->tmem_allocated) die("tensor memory not freed at the end of the block");
  blk.reset();  // drains the engines while the block is still current
  g_block = nullptr;
}
// The same for a block with a three-dimensional index.
template <class F>
void run_block3(unsigned bx, unsigned by, unsigned bz, int n, F body, unsigned seed = 1) {
  run_block(bx, by, n, [&] { blockIdx.z = bz; body(); }, seed);
}
}  // namespace emu
