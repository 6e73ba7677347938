// Host stand-in for the CUDA runtime header when a kernel's source is run
// on the CPU block emulator (emu_core.h): the qualifiers compile away, the
// vector types are plain structs, and the block built-ins go to the emulator.
#pragma once
#include <cmath>
#include <cstdint>
#include <cstring>

#include "emu_core.h"

#define __global__
#define __device__
#define __host__
#define __forceinline__ inline
#define __restrict__
#define __shared__
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
inline unsigned atomicExch(unsigned* p, unsigned v) {
  const unsigned o = *p;
  *p = v;
  return o;
}
inline void __syncthreads() { emu::syncthreads(); }
inline int __syncthreads_or(int p) { return emu::syncthreads_or(p); }
inline float __shfl_up_sync(unsigned, float x, int off) { return emu::shfl_up(x, off); }
inline int __all_sync(unsigned, int p) { return emu::all_sync(p); }

typedef int cudaError_t;
typedef void* cudaStream_t;

namespace emu {
template <class F>
void run_block(unsigned bx, unsigned by, int n, F body) {
  std::unique_ptr<Block> blk(new Block(n));
  std::memset(blk->tmem, 0xff, sizeof(blk->tmem));  // NaN-like poison: unwritten TMEM shows
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
  g_block = nullptr;
}
}  // namespace emu
