// The PTX building blocks of the tensor-core kernels, emulated on the host
// (CPU block emulator, emu_core.h).  Same names and encodings as the device
// versions; the descriptor and instruction-descriptor bit layouts are the
// library's, so the emulator decodes exactly what the kernel encodes.
#pragma once
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

namespace ls {
namespace tc {

inline uint32_t smem_u32(const void* p) { return emu::smem_addr(p); }
inline void mbar_init(uint32_t bar, uint32_t count) { emu::mbar_init(bar, count); }
inline void fence_mbar_init() {}
inline bool mbar_wait(uint32_t bar, uint32_t parity, const volatile uint32_t*) {
  return emu::mbar_wait(bar, parity);
}
inline bool mbar_wait_warp(uint32_t bar, uint32_t parity, const volatile uint32_t* abort) {
  const bool ok = mbar_wait(bar, parity, abort);
  return __all_sync(0xffffffffu, ok) != 0;
}
inline void fence_proxy_async_smem() {}
inline void tmem_alloc(uint32_t dst, uint32_t ncols) { emu::tmem_alloc(dst, ncols); }
inline void tmem_relinquish() {}
inline void tmem_dealloc(uint32_t, uint32_t) { emu::tmem_dealloc(); }
inline void tc_fence_before() {}
inline void tc_fence_after() {}

constexpr uint32_t idesc_bf16(int M, int N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
inline uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
inline void mma_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                   uint32_t accumulate) {
  emu::mma_ss(d_tmem, adesc, bdesc, idesc, accumulate);
}
inline void mma_commit(uint32_t bar) { emu::mbar_arrive(bar); }
inline void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) { emu::tmem_ld32(taddr, r); }
inline void tmem_wait_ld_r(uint32_t (&)[32]) {}
inline void reg_dep(uint32_t (&)[32]) {}
inline uint32_t sw128_offset(uint32_t row, uint32_t chunk) {
  return row * 128u + (((chunk ^ (row & 7u)) & 7u) << 4);
}
inline uint32_t pack_bf16x2(float lo, float hi) {
  return emu::bf16_bits(lo) | (emu::bf16_bits(hi) << 16);
}
inline float2 unpack_bf16x2(uint32_t u) { return {emu::bf16_float(u), emu::bf16_float(u >> 16)}; }
inline uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  std::memcpy(&v, emu::smem_ptr(addr, 16), 16);
  return v;
}
inline void st_shared_v4(uint32_t addr, uint4 v) { std::memcpy(emu::smem_ptr(addr, 16), &v, 16); }

}  // namespace tc
}  // namespace ls
