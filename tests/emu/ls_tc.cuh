// The PTX building blocks of the tensor-core kernels, emulated on the host
// (CPU block emulator, emu_core.h).  Same names and encodings as the device
// versions; the descriptor and instruction-descriptor bit layouts are the
// library's, so the emulator decodes exactly what the kernel encodes.
#pragma once
#include <cuda.h>
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

constexpr uint32_t idesc_bf16(int M, int N, bool b_mn_major, bool a_mn_major = false) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
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
  emu::mma(d_tmem, adesc, -1, bdesc, idesc, accumulate);
}
inline void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                   uint32_t accumulate) {
  emu::mma(d_tmem, 0, (int64_t)a_tmem, bdesc, idesc, accumulate);
}
inline void mma_commit(uint32_t bar) { emu::mma_commit(bar); }
inline void mbar_arrive(uint32_t bar) { emu::mbar_arrive(bar); }
inline void mbar_expect_tx(uint32_t bar, uint32_t bytes) { emu::mbar_expect_tx(bar, bytes); }
inline void prefetch_tmap(const CUtensorMap*) {}
inline void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  emu::bulk_load(dst, src, bytes, bar);
}
inline void prefetch_l2(const void* p, uint32_t bytes) {  // a hint: only its arguments are checked
  if (reinterpret_cast<uintptr_t>(p) % 16 || bytes % 16 || bytes == 0) emu::die("L2 prefetch arguments", bytes);
}
inline void tma_load_2d(uint32_t dst, const CUtensorMap* m, uint32_t bar, int32_t c0, int32_t c1) {
  const int32_t c[2] = {c0, c1};
  emu::tma_load(dst, m, bar, c);
}
inline void tma_load_3d(uint32_t dst, const CUtensorMap* m, uint32_t bar, int32_t c0, int32_t c1,
                        int32_t c2) {
  const int32_t c[3] = {c0, c1, c2};
  emu::tma_load(dst, m, bar, c);
}
inline void tma_load_4d(uint32_t dst, const CUtensorMap* m, uint32_t bar, int32_t c0, int32_t c1,
                        int32_t c2, int32_t c3) {
  const int32_t c[4] = {c0, c1, c2, c3};
  emu::tma_load(dst, m, bar, c);
}
inline void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) { emu::tmem_ld(taddr, r, 32); }
inline void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) { emu::tmem_st(taddr, r, 32); }
inline void tmem_st16(uint32_t taddr, const uint32_t* r) { emu::tmem_st(taddr, r, 16); }
inline void tmem_st1(uint32_t taddr, uint32_t v) { emu::tmem_st(taddr, &v, 1); }
inline void tmem_ld1x2(uint32_t a0, uint32_t a1, uint32_t& a, uint32_t& b) {
  emu::tmem_ld(a0, &a, 1);
  emu::tmem_ld(a1, &b, 1);
}
inline void tmem_wait_ld() {}
inline void tmem_wait_st() {}
inline void named_bar_sync(uint32_t id, uint32_t n) { emu::named_bar_sync(id, n); }
inline void tmem_wait_ld_r(uint32_t (&)[32]) {}
inline void reg_dep(uint32_t (&)[32]) {}
inline uint32_t sw128_offset(uint32_t row, uint32_t chunk) {
  return row * 128u + (((chunk ^ (row & 7u)) & 7u) << 4);
}
inline uint32_t pack_bf16x2(float lo, float hi) {
  return emu::bf16_bits(lo) | (emu::bf16_bits(hi) << 16);
}
inline float2 unpack_bf16x2(uint32_t u) { return {emu::bf16_float(u), emu::bf16_float(u >> 16)}; }
// packed float32 pairs: lane 0 in the low word, each lane rounded as the
// scalar operation
inline uint64_t f2(float lo, float hi) { return (uint64_t)__float_as_uint(lo) | ((uint64_t)__float_as_uint(hi) << 32); }
inline void f2_split(uint64_t r, float& lo, float& hi) {
  lo = __uint_as_float((uint32_t)r);
  hi = __uint_as_float((uint32_t)(r >> 32));
}
inline uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  float a0, a1, b0, b1, c0, c1;
  f2_split(a, a0, a1), f2_split(b, b0, b1), f2_split(c, c0, c1);
  return f2(std::fma(a0, b0, c0), std::fma(a1, b1, c1));
}
inline uint64_t f2_add(uint64_t a, uint64_t b) {
  float a0, a1, b0, b1;
  f2_split(a, a0, a1), f2_split(b, b0, b1);
  return f2(a0 + b0, a1 + b1);
}
inline uint64_t f2_mul(uint64_t a, uint64_t b) {
  float a0, a1, b0, b1;
  f2_split(a, a0, a1), f2_split(b, b0, b1);
  return f2(a0 * b0, a1 * b1);
}
inline uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  std::memcpy(&v, emu::smem_ptr(addr, 16), 16);
  return v;
}
inline void st_shared_v4(uint32_t addr, uint4 v) { std::memcpy(emu::smem_ptr(addr, 16), &v, 16); }
inline void st_shared_u16(uint32_t addr, uint16_t v) { std::memcpy(emu::smem_ptr(addr, 2), &v, 2); }

}  // namespace tc
}  // namespace ls
