// CPU emulation of one CUDA thread block, for running a tensor-core kernel's
// source on the host in tests.  Every CUDA thread is a std::thread; block
// and warp barriers are std::barrier; shared memory, tensor memory and
// mbarriers are host arrays.  tcgen05.mma runs synchronously in the issuing
// thread, so a commit completes its mbarrier phase at once.  Shared-memory
// operand tiles are read through the descriptor layouts the library's
// kernels use (128-byte swizzle; K-major with 1024-byte atom stride, or
// MN-major with the 64-element group stride in the leading-byte offset).
// What this checks: indexing, phase order, barrier protocol and tensor-memory
// lane rules of the kernel source, under that reading of the layouts.  What
// it does not: timing, proxy-ordering races, or hardware behaviour outside it.
#pragma once
#include <atomic>
#include <barrier>
#include <chrono>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <memory>
#include <mutex>
#include <thread>
#include <vector>

namespace emu {

constexpr size_t kSmemBytes = 240 * 1024;
constexpr int kTmemLanes = 128, kTmemCols = 512;

[[noreturn]] inline void die(const char* what, long a = 0, long b = 0) {
  std::fprintf(stderr, "emulator: %s (%ld, %ld)\n", what, a, b);
  std::fflush(stderr);
  std::abort();
}

struct Mbar {
  uint32_t addr = 0, count = 1;
  std::atomic<uint32_t> phase{0}, pending{1};
};

struct Block {
  explicit Block(int n) : nthreads(n), bar(n) {
    for (int w = 0; w < (n + 31) / 32; ++w) warp_bar.emplace_back(new std::barrier<>(32));
  }
  int nthreads;
  std::barrier<> bar;
  std::vector<std::unique_ptr<std::barrier<>>> warp_bar;
  float warp_f[32][32];
  int warp_i[32][32];
  std::atomic<int> or_acc{0};
  std::mutex mu;
  Mbar mbars[16];
  int n_mbars = 0;
  uint32_t tmem[kTmemLanes][kTmemCols];
  bool tmem_allocated = false;
};

inline Block* g_block = nullptr;
inline unsigned char* g_smem = nullptr;  // the kernel's dynamic shared memory
inline thread_local int t_tid = 0;

inline uint32_t smem_addr(const void* p) {
  const auto d = reinterpret_cast<const unsigned char*>(p) - g_smem;
  if (d < 0 || (size_t)d >= kSmemBytes) die("pointer outside shared memory", (long)d);
  return (uint32_t)d;
}
inline unsigned char* smem_ptr(uint32_t addr, uint32_t bytes) {
  if ((size_t)addr + bytes > kSmemBytes) die("shared-memory access out of range", addr, bytes);
  if (addr % bytes) die("misaligned shared-memory access", addr, bytes);
  return g_smem + addr;
}

// ------------------------------------------------------------ barriers
inline void syncthreads() { g_block->bar.arrive_and_wait(); }
inline int syncthreads_or(int p) {
  Block& b = *g_block;
  b.bar.arrive_and_wait();
  if (p) b.or_acc.fetch_or(1);
  b.bar.arrive_and_wait();
  const int r = b.or_acc.load();
  b.bar.arrive_and_wait();
  if (t_tid == 0) b.or_acc.store(0);
  b.bar.arrive_and_wait();
  return r;
}
inline float shfl_up(float x, int off) {
  Block& b = *g_block;
  const int w = t_tid >> 5, l = t_tid & 31;
  b.warp_f[w][l] = x;
  b.warp_bar[w]->arrive_and_wait();
  const float y = l >= off ? b.warp_f[w][l - off] : x;
  b.warp_bar[w]->arrive_and_wait();
  return y;
}
inline int all_sync(int p) {
  Block& b = *g_block;
  const int w = t_tid >> 5, l = t_tid & 31;
  b.warp_i[w][l] = p ? 1 : 0;
  b.warp_bar[w]->arrive_and_wait();
  int r = 1;
  for (int i = 0; i < 32; ++i) r &= b.warp_i[w][i];
  b.warp_bar[w]->arrive_and_wait();
  return r;
}

// ------------------------------------------------------------ mbarriers
inline Mbar& mbar_at(uint32_t addr) {
  Block& b = *g_block;
  std::lock_guard<std::mutex> lk(b.mu);
  for (int i = 0; i < b.n_mbars; ++i)
    if (b.mbars[i].addr == addr) return b.mbars[i];
  die("mbarrier used before mbarrier.init", addr);
}
inline void mbar_init(uint32_t addr, uint32_t count) {
  Block& b = *g_block;
  std::lock_guard<std::mutex> lk(b.mu);
  if (addr & 7) die("misaligned mbarrier", addr);
  if (b.n_mbars == 16) die("too many mbarriers");
  Mbar& m = b.mbars[b.n_mbars++];
  m.addr = addr, m.count = count;
  m.phase = 0, m.pending = count;
}
inline void mbar_arrive(uint32_t addr) {
  Mbar& m = mbar_at(addr);
  if (m.pending.fetch_sub(1) == 1) {
    m.pending = m.count;
    m.phase.fetch_add(1);
  }
}
// Succeeds once the phase with the given parity has completed; gives up after
// 5 s, as the kernels' bounded waits do.
inline bool mbar_wait(uint32_t addr, uint32_t parity) {
  Mbar& m = mbar_at(addr);
  const auto t0 = std::chrono::steady_clock::now();
  while ((m.phase.load() & 1u) == (parity & 1u)) {
    if (std::chrono::steady_clock::now() - t0 > std::chrono::seconds(5)) return false;
    std::this_thread::yield();
  }
  return true;
}

// ------------------------------------------------------------ bf16
inline uint32_t bf16_bits(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0x7fc0u;  // NaN
  u += 0x7fffu + ((u >> 16) & 1u);                       // round to nearest even
  return u >> 16;
}
inline float bf16_float(uint32_t h) {
  const uint32_t u = (h & 0xffffu) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// ------------------------------------------------------------ tensor memory
inline void tmem_alloc(uint32_t dst, uint32_t ncols) {
  Block& b = *g_block;
  if ((t_tid & 31) != 0) return;
  if (ncols != 512 && ncols != 256 && ncols != 128 && ncols != 64 && ncols != 32)
    die("tcgen05.alloc: column count", ncols);
  if (b.tmem_allocated) die("tcgen05.alloc twice");
  b.tmem_allocated = true;
  const uint32_t base = 0;
  std::memcpy(smem_ptr(dst, 4), &base, 4);
}
inline void tmem_dealloc() {
  if ((t_tid & 31) == 0) g_block->tmem_allocated = false;
}
inline void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  Block& b = *g_block;
  const int warp = t_tid >> 5;
  const uint32_t lane0 = taddr >> 16, col = taddr & 0xffffu;
  if (lane0 != (uint32_t)(32 * (warp % 4))) die("tcgen05.ld: warp reads another lane quarter", warp, lane0);
  if (col + 32 > (uint32_t)kTmemCols) die("tcgen05.ld: column out of range", col);
  const uint32_t lane = lane0 + (t_tid & 31);
  for (int i = 0; i < 32; ++i) r[i] = b.tmem[lane][col + i];
}

// ------------------------------------------------------------ MMA
// Byte address of element (row, k) of an operand (row = M for A, N for B).
inline uint32_t operand_addr(uint64_t desc, bool mn_major, int row, int k) {
  const uint32_t start = (uint32_t)(desc & 0x3fffu) << 4;
  const uint32_t lbo = (uint32_t)((desc >> 16) & 0x3fffu) << 4;
  const uint32_t sbo = (uint32_t)((desc >> 32) & 0x3fffu) << 4;
  if (((desc >> 61) & 7u) != 2u) die("only the 128-byte swizzle is emulated");
  uint32_t a;
  if (!mn_major)  // rows of 128 bytes along K; 8-row atoms SBO apart
    a = start + (uint32_t)(row / 8) * sbo + (uint32_t)(row % 8) * 128u + (uint32_t)k * 2u;
  else  // 64-element groups of the M/N index LBO apart; K rows of 128 bytes, 8-row atoms SBO apart
    a = start + (uint32_t)(row / 64) * lbo + (uint32_t)(k / 8) * sbo + (uint32_t)(k % 8) * 128u +
        (uint32_t)(row % 64) * 2u;
  return a ^ (((a >> 7) & 7u) << 4);
}
// tcgen05.mma.cta_group::1.kind::f16, bf16 A/B from shared memory, f32 D.
inline void mma_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
  Block& b = *g_block;
  if (!b.tmem_allocated) die("tcgen05.mma without tensor memory");
  const int M = (int)((idesc >> 24) & 0x1fu) << 4, N = (int)((idesc >> 17) & 0x3fu) << 3;
  const bool a_mn = (idesc >> 15) & 1u, b_mn = (idesc >> 16) & 1u;
  if (((idesc >> 4) & 3u) != 1u || ((idesc >> 7) & 7u) != 1u || ((idesc >> 10) & 7u) != 1u)
    die("idesc: only bf16 x bf16 -> f32 is emulated", idesc);
  if (M != 128) die("only M = 128 is emulated", M);
  const uint32_t lane0 = d_tmem >> 16, col0 = d_tmem & 0xffffu;
  if (lane0 != 0 || col0 + N > (uint32_t)kTmemCols) die("MMA accumulator out of range", lane0, col0);
  float av[128][16], bv[256][16];
  for (int m = 0; m < M; ++m)
    for (int k = 0; k < 16; ++k) {
      uint16_t h;
      std::memcpy(&h, smem_ptr(operand_addr(adesc, a_mn, m, k), 2), 2);
      av[m][k] = bf16_float(h);
    }
  for (int n = 0; n < N; ++n)
    for (int k = 0; k < 16; ++k) {
      uint16_t h;
      std::memcpy(&h, smem_ptr(operand_addr(bdesc, b_mn, n, k), 2), 2);
      bv[n][k] = bf16_float(h);
    }
  for (int m = 0; m < M; ++m)
    for (int n = 0; n < N; ++n) {
      float s = 0.f;
      if (acc) std::memcpy(&s, &b.tmem[m][col0 + n], 4);
      for (int k = 0; k < 16; ++k) s = std::fma(av[m][k], bv[n][k], s);
      std::memcpy(&b.tmem[m][col0 + n], &s, 4);
    }
}

// ------------------------------------------------------------ launch
// Runs body() once per thread of one block of n threads.
template <class F>
void run_block(unsigned bx, unsigned by, int n, F body);

}  // namespace emu
