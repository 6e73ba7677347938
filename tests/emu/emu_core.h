// CPU emulation of one CUDA thread block, for running a tensor-core kernel's
// source on the host in tests.  Every CUDA thread is a std::thread; block
// and warp barriers are std::barrier; shared memory, tensor memory and
// mbarriers are host state.  tcgen05.mma / tcgen05.commit and TMA copies run
// asynchronously, in issue order, on two engine threads (one for the tensor
// core, one for the copy engine) with random delays, so that a kernel which
// reads a result before waiting for it, or overwrites an operand that an
// issued MMA has not read yet, sees wrong data.  Shared-memory operand tiles
// are read through the descriptor layouts the library's kernels use
// (128-byte swizzle; K-major with the 1024-byte atom stride, or MN-major with
// the 64-element group stride in the leading-byte offset); TMA boxes land in
// the same swizzled layout.  What this checks: indexing, phase order, barrier
// protocol and tensor-memory lane rules of the kernel source, under that
// reading of the layouts.  What it does not: timing, the memory model beyond
// these orderings, or hardware behaviour outside it.
#pragma once
#include <atomic>
#include <barrier>
#include <chrono>
#include <cmath>
#include <condition_variable>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <deque>
#include <functional>
#include <memory>
#include <mutex>
#include <random>
#include <thread>
#include <vector>

namespace emu {

constexpr size_t kSmemBytes = 240 * 1024;
constexpr uint32_t kStaticBase = 0x40000;  // addresses of static __shared__ objects
constexpr int kTmemLanes = 128, kTmemCols = 512;

[[noreturn]] inline void die(const char* what, long a = 0, long b = 0) {
  std::fprintf(stderr, "emulator: %s (%ld, %ld)\n", what, a, b);
  std::fflush(stderr);
  std::abort();
}

// In-order asynchronous executor with random delays.
class Engine {
 public:
  explicit Engine(unsigned seed) : rng_(seed), th_([this] { loop(); }) {}
  ~Engine() {
    {
      std::lock_guard<std::mutex> lk(mu_);
      stop_ = true;
    }
    cv_.notify_all();
    th_.join();
  }
  void push(std::function<void()> f) {
    {
      std::lock_guard<std::mutex> lk(mu_);
      q_.push_back(std::move(f));
    }
    cv_.notify_all();
  }

 private:
  void loop() {
    for (;;) {
      std::function<void()> f;
      {
        std::unique_lock<std::mutex> lk(mu_);
        cv_.wait(lk, [&] { return stop_ || !q_.empty(); });
        if (q_.empty()) return;
        f = std::move(q_.front());
        q_.pop_front();
      }
      if (rng_() % 4 == 0) std::this_thread::sleep_for(std::chrono::microseconds(rng_() % 50));
      f();
    }
  }
  std::mt19937 rng_;
  std::mutex mu_;
  std::condition_variable cv_;
  std::deque<std::function<void()>> q_;
  bool stop_ = false;
  std::thread th_;
};

struct Mbar {
  uint32_t addr = 0, count = 1;
  int pending = 1;
  int64_t tx = 0;
  std::atomic<uint32_t> phase{0};
};

struct Block {
  explicit Block(int n, unsigned seed) : nthreads(n), bar(n), tensor(seed), copy(seed * 7 + 1) {
    for (int w = 0; w < (n + 31) / 32; ++w) warp_bar.emplace_back(new std::barrier<>(32));
  }
  int nthreads;
  std::barrier<> bar;
  std::vector<std::unique_ptr<std::barrier<>>> warp_bar;
  float warp_f[32][32];
  int warp_i[32][32];
  std::atomic<int> or_acc{0};
  std::mutex mu;  // mbarriers and the static-shared registry
  Mbar mbars[32];
  int n_mbars = 0;
  std::vector<std::pair<const void*, uint32_t>> statics;
  uint32_t tmem[kTmemLanes][kTmemCols];
  bool tmem_allocated = false;
  std::unique_ptr<std::barrier<>> named[16];  // bar.sync id, n (id 1..15), made on first use
  uint32_t named_n[16] = {};
  Engine tensor, copy;  // declared last: destroyed (drained) first
};

inline Block* g_block = nullptr;
inline unsigned char* g_smem = nullptr;  // the kernel's dynamic shared memory
inline thread_local int t_tid = 0;

// ------------------------------------------------------------ shared memory
inline uint32_t smem_addr(const void* p) {
  const auto d = reinterpret_cast<const unsigned char*>(p) - g_smem;
  if (d >= 0 && (size_t)d < kSmemBytes) return (uint32_t)d;
  Block& b = *g_block;  // a static __shared__ object: give it an address of its own
  std::lock_guard<std::mutex> lk(b.mu);
  for (auto& e : b.statics)
    if (e.first == p) return e.second;
  const uint32_t a = kStaticBase + 16u * (uint32_t)b.statics.size();
  b.statics.emplace_back(p, a);
  return a;
}
inline unsigned char* smem_ptr(uint32_t addr, uint32_t bytes) {
  if (addr % bytes) die("misaligned shared-memory access", addr, bytes);
  if (addr < kSmemBytes) {
    if ((size_t)addr + bytes > kSmemBytes) die("shared-memory access out of range", addr, bytes);
    return g_smem + addr;
  }
  Block& b = *g_block;
  std::lock_guard<std::mutex> lk(b.mu);
  for (auto& e : b.statics)
    if (e.second == addr) return (unsigned char*)e.first;
  die("access to an unknown shared address", addr);
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
inline void syncwarp() { g_block->warp_bar[t_tid >> 5]->arrive_and_wait(); }
// A named barrier among n threads (whole warps); every use of one id must
// name the same count.
inline void named_bar_sync(uint32_t id, uint32_t n) {
  Block& b = *g_block;
  if (id == 0 || id >= 16 || n == 0 || n % 32 || (int)n > b.nthreads) die("named barrier", id, n);
  std::barrier<>* br;
  {
    std::lock_guard<std::mutex> lk(b.mu);
    if (!b.named[id]) {
      b.named[id].reset(new std::barrier<>(n));
      b.named_n[id] = n;
    } else if (b.named_n[id] != n) {
      die("named barrier used with two thread counts", id, n);
    }
    br = b.named[id].get();
  }
  br->arrive_and_wait();
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

inline float shfl_down(float x, int off) {
  Block& b = *g_block;
  const int w = t_tid >> 5, l = t_tid & 31;
  b.warp_f[w][l] = x;
  b.warp_bar[w]->arrive_and_wait();
  const float y = l + off < 32 ? b.warp_f[w][l + off] : x;
  b.warp_bar[w]->arrive_and_wait();
  return y;
}
inline float shfl_xor(float x, int mask) {
  Block& b = *g_block;
  const int w = t_tid >> 5, l = t_tid & 31;
  b.warp_f[w][l] = x;
  b.warp_bar[w]->arrive_and_wait();
  const float y = b.warp_f[w][l ^ mask];
  b.warp_bar[w]->arrive_and_wait();
  return y;
}
inline int any_sync(int p) {
  Block& b = *g_block;
  const int w = t_tid >> 5, l = t_tid & 31;
  b.warp_i[w][l] = p ? 1 : 0;
  b.warp_bar[w]->arrive_and_wait();
  int r = 0;
  for (int i = 0; i < 32; ++i) r |= b.warp_i[w][i];
  b.warp_bar[w]->arrive_and_wait();
  return r;
}

// ------------------------------------------------------------ mbarriers
// An mbarrier in dynamic shared memory keeps this word in its 8 bytes for the
// emulator's own check: a kernel store that lands on the barrier (an
// overlapping array, say) would corrupt a real barrier's state, and here it
// fails the next operation on it.
constexpr uint64_t kMbarMagic = 0x6d6261725f656d75ull;
inline Mbar& mbar_locked(Block& b, uint32_t addr) {
  for (int i = 0; i < b.n_mbars; ++i)
    if (b.mbars[i].addr == addr) {
      if (addr < kSmemBytes) {
        uint64_t w;
        std::memcpy(&w, g_smem + addr, 8);
        if (w != kMbarMagic) die("an mbarrier in shared memory was overwritten by a store", addr);
      }
      return b.mbars[i];
    }
  die("mbarrier used before mbarrier.init", addr);
}
inline void mbar_init(uint32_t addr, uint32_t count) {
  Block& b = *g_block;
  std::lock_guard<std::mutex> lk(b.mu);
  if (addr & 7) die("misaligned mbarrier", addr);
  if (b.n_mbars == 32) die("too many mbarriers");
  Mbar& m = b.mbars[b.n_mbars++];
  m.addr = addr, m.count = count, m.pending = (int)count, m.tx = 0;
  m.phase = 0;
  if (addr < kSmemBytes) std::memcpy(g_smem + addr, &kMbarMagic, 8);
}
inline void mbar_update_locked(Mbar& m, int arrivals, int64_t tx_add) {
  m.pending -= arrivals;
  m.tx += tx_add;
  if (m.pending < 0) die("mbarrier: more arrivals than its count", m.addr);
  if (m.pending == 0 && m.tx == 0) {
    m.pending = (int)m.count;
    m.phase.fetch_add(1);
  }
}
inline void mbar_arrive(uint32_t addr) {
  Block& b = *g_block;
  std::lock_guard<std::mutex> lk(b.mu);
  mbar_update_locked(mbar_locked(b, addr), 1, 0);
}
inline void mbar_expect_tx(uint32_t addr, uint32_t bytes) {  // expect then arrive
  Block& b = *g_block;
  std::lock_guard<std::mutex> lk(b.mu);
  mbar_update_locked(mbar_locked(b, addr), 1, (int64_t)bytes);
}
inline void mbar_complete_tx(uint32_t addr, uint32_t bytes) {
  Block& b = *g_block;
  std::lock_guard<std::mutex> lk(b.mu);
  mbar_update_locked(mbar_locked(b, addr), 0, -(int64_t)bytes);
}
// Succeeds once the phase with the given parity has completed; gives up after
// 20 s, as the kernels' bounded waits do.
inline bool mbar_wait(uint32_t addr, uint32_t parity) {
  Mbar* m;
  {
    Block& b = *g_block;
    std::lock_guard<std::mutex> lk(b.mu);
    m = &mbar_locked(b, addr);
  }
  const auto t0 = std::chrono::steady_clock::now();
  while ((m->phase.load() & 1u) == (parity & 1u)) {
    if (std::chrono::steady_clock::now() - t0 > std::chrono::seconds(20)) return false;
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
inline uint32_t tmem_lane(uint32_t taddr, uint32_t ncols) {
  const int warp = t_tid >> 5;
  const uint32_t lane0 = taddr >> 16, col = taddr & 0xffffu;
  if (lane0 != (uint32_t)(32 * (warp % 4))) die("tcgen05.ld/st: warp uses another lane quarter", warp, lane0);
  if (col + ncols > (uint32_t)kTmemCols) die("tcgen05.ld/st: column out of range", col);
  return lane0 + (uint32_t)(t_tid & 31);
}
inline void tmem_ld(uint32_t taddr, uint32_t* r, int n) {
  const uint32_t lane = tmem_lane(taddr, n), col = taddr & 0xffffu;
  for (int i = 0; i < n; ++i) r[i] = g_block->tmem[lane][col + i];
}
inline void tmem_st(uint32_t taddr, const uint32_t* r, int n) {
  const uint32_t lane = tmem_lane(taddr, n), col = taddr & 0xffffu;
  for (int i = 0; i < n; ++i) g_block->tmem[lane][col + i] = r[i];
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
inline float smem_bf16(uint32_t addr) {
  uint16_t h;
  std::memcpy(&h, smem_ptr(addr, 2), 2);
  return bf16_float(h);
}
// tcgen05.mma.cta_group::1.kind::f16, bf16 A/B, f32 D; A from shared memory
// (a_tmem < 0) or tensor memory (bf16 pairs, K/2 columns).
inline void mma(uint32_t d_tmem, uint64_t adesc, int64_t a_tmem, uint64_t bdesc, uint32_t idesc,
                uint32_t acc) {
  Block& b = *g_block;
  if (!b.tmem_allocated) die("tcgen05.mma without tensor memory");
  const int M = (int)((idesc >> 24) & 0x1fu) << 4, N = (int)((idesc >> 17) & 0x3fu) << 3;
  const bool a_mn = (idesc >> 15) & 1u, b_mn = (idesc >> 16) & 1u;
  if (((idesc >> 4) & 3u) != 1u || ((idesc >> 7) & 7u) != 1u || ((idesc >> 10) & 7u) != 1u)
    die("idesc: only bf16 x bf16 -> f32 is emulated", idesc);
  if (M != 128) die("only M = 128 is emulated", M);
  if (N < 8 || N > 256 || N % 8) die("MMA N", N);
  const uint32_t lane0 = d_tmem >> 16, col0 = d_tmem & 0xffffu;
  if (lane0 != 0 || col0 + N > (uint32_t)kTmemCols) die("MMA accumulator out of range", lane0, col0);
  b.tensor.push([=, &b] {
    static thread_local float av[128][16], bv[256][16];
    for (int m = 0; m < M; ++m)
      for (int k = 0; k < 16; ++k) {
        if (a_tmem < 0) {
          av[m][k] = smem_bf16(operand_addr(adesc, a_mn, m, k));
        } else {
          const uint32_t ac = (uint32_t)a_tmem & 0xffffu;
          if ((a_tmem >> 16) != 0 || ac + 8 > (uint32_t)kTmemCols) die("MMA A in tensor memory", (long)a_tmem);
          av[m][k] = bf16_float(b.tmem[m][ac + k / 2] >> (16 * (k & 1)));
        }
      }
    for (int n = 0; n < N; ++n)
      for (int k = 0; k < 16; ++k) bv[n][k] = smem_bf16(operand_addr(bdesc, b_mn, n, k));
    for (int m = 0; m < M; ++m)
      for (int n = 0; n < N; ++n) {
        float s = 0.f;
        if (acc) std::memcpy(&s, &b.tmem[m][col0 + n], 4);
        for (int k = 0; k < 16; ++k) s = std::fma(av[m][k], bv[n][k], s);
        std::memcpy(&b.tmem[m][col0 + n], &s, 4);
      }
  });
}
// tcgen05.commit: arrives once every MMA issued before it has completed.
inline void mma_commit(uint32_t bar) {
  g_block->tensor.push([bar] { mbar_arrive(bar); });
}

// ------------------------------------------------------------ TMA
struct TensorMap {  // what cuTensorMapEncodeTiled records, for the copy engine
  const void* base;
  int rank;
  uint64_t dim[5];
  uint64_t stride[5];  // bytes; stride[0] = element size
  uint32_t box[5];
};
// Tiled load with the 128-byte swizzle: the box lands densely (dimension 0
// fastest, 128-byte rows), swizzled within 1024-byte atoms; elements outside
// the tensor read as zero.  Completes `bytes` of transaction on bar.
inline void tma_load(uint32_t dst, const TensorMap* m, uint32_t bar, const int32_t* c) {
  if (dst % 1024) die("TMA destination not 1024-byte aligned", dst);
  if ((c[0] * 2) % 16) die("TMA x coordinate not 16-byte aligned", c[0]);
  const TensorMap map = *m;
  int32_t cc[5] = {0, 0, 0, 0, 0};
  for (int i = 0; i < map.rank; ++i) cc[i] = c[i];
  uint32_t n = 1;
  for (int i = 0; i < map.rank; ++i) n *= map.box[i];
  if (map.box[0] * 2 != 128) die("emulated TMA boxes are 128 bytes wide", map.box[0]);
  g_block->copy.push([=] {
    for (uint32_t e = 0; e < n; ++e) {
      uint32_t rem = e;
      int64_t off = 0;
      bool in = true;
      for (int i = 0; i < map.rank; ++i) {
        const int64_t gi = (int64_t)cc[i] + rem % map.box[i];
        rem /= map.box[i];
        if (gi < 0 || gi >= (int64_t)map.dim[i]) in = false;
        off += gi * (int64_t)map.stride[i];
      }
      uint16_t v = 0;
      if (in) std::memcpy(&v, (const unsigned char*)map.base + off, 2);
      uint32_t a = dst + e * 2u;
      a ^= ((a >> 7) & 7u) << 4;
      std::memcpy(smem_ptr(a, 2), &v, 2);
    }
    mbar_complete_tx(bar, n * 2u);
  });
}

// Untiled bulk copy (cp.async.bulk): bytes land unchanged at dst.
inline void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  if (dst % 16 || reinterpret_cast<uintptr_t>(src) % 16 || bytes % 16 || bytes == 0)
    die("bulk copy: addresses and size must be 16-byte multiples", dst, bytes);
  smem_ptr(dst, 16);
  smem_ptr(dst + bytes - 16, 16);  // the whole destination inside shared memory
  g_block->copy.push([=] {
    std::memcpy(smem_ptr(dst, 16), src, bytes);
    mbar_complete_tx(bar, bytes);
  });
}

}  // namespace emu
