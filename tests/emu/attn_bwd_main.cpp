// Runs the prompt-attention backward kernel's source (tc_bwd_dq_ring_kernel) on
// the CPU block emulator:  attn_bwd_emu <in.bin> <out.bin>
// in.bin: int64 hq, hkv, R, P, page_size, pool_pages, num_pages, ns,
// split_span; float32 scale; then bf16 k_pool, v_pool [pool_pages][hkv][page][256],
// int32 page_table [num_pages], bf16 q, d_o [R][hq][256], bf16 k_resp,
// v_resp [R][hkv][256], float32 lse, delta [R][hq].
// out.bin: uint32 status[2]; float32 dq_parts [ns+1][R*hq][256] (unscaled).
#include <cuda_runtime.h>

#include <cstdio>
#include <vector>

namespace ls {
namespace {
alignas(1024) unsigned char smem_raw[emu::kSmemBytes];
}  // namespace
}  // namespace ls

#include "kernel.cu"  // the kernel's source: its constants, parameter block and the kernel

namespace ls {
namespace {
// The tensor maps the library encodes for these kernels (whole [rows x 64*blocks]
// tiles landing as `blocks` swizzled [rows x 64] column boxes).
emu::TensorMap pool_tile_map(const void* base, int64_t rows, int box_rows, int blocks) {
  return {base, 3, {64, (uint64_t)rows, 4}, {2, 512, 128}, {64, (uint32_t)box_rows, (uint32_t)blocks}};
}
emu::TensorMap rows_tile_map(const void* base, int heads, int64_t rows, int box_rows, int blocks) {
  return {base, 4, {64, (uint64_t)rows, 4, (uint64_t)heads}, {2, (uint64_t)heads * 512, 128, 512},
          {64, (uint32_t)box_rows, (uint32_t)blocks, 1}};
}

// the 128-key ring kernel: K and V chunks of [128 keys x 128 columns]
constexpr int kBoxBlocks = 2;
#define LS_EMU_KERNEL tc_bwd_dq_ring_kernel
#define LS_EMU_THREADS kThreadsRing
using EmuLayout = BwdRingLayout;

void emulate(BwdKParams p, const void* k_pool, const void* v_pool, const void* k_resp,
             const void* v_resp) {
  using L = EmuLayout;
  const CUtensorMap tk = pool_tile_map(k_pool, p.pool_rows, L::BN, kBoxBlocks);
  const CUtensorMap tv = pool_tile_map(v_pool, p.pool_rows, L::BN, kBoxBlocks);
  const CUtensorMap tkr = rows_tile_map(k_resp, p.hkv, p.R, L::BN, kBoxBlocks);
  const CUtensorMap tvr = rows_tile_map(v_resp, p.hkv, p.R, L::BN, kBoxBlocks);
  emu::g_smem = smem_raw;
  const int units = (p.ns + 1) * p.hkv * p.n_mt;
  for (int u = 0; u < units; ++u)
    emu::run_block((unsigned)u, 0, LS_EMU_THREADS, [&] { LS_EMU_KERNEL(tk, tv, tkr, tvr, p); },
                   (unsigned)(u + 1));
}
}  // namespace
}  // namespace ls

template <class T>
static bool rd(FILE* f, std::vector<T>& v, size_t n) {
  v.resize(n);
  return std::fread(v.data(), sizeof(T), n, f) == n;
}

int main(int argc, char** argv) {
  if (argc != 3) return 2;
  FILE* f = std::fopen(argv[1], "rb");
  if (!f) return 3;
  int64_t h[9];
  float scale;
  if (std::fread(h, 8, 9, f) != 9 || std::fread(&scale, 4, 1, f) != 1) return 4;
  const int64_t hq = h[0], hkv = h[1], R = h[2], P = h[3], page = h[4], pool_pages = h[5],
                num_pages = h[6], ns = h[7], span = h[8];
  std::vector<uint16_t> kp, vp, q, dO, kr, vr;
  std::vector<int32_t> pt;
  std::vector<float> lse, delta;
  const size_t npool = (size_t)pool_pages * hkv * page * 256;
  if (!rd(f, kp, npool) || !rd(f, vp, npool) || !rd(f, pt, (size_t)num_pages) ||
      !rd(f, q, (size_t)R * hq * 256) || !rd(f, dO, (size_t)R * hq * 256) ||
      !rd(f, kr, (size_t)R * hkv * 256) || !rd(f, vr, (size_t)R * hkv * 256) ||
      !rd(f, lse, (size_t)R * hq) || !rd(f, delta, (size_t)R * hq))
    return 5;
  std::fclose(f);
  std::vector<float> dq_parts((size_t)(ns + 1) * R * hq * 256, 0.f);
  uint32_t status[2] = {0, 0};
  ls::BwdKParams p{};
  p.hq = (int32_t)hq, p.hkv = (int32_t)hkv, p.gq = (int32_t)(hq / hkv), p.R = (int32_t)R;
  p.P = P, p.pool_rows = pool_pages * hkv * page, p.pool_pages = pool_pages;
  p.page_size = (int32_t)page, p.ns = (int32_t)ns, p.split_span = span;
  p.n_mt = (int32_t)((p.gq * R + 127) / 128);
  p.scale_log2 = scale * 1.4426950408889634f;
  p.q = reinterpret_cast<const __nv_bfloat16*>(q.data());
  p.d_o = reinterpret_cast<const __nv_bfloat16*>(dO.data());
  p.lse = lse.data(), p.delta = delta.data(), p.page_table = pt.data();
  p.dq_parts = dq_parts.data(), p.status = status;
  ls::emulate(p, kp.data(), vp.data(), kr.data(), vr.data());
  f = std::fopen(argv[2], "wb");
  if (!f) return 6;
  std::fwrite(status, 4, 2, f);
  std::fwrite(dq_parts.data(), 4, dq_parts.size(), f);
  std::fclose(f);
  return 0;
}
