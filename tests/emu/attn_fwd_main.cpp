// Runs the prompt-attention forward kernel's source (tc_fwd_ring_kernel) on
// the CPU block emulator:  attn_fwd_emu <in.bin> <out.bin>
// in.bin: as for the backward harness without d_o, lse and delta.
// out.bin: uint32 status[2]; float32 o_parts [ns+1][R*hq][256],
// lse_parts [ns+1][R*hq].
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
// The tensor maps the library encodes for this kernel: K units of
// [128 keys x 128 columns] (two column boxes), V units of [64 keys x 256].
emu::TensorMap pool_tile_map(const void* base, int64_t rows, int box_rows, int blocks) {
  return {base, 3, {64, (uint64_t)rows, 4}, {2, 512, 128}, {64, (uint32_t)box_rows, (uint32_t)blocks}};
}
emu::TensorMap rows_tile_map(const void* base, int heads, int64_t rows, int box_rows, int blocks) {
  return {base, 4, {64, (uint64_t)rows, 4, (uint64_t)heads}, {2, (uint64_t)heads * 512, 128, 512},
          {64, (uint32_t)box_rows, (uint32_t)blocks, 1}};
}

void emulate(FwdKParams p, const void* k_pool, const void* v_pool, const void* k_resp,
             const void* v_resp) {
  using L = FwdRingLayout;
  const CUtensorMap tk = pool_tile_map(k_pool, p.pool_rows, L::BN, 2);
  const CUtensorMap tv = pool_tile_map(v_pool, p.pool_rows, L::BN / 2, 4);
  const CUtensorMap tkr = rows_tile_map(k_resp, p.hkv, p.R, L::BN, 2);
  const CUtensorMap tvr = rows_tile_map(v_resp, p.hkv, p.R, L::BN / 2, 4);
  emu::g_smem = smem_raw;
  const int units = (p.ns + 1) * p.hkv * p.n_mt;
  for (int u = 0; u < units; ++u)
    emu::run_block((unsigned)u, 0, kThreadsRing,
                   [&] { tc_fwd_ring_kernel(tk, tv, tkr, tvr, p); }, (unsigned)(u + 1));
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
  std::vector<uint16_t> kp, vp, q, kr, vr;
  std::vector<int32_t> pt;
  const size_t npool = (size_t)pool_pages * hkv * page * 256;
  if (!rd(f, kp, npool) || !rd(f, vp, npool) || !rd(f, pt, (size_t)num_pages) ||
      !rd(f, q, (size_t)R * hq * 256) || !rd(f, kr, (size_t)R * hkv * 256) ||
      !rd(f, vr, (size_t)R * hkv * 256))
    return 5;
  std::fclose(f);
  std::vector<float> o_parts((size_t)(ns + 1) * R * hq * 256, 0.f), lse_parts((size_t)(ns + 1) * R * hq);
  uint32_t status[2] = {0, 0};
  ls::FwdKParams p{};
  p.hq = (int32_t)hq, p.hkv = (int32_t)hkv, p.gq = (int32_t)(hq / hkv), p.R = (int32_t)R;
  p.P = P, p.pool_rows = pool_pages * hkv * page, p.pool_pages = pool_pages;
  p.page_size = (int32_t)page, p.ns = (int32_t)ns, p.split_span = span;
  p.n_mt = (int32_t)((p.gq * R + 127) / 128);
  p.scale_log2 = scale * 1.4426950408889634f;
  p.q = reinterpret_cast<const __nv_bfloat16*>(q.data());
  p.page_table = pt.data(), p.o_parts = o_parts.data(), p.lse_parts = lse_parts.data();
  p.status = status;
  ls::emulate(p, kp.data(), vp.data(), kr.data(), vr.data());
  f = std::fopen(argv[2], "wb");
  if (!f) return 6;
  std::fwrite(status, 4, 2, f);
  std::fwrite(o_parts.data(), 4, o_parts.size(), f);
  std::fwrite(lse_parts.data(), 4, lse_parts.size(), f);
  std::fclose(f);
  return 0;
}
