// Runs the response dK/dV kernel's source (tc_dkdv_kernel) on the CPU block
// emulator:  attn_dkdv_emu <in.bin> <out.bin>
// in.bin: int64 hq, hkv, R; float32 scale; bf16 q, d_o [R][hq][256],
// k_resp, v_resp [R][hkv][256]; float32 lse, delta [R][hq].
// out.bin: uint32 status[2]; bf16 dk, dv [R][hkv][256].
#include <cuda_runtime.h>

#include <cstdio>
#include <vector>

namespace ls {
namespace {
alignas(1024) unsigned char smem_raw[emu::kSmemBytes];
}  // namespace
}  // namespace ls

#include "kernel.cu"  // the kernel's source, its launcher left out

namespace ls {
namespace {
// The library's 3-D map over token-major [rows][heads][256] bf16 data:
// [box_rows x 1 x 64] boxes.
emu::TensorMap rows_map(const void* base, int heads, int64_t rows, int box_rows) {
  return {base, 3, {256, (uint64_t)heads, (uint64_t)rows}, {2, 512, (uint64_t)heads * 512},
          {64, 1, (uint32_t)box_rows}};
}
void emulate(DkdvKParams p, const void* q, const void* d_o, const void* k, const void* v) {
  const CUtensorMap tk = rows_map(k, p.hkv, p.R, kBK), tv = rows_map(v, p.hkv, p.R, kBK);
  const CUtensorMap tq = rows_map(q, p.hq, p.R, kBR), to = rows_map(d_o, p.hq, p.R, kBR);
  emu::g_smem = smem_raw;
  const int grid = p.hkv * p.n_kt * 2;
  for (int u = 0; u < grid; ++u)
    emu::run_block((unsigned)u, 0, kThreads, [&] { tc_dkdv_kernel(tk, tv, tq, to, p); },
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
  int64_t h[3];
  float scale;
  if (std::fread(h, 8, 3, f) != 3 || std::fread(&scale, 4, 1, f) != 1) return 4;
  const int64_t hq = h[0], hkv = h[1], R = h[2];
  std::vector<uint16_t> q, dO, k, v;
  std::vector<float> lse, delta;
  if (!rd(f, q, (size_t)R * hq * 256) || !rd(f, dO, (size_t)R * hq * 256) ||
      !rd(f, k, (size_t)R * hkv * 256) || !rd(f, v, (size_t)R * hkv * 256) ||
      !rd(f, lse, (size_t)R * hq) || !rd(f, delta, (size_t)R * hq))
    return 5;
  std::fclose(f);
  std::vector<uint16_t> dk((size_t)R * hkv * 256, 0xffff), dv((size_t)R * hkv * 256, 0xffff);
  uint32_t status[2] = {0, 0};
  ls::DkdvKParams p{};
  p.hq = (int32_t)hq, p.hkv = (int32_t)hkv, p.gq = (int32_t)(hq / hkv), p.R = (int32_t)R;
  p.n_kt = (int32_t)((R + 127) / 128);
  p.scale = scale, p.scale_log2 = scale * 1.4426950408889634f;
  p.lse = lse.data(), p.delta = delta.data();
  p.dk = reinterpret_cast<__nv_bfloat16*>(dk.data());
  p.dv = reinterpret_cast<__nv_bfloat16*>(dv.data());
  p.status = status;
  ls::emulate(p, q.data(), dO.data(), k.data(), v.data());
  f = std::fopen(argv[2], "wb");
  if (!f) return 6;
  std::fwrite(status, 4, 2, f);
  std::fwrite(dk.data(), 2, dk.size(), f);
  std::fwrite(dv.data(), 2, dv.size(), f);
  std::fclose(f);
  return 0;
}
