// Runs the chunkwise GDN forward kernel's source on the CPU block emulator:
//   gdn_chunk_emu <in.bin> <out.bin>
// in.bin: int32 B, H, R; float32 s0 [H][128][128], q, k, v [B][R][H][128],
// g, beta [B][R][H].  out.bin: float32 o [B][R][H][128], s_final [B][H][128][128].
#include <cuda_runtime.h>

#include <cstdio>
#include <vector>

namespace ls {
namespace {
alignas(1024) unsigned char smem_raw[emu::kSmemBytes];
}  // namespace
}  // namespace ls

#include "kernel.cu"  // the kernel source up to the end of its anonymous namespace

namespace ls {
namespace {
void emulate(int B, int H, int R, const float* s0, const float* q, const float* k, const float* v,
             const float* g, const float* beta, float* o, float* s_final) {
  emu::g_smem = smem_raw;
  for (int m = 0; m < B; ++m)
    for (int h = 0; h < H; ++h)
      emu::run_block((unsigned)h, (unsigned)m, kThr, [&] {
        gdn_chunk_fwd_kernel(H, R, s0, q, k, v, g, beta, o, s_final, nullptr);
      });
}
}  // namespace
}  // namespace ls

int main(int argc, char** argv) {
  if (argc != 3) return 2;
  FILE* f = std::fopen(argv[1], "rb");
  if (!f) return 3;
  int32_t hdr[3];
  if (std::fread(hdr, 4, 3, f) != 3) return 4;
  const int B = hdr[0], H = hdr[1], R = hdr[2];
  const size_t ns = (size_t)H * 128 * 128, nt = (size_t)B * R * H * 128, nsc = (size_t)B * R * H;
  std::vector<float> s0(ns), q(nt), k(nt), v(nt), g(nsc), beta(nsc);
  for (auto* x : {&s0, &q, &k, &v, &g, &beta})
    if (std::fread(x->data(), 4, x->size(), f) != x->size()) return 5;
  std::fclose(f);
  std::vector<float> o(nt, 0.f), s_final((size_t)B * ns, 0.f);
  ls::emulate(B, H, R, s0.data(), q.data(), k.data(), v.data(), g.data(), beta.data(), o.data(),
              s_final.data());
  f = std::fopen(argv[2], "wb");
  if (!f) return 6;
  std::fwrite(o.data(), 4, o.size(), f);
  std::fwrite(s_final.data(), 4, s_final.size(), f);
  std::fclose(f);
  return 0;
}
