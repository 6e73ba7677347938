// Runs the chunk-parallel GDN kernels' source on the CPU block emulator:
//   gdn_cp_emu <stage> <in.bin> <out.bin>      stage: prep | all | fwd | fwd_bwd
// in.bin: int32 B, H, R; float32 s0 [H][128][128], q, k, v, d_o [B][R][H][128],
// g, beta [B][R][H].  out.bin: uint32 status; the float32 scratch; then (all,
// fwd, fwd_bwd) o, s_final, dq, dk, dv, dg, dbeta (the gradients zero after fwd).
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>
#include <vector>

namespace ls {
namespace {
alignas(1024) unsigned char smem_raw[emu::kSmemBytes];
}  // namespace
}  // namespace ls

#include "kernel.cu"  // the kernels' source, host launchers left out

int main(int argc, char** argv) {
  if (argc != 4) return 2;
  const int mode = std::strcmp(argv[1], "all") == 0       ? 1
                   : std::strcmp(argv[1], "fwd") == 0     ? 2
                   : std::strcmp(argv[1], "fwd_bwd") == 0 ? 3
                                                          : 0;
  FILE* f = std::fopen(argv[2], "rb");
  if (!f) return 3;
  int32_t hdr[3];
  if (std::fread(hdr, 4, 3, f) != 3) return 4;
  const int B = hdr[0], H = hdr[1], R = hdr[2];
  const int nch = (R + 127) / 128;
  const size_t ns = (size_t)H * 128 * 128, nt = (size_t)B * R * H * 128, nsc = (size_t)B * R * H;
  std::vector<float> s0(ns), q(nt), k(nt), v(nt), d_o(nt), g(nsc), beta(nsc);
  for (auto* x : {&s0, &q, &k, &v, &d_o, &g, &beta})
    if (std::fread(x->data(), 4, x->size(), f) != x->size()) return 5;
  std::fclose(f);
  std::vector<float> scr((size_t)B * H * nch * ls::kScrFloats, 0.f);
  std::vector<float> o(nt), s_final((size_t)B * ns), dq(nt), dk(nt), dv(nt), dg(nsc), dbeta(nsc);
  uint32_t status = 0;
  ls::emu_run(mode, B, H, R, s0.data(), q.data(), k.data(), v.data(), g.data(), beta.data(),
              d_o.data(), scr.data(), o.data(), s_final.data(), dq.data(), dk.data(), dv.data(),
              dg.data(), dbeta.data(), &status);
  f = std::fopen(argv[3], "wb");
  if (!f) return 6;
  std::fwrite(&status, 4, 1, f);
  std::fwrite(scr.data(), 4, scr.size(), f);
  if (mode != 0)
    for (auto* x : {&o, &s_final, &dq, &dk, &dv, &dg, &dbeta}) std::fwrite(x->data(), 4, x->size(), f);
  std::fclose(f);
  return 0;
}
