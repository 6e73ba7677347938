// Runs the recurrent GDN replay kernels' source (gdn_fwd_kernel and
// gdn_bwd_kernel) on the CPU block emulator:  gdn_rec_emu <in.bin> <out.bin>
// in.bin: int32 B, H, R; float32 s0 [H][128][128], q, k, v, d_o [B][R][H][128],
// g, beta [B][R][H].  out.bin: float32 o, s_final, dq, dk, dv, dg, dbeta.
#include <cuda_runtime.h>

#include <cstdio>
#include <vector>

namespace ls {
namespace {
float red[2 * 2 * (128 * 65 + 16)];  // the backward's dynamic shared memory
}  // namespace
}  // namespace ls

#include "kernel.cu"  // the kernels' source, host launchers left out

namespace ls {
namespace {
void emulate(int B, int H, int R, const float* s0, const float* q, const float* k, const float* v,
             const float* g, const float* beta, const float* d_o, float* o, float* s_final,
             float* dq, float* dk, float* dv, float* dg, float* dbeta) {
  std::vector<float> ws(gdn_workspace_bytes(B, H, R) / sizeof(float));
  static unsigned char dummy[1024];
  emu::g_smem = dummy;
  for (int m = 0; m < B; ++m)
    for (int h = 0; h < H; ++h) {
      emu::run_block((unsigned)h, (unsigned)m, kThreads,
                     [&] { gdn_fwd_kernel(H, R, s0, q, k, v, g, beta, o, s_final); });
      if (R > 0)
        emu::run_block((unsigned)h, (unsigned)m, kThreads, [&] {
          gdn_bwd_kernel(H, R, s0, q, k, v, g, beta, d_o, dq, dk, dv, dg, dbeta, ws.data());
        });
    }
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
  std::vector<float> s0(ns), q(nt), k(nt), v(nt), d_o(nt), g(nsc), beta(nsc);
  for (auto* x : {&s0, &q, &k, &v, &d_o, &g, &beta})
    if (std::fread(x->data(), 4, x->size(), f) != x->size()) return 5;
  std::fclose(f);
  std::vector<float> o(nt), s_final((size_t)B * ns), dq(nt), dk(nt), dv(nt), dg(nsc), dbeta(nsc);
  ls::emulate(B, H, R, s0.data(), q.data(), k.data(), v.data(), g.data(), beta.data(), d_o.data(),
              o.data(), s_final.data(), dq.data(), dk.data(), dv.data(), dg.data(), dbeta.data());
  f = std::fopen(argv[2], "wb");
  if (!f) return 6;
  for (auto* x : {&o, &s_final, &dq, &dk, &dv, &dg, &dbeta}) std::fwrite(x->data(), 4, x->size(), f);
  std::fclose(f);
  return 0;
}
