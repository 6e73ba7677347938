// Gated-DeltaNet state replay (the Qwen model's recurrent layers keep a
// fixed-size state for the prompt and replay each response from it with the
// prompt state detached: LongStraw DeepRead summary, section Method, Qwen
// path).  The recurrence, per head, with state S [dv][dk] (the published
// gated delta rule; the pages name the layer but do not print it):
//   a_t = exp(g_t),  u_t = S_{t-1} k_t,  w_t = v_t - a_t u_t
//   S_t = a_t S_{t-1} + b_t w_t k_t^T        (= a_t S_{t-1}(I - b_t k_t k_t^T) + b_t v_t k_t^T)
//   o_t = S_t q_t
//
// One CTA per (head, member), 256 threads, dk = dv = 128.  The members of a
// group replay from the same captured state and run side by side.  Thread (i = tid/2, half =
// tid%2) holds row i, columns 64*half .. 64*half+63 of S in registers, so a
// step needs no barrier: the row products S k and S q are a 64-term dot
// product plus one shuffle with the partner thread.  The time loop is
// sequential; heads run in parallel.
//
// Backward (the gradient of sum(dO * o) for q, k, v, g, b; none for S_0):
//   G_t  += dO_t q_t^T                       (G = dL/dS_t, in registers)
//   dq_t  = S_t^T dO_t
//   gk    = G_t k_t,  dw = b_t gk,  dv_t = dw,  db_t = w_t . gk
//   dg_t  = a_t (<G_t, S_{t-1}> - dw . u_t)
//   dk_t  = b_t G_t^T w_t - a_t S_{t-1}^T dw
//   G_{t-1} = a_t (G_t - dw k_t^T)
// S_{t-1} is needed in reverse order: the forward is re-run with a
// checkpoint of S every kSegB = 8 steps, and each segment is recomputed into
// a per-(member, head) buffer of 8 states (512 KB, so the buffers of all
// resident CTAs stay in L2) before it is walked backwards.  The column sums
// (dq_t, dk_t) go through shared memory; the two scalars through a block
// reduction.
#include <cuda_runtime.h>

#include <cstdint>

#include "ls_internal.h"

namespace ls {
namespace {

constexpr int kD = 128;    // dk = dv
constexpr int kTB = 16;    // tokens staged per block in the forward
constexpr int kSegB = 8;   // checkpoint interval of the backward
constexpr int kThreads = 256;
// Column-sum buffers of the backward: quantity (0: dq, 1: dk) x column half
// x 128 rows x 64 columns, rows padded to 65 floats and the second half
// shifted by 16 banks, so that both the row writes (thread (i, half)) and the
// column reads are free of bank conflicts.
constexpr int kRedPitch = 65;
constexpr int kRedHalf = kD * kRedPitch + 16;
constexpr int kRedQty = 2 * kRedHalf;
constexpr int kRedFloats = 2 * kRedQty;
__device__ __forceinline__ int red_at(int qty, int half, int row, int col) {
  return qty * kRedQty + half * kRedHalf + row * kRedPitch + col;
}

__device__ __forceinline__ float pair_sum(float x) { return x + __shfl_xor_sync(0xffffffffu, x, 1); }

__global__ void __launch_bounds__(kThreads, 1)
    gdn_fwd_kernel(int H, int R, const float* __restrict__ s0, const float* __restrict__ q,
                   const float* __restrict__ k, const float* __restrict__ v,
                   const float* __restrict__ g, const float* __restrict__ beta, float* __restrict__ o,
                   float* __restrict__ s_final) {
  __shared__ float ks[kTB][kD], qs[kTB][kD], vs[kTB][kD], gs[kTB], bs[kTB];
  const int h = blockIdx.x, tid = threadIdx.x;
  {  // member blockIdx.y: its tokens and final state (s0 is shared by the group)
    const int64_t tok = (int64_t)blockIdx.y * R * H;
    q += tok * kD, k += tok * kD, v += tok * kD, o += tok * kD, g += tok, beta += tok;
    if (s_final) s_final += (int64_t)blockIdx.y * H * kD * kD;
  }
  const int i = tid >> 1, half = tid & 1;
  float s[64];
  const float* src = s0 + ((int64_t)h * kD + i) * kD + half * 64;
#pragma unroll
  for (int c = 0; c < 64; ++c) s[c] = src[c];
  for (int t0 = 0; t0 < R; t0 += kTB) {
    const int nt = R - t0 < kTB ? R - t0 : kTB;
    __syncthreads();
    for (int x = tid; x < nt * kD; x += kThreads) {
      const int tt = x / kD, j = x % kD;
      const int64_t row = (int64_t)(t0 + tt) * H + h;
      ks[tt][j] = k[row * kD + j];
      qs[tt][j] = q[row * kD + j];
      vs[tt][j] = v[row * kD + j];
    }
    if (tid < nt) {
      gs[tid] = g[(int64_t)(t0 + tid) * H + h];
      bs[tid] = beta[(int64_t)(t0 + tid) * H + h];
    }
    __syncthreads();
    for (int tt = 0; tt < nt; ++tt) {
      const float a = expf(gs[tt]);
      const float* kr = &ks[tt][half * 64];
      const float* qr = &qs[tt][half * 64];
      float u = 0.f;
#pragma unroll
      for (int c = 0; c < 64; ++c) u = fmaf(s[c], kr[c], u);
      u = pair_sum(u);
      const float bw = bs[tt] * (vs[tt][i] - a * u);
      float acc = 0.f;
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        s[c] = fmaf(a, s[c], bw * kr[c]);
        acc = fmaf(s[c], qr[c], acc);
      }
      acc = pair_sum(acc);
      if (half == 0) o[((int64_t)(t0 + tt) * H + h) * kD + i] = acc;
    }
  }
  if (s_final) {
    float* dst = s_final + ((int64_t)h * kD + i) * kD + half * 64;
#pragma unroll
    for (int c = 0; c < 64; ++c) dst[c] = s[c];
  }
}

// Thread-private state scratch, laid out so that a warp's accesses are
// coalesced: element c of thread tid sits at float4 (c/4) * kThreads + tid.
__device__ __forceinline__ void put_state(float* base, int tid, const float (&s)[64]) {
  float4* p = reinterpret_cast<float4*>(base) + tid;
#pragma unroll
  for (int j = 0; j < 16; ++j) p[j * kThreads] = make_float4(s[4 * j], s[4 * j + 1], s[4 * j + 2], s[4 * j + 3]);
}
__device__ __forceinline__ void get_state(const float* base, int tid, float (&s)[64]) {
  const float4* p = reinterpret_cast<const float4*>(base) + tid;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float4 x = p[j * kThreads];
    s[4 * j] = x.x, s[4 * j + 1] = x.y, s[4 * j + 2] = x.z, s[4 * j + 3] = x.w;
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    gdn_bwd_kernel(int H, int R, const float* __restrict__ s0, const float* __restrict__ q,
                   const float* __restrict__ k, const float* __restrict__ v,
                   const float* __restrict__ g, const float* __restrict__ beta,
                   const float* __restrict__ d_o, float* __restrict__ dq, float* __restrict__ dk,
                   float* __restrict__ dv, float* __restrict__ dg, float* __restrict__ dbeta,
                   float* __restrict__ ws) {
  extern __shared__ float red[];  // column-sum buffers, see red_at
  __shared__ float tk[kSegB][kD], tv[kSegB][kD], tq[kSegB][kD], tdo[kSegB][kD];
  __shared__ float tg[kSegB], tb[kSegB], part[2][kThreads / 32];
  const int h = blockIdx.x, tid = threadIdx.x;
  const int i = tid >> 1, half = tid & 1;
  const int lane = tid & 31, wid = tid >> 5;
  const int nseg = (R + kSegB - 1) / kSegB;
  {  // member blockIdx.y
    const int64_t tok = (int64_t)blockIdx.y * R * H;
    q += tok * kD, k += tok * kD, v += tok * kD, d_o += tok * kD, g += tok, beta += tok;
    dq += tok * kD, dk += tok * kD, dv += tok * kD, dg += tok, dbeta += tok;
  }
  // per (member, head) workspace: nseg checkpoints, then the kSegB states of one segment
  float* ckpt = ws + ((int64_t)blockIdx.y * H + h) * (nseg + kSegB) * kD * kD;
  float* segs = ckpt + (int64_t)nseg * kD * kD;

  // tokens t0 .. t0+nt-1 into shared memory (q and dO only for the reverse walk)
  auto stage = [&](int t0, int nt, bool with_q) {
    __syncthreads();
    for (int x = tid; x < nt * kD; x += kThreads) {
      const int tt = x / kD, j = x % kD;
      const int64_t e = ((int64_t)(t0 + tt) * H + h) * kD + j;
      tk[tt][j] = k[e];
      tv[tt][j] = v[e];
      if (with_q) {
        tq[tt][j] = q[e];
        tdo[tt][j] = d_o[e];
      }
    }
    if (tid < nt) {
      tg[tid] = g[(int64_t)(t0 + tid) * H + h];
      tb[tid] = beta[(int64_t)(t0 + tid) * H + h];
    }
    __syncthreads();
  };
  auto step = [&](float (&s)[64], int tt) {  // S <- a S + b w k^T with staged token tt
    const float a = expf(tg[tt]);
    const float* kr = &tk[tt][half * 64];
    float u = 0.f;
#pragma unroll
    for (int c = 0; c < 64; ++c) u = fmaf(s[c], kr[c], u);
    u = pair_sum(u);
    const float bw = tb[tt] * (tv[tt][i] - a * u);
#pragma unroll
    for (int c = 0; c < 64; ++c) s[c] = fmaf(a, s[c], bw * kr[c]);
  };

  // ---- pass 1: forward, keeping S at the start of every segment
  float s[64];
#pragma unroll
  for (int c = 0; c < 64; ++c) s[c] = s0[(int64_t)h * kD * kD + (int64_t)i * kD + half * 64 + c];
  for (int sg = 0; sg < nseg; ++sg) {
    put_state(ckpt + (int64_t)sg * kD * kD, tid, s);
    if (sg == nseg - 1) break;  // the last segment is recomputed in pass 2
    stage(sg * kSegB, kSegB, false);
    for (int tt = 0; tt < kSegB; ++tt) step(s, tt);
  }

  // ---- pass 2: segments in reverse; G = dL/dS in registers
  float gg[64];
#pragma unroll
  for (int c = 0; c < 64; ++c) gg[c] = 0.f;
  float* r0 = red + red_at(0, half, i, 0);  // this thread's row of the dq buffer
  float* r1 = red + red_at(1, half, i, 0);  // and of the dk buffer
  for (int sg = nseg - 1; sg >= 0; --sg) {
    const int t0 = sg * kSegB, nt = (R - t0 < kSegB) ? R - t0 : kSegB;
    stage(t0, nt, true);
    get_state(ckpt + (int64_t)sg * kD * kD, tid, s);
    for (int tt = 0; tt < nt; ++tt) {  // S before each token of the segment
      put_state(segs + (int64_t)tt * kD * kD, tid, s);
      step(s, tt);
    }
    for (int tt = nt - 1; tt >= 0; --tt) {
      float sp[64];
      get_state(segs + (int64_t)tt * kD * kD, tid, sp);  // S_{t-1}, written by this thread
      const float a = expf(tg[tt]), b = tb[tt];
      const float* kr = &tk[tt][half * 64];
      const float* qr = &tq[tt][half * 64];
      float u = 0.f;
#pragma unroll
      for (int c = 0; c < 64; ++c) u = fmaf(sp[c], kr[c], u);
      u = pair_sum(u);
      const float w = tv[tt][i] - a * u;
      const float doi = tdo[tt][i];
      float gk = 0.f;
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        gg[c] = fmaf(doi, qr[c], gg[c]);
        gk = fmaf(gg[c], kr[c], gk);
      }
      gk = pair_sum(gk);
      const float dw = b * gk;
      float gs_dot = 0.f;
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const float st = fmaf(a, sp[c], b * w * kr[c]);  // S_t
        r0[c] = st * doi;                                // -> dq_t
        r1[c] = b * gg[c] * w - a * sp[c] * dw;          // -> dk_t
        gs_dot = fmaf(gg[c], sp[c], gs_dot);
        gg[c] = a * (gg[c] - dw * kr[c]);                // G_{t-1}
      }
      // scalars: db = sum_i w_i gk_i, dalpha = <G, S_{t-1}> - sum_i dw_i u_i
      float pdb = half == 0 ? w * gk : 0.f;
      float pda = gs_dot - (half == 0 ? dw * u : 0.f);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        pdb += __shfl_xor_sync(0xffffffffu, pdb, off);
        pda += __shfl_xor_sync(0xffffffffu, pda, off);
      }
      if (lane == 0) {
        part[0][wid] = pdb;
        part[1][wid] = pda;
      }
      const int64_t row = (int64_t)(t0 + tt) * H + h;
      if (half == 0) dv[row * kD + i] = dw;
      __syncthreads();
      {  // column j of dq (threads 0..127) or dk (128..255): the sum over the 128 rows
        const int which = tid >> 7, j = tid & (kD - 1);
        const float* col = red + red_at(which, j >> 6, 0, j & 63);
        float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
#pragma unroll 8
        for (int r = 0; r < kD; r += 4) {
          acc0 += col[(r + 0) * kRedPitch];
          acc1 += col[(r + 1) * kRedPitch];
          acc2 += col[(r + 2) * kRedPitch];
          acc3 += col[(r + 3) * kRedPitch];
        }
        (which == 0 ? dq : dk)[row * kD + j] = (acc0 + acc1) + (acc2 + acc3);
      }
      if (tid == 0) {
        float sdb = 0.f, sda = 0.f;
        for (int x = 0; x < kThreads / 32; ++x) {
          sdb += part[0][x];
          sda += part[1][x];
        }
        dbeta[row] = sdb;
        dg[row] = sda * a;
      }
      __syncthreads();  // the buffers and part[] are rewritten by the next step
    }
  }
}

}  // namespace

size_t gdn_workspace_bytes(int B, int H, int R) {
  const int64_t nseg = (R + kSegB - 1) / kSegB;
  return (size_t)B * H * (size_t)(nseg + kSegB) * kD * kD * sizeof(float);
}

bool gdn_supported(int dk, int dv) { return dk == kD && dv == kD; }

cudaError_t launch_gdn_fwd(int B, int H, int R, const float* s0, const float* q, const float* k,
                           const float* v, const float* g, const float* beta, float* o,
                           float* s_final, cudaStream_t st) {
  if (B == 0 || H == 0) return cudaSuccess;
  LaunchScope ls(kKGdnFwd, st);
  gdn_fwd_kernel<<<dim3(H, B), kThreads, 0, st>>>(H, R, s0, q, k, v, g, beta, o, s_final);
  return cudaGetLastError();
}

cudaError_t launch_gdn_bwd(int B, int H, int R, const float* s0, const float* q, const float* k,
                           const float* v, const float* g, const float* beta, const float* d_o,
                           float* dq, float* dk, float* dv, float* dg, float* dbeta, float* ws,
                           cudaStream_t st) {
  if (B == 0 || H == 0 || R == 0) return cudaSuccess;
  const int smem = kRedFloats * (int)sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(gdn_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  LaunchScope ls(kKGdnBwd, st);
  gdn_bwd_kernel<<<dim3(H, B), kThreads, smem, st>>>(H, R, s0, q, k, v, g, beta, d_o, dq, dk, dv, dg, dbeta,
                                            ws);
  return cudaGetLastError();
}

}  // namespace ls
