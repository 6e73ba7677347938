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
// checkpoint of S every kSeg steps, and each segment is recomputed into a
// per-head buffer before it is walked backwards.  The column sums (dq_t,
// dk_t) go through shared memory; the two scalars through a block reduction.
#include <cuda_runtime.h>

#include <cstdint>

#include "ls_internal.h"

namespace ls {
namespace {

constexpr int kD = 128;    // dk = dv
constexpr int kTB = 16;    // tokens staged per block in the forward
constexpr int kSeg = 64;   // checkpoint interval of the backward
constexpr int kThreads = 256;
constexpr int kRedPitch = kD + 1;  // padded rows of the column-sum buffers

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

__global__ void __launch_bounds__(kThreads, 1)
    gdn_bwd_kernel(int H, int R, const float* __restrict__ s0, const float* __restrict__ q,
                   const float* __restrict__ k, const float* __restrict__ v,
                   const float* __restrict__ g, const float* __restrict__ beta,
                   const float* __restrict__ d_o, float* __restrict__ dq, float* __restrict__ dk,
                   float* __restrict__ dv, float* __restrict__ dg, float* __restrict__ dbeta,
                   float* __restrict__ ws) {
  extern __shared__ float red[];  // [2][kD][kRedPitch]
  __shared__ float kv_k[kD], kv_q[kD], kv_v[kD], kv_do[kD], sc[2];
  __shared__ float part[2][kThreads / 32];
  const int h = blockIdx.x, tid = threadIdx.x;
  const int i = tid >> 1, half = tid & 1;
  const int lane = tid & 31, wid = tid >> 5;
  const int nseg = (R + kSeg - 1) / kSeg;
  {  // member blockIdx.y
    const int64_t tok = (int64_t)blockIdx.y * R * H;
    q += tok * kD, k += tok * kD, v += tok * kD, d_o += tok * kD, g += tok, beta += tok;
    dq += tok * kD, dk += tok * kD, dv += tok * kD, dg += tok, dbeta += tok;
  }
  // per (member, head) workspace: nseg checkpoints, then kSeg states of one segment
  float* ckpt = ws + ((int64_t)blockIdx.y * H + h) * (nseg + kSeg) * kD * kD;
  float* seg = ckpt + (int64_t)nseg * kD * kD;
  const int64_t my = (int64_t)i * kD + half * 64;  // this thread's slice of a state

  auto stage = [&](int t, bool with_q) {  // vectors of token t into shared memory
    __syncthreads();
    const int64_t row = (int64_t)t * H + h;
    if (tid < kD) {
      kv_k[tid] = k[row * kD + tid];
      kv_v[tid] = v[row * kD + tid];
    } else if (with_q) {
      kv_q[tid - kD] = q[row * kD + tid - kD];
      kv_do[tid - kD] = d_o[row * kD + tid - kD];
    }
    if (tid == 0) {
      sc[0] = g[row];
      sc[1] = beta[row];
    }
    __syncthreads();
  };
  auto step = [&](float (&s)[64]) {  // S <- a S + b w k^T with the staged token
    const float a = expf(sc[0]);
    const float* kr = &kv_k[half * 64];
    float u = 0.f;
#pragma unroll
    for (int c = 0; c < 64; ++c) u = fmaf(s[c], kr[c], u);
    u = pair_sum(u);
    const float bw = sc[1] * (kv_v[i] - a * u);
#pragma unroll
    for (int c = 0; c < 64; ++c) s[c] = fmaf(a, s[c], bw * kr[c]);
  };

  // ---- pass 1: forward, keeping S before every kSeg-th token
  float s[64];
#pragma unroll
  for (int c = 0; c < 64; ++c) s[c] = s0[(int64_t)h * kD * kD + my + c];
  for (int t = 0; t < R; ++t) {
    if (t % kSeg == 0) {
      float* dst = ckpt + (int64_t)(t / kSeg) * kD * kD + my;
#pragma unroll
      for (int c = 0; c < 64; ++c) dst[c] = s[c];
    }
    stage(t, false);
    step(s);
  }

  // ---- pass 2: segments in reverse; G = dL/dS in registers
  float gg[64];
#pragma unroll
  for (int c = 0; c < 64; ++c) gg[c] = 0.f;
  float* red0 = red;
  float* red1 = red + kD * kRedPitch;
  for (int sgi = nseg - 1; sgi >= 0; --sgi) {
    const int t0 = sgi * kSeg, t1 = (t0 + kSeg < R) ? t0 + kSeg : R;
    const float* c0 = ckpt + (int64_t)sgi * kD * kD + my;
#pragma unroll
    for (int c = 0; c < 64; ++c) s[c] = c0[c];
    for (int t = t0; t < t1; ++t) {  // S before each token of the segment
      float* dst = seg + (int64_t)(t - t0) * kD * kD + my;
#pragma unroll
      for (int c = 0; c < 64; ++c) dst[c] = s[c];
      stage(t, false);
      step(s);
    }
    for (int t = t1 - 1; t >= t0; --t) {
      stage(t, true);  // also orders the previous step's column sums before reuse
      const float* spp = seg + (int64_t)(t - t0) * kD * kD + my;
      float sp[64];
#pragma unroll
      for (int c = 0; c < 64; ++c) sp[c] = spp[c];
      const float a = expf(sc[0]), b = sc[1];
      const float* kr = &kv_k[half * 64];
      const float* qr = &kv_q[half * 64];
      float u = 0.f;
#pragma unroll
      for (int c = 0; c < 64; ++c) u = fmaf(sp[c], kr[c], u);
      u = pair_sum(u);
      const float w = kv_v[i] - a * u;
      const float doi = kv_do[i];
      float gk = 0.f;
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        gg[c] = fmaf(doi, qr[c], gg[c]);
        gk = fmaf(gg[c], kr[c], gk);
      }
      gk = pair_sum(gk);
      const float dw = b * gk;
      float gs_dot = 0.f;
      float* r0 = red0 + i * kRedPitch + half * 64;
      float* r1 = red1 + i * kRedPitch + half * 64;
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
      if (half == 0) dv[((int64_t)t * H + h) * kD + i] = dw;
      __syncthreads();
      const int64_t row = (int64_t)t * H + h;
      if (tid < kD) {
        float acc = 0.f;
        for (int r = 0; r < kD; ++r) acc += red0[r * kRedPitch + tid];
        dq[row * kD + tid] = acc;
      } else {
        const int j = tid - kD;
        float acc = 0.f;
        for (int r = 0; r < kD; ++r) acc += red1[r * kRedPitch + j];
        dk[row * kD + j] = acc;
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
    }
  }
}

}  // namespace

size_t gdn_workspace_bytes(int B, int H, int R) {
  const int64_t nseg = (R + kSeg - 1) / kSeg;
  return (size_t)B * H * (size_t)(nseg + kSeg) * kD * kD * sizeof(float);
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
  const int smem = 2 * kD * kRedPitch * (int)sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(gdn_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  LaunchScope ls(kKGdnBwd, st);
  gdn_bwd_kernel<<<dim3(H, B), kThreads, smem, st>>>(H, R, s0, q, k, v, g, beta, d_o, dq, dk, dv, dg, dbeta,
                                            ws);
  return cudaGetLastError();
}

}  // namespace ls
