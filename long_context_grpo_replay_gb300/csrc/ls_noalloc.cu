// Replay forward for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the
// point where they run the forward: code inside a framework that owns every
// allocation, an allocator-free embedding of the library, or a host thread
// that must not take the driver's allocation locks.  For them this file keeps
// one fixed block of device memory as the forward's scratch (the float32
// partial results and the status word that ls_replay_fwd otherwise keeps in
// the caller's workspace).  The block is a file-scope __device__ array, so
// every GPU that loads the library holds it until the process exits.
//
// In host code the array's name is only a host-side handle, never a device
// address: its device address is fetched once per device with
// cudaGetSymbolAddress (the first call on each device does this, with that
// device current; make that first call before any stream capture) and that
// address is what the kernels receive.  Every call shares the block and it
// keeps the last call's contents, so calls that overlap on the GPU (two
// streams, two threads) race on it.  The status word at its head is cleared
// before each call.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "ls_internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(64) << 20;  // 64 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_fwd_scratch[kScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

thread_local char g_noalloc_err[512] = "";

}  // namespace

extern "C" {

LS_API ls_status ls_replay_fwd_noalloc(const ls_attn_desc* desc, const ls_prompt_kv* prompt,
                                       const void* q, const void* k_resp, const void* v_resp,
                                       int32_t resp_len, void* o, float* lse, void* stream) {
  // Every check comes first: a refused call enqueues nothing and leaves the
  // scratch (and a status word an earlier call may still be setting) alone.
  size_t need = 0;
  const ls_status vs =
      ls::replay_fwd_validate(desc, prompt, q, k_resp, v_resp, resp_len, o, lse, &need);
  if (vs != LS_OK) return vs;
  if (resp_len == 0) return LS_OK;
  if (need > kScratchBytes) {
    snprintf(g_noalloc_err, sizeof(g_noalloc_err),
             "ls_replay_fwd_noalloc: this call needs %zu bytes of scratch, more than the fixed "
             "%zu-byte (64 MiB) scratch; use ls_replay_fwd with a caller-owned workspace",
             need, kScratchBytes);
    ls::set_last_error(g_noalloc_err);
    return LS_ERR_WORKSPACE_TOO_SMALL;
  }
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    snprintf(g_noalloc_err, sizeof(g_noalloc_err), "ls_replay_fwd_noalloc: no usable device (%s)",
             cudaGetErrorString(e));
    ls::set_last_error(g_noalloc_err);
    return LS_ERR_CUDA;
  }
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_fwd_scratch);
      if (e != cudaSuccess || !p) {
        snprintf(g_noalloc_err, sizeof(g_noalloc_err),
                 "ls_replay_fwd_noalloc: cannot resolve the static scratch on device %d (%s)", dev,
                 cudaGetErrorString(e));
        ls::set_last_error(g_noalloc_err);
        return LS_ERR_CUDA;
      }
      g_scratch_addr[dev] = p;
    }
    scratch = g_scratch_addr[dev];
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  e = cudaMemsetAsync(scratch, 0, ls::kWsHeader, s);  // status word starts at zero
  if (e != cudaSuccess) {
    snprintf(g_noalloc_err, sizeof(g_noalloc_err),
             "ls_replay_fwd_noalloc: clearing the scratch status failed (%s)",
             cudaGetErrorString(e));
    ls::set_last_error(g_noalloc_err);
    return LS_ERR_CUDA;
  }
  return ls_replay_fwd(desc, prompt, q, k_resp, v_resp, resp_len, o, lse, scratch, kScratchBytes,
                       stream);
}

size_t ls_replay_fwd_noalloc_scratch_bytes(void) { return kScratchBytes; }

}  // extern "C"
