// bwd_noalloc.cu -- ra_bwd_noalloc: the backward pass for callers that cannot
// allocate device memory.
//
// ra_bwd needs a workspace that the caller allocates: two float32 vectors
// per padded query row (-LSE*log2(e) and -D_vec, rows padded to 128-row
// tiles per ring block).  Some callers cannot do that: a plugin
// running inside a host framework that owns every byte of device memory
// through its own pool and forbids side allocations, or a latency-critical
// path that must not call cudaMalloc (which can synchronise the whole
// device).  For them the workspace lives here instead, in one file-scope
// device array of fixed size that every GPU which loads this library holds
// until the process exits.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>
#include <string>

#include "../../include/ringattn.h"

namespace ra {
void set_last_error(const std::string& msg);  // host.cu: the message ra_last_error() returns
}

namespace {

// Largest workspace ra_bwd_noalloc can serve: 48 MiB, 8 bytes per query row
// (padded to 128-row tiles per block): about 6 million rows B*H*S.
constexpr size_t kScratchBytes = size_t(48) << 20;
static __device__ __align__(256) unsigned char g_bwd_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of g_bwd_scratch on the current device.  Looked up once per
// device, with that device current; the name g_bwd_scratch itself is only a
// host-side handle and must never be handed to a kernel.
int scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    ra::set_last_error(std::string("ra_bwd_noalloc: cudaGetDevice failed: ") + cudaGetErrorString(e));
    return RA_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_bwd_scratch);
    if (e != cudaSuccess || p == nullptr) {
      ra::set_last_error(std::string("ra_bwd_noalloc: cudaGetSymbolAddress failed: ") + cudaGetErrorString(e));
      return RA_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return RA_OK;
}

}  // namespace

extern "C" {

int ra_bwd_noalloc(const void* Q, const void* K, const void* V, const void* O, const float* LSE, const void* dO,
                   void* dQ, void* dK, void* dV, int64_t B, int64_t H, int64_t S, int64_t D, int64_t N,
                   int causal, int layout, int dtype, void* stream) {
  const size_t need = ra_bwd_workspace_bytes(B, H, S, D, N);
  if (need == 0) {
    ra::set_last_error("ra_bwd_noalloc: invalid sizes (B=" + std::to_string(B) + " H=" + std::to_string(H) +
                       " S=" + std::to_string(S) + " D=" + std::to_string(D) + " N=" + std::to_string(N) +
                       "): each must be >= 1, S a multiple of N, and B*H*S*D within range");
    return RA_ERR_ARG;
  }
  if (need > kScratchBytes) {
    ra::set_last_error("ra_bwd_noalloc: these sizes need " + std::to_string(need) +
                       " bytes of workspace, more than the fixed " + std::to_string(kScratchBytes) +
                       " bytes it has; call ra_bwd with a caller-allocated workspace instead");
    return RA_ERR_ARG;
  }
  void* scratch = nullptr;
  int rc = scratch_address(&scratch);
  if (rc != RA_OK) return rc;
  return ra_bwd(Q, K, V, O, LSE, dO, dQ, dK, dV, B, H, S, D, N, causal, layout, dtype, scratch, kScratchBytes,
                stream);
}

}  // extern "C"
