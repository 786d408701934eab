// Backward pass for callers that must not allocate device memory.
//
// fa2_bwd needs a small scratch workspace (the row sums D and L * log2(e), and
// the work counter of its persistent main launch).
// Some callers cannot provide one: code running inside a memory pool they do
// not own, a plugin of a framework whose allocator must not be bypassed, or a
// process that has fixed its device footprint in advance and forbids
// cudaMalloc after start-up. For them fa2_bwd_noalloc keeps that scratch in
// a fixed-size array compiled into the library instead.
#include <cstddef>
#include <mutex>
#include <cuda_runtime.h>

#include "../../include/fa2.h"

namespace {

// Size of the built-in scratch: D and L*log2e take 8 bytes per query row,
// rows padded to 128 per head, and the work counter 256 bytes, so 16 MiB + 256
// serves up to about two million padded rows (for example B*H = 256 heads of
// 8192 rows).
constexpr size_t kNoAllocScratchBytes = (size_t(16) << 20) + 256;
constexpr int kMaxDevices = 64;

// One copy per GPU that loads the library, held until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices];  // device address of g_noalloc_scratch, per device

// The array's name is only a host-side stand-in: the device address has to be
// looked up once per device, with that device current.
int scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA2_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) return FA2_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return FA2_OK;
}

}  // namespace

extern "C" int fa2_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                               const float* lse, const void* dO, void* dq, void* dk, void* dv,
                               int B, int H, int N, int d, int causal, float scale, int dtype,
                               void* stream) {
  const size_t need = fa2_bwd_workspace_size(B, H, N, d);
  if (need == 0)  // invalid sizes: let fa2_bwd name the problem
    return fa2_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, causal, scale, dtype, nullptr, 0,
                   stream);
  if (need > kNoAllocScratchBytes) return FA2_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  const int st = scratch_address(&scratch);
  if (st != FA2_OK) return st;
  // Every scratch entry the kernels read is written first by the
  // preprocessing kernel (padding rows included), so nothing needs clearing.
  return fa2_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, causal, scale, dtype, scratch,
                 kNoAllocScratchBytes, stream);
}
