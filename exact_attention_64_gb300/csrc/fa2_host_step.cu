// Forward + backward on host buffers, pipelined by head chunks.
//
// Every (batch, head) of the attention is independent ("FlashAttention学习笔记
// (2)", V2中的thread blocks排布: the grid's batch and head axes share nothing),
// so a step over host-resident tensors can be cut into chunks of consecutive
// heads -- contiguous slabs of every [B][H][N][d] tensor -- and run as a
// three-stage pipeline on internal streams:
//   copy stream 1  : host -> device  of chunk c+1 (q, k, v, dO)
//   compute streams: fa2_fwd + fa2_bwd of chunk c, on the stream of its slot
//                    (consecutive chunks' kernels may overlap)
//   copy stream 2  : device -> host  of chunk c-1 (o, lse, dq, dk, dv)
// The first and last chunks are a quarter of the others, since their upload
// and download are not overlapped with anything.
// Two device slots hold a chunk's inputs and outputs; a slot is refilled only
// after the compute and the download of the chunk that used it two chunks
// earlier (event waits). The chain starts after the work already queued on the
// caller's stream and the caller's stream waits for its end, so the call is
// asynchronous like every other entry point. Each chunk runs the same kernels
// on the same per-head data as one whole-tensor launch: the results are the
// same bits.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/fa2.h"

namespace {

constexpr int kSlots = 2;
constexpr int kAutoChunks = 8;

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

struct ChunkLayout {
  size_t t16;      // bytes of one [hc][N][d] 16-bit tensor, rounded to 256
  size_t lse;      // bytes of one [hc][N] fp32 tensor, rounded to 256
  size_t slot;     // bytes of one slot: 8 16-bit tensors + lse, then fa2_bwd's workspace
  size_t bwd_ws;   // fa2_bwd workspace for one chunk
  size_t total;
};

bool layout(int B, int H, int N, int d, int hc, ChunkLayout* L) {
  const long long BH = static_cast<long long>(B) * H;
  if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128) || hc < 1 || hc > BH || hc > 65535)
    return false;
  L->t16 = up256(static_cast<size_t>(hc) * N * d * 2);
  L->lse = up256(static_cast<size_t>(hc) * N * 4);
  L->bwd_ws = up256(fa2_bwd_workspace_size(1, hc, N, d));
  if (L->bwd_ws == 0) return false;
  L->slot = 8 * L->t16 + L->lse + L->bwd_ws;
  L->total = kSlots * L->slot;
  return true;
}

int chunk_heads(int B, int H, int heads_per_chunk) {
  const int BH = B * H;
  if (heads_per_chunk > 0) return heads_per_chunk;
  int hc = (BH + kAutoChunks - 1) / kAutoChunks;
  return hc > 65535 ? 65535 : hc;
}

// Internal streams and events of one device, created on first use.
struct Pipe {
  bool ready = false;
  cudaStream_t up = nullptr, cmp[kSlots] = {}, down = nullptr;
  cudaEvent_t start = nullptr, done[kSlots + 2] = {};  // done: end of every internal stream
  cudaEvent_t uploaded[kSlots] = {}, computed[kSlots] = {}, downloaded[kSlots] = {};
};

constexpr int kMaxDevices = 64;
Pipe g_pipes[kMaxDevices];
// One lock per device: a call holds its device's lock while it enqueues (the
// events of the device's pipeline are shared by its calls); calls on other
// devices proceed.
std::mutex g_pipe_mu[kMaxDevices];

cudaError_t pipe_init(Pipe& p) {
  if (p.ready) return cudaSuccess;
  cudaError_t e = cudaSuccess;
  auto mk_stream = [&](cudaStream_t* s) {
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(s, cudaStreamNonBlocking);
  };
  auto mk_event = [&](cudaEvent_t* ev) {
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
  };
  mk_stream(&p.up);
  for (int s = 0; s < kSlots; ++s) mk_stream(&p.cmp[s]);
  mk_stream(&p.down);
  mk_event(&p.start);
  for (int i = 0; i < kSlots + 2; ++i) mk_event(&p.done[i]);
  for (int s = 0; s < kSlots; ++s) {
    mk_event(&p.uploaded[s]);
    mk_event(&p.computed[s]);
    mk_event(&p.downloaded[s]);
  }
  if (e == cudaSuccess) p.ready = true;
  return e;
}

}  // namespace

extern "C" {

size_t fa2_step_host_workspace_size(int B, int H, int N, int d, int heads_per_chunk) {
  if (B < 1 || H < 1 || heads_per_chunk < 0) return 0;
  ChunkLayout L;
  if (!layout(B, H, N, d, chunk_heads(B, H, heads_per_chunk), &L)) return 0;
  return L.total;
}

int fa2_step_host(const void* q, const void* k, const void* v, const void* dO, void* o, float* lse,
                  void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal, float scale,
                  int dtype, int heads_per_chunk, void* workspace, size_t workspace_bytes,
                  void* stream) {
  if (!q || !k || !v || !dO || !o || !lse || !dq || !dk || !dv || heads_per_chunk < 0 || B < 1 ||
      H < 1)
    return FA2_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA2_ERR_INVALID_ARG;
  if (dtype != FA2_FP16 && dtype != FA2_BF16) return FA2_ERR_INVALID_ARG;
  const int hc = chunk_heads(B, H, heads_per_chunk);
  ChunkLayout L;
  if (!layout(B, H, N, d, hc, &L)) return (d != 64 && d != 128) ? FA2_ERR_UNSUPPORTED : FA2_ERR_INVALID_ARG;
  if (workspace == nullptr || workspace_bytes < L.total) return FA2_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return FA2_ERR_ALIGNMENT;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA2_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_pipe_mu[dev]);
  Pipe& p = g_pipes[dev];
  if (pipe_init(p) != cudaSuccess) return FA2_ERR_CUDA;

  const cudaStream_t caller = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  const int BH = B * H;
  const size_t row16 = static_cast<size_t>(N) * d * 2;  // one head of a 16-bit tensor
  const size_t row32 = static_cast<size_t>(N) * 4;      // one head of lse
  const char* hin[4] = {static_cast<const char*>(q), static_cast<const char*>(k),
                        static_cast<const char*>(v), static_cast<const char*>(dO)};
  char* hout16[4] = {static_cast<char*>(o), static_cast<char*>(dq), static_cast<char*>(dk),
                     static_cast<char*>(dv)};

  cudaError_t e = cudaEventRecord(p.start, caller);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(p.up, p.start, 0);
  for (int i = 0; i < kSlots && e == cudaSuccess; ++i) e = cudaStreamWaitEvent(p.cmp[i], p.start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(p.down, p.start, 0);
  // Chunk sizes: the first upload and the last download are not overlapped
  // with anything, so the first and last chunks are a quarter of the others.
  const int small = hc / 4 > 1 ? hc / 4 : 1;
  auto next_chunk = [&](int rem, bool first) {
    if (first && rem > small) return small;
    if (rem > hc + small) return hc;
    return rem > small ? rem - small : rem;  // <= hc, then the last small chunk
  };
  int st = FA2_OK;
  for (int h0 = 0, c = 0, n = 0; h0 < BH && e == cudaSuccess && st == FA2_OK; h0 += n, ++c) {
    n = next_chunk(BH - h0, c == 0);
    const int s = c % kSlots;
    char* slot = ws + s * L.slot;
    char* din[4] = {slot, slot + L.t16, slot + 2 * L.t16, slot + 3 * L.t16};          // q k v dO
    char* dout[4] = {slot + 4 * L.t16, slot + 5 * L.t16, slot + 6 * L.t16, slot + 7 * L.t16};  // o dq dk dv
    float* dlse = reinterpret_cast<float*>(slot + 8 * L.t16);
    char* bwd_ws = slot + 8 * L.t16 + L.lse;
    // Chunk c computes on the stream of its slot, so consecutive chunks'
    // kernels may overlap and fill each other's tails.
    const cudaStream_t cmp = p.cmp[s];
    const size_t off16 = static_cast<size_t>(h0) * row16, bytes16 = static_cast<size_t>(n) * row16;
    // Upload: the slot's inputs are free once the compute of chunk c - 2 is done.
    if (c >= kSlots) e = cudaStreamWaitEvent(p.up, p.computed[s], 0);
    for (int t = 0; t < 4 && e == cudaSuccess; ++t)
      e = cudaMemcpyAsync(din[t], hin[t] + off16, bytes16, cudaMemcpyHostToDevice, p.up);
    if (e == cudaSuccess) e = cudaEventRecord(p.uploaded[s], p.up);
    // Compute: after the upload, and after the download of chunk c - 2 has read
    // the slot's outputs.
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cmp, p.uploaded[s], 0);
    if (e == cudaSuccess && c >= kSlots) e = cudaStreamWaitEvent(cmp, p.downloaded[s], 0);
    if (e != cudaSuccess) break;
    st = fa2_fwd(din[0], din[1], din[2], dout[0], dlse, 1, n, N, d, causal, scale, dtype, cmp);
    if (st == FA2_OK)
      st = fa2_bwd(din[0], din[1], din[2], dout[0], dlse, din[3], dout[1], dout[2], dout[3], 1, n, N,
                   d, causal, scale, dtype, bwd_ws, L.bwd_ws, cmp);
    if (st != FA2_OK) break;
    e = cudaEventRecord(p.computed[s], cmp);
    // Download.
    if (e == cudaSuccess) e = cudaStreamWaitEvent(p.down, p.computed[s], 0);
    for (int t = 0; t < 4 && e == cudaSuccess; ++t)
      e = cudaMemcpyAsync(hout16[t] + off16, dout[t], bytes16, cudaMemcpyDeviceToHost, p.down);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(reinterpret_cast<char*>(lse) + static_cast<size_t>(h0) * row32, dlse,
                          static_cast<size_t>(n) * row32, cudaMemcpyDeviceToHost, p.down);
    if (e == cudaSuccess) e = cudaEventRecord(p.downloaded[s], p.down);
  }
  // Join: the caller's stream continues after everything queued on the three
  // internal streams, on the error paths too, so that nothing queued here
  // outlives what the caller waits for.
  cudaStream_t internal[kSlots + 2];
  internal[0] = p.up;
  internal[1] = p.down;
  for (int i = 0; i < kSlots; ++i) internal[2 + i] = p.cmp[i];
  cudaError_t ej = cudaSuccess;
  for (int i = 0; i < kSlots + 2; ++i) {
    const cudaError_t a = cudaEventRecord(p.done[i], internal[i]);
    const cudaError_t b = a == cudaSuccess ? cudaStreamWaitEvent(caller, p.done[i], 0) : a;
    if (ej == cudaSuccess) ej = b;
  }
  if (st != FA2_OK) return st;
  if (e == cudaSuccess) e = ej;
  return e == cudaSuccess ? FA2_OK : FA2_ERR_CUDA;
}

}  // extern "C"
