// C ABI of libfa2.so: argument validation, TMA tensor maps, the device status
// word and the kernel launches. Declarations and argument contracts live in
// include/fa2.h.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <functional>
#include <map>
#include <mutex>
#include <queue>
#include <tuple>
#include <vector>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/fa2.h"
#include "fa2_common.cuh"

namespace fa2 {
cudaError_t launch_fwd(int d, bool bf16, bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const CUtensorMap& to, const FwdArgs& a,
                       cudaStream_t stream);
cudaError_t launch_fa1_order_fwd(int d, bool bf16, bool causal, const CUtensorMap& tq,
                                 const CUtensorMap& tk, const CUtensorMap& tv, const Fa1Args& a,
                                 cudaStream_t stream);
cudaError_t launch_bwd(int d, bool bf16, bool causal, const void* o, const void* dO,
                       const float* lse, const CUtensorMap* maps, const BwdArgs& a, float* dsum,
                       float* l2, cudaStream_t stream, cudaEvent_t* ev);
cudaError_t launch_bwd_fused(int d, bool bf16, bool causal, const void* o, const void* dO,
                             const float* lse, const CUtensorMap* maps, const BwdArgs& a, float* dsum,
                             float* l2, float* dq_acc, void* dq, int num_sms, cudaStream_t stream,
                             cudaEvent_t* ev);
}  // namespace fa2

namespace {

// One status word per device: a static device variable, so the library makes
// no allocation of its own.
__device__ int g_device_status;

constexpr int kMaxDevices = 64;
constexpr int kMaxFwdSplits = 128;  // largest K/V split count fa2_fwd_split accepts

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

std::mutex g_mu;
EncodeTiledFn g_encode = nullptr;
int g_arch_ok[kMaxDevices];        // 0 unknown, 1 sm_103, -1 other
int g_num_sms[kMaxDevices];        // multiprocessor count, per device
int* g_status_ptr[kMaxDevices];    // device address of g_device_status, per device
int g_fault_kind = 0;              // armed by fa2_debug_arm_fault, consumed by the next call of its kind
unsigned long long g_fault_timeout_ns = 0;
thread_local int g_last_cuda_error = 0;  // last cudaError_t behind an FA2_ERR_CUDA, per thread

int cuda_fail(cudaError_t e) {
  g_last_cuda_error = static_cast<int>(e);
  return FA2_ERR_CUDA;
}

int current_device(int* dev) {
  return cudaGetDevice(dev) == cudaSuccess && *dev >= 0 && *dev < kMaxDevices ? FA2_OK
                                                                               : FA2_ERR_CUDA;
}

// Per-device set-up: architecture check and the status word's device address.
int device_setup(int* dev_out, int** status_out) {
  int dev = 0;
  if (current_device(&dev) != FA2_OK) return FA2_ERR_CUDA;
  // Binds the device's primary context to the calling thread. The driver-API
  // tensor-map encoder needs a current context, and a thread that has so far
  // only used the runtime lazily (an autograd worker, say) may not have one.
  {
    const cudaError_t e = cudaSetDevice(dev);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_arch_ok[dev] == 0) {
    int major = 0, minor = 0;
    cudaError_t e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e != cudaSuccess) return cuda_fail(e);
    g_arch_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e);
    g_num_sms[dev] = sms > 0 ? sms : 1;
  }
  if (g_arch_ok[dev] != 1) return FA2_ERR_ARCH;
  if (g_status_ptr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_device_status);
    if (e != cudaSuccess) return cuda_fail(e);
    g_status_ptr[dev] = static_cast<int*>(p);
  }
  if (g_encode == nullptr) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
      return FA2_ERR_CUDA;
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  *dev_out = dev;
  *status_out = g_status_ptr[dev];
  return FA2_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

int check_common(int B, int H, int N, int d, int causal, float scale, int dtype) {
  if (B < 1 || H < 1 || N < 1) return FA2_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA2_ERR_INVALID_ARG;
  if (dtype != FA2_FP16 && dtype != FA2_BF16) return FA2_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA2_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA2_ERR_UNSUPPORTED;
  if (B > 65535 || H > 65535) return FA2_ERR_UNSUPPORTED;
  // Row indices of [B*H*N] stay within int32 (TMA coordinates and padded row
  // offsets); element offsets are computed in 64 bits.
  const long long rows = static_cast<long long>(B) * H * (N + 127);
  if (rows > (1LL << 31) - 1) return FA2_ERR_UNSUPPORTED;
  return FA2_OK;
}

// 3-D tensor map over a [B*H][N][d] 16-bit tensor, boxes of box_rows rows
// (128: one tile) x 64 columns (one 128-byte-swizzled slab), zero fill past row
// N of each head; stores clip there.
int make_map_16bit(CUtensorMap* m, const void* ptr, int BH, int N, int d, int dtype,
                   int box_rows = fa2::kTileRows) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(N) * d * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t es[3] = {1, 1, 1};
  const CUresult r =
      g_encode(m, dtype == FA2_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
               3, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    g_last_cuda_error = 1000 + static_cast<int>(r);  // driver codes offset by 1000
    return FA2_ERR_CUDA;
  }
  return FA2_OK;
}

// 3-D tensor map over the fp32 dQ accumulator of fa2_bwd_atomic
// [B*H][n_pad][d]: boxes of 32 rows x 32 columns (rows of 128 bytes, 128-byte
// swizzled), the unit of its reduce-adds (one warp's rows).
int make_map_dqacc(CUtensorMap* m, void* ptr, int BH, int n_pad, int d) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(n_pad),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4, static_cast<cuuint64_t>(n_pad) * d * 4};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t es[3] = {1, 1, 1};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box, es,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    g_last_cuda_error = 1000 + static_cast<int>(r);
    return FA2_ERR_CUDA;
  }
  return FA2_OK;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// N: query length (q, o, lse); Nk: key length (k, v).
int fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
             int Nk, int d, int causal, float scale, int dtype, int* tile_counts, void* stream,
             int num_splits = 1, void* workspace = nullptr, size_t workspace_bytes = 0) {
  if (!q || !k || !v || !o || !lse) return FA2_ERR_INVALID_ARG;
  int st = check_common(B, H, N, d, causal, scale, dtype);
  if (st != FA2_OK) return st;
  st = check_common(B, H, Nk, d, causal, scale, dtype);
  if (st != FA2_OK) return st;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
    return FA2_ERR_ALIGNMENT;
  const size_t tbytes = static_cast<size_t>(B) * H * N * d * 2;   // q, o
  const size_t kbytes = static_cast<size_t>(B) * H * Nk * d * 2;  // k, v
  const size_t lbytes = static_cast<size_t>(B) * H * N * 4;
  const void* ins[3] = {q, k, v};
  const size_t in_bytes[3] = {tbytes, kbytes, kbytes};
  for (int x = 0; x < 3; ++x)
    if (overlap(o, tbytes, ins[x], in_bytes[x]) || overlap(lse, lbytes, ins[x], in_bytes[x]))
      return FA2_ERR_OVERLAP;
  if (overlap(o, tbytes, lse, lbytes)) return FA2_ERR_OVERLAP;
  const int BH = B * H;
  float* o_part = nullptr;
  float* lse_part = nullptr;
  int* part_done = nullptr;
  size_t part_done_bytes = 0;
  if (num_splits > 1) {
    const size_t need = fa2_fwd_split_workspace_size(B, H, N, d, num_splits);
    if (workspace == nullptr || workspace_bytes < need) return FA2_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return FA2_ERR_ALIGNMENT;
    for (int x = 0; x < 3; ++x)
      if (overlap(workspace, need, ins[x], in_bytes[x])) return FA2_ERR_OVERLAP;
    if (overlap(workspace, need, o, tbytes) || overlap(workspace, need, lse, lbytes))
      return FA2_ERR_OVERLAP;
    o_part = static_cast<float*>(workspace);
    const size_t rows = static_cast<size_t>(num_splits) * BH * N;
    lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + align_up(rows * d * 4, 256));
    part_done = reinterpret_cast<int*>(static_cast<char*>(workspace) + align_up(rows * d * 4, 256) +
                                       align_up(rows * 4, 256));
    part_done_bytes = static_cast<size_t>(BH) * fa2::fwd_num_m_blocks(N) * 2 * sizeof(int);
  }
  int dev = 0;
  int* status = nullptr;
  st = device_setup(&dev, &status);
  if (st != FA2_OK) return st;
  CUtensorMap tq, tk, tv, to;
  if (make_map_16bit(&tq, q, BH, N, d, dtype) || make_map_16bit(&tk, k, BH, Nk, d, dtype) ||
      make_map_16bit(&tv, v, BH, Nk, d, dtype) ||
      make_map_16bit(&to, o, BH, N, d, dtype, num_splits > 1 ? fa2::kTileRows : 32))
    return FA2_ERR_CUDA;
  fa2::FwdArgs a{};
  a.lse = lse;
  a.B = B;
  a.H = H;
  a.N = N;
  a.Nk = Nk;
  a.num_m_blocks = fa2::fwd_num_m_blocks(N);
  a.scale_log2 = scale * 1.4426950408889634f;
  a.status = status;
  a.tile_count = tile_counts;
  a.timeout_ns = fa2::kDefaultWaitTimeoutNs;
  a.fault = 0;
  a.num_splits = num_splits;
  a.kv_tiles_max = 0;
  for (int m = 0; m < a.num_m_blocks; ++m)
    a.kv_tiles_max = std::max(a.kv_tiles_max, fa2::fwd_block_tiles(m, N, Nk, causal));
  a.o = o;
  a.o_part = o_part;
  a.lse_part = lse_part;
  a.part_done = part_done;
  a.sched = fa2::fwd_sched_make(BH, a.num_m_blocks, causal, g_num_sms[dev]);
  {
    // An armed failure-path fault is consumed by the next call of its kind:
    // 1 by an unsplit forward, 2 by a split one; both make the producer skip
    // the first V tile.
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_fault_kind == (num_splits <= 1 ? 1 : 2)) {
      a.fault = 1;
      a.timeout_ns = g_fault_timeout_ns;
      g_fault_kind = 0;
    }
  }
  // A non-sticky error left in this thread by another caller would otherwise be
  // reported as ours by the post-launch check.
  (void)cudaGetLastError();
  cudaError_t e = cudaSuccess;
  // The split kernel's arrival counters start at zero on every call.
  if (part_done != nullptr)
    e = cudaMemsetAsync(part_done, 0, part_done_bytes, static_cast<cudaStream_t>(stream));
  if (e == cudaSuccess)
    e = fa2::launch_fwd(d, dtype == FA2_BF16, causal != 0, tq, tk, tv, to, a,
                        static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA2_OK : cuda_fail(e);
}

// ---------------------------------------------------------------------------
// The K/V split count ("大猿搬砖简记", thread-block section, the
// num_splits_heuristic_fwd paragraph): the SM utilisation of every candidate
// split count, the best of them, and the smallest candidate within 0.95 of the
// best. Utilisation, which the page leaves undefined, is read as the fraction
// of the SMs' time spent on K/V tiles: useful tiles / (num_sms * makespan)
// when the launch's CTAs (row blocks longest first, each block's parts in
// order, heads fastest) start in launch order on the SM that frees first, a
// CTA taking its tiles plus kCtaCost, plus kPartCost more if its block is
// split. The costs are in tiles, measured on GB300. Integer arithmetic up to
// the one division per candidate, as in the fp64 reference of the rule.
// ---------------------------------------------------------------------------
constexpr long long kCtaCost = 1;
constexpr long long kPartCost = 6;

double split_utilisation_makespan(const std::vector<int>& tiles, int BH, int num_sms, int s) {
  const int n_max = tiles.empty() ? 0 : tiles[0];
  std::priority_queue<long long, std::vector<long long>, std::greater<long long>> free_at;
  for (int k = 0; k < num_sms; ++k) free_at.push(0);
  long long useful = 0;
  for (const int n : tiles) {
    const int p = fa2::fwd_num_parts(n, s, n_max);
    for (int part = 0; part < p; ++part) {
      int lo = 0, hi = 0;
      fa2::fwd_part_range(n, p, part, &lo, &hi);
      const long long cost = (hi - lo) + kCtaCost + (p > 1 ? kPartCost : 0);
      for (int h = 0; h < BH; ++h) {
        const long long t = free_at.top();
        free_at.pop();
        free_at.push(t + cost);
        useful += hi - lo;
      }
    }
  }
  long long span = 0;
  while (!free_at.empty()) {
    span = std::max(span, free_at.top());
    free_at.pop();
  }
  return span > 0 ? static_cast<double>(useful) / (static_cast<double>(num_sms) * span) : 1.0;
}

std::mutex g_split_mu;
std::map<std::tuple<int, int, int, int>, int> g_split_cache;  // (BH, N, causal, SMs) -> count

int num_splits_makespan(int BH, int N, int causal, int num_sms) {
  const auto key = std::make_tuple(BH, N, causal, num_sms);
  {
    std::lock_guard<std::mutex> lock(g_split_mu);
    const auto it = g_split_cache.find(key);
    if (it != g_split_cache.end()) return it->second;
  }
  // Row blocks in launch order (causal: longest first) with their K/V tiles.
  const int nm = fa2::fwd_num_m_blocks(N);
  std::vector<int> tiles(nm);
  for (int k = 0; k < nm; ++k)
    tiles[k] = fa2::fwd_block_tiles(fa2::fwd_m_block_of(k, nm, causal), N, N, causal);
  const int top = std::max(1, std::min(std::min(kMaxFwdSplits, num_sms), tiles[0]));
  std::vector<double> eff(top + 1, 0.0);
  double best = 0.0;
  eff[1] = split_utilisation_makespan(tiles, BH, num_sms, 1);
  int pick = 1;
  // With utilisation >= 0.95 unsplit, 1 is the smallest candidate within 0.95
  // of any best (<= 1): the other candidates need not be evaluated.
  if (eff[1] < 0.95) {
    for (int s = 1; s <= top; ++s) {
      if (s > 1) eff[s] = split_utilisation_makespan(tiles, BH, num_sms, s);
      best = std::max(best, eff[s]);
    }
    for (int s = 1; s <= top; ++s)
      if (eff[s] >= 0.95 * best) {
        pick = s;
        break;
      }
  }
  std::lock_guard<std::mutex> lock(g_split_mu);
  if (g_split_cache.size() > 4096) g_split_cache.clear();
  g_split_cache[key] = pick;
  return pick;
}

}  // namespace

extern "C" {

int fa2_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
            int d, int causal, float scale, int dtype, void* stream) {
  return fwd_impl(q, k, v, o, lse, B, H, N, N, d, causal, scale, dtype, nullptr, stream);
}

int fa2_fwd_qk(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
               int Nq, int Nk, int d, int causal, float scale, int dtype, void* stream) {
  return fwd_impl(q, k, v, o, lse, B, H, Nq, Nk, d, causal, scale, dtype, nullptr, stream);
}

size_t fa2_fwd_split_workspace_size(int B, int H, int N, int d, int num_splits) {
  if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128) || num_splits < 1 ||
      num_splits > kMaxFwdSplits)
    return 0;
  // [O parts: num_splits x B*H x N x d fp32][lse parts: num_splits x B*H x N fp32]
  // [arrival counters: B*H x ceil(N / 256) x 2 int32]
  const size_t rows = static_cast<size_t>(num_splits) * B * H * N;
  const size_t counters = static_cast<size_t>(B) * H * fa2::fwd_num_m_blocks(N) * 2 * sizeof(int);
  return align_up(rows * d * 4, 256) + align_up(rows * 4, 256) + align_up(counters, 256);
}

int fa2_num_splits(int B, int H, int N, int d, int causal, int num_sms) {
  if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128) || (causal != 0 && causal != 1) ||
      num_sms < 1 || static_cast<long long>(B) * H > (1 << 30))
    return 0;
  return num_splits_makespan(B * H, N, causal, num_sms);
}

int fa2_fwd_split(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                  int N, int d, int causal, float scale, int dtype, int num_splits, void* workspace,
                  size_t workspace_bytes, void* stream) {
  if (num_splits < 1 || num_splits > kMaxFwdSplits) return FA2_ERR_INVALID_ARG;
  return fwd_impl(q, k, v, o, lse, B, H, N, N, d, causal, scale, dtype, nullptr, stream, num_splits,
                  workspace, workspace_bytes);
}

size_t fa2_fwd_kv_outer_workspace_size(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128)) return 0;
  // [O_i: B*H x N x d fp32][m_i: B*H x N fp32][l_i: B*H x N fp32]
  const size_t rows = static_cast<size_t>(B) * H * N;
  return align_up(rows * d * 4, 256) + 2 * align_up(rows * 4, 256);
}

int fa2_fwd_kv_outer(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                     int N, int d, int causal, float scale, int dtype, void* workspace,
                     size_t workspace_bytes, void* stream) {
  if (!q || !k || !v || !o || !lse) return FA2_ERR_INVALID_ARG;
  int st = check_common(B, H, N, d, causal, scale, dtype);
  if (st != FA2_OK) return st;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
    return FA2_ERR_ALIGNMENT;
  const size_t need = fa2_fwd_kv_outer_workspace_size(B, H, N, d);
  if (workspace == nullptr || workspace_bytes < need) return FA2_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return FA2_ERR_ALIGNMENT;
  const size_t tbytes = static_cast<size_t>(B) * H * N * d * 2;
  const size_t lbytes = static_cast<size_t>(B) * H * N * 4;
  const void* ins[3] = {q, k, v};
  for (int x = 0; x < 3; ++x)
    if (overlap(o, tbytes, ins[x], tbytes) || overlap(lse, lbytes, ins[x], tbytes) ||
        overlap(workspace, need, ins[x], tbytes))
      return FA2_ERR_OVERLAP;
  if (overlap(o, tbytes, lse, lbytes) || overlap(workspace, need, o, tbytes) ||
      overlap(workspace, need, lse, lbytes))
    return FA2_ERR_OVERLAP;
  int dev = 0;
  int* status = nullptr;
  st = device_setup(&dev, &status);
  if (st != FA2_OK) return st;
  const int BH = B * H;
  CUtensorMap tq, tk, tv;
  if (make_map_16bit(&tq, q, BH, N, d, dtype) || make_map_16bit(&tk, k, BH, N, d, dtype) ||
      make_map_16bit(&tv, v, BH, N, d, dtype))
    return FA2_ERR_CUDA;
  const size_t rows = static_cast<size_t>(BH) * N;
  char* ws = static_cast<char*>(workspace);
  fa2::Fa1Args a{};
  a.o = o;
  a.lse = lse;
  a.o_acc = reinterpret_cast<float*>(ws);
  a.m_acc = reinterpret_cast<float*>(ws + align_up(rows * d * 4, 256));
  a.l_acc = reinterpret_cast<float*>(ws + align_up(rows * d * 4, 256) + align_up(rows * 4, 256));
  a.B = B;
  a.H = H;
  a.N = N;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.status = status;
  a.timeout_ns = fa2::kDefaultWaitTimeoutNs;
  (void)cudaGetLastError();
  const cudaError_t e = fa2::launch_fa1_order_fwd(d, dtype == FA2_BF16, causal != 0, tq, tk, tv, a,
                                                  static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA2_OK : cuda_fail(e);
}

int fa2_fwd_instrumented(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                         int H, int N, int d, int causal, float scale, int dtype, int* tile_counts,
                         void* stream) {
  return fwd_impl(q, k, v, o, lse, B, H, N, N, d, causal, scale, dtype, tile_counts, stream);
}

size_t fa2_bwd_workspace_size(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128)) return 0;
  // [D: B*H x N_pad fp32][L*log2e: B*H x N_pad fp32][work counter: 256 bytes],
  // N_pad = N rounded up to the 128-row tile of the backward kernels.
  const size_t bh = static_cast<size_t>(B) * H;
  const size_t n_pad = align_up(static_cast<size_t>(N), 128);
  return 2 * align_up(bh * n_pad * 4, 256) + 256;
}

size_t fa2_bwd_atomic_workspace_size(int B, int H, int N, int d) {
  const size_t rows = fa2_bwd_workspace_size(B, H, N, d);
  if (rows == 0) return 0;
  // ... followed by the fp32 dQ accumulator [B*H][N_pad][d].
  const size_t n_pad = align_up(static_cast<size_t>(N), 128);
  return rows + align_up(static_cast<size_t>(B) * H * n_pad * d * 4, 256);
}

namespace {
// N: query length (q, o, dO, dq, lse); Nk: key length (k, v, dk, dv).
// atomic = 0: the split backward (dK/dV workers and dQ workers in one launch,
// no atomics, bit-reproducible); 1: the column workers with fp32 dQ
// reduce-adds (fa2_bwd_atomic).
int bwd_impl(const void* q, const void* k, const void* v, const void* o, const float* lse,
             const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int Nk, int d,
             int causal, float scale, int dtype, void* workspace, size_t workspace_bytes,
             void* const* phase_events, void* stream, int atomic) {
  if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv) return FA2_ERR_INVALID_ARG;
  int st = check_common(B, H, N, d, causal, scale, dtype);
  if (st != FA2_OK) return st;
  st = check_common(B, H, Nk, d, causal, scale, dtype);
  if (st != FA2_OK) return st;
  const void* in16[5] = {q, k, v, o, dO};
  void* out16[3] = {dq, dk, dv};
  for (const void* p : in16)
    if (!aligned(p, 16)) return FA2_ERR_ALIGNMENT;
  for (void* p : out16)
    if (!aligned(p, 16)) return FA2_ERR_ALIGNMENT;
  if (!aligned(lse, 4)) return FA2_ERR_ALIGNMENT;
  const size_t need = atomic ? fa2_bwd_atomic_workspace_size(B, H, N, d)
                             : fa2_bwd_workspace_size(B, H, N, d);
  if (workspace == nullptr || workspace_bytes < need) return FA2_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return FA2_ERR_ALIGNMENT;
  const size_t qb = static_cast<size_t>(B) * H * N * d * 2;   // q, o, dO, dq
  const size_t kb = static_cast<size_t>(B) * H * Nk * d * 2;  // k, v, dk, dv
  const size_t lbytes = static_cast<size_t>(B) * H * N * 4;
  const size_t in_b[5] = {qb, kb, kb, qb, qb};
  const size_t out_b[3] = {qb, kb, kb};
  for (int x = 0; x < 3; ++x) {
    for (int y = 0; y < 5; ++y)
      if (overlap(out16[x], out_b[x], in16[y], in_b[y])) return FA2_ERR_OVERLAP;
    if (overlap(out16[x], out_b[x], lse, lbytes) || overlap(out16[x], out_b[x], workspace, need))
      return FA2_ERR_OVERLAP;
  }
  if (overlap(dq, qb, dk, kb) || overlap(dq, qb, dv, kb) || overlap(dk, kb, dv, kb))
    return FA2_ERR_OVERLAP;
  for (int y = 0; y < 5; ++y)
    if (overlap(workspace, need, in16[y], in_b[y])) return FA2_ERR_OVERLAP;
  if (overlap(workspace, need, lse, lbytes)) return FA2_ERR_OVERLAP;
  int dev = 0;
  int* status = nullptr;
  st = device_setup(&dev, &status);
  if (st != FA2_OK) return st;
  const int BH = B * H;
  // Tensor maps: q, k, v, dO (loads), dk, dv, dq (stores); all 128-row boxes;
  // fa2_bwd_atomic adds the fp32 dQ accumulator (reduce-adds).
  CUtensorMap maps[8];
  const void* src[7] = {q, k, v, dO, dk, dv, dq};
  const int rows[7] = {N, Nk, Nk, N, Nk, Nk, N};
  for (int i = 0; i < 7; ++i)
    if (make_map_16bit(&maps[i], src[i], BH, rows[i], d, dtype) != FA2_OK) return FA2_ERR_CUDA;
  const size_t n_pad = align_up(static_cast<size_t>(N), 128);
  const size_t lbytes_pad = align_up(static_cast<size_t>(BH) * n_pad * 4, 256);
  float* dsum = static_cast<float*>(workspace);
  float* l2 = reinterpret_cast<float*>(static_cast<char*>(workspace) + lbytes_pad);
  int* item_counter = reinterpret_cast<int*>(static_cast<char*>(workspace) + 2 * lbytes_pad);
  float* dq_acc = reinterpret_cast<float*>(static_cast<char*>(workspace) + 2 * lbytes_pad + 256);
  if (atomic && make_map_dqacc(&maps[7], dq_acc, BH, static_cast<int>(n_pad), d) != FA2_OK)
    return FA2_ERR_CUDA;
  fa2::BwdArgs a{};
  a.l2_pad = l2;
  a.dsum_pad = dsum;
  a.n_pad = static_cast<int>(n_pad);
  a.B = B;
  a.H = H;
  a.N = N;
  a.Nk = Nk;
  a.scale = scale;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.status = status;
  a.timeout_ns = fa2::kDefaultWaitTimeoutNs;
  a.fault = 0;
  a.item_counter = item_counter;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  {
    // Kind 3 is consumed by the next backward of either kind: the producer of
    // the K/V column workers skips the first dO tile. Kind 4 by the next
    // fa2_bwd: the dQ workers' producer skips the first V tile.
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_fault_kind == 3 || (g_fault_kind == 4 && !atomic)) {
      a.fault = g_fault_kind - 2;
      a.timeout_ns = g_fault_timeout_ns;
      g_fault_kind = 0;
    }
  }
  (void)cudaGetLastError();  // see fwd_impl
  cudaEvent_t* ev = reinterpret_cast<cudaEvent_t*>(const_cast<void**>(phase_events));
  const cudaError_t e =
      atomic ? fa2::launch_bwd_fused(d, dtype == FA2_BF16, causal != 0, o, dO, lse, maps, a, dsum,
                                     l2, dq_acc, dq, g_num_sms[dev], static_cast<cudaStream_t>(stream),
                                     ev)
             : fa2::launch_bwd(d, dtype == FA2_BF16, causal != 0, o, dO, lse, maps, a, dsum, l2,
                               static_cast<cudaStream_t>(stream), ev);
  return e == cudaSuccess ? FA2_OK : cuda_fail(e);
}
}  // namespace

int fa2_bwd_timed(const void* q, const void* k, const void* v, const void* o, const float* lse,
                  const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                  int causal, float scale, int dtype, void* workspace, size_t workspace_bytes,
                  void* const* phase_events, void* stream) {
  return bwd_impl(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, N, d, causal, scale, dtype, workspace,
                  workspace_bytes, phase_events, stream, 0);
}

int fa2_bwd_atomic(const void* q, const void* k, const void* v, const void* o, const float* lse,
                   const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                   int causal, float scale, int dtype, void* workspace, size_t workspace_bytes,
                   void* stream) {
  return bwd_impl(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, N, d, causal, scale, dtype, workspace,
                  workspace_bytes, nullptr, stream, 1);
}

int fa2_bwd_atomic_timed(const void* q, const void* k, const void* v, const void* o,
                         const float* lse, const void* dO, void* dq, void* dk, void* dv, int B,
                         int H, int N, int d, int causal, float scale, int dtype, void* workspace,
                         size_t workspace_bytes, void* const* phase_events, void* stream) {
  return bwd_impl(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, N, d, causal, scale, dtype, workspace,
                  workspace_bytes, phase_events, stream, 1);
}

int fa2_bwd_qk(const void* q, const void* k, const void* v, const void* o, const float* lse,
               const void* dO, void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d,
               int causal, float scale, int dtype, void* workspace, size_t workspace_bytes,
               void* stream) {
  return bwd_impl(q, k, v, o, lse, dO, dq, dk, dv, B, H, Nq, Nk, d, causal, scale, dtype,
                  workspace, workspace_bytes, nullptr, stream, 0);
}

int fa2_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
            const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal,
            float scale, int dtype, void* workspace, size_t workspace_bytes, void* stream) {
  return fa2_bwd_timed(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, causal, scale, dtype,
                       workspace, workspace_bytes, nullptr, stream);
}

int fa2_get_device_status(void* stream) {
  int dev = 0;
  int* status = nullptr;
  const int st = device_setup(&dev, &status);
  if (st != FA2_OK) return st;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  int h = 0;
  e = cudaMemcpy(&h, status, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e);
  if (h != 0) {
    const int zero = 0;
    if (cudaMemcpy(status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      return FA2_ERR_CUDA;
  }
  return h == 0 ? FA2_OK : h;
}

const char* fa2_status_string(int status) {
  switch (status) {
    case FA2_OK: return "FA2_OK";
    case FA2_ERR_INVALID_ARG: return "FA2_ERR_INVALID_ARG";
    case FA2_ERR_UNSUPPORTED: return "FA2_ERR_UNSUPPORTED";
    case FA2_ERR_ALIGNMENT: return "FA2_ERR_ALIGNMENT";
    case FA2_ERR_ARCH: return "FA2_ERR_ARCH";
    case FA2_ERR_CUDA: return "FA2_ERR_CUDA";
    case FA2_ERR_DEVICE_TIMEOUT: return "FA2_ERR_DEVICE_TIMEOUT";
    case FA2_ERR_WORKSPACE: return "FA2_ERR_WORKSPACE";
    case FA2_ERR_OVERLAP: return "FA2_ERR_OVERLAP";
    default: return "FA2_ERR_UNKNOWN";
  }
}

int fa2_fwd_grid(int B, int H, int N, int grid_out[3], int* rows_per_cta) {
  if (B < 1 || H < 1 || N < 1 || grid_out == nullptr) return FA2_ERR_INVALID_ARG;
  grid_out[0] = fa2::fwd_num_m_blocks(N);
  grid_out[1] = B;
  grid_out[2] = H;
  if (rows_per_cta) *rows_per_cta = fa2::kFwdRowsPerCta;
  return FA2_OK;
}

int fa2_fwd_block_work(int block_x, int N, int causal, int* row_begin, int* row_end,
                       int* kv_tiles) {
  const int nm = N >= 1 ? fa2::fwd_num_m_blocks(N) : 0;
  if (N < 1 || block_x < 0 || block_x >= nm || (causal != 0 && causal != 1))
    return FA2_ERR_INVALID_ARG;
  const int mb = fa2::fwd_m_block_of(block_x, nm, causal);
  const int r0 = mb * fa2::kFwdRowsPerCta;
  const int r1 = r0 + fa2::kFwdRowsPerCta < N ? r0 + fa2::kFwdRowsPerCta : N;
  if (row_begin) *row_begin = r0;
  if (row_end) *row_end = r1;
  if (kv_tiles) *kv_tiles = fa2::fwd_kv_tile_end(r0, r1, N, causal);
  return FA2_OK;
}

int fa2_fwd_schedule(int B, int H, int N, int causal, int num_sms, int* num_ctas, int* cta_of_block,
                     int* pos_of_block) {
  if (B < 1 || H < 1 || N < 1 || num_sms < 1 || (causal != 0 && causal != 1) || num_ctas == nullptr)
    return FA2_ERR_INVALID_ARG;
  const int nm = fa2::fwd_num_m_blocks(N);
  if (static_cast<long long>(B) * H * nm > (1LL << 31) - 1) return FA2_ERR_UNSUPPORTED;
  const fa2::FwdSched s = fa2::fwd_sched_make(B * H, nm, causal, num_sms);
  *num_ctas = s.G;
  if (cta_of_block == nullptr && pos_of_block == nullptr) return FA2_OK;
  const long long blocks = static_cast<long long>(B) * H * nm;
  for (long long i = 0; i < blocks; ++i) {
    if (cta_of_block) cta_of_block[i] = -1;
    if (pos_of_block) pos_of_block[i] = -1;
  }
  for (int c = 0; c < s.G; ++c) {
    fa2::FwdCursor cur{};
    int hb = 0, rank = 0;
    for (int k = 0; fa2::fwd_sched_next(s, c, cur, &hb, &rank); ++k) {
      if (hb < 0 || hb >= B * H || rank < 0 || rank >= nm) return FA2_ERR_INVALID_ARG;
      const long long lin = static_cast<long long>(hb) * nm + rank;
      if (cta_of_block) cta_of_block[lin] = c;
      if (pos_of_block) pos_of_block[lin] = k;
    }
  }
  return FA2_OK;
}

int fa2_last_cuda_error(void) { return g_last_cuda_error; }

int fa2_debug_arm_fault(int kind, int timeout_ms) {
  if (kind < 0 || kind > 4) return FA2_ERR_INVALID_ARG;
  if (kind != 0 && (timeout_ms < 1 || timeout_ms > 5000)) return FA2_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mu);
  g_fault_kind = kind;
  g_fault_timeout_ns = static_cast<unsigned long long>(timeout_ms) * 1000000ull;
  return FA2_OK;
}

}  // extern "C"
