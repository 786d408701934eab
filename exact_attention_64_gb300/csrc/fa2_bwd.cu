// FlashAttention-2 backward for sm_103a: two launches on one stream, the
// preprocessing pass and one main launch (fa2_bwd_main_kernel) whose CTAs run
// the dK/dV workers' and the dQ workers' blocks as work items.
//
//  1. fa2_bwd_pre_kernel  D_i = sum_c dO[i][c] * O[i][c] in fp32 from the stored
//                         O, and L_i * log2(e). The D shortcut stands in for
//                         rowsum(P o dP) ("大猿搬砖简记", V2 backward, last
//                         paragraph). It also zeroes the main launch's work
//                         counter.
//  2. dK/dV items         K/V outer, Q inner ("FlashAttention学习笔记(2)",
//                         Foward和backward中的thread block划分; "大猿搬砖简记",
//                         V2 backward): one item per 128-key column block keeps
//                         K_j, V_j in shared memory and dK_j, dV_j in TMEM while
//                         128-row query tiles stream past; S and P are
//                         recomputed from L ("flash-attention123和ring-attention",
//                         优化1).
//  3. dQ items            dQ, which accumulates along the key direction (the
//                         "awkward" gradient of the V2 backward), gets a worker
//                         of its own that owns a 128-row query tile and
//                         accumulates dQ in fp32 TMEM over the visible K/V
//                         tiles, recomputing S, dP and dS. This is the split
//                         variant: no atomics, and dQ is bit-reproducible.
//
// Products (tcgen05, 16-bit operands, fp32 accumulate in TMEM):
//   dK/dV item, per query tile i:  S^T = K Q_i^T, dP^T = V dO_i^T   (SS, M=128 keys, N=128 queries)
//                                  dV += P^T dO_i, dK += dS^T Q_i   (TS, A from TMEM, M=128 keys, N=d)
//   dQ item, per K/V tile j:       S = Q K_j^T, dP = dO V_j^T        (SS, M=128 queries, N=128 keys)
//                                  dQ += dS K_j                      (TS, A from TMEM, M=128 queries, N=d)
// with P = exp2(S * scale*log2e - L*log2e) and dS = P o (dP - D).
// The CTAs and their warp roles are in fa2_bwd_persist.cuh.
#include <cuda_fp16.h>
#include "fa2_bwd_parts.cuh"
#include "../../include/fa2.h"

namespace fa2 {

template <int D>
struct BwdCfg {
  static constexpr int SLAB_BYTES = kTileRows * 128;    // 128 rows x 128 bytes
  static constexpr int TILE_BYTES = kTileRows * D * 2;  // one 128-row Q, K, V or dO tile
  static constexpr int NS = 2;                          // ring depth of the streamed pair
  static constexpr int OFF_FIX0 = 0;                    // resident pair (K,V) or (Q,dO)
  static constexpr int OFF_FIX1 = TILE_BYTES;
  static constexpr int OFF_STR0 = 2 * TILE_BYTES;       // streamed pair, NS stages each
  static constexpr int OFF_STR1 = OFF_STR0 + NS * TILE_BYTES;
  // dK/dV workers: per-warp copies of L*log2e and D for its 64 query columns
  // (8 warps x 128 floats), read as shared-memory broadcasts.
  static constexpr int OFF_LD = OFF_STR1 + NS * TILE_BYTES;
  static constexpr int SMEM_BYTES = OFF_LD + 8 * 128 * 4;
  // >= 116 KiB so that at most one CTA (one 512-column TMEM allocation) lives on an SM.
  static constexpr int SMEM_ALLOC = (SMEM_BYTES + 1024 > 118784) ? SMEM_BYTES + 1024 : 118784;
  static constexpr int THREADS = 384;
  static constexpr uint32_t TMEM_COLS = 512;
  // dK/dV worker TMEM: dV, dK accumulators, S^T and dP^T. A warpgroup owns 64
  // query columns of each region. Once it has read its S^T columns it writes
  // P^T over the first 32 of them (16-bit pairs, query 2c and 2c+1 in column
  // c), and once it has read its dP^T columns it writes dS^T over the first 32
  // of those, so the A operand of dV (dK) for 16-query block kk sits at column
  // KV_ST (KV_DPT) + 64 * (kk / 4) + 8 * (kk % 4).
  static constexpr uint32_t KV_DV = 0, KV_DK = D, KV_ST = 2 * D, KV_DPT = 2 * D + 128;
  __host__ __device__ static constexpr uint32_t pair_col(int kk) { return 64u * (kk / 4) + 8u * (kk % 4); }
  // dQ worker TMEM: S, dP, the dQ accumulator and two dS buffers.
  static constexpr uint32_t Q_S = 0, Q_DP = 128, Q_DQ = 256;
  __host__ __device__ static constexpr uint32_t Q_DS(int b) { return 256 + D + 64 * b; }
};

// dQ worker shared-memory plan: Q, dO resident; K_j in a 3-deep ring (it is
// read by S(j) and, last, by dQ(j)); V_j in a 2-deep ring (read only by
// dP(j), so it is freed early). 224 KiB at d = 128.
template <int D>
struct DqCfg {
  static constexpr int TILE_BYTES = BwdCfg<D>::TILE_BYTES;
  static constexpr int NK = 3, NV = 2;
  static constexpr int OFF_Q = 0, OFF_DO = TILE_BYTES;
  static constexpr int OFF_K = 2 * TILE_BYTES;
  static constexpr int OFF_V = OFF_K + NK * TILE_BYTES;
  static constexpr int SMEM_BYTES = OFF_V + NV * TILE_BYTES;
  static constexpr int SMEM_ALLOC = (SMEM_BYTES + 1024 > 118784) ? SMEM_BYTES + 1024 : 118784;
};

// ---------------------------------------------------------------------------
// 1. preprocess
// ---------------------------------------------------------------------------
template <int D, bool BF16>
__device__ __forceinline__ float dot8(uint4 x, uint4 y) {
  const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
  float acc = 0.f;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    float x0, x1, y0, y1;
    if constexpr (BF16) {
      x0 = __uint_as_float(xs[w] << 16); x1 = __uint_as_float(xs[w] & 0xffff0000u);
      y0 = __uint_as_float(ys[w] << 16); y1 = __uint_as_float(ys[w] & 0xffff0000u);
    } else {
      const __half2 xh = *reinterpret_cast<const __half2*>(&xs[w]);
      const __half2 yh = *reinterpret_cast<const __half2*>(&ys[w]);
      x0 = __low2float(xh); x1 = __high2float(xh);
      y0 = __low2float(yh); y1 = __high2float(yh);
    }
    acc = fmaf(x0, y0, acc);
    acc = fmaf(x1, y1, acc);
  }
  return acc;
}

// One row is D/8 lanes of 16 bytes, so a warp covers 32/(D/8) rows per pass,
// and each warp keeps kPrePasses passes of loads in flight before reducing.
constexpr int kPrePasses = 4;

// With dq_acc (the fused backward's fp32 dQ accumulator, [BH][n_pad][D]), the
// same pass also zeroes it, padding rows included: each lane clears the D/LPR
// floats of its row that line up with its 8 elements of O.
template <int D, bool BF16>
__global__ void __launch_bounds__(256)
    fa2_bwd_pre_kernel(const uint16_t* __restrict__ o, const uint16_t* __restrict__ dout,
                       const float* __restrict__ lse, float* __restrict__ dsum_pad,
                       float* __restrict__ l2_pad, float* __restrict__ dq_acc,
                       int* __restrict__ item_counter, int BH, int N, int n_pad) {
  constexpr int LPR = D / 8;     // lanes per row
  constexpr int RPW = 32 / LPR;  // rows per warp per pass
  constexpr int U = kPrePasses;
  const int lane = threadIdx.x & 31, sub = lane / LPR, li = lane % LPR;
  const long long total = static_cast<long long>(BH) * n_pad;
  if (item_counter != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *item_counter = 0;
  const long long warp_id = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const long long stride = static_cast<long long>(gridDim.x) * (blockDim.x >> 5) * RPW * U;
  for (long long base = warp_id * RPW * U; base < total; base += stride) {
    uint4 ov[U], dv[U];
    bool valid[U];
    size_t src[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const long long r = base + u * RPW + sub;
      const int bh = static_cast<int>(r / n_pad), i = static_cast<int>(r % n_pad);
      valid[u] = r < total && i < N;
      src[u] = valid[u] ? static_cast<size_t>(bh) * N + i : 0;
      ov[u] = make_uint4(0u, 0u, 0u, 0u);
      dv[u] = make_uint4(0u, 0u, 0u, 0u);
      if (valid[u]) {
        ov[u] = *reinterpret_cast<const uint4*>(o + src[u] * D + li * 8);
        dv[u] = *reinterpret_cast<const uint4*>(dout + src[u] * D + li * 8);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float acc = dot8<D, BF16>(ov[u], dv[u]);
#pragma unroll
      for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      const long long r = base + u * RPW + sub;
      if (li == 0 && r < total) {
        dsum_pad[r] = valid[u] ? acc : 0.f;
        l2_pad[r] = valid[u] ? lse[src[u]] * kLog2e : 0.f;
      }
      if (dq_acc != nullptr && r < total) {
        float4* z = reinterpret_cast<float4*>(dq_acc + r * D + li * 8);
        z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  }
}

}  // namespace fa2

#include "fa2_bwd_persist.cuh"

namespace fa2 {

// ---------------------------------------------------------------------------
// Host-side launcher
// ---------------------------------------------------------------------------
static int g_num_sms = 0;

static int num_sms() {
  if (g_num_sms == 0) {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    g_num_sms = n > 0 ? n : 148;
  }
  return g_num_sms;
}

template <int D, bool BF16>
static cudaError_t launch_bwd_pre_t(const void* o, const void* dO, const float* lse, float* dsum,
                                    float* l2, float* dq_acc, int* item_counter, int BH, int N,
                                    int n_pad, cudaStream_t stream) {
  const long long rows = static_cast<long long>(BH) * n_pad;
  const long long rows_per_block = 8LL * (32 / (D / 8)) * kPrePasses;  // 8 warps
  long long blocks = (rows + rows_per_block - 1) / rows_per_block;
  const long long cap = static_cast<long long>(num_sms()) * 8;
  if (blocks > cap) blocks = cap;
  fa2_bwd_pre_kernel<D, BF16><<<static_cast<int>(blocks), 256, 0, stream>>>(
      static_cast<const uint16_t*>(o), static_cast<const uint16_t*>(dO), lse, dsum, l2, dq_acc,
      item_counter, BH, N, n_pad);
  return cudaGetLastError();
}

// The preprocessing pass of both backward variants (dq_acc: nullptr, or the
// fused backward's fp32 dQ accumulator to zero; item_counter: nullptr, or the
// persistent main launch's work counter to zero).
cudaError_t launch_bwd_pre(int d, bool bf16, const void* o, const void* dO, const float* lse,
                           float* dsum, float* l2, float* dq_acc, int* item_counter, int BH, int N,
                           int n_pad, cudaStream_t stream) {
#define FA2_PRE_CASE(DD, BB) \
  if (d == DD && bf16 == BB) \
    return launch_bwd_pre_t<DD, BB>(o, dO, lse, dsum, l2, dq_acc, item_counter, BH, N, n_pad, stream);
  FA2_PRE_CASE(64, true)
  FA2_PRE_CASE(64, false)
  FA2_PRE_CASE(128, true)
  FA2_PRE_CASE(128, false)
#undef FA2_PRE_CASE
  return cudaErrorInvalidValue;
}

template <int D, bool BF16, bool CAUSAL>
static cudaError_t launch_bwd_t(const void* o, const void* dO, const float* lse,
                                const CUtensorMap* maps, const BwdArgs& a, float* dsum,
                                float* l2, cudaStream_t stream, cudaEvent_t* ev) {
  using C = BwdCfg<D>;
  const int BH = a.B * a.H;
  if (ev) cudaEventRecord(ev[0], stream);
  {
    const cudaError_t e = launch_bwd_pre(D, BF16, o, dO, lse, dsum, l2, nullptr, a.item_counter, BH, a.N, a.n_pad, stream);
    if (e != cudaSuccess) return e;
  }
  if (ev) cudaEventRecord(ev[1], stream);
  {
    auto kern = fa2_bwd_main_kernel<D, BF16, CAUSAL>;
    const int smem = C::SMEM_ALLOC > DqCfg<D>::SMEM_ALLOC ? C::SMEM_ALLOC : DqCfg<D>::SMEM_ALLOC;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int nm = dq_num_m_blocks(a.N);
    const int nkb = bwd_num_n_blocks(a.Nk);
    const long long kv_items = static_cast<long long>(nkb) * BH;
    const long long total = kv_items + static_cast<long long>(nm) * BH;
    if (total > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const long long grid = total < num_sms() ? total : num_sms();
    kern<<<static_cast<unsigned>(grid), C::THREADS, smem, stream>>>(maps[0], maps[1], maps[2], maps[3],
                                                                   a, nm, nkb, kv_items, total);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // The dK/dV and dQ workers share one launch: the third and fourth events
  // both mark its end.
  if (ev) cudaEventRecord(ev[2], stream);
  if (ev) cudaEventRecord(ev[3], stream);
  return cudaSuccess;
}

cudaError_t launch_bwd(int d, bool bf16, bool causal, const void* o, const void* dO,
                       const float* lse, const CUtensorMap* maps, const BwdArgs& a, float* dsum,
                       float* l2, cudaStream_t stream, cudaEvent_t* ev) {
#define FA2_BWD_CASE(DD, BB, CC) \
  if (d == DD && bf16 == BB && causal == CC) \
    return launch_bwd_t<DD, BB, CC>(o, dO, lse, maps, a, dsum, l2, stream, ev);
  FA2_BWD_CASE(64, true, false)
  FA2_BWD_CASE(64, true, true)
  FA2_BWD_CASE(64, false, false)
  FA2_BWD_CASE(64, false, true)
  FA2_BWD_CASE(128, true, false)
  FA2_BWD_CASE(128, true, true)
  FA2_BWD_CASE(128, false, false)
  FA2_BWD_CASE(128, false, true)
#undef FA2_BWD_CASE
  return cudaErrorInvalidValue;
}

}  // namespace fa2

extern "C" int fa2_bwd_grid(int B, int H, int N, int d, int grid_out[3], int* keys_per_cta,
                            int* q_rows_per_tile) {
  if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128) || !grid_out) return FA2_ERR_INVALID_ARG;
  grid_out[0] = fa2::bwd_num_n_blocks(N);
  grid_out[1] = B;
  grid_out[2] = H;
  if (keys_per_cta) *keys_per_cta = fa2::kTileRows;
  if (q_rows_per_tile) *q_rows_per_tile = fa2::kTileRows;
  return FA2_OK;
}

extern "C" int fa2_bwd_block_work(int block_x, int N, int d, int causal, int* key_begin,
                                  int* key_end, int* q_tile_begin, int* q_tile_end) {
  if (N < 1 || (d != 64 && d != 128) || block_x < 0 || block_x >= fa2::bwd_num_n_blocks(N) ||
      (causal != 0 && causal != 1))
    return FA2_ERR_INVALID_ARG;
  const int k0 = block_x * fa2::kTileRows;
  if (key_begin) *key_begin = k0;
  if (key_end) *key_end = (k0 + fa2::kTileRows < N) ? k0 + fa2::kTileRows : N;
  if (q_tile_begin) *q_tile_begin = fa2::bwd_q_tile_begin(block_x, causal);
  if (q_tile_end) *q_tile_end = fa2::ceil_div(N, fa2::kTileRows);
  return FA2_OK;
}
