// FlashAttention-2 backward for sm_103a: two launches on one stream, the
// preprocessing pass and one main launch that runs the dK/dV workers and the
// dQ workers (fa2_bwd_main_kernel).
//
//  1. fa2_bwd_pre_kernel  D_i = sum_c dO[i][c] * O[i][c] in fp32 from the stored
//                         O, and L_i * log2(e). The D shortcut stands in for
//                         rowsum(P o dP) ("大猿搬砖简记", V2 backward, last
//                         paragraph).
//  2. dK/dV workers      K/V outer, Q inner ("FlashAttention学习笔记(2)",
//                         Foward和backward中的thread block划分; "大猿搬砖简记",
//                         V2 backward): one CTA per 128-key column block keeps
//                         K_j, V_j in shared memory and dK_j, dV_j in TMEM while
//                         128-row query tiles stream past; S and P are
//                         recomputed from L ("flash-attention123和ring-attention",
//                         优化1).
//  3. dQ workers         dQ, which accumulates along the key direction (the
//                         "awkward" gradient of the V2 backward), gets a worker
//                         of its own that owns a 128-row query tile and
//                         accumulates dQ in fp32 TMEM over the visible K/V
//                         tiles, recomputing S, dP and dS. This is the split
//                         variant: no atomics, and dQ is bit-reproducible.
//
// Products (tcgen05, 16-bit operands, fp32 accumulate in TMEM):
//   dK/dV worker, per query tile i:  S^T = K Q_i^T, dP^T = V dO_i^T   (SS, M=128 keys, N=128 queries)
//                                    dV += P^T dO_i, dK += dS^T Q_i   (TS, A from TMEM, M=128 keys, N=d)
//   dQ worker, per K/V tile j:       S = Q K_j^T, dP = dO V_j^T        (SS, M=128 queries, N=128 keys)
//                                    dQ += dS K_j                      (TS, A from TMEM, M=128 queries, N=d)
// with P = exp2(S * scale*log2e - L*log2e) and dS = P o (dP - D).
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

struct BwdKvShared {
  uint64_t kv_full;
  uint64_t q_full[2], do_full[2];  // streamed pair ring: Q_i and dO_i landed (separately, so
  uint64_t s_empty[2];             // S^T(i) need not wait for dO_i); both free again
  uint64_t st_full;                // S^T(i) complete
  uint64_t dpt_full;               // dP^T(i) complete
  uint64_t p_done;                 // P^T(i) written over S^T(i) by all 8 compute warps
  uint64_t ds_done;                // dS^T(i) written over dP^T(i) by all 8 compute warps
  uint64_t mma_done;               // every product of the block has completed
  uint32_t tmem_base;
  int abort_flag;
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

struct BwdQShared {
  uint64_t q_full;
  uint64_t k_full[3], k_empty[3];  // K_j ring
  uint64_t v_full[2], v_empty[2];  // V_j ring
  uint64_t st_full, s_free, ds_full, mma_done;
  uint32_t tmem_base;
  int abort_flag;
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
                       float* __restrict__ l2_pad, float* __restrict__ dq_acc, int BH, int N,
                       int n_pad) {
  constexpr int LPR = D / 8;     // lanes per row
  constexpr int RPW = 32 / LPR;  // rows per warp per pass
  constexpr int U = kPrePasses;
  const int lane = threadIdx.x & 31, sub = lane / LPR, li = lane % LPR;
  const long long total = static_cast<long long>(BH) * n_pad;
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

// ---------------------------------------------------------------------------
// 2. dK / dV workers (K/V outer, Q inner)
// ---------------------------------------------------------------------------
// Warp roles: warp 0 TMA; warp 1 issues every product; warps 4-7 and 8-11
// compute P^T and dS^T for query columns [0,64) and [64,128) of each tile
// (TMEM lane = key). P^T(i) replaces S^T(i) in TMEM as soon as it is formed,
// so dV(i) runs before dS^T(i) exists, and dS^T(i) replaces dP^T(i). The
// tensor core runs
//   ... dV(i), S^T(i+1), dK(i), dP^T(i+1), dV(i+1) ...
// in issue order, which also orders each product that overwrites a TMEM region
// after the product that reads it. Two chains cross from tile to tile:
// S^T -> P^T -> dV -> S^T and dP^T -> dS^T -> dK -> dP^T; each holds two
// products and one step of the compute warps, so while the compute warps form
// P^T(i+1) the tensor core runs dK(i) and dP^T(i+1).
// One dK/dV worker (key block nb of batch*head bh), run by a CTA of the
// backward's main launch.
template <int D, bool BF16, bool CAUSAL>
__device__ __forceinline__ void bwd_dkdv_cta(const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                                             const CUtensorMap& tm_v, const CUtensorMap& tm_do,
                                             const CUtensorMap& tm_dk, const CUtensorMap& tm_dv,
                                             const BwdArgs& a, const int nb, const int bh) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  __shared__ BwdKvShared sh;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = a.N;    // queries
  const int Nk = a.Nk;  // keys and values
  const int n0 = nb * kTileRows;
  const int i_begin = bwd_q_tile_begin(nb, CAUSAL);
  // 0 when no query sees these keys (causal, more keys than queries): the
  // block then loads and issues nothing and writes dK = dV = 0.
  const int n_steps = max(0, ceil_div(N, kTileRows) - i_begin);

  if (threadIdx.x == 0) {
    mbar_init(&sh.kv_full, 1);
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&sh.q_full[s], 1);
      mbar_init(&sh.do_full[s], 1);
      mbar_init(&sh.s_empty[s], 1);
    }
    mbar_init(&sh.st_full, 1);
    mbar_init(&sh.dpt_full, 1);
    mbar_init(&sh.p_done, 8);  // the eight compute warps
    mbar_init(&sh.ds_done, 8);
    mbar_init(&sh.mma_done, 1);
    sh.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sh.tmem_base, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;
  volatile int* abort_flag = &sh.abort_flag;
  const WaitCtx wc{a.status, abort_flag, a.timeout_ns};

  if (warp < 4) {
    setmaxnreg_dec<64>();
    if (warp == 0 && lane == 0) {
      // ---------------- TMA producer ----------------
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      if (n_steps > 0) {
        mbar_arrive_expect_tx(&sh.kv_full, 2 * C::TILE_BYTES);
        load_tile<D>(smem + C::OFF_FIX0, &tm_k, &sh.kv_full, n0, bh);
        load_tile<D>(smem + C::OFF_FIX1, &tm_v, &sh.kv_full, n0, bh);
      }
      int i = 0;
      bool ok = true;
      for (; i < n_steps; ++i) {
        const int st = i % C::NS, ph = (i / C::NS) & 1;
        ok = mbar_wait(&sh.s_empty[st], ph ^ 1, wc);
        if (!ok) break;
        const int q0 = (i_begin + i) * kTileRows;
        mbar_arrive_expect_tx(&sh.q_full[st], C::TILE_BYTES);
        load_tile<D>(smem + C::OFF_STR0 + st * C::TILE_BYTES, &tm_q, &sh.q_full[st], q0, bh);
        if (a.fault == 1 && i == 0) continue;  // failure-path test: dO_0 never arrives
        mbar_arrive_expect_tx(&sh.do_full[st], C::TILE_BYTES);
        load_tile<D>(smem + C::OFF_STR1 + st * C::TILE_BYTES, &tm_do, &sh.do_full[st], q0, bh);
      }
      if (!ok) {
        if (n_steps > 0) mbar_wait_drain(&sh.kv_full, 0, a.timeout_ns);
        for (int ii = max(0, i - C::NS); ii < i; ++ii) {
          mbar_wait_drain(&sh.q_full[ii % C::NS], (ii / C::NS) & 1, a.timeout_ns);
          if (!(a.fault == 1 && ii == 0))
            mbar_wait_drain(&sh.do_full[ii % C::NS], (ii / C::NS) & 1, a.timeout_ns);
        }
      }
    } else if (warp == 1) {
      // ---------------- tcgen05.mma issuer (whole warp, one lane issues) ----------------
      const uint32_t k_s = smem_u32(smem + C::OFF_FIX0), v_s = smem_u32(smem + C::OFF_FIX1);
      auto q_at = [&](int i) { return smem_u32(smem + C::OFF_STR0 + (i % C::NS) * C::TILE_BYTES); };
      auto do_at = [&](int i) { return smem_u32(smem + C::OFF_STR1 + (i % C::NS) * C::TILE_BYTES); };
      const uint32_t t_pt = tmem + C::KV_ST, t_dst = tmem + C::KV_DPT;
      auto pt_col = [t_pt](int kk) { return t_pt + C::pair_col(kk); };
      auto dst_col = [t_dst](int kk) { return t_dst + C::pair_col(kk); };
      bool ok = n_steps == 0 ||
                (mbar_wait_warp(&sh.kv_full, 0, wc) && mbar_wait_warp(&sh.q_full[0], 0, wc));
      if (ok && n_steps > 0) {
        tc_fence_after();
        mma_rows_x_rows<D, BF16>(tmem + C::KV_ST, k_s, q_at(0));
        umma_commit_warp(&sh.st_full);
        ok = mbar_wait_warp(&sh.do_full[0], 0, wc);
        if (ok) {
          tc_fence_after();
          mma_rows_x_rows<D, BF16>(tmem + C::KV_DPT, v_s, do_at(0));
          umma_commit_warp(&sh.dpt_full);
        }
      }
      for (int i = 0; i < n_steps && ok; ++i) {
        const int nx = i + 1;
        // dV += P^T(i) dO_i, then S^T(i+1) over the region P^T(i) is read from.
        ok = mbar_wait_warp(&sh.p_done, i & 1, wc);
        if (!ok) break;
        tc_fence_after();
        mma_tmem_x_tile<D, BF16>(tmem + C::KV_DV, pt_col, do_at(i), i > 0);
        if (nx < n_steps) {
          ok = mbar_wait_warp(&sh.q_full[nx % C::NS], (nx / C::NS) & 1, wc);
          if (!ok) break;
          tc_fence_after();
          mma_rows_x_rows<D, BF16>(tmem + C::KV_ST, k_s, q_at(nx));
          umma_commit_warp(&sh.st_full);
        }
        // dK += dS^T(i) Q_i, then dP^T(i+1) over the region dS^T(i) is read
        // from. dK(i) is the last reader of Q_i and dO_i: its commit frees the stage.
        ok = mbar_wait_warp(&sh.ds_done, i & 1, wc);
        if (!ok) break;
        tc_fence_after();
        mma_tmem_x_tile<D, BF16>(tmem + C::KV_DK, dst_col, q_at(i), i > 0);
        umma_commit_warp(&sh.s_empty[i % C::NS]);
        if (nx < n_steps) {
          ok = mbar_wait_warp(&sh.do_full[nx % C::NS], (nx / C::NS) & 1, wc);
          if (!ok) break;
          tc_fence_after();
          mma_rows_x_rows<D, BF16>(tmem + C::KV_DPT, v_s, do_at(nx));
          umma_commit_warp(&sh.dpt_full);
        }
      }
      umma_commit_warp(&sh.mma_done);
      mbar_wait_drain(&sh.mma_done, 0, a.timeout_ns);
    }
  } else {
    setmaxnreg_inc<208>();
    // ---------------- P^T / dS^T warpgroups ----------------
    const int wg = (warp - 4) >> 2;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // key row of the block == TMEM lane
    const int kg = n0 + r;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t t_st = tmem + lane_off + C::KV_ST + 64 * wg;
    const uint32_t t_dpt = tmem + lane_off + C::KV_DPT + 64 * wg;
    const float sl2 = a.scale_log2;
    // This warp's copy of -L*log2e [0,64) and D [64,128) for its 64 query columns.
    float* ld_s = reinterpret_cast<float*>(smem + C::OFF_LD) + (warp - 4) * 128;
    bool ok = true;
    for (int i = 0; i < n_steps; ++i) {
      const int q0 = (i_begin + i) * kTileRows;
      const int qc0 = q0 + 64 * wg;  // first query column of this warpgroup
      {
        // Coalesced loads (they do not depend on S) before waiting for the scores.
        const size_t row = static_cast<size_t>(bh) * a.n_pad + qc0 + 2 * lane;
        const float2 l2v = *reinterpret_cast<const float2*>(a.l2_pad + row);
        const float2 dv2 = *reinterpret_cast<const float2*>(a.dsum_pad + row);
        __syncwarp();  // every lane is done with the previous step's values
        *reinterpret_cast<float2*>(ld_s + 2 * lane) = make_float2(-l2v.x, -l2v.y);
        *reinterpret_cast<float2*>(ld_s + 64 + 2 * lane) = dv2;
        __syncwarp();
      }
      // Shared-memory loads return slowly while the score products stream their
      // operands from shared memory, so -L*log2e (and D below) are loaded into
      // registers ahead of the waits rather than inside the exponent loops.
      float lreg[64];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const float4 l4 = reinterpret_cast<const float4*>(ld_s)[u];
        lreg[4 * u] = l4.x; lreg[4 * u + 1] = l4.y; lreg[4 * u + 2] = l4.z; lreg[4 * u + 3] = l4.w;
      }
      ok = mbar_wait_warp(&sh.st_full, i & 1, wc);
      if (!ok) break;
      __syncwarp();  // the warp-collective TMEM loads below need a converged warp
      tc_fence_after();
      // All 64 columns of S^T into registers; P^T then goes over the first 32.
      uint32_t sv[64];
      tmem_ld_32x32b_x32(t_st, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
      tmem_ld_32x32b_x32(t_st + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
      tmem_wait_ld();
      reg_fence(sv);
      const bool need_mask = (CAUSAL && qc0 < n0 + kTileRows - 1) || (qc0 + 64 > N) ||
                             (n0 + kTileRows > Nk);
      // P^T as 16-bit pairs; dS^T below is formed from these rounded values.
      uint32_t pk[32];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float p[32];
        const uint32_t(&sh_h)[32] = *reinterpret_cast<const uint32_t(*)[32]>(&sv[32 * h]);
        if (need_mask)
          dkdv_p_cols<true, CAUSAL>(sh_h, lreg + 32 * h, sl2, kg, qc0 + 32 * h, N, Nk, p);
        else
          dkdv_p_cols<false, CAUSAL>(sh_h, lreg + 32 * h, sl2, kg, qc0 + 32 * h, N, Nk, p);
#pragma unroll
        for (int j = 0; j < 16; ++j) pk[16 * h + j] = pack_x2<BF16>(p[2 * j], p[2 * j + 1]);
      }
      tmem_st_32x32b_x32(t_st, pk);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.p_done);
      float dreg[64];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const float4 d4 = reinterpret_cast<const float4*>(ld_s + 64)[u];
        dreg[4 * u] = d4.x; dreg[4 * u + 1] = d4.y; dreg[4 * u + 2] = d4.z; dreg[4 * u + 3] = d4.w;
      }

      ok = mbar_wait_warp(&sh.dpt_full, i & 1, wc);
      if (!ok) break;
      __syncwarp();
      tc_fence_after();
      // dS^T = P^T o (dP^T - D) from the rounded P^T, over the first 32 dP^T
      // columns once all 64 have been read.
      uint32_t dsk[32];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t dp[32];
        tmem_ld_32x32b_x32(t_dpt + 32 * h, dp);
        tmem_wait_ld();
        reg_fence(dp);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int c = 32 * h + 2 * j;
          const float2 ds = f2_mul(unpack_x2<BF16>(pk[16 * h + j]),
                                   f2_sub(make_float2(__uint_as_float(dp[2 * j]), __uint_as_float(dp[2 * j + 1])),
                                          make_float2(dreg[c], dreg[c + 1])));
          dsk[16 * h + j] = pack_x2<BF16>(ds.x, ds.y);
        }
      }
      tmem_st_32x32b_x32(t_dpt, dsk);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.ds_done);
    }
    // ---------------- epilogue: dV, scale*dK -> 16-bit, TMA store ----------------
    if (ok) ok = mbar_wait_warp(&sh.mma_done, 0, wc);
    // All MMAs have completed, so the K and V buffers are free for staging.
    uint8_t* stage = smem + (wg == 0 ? C::OFF_FIX1 : C::OFF_FIX0);
    if (ok && n_steps > 0) {
      __syncwarp();
      tc_fence_after();
      stage_rows<D, BF16>(stage, tmem + lane_off + (wg == 0 ? C::KV_DV : C::KV_DK), r,
                          wg == 0 ? 1.f : a.scale);
      fence_proxy_async_smem();
    } else if (ok) {
      // No query sees these keys: their gradients are zero.
#pragma unroll
      for (int sl = 0; sl < D / 64; ++sl)
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(stage + sl * C::SLAB_BYTES + r * 128 + c * 16) = make_uint4(0u, 0u, 0u, 0u);
      fence_proxy_async_smem();
    }
    named_bar_sync(1 + wg, 128);
    if ((threadIdx.x & 127) == 0 && *abort_flag == 0) {
      const CUtensorMap* map = (wg == 0) ? &tm_dv : &tm_dk;
#pragma unroll
      for (int s = 0; s < D / 64; ++s) tma_store_3d(map, stage + s * C::SLAB_BYTES, s * 64, n0, bh);
      bulk_commit_group();
      bulk_wait_group_read0();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// 3. dQ workers (Q outer, K/V inner)
// ---------------------------------------------------------------------------
// Warp roles: warp 0 TMA, warp 1 MMA, warps 4-7 and 8-11 compute dS for key
// columns [0,64) and [64,128) of each K/V tile (TMEM lane = query row).
// One dQ worker (query block of longest-first rank `rank`, batch*head bh),
// run by a CTA of the backward's main launch.
template <int D, bool BF16, bool CAUSAL>
__device__ __forceinline__ void bwd_dq_cta(const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                                           const CUtensorMap& tm_v, const CUtensorMap& tm_do,
                                           const CUtensorMap& tm_dq, const BwdArgs& a,
                                           const int num_m_blocks, const int rank, const int bh) {
  using C = BwdCfg<D>;
  using Q = DqCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  __shared__ BwdQShared sh;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = a.N;
  const int mb = dq_m_block_of(rank, num_m_blocks, CAUSAL);
  const int q0 = mb * kTileRows;
  const int n_kv = fwd_kv_tile_end(q0, min(N, q0 + kTileRows), a.Nk, CAUSAL);

  if (threadIdx.x == 0) {
    mbar_init(&sh.q_full, 1);
    for (int s = 0; s < Q::NK; ++s) { mbar_init(&sh.k_full[s], 1); mbar_init(&sh.k_empty[s], 1); }
    for (int s = 0; s < Q::NV; ++s) { mbar_init(&sh.v_full[s], 1); mbar_init(&sh.v_empty[s], 1); }
    mbar_init(&sh.st_full, 1);
    mbar_init(&sh.s_free, 8);
    mbar_init(&sh.ds_full, 8);
    mbar_init(&sh.mma_done, 1);
    sh.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sh.tmem_base, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;
  volatile int* abort_flag = &sh.abort_flag;
  const WaitCtx wc{a.status, abort_flag, a.timeout_ns};

  if (warp < 4) {
    setmaxnreg_dec<64>();
    if (warp == 0 && lane == 0) {
      // ---------------- TMA producer ----------------
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(&sh.q_full, 2 * C::TILE_BYTES);
      load_tile<D>(smem + Q::OFF_Q, &tm_q, &sh.q_full, q0, bh);
      load_tile<D>(smem + Q::OFF_DO, &tm_do, &sh.q_full, q0, bh);
      int j = 0, kj = 0, vj = 0;  // K_j / V_j loads issued
      bool ok = true;
      for (; j < n_kv; ++j) {
        const int ks = j % Q::NK, vs = j % Q::NV;
        ok = mbar_wait(&sh.k_empty[ks], ((j / Q::NK) & 1) ^ 1, wc);
        if (!ok) break;
        mbar_arrive_expect_tx(&sh.k_full[ks], C::TILE_BYTES);
        load_tile<D>(smem + Q::OFF_K + ks * C::TILE_BYTES, &tm_k, &sh.k_full[ks], j * kTileRows, bh);
        kj = j + 1;
        ok = mbar_wait(&sh.v_empty[vs], ((j / Q::NV) & 1) ^ 1, wc);
        if (!ok) break;
        vj = j + 1;
        if (a.fault == 2 && j == 0) continue;  // failure-path test: V_0 never arrives
        mbar_arrive_expect_tx(&sh.v_full[vs], C::TILE_BYTES);
        load_tile<D>(smem + Q::OFF_V + vs * C::TILE_BYTES, &tm_v, &sh.v_full[vs], j * kTileRows, bh);
      }
      if (!ok) {
        mbar_wait_drain(&sh.q_full, 0, a.timeout_ns);
        for (int jj = max(0, kj - Q::NK); jj < kj; ++jj)
          mbar_wait_drain(&sh.k_full[jj % Q::NK], (jj / Q::NK) & 1, a.timeout_ns);
        for (int jj = max(0, vj - Q::NV); jj < vj; ++jj)
          if (!(a.fault == 2 && jj == 0))
            mbar_wait_drain(&sh.v_full[jj % Q::NV], (jj / Q::NV) & 1, a.timeout_ns);
      }
    } else if (warp == 1) {
      // ---------------- tcgen05.mma issuer (the whole warp; one lane issues) ----------------
      const uint32_t q_s = smem_u32(smem + Q::OFF_Q), do_s = smem_u32(smem + Q::OFF_DO);
      auto k_at = [&](int j) { return smem_u32(smem + Q::OFF_K + (j % Q::NK) * C::TILE_BYTES); };
      auto v_at = [&](int j) { return smem_u32(smem + Q::OFF_V + (j % Q::NV) * C::TILE_BYTES); };
      bool ok = mbar_wait_warp(&sh.q_full, 0, wc) && mbar_wait_warp(&sh.k_full[0], 0, wc) &&
                mbar_wait_warp(&sh.v_full[0], 0, wc);
      if (ok) {
        tc_fence_after();
        mma_rows_x_rows<D, BF16>(tmem + C::Q_S, q_s, k_at(0));
        mma_rows_x_rows<D, BF16>(tmem + C::Q_DP, do_s, v_at(0));
        umma_commit_warp(&sh.st_full);
        umma_commit_warp(&sh.v_empty[0]);  // V_0 is read by dP(0) only
      }
      for (int j = 0; j < n_kv && ok; ++j) {
        const int b = j & 1;
        // S(j), dP(j) have been read into registers: issue the next pair at once.
        ok = mbar_wait_warp(&sh.s_free, j & 1, wc);
        if (!ok) break;
        tc_fence_after();
        if (j + 1 < n_kv) {
          const int jn = j + 1;
          ok = mbar_wait2_warp(&sh.k_full[jn % Q::NK], (jn / Q::NK) & 1, &sh.v_full[jn % Q::NV],
                               (jn / Q::NV) & 1, wc);
          if (!ok) break;
          tc_fence_after();
          mma_rows_x_rows<D, BF16>(tmem + C::Q_S, q_s, k_at(jn));
          mma_rows_x_rows<D, BF16>(tmem + C::Q_DP, do_s, v_at(jn));
          umma_commit_warp(&sh.st_full);
          umma_commit_warp(&sh.v_empty[jn % Q::NV]);
        }
        ok = mbar_wait_warp(&sh.ds_full, j & 1, wc);
        if (!ok) break;
        tc_fence_after();
        const uint32_t ds_col = tmem + C::Q_DS(b);
        mma_tmem_x_tile<D, BF16>(tmem + C::Q_DQ, [ds_col](int kk) { return ds_col + 8u * kk; },
                                       k_at(j), j > 0);
        umma_commit_warp(&sh.k_empty[j % Q::NK]);  // K_j's last reader is dQ(j)
      }
      umma_commit_warp(&sh.mma_done);
      mbar_wait_drain(&sh.mma_done, 0, a.timeout_ns);
    }
  } else {
    setmaxnreg_inc<208>();
    // ---------------- dS warpgroups ----------------
    const int wg = (warp - 4) >> 2;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // query row of the tile == TMEM lane
    const int my_row = q0 + r;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const float sl2 = a.scale_log2;
    const float l2 = a.l2_pad[static_cast<size_t>(bh) * a.n_pad + my_row];
    const float dsum = a.dsum_pad[static_cast<size_t>(bh) * a.n_pad + my_row];
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const int b = j & 1;
      const int kc0 = j * kTileRows + 64 * wg;  // first key column of this warpgroup
      ok = mbar_wait_warp(&sh.st_full, j & 1, wc);
      if (!ok) break;
      __syncwarp();  // the warp-collective TMEM loads below need a converged warp
      tc_fence_after();
      uint32_t s[64], dp[64];
      tmem_ld_32x32b_x32(tmem + lane_off + C::Q_S + 64 * wg, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
      tmem_ld_32x32b_x32(tmem + lane_off + C::Q_S + 64 * wg + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
      tmem_ld_32x32b_x32(tmem + lane_off + C::Q_DP + 64 * wg, *reinterpret_cast<uint32_t(*)[32]>(&dp[0]));
      tmem_ld_32x32b_x32(tmem + lane_off + C::Q_DP + 64 * wg + 32, *reinterpret_cast<uint32_t(*)[32]>(&dp[32]));
      tmem_wait_ld();
      reg_fence(s);
      reg_fence(dp);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.s_free);
      const bool need_mask = (CAUSAL && kc0 + 63 > q0) || (kc0 + 64 > a.Nk) || (q0 + kTileRows > N);
      const int lim = CAUSAL ? min(a.Nk, my_row + 1) : a.Nk;  // keys < lim are visible
      const bool row_ok = my_row < N;
      uint32_t dsp[32];
      if (need_mask)
        dq_ds_cols<true, BF16>(s, dp, sl2, l2, dsum, kc0, lim, row_ok, dsp);
      else
        dq_ds_cols<false, BF16>(s, dp, sl2, l2, dsum, kc0, lim, row_ok, dsp);
      tmem_st_32x32b_x32(tmem + lane_off + C::Q_DS(b) + 32 * wg, dsp);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.ds_full);
    }
    // ---------------- epilogue: scale * dQ -> 16-bit, TMA store ----------------
    if (ok) ok = mbar_wait_warp(&sh.mma_done, 0, wc);
    // Every MMA has completed: the Q buffer is free for staging.
    uint8_t* stage = smem + Q::OFF_Q;
    if (ok && wg == 0) {
      __syncwarp();
      tc_fence_after();
      stage_rows<D, BF16>(stage, tmem + lane_off + C::Q_DQ, r, a.scale);
      fence_proxy_async_smem();
    }
    named_bar_sync(1 + wg, 128);
    if (wg == 0 && (threadIdx.x & 127) == 0 && *abort_flag == 0) {
#pragma unroll
      for (int s = 0; s < D / 64; ++s) tma_store_3d(&tm_dq, stage + s * C::SLAB_BYTES, s * 64, q0, bh);
      bulk_commit_group();
      bulk_wait_group_read0();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// 4. The backward's main launch: the dK/dV workers, then the dQ workers
// ---------------------------------------------------------------------------
// The two passes read the same inputs and D, L from the preprocessing pass,
// and write different outputs, so they share one grid: CTAs [0, kv_ctas) are
// dK/dV workers in the pages' (key block, batch, head) order (key block
// fastest, then batch, then head), the rest dQ workers in the same order over
// the longest-first query-block ranks. CTAs start in index order, so dQ
// workers take the SMs that short dK/dV workers free while the long ones are
// still running.
template <int D, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(384, 1)
    fa2_bwd_main_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                        const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                        const __grid_constant__ CUtensorMap tm_dq, const BwdArgs a, int num_m_blocks,
                        int kv_ctas) {
  const int x = blockIdx.x;
  if (x < kv_ctas) {
    const int nkb = bwd_num_n_blocks(a.Nk);
    const int rest = x / nkb;  // batch + B * head
    bwd_dkdv_cta<D, BF16, CAUSAL>(tm_q, tm_k, tm_v, tm_do, tm_dk, tm_dv, a, x % nkb,
                                  (rest % a.B) * a.H + rest / a.B);
  } else {
    const int y = x - kv_ctas;
    const int rest = y / num_m_blocks;
    bwd_dq_cta<D, BF16, CAUSAL>(tm_q, tm_k, tm_v, tm_do, tm_dq, a, num_m_blocks, y % num_m_blocks,
                                (rest % a.B) * a.H + rest / a.B);
  }
}

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
                                    float* l2, float* dq_acc, int BH, int N, int n_pad,
                                    cudaStream_t stream) {
  const long long rows = static_cast<long long>(BH) * n_pad;
  const long long rows_per_block = 8LL * (32 / (D / 8)) * kPrePasses;  // 8 warps
  long long blocks = (rows + rows_per_block - 1) / rows_per_block;
  const long long cap = static_cast<long long>(num_sms()) * 8;
  if (blocks > cap) blocks = cap;
  fa2_bwd_pre_kernel<D, BF16><<<static_cast<int>(blocks), 256, 0, stream>>>(
      static_cast<const uint16_t*>(o), static_cast<const uint16_t*>(dO), lse, dsum, l2, dq_acc, BH,
      N, n_pad);
  return cudaGetLastError();
}

// The preprocessing pass of both backward variants (dq_acc: nullptr, or the
// fused backward's fp32 dQ accumulator to zero).
cudaError_t launch_bwd_pre(int d, bool bf16, const void* o, const void* dO, const float* lse,
                           float* dsum, float* l2, float* dq_acc, int BH, int N, int n_pad,
                           cudaStream_t stream) {
  if (d == 64 && bf16) return launch_bwd_pre_t<64, true>(o, dO, lse, dsum, l2, dq_acc, BH, N, n_pad, stream);
  if (d == 64 && !bf16) return launch_bwd_pre_t<64, false>(o, dO, lse, dsum, l2, dq_acc, BH, N, n_pad, stream);
  if (d == 128 && bf16) return launch_bwd_pre_t<128, true>(o, dO, lse, dsum, l2, dq_acc, BH, N, n_pad, stream);
  if (d == 128 && !bf16) return launch_bwd_pre_t<128, false>(o, dO, lse, dsum, l2, dq_acc, BH, N, n_pad, stream);
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
    const cudaError_t e = launch_bwd_pre(D, BF16, o, dO, lse, dsum, l2, nullptr, BH, a.N, a.n_pad, stream);
    if (e != cudaSuccess) return e;
  }
  if (ev) cudaEventRecord(ev[1], stream);
  {
    auto kern = fa2_bwd_main_kernel<D, BF16, CAUSAL>;
    const int smem = C::SMEM_ALLOC > DqCfg<D>::SMEM_ALLOC ? C::SMEM_ALLOC : DqCfg<D>::SMEM_ALLOC;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int nm = dq_num_m_blocks(a.N);
    const long long kv_ctas = static_cast<long long>(bwd_num_n_blocks(a.Nk)) * BH;
    const long long total = kv_ctas + static_cast<long long>(nm) * BH;
    if (total > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    kern<<<static_cast<unsigned>(total), C::THREADS, smem, stream>>>(
        maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], maps[6], a, nm, static_cast<int>(kv_ctas));
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
