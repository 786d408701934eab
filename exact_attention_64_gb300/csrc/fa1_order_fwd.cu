// Forward pass in the FlashAttention-1 loop order: K/V blocks outer, Q blocks
// inner ("FlashAttention学习笔记(2)", the FlashAttention-1 forward algorithm
// and the loop-order comparison that motivates FlashAttention-2; "flash-
// attention123和ring-attention", FlashAttention-1 section).
//
// One CTA per (batch, head) -- FlashAttention-1 parallelises over batch and
// heads only. For every K/V block j it visits every query block i that sees
// it; at each step the running output O_i, row max m_i and row sum l_i of that
// block are read from HBM, combined with the step's block result, and written
// back, O_i kept normalised by l_i as in the first version of the algorithm:
//   S = Q_i K_j^T,  m~ = rowmax(S),  P~ = exp(S - m~),  l~ = rowsum(P~),
//   m_new = max(m_i, m~),  l_new = e^(m_i - m_new) l_i + e^(m~ - m_new) l~,
//   O_i <- (l_i e^(m_i - m_new) O_i + e^(m~ - m_new) P~ V_j) / l_new.
// O_i, m_i, l_i live in an fp32 workspace; at the last K/V block of a query
// block the result is written as the 16-bit O and L = m + ln l instead.
// This kernel exists to measure the loop order against the FlashAttention-2
// kernel (fa2_fwd.cu): same tensor-core and TMA machinery, the other order.
//
// Warp roles (6 warps):
//   warp 0    : TMA producer -- K_j and V_j once per j, Q_i through a 2-slot ring
//   warp 1    : tcgen05.mma issuer (converged warp, one lane elected)
//   warps 2-5 : one warpgroup, thread = query row: softmax of step g, then the
//               HBM correction of step g-1 (software pipelined with the MMAs)
// TMEM: S/P of steps g mod 2 in columns [0,128) and [128,256); P V of steps
// g mod 2 in [256, 256+d) and [256+d, 256+2d).
#include <cuda_fp16.h>
#include "fa2_common.cuh"

namespace fa2 {

namespace {

constexpr float kLn2Fa1 = 0.6931471805599453f;

template <int D>
struct Fa1Cfg {
  static constexpr int SLAB_BYTES = kTileRows * 128;
  static constexpr int TILE_BYTES = kTileRows * D * 2;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = TILE_BYTES;
  static constexpr int OFF_Q = 2 * TILE_BYTES;  // two slots
  static constexpr int SMEM_BYTES = 4 * TILE_BYTES;
  static constexpr int SMEM_ALLOC = SMEM_BYTES + 1024;
  static constexpr int THREADS = 192;
  __host__ __device__ static constexpr uint32_t TM_S(int b) { return b ? 128u : 0u; }
  __host__ __device__ static constexpr uint32_t TM_PV(int b) { return b ? 256u + D : 256u; }
  static constexpr uint32_t TM_P_OFF = 64u;
  static constexpr uint32_t TMEM_COLS = 512u;
};

struct Fa1Shared {
  uint64_t kv_full, kv_empty;
  uint64_t q_full[2], q_empty[2];
  uint64_t s_full[2], p_full[2], pv_full[2], pv_free[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort_flag;
};

// First query tile that sees K/V tile j (top-left causal: key <= query).
__device__ __forceinline__ int fa1_i_begin(int j, bool causal) { return causal ? j : 0; }
// Last K/V tile that query tile i sees.
__device__ __forceinline__ int fa1_j_last(int i, int n_tiles, bool causal) {
  return causal ? min(i, n_tiles - 1) : n_tiles - 1;
}

template <int D, bool BF16>
__device__ __forceinline__ void fa1_issue_qk(uint32_t d_tmem, uint32_t q_smem, uint32_t k_smem) {
  constexpr uint32_t idesc = make_idesc_f16(128, 128, BF16, false, false);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = (kk / 4) * Fa1Cfg<D>::SLAB_BYTES + (kk % 4) * 32;
    umma_ss_warp(d_tmem, make_sdesc_sw128(q_smem + off, 16, 1024),
                 make_sdesc_sw128(k_smem + off, 16, 1024), idesc, kk > 0 ? 1u : 0u);
  }
}

template <int D, bool BF16>
__device__ __forceinline__ void fa1_issue_pv(uint32_t o_tmem, uint32_t p_tmem, uint32_t v_smem) {
  constexpr uint32_t idesc = make_idesc_f16(128, D, BF16, false, true);
#pragma unroll
  for (int kk = 0; kk < kTileRows / 16; ++kk)
    umma_ts_warp(o_tmem, p_tmem + kk * 8,
                 make_sdesc_sw128(v_smem + kk * 2048, Fa1Cfg<D>::SLAB_BYTES, 1024), idesc,
                 kk > 0 ? 1u : 0u);
}

template <int D>
__device__ __forceinline__ void fa1_load_tile(uint8_t* dst, const CUtensorMap* map, uint64_t* bar,
                                              int row, int bh) {
#pragma unroll
  for (int s = 0; s < D / 64; ++s)
    tma_load_3d(dst + s * Fa1Cfg<D>::SLAB_BYTES, map, bar, s * 64, row, bh);
}

template <int D, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(192, 1)
    fa1_order_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const Fa1Args a) {
  using C = Fa1Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  __shared__ Fa1Shared sh;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = a.N;
  const int bh = blockIdx.x;
  const int nt = ceil_div(N, kTileRows);

  if (threadIdx.x == 0) {
    mbar_init(&sh.kv_full, 1);
    mbar_init(&sh.kv_empty, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sh.q_full[b], 1);
      mbar_init(&sh.q_empty[b], 1);
      mbar_init(&sh.s_full[b], 1);
      mbar_init(&sh.p_full[b], 4);   // one arrival per warp of the group
      mbar_init(&sh.pv_full[b], 1);
      mbar_init(&sh.pv_free[b], 4);
    }
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

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      bool ok = true;
      int g = 0, j = 0;
      int kv_loaded = 0;  // K/V copies issued (for the drain on abort)
      for (; j < nt && ok; ++j) {
        ok = mbar_wait(&sh.kv_empty, (j & 1) ^ 1, wc);
        if (!ok) break;
        mbar_arrive_expect_tx(&sh.kv_full, 2 * C::TILE_BYTES);
        fa1_load_tile<D>(smem + C::OFF_K, &tm_k, &sh.kv_full, j * kTileRows, bh);
        fa1_load_tile<D>(smem + C::OFF_V, &tm_v, &sh.kv_full, j * kTileRows, bh);
        ++kv_loaded;
        for (int i = fa1_i_begin(j, CAUSAL); i < nt; ++i, ++g) {
          const int qs = g & 1;
          ok = mbar_wait(&sh.q_empty[qs], ((g >> 1) & 1) ^ 1, wc);
          if (!ok) break;
          mbar_arrive_expect_tx(&sh.q_full[qs], C::TILE_BYTES);
          fa1_load_tile<D>(smem + C::OFF_Q + qs * C::TILE_BYTES, &tm_q, &sh.q_full[qs], i * kTileRows, bh);
        }
      }
      if (!ok) {
        // Drain the copies that may still be in flight: the last K/V pair and
        // the last two Q slots.
        if (kv_loaded > 0) mbar_wait_drain(&sh.kv_full, (kv_loaded - 1) & 1, a.timeout_ns);
        for (int gg = max(0, g - 2); gg < g; ++gg)
          mbar_wait_drain(&sh.q_full[gg & 1], (gg >> 1) & 1, a.timeout_ns);
      }
    }
  } else if (warp == 1) {
    // ---------------- tcgen05.mma issuer ----------------
    const uint32_t k_s = smem_u32(smem + C::OFF_K);
    const uint32_t v_s = smem_u32(smem + C::OFF_V);
    bool ok = true;
    int g = 0;
    // P V of step h into PV buffer h mod 2, once its P is in TMEM and the
    // correction of step h - 2 has read that buffer.
    auto issue_pv_step = [&](int h) -> bool {
      if (!mbar_wait2_warp(&sh.p_full[h & 1], (h >> 1) & 1, &sh.pv_free[h & 1], ((h >> 1) & 1) ^ 1, wc))
        return false;
      tc_fence_after();
      fa1_issue_pv<D, BF16>(tmem + C::TM_PV(h & 1), tmem + C::TM_S(h & 1) + C::TM_P_OFF, v_s);
      umma_commit_warp(&sh.pv_full[h & 1]);
      return true;
    };
    for (int j = 0; j < nt && ok; ++j) {
      ok = mbar_wait_warp(&sh.kv_full, j & 1, wc);
      if (!ok) break;
      const int i0 = fa1_i_begin(j, CAUSAL);
      for (int i = i0; i < nt; ++i, ++g) {
        const int qs = g & 1;
        // S of step g. Its buffer was last read (as P) by P V of step g - 2,
        // issued earlier: tcgen05 operations of one CTA run in issue order.
        ok = mbar_wait_warp(&sh.q_full[qs], (g >> 1) & 1, wc);
        if (!ok) break;
        tc_fence_after();
        fa1_issue_qk<D, BF16>(tmem + C::TM_S(qs), smem_u32(smem + C::OFF_Q + qs * C::TILE_BYTES), k_s);
        umma_commit_warp(&sh.s_full[qs]);
        umma_commit_warp(&sh.q_empty[qs]);
        if (i > i0) {
          ok = issue_pv_step(g - 1);
          if (!ok) break;
        }
      }
      if (!ok) break;
      ok = issue_pv_step(g - 1);  // the last step of this K/V block
      if (!ok) break;
      umma_commit_warp(&sh.kv_empty);
    }
    umma_commit_warp(&sh.mma_done);
    mbar_wait_drain(&sh.mma_done, 0, a.timeout_ns);
  } else {
    // ---------------- softmax + correction warpgroup ----------------
    const int quad = warp & 3;                // TMEM lane quadrant of this warp
    const int r = quad * 32 + lane;           // row inside the Q tile
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const float sl2 = a.scale_log2;
    const size_t rows_bh = static_cast<size_t>(bh) * N;
    bool ok = true;
    int g = 0;
    float mt_prev = 0.f, lt_prev = 0.f;  // m~ (scaled, log2 units) and l~ of step g - 1

    auto softmax_step = [&](int i, int j, float& mt, float& lt) -> bool {
      const int b = g & 1;
      if (!mbar_wait_warp(&sh.s_full[b], (g >> 1) & 1, wc)) return false;
      __syncwarp();
      tc_fence_after();
      const uint32_t t_s = tmem + lane_off + C::TM_S(b);
      uint32_t s[128];
#pragma unroll
      for (int c = 0; c < 4; ++c)
        tmem_ld_32x32b_x32(t_s + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&s[32 * c]));
      tmem_wait_ld();
      reg_fence(s);
      const int kv0 = j * kTileRows;
      const int row = i * kTileRows + r;
      const bool need_mask = (kv0 + kTileRows > N) || (CAUSAL && i == j);
      if (need_mask) {
        // At least one key stays: kv0 < N, and on the diagonal key kv0 <= row.
        const int lim = CAUSAL && i == j ? min(N - kv0, row - kv0 + 1) : N - kv0;
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c >= lim) s[c] = __float_as_uint(-INFINITY);
      }
      float mx = __uint_as_float(s[0]);
#pragma unroll
      for (int c = 1; c < 128; ++c) mx = fmaxf(mx, __uint_as_float(s[c]));
      const float neg = -mx * sl2;
      float l0 = 0.f, l1 = 0.f;
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const float p0 = ex2_approx(fmaf(__uint_as_float(s[2 * c]), sl2, neg));
        const float p1 = ex2_approx(fmaf(__uint_as_float(s[2 * c + 1]), sl2, neg));
        l0 += p0;
        l1 += p1;
        s[c] = pack_x2<BF16>(p0, p1);
      }
      const uint32_t t_p = t_s + C::TM_P_OFF;
      tmem_st_32x32b_x32(t_p, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
      tmem_st_32x32b_x32(t_p + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.p_full[b]);
      mt = mx * sl2;
      lt = l0 + l1;
      return true;
    };

    // HBM round trip of step h = (query tile i, K/V tile j) with block stats (mt, lt).
    auto correction_step = [&](int h, int i, int j, float mt, float lt) -> bool {
      const int b = h & 1;
      if (!mbar_wait_warp(&sh.pv_full[b], (h >> 1) & 1, wc)) return false;
      __syncwarp();
      tc_fence_after();
      uint32_t pv[D];
#pragma unroll
      for (int c = 0; c < D / 32; ++c)
        tmem_ld_32x32b_x32(tmem + lane_off + C::TM_PV(b) + 32 * c,
                           *reinterpret_cast<uint32_t(*)[32]>(&pv[32 * c]));
      tmem_wait_ld();
      reg_fence(pv);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.pv_free[b]);
      const int row = i * kTileRows + r;
      if (row < N) {
        const size_t ri = rows_bh + row;
        const bool first = j == 0;  // every query tile is first visited by K/V tile 0
        const bool last = j == fa1_j_last(i, nt, CAUSAL);
        const float m_old = first ? -INFINITY : a.m_acc[ri];
        const float l_old = first ? 0.f : a.l_acc[ri];
        const float m_new = fmaxf(m_old, mt);
        const float alpha = first ? 0.f : ex2_approx(m_old - m_new) * l_old;
        const float beta = ex2_approx(mt - m_new);
        const float l_new = alpha + beta * lt;
        const float inv = 1.f / l_new;
        const float ca = alpha * inv, cb = beta * inv;
        float4* acc = reinterpret_cast<float4*>(a.o_acc + ri * D);
        if (last) {
          uint4* out = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.o) + ri * D);
#pragma unroll
          for (int c = 0; c < D / 8; ++c) {
            float v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = cb * __uint_as_float(pv[8 * c + e]);
            if (!first) {
              const float4 x0 = acc[2 * c], x1 = acc[2 * c + 1];
              v[0] = fmaf(ca, x0.x, v[0]); v[1] = fmaf(ca, x0.y, v[1]);
              v[2] = fmaf(ca, x0.z, v[2]); v[3] = fmaf(ca, x0.w, v[3]);
              v[4] = fmaf(ca, x1.x, v[4]); v[5] = fmaf(ca, x1.y, v[5]);
              v[6] = fmaf(ca, x1.z, v[6]); v[7] = fmaf(ca, x1.w, v[7]);
            }
            out[c] = make_uint4(pack_x2<BF16>(v[0], v[1]), pack_x2<BF16>(v[2], v[3]),
                                pack_x2<BF16>(v[4], v[5]), pack_x2<BF16>(v[6], v[7]));
          }
          a.lse[ri] = (m_new + lg2_approx(l_new)) * kLn2Fa1;
        } else {
#pragma unroll
          for (int c = 0; c < D / 4; ++c) {
            float4 v = make_float4(cb * __uint_as_float(pv[4 * c]), cb * __uint_as_float(pv[4 * c + 1]),
                                   cb * __uint_as_float(pv[4 * c + 2]), cb * __uint_as_float(pv[4 * c + 3]));
            if (!first) {
              const float4 x = acc[c];
              v.x = fmaf(ca, x.x, v.x); v.y = fmaf(ca, x.y, v.y);
              v.z = fmaf(ca, x.z, v.z); v.w = fmaf(ca, x.w, v.w);
            }
            acc[c] = v;
          }
          a.m_acc[ri] = m_new;
          a.l_acc[ri] = l_new;
        }
      }
      return true;
    };

    for (int j = 0; j < nt && ok; ++j) {
      const int i0 = fa1_i_begin(j, CAUSAL);
      for (int i = i0; i < nt; ++i, ++g) {
        float mt, lt;
        ok = softmax_step(i, j, mt, lt);
        if (!ok) break;
        if (i > i0) {
          ok = correction_step(g - 1, i - 1, j, mt_prev, lt_prev);
          if (!ok) break;
        }
        mt_prev = mt;
        lt_prev = lt;
      }
      if (!ok) break;
      ok = correction_step(g - 1, nt - 1, j, mt_prev, lt_prev);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D, bool BF16, bool CAUSAL>
cudaError_t launch_fa1_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const Fa1Args& a, cudaStream_t stream) {
  using C = Fa1Cfg<D>;
  auto kern = fa1_order_fwd_kernel<D, BF16, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  kern<<<a.B * a.H, C::THREADS, C::SMEM_ALLOC, stream>>>(tq, tk, tv, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fa1_order_fwd(int d, bool bf16, bool causal, const CUtensorMap& tq,
                                 const CUtensorMap& tk, const CUtensorMap& tv, const Fa1Args& a,
                                 cudaStream_t stream) {
#define FA1_CASE(DD, BB, CC) \
  if (d == DD && bf16 == BB && causal == CC) return launch_fa1_t<DD, BB, CC>(tq, tk, tv, a, stream);
  FA1_CASE(64, true, false)
  FA1_CASE(64, true, true)
  FA1_CASE(64, false, false)
  FA1_CASE(64, false, true)
  FA1_CASE(128, true, false)
  FA1_CASE(128, true, true)
  FA1_CASE(128, false, false)
  FA1_CASE(128, false, true)
#undef FA1_CASE
  return cudaErrorInvalidValue;
}

}  // namespace fa2
