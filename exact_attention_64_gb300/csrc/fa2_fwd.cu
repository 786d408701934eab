// FlashAttention-2 forward for sm_103a (tcgen05 + TMA + TMEM).
//
// What it computes (per (batch, head), rows independent):
//   S = scale * Q K^T, causal mask j > i -> -inf,
//   O = softmax(S) V,   L = m + ln(l)  (logsumexp, the only statistic stored).
// The loop order is the FlashAttention-2 one: Q is the outer loop (each CTA
// owns query rows), K/V is the inner loop streamed through shared memory, and
// nothing but O and L ever leaves the chip ("FlashAttention学习笔记(2)", opening
// section; "flash-attention123和ring-attention", 优化1). The online softmax keeps
// a running row max m and row sum l; O accumulates un-normalised and is divided
// by l once at the end ("flash-attention123和ring-attention", 优化2). K/V tiles
// that the causal mask hides completely are skipped, not loaded (优化3).
//
// GB300 mapping (one CTA = two 128-row Q tiles "A" and "B" of one head):
//   warp 0        TMA producer: Q_A, Q_B once, then K_j through a multi-stage
//                 shared-memory ring (mbarrier full/empty pairs).
//   warp 3        TMA producer of the V_j ring.
//   warp 1        tcgen05.mma issuer (the whole warp, one lane elected):
//                 S_t = Q_t K_j^T into TMEM, O_t += P_t V_j with P_t read
//                 straight from TMEM.
//   warps 4-7     softmax of tile A, warps 8-11 softmax of tile B. TMEM lane i
//                 is query row i, so one thread owns one whole row: the row max
//                 and row sum need no shuffles. The two tiles ping-pong, so the
//                 tensor core works on one tile while the other's exponentials
//                 run.
// TMEM (512 columns): S_A [0,128) S_B [128,256) O_A [256,256+d) O_B [256+d,256+2d).
// P_t (16-bit, two per column) overwrites the upper half of S_t.
// Rescaling of O is lazy: the reference max only moves when the row max grows
// by more than kRescaleLog2 (in log2 units). Using a stale, smaller reference
// max is exact -- O and l share it and the final O / l cancels it -- and
// bounds every P by 2^kRescaleLog2, so nothing overflows.
#include "fa2_common.cuh"

namespace fa2 {

constexpr float kRescaleLog2 = 8.0f;
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct FwdCfg {
  static constexpr int SLAB_BYTES = kTileRows * 128;     // 128 rows x 128 bytes (64 elems)
  static constexpr int TILE_BYTES = kTileRows * D * 2;   // one Q, K or V tile
  static constexpr int NK = (D == 128) ? 2 : 4;          // K ring depth
  static constexpr int NV = (D == 128) ? 2 : 4;          // V ring depth
  static constexpr int OFF_Q = 0;                        // Q_A, Q_B
  static constexpr int OFF_K = 2 * TILE_BYTES;
  static constexpr int OFF_V = OFF_K + NK * TILE_BYTES;
  static constexpr int SMEM_BYTES = OFF_V + NV * TILE_BYTES;
  static constexpr int SMEM_ALLOC = SMEM_BYTES + 1024;   // slack for 1024-byte alignment
  static constexpr int THREADS = 384;
  __host__ __device__ static constexpr uint32_t TM_S(int t) { return t ? 128u : 0u; }
  __host__ __device__ static constexpr uint32_t TM_O(int t) { return t ? 256u + D : 256u; }
  static constexpr uint32_t TM_P_OFF = 64u;
  static constexpr uint32_t TMEM_COLS = 512u;
};

template <int D>
struct FwdShared {
  uint64_t q_full;
  uint64_t k_full[FwdCfg<D>::NK], k_empty[FwdCfg<D>::NK];
  uint64_t v_full[FwdCfg<D>::NV], v_empty[FwdCfg<D>::NV];
  uint64_t s_full[2], p_full[2], o_full[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort_flag;
  int work[4];  // split mode: row block, batch*head, part, part count
  int merge[2];  // split mode: this CTA's row tile t arrived last and merges it
};

// Merge of a row tile's K/V parts, run by the warpgroup whose part arrived
// last ("大猿搬砖简记", thread-block section: the partial results of the
// blocks that share a worker's K/V range are combined to recover the global
// softmax). Part s of a row holds O_s = (sum over its keys of exp(S - m_s) V)
// / l_s and lse_s = m_s + ln l_s (-inf: no key of the part is visible); then
//   L = ln sum_s exp(lse_s),   O = sum_s exp(lse_s - L) O_s,
// with O rounded once to the 16-bit type. Each warp merges its 32 rows: lane =
// row reads its row's logsumexps (32 parts per batch of loads, all in flight
// together), forms L with a running max, and stages the weights in the warp's
// 4 KiB shared slice (XOR-swizzled); then the lanes cover 4 rows x 64 columns
// per part so that every read of the parts is a whole 128-byte segment and 16
// reads are in flight per lane and part. The parts were written by other CTAs:
// they are read through L2 (ld.global.cg).
template <int D, bool BF16>
__device__ __forceinline__ void fwd_merge_rows(const FwdArgs& a, int bh, int wrow0, int parts,
                                               int lane, float* wsm) {
  constexpr float kLog2e = 1.4426950408889634f;
  const int N = a.N;
  const size_t bhn = static_cast<size_t>(a.B) * a.H * N;
  const size_t rbase = static_cast<size_t>(bh) * N;
  const int my_row = wrow0 + lane;
  const bool row_in = my_row < N;
  // This lane's logsumexps of parts [s0, s0 + 32).
  auto load_lse = [&](int s0, float (&l)[32]) {
#pragma unroll
    for (int k = 0; k < 32; ++k)
      l[k] = (row_in && s0 + k < parts) ? __ldcg(a.lse_part + (s0 + k) * bhn + rbase + my_row)
                                        : -INFINITY;
  };
  float lb[32];
  float mx = -INFINITY, tot = 0.f;
  for (int s0 = 0; s0 < parts; s0 += 32) {
    load_lse(s0, lb);
    float cm = mx;
#pragma unroll
    for (int k = 0; k < 32; ++k) cm = fmaxf(cm, lb[k]);
    if (cm != -INFINITY) {
      if (mx != -INFINITY) tot *= ex2_approx((mx - cm) * kLog2e);
#pragma unroll
      for (int k = 0; k < 32; ++k) tot += ex2_approx((lb[k] - cm) * kLog2e);  // -inf -> 0
      mx = cm;
    }
  }
  const float L = (mx == -INFINITY) ? -INFINITY : mx + lg2_approx(tot) * kLn2;
  if (row_in) a.lse[rbase + my_row] = L;
  // Weights of parts [s0, s0 + 32) of this lane's row: wsm[row][k ^ row]. With
  // at most 32 parts the logsumexps are still in registers.
  auto stage_weights = [&](int s0) {
    if (parts > 32) load_lse(s0, lb);
    __syncwarp();
#pragma unroll
    for (int k = 0; k < 32; ++k)
      wsm[lane * 32 + (k ^ lane)] = (L == -INFINITY) ? 0.f : ex2_approx((lb[k] - L) * kLog2e);
    __syncwarp();
  };
  const int sub = lane >> 3, seg = lane & 7;
  const bool once = parts <= 32;
  if (once) stage_weights(0);
  constexpr int CW = D < 64 ? D : 64;  // columns per pass
#pragma unroll 1
  for (int c = 0; c < D; c += CW) {
    float4 acc[CW / 32][8];
#pragma unroll
    for (int h = 0; h < CW / 32; ++h)
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[h][i] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < parts; s0 += 32) {
      if (!once) stage_weights(s0);
      const int cnt = min(32, parts - s0);
#pragma unroll 2
      for (int k = 0; k < cnt; ++k) {
        const float* src = a.o_part + ((s0 + k) * bhn + rbase) * D + c + seg * 4;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int rr = 4 * i + sub;
          if (wrow0 + rr < N) {
            const float w = wsm[rr * 32 + (k ^ rr)];
#pragma unroll
            for (int h = 0; h < CW / 32; ++h) {
              const float4 x = __ldcg(reinterpret_cast<const float4*>(
                  src + static_cast<size_t>(wrow0 + rr) * D + 32 * h));
              acc[h][i].x = fmaf(w, x.x, acc[h][i].x);
              acc[h][i].y = fmaf(w, x.y, acc[h][i].y);
              acc[h][i].z = fmaf(w, x.z, acc[h][i].z);
              acc[h][i].w = fmaf(w, x.w, acc[h][i].w);
            }
          }
        }
      }
    }
    uint16_t* o16 = static_cast<uint16_t*>(a.o);
#pragma unroll
    for (int h = 0; h < CW / 32; ++h)
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int rr = 4 * i + sub;
        if (wrow0 + rr < N)
          *reinterpret_cast<uint2*>(o16 + (rbase + wrow0 + rr) * D + c + 32 * h + seg * 4) =
              make_uint2(pack_x2<BF16>(acc[h][i].x, acc[h][i].y),
                         pack_x2<BF16>(acc[h][i].z, acc[h][i].w));
      }
  }
}

// S_t = Q_t K^T : M=128 queries, N=128 keys, K=d. Both operands K-major,
// 128-byte swizzled, one 64-element slab per 16 KiB. Issued by a converged
// warp (one lane elected), like every MMA helper in this file.
template <int D, bool BF16>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t q_smem, uint32_t k_smem) {
  constexpr uint32_t idesc = make_idesc_f16(128, 128, BF16, false, false);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = (kk / 4) * FwdCfg<D>::SLAB_BYTES + (kk % 4) * 32;
    umma_ss_warp(d_tmem, make_sdesc_sw128(q_smem + off, 16, 1024),
                 make_sdesc_sw128(k_smem + off, 16, 1024), idesc, kk > 0 ? 1u : 0u);
  }
}

// O_t (+)= P_t V : M=128 queries, N=d, K=128 keys. P from TMEM (16-bit pairs),
// V is [key][d] in shared memory, i.e. MN-major for this product.
template <int D, bool BF16>
__device__ __forceinline__ void issue_pv(uint32_t o_tmem, uint32_t p_tmem, uint32_t v_smem,
                                         bool accumulate) {
  constexpr uint32_t idesc = make_idesc_f16(128, D, BF16, false, true);
#pragma unroll
  for (int kk = 0; kk < kTileRows / 16; ++kk) {
    umma_ts_warp(o_tmem, p_tmem + kk * 8,
                 make_sdesc_sw128(v_smem + kk * 2048, FwdCfg<D>::SLAB_BYTES, 1024), idesc,
                 (accumulate || kk > 0) ? 1u : 0u);
  }
}

template <int D>
__device__ __forceinline__ void tma_load_tile(uint8_t* dst, const CUtensorMap* map,
                                              uint64_t* bar, int row, int bh) {
#pragma unroll
  for (int s = 0; s < D / 64; ++s)
    tma_load_3d(dst + s * FwdCfg<D>::SLAB_BYTES, map, bar, s * 64, row, bh);
}

// One K/V step of a softmax warp, for its row my_row of tile t: S from TMEM,
// the mask, the row max, the lazy rescale of O (exact: O and l share the
// reference max), P into TMEM over the upper half of S, and the arrival on
// p_full. s_par is this step's s_full parity, o_prev_par the previous step's
// o_full parity; first marks the tile's first step. Returns false if a wait
// gave up.
template <int D, bool BF16, bool CAUSAL>
__device__ __forceinline__ bool fwd_softmax_step(uint64_t* s_full, uint64_t* o_full, uint64_t* p_full,
                                                 uint32_t t_s, uint32_t t_p, uint32_t t_o, int kv0,
                                                 int row_base, int my_row, int Nk, float sl2, bool first,
                                                 uint32_t s_par, uint32_t o_prev_par, float& m_ref,
                                                 float& l, int lane, const WaitCtx& wc) {
  bool ok = mbar_wait_warp(s_full, s_par, wc);
  if (!ok) return false;
  __syncwarp();  // the warp-collective TMEM loads below need a converged warp
  tc_fence_after();
  uint32_t s[128];
#pragma unroll
  for (int c = 0; c < 4; ++c)
    tmem_ld_32x32b_x32(t_s + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&s[32 * c]));
  tmem_wait_ld();
  reg_fence(s);
  // Mask keys past the sequence end and, on the diagonal tile, keys after the query.
  const bool need_mask = (kv0 + kTileRows > Nk) || (CAUSAL && kv0 + kTileRows - 1 > row_base);
  if (need_mask) {
    const int lim = CAUSAL ? min(Nk - kv0, my_row - kv0 + 1) : (Nk - kv0);
#pragma unroll
    for (int c = 0; c < 128; ++c)
      if (c >= lim) s[c] = __float_as_uint(-INFINITY);
  }
  // Row max as eight independent chains of three-input maxima (short
  // dependency chains, half the instructions of two-input maxima).
  float mx8[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) mx8[u] = fmaxf(__uint_as_float(s[u]), __uint_as_float(s[8 + u]));
#pragma unroll
  for (int c = 16; c < 128; c += 16)
#pragma unroll
    for (int u = 0; u < 8; ++u)
      mx8[u] = fmax3(mx8[u], __uint_as_float(s[c + u]), __uint_as_float(s[c + 8 + u]));
  const float mx = fmaxf(fmax3(mx8[0], mx8[1], mx8[2]),
                         fmax3(fmax3(mx8[3], mx8[4], mx8[5]), mx8[6], mx8[7]));
  const float m_new = fmaxf(m_ref, mx);
  const bool rescale = (m_new - m_ref) * sl2 > kRescaleLog2;  // also true when m_ref = -inf
  float alpha = 1.f;
  if (rescale) {
    alpha = ex2_approx((m_ref - m_new) * sl2);
    m_ref = m_new;
  }
  const float neg = (m_ref == -INFINITY) ? 0.f : -m_ref * sl2;
  // Packed fp32 pairs (f32x2) for the exponent arguments and the row-sum
  // partials: half the FMA-pipe instructions of the scalar form, same
  // results. rs[k] accumulates columns 8u+2k and 8u+2k+1.
  float2 rs[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                  make_float2(0.f, 0.f)};
  const float2 sl2x2 = make_float2(sl2, sl2), negx2 = make_float2(neg, neg);
#pragma unroll
  for (int c = 0; c < 64; ++c) {
    const float2 x = f2_fma(make_float2(__uint_as_float(s[2 * c]), __uint_as_float(s[2 * c + 1])),
                            sl2x2, negx2);
    const float2 p = make_float2(ex2_approx(x.x), ex2_approx(x.y));
    rs[c & 3] = f2_add(rs[c & 3], p);
    s[c] = pack_x2<BF16>(p.x, p.y);
  }
  l = l * alpha + (((rs[0].x + rs[0].y) + (rs[1].x + rs[1].y)) +
                   ((rs[2].x + rs[2].y) + (rs[3].x + rs[3].y)));
  tmem_st_32x32b_x32(t_p, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
  tmem_st_32x32b_x32(t_p + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
  tmem_wait_st();
  if (!first && __any_sync(0xffffffffu, rescale)) {
    // O_t still holds the sum up to the previous step: wait for that product, then rescale.
    ok = mbar_wait_warp(o_full, o_prev_par, wc);
    if (!ok) return false;
    __syncwarp();
    tc_fence_after();
#pragma unroll
    for (int c = 0; c < D; c += 32) {
      uint32_t o[32];
      tmem_ld_32x32b_x32(t_o + c, o);
      tmem_wait_ld();
      reg_fence(o);
#pragma unroll
      for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
      tmem_st_32x32b_x32(t_o + c, o);
    }
    tmem_wait_st();
  }
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(p_full);
  return true;
}

template <int D, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(384, 1)
    fa2_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                   const FwdArgs a) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  __shared__ FwdShared<D> sh;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = a.N;    // queries
  const int Nk = a.Nk;  // keys and values
  const int S = a.num_splits > 1 ? a.num_splits : 1;
  if (threadIdx.x == 0) {
    mbar_init(&sh.q_full, 1);
    for (int i = 0; i < C::NK; ++i) { mbar_init(&sh.k_full[i], 1); mbar_init(&sh.k_empty[i], 1); }
    for (int i = 0; i < C::NV; ++i) { mbar_init(&sh.v_full[i], 1); mbar_init(&sh.v_empty[i], 1); }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&sh.s_full[t], 1);
      mbar_init(&sh.p_full[t], 4);  // one arrival per softmax warp
      mbar_init(&sh.o_full[t], 1);
    }
    mbar_init(&sh.mma_done, 1);
    sh.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sh.tmem_base, C::TMEM_COLS);
    tmem_relinquish();
  }
  // Split mode: one warp places this CTA (row blocks ranked longest first).
  if (S > 1 && warp == 2)
    split_locate(blockIdx.x, a.num_m_blocks, S, a.kv_tiles_max, a.B * a.H, lane,
                 [&](int k, int* blk, int* tiles) {
                   *blk = fwd_m_block_of(k, a.num_m_blocks, CAUSAL);
                   *tiles = fwd_block_tiles(*blk, N, Nk, CAUSAL);
                 },
                 sh.work);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // Without a split the grid is (row block, batch, head) with one part per
  // block; with one it is 1-D and the locator above placed this CTA.
  const int mb = S > 1 ? sh.work[0] : fwd_m_block_of(blockIdx.x, a.num_m_blocks, CAUSAL);
  const int bh = S > 1 ? sh.work[1] : blockIdx.y * a.H + blockIdx.z;
  const int split = S > 1 ? sh.work[2] : 0;
  const int parts = S > 1 ? sh.work[3] : 1;
  const int row0 = mb * kFwdRowsPerCta;
  const int rows_a = min(kTileRows, N - row0);
  const int rows_b = max(0, min(kTileRows, N - row0 - kTileRows));
  // Per-tile values are kept as scalars: a two-element array indexed by the
  // warp's tile would live in local memory and be reloaded in the loops.
  const int end_a = fwd_kv_tile_end(row0, row0 + rows_a, Nk, CAUSAL);
  const int end_b = fwd_kv_tile_end(row0 + kTileRows, row0 + kTileRows + rows_b, Nk, CAUSAL);
  // This CTA's part [kv_lo, kv_hi) of the block's K/V tiles. Below, j counts
  // tiles within the part (ring slots, phases, first-tile flags); kv_lo + j is
  // the K/V tile itself (TMA coordinates, masks).
  int kv_lo, kv_hi;
  fwd_part_range(max(end_a, end_b), parts, split, &kv_lo, &kv_hi);
  const int n_a = max(0, min(kv_hi, end_a) - kv_lo), n_b = max(0, min(kv_hi, end_b) - kv_lo);
  const int n_total = max(n_a, n_b);
  const uint32_t tmem = sh.tmem_base;
  volatile int* abort_flag = &sh.abort_flag;
  const WaitCtx wc{a.status, abort_flag, a.timeout_ns};

  if (warp < 4) {
    setmaxnreg_dec<64>();
    if (warp == 0 && lane == 0) {
      // ---------------- TMA producer: Q, then the K ring ----------------
      // K and V have producers of their own so that a V slot that frees late
      // (V_j is read by the last products of step j) never holds up K_{j+1}.
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      if (n_total > 0) {  // an empty part loads nothing
        mbar_arrive_expect_tx(&sh.q_full, (rows_b > 0 ? 2 : 1) * C::TILE_BYTES);
        tma_load_tile<D>(smem + C::OFF_Q, &tm_q, &sh.q_full, row0, bh);
        if (rows_b > 0)
          tma_load_tile<D>(smem + C::OFF_Q + C::TILE_BYTES, &tm_q, &sh.q_full, row0 + kTileRows, bh);
      }
      int j = 0;
      bool ok = true;
      for (; j < n_total && ok; ++j) {
        const int ks = j % C::NK, kp = (j / C::NK) & 1;
        ok = mbar_wait(&sh.k_empty[ks], kp ^ 1, wc);
        if (!ok) break;
        mbar_arrive_expect_tx(&sh.k_full[ks], C::TILE_BYTES);
        tma_load_tile<D>(smem + C::OFF_K + ks * C::TILE_BYTES, &tm_k, &sh.k_full[ks],
                         (kv_lo + j) * kTileRows, bh);
      }
      if (!ok) {
        // Drain every copy that may still be in flight (Q and the last NK K tiles).
        if (n_total > 0) mbar_wait_drain(&sh.q_full, 0, a.timeout_ns);
        for (int jj = max(0, j - C::NK); jj < j; ++jj)
          mbar_wait_drain(&sh.k_full[jj % C::NK], (jj / C::NK) & 1, a.timeout_ns);
      }
      if (a.tile_count != nullptr) {
        const int cta = (blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
        a.tile_count[cta] = j;
      }
    } else if (warp == 3 && lane == 0) {
      // ---------------- TMA producer: the V ring ----------------
      tma_prefetch_desc(&tm_v);
      int j = 0;
      bool ok = true;
      for (; j < n_total && ok; ++j) {
        const int vs = j % C::NV, vp = (j / C::NV) & 1;
        ok = mbar_wait(&sh.v_empty[vs], vp ^ 1, wc);
        if (!ok) break;
        if (a.fault == 1 && j == 0) continue;  // failure-path test: V_0 never arrives
        mbar_arrive_expect_tx(&sh.v_full[vs], C::TILE_BYTES);
        tma_load_tile<D>(smem + C::OFF_V + vs * C::TILE_BYTES, &tm_v, &sh.v_full[vs],
                         (kv_lo + j) * kTileRows, bh);
      }
      if (!ok) {
        for (int jj = max(0, j - C::NV); jj < j; ++jj)
          if (!(a.fault == 1 && jj == 0))
            mbar_wait_drain(&sh.v_full[jj % C::NV], (jj / C::NV) & 1, a.timeout_ns);
      }
    } else if (warp == 1) {
      // ---------------- tcgen05.mma issuer (the whole warp; one lane issues) ----------------
      const uint32_t q_s[2] = {smem_u32(smem + C::OFF_Q), smem_u32(smem + C::OFF_Q + C::TILE_BYTES)};
      // An empty part (n_total == 0) has nothing to wait for or issue.
      bool ok = n_total == 0 || (mbar_wait_warp(&sh.q_full, 0, wc) && mbar_wait_warp(&sh.k_full[0], 0, wc));
      if (ok && n_total > 0) {
        tc_fence_after();
        const uint32_t k0 = smem_u32(smem + C::OFF_K);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if ((t == 0 ? n_a : n_b) > 0) {
            issue_qk<D, BF16>(tmem + C::TM_S(t), q_s[t], k0);
            umma_commit_warp(&sh.s_full[t]);
          }
        }
        umma_commit_warp(&sh.k_empty[0]);
      }
      for (int j = 0; j < n_total && ok; ++j) {
        const bool more = (j + 1 < n_total);
        const int ks = (j + 1) % C::NK, vs = j % C::NV;
        ok = more ? mbar_wait2_warp(&sh.k_full[ks], ((j + 1) / C::NK) & 1, &sh.v_full[vs],
                                    (j / C::NV) & 1, wc)
                  : mbar_wait_warp(&sh.v_full[vs], (j / C::NV) & 1, wc);
        if (!ok) break;
        const uint32_t v_smem = smem_u32(smem + C::OFF_V + vs * C::TILE_BYTES);
        const uint32_t k_next = smem_u32(smem + C::OFF_K + ((j + 1) % C::NK) * C::TILE_BYTES);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int n_this = t == 0 ? n_a : n_b;
          if (j < n_this) {
            ok = mbar_wait_warp(&sh.p_full[t], j & 1, wc);
            if (!ok) break;
            tc_fence_after();
            issue_pv<D, BF16>(tmem + C::TM_O(t), tmem + C::TM_S(t) + C::TM_P_OFF, v_smem, j > 0);
            umma_commit_warp(&sh.o_full[t]);
            if (j + 1 < n_this) {
              issue_qk<D, BF16>(tmem + C::TM_S(t), q_s[t], k_next);
              umma_commit_warp(&sh.s_full[t]);
            }
          }
        }
        if (!ok) break;
        umma_commit_warp(&sh.v_empty[vs]);
        if (more) umma_commit_warp(&sh.k_empty[(j + 1) % C::NK]);
      }
      // Every MMA this warp issued must complete before TMEM is released.
      umma_commit_warp(&sh.mma_done);
      mbar_wait_drain(&sh.mma_done, 0, a.timeout_ns);
    }
  } else {
    setmaxnreg_inc<208>();
    // ---------------- softmax warpgroups ----------------
    const int t = (warp - 4) >> 2;  // 0: tile A, 1: tile B
    const int quad = warp & 3;      // TMEM lane quadrant this warp may access
    const int r = quad * 32 + lane; // row inside the tile == TMEM lane
    const int row_base = row0 + t * kTileRows;
    const int my_row = row_base + r;
    const int nt = t == 0 ? n_a : n_b;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t t_s = tmem + lane_off + C::TM_S(t);
    const uint32_t t_p = t_s + C::TM_P_OFF;
    const uint32_t t_o = tmem + lane_off + C::TM_O(t);
    const float sl2 = a.scale_log2;
    float m_ref = -INFINITY;  // reference max (raw score units) used by exp
    float l = 0.f;
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      ok = fwd_softmax_step<D, BF16, CAUSAL>(&sh.s_full[t], &sh.o_full[t], &sh.p_full[t], t_s, t_p, t_o,
                                             (kv_lo + j) * kTileRows, row_base, my_row, Nk, sl2, j == 0,
                                             j & 1, (j - 1) & 1, m_ref, l, lane, wc);
      if (!ok) break;
    }
    // ---------------- epilogue: O / l -> 16-bit, L = m + ln l ----------------
    if (ok && nt > 0) ok = mbar_wait_warp(&sh.o_full[t], (nt - 1) & 1, wc);
    if (a.o_part != nullptr && parts > 1) {
      // K/V split: this part's O / l in fp32 and its logsumexp, for the merge
      // pass; a part with no key of this tile's rows (causal: the part lies
      // past them) contributes O = 0 with logsumexp -inf. A block with a single
      // part takes the plain epilogue below and writes O and L itself. The TMEM
      // loads are warp-collective: the whole warp runs them, and only the
      // stores are limited to rows inside the sequence. Each warp stages its
      // rows through a private 4 KiB slice of Q_t's buffer, free once Q_t's
      // last product has completed.
      const bool row_in = my_row < N;
      const size_t part_base =
          (static_cast<size_t>(split) * (static_cast<size_t>(a.B) * a.H) + bh) * static_cast<size_t>(N);
      const int wrow0 = row_base + quad * 32;  // first row of this warp
      const int sub = lane >> 3, seg = lane & 7;  // store phase: 4 rows x 8 chunks of 16 bytes
      if (ok && nt > 0) {
        __syncwarp();
        tc_fence_after();
        tmem_rows_to_f32<D>(t_o, 1.f / l, a.o_part + (part_base + wrow0) * D, N - wrow0, lane,
                            reinterpret_cast<float4*>(smem + C::OFF_Q + t * C::TILE_BYTES + quad * 4096));
        if (row_in) a.lse_part[part_base + my_row] = (m_ref * sl2 + lg2_approx(l)) * kLn2;
      } else if (ok) {
        const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
        for (int c = 0; c < D; c += 32) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int rr = 4 * i + sub;
            if (wrow0 + rr < N)
              reinterpret_cast<float4*>(a.o_part + (part_base + wrow0 + rr) * D + c)[seg] = zero;
          }
        }
        if (row_in) a.lse_part[part_base + my_row] = -INFINITY;
      }
      // Arrival on the row tile's part counter; the group whose arrival
      // completes the count merges the parts. Every warp of the group gets
      // here on every path, aborted or not.
      const size_t ci = (static_cast<size_t>(bh) * a.num_m_blocks + mb) * 2 + t;
      if (arrive_last(a.part_done + ci, parts, 1 + t, &sh.merge[t])) {
        // The merge stages its weights in Q_t's buffer. A group with no key in
        // this part skipped every wait, so Q's copy may still be landing there.
        bool q_in = true;
        if (nt == 0 && n_total > 0) q_in = mbar_wait_warp(&sh.q_full, 0, wc);
        if (q_in && *abort_flag == 0)
          fwd_merge_rows<D, BF16>(a, bh, wrow0, parts, lane,
                                  reinterpret_cast<float*>(smem + C::OFF_Q + t * C::TILE_BYTES + quad * 4096));
      }
    } else {
      // Q_t's shared buffer is free (its last S product has completed): stage O
      // there in the same 128-byte-swizzled layout and store it with TMA, which
      // also clips rows past the sequence end.
      uint8_t* stage = smem + C::OFF_Q + t * C::TILE_BYTES;
      if (ok && nt > 0) {
        __syncwarp();
        tc_fence_after();
        const float inv_l = 1.f / l;
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(t_o + c, o);
          tmem_wait_ld();
          reg_fence(o);
          const int slab = c / 64;
          const int chunk0 = (c % 64) / 8;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint4 val;
            val.x = pack_x2<BF16>(__uint_as_float(o[8 * k + 0]) * inv_l, __uint_as_float(o[8 * k + 1]) * inv_l);
            val.y = pack_x2<BF16>(__uint_as_float(o[8 * k + 2]) * inv_l, __uint_as_float(o[8 * k + 3]) * inv_l);
            val.z = pack_x2<BF16>(__uint_as_float(o[8 * k + 4]) * inv_l, __uint_as_float(o[8 * k + 5]) * inv_l);
            val.w = pack_x2<BF16>(__uint_as_float(o[8 * k + 6]) * inv_l, __uint_as_float(o[8 * k + 7]) * inv_l);
            const int phys = (chunk0 + k) ^ (r & 7);
            *reinterpret_cast<uint4*>(stage + slab * C::SLAB_BYTES + r * 128 + phys * 16) = val;
          }
        }
        fence_proxy_async_smem();
        if (my_row < N) a.lse[static_cast<size_t>(bh) * N + my_row] = (m_ref * sl2 + lg2_approx(l)) * kLn2;
      }
      // Every warp of the group reaches this barrier on every path, aborted or not.
      named_bar_sync(1 + t, 128);
      if ((threadIdx.x & 127) == 0 && nt > 0 && *abort_flag == 0) {
#pragma unroll
        for (int s = 0; s < D / 64; ++s)
          tma_store_3d(&tm_o, stage + s * C::SLAB_BYTES, s * 64, row_base, bh);
        bulk_commit_group();
        bulk_wait_group_read0();
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace fa2

#include "fa2_fwd_persist.cuh"

namespace fa2 {

// ---------------------------------------------------------------------------
// Host-side launcher (called by the C ABI after validation). Without a K/V
// split the persistent kernel runs the row blocks (a.sched: at most one CTA
// per SM; `to` has 32-row boxes, one softmax warp's rows); with one, the
// per-block kernel runs one CTA per (row block, part) (`to`: 128-row boxes).
// ---------------------------------------------------------------------------
template <int D, bool BF16, bool CAUSAL>
static cudaError_t launch_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                const CUtensorMap& to, const FwdArgs& a, cudaStream_t stream) {
  using C = FwdCfg<D>;
  if (a.num_splits <= 1) {
    auto pk = fa2_fwd_persist_kernel<D, BF16, CAUSAL>;
    constexpr int smem = FwdPCfg<D>::SMEM_ALLOC;
    cudaError_t e = cudaFuncSetAttribute(pk, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (a.sched.G < 1) return cudaErrorInvalidConfiguration;
    pk<<<a.sched.G, C::THREADS, smem, stream>>>(tq, tk, tv, to, a);
    return cudaGetLastError();
  }
  auto kern = fa2_fwd_kernel<D, BF16, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  const long long ctas = split_ctas(a.num_m_blocks, a.num_splits, a.kv_tiles_max, a.B * a.H, [&](int k) {
    return fwd_block_tiles(fwd_m_block_of(k, a.num_m_blocks, CAUSAL), a.N, a.Nk, CAUSAL);
  });
  if (ctas < 1 || ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  kern<<<static_cast<unsigned>(ctas), C::THREADS, C::SMEM_ALLOC, stream>>>(tq, tk, tv, to, a);
  return cudaGetLastError();
}

cudaError_t launch_fwd(int d, bool bf16, bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const CUtensorMap& to, const FwdArgs& a,
                       cudaStream_t stream) {
#define FA2_FWD_CASE(DD, BB, CC) \
  if (d == DD && bf16 == BB && causal == CC) return launch_fwd_t<DD, BB, CC>(tq, tk, tv, to, a, stream);
  FA2_FWD_CASE(64, true, false)
  FA2_FWD_CASE(64, true, true)
  FA2_FWD_CASE(64, false, false)
  FA2_FWD_CASE(64, false, true)
  FA2_FWD_CASE(128, true, false)
  FA2_FWD_CASE(128, true, true)
  FA2_FWD_CASE(128, false, false)
  FA2_FWD_CASE(128, false, true)
#undef FA2_FWD_CASE
  return cudaErrorInvalidValue;
}

}  // namespace fa2
