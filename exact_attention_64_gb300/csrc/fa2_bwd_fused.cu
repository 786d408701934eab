// FlashAttention-2 backward with the column workers of the pages: K/V outer,
// Q inner, and dQ accumulated across the column workers by fp32 reduce-adds
// ("FlashAttention学习笔记(2)", Foward和backward中的thread block划分: dK and dV
// accumulate along the query direction inside one worker, dQ along the key
// direction across workers; "大猿搬砖简记", V2 backward). Three launches on one
// stream:
//
//  1. fa2_bwd_pre_kernel       D = rowsum(dO o O), L*log2(e), and dQaccum = 0.
//  2. fa2_bwd_fused_kernel     one CTA per 128-key column block: K_j, V_j stay in
//                              shared memory and dK_j, dV_j in TMEM while the
//                              128-row query tiles stream past; per tile
//                                S^T = K Q_i^T, dP^T = V dO_i^T          (SS, M=128 keys)
//                                P^T = exp2(S^T*scale*log2e - L*log2e),  dS^T = P^T o (dP^T - D)
//                                dK += dS^T Q_i   (SS, A = dS^T in shared memory, K-major)
//                                dQ_i = dS K      (SS, A = the same dS^T buffer read MN-major)
//                                dV += P^T dO_i   (TS, A = P^T in TMEM)
//                              and dQ_i (fp32, in TMEM) is added into dQaccum with
//                              TMA reduce-adds through shared memory, 32 rows x 32
//                              columns per warp and box.
//  3. fa2_bwd_dq_convert_kernel  dQ = scale * dQaccum -> 16 bit.
//
// Five GEMM units per (key block, query tile) pair, none recomputed. The sum
// order of dQ's reduce-adds depends on which column worker arrives first, so
// dQ is not bit-reproducible run to run (the split backward in fa2_bwd.cu is).
//
// TMEM (512 columns): dV [0,d), dK [d,2d) and two 128-column regions X, Y that
// swap roles from one query tile to the next: tile i computes S^T into R_S(i)
// and dP^T into R_P(i), writes P^T back into R_P(i) and lands dQ_i in R_S(i)
// once S^T(i) has been read; tile i+1 uses R_S(i+1) = R_P(i) (free once dV(i),
// the last reader of P^T(i), was issued) and R_P(i+1) = R_S(i) (free once dQ_i
// has been read out). The tensor core runs, per tile,
//   dV(i), S^T(i+1), dQ_i, dK(i), dP^T(i+1)
// so the exponentials of P^T(i+1) overlap dQ_i and dK(i), and the read-out of
// dQ_i overlaps dK(i).
#include "fa2_bwd_parts.cuh"
#include "../../include/fa2.h"

namespace fa2 {

template <int D>
struct FusedCfg {
  static constexpr int TILE = BwdTile<D>::TILE_BYTES;
  static constexpr int SLAB = BwdTile<D>::SLAB_BYTES;   // 128 rows x 128 bytes
  static constexpr int OFF_K = 0, OFF_V = TILE;          // resident K_j, V_j
  static constexpr int OFF_Q = 2 * TILE;                 // Q_i ring, 2 stages
  static constexpr int OFF_DO = OFF_Q + 2 * TILE;        // dO_i ring, 2 stages
  // dS^T [key][query] 16-bit as two slabs of 64 queries (one per compute
  // warpgroup); between tiles, each slab stages that warpgroup's dQ_i boxes
  // (4 KiB per warp: 32 rows x 32 fp32 columns).
  static constexpr int OFF_DS = OFF_DO + 2 * TILE;
  static constexpr int SMEM_BYTES = OFF_DS + 2 * SLAB;
  // >= 116 KiB so that at most one CTA (one 512-column TMEM allocation) lives on an SM.
  static constexpr int SMEM_ALLOC = (SMEM_BYTES + 1024 > 118784) ? SMEM_BYTES + 1024 : 118784;
  static constexpr int THREADS = 384;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t T_DV = 0, T_DK = D, T_X = 2 * D, T_Y = 2 * D + 128;
};

struct FusedShared {
  uint64_t kv_full;
  uint64_t q_full[2], do_full[2];    // ring stages landed
  uint64_t q_empty[2], do_empty[2];  // ring stages read by their last product (dK / dV)
  uint64_t st_full;                  // S^T(i) complete
  uint64_t dpt_full;                 // dP^T(i) complete
  uint64_t ds_ready;                 // P^T(i) in TMEM and dS^T(i) in shared memory, from all 8 compute warps
  uint64_t dq_full;                  // dQ_i complete: readable in TMEM
  uint64_t dk_done;                  // dK(i) complete: the dS^T buffer free (dQ_i, its other reader, came first)
  uint64_t dq_drained;               // dQ_i read out of TMEM by all 8 compute warps
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort_flag;
};

// D[tmem] (+)= A X with A = 128 x 128 16-bit from the dS^T buffer and X a
// 128-row tile [row][d] (MN-major for this product). A_MN = false reads the
// buffer as dS^T (rows = keys = M, K-major); A_MN = true reads it as dS (M =
// queries, the buffer's columns: MN-major, the same descriptor form as an
// MN-major B tile).
template <int D, bool BF16, bool A_MN>
__device__ __forceinline__ void mma_ds_x_tile(uint32_t d_tmem, uint32_t ds_smem, uint32_t x_smem,
                                              bool accumulate) {
  constexpr uint32_t idesc = make_idesc_f16(128, D, BF16, A_MN, true);
  constexpr uint32_t SLAB = FusedCfg<D>::SLAB;
#pragma unroll
  for (int kk = 0; kk < kTileRows / 16; ++kk) {
    const uint64_t ad = A_MN ? make_sdesc_sw128(ds_smem + kk * 2048, SLAB, 1024)
                             : make_sdesc_sw128(ds_smem + (kk / 4) * SLAB + (kk % 4) * 32, 16, 1024);
    const uint64_t bd = make_sdesc_sw128(x_smem + kk * 2048, SLAB, 1024);
    umma_ss_warp(d_tmem, ad, bd, idesc, (accumulate || kk > 0) ? 1u : 0u);
  }
}

template <int D, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(384, 1)
    fa2_bwd_fused_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                         const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                         const __grid_constant__ CUtensorMap tm_dqa, const BwdArgs a) {
  using C = FusedCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  __shared__ FusedShared sh;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = a.N;    // queries
  const int Nk = a.Nk;  // keys and values
  // The pages' (key block, batch, head) order, key block fastest; under the
  // causal mask key block 0 has the most query tiles, so blocks start longest first.
  const int nkb = bwd_num_n_blocks(Nk);
  const int nb = blockIdx.x % nkb;
  const int rest = blockIdx.x / nkb;
  const int bh = (rest % a.B) * a.H + rest / a.B;
  const int n0 = nb * kTileRows;
  const int i_begin = bwd_q_tile_begin(nb, CAUSAL);
  // 0 when no query sees these keys (causal, more keys than queries): the
  // block then loads and issues nothing and writes dK = dV = 0.
  const int n_steps = max(0, ceil_div(N, kTileRows) - i_begin);

  if (threadIdx.x == 0) {
    mbar_init(&sh.kv_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sh.q_full[s], 1);
      mbar_init(&sh.do_full[s], 1);
      mbar_init(&sh.q_empty[s], 1);
      mbar_init(&sh.do_empty[s], 1);
    }
    mbar_init(&sh.st_full, 1);
    mbar_init(&sh.dpt_full, 1);
    mbar_init(&sh.ds_ready, 8);    // the eight compute warps
    mbar_init(&sh.dq_full, 1);
    mbar_init(&sh.dk_done, 1);
    mbar_init(&sh.dq_drained, 8);
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
      tma_prefetch_desc(&tm_dqa);
      if (n_steps > 0) {
        mbar_arrive_expect_tx(&sh.kv_full, 2 * C::TILE);
        load_tile<D>(smem + C::OFF_K, &tm_k, &sh.kv_full, n0, bh);
        load_tile<D>(smem + C::OFF_V, &tm_v, &sh.kv_full, n0, bh);
      }
      int iq = 0, ido = 0;  // Q_i / dO_i loads issued (or, for the faulted one, skipped)
      bool ok = true;
      for (int i = 0; i < n_steps; ++i) {
        const int st = i & 1, ph = (i >> 1) & 1;
        const int q0 = (i_begin + i) * kTileRows;
        ok = mbar_wait(&sh.q_empty[st], ph ^ 1, wc);
        if (!ok) break;
        mbar_arrive_expect_tx(&sh.q_full[st], C::TILE);
        load_tile<D>(smem + C::OFF_Q + st * C::TILE, &tm_q, &sh.q_full[st], q0, bh);
        iq = i + 1;
        ok = mbar_wait(&sh.do_empty[st], ph ^ 1, wc);
        if (!ok) break;
        ido = i + 1;
        if (a.fault == 1 && i == 0) continue;  // failure-path test: dO_0 never arrives
        mbar_arrive_expect_tx(&sh.do_full[st], C::TILE);
        load_tile<D>(smem + C::OFF_DO + st * C::TILE, &tm_do, &sh.do_full[st], q0, bh);
      }
      if (!ok) {
        // Let every copy that may still be in flight land before the CTA exits.
        if (n_steps > 0) mbar_wait_drain(&sh.kv_full, 0, a.timeout_ns);
        for (int ii = max(0, iq - 2); ii < iq; ++ii)
          mbar_wait_drain(&sh.q_full[ii & 1], (ii >> 1) & 1, a.timeout_ns);
        for (int ii = max(0, ido - 2); ii < ido; ++ii)
          if (!(a.fault == 1 && ii == 0))
            mbar_wait_drain(&sh.do_full[ii & 1], (ii >> 1) & 1, a.timeout_ns);
      }
    } else if (warp == 1) {
      // ---------------- tcgen05.mma issuer (the whole warp; one lane issues) ----------------
      // One issuer for all five products, so that every reuse of a TMEM
      // region follows issue order. Per tile, once P^T(i) and dS^T(i) are
      // ready: dV(i); S^T(i+1) into R_P(i) (behind dV(i), the last reader of
      // P^T(i)); dQ_i into R_S(i); dK(i); and, once dQ_i has been read out,
      // dP^T(i+1) into R_S(i).
      const uint32_t k_s = smem_u32(smem + C::OFF_K), v_s = smem_u32(smem + C::OFF_V);
      const uint32_t ds_s = smem_u32(smem + C::OFF_DS);
      auto q_at = [&](int i) { return smem_u32(smem + C::OFF_Q + (i & 1) * C::TILE); };
      auto do_at = [&](int i) { return smem_u32(smem + C::OFF_DO + (i & 1) * C::TILE); };
      auto r_s = [&](int i) { return tmem + ((i & 1) ? C::T_Y : C::T_X); };
      auto r_p = [&](int i) { return tmem + ((i & 1) ? C::T_X : C::T_Y); };
      bool ok = n_steps == 0 ||
                (mbar_wait_warp(&sh.kv_full, 0, wc) && mbar_wait_warp(&sh.q_full[0], 0, wc));
      if (ok && n_steps > 0) {
        tc_fence_after();
        mma_rows_x_rows<D, BF16>(r_s(0), k_s, q_at(0));
        umma_commit_warp(&sh.st_full);
        ok = mbar_wait_warp(&sh.do_full[0], 0, wc);
        if (ok) {
          tc_fence_after();
          mma_rows_x_rows<D, BF16>(r_p(0), v_s, do_at(0));
          umma_commit_warp(&sh.dpt_full);
        }
      }
      for (int i = 0; i < n_steps && ok; ++i) {
        const int st = i & 1;
        const bool more = i + 1 < n_steps;
        ok = mbar_wait_warp(&sh.ds_ready, i & 1, wc);
        if (!ok) break;
        tc_fence_after();
        const uint32_t rp = r_p(i);
        mma_tmem_x_tile<D, BF16>(
            tmem + C::T_DV, [rp](int kk) { return rp + 64u * static_cast<uint32_t>(kk >> 2) + 8u * (kk & 3); },
            do_at(i), i > 0);  // dV += P^T dO_i
        umma_commit_warp(&sh.do_empty[st]);  // dO_i's last reader was dV(i)
        if (more) {
          ok = mbar_wait_warp(&sh.q_full[(i + 1) & 1], ((i + 1) >> 1) & 1, wc);
          if (!ok) break;
          tc_fence_after();
          mma_rows_x_rows<D, BF16>(r_s(i + 1), k_s, q_at(i + 1));  // into R_P(i), behind dV(i)
          umma_commit_warp(&sh.st_full);
        }
        mma_ds_x_tile<D, BF16, true>(r_s(i), ds_s, k_s, false);              // dQ_i = dS K
        umma_commit_warp(&sh.dq_full);
        mma_ds_x_tile<D, BF16, false>(tmem + C::T_DK, ds_s, q_at(i), i > 0);  // dK += dS^T Q_i
        umma_commit_warp(&sh.dk_done);
        umma_commit_warp(&sh.q_empty[st]);  // Q_i's last reader was dK(i)
        if (more) {
          const int in = i + 1;
          ok = mbar_wait2_warp(&sh.do_full[in & 1], (in >> 1) & 1, &sh.dq_drained, i & 1, wc);
          if (!ok) break;
          tc_fence_after();
          mma_rows_x_rows<D, BF16>(r_p(in), v_s, do_at(in));  // into R_S(i), dQ_i read out
          umma_commit_warp(&sh.dpt_full);
        }
      }
      // Every MMA this warp issued must complete before TMEM is released.
      umma_commit_warp(&sh.mma_done);
      mbar_wait_drain(&sh.mma_done, 0, a.timeout_ns);
    }
  } else {
    setmaxnreg_inc<208>();
    // ---------------- compute warpgroups: P^T, dS^T, the dQ drain ----------------
    const int wg = (warp - 4) >> 2;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // TMEM lane: key row of the block for S^T and dP^T, query row for dQ
    const int kg = n0 + r;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const float sl2 = a.scale_log2;
    uint8_t* slab = smem + C::OFF_DS + wg * C::SLAB;  // this warpgroup's 64 query columns of dS^T
    // P^T of tile t as 16-bit pairs: -L*log2e of this warpgroup's 64 queries
    // (every lane reads the same values: broadcast loads), S^T(t) from TMEM,
    // exponentials. dS^T(t) is later formed from these rounded values.
    auto p_tile = [&](int t, uint32_t (&pk)[32]) -> bool {
      const int qc0 = (i_begin + t) * kTileRows + 64 * wg;  // first query column of this warpgroup
      const uint32_t rs = tmem + lane_off + ((t & 1) ? C::T_Y : C::T_X);
      const float* lrow = a.l2_pad + static_cast<size_t>(bh) * a.n_pad + qc0;
      float lreg[64];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const float4 l4 = __ldg(reinterpret_cast<const float4*>(lrow) + u);
        lreg[4 * u] = -l4.x; lreg[4 * u + 1] = -l4.y; lreg[4 * u + 2] = -l4.z; lreg[4 * u + 3] = -l4.w;
      }
      if (!mbar_wait_warp(&sh.st_full, t & 1, wc)) return false;
      __syncwarp();  // the warp-collective TMEM loads below need a converged warp
      tc_fence_after();
      uint32_t sv[64];
      tmem_ld_32x32b_x32(rs + 64 * wg, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
      tmem_ld_32x32b_x32(rs + 64 * wg + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
      tmem_wait_ld();
      reg_fence(sv);
      const bool need_mask = (CAUSAL && qc0 < n0 + kTileRows - 1) || (qc0 + 64 > N) ||
                             (n0 + kTileRows > Nk);
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
      return true;
    };
    uint32_t pk[32];
    bool ok = n_steps == 0 || p_tile(0, pk);
    for (int i = 0; i < n_steps && ok; ++i) {
      const int q0 = (i_begin + i) * kTileRows;
      const int qc0 = q0 + 64 * wg;
      const uint32_t rs = tmem + lane_off + ((i & 1) ? C::T_Y : C::T_X);
      const uint32_t rp = tmem + lane_off + ((i & 1) ? C::T_X : C::T_Y);
      const float* drow = a.dsum_pad + static_cast<size_t>(bh) * a.n_pad + qc0;
      float dreg[64];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const float4 d4 = __ldg(reinterpret_cast<const float4*>(drow) + u);
        dreg[4 * u] = d4.x; dreg[4 * u + 1] = d4.y; dreg[4 * u + 2] = d4.z; dreg[4 * u + 3] = d4.w;
      }
      ok = mbar_wait_warp(&sh.dpt_full, i & 1, wc);
      if (!ok) break;
      __syncwarp();
      tc_fence_after();
      uint32_t dsk[32];  // dS^T of this key row, 64 queries as 16-bit pairs
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t dp[32];
        tmem_ld_32x32b_x32(rp + 64 * wg + 32 * h, dp);
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
      // dP^T(i) has been read: P^T(i) takes this warpgroup's first 32 columns
      // of R_P(i) (the dV product's A operand), and dS^T(i) goes to this
      // warpgroup's slab, row r = 128 bytes, 16-byte chunks XOR-swizzled by row.
      tmem_st_32x32b_x32(rp + 64 * wg, pk);
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(slab + r * 128 + ((c ^ (r & 7)) * 16)) =
            make_uint4(dsk[4 * c], dsk[4 * c + 1], dsk[4 * c + 2], dsk[4 * c + 3]);
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.ds_ready);

      // The next tile's exponentials while the tensor core runs dV(i),
      // S^T(i+1), dQ_i and dK(i).
      if (i + 1 < n_steps) {
        ok = p_tile(i + 1, pk);
        if (!ok) break;
      }

      // dQ_i (lane = query row q0 + r) into dQaccum: this warpgroup's d/2
      // columns. First all of them into registers, which frees R_S(i) for
      // dP^T(i+1); then, once dK(i) has read dS^T(i), 32 columns at a time
      // through the slab: each warp stages its own 32 rows (its 4 KiB) as one
      // 32-row x 32-column fp32 box of the reduce-add's tensor map and issues
      // that box itself, so no warp waits for another.
      ok = mbar_wait_warp(&sh.dq_full, i & 1, wc);
      if (!ok) break;
      __syncwarp();
      tc_fence_after();
      uint32_t xq[D / 2];
#pragma unroll
      for (int c = 0; c < D / 2; c += 32)
        tmem_ld_32x32b_x32(rs + wg * (D / 2) + c, *reinterpret_cast<uint32_t(*)[32]>(&xq[c]));
      tmem_wait_ld();
      reg_fence(xq);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.dq_drained);
      ok = mbar_wait_warp(&sh.dk_done, i & 1, wc);
      if (!ok) break;
      uint8_t* box = slab + quad * 4096;
#pragma unroll
      for (int c = 0; c < D / 2; c += 32) {
        float4* dst = reinterpret_cast<float4*>(box + lane * 128);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          dst[k ^ (lane & 7)] = make_float4(__uint_as_float(xq[c + 4 * k]), __uint_as_float(xq[c + 4 * k + 1]),
                                            __uint_as_float(xq[c + 4 * k + 2]), __uint_as_float(xq[c + 4 * k + 3]));
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_reduce_add_3d(&tm_dqa, box, wg * (D / 2) + c, q0 + quad * 32, bh);
          bulk_commit_group();
          bulk_wait_group_read0();
        }
        __syncwarp();
      }
    }
    // ---------------- epilogue: dV, scale*dK -> 16-bit, TMA store ----------------
    if (ok) ok = mbar_wait_warp(&sh.mma_done, 0, wc);
    // All MMAs have completed, so the K and V buffers are free for staging.
    uint8_t* stage = smem + (wg == 0 ? C::OFF_V : C::OFF_K);
    if (ok && n_steps > 0) {
      __syncwarp();
      tc_fence_after();
      stage_rows<D, BF16>(stage, tmem + lane_off + (wg == 0 ? C::T_DV : C::T_DK), r,
                          wg == 0 ? 1.f : a.scale);
      fence_proxy_async_smem();
    } else if (ok) {
      // No query sees these keys: their gradients are zero.
#pragma unroll
      for (int sl = 0; sl < D / 64; ++sl)
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(stage + sl * C::SLAB + r * 128 + c * 16) = make_uint4(0u, 0u, 0u, 0u);
      fence_proxy_async_smem();
    }
    named_bar_sync(1 + wg, 128);
    if ((threadIdx.x & 127) == 0 && *abort_flag == 0) {
      const CUtensorMap* map = (wg == 0) ? &tm_dv : &tm_dk;
#pragma unroll
      for (int s = 0; s < D / 64; ++s) tma_store_3d(map, stage + s * C::SLAB, s * 64, n0, bh);
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

// dQ = scale * dQaccum, rounded once to the 16-bit type: 8 elements per
// thread, 32-byte loads of dQaccum ([B*H][n_pad][d] fp32) and 16-byte stores of
// dQ ([B*H][N][d]). HBM-bound.
template <int D, bool BF16>
__global__ void __launch_bounds__(256)
    fa2_bwd_dq_convert_kernel(const float* __restrict__ dq_acc, uint16_t* __restrict__ dq, int BH,
                              int N, int n_pad, float scale) {
  const long long per_head = static_cast<long long>(N) * (D / 8);
  const long long total = static_cast<long long>(BH) * per_head;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; t < total;
       t += stride) {
    const long long h = t / per_head;
    const long long e = (t - h * per_head) * 8;  // element offset inside the head's [N][d]
    const float4* src = reinterpret_cast<const float4*>(dq_acc + h * n_pad * D + e);
    const float4 x0 = __ldcs(src), x1 = __ldcs(src + 1);
    uint4 o;
    o.x = pack_x2<BF16>(x0.x * scale, x0.y * scale);
    o.y = pack_x2<BF16>(x0.z * scale, x0.w * scale);
    o.z = pack_x2<BF16>(x1.x * scale, x1.y * scale);
    o.w = pack_x2<BF16>(x1.z * scale, x1.w * scale);
    *reinterpret_cast<uint4*>(dq + h * N * D + e) = o;
  }
}

// ---------------------------------------------------------------------------
// Host-side launcher
// ---------------------------------------------------------------------------
cudaError_t launch_bwd_pre(int d, bool bf16, const void* o, const void* dO, const float* lse,
                           float* dsum, float* l2, float* dq_acc, int* item_counter, int BH, int N,
                           int n_pad, cudaStream_t stream);

template <int D, bool BF16, bool CAUSAL>
static cudaError_t launch_bwd_fused_t(const void* o, const void* dO, const float* lse,
                                      const CUtensorMap* maps, const BwdArgs& a, float* dsum, float* l2,
                                      float* dq_acc, void* dq, int num_sms, cudaStream_t stream,
                                      cudaEvent_t* ev) {
  using C = FusedCfg<D>;
  const int BH = a.B * a.H;
  if (ev) cudaEventRecord(ev[0], stream);
  cudaError_t e = launch_bwd_pre(D, BF16, o, dO, lse, dsum, l2, dq_acc, nullptr, BH, a.N, a.n_pad, stream);
  if (e != cudaSuccess) return e;
  if (ev) cudaEventRecord(ev[1], stream);
  {
    auto kern = fa2_bwd_fused_kernel<D, BF16, CAUSAL>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    const long long ctas = static_cast<long long>(bwd_num_n_blocks(a.Nk)) * BH;
    if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    kern<<<static_cast<unsigned>(ctas), C::THREADS, C::SMEM_ALLOC, stream>>>(
        maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], maps[7], a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (ev) cudaEventRecord(ev[2], stream);
  {
    const long long chunks = static_cast<long long>(BH) * a.N * (D / 8);
    long long blocks = (chunks + 255) / 256;
    const long long cap = static_cast<long long>(num_sms) * 16;
    if (blocks > cap) blocks = cap;
    fa2_bwd_dq_convert_kernel<D, BF16><<<static_cast<int>(blocks), 256, 0, stream>>>(
        dq_acc, static_cast<uint16_t*>(dq), BH, a.N, a.n_pad, a.scale);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (ev) cudaEventRecord(ev[3], stream);
  return cudaSuccess;
}

cudaError_t launch_bwd_fused(int d, bool bf16, bool causal, const void* o, const void* dO,
                             const float* lse, const CUtensorMap* maps, const BwdArgs& a, float* dsum,
                             float* l2, float* dq_acc, void* dq, int num_sms, cudaStream_t stream,
                             cudaEvent_t* ev) {
#define FA2_FUSED_CASE(DD, BB, CC)         \
  if (d == DD && bf16 == BB && causal == CC) \
    return launch_bwd_fused_t<DD, BB, CC>(o, dO, lse, maps, a, dsum, l2, dq_acc, dq, num_sms, stream, ev);
  FA2_FUSED_CASE(64, true, false)
  FA2_FUSED_CASE(64, true, true)
  FA2_FUSED_CASE(64, false, false)
  FA2_FUSED_CASE(64, false, true)
  FA2_FUSED_CASE(128, true, false)
  FA2_FUSED_CASE(128, true, true)
  FA2_FUSED_CASE(128, false, false)
  FA2_FUSED_CASE(128, false, true)
#undef FA2_FUSED_CASE
  return cudaErrorInvalidValue;
}

}  // namespace fa2
