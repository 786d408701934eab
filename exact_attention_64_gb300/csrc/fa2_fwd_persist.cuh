// Persistent form of the unsplit forward (included by fa2_fwd.cu after the
// tile layout, the MMA helpers and the softmax step it shares with the
// per-block kernel).
//
// The work items are the per-block kernel's thread blocks ("FlashAttention学习笔记(2)",
// V2中的thread blocks排布): 256 query rows (tiles A and B, 128 rows each) of one
// head. One CTA per SM runs the fixed list FwdSched gives it (see
// fwd_sched_make: causal pairs of row blocks with a constant K/V total, the
// last partial round split into halves), so there is no counter and no
// workspace, and every role of the CTA walks the same list by itself.
//
// Inside a CTA the K/V rings and every pipeline barrier keep counting across
// items. Q_A and Q_B have barriers of their own: Q_t of the next item loads as
// soon as tile t's last S product of the current item has completed, and that
// next item's first S_t product follows tile t's last P V product as soon as
// its copies have landed, so the tensor core moves on to the next item while
// the softmax warps finish the current one. The epilogue stages O in buffers
// of its own (the Q buffers are already being refilled) and stores it with
// TMA.
#pragma once

namespace fa2 {

// Shared memory: the per-block kernel's Q, K, V layout, then one 4 KiB
// staging buffer per softmax warp for its 32 output rows x 64 columns (128-byte
// rows, 128-byte swizzled), which a 32-row TMA store writes out.
template <int D>
struct FwdPCfg {
  static constexpr int OFF_O = FwdCfg<D>::SMEM_BYTES;
  static constexpr int STAGE_BYTES = 32 * 128;
  static constexpr int SMEM_ALLOC = OFF_O + 8 * STAGE_BYTES + 1024;  // + slack for 1024-byte alignment
};

template <int D>
struct FwdPShared {
  uint64_t q_full[2], q_free[2];  // Q_t landed / read by the item's last S_t product
  uint64_t k_full[FwdCfg<D>::NK], k_empty[FwdCfg<D>::NK];
  uint64_t v_full[FwdCfg<D>::NV], v_empty[FwdCfg<D>::NV];
  uint64_t s_full[2], p_full[2], o_full[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort_flag;
};

// One work item: row block mb (rows [256 mb, 256 mb + 256)) of head bh, the
// K/V tile counts of tiles A and B (n_b = 0 when the block has no second
// tile), and its linear index in the per-block grid (hb * nm + rank).
struct FwdItem {
  int mb, bh, n_a, n_b, lin;
};

template <bool CAUSAL>
__device__ __forceinline__ FwdItem fwd_item(int hb, int rank, const FwdArgs& a) {
  FwdItem it;
  const int nm = a.num_m_blocks;
  it.mb = fwd_m_block_of(rank, nm, CAUSAL);
  it.bh = (hb % a.B) * a.H + hb / a.B;  // the per-block grid's (batch, head) = (y, z)
  it.lin = hb * nm + rank;
  const int row0 = it.mb * kFwdRowsPerCta;
  const int rows_a = min(kTileRows, a.N - row0);
  const int rows_b = max(0, min(kTileRows, a.N - row0 - kTileRows));
  it.n_a = fwd_kv_tile_end(row0, row0 + rows_a, a.Nk, CAUSAL);
  it.n_b = fwd_kv_tile_end(row0 + kTileRows, row0 + kTileRows + rows_b, a.Nk, CAUSAL);
  return it;
}

// Next item of this CTA; false when its list is exhausted.
template <bool CAUSAL>
__device__ __forceinline__ bool fwd_next(const FwdArgs& a, FwdCursor& cur, FwdItem& it) {
  int hb, rank;
  if (!fwd_sched_next(a.sched, blockIdx.x, cur, &hb, &rank)) return false;
  it = fwd_item<CAUSAL>(hb, rank, a);
  return true;
}

// Epilogue of one softmax warp: O / l of its 32 rows, rounded to 16 bits, in
// 64-column chunks through the warp's staging buffer and a TMA store of a
// 32-row box at rows [wrow0, wrow0 + 32) of head bh (the store clips rows past
// the sequence end). Before a chunk overwrites the buffer, the warp's
// previous store must have finished reading it. The TMEM loads are
// warp-collective.
template <int D, bool BF16>
__device__ __forceinline__ void fwd_store_rows(uint32_t t_o, uint8_t* stage, const CUtensorMap* tm_o,
                                               int wrow0, int bh, float inv_l, int lane) {
#pragma unroll
  for (int c = 0; c < D; c += 64) {
    if (lane == 0) bulk_wait_group_read0();
    __syncwarp();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t x[32];
      tmem_ld_32x32b_x32(t_o + c + 32 * h, x);
      tmem_wait_ld();
      reg_fence(x);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint4 val;
        val.x = pack_x2<BF16>(__uint_as_float(x[8 * k + 0]) * inv_l, __uint_as_float(x[8 * k + 1]) * inv_l);
        val.y = pack_x2<BF16>(__uint_as_float(x[8 * k + 2]) * inv_l, __uint_as_float(x[8 * k + 3]) * inv_l);
        val.z = pack_x2<BF16>(__uint_as_float(x[8 * k + 4]) * inv_l, __uint_as_float(x[8 * k + 5]) * inv_l);
        val.w = pack_x2<BF16>(__uint_as_float(x[8 * k + 6]) * inv_l, __uint_as_float(x[8 * k + 7]) * inv_l);
        const int phys = (4 * h + k) ^ (lane & 7);
        *reinterpret_cast<uint4*>(stage + lane * 128 + phys * 16) = val;
      }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_3d(tm_o, stage, c, wrow0, bh);
      bulk_commit_group();
    }
  }
}

// ---------------- producers (one thread each) ----------------
// Q_t of an item waits for the previous item's q_free[t] (its last S_t product
// has completed). Per item the K producer issues Q_A, K_0, Q_B, K_1, ...: the
// first products of an item need Q_A and K_0 first, and Q_B's wait (on the
// current item's last S_B product) then never holds up K_0. On a failed wait
// the producer drains every copy it issued (last_*: the phase number last
// armed on each barrier, -1 never) and returns false.
template <int D, bool CAUSAL>
__device__ bool fwd_persist_k_producer(FwdPShared<D>& sh, uint8_t* smem, const CUtensorMap& tm_q,
                                       const CUtensorMap& tm_k, const FwdArgs& a, const WaitCtx& wc) {
  using C = FwdCfg<D>;
  int g = 0, qa = 0, qb = 0, last_qa = -1, last_qb = -1;
  int last_k[C::NK];
#pragma unroll
  for (int i = 0; i < C::NK; ++i) last_k[i] = -1;
  bool ok = true;
  FwdCursor cur{};
  FwdItem it;
  while (ok && fwd_next<CAUSAL>(a, cur, it)) {
    const int n_total = max(it.n_a, it.n_b);
    const int row0 = it.mb * kFwdRowsPerCta;
    int loaded = 0;
    if (it.n_a > 0) {
      if (qa > 0) ok = mbar_wait(&sh.q_free[0], (qa - 1) & 1, wc);
      if (ok) {
        mbar_arrive_expect_tx(&sh.q_full[0], C::TILE_BYTES);
        tma_load_tile<D>(smem + C::OFF_Q, &tm_q, &sh.q_full[0], row0, it.bh);
        last_qa = qa++;
      }
    }
    for (int j = 0; j < n_total && ok; ++j, ++g) {
      const int ks = g % C::NK;
      ok = mbar_wait(&sh.k_empty[ks], ((g / C::NK) & 1) ^ 1, wc);
      if (!ok) break;
      mbar_arrive_expect_tx(&sh.k_full[ks], C::TILE_BYTES);
      tma_load_tile<D>(smem + C::OFF_K + ks * C::TILE_BYTES, &tm_k, &sh.k_full[ks], j * kTileRows, it.bh);
      last_k[ks] = g / C::NK;
      ++loaded;
      if (j == 0 && it.n_b > 0) {
        if (qb > 0) ok = mbar_wait(&sh.q_free[1], (qb - 1) & 1, wc);
        if (ok) {
          mbar_arrive_expect_tx(&sh.q_full[1], C::TILE_BYTES);
          tma_load_tile<D>(smem + C::OFF_Q + C::TILE_BYTES, &tm_q, &sh.q_full[1], row0 + kTileRows, it.bh);
          last_qb = qb++;
        }
      }
    }
    if (a.tile_count != nullptr) a.tile_count[it.lin] = loaded;
  }
  if (!ok) {
    if (last_qa >= 0) mbar_wait_drain(&sh.q_full[0], last_qa & 1, a.timeout_ns);
    if (last_qb >= 0) mbar_wait_drain(&sh.q_full[1], last_qb & 1, a.timeout_ns);
#pragma unroll
    for (int i = 0; i < C::NK; ++i)
      if (last_k[i] >= 0) mbar_wait_drain(&sh.k_full[i], last_k[i] & 1, a.timeout_ns);
  }
  return ok;
}

// V producer: the items' V tiles through the ring. Failure-path test: the
// first V tile of CTA 0 never arrives.
template <int D, bool CAUSAL>
__device__ bool fwd_persist_v_producer(FwdPShared<D>& sh, uint8_t* smem, const CUtensorMap& tm_v,
                                       const FwdArgs& a, const WaitCtx& wc) {
  using C = FwdCfg<D>;
  int g = 0;
  int last_v[C::NV];
#pragma unroll
  for (int i = 0; i < C::NV; ++i) last_v[i] = -1;
  bool ok = true;
  FwdCursor cur{};
  FwdItem it;
  while (ok && fwd_next<CAUSAL>(a, cur, it)) {
    const int n_total = max(it.n_a, it.n_b);
    for (int j = 0; j < n_total; ++j, ++g) {
      const int vs = g % C::NV;
      ok = mbar_wait(&sh.v_empty[vs], ((g / C::NV) & 1) ^ 1, wc);
      if (!ok) break;
      if (a.fault == 1 && g == 0 && blockIdx.x == 0) continue;
      mbar_arrive_expect_tx(&sh.v_full[vs], C::TILE_BYTES);
      tma_load_tile<D>(smem + C::OFF_V + vs * C::TILE_BYTES, &tm_v, &sh.v_full[vs], j * kTileRows, it.bh);
      last_v[vs] = g / C::NV;
    }
  }
  if (!ok) {
#pragma unroll
    for (int i = 0; i < C::NV; ++i)
      if (last_v[i] >= 0) mbar_wait_drain(&sh.v_full[i], last_v[i] & 1, a.timeout_ns);
  }
  return ok;
}

// ---------------- tcgen05.mma issuer (the whole warp; one lane issues) ----------------
// Per K/V step g of an item (j = g - g0) and tile t with j < n_t: P_t V_g
// into O_t once the softmax has written P_t, then tile t's next S product,
// S_t(j+1) with K_{g+1}, inside the item. After tile t's last step, S_t(0) of
// the next item (its Q_t and first K tile) is pending: it is issued as soon as
// both copies have landed, tested without blocking between the other tile's
// products, and waited for only once the current item has issued everything
// else, so a copy still in flight never holds up the other tile's work (under
// a causal mask tile A runs one step fewer than tile B). These copies depend
// only on products issued earlier (the next Q_t on this item's last S_t
// product, the next K tile on the ring slot of K_{g-1}), so no wait can close
// a cycle. q_free[t] is committed after the item's last S_t product, k_empty(g)
// after every S product that reads K_g, v_empty(g) after both P V products of
// step g. The counters sa, sb (products of tile A / B so far) and qa, qb
// (items in which the tile is active) continue across items, as do the
// barrier phases they select.
template <int D, bool BF16>
__device__ __forceinline__ void fwd_issue_s(uint32_t tmem, int t, uint32_t q_smem, uint32_t k_smem,
                                            FwdPShared<D>& sh, bool last_of_item) {
  using C = FwdCfg<D>;
  issue_qk<D, BF16>(tmem + C::TM_S(t), q_smem, k_smem);
  umma_commit_warp(&sh.s_full[t]);
  if (last_of_item) umma_commit_warp(&sh.q_free[t]);
}

template <int D, bool BF16, bool CAUSAL>
__device__ bool fwd_persist_issuer(FwdPShared<D>& sh, uint8_t* smem, uint32_t tmem, const FwdArgs& a,
                                   const WaitCtx& wc) {
  using C = FwdCfg<D>;
  const uint32_t q_a = smem_u32(smem + C::OFF_Q), q_b = q_a + C::TILE_BYTES;
  const uint32_t k_base = smem_u32(smem + C::OFF_K), v_base = smem_u32(smem + C::OFF_V);
  int g0 = 0, sa = 0, sb = 0, qa = 0, qb = 0;
  bool pre_a = false, pre_b = false;  // S_t(0) of the current item issued by the previous one
  bool ok = true;
  FwdCursor cur{};
  FwdItem it, nx;
  bool have = fwd_next<CAUSAL>(a, cur, it);
  while (have && ok) {
    const bool have_nx = fwd_next<CAUSAL>(a, cur, nx);
    const int n_a = it.n_a, n_b = it.n_b;
    const int n_total = max(n_a, n_b);
    const int g1 = g0 + n_total;  // first K/V step of the next item
    // S_t(0) of tiles that the previous item did not start.
    if ((n_a > 0 && !pre_a) || (n_b > 0 && !pre_b)) {
      ok = mbar_wait_warp(&sh.k_full[g0 % C::NK], (g0 / C::NK) & 1, wc);
      const uint32_t k0 = k_base + (g0 % C::NK) * C::TILE_BYTES;
      if (ok && n_a > 0 && !pre_a) {
        ok = mbar_wait_warp(&sh.q_full[0], qa & 1, wc);
        if (ok) {
          tc_fence_after();
          fwd_issue_s<D, BF16>(tmem, 0, q_a, k0, sh, n_a == 1);
          ++qa;
        }
      }
      if (ok && n_b > 0 && !pre_b) {
        ok = mbar_wait_warp(&sh.q_full[1], qb & 1, wc);
        if (ok) {
          tc_fence_after();
          fwd_issue_s<D, BF16>(tmem, 1, q_b, k0, sh, n_b == 1);
          ++qb;
        }
      }
      if (!ok) break;
    }
    if (n_total > 0) umma_commit_warp(&sh.k_empty[g0 % C::NK]);
    pre_a = pre_b = false;
    bool pend_a = false, pend_b = false;  // S_t(0) of the next item not issued yet
    const uint32_t k_first_next = k_base + (g1 % C::NK) * C::TILE_BYTES;
    const uint32_t k1_par = (g1 / C::NK) & 1;
    // Issues the pending S_A(0) of the next item if its copies have landed.
    auto try_pending_a = [&]() {
      if (pend_a && __all_sync(0xffffffffu, mbar_test_wait(smem_u32(&sh.q_full[0]), qa & 1) &&
                                                mbar_test_wait(smem_u32(&sh.k_full[g1 % C::NK]), k1_par))) {
        tc_fence_after();
        fwd_issue_s<D, BF16>(tmem, 0, q_a, k_first_next, sh, nx.n_a == 1);
        ++qa;
        pre_a = true;
        pend_a = false;
      }
    };
    for (int j = 0; j < n_total && ok; ++j) {
      const int g = g0 + j;
      const bool more = j + 1 < n_total;
      ok = more ? mbar_wait2_warp(&sh.k_full[(g + 1) % C::NK], ((g + 1) / C::NK) & 1,
                                  &sh.v_full[g % C::NV], (g / C::NV) & 1, wc)
                : mbar_wait_warp(&sh.v_full[g % C::NV], (g / C::NV) & 1, wc);
      if (!ok) break;
      const uint32_t v_smem = v_base + (g % C::NV) * C::TILE_BYTES;
      const uint32_t k_next = k_base + ((g + 1) % C::NK) * C::TILE_BYTES;
      if (j < n_a) {
        ok = mbar_wait_warp(&sh.p_full[0], sa & 1, wc);
        if (!ok) break;
        tc_fence_after();
        issue_pv<D, BF16>(tmem + C::TM_O(0), tmem + C::TM_S(0) + C::TM_P_OFF, v_smem, j > 0);
        umma_commit_warp(&sh.o_full[0]);
        ++sa;
        if (j + 1 < n_a)
          fwd_issue_s<D, BF16>(tmem, 0, q_a, k_next, sh, j + 2 == n_a);
        else
          pend_a = have_nx && nx.n_a > 0;
      }
      try_pending_a();
      if (j < n_b) {
        ok = mbar_wait_warp(&sh.p_full[1], sb & 1, wc);
        if (!ok) break;
        tc_fence_after();
        issue_pv<D, BF16>(tmem + C::TM_O(1), tmem + C::TM_S(1) + C::TM_P_OFF, v_smem, j > 0);
        umma_commit_warp(&sh.o_full[1]);
        ++sb;
        if (j + 1 < n_b)
          fwd_issue_s<D, BF16>(tmem, 1, q_b, k_next, sh, j + 2 == n_b);
        else
          pend_b = have_nx && nx.n_b > 0;
      }
      if (more) umma_commit_warp(&sh.k_empty[(g + 1) % C::NK]);
      umma_commit_warp(&sh.v_empty[g % C::NV]);
    }
    if (!ok) break;
    // The next item's first products that are still pending: everything else
    // of this item has been issued, so now they may wait.
    if (pend_a) {
      ok = mbar_wait_warp(&sh.q_full[0], qa & 1, wc) && mbar_wait_warp(&sh.k_full[g1 % C::NK], k1_par, wc);
      if (!ok) break;
      tc_fence_after();
      fwd_issue_s<D, BF16>(tmem, 0, q_a, k_first_next, sh, nx.n_a == 1);
      ++qa;
      pre_a = true;
    }
    if (pend_b) {
      ok = mbar_wait_warp(&sh.q_full[1], qb & 1, wc) && mbar_wait_warp(&sh.k_full[g1 % C::NK], k1_par, wc);
      if (!ok) break;
      tc_fence_after();
      fwd_issue_s<D, BF16>(tmem, 1, q_b, k_first_next, sh, nx.n_b == 1);
      ++qb;
      pre_b = true;
    }
    g0 = g1;
    it = nx;
    have = have_nx;
  }
  // Every product this warp issued must complete before TMEM is released.
  umma_commit_warp(&sh.mma_done);
  mbar_wait_drain(&sh.mma_done, 0, a.timeout_ns);
  return ok;
}

// ---------------- softmax warpgroups ----------------
// Warps 4-7 own tile A, warps 8-11 tile B of every item; TMEM lane = row of
// the tile, one thread per row. Per item: the steps of fwd_softmax_step
// (their barrier phases continue across items in st), then the epilogue
// O / l -> 16-bit rows and L = m + ln l, written straight to global memory.
// The next item's first P V product, which overwrites O_t, waits on this
// warp's next p_full arrival, which comes after these TMEM loads.
template <int D, bool BF16, bool CAUSAL>
__device__ bool fwd_persist_softmax(FwdPShared<D>& sh, uint8_t* smem, uint32_t tmem, const CUtensorMap& tm_o,
                                    const FwdArgs& a, int warp, int lane, const WaitCtx& wc) {
  using C = FwdCfg<D>;
  const int t = (warp - 4) >> 2;   // 0: tile A, 1: tile B
  const int quad = warp & 3;       // TMEM lane quadrant this warp may access
  const int r = quad * 32 + lane;  // row inside the tile == TMEM lane
  const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
  const uint32_t t_s = tmem + lane_off + C::TM_S(t);
  const uint32_t t_p = t_s + C::TM_P_OFF;
  const uint32_t t_o = tmem + lane_off + C::TM_O(t);
  const float sl2 = a.scale_log2;
  const int N = a.N;
  uint8_t* stage = smem + FwdPCfg<D>::OFF_O + (warp - 4) * FwdPCfg<D>::STAGE_BYTES;
  int st = 0;
  bool ok = true;
  FwdCursor cur{};
  FwdItem it;
  while (ok && fwd_next<CAUSAL>(a, cur, it)) {
    const int nt = t == 0 ? it.n_a : it.n_b;
    if (nt == 0) continue;
    const int row_base = it.mb * kFwdRowsPerCta + t * kTileRows;
    const int my_row = row_base + r;
    float m_ref = -INFINITY;  // reference max (raw score units) used by exp
    float l = 0.f;
    for (int j = 0; j < nt; ++j, ++st) {
      ok = fwd_softmax_step<D, BF16, CAUSAL>(&sh.s_full[t], &sh.o_full[t], &sh.p_full[t], t_s, t_p, t_o,
                                             j * kTileRows, row_base, my_row, a.Nk, sl2, j == 0, st & 1,
                                             (st - 1) & 1, m_ref, l, lane, wc);
      if (!ok) break;
    }
    if (ok) ok = mbar_wait_warp(&sh.o_full[t], (st - 1) & 1, wc);
    if (!ok) break;
    __syncwarp();
    tc_fence_after();
    fwd_store_rows<D, BF16>(t_o, stage, &tm_o, row_base + quad * 32, it.bh, 1.f / l, lane);
    if (my_row < N) a.lse[static_cast<size_t>(it.bh) * N + my_row] = (m_ref * sl2 + lg2_approx(l)) * kLn2;
  }
  // The last stores must have read the staging buffer before the CTA exits.
  if (lane == 0) bulk_wait_group_read0();
  __syncwarp();
  return ok;
}

template <int D, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(384, 1)
    fa2_fwd_persist_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                           const FwdArgs a) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  __shared__ FwdPShared<D> sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(&sh.q_full[t], 1);
      mbar_init(&sh.q_free[t], 1);
      mbar_init(&sh.s_full[t], 1);
      mbar_init(&sh.p_full[t], 4);  // one arrival per softmax warp of the tile
      mbar_init(&sh.o_full[t], 1);
    }
    for (int i = 0; i < C::NK; ++i) { mbar_init(&sh.k_full[i], 1); mbar_init(&sh.k_empty[i], 1); }
    for (int i = 0; i < C::NV; ++i) { mbar_init(&sh.v_full[i], 1); mbar_init(&sh.v_empty[i], 1); }
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
  const WaitCtx wc{a.status, &sh.abort_flag, a.timeout_ns};
  if (warp < 4) {
    // 4 x 32 x 120 + 8 x 32 x 192 = 64,512 = the launch's 384 x 168 registers
    // (the issuer, which carries two items and all pipeline counters, spills
    // below 120; the softmax needs no more than 192).
    setmaxnreg_dec<120>();
    if (warp == 0 && lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      fwd_persist_k_producer<D, CAUSAL>(sh, smem, tm_q, tm_k, a, wc);
    } else if (warp == 3 && lane == 0) {
      tma_prefetch_desc(&tm_v);
      fwd_persist_v_producer<D, CAUSAL>(sh, smem, tm_v, a, wc);
    } else if (warp == 1) {
      fwd_persist_issuer<D, BF16, CAUSAL>(sh, smem, tmem, a, wc);
    }
  } else {
    setmaxnreg_inc<192>();
    fwd_persist_softmax<D, BF16, CAUSAL>(sh, smem, tmem, tm_o, a, warp, lane, wc);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace fa2
