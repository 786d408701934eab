// The backward's main launch (included by fa2_bwd.cu after the shared-memory
// and TMEM layouts it uses, BwdCfg and DqCfg).
//
// One CTA per SM takes work items from a counter in the workspace (its first
// item is its own index): first the
// dK/dV workers' key blocks ("FlashAttention学习笔记(2)", Foward和backward中的
// thread block划分: one worker per K/V column block), then the dQ workers'
// query blocks, each in the order the per-block launch used (block fastest,
// then batch, then head; longest first under a causal mask). Taking items from
// a counter balances unequal causal blocks without a schedule.
//
// Inside a CTA the producer warp takes an item, publishes it in a small ring
// of item slots, and loads its operands; the MMA issuer and the compute warps
// read the same slots. The streamed-operand rings and every pipeline barrier
// keep counting across items, so the next item's loads and first products
// overlap the current item's last tile and its epilogue, and nothing waits for
// a new CTA to start. The epilogues write dK, dV and dQ from TMEM straight to
// global memory (each thread owns one row), so they need no staging buffer.
#pragma once

namespace fa2 {

constexpr int kItemSlots = 4;

struct BwdItem {
  int kind;  // 0: dK/dV worker (blk = key block), 1: dQ worker (blk = longest-first rank), 2: none left
  int blk;
  int bh;
};

struct BwdPShared {
  // dK/dV role
  uint64_t kv_full;                // K_j, V_j of the item landed (one phase per item with work)
  uint64_t q_full[2], do_full[2];  // streamed Q_i / dO_i ring
  uint64_t s_empty[2];             // ring stage free (committed after dK of its tile)
  uint64_t st_full, dpt_full;      // S^T(i), dP^T(i) complete
  uint64_t p_done, ds_done;        // P^T(i), dS^T(i) written by the 8 compute warps
  uint64_t kv_res_free;            // the item's last S^T and dP^T complete: K, V may be replaced
  uint64_t kv_acc_done;            // the item's last dK complete: dV, dK final in TMEM
  // dQ role
  uint64_t qq_full;                // Q, dO of the item landed
  uint64_t k_full[3], k_empty[3];  // K ring
  uint64_t v_full[2], v_empty[2];  // V ring
  uint64_t sq_full, sq_free;
  uint64_t dsq_full[2];            // dS(h) written by the 8 compute warps, one barrier per dS
                                   // buffer: the warps may finish dS(h+1) before the issuer has
                                   // waited for dS(h), and a parity wait must never fall two
                                   // phases behind its barrier
  uint64_t q_res_free;             // the item's last S and dP complete: Q, dO may be replaced
  uint64_t dq_acc_done;            // the item's last dQ product complete
  // items
  uint64_t item_full[kItemSlots], item_empty[kItemSlots];
  BwdItem items[kItemSlots];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort_flag;
};

// The item with index idx of the combined list: kv_items dK/dV key blocks, then
// the dQ query blocks.
__device__ __forceinline__ BwdItem bwd_item_of(long long idx, const BwdArgs& a, int nkb, int nm,
                                               long long kv_items, long long total) {
  BwdItem it;
  if (idx >= total) {
    it.kind = 2;
    it.blk = 0;
    it.bh = 0;
  } else if (idx < kv_items) {
    const int x = static_cast<int>(idx);
    const int rest = x / nkb;
    it.kind = 0;
    it.blk = x % nkb;
    it.bh = (rest % a.B) * a.H + rest / a.B;
  } else {
    const int y = static_cast<int>(idx - kv_items);
    const int rest = y / nm;
    it.kind = 1;
    it.blk = y % nm;
    it.bh = (rest % a.B) * a.H + rest / a.B;
  }
  return it;
}

// Query tiles of a dK/dV item (key block nb) and K/V tiles of a dQ item.
template <bool CAUSAL>
__device__ __forceinline__ int kv_item_steps(int nb, int N) {
  return max(0, ceil_div(N, kTileRows) - bwd_q_tile_begin(nb, CAUSAL));
}
template <bool CAUSAL>
__device__ __forceinline__ int dq_item_tiles(int rank, int nm, const BwdArgs& a) {
  const int q0 = dq_m_block_of(rank, nm, CAUSAL) * kTileRows;
  return fwd_kv_tile_end(q0, min(a.N, q0 + kTileRows), a.Nk, CAUSAL);
}

// Counters each role keeps across items (phases of the rings and barriers).
struct BwdRoleCount {
  int kv_items;   // dK/dV items with at least one query tile
  int kv_tiles;   // query tiles of all dK/dV items
  int q_items;    // dQ items with at least one K/V tile
  int q_tiles;    // K/V tiles of all dQ items
};

// ---------------- producer (one thread of warp 0) ----------------
// Returns false if a wait gave up; every copy it issued has then been drained.
// last_*[i] is the phase number last armed on barrier i (-1: never), so the
// drain waits only for copies that were issued.
template <int D, bool CAUSAL>
__device__ bool bwd_persist_producer(BwdPShared& sh, uint8_t* smem, const CUtensorMap& tm_q,
                                     const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                     const CUtensorMap& tm_do, const BwdArgs& a, int nkb, int nm,
                                     long long kv_items, long long total, const WaitCtx& wc) {
  using C = BwdCfg<D>;
  using Q = DqCfg<D>;
  BwdRoleCount n{0, 0, 0, 0};
  int last_kv = -1, last_qq = -1;
  int last_q[C::NS], last_do[C::NS], last_k[Q::NK], last_v[Q::NV];
  for (int i = 0; i < C::NS; ++i) last_q[i] = last_do[i] = -1;
  for (int i = 0; i < Q::NK; ++i) last_k[i] = -1;
  for (int i = 0; i < Q::NV; ++i) last_v[i] = -1;
  int prev_kind = -1;
  bool ok = true;
  for (int k = 0; ok; ++k) {
    const int slot = k % kItemSlots;
    if (k >= kItemSlots) {
      ok = mbar_wait(&sh.item_empty[slot], ((k / kItemSlots) & 1) ^ 1, wc);
      if (!ok) break;
    }
    // The first item is the CTA's own index (the grid has at most as many
    // CTAs as items), so no CTA starts behind a global atomic; later items
    // come from the counter, past the first gridDim.x.
    const long long idx = (k == 0) ? static_cast<long long>(blockIdx.x)
                                   : static_cast<long long>(gridDim.x) + atomicAdd(a.item_counter, 1);
    const BwdItem it = bwd_item_of(idx, a, nkb, nm, kv_items, total);
    sh.items[slot] = it;
    mbar_arrive(&sh.item_full[slot]);  // release: the item is visible to the waiters
    if (it.kind == 2) break;
    if (it.kind == 1 && prev_kind == 0 && n.kv_tiles > 0) {
      // Role switch: the dQ layout reuses the dK/dV operands' shared memory, so
      // every dK/dV product must have completed, and with them every copy they
      // read. The ring stage of the last dK/dV tile is released by a commit
      // behind that tile's dK, the last product issued. A parity wait is only
      // exact while the phase before it has completed: this barrier's was
      // waited for when that tile was loaded, whereas the item-level barriers
      // may lag this thread by more than one phase.
      const int g = n.kv_tiles - 1;
      ok = mbar_wait(&sh.s_empty[g % C::NS], (g / C::NS) & 1, wc);
      if (!ok) break;
    }
    prev_kind = it.kind;
    if (it.kind == 0) {
      const int steps = kv_item_steps<CAUSAL>(it.blk, a.N);
      if (steps == 0) continue;
      const int n0 = it.blk * kTileRows;
      const int i_begin = bwd_q_tile_begin(it.blk, CAUSAL);
      if (n.kv_items > 0) {  // K, V of the previous item are read by its last S^T, dP^T
        ok = mbar_wait(&sh.kv_res_free, (n.kv_items - 1) & 1, wc);
        if (!ok) break;
      }
      mbar_arrive_expect_tx(&sh.kv_full, 2 * C::TILE_BYTES);
      load_tile<D>(smem + C::OFF_FIX0, &tm_k, &sh.kv_full, n0, it.bh);
      load_tile<D>(smem + C::OFF_FIX1, &tm_v, &sh.kv_full, n0, it.bh);
      last_kv = n.kv_items;
      for (int i = 0; i < steps && ok; ++i) {
        const int g = n.kv_tiles + i;
        const int st = g % C::NS, ph = g / C::NS;
        ok = mbar_wait(&sh.s_empty[st], (ph & 1) ^ 1, wc);
        if (!ok) break;
        const int q0 = (i_begin + i) * kTileRows;
        mbar_arrive_expect_tx(&sh.q_full[st], C::TILE_BYTES);
        load_tile<D>(smem + C::OFF_STR0 + st * C::TILE_BYTES, &tm_q, &sh.q_full[st], q0, it.bh);
        last_q[st] = ph;
        if (a.fault == 1 && idx == 0 && i == 0) continue;  // failure-path test: dO never arrives
        mbar_arrive_expect_tx(&sh.do_full[st], C::TILE_BYTES);
        load_tile<D>(smem + C::OFF_STR1 + st * C::TILE_BYTES, &tm_do, &sh.do_full[st], q0, it.bh);
        last_do[st] = ph;
      }
      if (!ok) break;
      n.kv_tiles += steps;
      ++n.kv_items;
    } else {
      const int tiles = dq_item_tiles<CAUSAL>(it.blk, nm, a);
      if (tiles == 0) continue;
      const int q0 = dq_m_block_of(it.blk, nm, CAUSAL) * kTileRows;
      if (n.q_items > 0) {  // Q, dO of the previous item are read by its last S, dP
        ok = mbar_wait(&sh.q_res_free, (n.q_items - 1) & 1, wc);
        if (!ok) break;
      }
      mbar_arrive_expect_tx(&sh.qq_full, 2 * C::TILE_BYTES);
      load_tile<D>(smem + Q::OFF_Q, &tm_q, &sh.qq_full, q0, it.bh);
      load_tile<D>(smem + Q::OFF_DO, &tm_do, &sh.qq_full, q0, it.bh);
      last_qq = n.q_items;
      for (int j = 0; j < tiles && ok; ++j) {
        const int h = n.q_tiles + j;
        const int ks = h % Q::NK, vs = h % Q::NV;
        ok = mbar_wait(&sh.k_empty[ks], ((h / Q::NK) & 1) ^ 1, wc);
        if (!ok) break;
        mbar_arrive_expect_tx(&sh.k_full[ks], C::TILE_BYTES);
        load_tile<D>(smem + Q::OFF_K + ks * C::TILE_BYTES, &tm_k, &sh.k_full[ks], j * kTileRows, it.bh);
        last_k[ks] = h / Q::NK;
        ok = mbar_wait(&sh.v_empty[vs], ((h / Q::NV) & 1) ^ 1, wc);
        if (!ok) break;
        if (a.fault == 2 && idx == kv_items && j == 0) continue;  // failure-path test: V never arrives
        mbar_arrive_expect_tx(&sh.v_full[vs], C::TILE_BYTES);
        load_tile<D>(smem + Q::OFF_V + vs * C::TILE_BYTES, &tm_v, &sh.v_full[vs], j * kTileRows, it.bh);
        last_v[vs] = h / Q::NV;
      }
      if (!ok) break;
      n.q_tiles += tiles;
      ++n.q_items;
    }
  }
  if (!ok) {
    // Drain every copy that may still be landing before the CTA gives up its
    // shared memory (a completed phase returns at once; the drain ignores the
    // abort flag and is bounded).
    if (last_kv >= 0) mbar_wait_drain(&sh.kv_full, last_kv & 1, a.timeout_ns);
    if (last_qq >= 0) mbar_wait_drain(&sh.qq_full, last_qq & 1, a.timeout_ns);
    for (int i = 0; i < C::NS; ++i) {
      if (last_q[i] >= 0) mbar_wait_drain(&sh.q_full[i], last_q[i] & 1, a.timeout_ns);
      if (last_do[i] >= 0) mbar_wait_drain(&sh.do_full[i], last_do[i] & 1, a.timeout_ns);
    }
    for (int i = 0; i < Q::NK; ++i)
      if (last_k[i] >= 0) mbar_wait_drain(&sh.k_full[i], last_k[i] & 1, a.timeout_ns);
    for (int i = 0; i < Q::NV; ++i)
      if (last_v[i] >= 0) mbar_wait_drain(&sh.v_full[i], last_v[i] & 1, a.timeout_ns);
  }
  return ok;
}

// ---------------- MMA issuer (warp 1; one lane issues) ----------------
// dK/dV item: S^T(0), dP^T(0), then per query tile dV(i), S^T(i+1), dK(i),
// dP^T(i+1). The compute warps write P^T(i) over S^T(i) in TMEM as soon as it
// is formed, so dV(i) runs before dS^T(i) exists, and dS^T(i) over dP^T(i).
// The tensor core runs products in issue order, which also orders each product
// that overwrites a TMEM region after the product that reads it. Two chains
// cross from tile to tile, S^T -> P^T -> dV -> S^T and dP^T -> dS^T -> dK ->
// dP^T; each holds two products and one step of the compute warps, so while
// the compute warps form P^T(i+1) the tensor core runs dK(i) and dP^T(i+1).
// dQ item: S(0), dP(0), then per K/V tile j: S(j+1), dP(j+1) as soon as the
// compute warps have read S(j), dP(j) (two dS buffers), and dQ(j). A new item's S^T(0) is issued
// behind the previous item's last dK, so it overlaps that item's epilogue; its
// first dV / dK (accumulate off) come after the compute warps' next arrivals,
// which they make only once the previous item's accumulators are read out.
template <int D, bool BF16, bool CAUSAL>
__device__ bool bwd_persist_issuer(BwdPShared& sh, uint8_t* smem, uint32_t tmem, const BwdArgs& a,
                                   int nm, const WaitCtx& wc) {
  using C = BwdCfg<D>;
  using Q = DqCfg<D>;
  BwdRoleCount n{0, 0, 0, 0};
  bool ok = true;
  int prev_kind = -1, prev_slot = 0, prev_k = 0;
  const uint32_t t_pt = tmem + C::KV_ST, t_dst = tmem + C::KV_DPT;
  auto pt_col = [t_pt](int kk) { return t_pt + C::pair_col(kk); };
  auto dst_col = [t_dst](int kk) { return t_dst + C::pair_col(kk); };
  for (int k = 0; ok; ++k) {
    const int slot = k % kItemSlots;
    ok = mbar_wait_warp(&sh.item_full[slot], (k / kItemSlots) & 1, wc);
    if (!ok) break;
    const BwdItem it = sh.items[slot];
    if (it.kind == 2) break;
    if (it.kind == 1 && prev_kind == 0) {
      // Role switch: the dQ products write TMEM columns that hold the last
      // dK/dV item's accumulators; wait until the compute warps have released
      // that item (after its epilogue).
      ok = mbar_wait_warp(&sh.item_empty[prev_slot], (prev_k / kItemSlots) & 1, wc);
      if (!ok) break;
    }
    if (it.kind == 0) {
      const int steps = kv_item_steps<CAUSAL>(it.blk, a.N);
      if (steps > 0) {
        const uint32_t k_s = smem_u32(smem + C::OFF_FIX0), v_s = smem_u32(smem + C::OFF_FIX1);
        auto q_at = [&](int g) { return smem_u32(smem + C::OFF_STR0 + (g % C::NS) * C::TILE_BYTES); };
        auto do_at = [&](int g) { return smem_u32(smem + C::OFF_STR1 + (g % C::NS) * C::TILE_BYTES); };
        const int g0 = n.kv_tiles;
        ok = mbar_wait_warp(&sh.kv_full, n.kv_items & 1, wc) &&
             mbar_wait_warp(&sh.q_full[g0 % C::NS], (g0 / C::NS) & 1, wc);
        if (ok) {
          tc_fence_after();
          mma_rows_x_rows<D, BF16>(tmem + C::KV_ST, k_s, q_at(g0));
          umma_commit_warp(&sh.st_full);
          ok = mbar_wait_warp(&sh.do_full[g0 % C::NS], (g0 / C::NS) & 1, wc);
        }
        if (ok) {
          tc_fence_after();
          mma_rows_x_rows<D, BF16>(tmem + C::KV_DPT, v_s, do_at(g0));
          umma_commit_warp(&sh.dpt_full);
          if (steps == 1) umma_commit_warp(&sh.kv_res_free);
        }
        for (int i = 0; i < steps && ok; ++i) {
          const int g = g0 + i, gx = g + 1;
          ok = mbar_wait_warp(&sh.p_done, g & 1, wc);
          if (!ok) break;
          tc_fence_after();
          mma_tmem_x_tile<D, BF16>(tmem + C::KV_DV, pt_col, do_at(g), i > 0);
          if (i + 1 < steps) {
            ok = mbar_wait_warp(&sh.q_full[gx % C::NS], (gx / C::NS) & 1, wc);
            if (!ok) break;
            tc_fence_after();
            mma_rows_x_rows<D, BF16>(tmem + C::KV_ST, k_s, q_at(gx));
            umma_commit_warp(&sh.st_full);
          }
          ok = mbar_wait_warp(&sh.ds_done, g & 1, wc);
          if (!ok) break;
          tc_fence_after();
          mma_tmem_x_tile<D, BF16>(tmem + C::KV_DK, dst_col, q_at(g), i > 0);
          umma_commit_warp(&sh.s_empty[g % C::NS]);
          if (i + 1 < steps) {
            ok = mbar_wait_warp(&sh.do_full[gx % C::NS], (gx / C::NS) & 1, wc);
            if (!ok) break;
            tc_fence_after();
            mma_rows_x_rows<D, BF16>(tmem + C::KV_DPT, v_s, do_at(gx));
            umma_commit_warp(&sh.dpt_full);
            if (i + 2 == steps) umma_commit_warp(&sh.kv_res_free);
          }
        }
        if (!ok) break;
        umma_commit_warp(&sh.kv_acc_done);
        n.kv_tiles += steps;
        ++n.kv_items;
      }
    } else {
      const int tiles = dq_item_tiles<CAUSAL>(it.blk, nm, a);
      if (tiles > 0) {
        const uint32_t q_s = smem_u32(smem + Q::OFF_Q), do_s = smem_u32(smem + Q::OFF_DO);
        auto k_at = [&](int h) { return smem_u32(smem + Q::OFF_K + (h % Q::NK) * C::TILE_BYTES); };
        auto v_at = [&](int h) { return smem_u32(smem + Q::OFF_V + (h % Q::NV) * C::TILE_BYTES); };
        const int h0 = n.q_tiles;
        ok = mbar_wait_warp(&sh.qq_full, n.q_items & 1, wc) &&
             mbar_wait_warp(&sh.k_full[h0 % Q::NK], (h0 / Q::NK) & 1, wc) &&
             mbar_wait_warp(&sh.v_full[h0 % Q::NV], (h0 / Q::NV) & 1, wc);
        if (ok) {
          tc_fence_after();
          mma_rows_x_rows<D, BF16>(tmem + C::Q_S, q_s, k_at(h0));
          mma_rows_x_rows<D, BF16>(tmem + C::Q_DP, do_s, v_at(h0));
          umma_commit_warp(&sh.sq_full);
          umma_commit_warp(&sh.v_empty[h0 % Q::NV]);
          if (tiles == 1) umma_commit_warp(&sh.q_res_free);
        }
        for (int j = 0; j < tiles && ok; ++j) {
          const int h = h0 + j, hx = h + 1;
          ok = mbar_wait_warp(&sh.sq_free, h & 1, wc);
          if (!ok) break;
          tc_fence_after();
          if (j + 1 < tiles) {
            ok = mbar_wait2_warp(&sh.k_full[hx % Q::NK], (hx / Q::NK) & 1, &sh.v_full[hx % Q::NV],
                                 (hx / Q::NV) & 1, wc);
            if (!ok) break;
            tc_fence_after();
            mma_rows_x_rows<D, BF16>(tmem + C::Q_S, q_s, k_at(hx));
            mma_rows_x_rows<D, BF16>(tmem + C::Q_DP, do_s, v_at(hx));
            umma_commit_warp(&sh.sq_full);
            umma_commit_warp(&sh.v_empty[hx % Q::NV]);
            if (j + 2 == tiles) umma_commit_warp(&sh.q_res_free);
          }
          ok = mbar_wait_warp(&sh.dsq_full[h & 1], (h >> 1) & 1, wc);
          if (!ok) break;
          tc_fence_after();
          const uint32_t ds_col = tmem + C::Q_DS(h & 1);
          mma_tmem_x_tile<D, BF16>(tmem + C::Q_DQ, [ds_col](int kk) { return ds_col + 8u * kk; },
                                         k_at(h), j > 0);
          umma_commit_warp(&sh.k_empty[h % Q::NK]);  // K_h's last reader is dQ(h)
        }
        if (!ok) break;
        umma_commit_warp(&sh.dq_acc_done);
        n.q_tiles += tiles;
        ++n.q_items;
      }
    }
    // Every role warp releases the slot once it is done with the item.
    if ((threadIdx.x & 31) == 0) mbar_arrive(&sh.item_empty[slot]);
    prev_kind = it.kind;
    prev_slot = slot;
    prev_k = k;
  }
  // Every product this warp issued must complete before TMEM is released.
  umma_commit_warp(&sh.mma_done);
  mbar_wait_drain(&sh.mma_done, 0, a.timeout_ns);
  return ok;
}

// Columns [c0, c1) of this thread's TMEM row, times mul, rounded to 16 bits and
// written to the row's global memory (dst = the row's first element; each
// thread owns one row). The TMEM loads are warp-collective: every lane runs
// them, and only rows inside the tensor (valid) store.
template <int D, bool BF16>
__device__ __forceinline__ void store_row_global(uint32_t t_row, uint16_t* dst, bool valid, float mul,
                                                 int c0, int c1) {
#pragma unroll
  for (int c = 0; c < D; c += 32) {
    if (c < c0 || c >= c1) continue;
    uint32_t x[32];
    tmem_ld_32x32b_x32(t_row + c, x);
    tmem_wait_ld();
    reg_fence(x);
    if (valid) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint4 val;
        val.x = pack_x2<BF16>(__uint_as_float(x[8 * k + 0]) * mul, __uint_as_float(x[8 * k + 1]) * mul);
        val.y = pack_x2<BF16>(__uint_as_float(x[8 * k + 2]) * mul, __uint_as_float(x[8 * k + 3]) * mul);
        val.z = pack_x2<BF16>(__uint_as_float(x[8 * k + 4]) * mul, __uint_as_float(x[8 * k + 5]) * mul);
        val.w = pack_x2<BF16>(__uint_as_float(x[8 * k + 6]) * mul, __uint_as_float(x[8 * k + 7]) * mul);
        *reinterpret_cast<uint4*>(dst + c + 8 * k) = val;
      }
    }
  }
}

// ---------------- compute warps (warps 4-11) ----------------
// dK/dV items: P^T and dS^T for query columns [0,64) / [64,128) of each tile
// (TMEM lane = key), as in the per-block worker; then dV (warpgroup 0) or
// scale * dK (warpgroup 1) of the block's 128 keys, straight to global memory.
// dQ items: dS for key columns [0,64) / [64,128) (TMEM lane = query); then
// scale * dQ, columns split between the two warpgroups.
template <int D, bool BF16, bool CAUSAL>
__device__ bool bwd_persist_compute(BwdPShared& sh, uint8_t* smem, uint32_t tmem, const BwdArgs& a,
                                    int nm, const WaitCtx& wc) {
  using C = BwdCfg<D>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wg = (warp - 4) >> 2;
  const int quad = warp & 3;
  const int r = quad * 32 + lane;  // TMEM lane of this thread
  const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
  const float sl2 = a.scale_log2;
  const int N = a.N, Nk = a.Nk;
  float* ld_s = reinterpret_cast<float*>(smem + C::OFF_LD) + (warp - 4) * 128;
  BwdRoleCount n{0, 0, 0, 0};
  bool ok = true;
  for (int k = 0; ok; ++k) {
    const int slot = k % kItemSlots;
    ok = mbar_wait_warp(&sh.item_full[slot], (k / kItemSlots) & 1, wc);
    if (!ok) break;
    const BwdItem it = sh.items[slot];
    if (it.kind == 2) break;
    const int bh = it.bh;
    if (it.kind == 0) {
      // ---------------- dK/dV item ----------------
      const int steps = kv_item_steps<CAUSAL>(it.blk, N);
      const int n0 = it.blk * kTileRows;
      const int i_begin = bwd_q_tile_begin(it.blk, CAUSAL);
      const int kg = n0 + r;
      const uint32_t t_st = tmem + lane_off + C::KV_ST + 64 * wg;
      const uint32_t t_dpt = tmem + lane_off + C::KV_DPT + 64 * wg;
      for (int i = 0; i < steps; ++i) {
        const int g = n.kv_tiles + i;
        const int q0 = (i_begin + i) * kTileRows;
        const int qc0 = q0 + 64 * wg;  // first query column of this warpgroup
        // L * log2e and D of this warpgroup's 64 query columns, the same for
        // every thread, loaded before waiting for the scores (they do not
        // depend on S). At d = 128 the warp stages them through its shared
        // slice (coalesced loads, then broadcast reads); at d = 64 warp-uniform
        // 16-byte loads through L1 measured faster (and slower at d = 128).
        const size_t crow = static_cast<size_t>(bh) * a.n_pad + qc0;
        if (D != 64) {
          const float2 l2v = *reinterpret_cast<const float2*>(a.l2_pad + crow + 2 * lane);
          const float2 dv2 = *reinterpret_cast<const float2*>(a.dsum_pad + crow + 2 * lane);
          __syncwarp();  // every lane is done with the previous step's values
          *reinterpret_cast<float2*>(ld_s + 2 * lane) = make_float2(-l2v.x, -l2v.y);
          *reinterpret_cast<float2*>(ld_s + 64 + 2 * lane) = dv2;
          __syncwarp();
        }
        float lreg[64];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          float4 l4;
          if (D == 64) {
            l4 = __ldg(reinterpret_cast<const float4*>(a.l2_pad + crow) + u);
            l4 = make_float4(-l4.x, -l4.y, -l4.z, -l4.w);
          } else {
            l4 = reinterpret_cast<const float4*>(ld_s)[u];
          }
          lreg[4 * u] = l4.x; lreg[4 * u + 1] = l4.y; lreg[4 * u + 2] = l4.z; lreg[4 * u + 3] = l4.w;
        }
        ok = mbar_wait_warp(&sh.st_full, g & 1, wc);
        if (!ok) break;
        __syncwarp();  // the warp-collective TMEM loads below need a converged warp
        tc_fence_after();
        uint32_t sv[64];
        tmem_ld_32x32b_x32(t_st, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
        tmem_ld_32x32b_x32(t_st + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
        tmem_wait_ld();
        reg_fence(sv);
        const bool need_mask = (CAUSAL && qc0 < n0 + kTileRows - 1) || (qc0 + 64 > N) ||
                               (n0 + kTileRows > Nk);
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
          const float4 d4 = D == 64 ? __ldg(reinterpret_cast<const float4*>(a.dsum_pad + crow) + u)
                                    : reinterpret_cast<const float4*>(ld_s + 64)[u];
          dreg[4 * u] = d4.x; dreg[4 * u + 1] = d4.y; dreg[4 * u + 2] = d4.z; dreg[4 * u + 3] = d4.w;
        }
        ok = mbar_wait_warp(&sh.dpt_full, g & 1, wc);
        if (!ok) break;
        __syncwarp();
        tc_fence_after();
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
      if (!ok) break;
      // Epilogue: dV (warpgroup 0) or scale * dK (warpgroup 1) of this block's keys.
      uint16_t* out = static_cast<uint16_t*>(wg == 0 ? a.dv : a.dk) +
                      (static_cast<size_t>(bh) * Nk + kg) * D;
      const bool row_in = kg < Nk;
      if (steps > 0) {
        ok = mbar_wait_warp(&sh.kv_acc_done, n.kv_items & 1, wc);
        if (!ok) break;
        __syncwarp();
        tc_fence_after();
        store_row_global<D, BF16>(tmem + lane_off + (wg == 0 ? C::KV_DV : C::KV_DK), out, row_in,
                                  wg == 0 ? 1.f : a.scale, 0, D);
        n.kv_tiles += steps;
        ++n.kv_items;
      } else if (row_in) {
        // No query sees these keys: their gradients are zero.
#pragma unroll
        for (int c = 0; c < D; c += 8) *reinterpret_cast<uint4*>(out + c) = make_uint4(0u, 0u, 0u, 0u);
      }
    } else {
      // ---------------- dQ item ----------------
      const int tiles = dq_item_tiles<CAUSAL>(it.blk, nm, a);
      const int q0 = dq_m_block_of(it.blk, nm, CAUSAL) * kTileRows;
      const int my_row = q0 + r;
      const float l2 = a.l2_pad[static_cast<size_t>(bh) * a.n_pad + my_row];
      const float dsum = a.dsum_pad[static_cast<size_t>(bh) * a.n_pad + my_row];
      const int lim = CAUSAL ? min(Nk, my_row + 1) : Nk;  // keys < lim are visible
      const bool row_ok = my_row < N;
      for (int j = 0; j < tiles; ++j) {
        const int h = n.q_tiles + j;
        const int kc0 = j * kTileRows + 64 * wg;  // first key column of this warpgroup
        ok = mbar_wait_warp(&sh.sq_full, h & 1, wc);
        if (!ok) break;
        __syncwarp();
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
        if (lane == 0) mbar_arrive(&sh.sq_free);
        const bool need_mask = (CAUSAL && kc0 + 63 > q0) || (kc0 + 64 > Nk) || (q0 + kTileRows > N);
        uint32_t dsp[32];
        if (need_mask)
          dq_ds_cols<true, BF16>(s, dp, sl2, l2, dsum, kc0, lim, row_ok, dsp);
        else
          dq_ds_cols<false, BF16>(s, dp, sl2, l2, dsum, kc0, lim, row_ok, dsp);
        tmem_st_32x32b_x32(tmem + lane_off + C::Q_DS(h & 1) + 32 * wg, dsp);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.dsq_full[h & 1]);
      }
      if (!ok) break;
      // Epilogue: scale * dQ of this block's rows; warpgroup w stores columns [w*D/2, (w+1)*D/2).
      if (tiles > 0) {
        ok = mbar_wait_warp(&sh.dq_acc_done, n.q_items & 1, wc);
        if (!ok) break;
        __syncwarp();
        tc_fence_after();
        uint16_t* out = static_cast<uint16_t*>(a.dq) + (static_cast<size_t>(bh) * N + my_row) * D;
        store_row_global<D, BF16>(tmem + lane_off + C::Q_DQ, out, row_ok, a.scale, wg * (D / 2),
                                  (wg + 1) * (D / 2));
        n.q_tiles += tiles;
        ++n.q_items;
      }
    }
    // The accumulators of this item have been read: release the slot (the MMA
    // issuer waits for that before a role switch reuses their TMEM columns).
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.item_empty[slot]);
  }
  return ok;
}

// ---------------- the persistent main launch ----------------
template <int D, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(384, 1)
    fa2_bwd_main_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                           const BwdArgs a, int num_m_blocks, int nkb, long long kv_items,
                           long long total) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  __shared__ BwdPShared sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&sh.kv_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sh.q_full[s], 1);
      mbar_init(&sh.do_full[s], 1);
      mbar_init(&sh.s_empty[s], 1);
      mbar_init(&sh.v_full[s], 1);
      mbar_init(&sh.v_empty[s], 1);
    }
    mbar_init(&sh.st_full, 1);
    mbar_init(&sh.dpt_full, 1);
    mbar_init(&sh.p_done, 8);  // the eight compute warps
    mbar_init(&sh.ds_done, 8);
    mbar_init(&sh.kv_res_free, 1);
    mbar_init(&sh.kv_acc_done, 1);
    mbar_init(&sh.qq_full, 1);
    for (int s = 0; s < 3; ++s) {
      mbar_init(&sh.k_full[s], 1);
      mbar_init(&sh.k_empty[s], 1);
    }
    mbar_init(&sh.sq_full, 1);
    mbar_init(&sh.sq_free, 8);
    mbar_init(&sh.dsq_full[0], 8);
    mbar_init(&sh.dsq_full[1], 8);
    mbar_init(&sh.q_res_free, 1);
    mbar_init(&sh.dq_acc_done, 1);
    for (int s = 0; s < kItemSlots; ++s) {
      mbar_init(&sh.item_full[s], 1);   // the producer
      mbar_init(&sh.item_empty[s], 9);  // the MMA warp and the eight compute warps
    }
    mbar_init(&sh.mma_done, 1);
    sh.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sh.tmem_base, BwdCfg<D>::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;
  const WaitCtx wc{a.status, &sh.abort_flag, a.timeout_ns};
  if (warp < 4) {
    // 4 x 32 x 88 + 8 x 32 x 208 = 64,512 = the launch's 384 x 168 registers;
    // the issuer, which carries both roles' loops, needs the 88.
    setmaxnreg_dec<88>();
    if (warp == 0 && lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      bwd_persist_producer<D, CAUSAL>(sh, smem, tm_q, tm_k, tm_v, tm_do, a, nkb, num_m_blocks,
                                      kv_items, total, wc);
    } else if (warp == 1) {
      bwd_persist_issuer<D, BF16, CAUSAL>(sh, smem, tmem, a, num_m_blocks, wc);
    }
  } else {
    setmaxnreg_inc<208>();
    bwd_persist_compute<D, BF16, CAUSAL>(sh, smem, tmem, a, num_m_blocks, wc);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, BwdCfg<D>::TMEM_COLS);
  }
}

}  // namespace fa2
