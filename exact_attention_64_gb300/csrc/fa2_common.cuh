// Shared definitions of the FlashAttention-2 library: argument blocks, the
// work mapping (which rows/keys each CTA owns) and small device utilities.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include "sm103_ptx.cuh"

namespace fa2 {

__host__ __device__ constexpr int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Q, K, V row tiles are 128 rows: one tcgen05 M=128 MMA covers one tile and
// TMEM lane i holds row i of it.
constexpr int kTileRows = 128;
// A forward CTA owns two adjacent Q tiles (256 query rows) of one (batch, head)
// and streams every visible K/V tile once for both of them.
constexpr int kFwdRowsPerCta = 2 * kTileRows;

// Forward work mapping. The grid is (num_m_block, batch, heads) with the row
// block varying fastest, as in the FlashAttention-2 thread-block layout
// ("FlashAttention学习笔记(2)", V2中的thread blocks排布): CTAs that read the same
// K/V run back to back and share it through L2. Under a causal mask the row
// blocks are launched longest first.
__host__ __device__ inline int fwd_num_m_blocks(int N) { return ceil_div(N, kFwdRowsPerCta); }

__host__ __device__ inline int fwd_m_block_of(int block_x, int num_m_blocks, int causal) {
  return causal ? (num_m_blocks - 1 - block_x) : block_x;
}

// Half-open K/V tile range [0, end) that query rows [row_begin, row_end) visit.
// Under the causal mask a K/V tile whose first key is past the last query row
// is entirely masked and is skipped, neither loaded nor computed
// ("flash-attention123和ring-attention", 优化3).
// N_k is the key length; with causal masking (top-left: key j visible to
// query i iff j <= i) the range also stops at the last tile of the keys.
__host__ __device__ inline int fwd_kv_tile_end(int row_begin, int row_end, int N_k, int causal) {
  if (row_end <= row_begin) return 0;
  const int all = ceil_div(N_k, kTileRows);
  return causal ? min(ceil_div(row_end, kTileRows), all) : all;
}

// KV split ("大猿搬砖简记", thread-block section, the num_splits_heuristic_fwd
// paragraph). When the (row block, batch, head) workers cannot fill the SMs,
// the K/V tile range [0, n) of a worker is cut into contiguous parts merged
// later by the online-softmax rule. num_splits is the part count of the
// longest range (n_max tiles); a shorter range (causal row blocks) gets
// proportionally fewer parts, min(n, ceil(n * num_splits / n_max)), so that no
// part is empty and none is longer than ceil(n_max / num_splits) tiles.
__host__ __device__ inline int fwd_num_parts(int n, int num_splits, int n_max) {
  if (n <= 0) return 0;
  if (num_splits <= 1 || n_max <= 0) return 1;
  const long long p = (static_cast<long long>(n) * num_splits + n_max - 1) / n_max;
  return static_cast<int>(p < n ? p : n);
}

// Part `part` of `parts` balanced parts of [0, n): [floor(part n / parts),
// floor((part + 1) n / parts)); every part is non-empty when parts <= n.
__host__ __device__ inline void fwd_part_range(int n, int parts, int part, int* lo, int* hi) {
  if (parts <= 0) { *lo = *hi = 0; return; }
  *lo = static_cast<int>(static_cast<long long>(part) * n / parts);
  *hi = static_cast<int>(static_cast<long long>(part + 1) * n / parts);
}

// K/V tile count of row block m (kFwdRowsPerCta query rows).
__host__ __device__ inline int fwd_block_tiles(int m, int N, int N_k, int causal) {
  const int r0 = m * kFwdRowsPerCta;
  return fwd_kv_tile_end(r0, min(N, r0 + kFwdRowsPerCta), N_k, causal);
}

// Schedule of the persistent forward: G CTAs (at most one per SM) each run a
// fixed list of row blocks ("items"). Item (hb, rank) is the row block the
// per-block grid runs as blockIdx = (rank, hb % B, hb / B), i.e. linear block
// index hb * nm + rank, and covers rows of block fwd_m_block_of(rank).
//
// Without a causal mask every item has the same K/V range: items are dealt
// round robin (CTA c takes items c, c + G, ...), heads in order, so the CTAs
// running at any moment share a few heads' K/V through L2.
//
// Under a causal mask row block m visits about 2(m + 1) K/V tiles, so ranks q
// and nm-1-q of a head (blocks nm-1-q and q) form a pair with a constant total.
// Pairs are dealt round robin, longer block first. The last, partial round
// would leave most CTAs idle while a few run a whole pair; instead the R
// leftover pairs are chosen among the most balanced ones (q near the middle,
// whose two blocks are nearly equal) of the last heads and run as halves, one
// half per CTA: every CTA then finishes within about half a pair of the mean.
// Concretely, with P pairs, G = min(P, SMs), R = P mod G, T = ceil(R / BH)
// middle pairs are reserved in each of the last BHr = ceil(R / T) heads
// (R' = BHr T >= R of them); the other P - R' = kG - (R' - R) pairs are dealt
// round robin, which leaves R' - R CTAs one pair short; those run R' - R of the
// reserved pairs whole, and the other R are split over CTAs 0 .. 2R-1. The
// reserve is used when nm is even (true pairs), R > 0, T <= pairs per head and
// R + R' <= G; otherwise the leftover pairs are dealt like the others. When
// there are at most as many items as SMs, every item gets its own CTA.
struct FwdSched {
  int BH, nm;     // heads (batch x heads) and row blocks per head
  int G;          // CTAs
  int pairs;      // 0: items round robin; 1: causal pairs
  int ph;         // pairs per head, ceil(nm / 2) (odd nm: the middle block alone)
  long long bulk; // pairs dealt round robin
  int T, BHr;     // reserve: T middle pairs in each of the last BHr heads
  int Rw, Rs;     // reserved pairs run whole (CTAs G-Rw .. G-1) / as halves (CTAs 0 .. 2Rs-1)
};

__host__ __device__ inline FwdSched fwd_sched_make(int BH, int nm, int causal, int num_sms) {
  FwdSched s{};
  s.BH = BH;
  s.nm = nm;
  s.ph = (nm + 1) / 2;
  const long long items = static_cast<long long>(BH) * nm;
  if (num_sms < 1) num_sms = 1;
  if (!causal || items <= num_sms) {
    s.pairs = 0;
    s.G = static_cast<int>(items < num_sms ? items : num_sms);
    return s;
  }
  s.pairs = 1;
  const long long P = static_cast<long long>(BH) * s.ph;
  s.G = static_cast<int>(P < num_sms ? P : num_sms);
  s.bulk = P;
  const long long R = P % s.G;
  if (nm % 2 == 0 && R > 0) {
    const long long T = (R + BH - 1) / BH;
    if (T <= s.ph) {
      const long long BHr = (R + T - 1) / T;
      const long long Rp = BHr * T;
      if (R + Rp <= s.G) {
        s.T = static_cast<int>(T);
        s.BHr = static_cast<int>(BHr);
        s.Rw = static_cast<int>(Rp - R);
        s.Rs = static_cast<int>(R);
        s.bulk = P - Rp;
      }
    }
  }
  return s;
}

// Position of a CTA in its item list.
struct FwdCursor {
  long long j;  // items mode: item round; pairs mode: bulk pair round
  int half;     // 0 / 1: first / second block of the current pair
  int stage;    // pairs mode: 0 bulk, 1 reserved pairs, 2 done
};

// Pair (hb, q) of bulk pair b (heads in order; the reserved heads skip their
// T middle pairs).
__host__ __device__ inline void fwd_sched_bulk_pair(const FwdSched& s, long long b, int* hb, int* q) {
  const long long A = static_cast<long long>(s.BH - s.BHr) * s.ph;
  if (b < A) {
    *hb = static_cast<int>(b / s.ph);
    *q = static_cast<int>(b % s.ph);
  } else {
    const int w = s.ph - s.T;
    *hb = s.BH - s.BHr + static_cast<int>((b - A) / w);
    *q = static_cast<int>((b - A) % w);
  }
}

// Reserved pair r: head BH - BHr + r / T, pair ph - 1 - r % T.
__host__ __device__ inline void fwd_sched_reserved_pair(const FwdSched& s, int r, int* hb, int* q) {
  *hb = s.BH - s.BHr + r / s.T;
  *q = s.ph - 1 - r % s.T;
}

// Next item of CTA c: writes its head index hb and rank and advances the
// cursor; returns false when the CTA's list is exhausted.
__host__ __device__ inline bool fwd_sched_next(const FwdSched& s, int c, FwdCursor& cur, int* hb,
                                               int* rank) {
  const int nm = s.nm;
  if (!s.pairs) {
    const long long u = c + cur.j * s.G;
    if (u >= static_cast<long long>(s.BH) * nm) return false;
    ++cur.j;
    *hb = static_cast<int>(u / nm);
    *rank = static_cast<int>(u % nm);
    return true;
  }
  for (;;) {
    int q;
    if (cur.stage == 0) {
      const long long b = c + cur.j * s.G;
      if (b >= s.bulk) {
        cur.stage = 1;
        cur.half = 0;
        continue;
      }
      fwd_sched_bulk_pair(s, b, hb, &q);
    } else if (cur.stage == 1) {
      if (c >= s.G - s.Rw) {  // a reserved pair run whole
        fwd_sched_reserved_pair(s, c - (s.G - s.Rw), hb, &q);
      } else if (c < 2 * s.Rs) {  // half of a reserved pair
        if (cur.half > 0) return false;
        fwd_sched_reserved_pair(s, s.Rw + c / 2, hb, &q);
        cur.half = 1;
        cur.stage = 2;
        *rank = (c % 2 == 0) ? q : nm - 1 - q;
        return true;
      } else {
        return false;
      }
    } else {
      return false;
    }
    // A pair: rank q, then rank nm-1-q (none when they coincide).
    if (cur.half == 0) {
      cur.half = 1;
      if (nm - 1 - q == q) {
        cur.half = 0;
        if (cur.stage == 0) ++cur.j; else cur.stage = 2;
      }
      *rank = q;
      return true;
    }
    cur.half = 0;
    if (cur.stage == 0) ++cur.j; else cur.stage = 2;
    *rank = nm - 1 - q;
    return true;
  }
}

// Backward work mapping. dK and dV accumulate along the query direction, so
// their worker owns a K/V column block ("FlashAttention学习笔记(2)",
// Foward和backward中的thread block划分): one CTA per 128-key block, the column
// block varying fastest, visiting 128-row query tiles from the first one that
// reaches the diagonal. dQ accumulates along the key direction; its worker owns
// a 128-row query tile and visits the K/V tiles up to the diagonal, like the
// forward (causal: longest first).
__host__ __device__ inline int bwd_num_n_blocks(int N) { return ceil_div(N, kTileRows); }

__host__ __device__ inline int bwd_q_tile_begin(int n_block, int causal) {
  return causal ? n_block : 0;
}

__host__ __device__ inline int dq_num_m_blocks(int N) { return ceil_div(N, kTileRows); }

__host__ __device__ inline int dq_m_block_of(int block_x, int num_m_blocks, int causal) {
  return causal ? (num_m_blocks - 1 - block_x) : block_x;
}

// Argument block of the forward kernel (tensor maps travel separately as
// __grid_constant__ parameters).
struct FwdArgs {
  float* lse;         // [B*H, N] fp32, natural-log logsumexp
  int B, H, N;        // N: query length
  int Nk;             // key (and value) length
  int num_m_blocks;   // ceil(N / 256)
  float scale_log2;   // scale * log2(e)
  int* status;        // device status word
  int* tile_count;    // optional: K/V tiles loaded per row block, in per-block grid order (nullptr = off)
  unsigned long long timeout_ns;  // bound on every mbarrier wait
  int fault;          // 0 normally; 1 = the first V tile (of the first CTA, unsplit) never loads (failure-path test)
  int num_splits;     // K/V parts of the longest worker; <= 1: no split
  int kv_tiles_max;   // split mode: K/V tile count of the longest row block
  FwdSched sched;     // unsplit: the persistent kernel's item lists
  void* o;            // [B*H][N][d] 16-bit output (unsplit: the persistent kernel's row stores;
                      // split: written by the merging group)
  float* o_part;      // split mode: [num_splits][B*H][N][d] fp32 O / l of each part
  float* lse_part;    // split mode: [num_splits][B*H][N] fp32 logsumexp of each part (-inf: empty)
  int* part_done;     // split mode: [B*H][num_m_blocks][2] arrivals per row tile, zero on entry
};

// Argument block of the K/V-outer (FlashAttention-1 order) forward kernel.
struct Fa1Args {
  void* o;            // [B*H][N][d] 16-bit output
  float* lse;         // [B*H][N] natural-log logsumexp
  float* o_acc;       // workspace [B*H][N][d] fp32: running O_i (normalised)
  float* m_acc;       // workspace [B*H][N] fp32: running max (scaled, log2 units)
  float* l_acc;       // workspace [B*H][N] fp32: running sum
  int B, H, N;
  float scale_log2;
  int* status;
  unsigned long long timeout_ns;
};

struct BwdArgs {
  const float* l2_pad;    // L * log2(e), [B*H, n_pad] fp32 (0 past row N)
  const float* dsum_pad;  // D = rowsum(dO o O), [B*H, n_pad] fp32 (0 past row N)
  int n_pad;              // N rounded up to 128
  int B, H, N;            // N: query length
  int Nk;                 // key (and value) length
  float scale;            // softmax scale
  float scale_log2;       // scale * log2(e)
  int* status;
  unsigned long long timeout_ns;
  int fault;              // 0 normally; failure-path tests: 1 = the producer skips the
                          // first dO tile of the first dK/dV item, 2 = the first V tile
                          // of the first dQ item
  int* item_counter;      // persistent main launch: work items taken so far; the
                          // preprocessing pass zeroes it
  void* dq;               // persistent main launch: outputs written from TMEM by row,
  void* dk;               // [B*H][N][d] (dq) and [B*H][Nk][d] (dk, dv), 16-bit
  void* dv;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

template <int N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// ---------------------------------------------------------------------------
// Split-mode building blocks shared by the forward and backward kernels.
// ---------------------------------------------------------------------------

// CTA `cta` of a split launch -> (block, batch*head, part, parts). Blocks are
// ranked longest first by rank_info(k, &block, &tiles); rank k owns
// parts(tiles) * BH consecutive CTAs, heads varying fastest. One whole warp
// scans 32 ranks at a time (inclusive prefix sum of the CTA counts); lane 0 of
// the hit writes out[0..3]. Past the last part: all zero (no work).
template <class RankInfo>
__device__ __forceinline__ void split_locate(int cta, int M, int S, int n_max, int BH, int lane,
                                             RankInfo rank_info, int* out) {
  int base = 0;
  for (int k0 = 0; k0 < M; k0 += 32) {
    const int k = k0 + lane;
    int blk = 0, p = 0;
    if (k < M) {
      int tiles = 0;
      rank_info(k, &blk, &tiles);
      p = fwd_num_parts(tiles, S, n_max);
    }
    const int c = p * BH;
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, k < M && cta < base + incl);
    if (hit != 0u) {
      if (lane == __ffs(hit) - 1) {
        const int r = cta - (base + incl - c);
        out[0] = blk;
        out[1] = r % BH;
        out[2] = r / BH;
        out[3] = p;
      }
      return;
    }
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) out[0] = out[1] = out[2] = out[3] = 0;
}

// CTAs of a split launch: sum over the ranks of their part counts, times BH.
template <class TilesOf>
inline long long split_ctas(int M, int S, int n_max, int BH, TilesOf tiles_of) {
  long long total = 0;
  for (int k = 0; k < M; ++k) total += fwd_num_parts(tiles_of(k), S, n_max);
  return total * BH;
}

// One warp's 32 TMEM lanes (rows) x D fp32 columns, times `mul` (per lane),
// to rows [0, rows_valid) of a row-major fp32 matrix starting at dst. Each 32-
// column block passes through the warp's 4 KiB shared slice (16-byte chunks
// XOR-swizzled by row) so that every global store is a whole 128-byte row
// segment. Warp-collective: the whole warp calls it.
template <int D>
__device__ __forceinline__ void tmem_rows_to_f32(uint32_t t_src, float mul, float* dst,
                                                 int rows_valid, int lane, float4* slice) {
  const int sub = lane >> 3, seg = lane & 7;
#pragma unroll 1
  for (int c = 0; c < D; c += 32) {
    uint32_t x[32];
    tmem_ld_32x32b_x32(t_src + c, x);
    tmem_wait_ld();
    reg_fence(x);
#pragma unroll
    for (int k = 0; k < 8; ++k)
      slice[lane * 8 + (k ^ (lane & 7))] =
          make_float4(__uint_as_float(x[4 * k]) * mul, __uint_as_float(x[4 * k + 1]) * mul,
                      __uint_as_float(x[4 * k + 2]) * mul, __uint_as_float(x[4 * k + 3]) * mul);
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int rr = 4 * i + sub;
      const float4 val = slice[rr * 8 + (seg ^ (rr & 7))];
      if (rr < rows_valid) reinterpret_cast<float4*>(dst + static_cast<size_t>(rr) * D + c)[seg] = val;
    }
    __syncwarp();
  }
}

// Arrival of a 128-thread group on a part counter: every thread's stores are
// made visible device-wide first, one thread adds 1, and the group learns
// whether its add completed the count (the group that then merges). Nobody
// waits on another CTA. Every thread of the group must call it.
__device__ __forceinline__ bool arrive_last(int* counter, int parts, int bar_id, int* flag) {
  __threadfence();
  named_bar_sync(bar_id, 128);
  if ((threadIdx.x & 127) == 0) *flag = atomicAdd(counter, 1) == parts - 1;
  named_bar_sync(bar_id, 128);
  const bool last = *flag != 0;
  if (last) __threadfence();
  return last;
}

}  // namespace fa2
