// Pieces shared by the backward kernels: tile loads, the MMA forms of the
// backward products, the exponentials of P^T and the 16-bit epilogue staging.
#pragma once
#include "fa2_common.cuh"

namespace fa2 {

constexpr float kLog2e = 1.4426950408889634f;

// A 128-row tile of a 16-bit [rows][d] tensor in shared memory: d/64 slabs of
// 128 rows x 128 bytes, 128-byte swizzled (the TMA box layout).
template <int D>
struct BwdTile {
  static constexpr int SLAB_BYTES = kTileRows * 128;
  static constexpr int TILE_BYTES = kTileRows * D * 2;
};

template <int D>
__device__ __forceinline__ void load_tile(uint8_t* dst, const CUtensorMap* map, uint64_t* bar,
                                          int row, int bh) {
#pragma unroll
  for (int s = 0; s < D / 64; ++s)
    tma_load_3d(dst + s * BwdTile<D>::SLAB_BYTES, map, bar, s * 64, row, bh);
}

// D[tmem] = A B^T over the head dimension: M=128 rows of A, N=128 rows of B,
// K=d. Both tiles K-major, 128-byte swizzled (the forward's Q K^T form).
// Like every MMA helper here, issued by a converged warp (one lane elected).
template <int D, bool BF16>
__device__ __forceinline__ void mma_rows_x_rows(uint32_t d_tmem, uint32_t a_smem, uint32_t b_smem) {
  constexpr uint32_t idesc = make_idesc_f16(128, 128, BF16, false, false);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = (kk / 4) * BwdTile<D>::SLAB_BYTES + (kk % 4) * 32;
    const uint64_t ad = make_sdesc_sw128(a_smem + off, 16, 1024);
    const uint64_t bd = make_sdesc_sw128(b_smem + off, 16, 1024);
    umma_ss_warp(d_tmem, ad, bd, idesc, kk > 0 ? 1u : 0u);
  }
}

// D[tmem] (+)= A[tmem] X with A = 128 x 128 16-bit pairs in TMEM and X a
// 128-row tile [row][d] in shared memory (MN-major for this product; the
// forward's P V form). a_col(kk) gives the TMEM column of A's 16-row block kk.
template <int D, bool BF16, typename ACol>
__device__ __forceinline__ void mma_tmem_x_tile(uint32_t d_tmem, ACol a_col, uint32_t x_smem,
                                                bool accumulate) {
  constexpr uint32_t idesc = make_idesc_f16(128, D, BF16, false, true);
#pragma unroll
  for (int kk = 0; kk < kTileRows / 16; ++kk) {
    const uint64_t bd = make_sdesc_sw128(x_smem + kk * 2048, BwdTile<D>::SLAB_BYTES, 1024);
    const uint32_t acc = (accumulate || kk > 0) ? 1u : 0u;
    umma_ts_warp(d_tmem, a_col(kk), bd, idesc, acc);
  }
}

// P^T for 32 query columns q_first.. of key row kg (dK/dV workers):
// p[c] = exp2(S^T[c] * scale*log2e + nl_cols[c]), nl_cols = -(L*log2e) in registers. With MASK, pairs outside the
// sequence or with key > query (causal) get 0. MASK is a template parameter so
// that tiles off the diagonal run a loop with no per-element branches, which
// would otherwise keep the exponentials from overlapping.
template <bool MASK, bool CAUSAL>
__device__ __forceinline__ void dkdv_p_cols(const uint32_t (&sv)[32], const float* nl_cols, float sl2,
                                            int kg, int q_first, int Nq, int Nk, float* p) {
#pragma unroll
  for (int c = 0; c < 32; c += 2) {
    const float2 x = f2_fma(make_float2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])),
                            make_float2(sl2, sl2), make_float2(nl_cols[c], nl_cols[c + 1]));
    float p0 = ex2_approx(x.x), p1 = ex2_approx(x.y);
    if constexpr (MASK) {
      const int q0 = q_first + c;
      p0 = (kg >= Nk || q0 >= Nq || (CAUSAL && kg > q0)) ? 0.f : p0;
      p1 = (kg >= Nk || q0 + 1 >= Nq || (CAUSAL && kg > q0 + 1)) ? 0.f : p1;
    }
    p[c] = p0;
    p[c + 1] = p1;
  }
}

// dS for 64 key columns of query row my_row (dQ workers), packed to 16-bit
// pairs: dS = P o (dP - D) with P = exp2(S * scale*log2e - L*log2e). With MASK,
// keys at or past lim and rows past the sequence get P = 0. Column pairs use
// packed fp32 (f32x2) arithmetic.
template <bool MASK, bool BF16>
__device__ __forceinline__ void dq_ds_cols(const uint32_t (&s)[64], const uint32_t (&dp)[64], float sl2,
                                           float l2, float dsum, int kc0, int lim, bool row_ok,
                                           uint32_t (&dsp)[32]) {
  const float2 sl2x2 = make_float2(sl2, sl2), nl2 = make_float2(-l2, -l2);
  const float2 dsum2 = make_float2(dsum, dsum);
#pragma unroll
  for (int c = 0; c < 64; c += 2) {
    const float2 x = f2_fma(make_float2(__uint_as_float(s[c]), __uint_as_float(s[c + 1])), sl2x2, nl2);
    float p0 = ex2_approx(x.x), p1 = ex2_approx(x.y);
    if constexpr (MASK) {
      p0 = (!row_ok || kc0 + c >= lim) ? 0.f : p0;
      p1 = (!row_ok || kc0 + c + 1 >= lim) ? 0.f : p1;
    }
    const float2 ds = f2_mul(make_float2(p0, p1),
                             f2_sub(make_float2(__uint_as_float(dp[c]), __uint_as_float(dp[c + 1])), dsum2));
    dsp[c / 2] = pack_x2<BF16>(ds.x, ds.y);
  }
}

// Stage a 128 x d fp32 TMEM accumulator (this thread's lane = row r) as 16-bit
// rows, multiplied by mul, into a 128-byte-swizzled tile in shared memory.
template <int D, bool BF16>
__device__ __forceinline__ void stage_rows(uint8_t* stage, uint32_t t_src, int r, float mul) {
#pragma unroll
  for (int c = 0; c < D; c += 32) {
    uint32_t x[32];
    tmem_ld_32x32b_x32(t_src + c, x);
    tmem_wait_ld();
    reg_fence(x);
    const int slab = c / 64, chunk0 = (c % 64) / 8;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint4 val;
      val.x = pack_x2<BF16>(__uint_as_float(x[8 * k + 0]) * mul, __uint_as_float(x[8 * k + 1]) * mul);
      val.y = pack_x2<BF16>(__uint_as_float(x[8 * k + 2]) * mul, __uint_as_float(x[8 * k + 3]) * mul);
      val.z = pack_x2<BF16>(__uint_as_float(x[8 * k + 4]) * mul, __uint_as_float(x[8 * k + 5]) * mul);
      val.w = pack_x2<BF16>(__uint_as_float(x[8 * k + 6]) * mul, __uint_as_float(x[8 * k + 7]) * mul);
      *reinterpret_cast<uint4*>(stage + slab * BwdTile<D>::SLAB_BYTES + r * 128 +
                                (((chunk0 + k) ^ (r & 7)) * 16)) = val;
    }
  }
}


}  // namespace fa2
