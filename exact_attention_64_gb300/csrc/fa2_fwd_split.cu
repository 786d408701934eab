// K/V-split forward: the merge pass ("大猿搬砖简记", thread-block section: the
// K/V range of a worker may be split across blocks when the SMs cannot be
// filled otherwise, and the blocks' partial results must then be combined to
// recover the global softmax).
//
// Each part s of a row holds O_s = (sum over its keys of exp(S - m_s) V) / l_s
// and its logsumexp lse_s = m_s + ln l_s (-inf for a part with no keys). The
// merge is the online-softmax rule applied to whole parts:
//   L = ln sum_s exp(lse_s),   O = sum_s exp(lse_s - L) O_s.
#include <cuda_fp16.h>
#include "fa2_common.cuh"

namespace fa2 {

constexpr float kLog2eSplit = 1.4426950408889634f;
constexpr float kLn2Split = 0.6931471805599453f;

// One warp per row; each lane owns D/32 consecutive columns.
template <int D, bool BF16>
__global__ void __launch_bounds__(256)
    fa2_fwd_combine_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part,
                           uint16_t* __restrict__ o, float* __restrict__ lse, int S, long long rows) {
  constexpr int EPL = D / 32;
  const int lane = threadIdx.x & 31;
  const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  for (long long row = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       row < rows; row += warps) {
    float m = -INFINITY;
    for (int s = 0; s < S; ++s) m = fmaxf(m, lse_part[s * rows + row]);
    float acc[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
    float L = -INFINITY;
    if (m != -INFINITY) {
      float tot = 0.f;
      for (int s = 0; s < S; ++s) {
        const float ls = lse_part[s * rows + row];
        const float w = ex2_approx((ls - m) * kLog2eSplit);  // 0 for an empty part
        tot += w;
        const float* src = o_part + (static_cast<size_t>(s) * rows + row) * D + lane * EPL;
        if constexpr (EPL == 4) {
          const float4 x = *reinterpret_cast<const float4*>(src);
          acc[0] = fmaf(w, x.x, acc[0]); acc[1] = fmaf(w, x.y, acc[1]);
          acc[2] = fmaf(w, x.z, acc[2]); acc[3] = fmaf(w, x.w, acc[3]);
        } else {
          const float2 x = *reinterpret_cast<const float2*>(src);
          acc[0] = fmaf(w, x.x, acc[0]); acc[1] = fmaf(w, x.y, acc[1]);
        }
      }
      const float inv = 1.f / tot;
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[e] *= inv;
      L = m + lg2_approx(tot) * kLn2Split;
    }
    uint16_t* dst = o + row * D + lane * EPL;
    if constexpr (EPL == 4) {
      *reinterpret_cast<uint2*>(dst) = make_uint2(pack_x2<BF16>(acc[0], acc[1]), pack_x2<BF16>(acc[2], acc[3]));
    } else {
      *reinterpret_cast<uint32_t*>(dst) = pack_x2<BF16>(acc[0], acc[1]);
    }
    if (lane == 0) lse[row] = L;
  }
}

cudaError_t launch_fwd_combine(int d, bool bf16, const float* o_part, const float* lse_part, void* o,
                               float* lse, int S, long long rows, int num_sms, cudaStream_t stream) {
  long long blocks = (rows + 7) / 8;
  const long long cap = static_cast<long long>(num_sms > 0 ? num_sms : 148) * 16;
  if (blocks > cap) blocks = cap;
  const dim3 grid(static_cast<unsigned>(blocks));
  uint16_t* o16 = static_cast<uint16_t*>(o);
  if (d == 128 && bf16) fa2_fwd_combine_kernel<128, true><<<grid, 256, 0, stream>>>(o_part, lse_part, o16, lse, S, rows);
  else if (d == 128) fa2_fwd_combine_kernel<128, false><<<grid, 256, 0, stream>>>(o_part, lse_part, o16, lse, S, rows);
  else if (bf16) fa2_fwd_combine_kernel<64, true><<<grid, 256, 0, stream>>>(o_part, lse_part, o16, lse, S, rows);
  else fa2_fwd_combine_kernel<64, false><<<grid, 256, 0, stream>>>(o_part, lse_part, o16, lse, S, rows);
  return cudaGetLastError();
}

}  // namespace fa2
