// attn_splitkv.cu -- merge of split-KV partial results into O and lse.
//
// Each key slice s of a query row left an unnormalised output a_s, a reference maximum m_s (log2
// units) and its fp32 row sum l_s.  The merge is the block merge
// of the CS336 GPU/attention notes, "Online softmax 回顾", applied to all slices at once:
//   M = max_s m_s,  w_s = 2^(m_s - M),  O = sum_s w_s a_s / sum_s w_s l_s,
//   lse = (M + log2 sum_s w_s l_s) * ln 2.
#include <cuda_bf16.h>

#include <cmath>

#include "attn_params.h"
#include "sm103_ptx.cuh"

namespace attn {
namespace {

template <int D>
__global__ void __launch_bounds__(256) splitkv_combine_kernel(const float* __restrict__ part_o,
                                                              const float* __restrict__ stat,
                                                              __nv_bfloat16* __restrict__ o,
                                                              float* __restrict__ lse,
                                                              long long rows, int S) {
  constexpr int kPer = D / 32;  // columns per lane
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int lane = threadIdx.x & 31;
  const long long plane = static_cast<long long>(S) * rows;
  float M = -INFINITY;
  for (int s = 0; s < S; ++s) M = fmaxf(M, stat[s * rows + row]);
  float acc[kPer];
  #pragma unroll
  for (int i = 0; i < kPer; ++i) acc[i] = 0.f;
  float le = 0.f;
  for (int s = 0; s < S; ++s) {
    const long long slot = s * rows + row;
    const float m = stat[slot];
    if (m == -INFINITY) continue;  // this slice held no key of the row
    const float w = ex2_approx(m - M);
    le += w * stat[plane + slot];
    const float* src = part_o + slot * D + lane * kPer;
    if constexpr (kPer == 4) {
      const float4 x = *reinterpret_cast<const float4*>(src);
      acc[0] += w * x.x; acc[1] += w * x.y; acc[2] += w * x.z; acc[3] += w * x.w;
    } else {
      const float2 x = *reinterpret_cast<const float2*>(src);
      acc[0] += w * x.x; acc[1] += w * x.y;
    }
  }
  const float inv = 1.f / le;
  __nv_bfloat16* dst = o + row * D + lane * kPer;
  if constexpr (kPer == 4) {
    *reinterpret_cast<uint2*>(dst) =
        make_uint2(pack_bf16x2(acc[0] * inv, acc[1] * inv), pack_bf16x2(acc[2] * inv, acc[3] * inv));
  } else {
    *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
  }
  if (lane == 0) lse[row] = (M + log2f(le)) * 0.69314718055994530942f;
}

}  // namespace

cudaError_t launch_splitkv_combine(int d, const float* part_o, const float* part_stat, void* o,
                                   float* lse, long long rows, int splits, cudaStream_t stream) {
  const long long blocks = (rows + 7) / 8;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(o);
  if (d == 64)
    splitkv_combine_kernel<64><<<static_cast<int>(blocks), 256, 0, stream>>>(part_o, part_stat, out,
                                                                            lse, rows, splits);
  else
    splitkv_combine_kernel<128><<<static_cast<int>(blocks), 256, 0, stream>>>(part_o, part_stat, out,
                                                                             lse, rows, splits);
  return cudaGetLastError();
}

}  // namespace attn
