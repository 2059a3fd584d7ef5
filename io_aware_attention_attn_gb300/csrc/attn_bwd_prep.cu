// attn_bwd_prep.cu -- per-row inputs of the backward tile kernels.
//
// D_i = dO_i . O_i (the softmax-gradient term: sum_k P_ik dP_ik = dO_i . O_i because
// sum_k P_ik V_k = O_i) and lse_i * log2(e), written negated to [B*H][n_pad] fp32 planes (the
// tile kernels add them with packed adds and fused multiply-adds); rows past N hold -D = 0 and
// -lse2 = -inf, so that a padded query row rebuilds P = 2^(-inf) = 0.
#include <cuda_bf16.h>

#include <cmath>

#include "attn_bwd.h"

namespace attn {
namespace {

template <int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const __nv_bfloat16* __restrict__ o,
                                                       const __nv_bfloat16* __restrict__ dout,
                                                       const float* __restrict__ lse,
                                                       float* __restrict__ nlse2,
                                                       float* __restrict__ nd, long long rows_pad,
                                                       int N, int n_pad) {
  constexpr int kPer = D / 32;  // elements per lane
  const long long w = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (w >= rows_pad) return;
  const int lane = threadIdx.x & 31;
  const long long z = w / n_pad;
  const int row = static_cast<int>(w % n_pad);
  if (row >= N) {
    if (lane == 0) {
      nlse2[w] = -INFINITY;
      nd[w] = 0.f;
    }
    return;
  }
  const size_t off = (static_cast<size_t>(z) * N + row) * D + lane * kPer;
  float acc = 0.f;
  if constexpr (kPer == 4) {
    const uint2 a = *reinterpret_cast<const uint2*>(o + off);
    const uint2 b = *reinterpret_cast<const uint2*>(dout + off);
    const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
    #pragma unroll
    for (int q = 0; q < 2; ++q) {
      const float2 x = __bfloat1622float2(a2[q]), y = __bfloat1622float2(b2[q]);
      acc = fmaf(x.x, y.x, acc);
      acc = fmaf(x.y, y.y, acc);
    }
  } else {
    const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(o + off));
    const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(dout + off));
    acc = fmaf(x.x, y.x, x.y * y.y);
  }
  #pragma unroll
  for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
  if (lane == 0) {
    nd[w] = -acc;
    nlse2[w] = -lse[static_cast<size_t>(z) * N + row] * 1.4426950408889634f;
  }
}

// Packed batches: block = one 128-row tile slot of one head (see bwd_locate_tile); its rows go
// to plane rows 128 * slot + r, rows past the end of the sequence get the padding values.
template <int D>
__global__ void __launch_bounds__(256) bwd_prep_varlen_kernel(
    const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
    const float* __restrict__ lse, float* __restrict__ nlse2, float* __restrict__ nd,
    const int32_t* __restrict__ cu, int n_seqs, int H, int T, int n_slots) {
  constexpr int kPer = D / 32;
  __shared__ int info[3];
  const int z = blockIdx.x % H, slot = blockIdx.x / H;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0) {
    int start, len, tile, base;
    bwd_locate_tile(cu, n_seqs, T, slot, lane, start, len, tile, base);
    if (lane == 0) {
      info[0] = start;
      info[1] = len;
      info[2] = tile;
    }
  }
  __syncthreads();
  const int start = info[0], len = info[1], tile = info[2];
  if (tile < 0) return;  // past the last tile: these plane rows are never read
  const size_t prow = static_cast<size_t>(z) * (static_cast<size_t>(n_slots) * kBM) +
                      static_cast<size_t>(slot) * kBM;
  for (int r = warp * 16; r < warp * 16 + 16; ++r) {
    const int in_seq = tile * kBM + r;
    if (in_seq >= len) {
      if (lane == 0) {
        nlse2[prow + r] = -INFINITY;
        nd[prow + r] = 0.f;
      }
      continue;
    }
    const size_t row = static_cast<size_t>(z) * T + start + in_seq;
    const size_t off = row * D + lane * kPer;
    float acc = 0.f;
    if constexpr (kPer == 4) {
      const uint2 a = *reinterpret_cast<const uint2*>(o + off);
      const uint2 b = *reinterpret_cast<const uint2*>(dout + off);
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
      const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
      #pragma unroll
      for (int q = 0; q < 2; ++q) {
        const float2 x = __bfloat1622float2(a2[q]), y = __bfloat1622float2(b2[q]);
        acc = fmaf(x.x, y.x, acc);
        acc = fmaf(x.y, y.y, acc);
      }
    } else {
      const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(o + off));
      const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(dout + off));
      acc = fmaf(x.x, y.x, x.y * y.y);
    }
    #pragma unroll
    for (int sft = 16; sft > 0; sft >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, sft);
    if (lane == 0) {
      nd[prow + r] = -acc;
      nlse2[prow + r] = -lse[row] * 1.4426950408889634f;
    }
  }
}

}  // namespace

cudaError_t launch_bwd_prep_varlen(const void* o, const void* dout, const float* lse,
                                   float* nlse2, float* nd, const int32_t* cu_seqlens, int n_seqs,
                                   int H, int T, int n_slots, int d, cudaStream_t stream) {
  const long long blocks = static_cast<long long>(H) * n_slots;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
  const auto* ob = static_cast<const __nv_bfloat16*>(o);
  const auto* db = static_cast<const __nv_bfloat16*>(dout);
  if (d == 64)
    bwd_prep_varlen_kernel<64><<<static_cast<int>(blocks), 256, 0, stream>>>(
        ob, db, lse, nlse2, nd, cu_seqlens, n_seqs, H, T, n_slots);
  else
    bwd_prep_varlen_kernel<128><<<static_cast<int>(blocks), 256, 0, stream>>>(
        ob, db, lse, nlse2, nd, cu_seqlens, n_seqs, H, T, n_slots);
  return cudaGetLastError();
}

cudaError_t launch_bwd_prep(const void* o, const void* dout, const float* lse, float* nlse2,
                            float* nd, int BH, int N, int n_pad, int d, cudaStream_t stream) {
  const long long rows_pad = static_cast<long long>(BH) * n_pad;
  const long long blocks = (rows_pad + 7) / 8;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
  const auto* ob = static_cast<const __nv_bfloat16*>(o);
  const auto* db = static_cast<const __nv_bfloat16*>(dout);
  if (d == 64)
    bwd_prep_kernel<64><<<static_cast<int>(blocks), 256, 0, stream>>>(ob, db, lse, nlse2, nd,
                                                                      rows_pad, N, n_pad);
  else
    bwd_prep_kernel<128><<<static_cast<int>(blocks), 256, 0, stream>>>(ob, db, lse, nlse2, nd,
                                                                       rows_pad, N, n_pad);
  return cudaGetLastError();
}

}  // namespace attn
