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

// One row of O and of dO is D/8 chunks of 16 bytes.  prep_dot is a lane's share of dO . O over
// its chunk; prep_reduce sums the shares of the D/8 lanes that hold one row.  Both passes below
// use them, in the same order, so a packed batch of one sequence reproduces the dense planes bit
// for bit.
template <int D>
__device__ __forceinline__ float prep_dot(const uint4& a, const uint4& b) {
  const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
  const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
  float acc = 0.f;
  #pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float2 x = __bfloat1622float2(a2[q]), y = __bfloat1622float2(b2[q]);
    acc = fmaf(x.x, y.x, acc);
    acc = fmaf(x.y, y.y, acc);
  }
  return acc;
}
template <int D>
__device__ __forceinline__ float prep_reduce(float acc) {
  #pragma unroll
  for (int sft = D / 16; sft > 0; sft >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, sft);
  return acc;
}

// Dense batches: each warp takes 8 consecutive plane rows (never across heads: n_pad is a
// multiple of 128).  A row of O and of dO is D/8 chunks of 16 bytes, one per lane, so a warp's
// load instruction covers 32 / (D/8) rows and every lane has 8 / (32 / (D/8)) loads of each
// tensor in flight before it reduces.
template <int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const __nv_bfloat16* __restrict__ o,
                                                       const __nv_bfloat16* __restrict__ dout,
                                                       const float* __restrict__ lse,
                                                       float* __restrict__ nlse2,
                                                       float* __restrict__ nd, long long rows_pad,
                                                       int N, int n_pad) {
  constexpr int kLanes = D / 8;          // 16-byte chunks per row
  constexpr int kRowsPer = 32 / kLanes;  // rows per warp-wide load
  constexpr int kIters = 8 / kRowsPer;
  const long long w0 = (static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5)) * 8;
  if (w0 >= rows_pad) return;
  const int lane = threadIdx.x & 31;
  const int sub = lane / kLanes, chunk = lane % kLanes;
  uint4 a[kIters], b[kIters];
  #pragma unroll
  for (int it = 0; it < kIters; ++it) {
    const long long w = w0 + it * kRowsPer + sub;
    const long long z = w / n_pad;
    const int row = static_cast<int>(w % n_pad);
    a[it] = make_uint4(0u, 0u, 0u, 0u);
    b[it] = make_uint4(0u, 0u, 0u, 0u);
    if (w < rows_pad && row < N) {
      const size_t off = (static_cast<size_t>(z) * N + row) * D + chunk * 8;
      a[it] = __ldg(reinterpret_cast<const uint4*>(o + off));
      b[it] = __ldg(reinterpret_cast<const uint4*>(dout + off));
    }
  }
  #pragma unroll
  for (int it = 0; it < kIters; ++it) {
    const float acc = prep_reduce<D>(prep_dot<D>(a[it], b[it]));
    const long long w = w0 + it * kRowsPer + sub;
    if (chunk == 0 && w < rows_pad) {
      const long long z = w / n_pad;
      const int row = static_cast<int>(w % n_pad);
      if (row < N) {
        nd[w] = -acc;
        nlse2[w] = -lse[static_cast<size_t>(z) * N + row] * 1.4426950408889634f;
      } else {
        nlse2[w] = -INFINITY;
        nd[w] = 0.f;
      }
    }
  }
}

// Packed batches: block = one 128-row tile slot of one head (see bwd_locate_tile); its rows go
// to plane rows 128 * slot + r, rows past the end of the sequence get the padding values.
template <int D>
__global__ void __launch_bounds__(256) bwd_prep_varlen_kernel(
    const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
    const float* __restrict__ lse, float* __restrict__ nlse2, float* __restrict__ nd,
    const int32_t* __restrict__ cu, int n_seqs, int H, int T, int n_slots) {
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
  // each warp takes 16 rows of the tile, 32 / (D/8) rows per load as in the dense pass
  constexpr int kLanes = D / 8, kRowsPer = 32 / kLanes;
  const int sub = lane / kLanes, chunk = lane % kLanes;
  for (int r0 = warp * 16; r0 < warp * 16 + 16; r0 += kRowsPer) {
    const int r = r0 + sub;
    const int in_seq = tile * kBM + r;
    const bool valid = in_seq < len;
    const size_t row = static_cast<size_t>(z) * T + start + (valid ? in_seq : 0);
    uint4 a = make_uint4(0u, 0u, 0u, 0u), b = make_uint4(0u, 0u, 0u, 0u);
    if (valid) {
      a = __ldg(reinterpret_cast<const uint4*>(o + row * D + chunk * 8));
      b = __ldg(reinterpret_cast<const uint4*>(dout + row * D + chunk * 8));
    }
    const float acc = prep_reduce<D>(prep_dot<D>(a, b));
    if (chunk == 0) {
      if (valid) {
        nd[prow + r] = -acc;
        nlse2[prow + r] = -lse[row] * 1.4426950408889634f;
      } else {
        nlse2[prow + r] = -INFINITY;
        nd[prow + r] = 0.f;
      }
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
  const long long blocks = (rows_pad + 63) / 64;  // 8 warps of 8 rows
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
