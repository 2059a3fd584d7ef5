// attn_fp8.cu -- per-tile E4M3 quantization and the launcher of the FP8 forward kernel.
//
// Quantization of a bf16 tensor [B*H][N][d], per tile of 128 rows of a head (CS336 Lecture 5
// notes, section 3.1: E4M3 for forward activations, with per-tile scaling):
//   scale = amax / 448 in fp32 (1 for an all-zero tile), code = E4M3 round-to-nearest-even of
//   x / scale (fp32 IEEE division), saturating at +-448.
// Codes are written row-major [B*H][N][d], or transposed [B*H][d][Npad] (Npad = N rounded up to
// 128, padding codes 0) for the V operand of the FP8 forward.
#include <atomic>

#include <cuda_bf16.h>

#include "attn_fwd_fp8_kernel.cuh"

namespace attn {
namespace {

constexpr int kQuantThreads = 256;

template <int D>
__global__ void __launch_bounds__(kQuantThreads) quantize_fp8_kernel(
    const __nv_bfloat16* __restrict__ x, uint8_t* __restrict__ codes, float* __restrict__ scales,
    int N, int n_tiles, int n_pad, int transpose) {
  constexpr int kPer = D / 2;  // elements per thread: row = tid / 2, half = tid % 2
  __shared__ float red[kQuantThreads / 32];
  __shared__ float s_scale;
  __shared__ __align__(16) uint8_t tile_t[D][kBM + 16];  // transposed codes (transpose only)
  const int z = blockIdx.x / n_tiles;
  const int t = blockIdx.x % n_tiles;
  const int r = threadIdx.x >> 1;
  const int c0 = (threadIdx.x & 1) * kPer;
  const int row = t * kBM + r;
  const bool valid = row < N;
  float v[kPer];
  const __nv_bfloat16* src = x + (static_cast<size_t>(z) * N + (valid ? row : 0)) * D + c0;
  #pragma unroll
  for (int i = 0; i < kPer / 8; ++i) {
    uint4 w = valid ? reinterpret_cast<const uint4*>(src)[i] : make_uint4(0, 0, 0, 0);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
    #pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 f = __bfloat1622float2(h[q]);
      v[8 * i + 2 * q] = f.x;
      v[8 * i + 2 * q + 1] = f.y;
    }
  }
  float amax = 0.f;
  #pragma unroll
  for (int i = 0; i < kPer; ++i) amax = fmaxf(amax, fabsf(v[i]));
  #pragma unroll
  for (int s = 16; s > 0; s >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, s));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = 0.f;
    for (int w = 0; w < kQuantThreads / 32; ++w) m = fmaxf(m, red[w]);
    const float sc = m > 0.f ? __fdiv_rn(m, 448.f) : 1.f;
    s_scale = sc;
    scales[blockIdx.x] = sc;
  }
  __syncthreads();
  const float sc = s_scale;
  uint32_t w32[kPer / 4];
  #pragma unroll
  for (int i = 0; i < kPer / 4; ++i)
    w32[i] = static_cast<uint32_t>(pack_e4m3x2(__fdiv_rn(v[4 * i], sc), __fdiv_rn(v[4 * i + 1], sc))) |
             (static_cast<uint32_t>(pack_e4m3x2(__fdiv_rn(v[4 * i + 2], sc),
                                                __fdiv_rn(v[4 * i + 3], sc)))
              << 16);
  if (!transpose) {
    if (valid) {
      uint4* dst = reinterpret_cast<uint4*>(codes + (static_cast<size_t>(z) * N + row) * D + c0);
      #pragma unroll
      for (int i = 0; i < kPer / 16; ++i)
        dst[i] = make_uint4(w32[4 * i], w32[4 * i + 1], w32[4 * i + 2], w32[4 * i + 3]);
    }
    return;
  }
  // transposed: stage [d][row] in shared memory, then write 128-byte rows of [d][Npad]
  #pragma unroll
  for (int i = 0; i < kPer; ++i) tile_t[c0 + i][r] = static_cast<uint8_t>(w32[i >> 2] >> (8 * (i & 3)));
  __syncthreads();
  for (int e = threadIdx.x; e < D * (kBM / 16); e += kQuantThreads) {
    const int c = e / (kBM / 16), seg = e % (kBM / 16);
    const uint4 val = *reinterpret_cast<const uint4*>(&tile_t[c][seg * 16]);
    *reinterpret_cast<uint4*>(codes + (static_cast<size_t>(z) * D + c) * n_pad + t * kBM +
                              seg * 16) = val;
  }
}

}  // namespace

cudaError_t launch_quantize_fp8(const void* x, void* codes, float* scales, int BH, int N, int d,
                                bool transpose, cudaStream_t stream) {
  const int n_tiles = (N + kBM - 1) / kBM;
  const long long blocks = static_cast<long long>(BH) * n_tiles;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
  const auto* xb = static_cast<const __nv_bfloat16*>(x);
  auto* cb = static_cast<uint8_t*>(codes);
  if (d == 64)
    quantize_fp8_kernel<64><<<static_cast<int>(blocks), kQuantThreads, 0, stream>>>(
        xb, cb, scales, N, n_tiles, n_tiles * kBM, transpose ? 1 : 0);
  else
    quantize_fp8_kernel<128><<<static_cast<int>(blocks), kQuantThreads, 0, stream>>>(
        xb, cb, scales, N, n_tiles, n_tiles * kBM, transpose ? 1 : 0);
  return cudaGetLastError();
}

namespace {

template <bool CAUSAL>
cudaError_t launch_fp8(const Fp8Params& p, cudaStream_t stream) {
  auto* kernel = attn_fwd_fp8_kernel<CAUSAL>;
  constexpr int kSmem = Fp8Layout::kDynBytes;
  static std::atomic<uint64_t> attr_done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_done.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    attr_done.fetch_or(bit, std::memory_order_acq_rel);
  }
  kernel<<<p.n_qt * p.B * p.H, kFp8Threads, kSmem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_fp8(const Fp8Params& p, bool causal, cudaStream_t stream) {
  return causal ? launch_fp8<true>(p, stream) : launch_fp8<false>(p, stream);
}

}  // namespace attn
