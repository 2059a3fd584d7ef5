// attn_fp8.cu -- per-tile E4M3 quantization and the launcher of the FP8 forward kernel.
//
// Quantization of a bf16 tensor [B*H][N][d], per tile of 128 rows of a head (CS336 Lecture 5
// notes, section 3.1: E4M3 for forward activations, with per-tile scaling):
//   scale = amax / 448 in fp32 (1 for an all-zero tile), code = E4M3 round-to-nearest-even of
//   x / scale rounded to nearest fp32 (the IEEE quotient), saturating at +-448.
// Codes are written row-major [B*H][N][d], or transposed [B*H][d][Npad] (Npad = N rounded up to
// 128, padding codes 0) for the V operand of the FP8 forward.
#include <atomic>

#include <cuda_bf16.h>

#include "attn_fwd_fp8_kernel.cuh"

namespace attn {
namespace {

constexpr int kQuantThreads = 256;

// x / sc rounded to nearest fp32, from rc = RN(1 / sc) and one remainder correction: with
// q0 = RN(x rc), the remainder x - sc q0 is exact under a fused multiply-add and RN(q0 + rem rc)
// is the rounded quotient (the correction step of FMA-based division: P. Markstein, "Computation
// of elementary functions on the IBM RISC System/6000 processor", IBM J. Res. Develop. 34(1),
// 1990).  The sign comes from x, so -0 stays -0.  For x below fp32's normal range the exact
// remainder can fall under the subnormal spacing and the quotient lose its last bit, but such
// quotients code to 0 either way.  Used for the scales of tiles whose reciprocal is far from the
// fp32 range's ends; attn_selftest_fp8_quotients compares the codes it gives with those of the
// IEEE division for every bf16 value and every scale a bf16 tile can have.
constexpr float kFastQuotientMinScale = 0x1p-100f;

__device__ __forceinline__ float quotient_rn(float x, float sc, float rc) {
  const float q0 = __fmul_rn(x, rc);
  return copysignf(__fmaf_rn(__fmaf_rn(-sc, q0, x), rc, q0), x);
}

// E4M3 codes of x0 / sc and x1 / sc (x0 in the low byte), as the quantizer forms them.
__device__ __forceinline__ uint16_t code_pair(float x0, float x1, float sc, float rc, bool fast) {
  return fast ? pack_e4m3x2(quotient_rn(x0, sc, rc), quotient_rn(x1, sc, rc))
              : pack_e4m3x2(__fdiv_rn(x0, sc), __fdiv_rn(x1, sc));
}

// One block per (head slice z, 128-row tile t).  The tile is 128 * D / 8 chunks of 16 bytes (8
// values); each thread holds D / 16 of them in registers as packed bf16, every load issued before
// the first use, so four blocks fit on an SM with their whole tiles (32 KB at d = 128) in flight.
// Row-major codes: thread i takes chunks i, i + 256, ..., so each load instruction of a warp reads
// 512 contiguous bytes and each store writes 256.  Transposed codes: thread 2r + h takes half h of
// row r, whose codes it writes down column r of the shared-memory staging tile.
template <int D>
__global__ void __launch_bounds__(kQuantThreads, 4) quantize_fp8_kernel(
    const __nv_bfloat16* __restrict__ x, uint8_t* __restrict__ codes, float* __restrict__ scales,
    int N, int n_tiles, int n_pad, int transpose) {
  constexpr int kRowChunks = D / 8;                          // chunks per row
  constexpr int kPer = kBM * kRowChunks / kQuantThreads;     // chunks per thread (D / 16)
  __shared__ float red[kQuantThreads / 32];
  __shared__ float s_scale, s_rcp;
  __shared__ __align__(16) uint8_t tile_t[D][kBM + 16];  // transposed codes (transpose only)
  const int z = blockIdx.x / n_tiles;
  const int t = blockIdx.x % n_tiles;
  const int rows = min(kBM, N - t * kBM);  // rows of this tile inside the tensor
  const size_t base = (static_cast<size_t>(z) * N + static_cast<size_t>(t) * kBM) * D;
  auto chunk = [&](int i) {
    return transpose ? (threadIdx.x >> 1) * kRowChunks + (threadIdx.x & 1) * kPer + i
                     : static_cast<int>(threadIdx.x) + kQuantThreads * i;
  };
  uint4 w[kPer];  // 8 bf16 values each
  const uint4* src = reinterpret_cast<const uint4*>(x + base);
  #pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int k = chunk(i);
    w[i] = k / kRowChunks < rows ? src[k] : make_uint4(0, 0, 0, 0);
  }
  // |x| maximum in bf16 (the maximum of bf16 values is one of them: exact)
  __nv_bfloat162 m2 = __float2bfloat162_rn(0.f);
  #pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w[i]);
    #pragma unroll
    for (int q = 0; q < 4; ++q) m2 = __hmax2(m2, __habs2(h[q]));
  }
  float amax = fmaxf(__low2float(m2), __high2float(m2));
  #pragma unroll
  for (int s = 16; s > 0; s >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, s));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = 0.f;
    for (int i = 0; i < kQuantThreads / 32; ++i) m = fmaxf(m, red[i]);
    const float sc = m > 0.f ? __fdiv_rn(m, 448.f) : 1.f;
    s_scale = sc;
    s_rcp = __frcp_rn(sc);
    scales[blockIdx.x] = sc;
  }
  __syncthreads();
  const float sc = s_scale, rc = s_rcp;
  const bool fast = sc >= kFastQuotientMinScale;
  uint2 cw[kPer];  // the 8 codes of each chunk
  #pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w[i]);
    uint32_t c[2];
    #pragma unroll
    for (int q = 0; q < 2; ++q) {
      const float2 a = __bfloat1622float2(h[2 * q]), b = __bfloat1622float2(h[2 * q + 1]);
      c[q] = static_cast<uint32_t>(code_pair(a.x, a.y, sc, rc, fast)) |
             (static_cast<uint32_t>(code_pair(b.x, b.y, sc, rc, fast)) << 16);
    }
    cw[i] = make_uint2(c[0], c[1]);
  }
  if (!transpose) {
    uint2* dst = reinterpret_cast<uint2*>(codes + base);
    #pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int k = chunk(i);
      if (k / kRowChunks < rows) dst[k] = cw[i];
    }
    return;
  }
  // transposed: stage [d][row] in shared memory, then write 128-byte rows of [d][Npad]
  const int r = threadIdx.x >> 1, c0 = (threadIdx.x & 1) * (D / 2);
  #pragma unroll
  for (int i = 0; i < kPer; ++i)
    #pragma unroll
    for (int e = 0; e < 8; ++e)
      tile_t[c0 + 8 * i + e][r] =
          static_cast<uint8_t>((e < 4 ? cw[i].x : cw[i].y) >> (8 * (e & 3)));
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

// Block b takes amax = the positive finite bf16 number with bits b + 1 (0x0001 .. 0x7F7F) and
// every bf16 x with |x| <= amax: the quantizer's code of x at the tile scale amax / 448 against
// the E4M3 code of the IEEE quotient.  Mismatching pairs are counted into *mismatches.
__global__ void __launch_bounds__(256) fp8_quotient_check_kernel(unsigned long long* mismatches) {
  const uint32_t abits = blockIdx.x + 1u;
  const float sc = __fdiv_rn(__uint_as_float(abits << 16), 448.f);
  const float rc = __frcp_rn(sc);
  const bool fast = sc >= kFastQuotientMinScale;
  unsigned int bad = 0;
  for (uint32_t xb = threadIdx.x; xb <= abits; xb += blockDim.x) {
    const float xp = __uint_as_float(xb << 16), xn = __uint_as_float((xb | 0x8000u) << 16);
    const uint16_t got = code_pair(xp, xn, sc, rc, fast);
    const uint16_t want = pack_e4m3x2(__fdiv_rn(xp, sc), __fdiv_rn(xn, sc));
    bad += ((got & 0xFFu) != (want & 0xFFu)) + ((got >> 8) != (want >> 8));
  }
  #pragma unroll
  for (int off = 16; off > 0; off >>= 1) bad += __shfl_xor_sync(0xffffffffu, bad, off);
  if ((threadIdx.x & 31) == 0 && bad) atomicAdd(mismatches, static_cast<unsigned long long>(bad));
}

}  // namespace

cudaError_t launch_fp8_quotient_check(unsigned long long* mismatches, cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(mismatches, 0, sizeof(unsigned long long), stream);
  if (e != cudaSuccess) return e;
  fp8_quotient_check_kernel<<<0x7F7F, 256, 0, stream>>>(mismatches);
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
