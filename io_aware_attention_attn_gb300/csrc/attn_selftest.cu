// attn_selftest.cu -- diagnostic: one 128-row tcgen05 MMA with the exact operand descriptors of
// the fused forward kernel, so descriptor or layout faults show up in isolation.
//   mode 0: D[128 x 128] = A[128 x dim] B[128 x dim]^T  (both K-major: the S = Q K^T product)
//   mode 1: D[128 x dim] = A[128 x 128] B[128 x dim]    (A K-major, B MN-major: the P V product)
//   mode 2: as mode 1 with A held in tensor memory (two bf16 per 32-bit column), written there by
//           tcgen05.st from the threads' registers: the P V product with P kept on chip
#include "attn_fp8.h"
#include "attn_gb300.h"
#include "attn_host.h"
#include "sm103_ptx.cuh"

namespace attn {
namespace {

struct SelftestParams {
  CUtensorMap tm_a;
  CUtensorMap tm_b;
  const void* a;
  float* d;
  int* status;
  int mode;
  int dim;
};

constexpr int kSelftestSmem = 2 * 32768 + 1024 + 64;

__global__ void __launch_bounds__(128, 1) mma_selftest_kernel(const __grid_constant__ SelftestParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  const uint32_t sbase = (raw_s + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw_s);
  const uint32_t sa = sbase, sb = sbase + 32768;
  const uint32_t bar_load = sbase + 65536, bar_mma = bar_load + 8;
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + 65536 + 16);
  const WaitCtx wc{reinterpret_cast<volatile int*>(misc + 1), p.status};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int a_cols = p.mode == 0 ? p.dim : 128;
  const int n_out = p.mode == 0 ? 128 : p.dim;
  const bool a_in_tmem = p.mode == 2;
  if (threadIdx.x == 0) {
    mbar_init(bar_load, 1);
    mbar_init(bar_mma, 1);
    fence_barrier_init();
    misc[1] = 0;
  }
  if (warp == 0) {
    tmem_alloc(sbase + 65536 + 16, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  if (a_in_tmem) {
    // thread r packs row r of A (128 bf16 = 64 words) into TMEM columns 256..319 of lane r
    const int r = warp * 32 + lane;
    const uint32_t* arow = reinterpret_cast<const uint32_t*>(p.a) + r * 64;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(warp * 32) << 16) + 256;
    for (int c = 0; c < 2; ++c) {
      uint32_t v[32];
      for (int i = 0; i < 32; ++i) v[i] = arow[c * 32 + i];
      tmem_st32(t_lane + c * 32, v);
    }
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  bool ok = true;
  if (threadIdx.x == 0) {
    tc_fence_after();
    mbar_arrive_expect_tx(bar_load, 128 * ((a_in_tmem ? 0 : a_cols) + p.dim) * 2);
    if (!a_in_tmem)
      for (int c = 0; c < a_cols / 64; ++c)
        tma_load_3d(sa + c * 16384, &p.tm_a, bar_load, c * 64, 0, 0);
    for (int c = 0; c < p.dim / 64; ++c) tma_load_3d(sb + c * 16384, &p.tm_b, bar_load, c * 64, 0, 0);
    ok = mbar_wait(bar_load, 0, wc, 3, 1);
    if (ok) {
      tc_fence_after();
      if (p.mode == 0) {
        const uint32_t id = idesc_bf16_f32(128, 128, false, false);
        for (int t = 0; t < p.dim / 16; ++t) {
          const uint32_t off = static_cast<uint32_t>((t >> 2) * 16384 + (t & 3) * 32);
          mma_bf16_ss(tmem, sdesc_sw128(sa + off, 16, 1024), sdesc_sw128(sb + off, 16, 1024), id,
                      t > 0 ? 1u : 0u);
        }
      } else if (!a_in_tmem) {
        const uint32_t id = idesc_bf16_f32(128, p.dim, false, true);
        for (int t = 0; t < 128 / 16; ++t) {
          const uint32_t aoff = static_cast<uint32_t>((t >> 2) * 16384 + (t & 3) * 32);
          mma_bf16_ss(tmem, sdesc_sw128(sa + aoff, 16, 1024), sdesc_sw128(sb + t * 2048, 16384, 1024),
                      id, t > 0 ? 1u : 0u);
        }
      } else {
        const uint32_t id = idesc_bf16_f32(128, p.dim, false, true);
        for (int t = 0; t < 128 / 16; ++t)
          mma_bf16_ts(tmem, tmem + 256 + t * 8, sdesc_sw128(sb + t * 2048, 16384, 1024), id,
                      t > 0 ? 1u : 0u);
      }
      mma_commit(bar_mma);
    } else {
      mbar_wait_drain(bar_load, 0);
    }
    misc[2] = ok ? 1u : 0u;
  }
  __syncthreads();
  if (misc[2]) {
    if (mbar_wait_warp(bar_mma, 0, wc, 3, 2)) {
      tc_fence_after();
      const int r = warp * 32 + lane;
      const uint32_t t_lane = tmem + (static_cast<uint32_t>(warp * 32) << 16);
      for (int c = 0; c < n_out / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(t_lane + c * 32, v);
        tmem_wait_ld_regs(v);
        for (int i = 0; i < 32; ++i) p.d[r * n_out + c * 32 + i] = __uint_as_float(v[i]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace
}  // namespace attn

extern "C" int attn_selftest_mma(const void* a, const void* b, float* d, int mode, int dim,
                                 void* stream) {
  using namespace attn;
  if (!a || !b || !d) return ATTN_ERR_NULL;
  if (dim != 64 && dim != 128) return ATTN_ERR_HEAD_DIM;
  if (mode < 0 || mode > 2) return ATTN_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b)) & 15u) return ATTN_ERR_ALIGN;
  int rc = check_device();
  if (rc != 0) return rc;
  SelftestParams p{};
  const int a_cols = mode == 0 ? dim : 128;
  if (encode_rows_map(&p.tm_a, a, a_cols, 128, 1) != CUDA_SUCCESS ||
      encode_rows_map(&p.tm_b, b, dim, 128, 1) != CUDA_SUCCESS)
    return ATTN_ERR_LAUNCH;
  p.a = a;
  p.d = d;
  p.status = status_word();
  if (!p.status) return ATTN_ERR_LAUNCH;
  p.mode = mode;
  p.dim = dim;
  if (cudaFuncSetAttribute(mma_selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kSelftestSmem) != cudaSuccess)
    return ATTN_ERR_LAUNCH;
  mma_selftest_kernel<<<1, 128, kSelftestSmem, static_cast<cudaStream_t>(stream)>>>(p);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

// ------------------------------------------------------------------ bounded-wait self-test
namespace attn {
namespace {

__global__ void wait_timeout_kernel(int* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);  // nobody ever arrives
    fence_barrier_init();
    abort_flag = 0;
  }
  __syncthreads();
  const WaitCtx wc{&abort_flag, status};
  mbar_wait_warp(b, 0, wc, 6, 1);  // gives up after kWaitLimitNs and records the status
}

}  // namespace
}  // namespace attn

extern "C" int attn_selftest_wait_timeout(void* stream) {
  using namespace attn;
  int rc = check_device();
  if (rc != 0) return rc;
  int* status = status_word();
  if (!status) return ATTN_ERR_LAUNCH;
  wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

extern "C" int attn_selftest_fp8_quotients(unsigned long long* mismatches, void* stream) {
  using namespace attn;
  if (!mismatches) return ATTN_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(mismatches) & 7u) return ATTN_ERR_ALIGN;
  int rc = check_device();
  if (rc != 0) return rc;
  return launch_fp8_quotient_check(mismatches, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? ATTN_OK
             : ATTN_ERR_LAUNCH;
}
