// attn_fwd_2sm.cu -- instantiations and launcher of the two-SM fused forward (head dim 128).
#include <atomic>

#include "attn_fwd_2sm_kernel.cuh"

namespace attn {
namespace {

template <bool CAUSAL>
cudaError_t launch(const FwdParams& p, int grid, cudaStream_t stream) {
  auto* kernel = attn_fwd_2sm_kernel<CAUSAL>;
  constexpr int kSmem = Fwd2smLayout::kDynBytes;
  // the opt-in for more than 48 KB of dynamic shared memory is per device; remember it
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
  // the kernel's cluster shape (2, 1, 1) is a compile-time attribute; grid is a multiple of 2
  kernel<<<grid, k2smThreads, kSmem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_d128_2sm(const FwdParams& p, bool causal, int grid, cudaStream_t stream) {
  if (grid % 2 != 0) return cudaErrorInvalidValue;
  return causal ? launch<true>(p, grid, stream) : launch<false>(p, grid, stream);
}

}  // namespace attn
