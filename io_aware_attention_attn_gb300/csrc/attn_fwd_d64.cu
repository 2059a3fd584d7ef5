// attn_fwd_d64.cu -- instantiations and launcher of the fused forward kernel for head dim 64.
#include <atomic>

#include "attn_fwd_pair_kernel.cuh"

namespace attn {
namespace {

template <bool CAUSAL, bool VARLEN>
cudaError_t launch(const FwdParams& p, int grid, cudaStream_t stream) {
  auto* kernel = attn_fwd_pair_kernel<64, CAUSAL, VARLEN>;
  constexpr int kSmem = PairLayout<64>::kDynBytes;
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
  kernel<<<grid, kPairThreads, kSmem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_d64(const FwdParams& p, bool causal, bool varlen, int grid,
                            cudaStream_t stream) {
  if (causal) return varlen ? launch<true, true>(p, grid, stream) : launch<true, false>(p, grid, stream);
  return varlen ? launch<false, true>(p, grid, stream) : launch<false, false>(p, grid, stream);
}

}  // namespace attn
