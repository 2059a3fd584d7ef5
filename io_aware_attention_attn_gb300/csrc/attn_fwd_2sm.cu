// attn_fwd_2sm.cu -- instantiations and launcher of the two-SM fused forward (head dims 64, 128).
#include <atomic>

#include "attn_fwd_2sm_kernel.cuh"

namespace attn {
namespace {

template <int D, bool CAUSAL, bool VARLEN>
cudaError_t launch(const FwdParams& p, int units, cudaStream_t stream) {
  auto* kernel = attn_fwd_2sm_kernel<D, CAUSAL, VARLEN>;
  constexpr int kSmem = Fwd2smLayout<D>::kDynBytes;
  // the opt-in for more than 48 KB of dynamic shared memory and the number of clusters that fit
  // at once are per device; remember them (0: not known yet)
  static std::atomic<int> fit[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int clusters = fit[dev & 63].load(std::memory_order_acquire);
  if (clusters == 0) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * kSmCount);
    cfg.blockDim = dim3(k2smThreads);
    cfg.dynamicSmemBytes = kSmem;
    int n = 0;
    // the kernel's cluster shape (2, 1, 1) is a compile-time attribute
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess || n <= 0) {
      (void)cudaGetLastError();
      n = kSmCount / 2;
    }
    clusters = n;
    fit[dev & 63].store(clusters, std::memory_order_release);
  }
  // persistent: one cluster of two CTAs per pair of SMs that fits, each looping over units (for a
  // packed batch `units` is an upper bound; the kernel counts the units from cu_seqlens)
  const int grid = 2 * (units < clusters ? units : clusters);
  kernel<<<grid, k2smThreads, kSmem, stream>>>(p);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const FwdParams& p, bool causal, bool varlen, int units,
                     cudaStream_t stream) {
  if (varlen)
    return causal ? launch<D, true, true>(p, units, stream)
                  : launch<D, false, true>(p, units, stream);
  return causal ? launch<D, true, false>(p, units, stream) : launch<D, false, false>(p, units, stream);
}

}  // namespace

cudaError_t launch_fwd_2sm(const FwdParams& p, int d, bool causal, bool varlen, int units,
                           cudaStream_t stream) {
  if (units <= 0) return cudaErrorInvalidValue;
  if (d == 64) return launch_d<64>(p, causal, varlen, units, stream);
  if (d == 128) return launch_d<128>(p, causal, varlen, units, stream);
  return cudaErrorInvalidValue;
}

}  // namespace attn
