// attn_bwd_d128.cu -- instantiations and launchers of the backward tile kernels for head dim 128.
#include <atomic>

#include "attn_bwd_kernels.cuh"

namespace attn {
namespace {

// The opt-in for more than 48 KB of dynamic shared memory is per device and per kernel.
template <typename Kernel>
cudaError_t allow_smem(Kernel kernel, int bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(done.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    done.fetch_or(bit, std::memory_order_acq_rel);
  }
  return cudaSuccess;
}

template <bool CAUSAL, bool VARLEN>
cudaError_t launch(const BwdParams& p, cudaStream_t stream) {
  static std::atomic<uint64_t> kv_done{0}, q_done{0};
  auto* kv = attn_bwd_dkdv_kernel<128, CAUSAL, VARLEN>;
  auto* qk = attn_bwd_dq_kernel<128, CAUSAL, VARLEN>;
  constexpr int kKvSmem = BwdKvLayout<128>::kDynBytes;
  constexpr int kQSmem = BwdQLayout<128>::kDynBytes;
  cudaError_t e = allow_smem(kv, kKvSmem, kv_done);
  if (e == cudaSuccess) e = allow_smem(qk, kQSmem, q_done);
  if (e != cudaSuccess) return e;
  // one CTA per (head, 128-row tile); packed batches: per (head, tile slot), past-the-end slots
  // return at once
  const int units = VARLEN ? p.n_tiles : p.n_tiles * p.B;
  kv<<<units * p.H_kv, kBwdThreads, kKvSmem, stream>>>(p);  // per K/V head
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  qk<<<units * p.H, kBwdThreads, kQSmem, stream>>>(p);      // per query head
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_d128(const BwdParams& p, bool causal, cudaStream_t stream) {
  if (p.cu_seqlens)
    return causal ? launch<true, true>(p, stream) : launch<false, true>(p, stream);
  return causal ? launch<true, false>(p, stream) : launch<false, false>(p, stream);
}

}  // namespace attn
