// attn_bwd_d64.cu -- instantiations and launchers of the backward tile kernels for head dim 64.
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
  static std::atomic<uint64_t> done{0};
  auto* kernel = attn_bwd_tiles_kernel<64, CAUSAL, VARLEN>;
  constexpr int kSmem = BwdKvLayout<64>::kDynBytes > BwdQLayout<64>::kDynBytes
                            ? BwdKvLayout<64>::kDynBytes
                            : BwdQLayout<64>::kDynBytes;
  cudaError_t e = allow_smem(kernel, kSmem, done);
  if (e != cudaSuccess) return e;
  // one CTA per (head, 128-row tile): the dK/dV pass per K/V head, then the dQ pass per query
  // head; packed batches: per (head, tile slot), past-the-end slots return at once
  const long long units = VARLEN ? p.n_tiles : static_cast<long long>(p.n_tiles) * p.B;
  const long long n_kv = units * p.H_kv, n_q = units * p.H;
  if (n_kv + n_q > 0x7FFFFFFF) return cudaErrorInvalidValue;
  // programmatic dependent launch: the CTAs set up while the row pass finishes, then wait for it
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(n_kv + n_q));
  cfg.blockDim = dim3(kBwdThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kernel, p, static_cast<int>(n_kv));
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_d64(const BwdParams& p, bool causal, cudaStream_t stream) {
  if (p.cu_seqlens)
    return causal ? launch<true, true>(p, stream) : launch<false, true>(p, stream);
  return causal ? launch<true, false>(p, stream) : launch<false, false>(p, stream);
}

}  // namespace attn
