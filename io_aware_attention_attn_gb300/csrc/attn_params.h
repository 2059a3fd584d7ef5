// attn_params.h -- launch parameters and shared-memory layout of the fused forward kernel,
// shared by the host launcher and the device code.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace attn {

constexpr int kBM = 128;           // query rows per tile
constexpr int kBN = 128;           // keys per tile
constexpr int kStages = 2;         // depth of the K and V rings
constexpr int kFwdThreads = 192;   // 6 warps: producer, MMA, 4 x softmax
constexpr float kTau = 8.0f;       // tolerated growth of the row max before O is rescaled (log2)

struct FwdParams {
  CUtensorMap tm_q;          // 3-D maps {d, rows, heads}, box {64, 128, 1}, 128-byte swizzle
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  __nv_bfloat16* o;
  float* lse;
  const int* cu_seqlens;     // packed layout only
  int* status;               // device status word (bounded-wait failures)
  int B, H, N;               // N: sequence length (dense) or total tokens T (packed)
  int n_qt;                  // dense: query tiles per head
  float scale_log2;          // scale * log2(e)
};

template <int D>
struct FwdLayout {
  static constexpr int kTile = kBM * D * 2;     // one 128-row x D bf16 tile (D/64 blocks of 16 KB)
  static constexpr int kPTile = kBM * kBN * 2;  // one 128 x 128 bf16 probability tile
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTile;
  static constexpr int kV = kK + kStages * kTile;
  static constexpr int kP = kV + kStages * kTile;
  static constexpr int kBar = kP + 2 * kPTile;
  enum {
    bQ = 0,                 // Q landed
    bKF = 1,                // K stage full  [kStages]
    bKE = bKF + kStages,    // K stage free  [kStages]
    bVF = bKE + kStages,    // V stage full  [kStages]
    bVE = bVF + kStages,    // V stage free  [kStages]
    bSF = bVE + kStages,    // S buffer written by the MMA  [2]
    bPF = bSF + 2,          // P_j written and O corrected (128 softmax threads arrive)
    bOD = bPF + 1,          // P_j V_j accumulated
    bDR = bOD + 1,          // drain after an abort
    kNumBars = bDR + 1
  };
  static constexpr int kMisc = kBar + kNumBars * 8;  // [0] tmem base [1] abort [2..4] tile info
  static constexpr int kBytes = kMisc + 32;
  static constexpr int kDynBytes = kBytes + 1024;    // slack to align the base to 1024 bytes
};

static_assert(FwdLayout<128>::kDynBytes <= 232448, "fused kernel exceeds 227 KB shared memory");

// Host launchers (one translation unit per head dimension).
cudaError_t launch_fwd_d64(const FwdParams& p, bool causal, bool varlen, int grid,
                           cudaStream_t stream);
cudaError_t launch_fwd_d128(const FwdParams& p, bool causal, bool varlen, int grid,
                            cudaStream_t stream);

// ---------------------------------------------------------------- unfused comparison path
struct UnfusedArgs {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  void* workspace;
  int* status;
  int B, H, N, d;
  bool causal;
  float scale;
};

// Workspace of the unfused path: S [BH][N][Npad] fp32, P [BH][N][Npad] bf16 (unnormalised
// exp(s - m), so the row maximum is exactly 1), and inv_l [BH][N] fp32 (1 / row sum of the
// rounded P), each region 256-byte aligned.  Npad = N rounded up to 128.
struct UnfusedLayout {
  size_t npad, s_off, p_off, l_off, total;
};

inline UnfusedLayout unfused_workspace_layout(int B, int H, int N) {
  UnfusedLayout L{};
  const size_t bh = static_cast<size_t>(B) * static_cast<size_t>(H);
  L.npad = (static_cast<size_t>(N) + 127) / 128 * 128;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  L.s_off = 0;
  L.p_off = up(bh * N * L.npad * 4);
  L.l_off = L.p_off + up(bh * N * L.npad * 2);
  L.total = L.l_off + up(bh * N * 4);
  return L;
}

cudaError_t launch_unfused(const UnfusedArgs& a, cudaStream_t stream);

}  // namespace attn
