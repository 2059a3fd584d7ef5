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
// A tile is exponentiated against the running reference maximum first; only when its row sum
// exceeds kSumLimit (so no P exceeds it either) is the tile maximum taken and the reference moved.
constexpr float kSumLimit = 65536.f;

struct FwdParams {
  CUtensorMap tm_q;          // 3-D maps {d, rows, heads}, box {64, 128, 1}, 128-byte swizzle
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  CUtensorMap tm_o;          // O as {d, rows, heads}, box {64, 32, 1}: two-SM epilogue stores
  __nv_bfloat16* o;
  float* lse;
  const int* cu_seqlens;     // packed layout only
  int* status;               // device status word (bounded-wait failures)
  int B, H, N;               // H: query heads; N: sequence length (dense) or total tokens T
  int group;                 // query heads per K/V head (1: multi-head; H: multi-query)
  int n_splits;              // key-range slices per query pair (1: the whole row in one CTA)
  float* part_o;             // split-KV partials [n_splits][B H N][D] fp32 (unnormalised O)
  float* part_stat;          // split-KV partials [2][n_splits][B H N]: reference max (log2),
                             // row sum
  int n_qt;                  // dense: query-tile pairs (256 rows) per head
  float scale_log2;          // scale * log2(e)
};

// ------------------------------------------------ fused kernel: one query tile per SM, two SMs
// per MMA (a cluster of two CTAs; see attn_fwd_2sm_kernel.cuh)
constexpr int k2smThreads = 224;  // 7 warps: producer, P V issuer, 4 softmax, S issuer
constexpr int k2smStagesK = 4;
constexpr int k2smStagesV = 4;
constexpr int k2smSBufs = 3;      // S / P buffers in tensor memory
constexpr int k2smPVN = 128;      // N of the P V product: D = 128, or D = 64 padded with zero V
template <int D>
struct Fwd2smLayout {
  static constexpr int kQBytes = kBM * D * 2;  // this CTA's 128 query rows (D/64 64-col blocks)
  static constexpr int kKBytes = 64 * D * 2;   // 64 keys of a key tile (D/64 blocks of 8 KB)
  static constexpr int kVBytes = kBN * 64 * 2; // a key tile's 64 value columns of this CTA
  static constexpr int kQ = 0;                 // [2]: the current and the next query pair
  static constexpr int kK = kQ + 2 * kQBytes;
  static constexpr int kV = kK + k2smStagesK * kKBytes;
  // epilogue staging [4 warps][2 halves][32 rows x 128 bytes], 1024-byte aligned: the TMA
  // stores of O read it in the 128-byte swizzle
  static constexpr int kOut = kV + k2smStagesV * kVBytes;
  static constexpr int kBar = kOut + 4 * 8192;
  enum {
    bQF = 0,                       // both CTAs' Q landed (leader's copy)   [2 Q buffers]
    bQE = bQF + 2,                 // Q buffer free: its S products done (both) [2]
    bKF = bQE + 2,                 // K stage full (leader's copy)  [k2smStagesK]
    bKE = bKF + k2smStagesK,       // K stage free (both)           [k2smStagesK]
    bVF = bKE + k2smStagesK,       // V stage full (leader's copy)  [k2smStagesV]
    bVE = bVF + k2smStagesV,       // V stage free (both)           [k2smStagesV]
    bSF = bVE + k2smStagesV,       // S written into buffer b (both)          [k2smSBufs]
    bPF = bSF + k2smSBufs,         // P written, O corrected (leader's copy)  [k2smSBufs]
    bPV = bPF + k2smSBufs,         // P V from buffer b completed (both)      [k2smSBufs]
    bOD = bPV + k2smSBufs,         // a pair's last P V completed (both)
    bOE = bOD + 1,                 // O read by the epilogue (leader's copy, 8 arrivals)
    bDR = bOE + 1,                 // drain after an abort (leader), one per issuer [2]
    kNumBars = bDR + 2
  };
  static constexpr int kMisc = kBar + kNumBars * 8;  // [0] tmem base [1] abort [2] units [3] pairs
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kDynBytes = kBytes + 1024;
  static_assert(kOut % 1024 == 0, "O staging must sit on the swizzle atom");
  static_assert(kDynBytes <= 232448, "two-SM kernel exceeds 227 KB shared memory");
};

// The forward on CTA pairs, persistent (head dim 64 or 128): `units` = query pairs x key slices
// (dense) or an upper bound on the query pairs of all sequences times the heads (packed), spread
// over as many clusters of two CTAs as fit on the device; p.tm_k has a 64-row box, p.tm_o a
// 32-row box.
cudaError_t launch_fwd_2sm(const FwdParams& p, int d, bool causal, bool varlen, int units,
                           cudaStream_t stream);

// Split-KV: slices per query pair the library picks when the caller passes num_splits <= 0, and
// the merge of the slices' partial results (attn_splitkv.cu).  The pick minimises a simple cost
// model of the launch: waves of (query pair, slice) units times the key tiles one slice visits
// plus about two tiles of fixed per-unit cost (prologue, epilogue, partial write-out).  A unit is
// a cluster of two CTAs on two SMs (76 at once).
constexpr int kSmCount = 152;
constexpr int kMaxSplits = 32;
inline int splitkv_pick(int B, int H, int N, int d, int num_splits) {
  (void)d;
  const long long slots = kSmCount / 2;
  const long long pairs = static_cast<long long>((N + 2 * kBM - 1) / (2 * kBM)) * B * H;
  const int key_tiles = (N + kBN - 1) / kBN;
  const int cap = key_tiles < kMaxSplits ? key_tiles : kMaxSplits;
  if (cap < 1 || pairs < 1) return 1;
  if (num_splits > 0) return num_splits < cap ? num_splits : cap;
  int best = 1;
  long long best_cost = -1;
  for (int s = 1; s <= cap; ++s) {
    const long long waves = (pairs * s + slots - 1) / slots;
    const long long cost = waves * ((key_tiles + s - 1) / s + 2);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}
cudaError_t launch_splitkv_combine(int d, const float* part_o, const float* part_stat, void* o,
                                   float* lse, long long rows, int splits, cudaStream_t stream);

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
