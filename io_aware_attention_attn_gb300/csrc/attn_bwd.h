// attn_bwd.h -- launch parameters, shared-memory layouts and launchers of the backward pass.
//
// The backward recomputes S and P tile by tile from the logsumexp the forward saved (CS336
// Lecture 5 notes, section 6.2, "反向传播怎么办") and applies the chain rule of the definition:
// dV = P^T dO, dP = dO V^T, dS = P * (dP - D) with D_i = dO_i . O_i, dQ = scale dS K,
// dK = scale dS^T Q.  Two launches:
//   bwd_prep_kernel         -D_i and -lse_i * log2(e) per query row, into padded fp32 planes
//   attn_bwd_tiles_kernel   the dK/dV pass, one CTA per (K/V head, 128-key tile): dK and dV
//                           accumulated in tensor memory over the query tiles; then the dQ pass,
//                           one CTA per (head, 128-query tile): dQ accumulated in tensor memory
//                           over the key tiles
// Every output element is written by exactly one CTA: no atomics, the result is deterministic.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "attn_params.h"

namespace attn {

// Programmatic dependent launch: the tile kernel is launched as the row pass's blocks finish, sets
// up its barriers and tensor memory, and waits here for the row pass's grid to complete (and its
// writes to be visible) before it reads the planes.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Status kind (low byte of the device status word, beside the kinds of the bounded waits): the
// launch's dynamic shared memory could not hold the dK/dV pass's 1024-byte-aligned layout; the
// CTA then did nothing.
constexpr int kStatusSmemLayout = 3;

constexpr int kBwdThreads = 384;    // warp 0 TMA, warps 1, 10, 11 MMA, warps 2..9 column halves
constexpr int kBwdStages = 2;       // depth of the streamed-tile rings
constexpr int kBwdStagesQ = 3;      // dK/dV kernel: depth of the Q ring

struct BwdParams {
  CUtensorMap tm_q;   // 3-D maps over [B*H][N][D] bf16, box {64, 128, 1}, 128-byte swizzle
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  CUtensorMap tm_do;
  CUtensorMap tm_dq;  // dense head dim 128: outputs, box {64, 32, 1}, 128-byte swizzle (TMA stores)
  CUtensorMap tm_dk;
  CUtensorMap tm_dv;
  __nv_bfloat16* dq;  // outputs [B, H, N, D] bf16
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  const float* nlse2;  // [B*H][n_pad]: -lse * log2(e); -inf in rows >= N
  const float* nd;     // [B*H][n_pad]: -rowsum(dO * O); 0 in rows >= N
  int* status;        // device status word (bounded waits)
  const int32_t* cu_seqlens;  // packed batches: int32[n_seqs + 1] offsets into the T rows; else NULL
  int n_seqs;         // packed batches: number of sequences
  int B, H, N;        // packed batches: N = T, the total number of rows
  int H_kv;           // key/value heads (H_kv divides H; query head h reads K/V head h / group)
  int group;          // H / H_kv
  int n_tiles;        // dense: ceil(N / 128); packed: tile slots ceil(T / 128) + n_seqs
  int n_pad;          // rows of a head in the -lse2 / -D planes: 128 * n_tiles
  float scale_log2;   // scale * log2(e)
  float scale;
};

// dK/dV kernel: K_j and V_j resident; Q_i with its -lse2 slice streams through a kBwdStagesQ ring
// (S^T of query tile t+2 is issued while tile t+1 is being processed, so its Q tile must have
// landed a tile earlier), dO_i with its -D slice through a kBwdStages ring.  At head dim 128 the
// tiles take 224 KB; the layout then fits the 227 KB limit only if the dynamic shared memory
// starts within 272 bytes of a 1024-byte boundary (the kernel checks, and reports
// kStatusSmemLayout instead of running otherwise).
template <int D>
struct BwdKvLayout {
  static constexpr int kTile = kBM * D * 2;
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTile;
  static constexpr int kQ = kV + kTile;                    // [kBwdStagesQ]
  static constexpr int kDO = kQ + kBwdStagesQ * kTile;     // [kBwdStages]
  static constexpr int kLse = kDO + kBwdStages * kTile;    // [kBwdStagesQ] x -lse2[128]
  static constexpr int kDvec = kLse + kBwdStagesQ * 512;   // [kBwdStages] x -D[128]
  static constexpr int kBar = kDvec + kBwdStages * 512;
  enum {
    bKV = 0,                   // K_j and V_j landed
    bQF = 1,                   // Q_i and its -lse2 landed  [kBwdStagesQ]
    bQE = bQF + kBwdStagesQ,   // Q stage free              [kBwdStagesQ]
    bOF = bQE + kBwdStagesQ,   // dO_i and its -D landed    [kBwdStages]
    bOE = bOF + kBwdStages,    // dO stage free             [kBwdStages]
    bS = bOE + kBwdStages,     // S^T = K Q^T written               [2 tensor-memory buffers]
    bSR = bS + 2,              // S^T read by every compute thread (256 arrivals)
    bDP,                       // dP^T = V dO^T written over the S^T just read
    bP,                        // P^T (bf16) written over dP^T (256 arrivals)  [2 buffers]
    bDS = bP + 2,              // dS^T (bf16) written over dP^T (256 arrivals) [2 buffers]
    bACC = bDS + 2,            // dV += P^T dO and dK += dS^T Q completed  [2 buffers]
    bEND = bACC + 2,           // every product of the CTA completed (dV and dK issuers)
    bVEND,                     // the last dV product completed
    bDR,                       // drain after an abort, one per issuer [3]
    kNumBars = bDR + 3
  };
  static constexpr int kMisc = kBar + kNumBars * 8;  // [0] tmem base [1] abort [2..5] tile
  static constexpr int kBytes = kMisc + 32;
  static constexpr int kDynBytes = kBytes + 1024 <= 232448 ? kBytes + 1024 : 232448;
};

// dQ kernel: Q_i and dO_i resident; K_j and V_j stream through rings (K three deep: K_j is
// still read by dQ_j while S_{j+1} reads K_{j+1} and K_{j+2} is in flight).
constexpr int kBwdStagesQK = 3;
template <int D>
struct BwdQLayout {
  static constexpr int kTile = kBM * D * 2;
  static constexpr int kQ = 0;
  static constexpr int kDO = kQ + kTile;
  static constexpr int kK = kDO + kTile;                   // [kBwdStagesQK]
  static constexpr int kV = kK + kBwdStagesQK * kTile;     // [kBwdStages]
  static constexpr int kBar = kV + kBwdStages * kTile;
  enum {
    bQ = 0,                   // Q_i and dO_i landed
    bKF = 1,                  // K stage full [kBwdStagesQK]
    bKE = bKF + kBwdStagesQK, // K stage free (both issuers) [kBwdStagesQK]
    bVF = bKE + kBwdStagesQK, // V stage full [kBwdStages]
    bVE = bVF + kBwdStages,   // V stage free [kBwdStages]
    bS = bVE + kBwdStages,    // S = Q K^T written
    bSR,                      // S read by every compute thread (256 arrivals)
    bDP,                      // dP = dO V^T written            [2 tensor-memory buffers]
    bDS = bDP + 2,            // dS (bf16) written over dP       [2] (256 arrivals)
    bDQ = bDS + 2,            // dQ += dS K from buffer completed [2]
    bDR = bDQ + 2,            // drain after an abort, one per issuer [3]
    kNumBars = bDR + 3
  };
  static constexpr int kMisc = kBar + kNumBars * 8;  // [0] tmem base [1] abort [2..5] tile
  static constexpr int kBytes = kMisc + 32;
  static constexpr int kDynBytes = kBytes + 1024;
};

static_assert(BwdKvLayout<128>::kDynBytes <= 232448, "dK/dV kernel exceeds 227 KB shared memory");
static_assert(BwdQLayout<128>::kDynBytes <= 232448, "dQ kernel exceeds 227 KB shared memory");

// Packed batches: the 128-row tiles of all sequences, numbered sequence after sequence, are the
// "slots" of a head.  A warp-collective scan of cu_seqlens maps a slot to its sequence (start
// row, length, tile within the sequence, slots of the earlier sequences); tile = -1 for a slot past
// the last tile.  Offsets are clamped into [0, N] so no access leaves the buffers.
__device__ __forceinline__ void bwd_locate_tile(const int32_t* cu, int n_seqs, int N, int slot,
                                                int lane, int& start, int& len, int& tile,
                                                int& base) {
  start = 0;
  len = 0;
  tile = -1;
  base = 0;
  int remaining = slot, before = 0;
  for (int b0 = 0; b0 < n_seqs; b0 += 32) {
    const int s = b0 + lane;
    int a = 0, e = 0;
    if (s < n_seqs) {
      a = min(max(__ldg(cu + s), 0), N);
      e = min(max(__ldg(cu + s + 1), a), N);
    }
    const int nt = (e - a + kBM - 1) / kBM;
    int incl = nt;
    #pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    const int excl = incl - nt;
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    if (remaining < total) {
      const unsigned hit = __ballot_sync(0xffffffffu, remaining >= excl && remaining < incl);
      const int src = __ffs(hit) - 1;  // hit != 0: the slots of this chunk cover `remaining`
      start = __shfl_sync(0xffffffffu, a, src);
      len = __shfl_sync(0xffffffffu, e - a, src);
      const int ex = __shfl_sync(0xffffffffu, excl, src);
      tile = remaining - ex;
      base = before + ex;
      return;
    }
    remaining -= total;
    before += total;
  }
}

// Launchers (one translation unit per head dimension for the tile kernels).
cudaError_t launch_bwd_d64(const BwdParams& p, bool causal, cudaStream_t stream);
cudaError_t launch_bwd_d128(const BwdParams& p, bool causal, cudaStream_t stream);
cudaError_t launch_bwd_prep(const void* o, const void* dout, const float* lse, float* nlse2,
                            float* nd, int BH, int N, int n_pad, int d, cudaStream_t stream);
// packed batches: planes of 128 * (ceil(T/128) + n_seqs) rows per head, one 128-row tile per slot
cudaError_t launch_bwd_prep_varlen(const void* o, const void* dout, const float* lse,
                                   float* nlse2, float* nd, const int32_t* cu_seqlens, int n_seqs,
                                   int H, int T, int n_slots, int d, cudaStream_t stream);

}  // namespace attn
