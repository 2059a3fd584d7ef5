// attn_fp8.h -- parameters, shared-memory layout and launchers of the FP8 (E4M3) forward.
//
// Inputs are E4M3 codes with one fp32 scale per 128-row tile of each head (value = code x scale;
// the E4M3 format and per-tile scaling: CS336 Lecture 5 notes, section 3.1).  Q and K are
// [B*H][N][128] codes; V is stored transposed, [B*H][128][Npad] (Npad = N rounded up to 128,
// padding codes 0), so that every tensor-core operand of the kind::f8f6f4 products is K-major.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "attn_params.h"

namespace attn {

constexpr int kFp8Threads = 320;  // warp 0 TMA, warp 1 MMA, warps 2..9 softmax (two tiles)
constexpr int kFp8StagesK = 3;
constexpr int kFp8StagesV = 3;
// The probabilities enter the P V product as E4M3 codes of P * 48 * (sv_j / sv_max): with the
// reference maximum allowed to trail the row maximum by at most kFp8Tau = 3 (log2 units), P <= 8
// and the codes stay at or below 384 < 448, while P down to 2^-14.6 of the reference stays above
// E4M3's smallest subnormal.  (A reference that moves on every 0.5 of growth with a factor of 256
// measured 1409 TFLOPS against 1478 here: the O rescales it forces cost more than they buy.)
constexpr float kFp8Tau = 3.0f;
constexpr float kFp8PScale = 48.f;

struct Fp8Params {
  CUtensorMap tm_q;    // [B*H][N][128] E4M3, box {128, 128, 1}, 128-byte swizzle
  CUtensorMap tm_k;
  CUtensorMap tm_vt;   // [B*H][128][Npad] E4M3, box {128, 128, 1}, 128-byte swizzle
  __nv_bfloat16* o;    // [B, H, N, 128] bf16
  float* lse;          // [B, H, N] fp32
  const float* sq;     // [B*H][n_tiles] tile scales
  const float* sk;
  const float* sv;
  int* status;
  int B, H, N;
  int n_tiles;         // ceil(N / 128)
  int n_qt;            // pairs of query tiles per head
  float scale_log2;    // softmax scale * log2(e)
};

struct Fp8Layout {
  static constexpr int kTile = kBM * 128;  // 128 rows x 128 one-byte codes
  static constexpr int kQ = 0;             // Q_0, Q_1
  static constexpr int kK = kQ + 2 * kTile;
  static constexpr int kV = kK + kFp8StagesK * kTile;
  static constexpr int kOut = kV + kFp8StagesV * kTile;  // O staging: 8 warps x 32 rows x 256 B
  static constexpr int kBar = kOut + 8 * 32 * 256;
  enum {
    bQ = 0,
    bKF = 1,
    bKE = bKF + kFp8StagesK,
    bVF = bKE + kFp8StagesK,
    bVE = bVF + kFp8StagesV,
    bSF = bVE + kFp8StagesV,  // [2]
    bPF = bSF + 2,            // [2] (128 arrivals)
    bPV = bPF + 2,            // [2]
    bOD = bPV + 2,            // [2]
    bDR = bOD + 2,
    kNumBars
  };
  static constexpr int kMisc = kBar + kNumBars * 8;  // [0] tmem base [1] abort flag
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kDynBytes = kBytes + 1024;
};

cudaError_t launch_fwd_fp8(const Fp8Params& p, bool causal, cudaStream_t stream);
cudaError_t launch_quantize_fp8(const void* x, void* codes, float* scales, int BH, int N, int d,
                                bool transpose, cudaStream_t stream);
// Compares the quantizer's codes with those of the IEEE quotient for every bf16 value x and every
// tile maximum amax >= |x| (attn_selftest_fp8_quotients); the count lands in *mismatches.
cudaError_t launch_fp8_quotient_check(unsigned long long* mismatches, cudaStream_t stream);

}  // namespace attn
