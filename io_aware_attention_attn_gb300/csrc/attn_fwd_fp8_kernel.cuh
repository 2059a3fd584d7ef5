// attn_fwd_fp8_kernel.cuh -- FP8 (E4M3) fused attention forward for sm_103a, head dim 128.
//
// The pipeline of the bf16 pair kernel (two 128-row query tiles per CTA; warp 0 TMA producer,
// warp 1 MMA issuer, warps 2..9 softmax, one row per thread) with kind::f8f6f4 products:
//   S_t  = Q_t K_j^T     A = Q codes, B = K codes, both K-major (4 instructions of K = 32)
//   O_t += P_t V_j       A = P codes from tensor memory, B = V^T codes (K-major: V is stored
//                        transposed, [d][keys]); 4 instructions of 32 keys
// Tile scales enter the softmax: the scores of (query tile t, key tile j) are the raw products
// times sq_t * sk_j * scale * log2(e).  V's tile scales are folded into the probabilities:
// P_t V_j uses the codes of P * kFp8PScale * sv_j / sv_max, and the epilogue multiplies by
// sv_max / (kFp8PScale l).  The reference maximum trails the row maximum by at most kFp8Tau, so
// P <= 2^kFp8Tau and the codes never saturate.  l and lse use the fp32 sums of the unrounded P.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "attn_fp8.h"
#include "sm103_ptx.cuh"

namespace attn {
namespace fp8k {
__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }
}  // namespace fp8k

template <bool CAUSAL>
__global__ void __launch_bounds__(kFp8Threads, 1)
    attn_fwd_fp8_kernel(const __grid_constant__ Fp8Params p) {
  using Lay = Fp8Layout;
  using fp8k::f2u;
  using fp8k::u2f;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  const uint32_t sbase = (raw_s + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw_s);
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + Lay::kMisc);
  const WaitCtx wc{reinterpret_cast<volatile int*>(misc + 1), p.status};
  auto bar = [&](int i) -> uint32_t { return sbase + Lay::kBar + 8u * static_cast<uint32_t>(i); };
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(bar(Lay::bQ), 1);
    for (int s = 0; s < kFp8StagesK; ++s) {
      mbar_init(bar(Lay::bKF + s), 1);
      mbar_init(bar(Lay::bKE + s), 1);
    }
    for (int s = 0; s < kFp8StagesV; ++s) {
      mbar_init(bar(Lay::bVF + s), 1);
      mbar_init(bar(Lay::bVE + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(Lay::bSF + t), 1);
      mbar_init(bar(Lay::bPF + t), 4);
      mbar_init(bar(Lay::bPV + t), 1);
      mbar_init(bar(Lay::bOD + t), 1);
    }
    mbar_init(bar(Lay::bDR), 1);
    fence_barrier_init();
    misc[1] = 0;
  }

  const int BH = p.B * p.H;
  const int L = static_cast<int>(blockIdx.x);
  int z, pt;
  if constexpr (CAUSAL) {  // heaviest pairs first
    pt = p.n_qt - 1 - L / BH;
    z = L % BH;
  } else {                 // the pairs of a head together: its K and V stay in L2
    z = L / p.n_qt;
    pt = L % p.n_qt;
  }
  const int seq_len = p.N;
  int n_kv[2];
  #pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int qt = 2 * pt + t;
    n_kv[t] = (qt * kBM >= seq_len) ? 0 : (CAUSAL ? qt + 1 : p.n_tiles);
  }
  const int n_max = n_kv[0] > n_kv[1] ? n_kv[0] : n_kv[1];

  __syncthreads();
  if (warp == 1) {
    tmem_alloc(sbase + Lay::kMisc, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  constexpr uint32_t kColS[2] = {0, 128};
  constexpr uint32_t kColO[2] = {256, 384};
  constexpr uint64_t kTileD = static_cast<uint64_t>(Lay::kTile >> 4);

  if (warp == 0) {
    // ================================================================ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_vt);
      const uint64_t keep = l2_policy_evict_last();
      const uint64_t once = l2_policy_evict_first();
      mbar_arrive_expect_tx(bar(Lay::bQ), 2 * Lay::kTile);
      #pragma unroll
      for (int t = 0; t < 2; ++t)
        tma_load_3d_hint(sbase + Lay::kQ + t * Lay::kTile, &p.tm_q, bar(Lay::bQ), 0,
                         (2 * pt + t) * kBM, z, once);
      int nk = 0, nv = 0;
      bool ok = true;
      for (int j = 0; j < n_max; ++j) {
        const int sk = j % kFp8StagesK, sv = j % kFp8StagesV;
        if (j >= kFp8StagesK &&
            !(ok = mbar_wait(bar(Lay::bKE + sk),
                             (static_cast<uint32_t>(j / kFp8StagesK) & 1u) ^ 1u, wc, 0, 1)))
          break;
        mbar_arrive_expect_tx(bar(Lay::bKF + sk), Lay::kTile);
        tma_load_3d_hint(sbase + Lay::kK + sk * Lay::kTile, &p.tm_k, bar(Lay::bKF + sk), 0,
                         j * kBN, z, keep);
        ++nk;
        if (j >= kFp8StagesV &&
            !(ok = mbar_wait(bar(Lay::bVE + sv),
                             (static_cast<uint32_t>(j / kFp8StagesV) & 1u) ^ 1u, wc, 0, 2)))
          break;
        mbar_arrive_expect_tx(bar(Lay::bVF + sv), Lay::kTile);
        tma_load_3d_hint(sbase + Lay::kV + sv * Lay::kTile, &p.tm_vt, bar(Lay::bVF + sv),
                         j * kBN, 0, z, keep);
        ++nv;
      }
      if (!ok) {
        mbar_wait_drain(bar(Lay::bQ), 0);
        for (int j = (nk > kFp8StagesK ? nk - kFp8StagesK : 0); j < nk; ++j)
          mbar_wait_drain(bar(Lay::bKF + j % kFp8StagesK),
                          static_cast<uint32_t>(j / kFp8StagesK) & 1u);
        for (int j = (nv > kFp8StagesV ? nv - kFp8StagesV : 0); j < nv; ++j)
          mbar_wait_drain(bar(Lay::bVF + j % kFp8StagesV),
                          static_cast<uint32_t>(j / kFp8StagesV) & 1u);
      }
    }
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    constexpr uint32_t kId = idesc_e4m3_f32(kBM, kBN);  // both products are M128 N128
    const uint64_t desc_q = sdesc_sw128(sbase + Lay::kQ, 16, 1024);
    const uint64_t desc_k = sdesc_sw128(sbase + Lay::kK, 16, 1024);
    const uint64_t desc_v = sdesc_sw128(sbase + Lay::kV, 16, 1024);
    auto issue_s = [&](int t, int j) {
      const uint64_t a = desc_q + static_cast<uint64_t>(t) * kTileD;
      const uint64_t b = desc_k + static_cast<uint64_t>(j % kFp8StagesK) * kTileD;
      #pragma unroll
      for (int k = 0; k < 4; ++k)  // K = 32 codes = 32 bytes per instruction
        mma_f8_ss(tmem + kColS[t], a + 2 * k, b + 2 * k, kId, k > 0 ? 1u : 0u);
      mma_commit(bar(Lay::bSF + t));
    };
    auto wait_k = [&](int j) {
      return mbar_wait_warp(bar(Lay::bKF + j % kFp8StagesK),
                            static_cast<uint32_t>(j / kFp8StagesK) & 1u, wc, 1, 3);
    };
    bool ok = mbar_wait_warp(bar(Lay::bQ), 0, wc, 1, 4) && wait_k(0);
    if (ok) {
      tc_fence_after();
      if (lane == 0) {
        if (n_kv[0] > 0) issue_s(0, 0);
        if (n_kv[1] > 0) issue_s(1, 0);
        mma_commit(bar(Lay::bKE + 0));
      }
      __syncwarp();
    }
    for (int j = 0; ok && j < n_max; ++j) {
      const int sv = j % kFp8StagesV;
      bool v_ready = false;
      #pragma unroll
      for (int t = 0; t < 2; ++t) {
        if (j >= n_kv[t]) continue;
        if (!(ok = mbar_wait_spin_warp(bar(Lay::bPF + t), static_cast<uint32_t>(j) & 1u, wc, 1, 5)))
          break;
        if (!v_ready) {
          if (!(ok = mbar_wait_warp(bar(Lay::bVF + sv),
                                    static_cast<uint32_t>(j / kFp8StagesV) & 1u, wc, 1, 6)))
            break;
          v_ready = true;
        }
        tc_fence_after();
        if (lane == 0) {
          const uint64_t b = desc_v + static_cast<uint64_t>(sv) * kTileD;
          #pragma unroll
          for (int k = 0; k < 4; ++k)  // 32 keys per instruction: 8 TMEM columns of P codes
            mma_f8_ts(tmem + kColO[t], tmem + kColS[t] + 8 * k, b + 2 * k, kId,
                      (j > 0 || k > 0) ? 1u : 0u);
          mma_commit(bar(Lay::bPV + t));
          if (j == n_kv[t] - 1) mma_commit(bar(Lay::bOD + t));
        }
        __syncwarp();
        if (j + 1 < n_kv[t]) {
          if (!(ok = wait_k(j + 1))) break;
          if (!(ok = mbar_wait_spin_warp(bar(Lay::bPV + t), static_cast<uint32_t>(j) & 1u, wc, 1, 7)))
            break;
          tc_fence_after();
          if (lane == 0) issue_s(t, j + 1);
          __syncwarp();
        }
      }
      if (!ok) break;
      if (lane == 0) {
        mma_commit(bar(Lay::bVE + sv));
        if (j + 1 < n_max) mma_commit(bar(Lay::bKE + (j + 1) % kFp8StagesK));
      }
      __syncwarp();
    }
    if (!ok) {
      if (lane == 0) mma_commit(bar(Lay::bDR));
      __syncwarp();
      mbar_wait_drain(bar(Lay::bDR), 0);
    }
  } else {
    // ================================================================ softmax
    const int t = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int qt = 2 * pt + t;
    const int row = qt * kBM + r;
    const int n = n_kv[t];
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t s_col = t_lane + kColS[t];
    const uint32_t o_col = t_lane + kColO[t];
    const float* sk = p.sk + static_cast<size_t>(z) * p.n_tiles;
    const float* svs = p.sv + static_cast<size_t>(z) * p.n_tiles;
    const float cq = (n > 0 ? p.sq[static_cast<size_t>(z) * p.n_tiles + qt] : 0.f) * p.scale_log2;
    float sv_max = 0.f;
    for (int i = 0; i < p.n_tiles; ++i) sv_max = fmaxf(sv_max, __ldg(svs + i));
    const float fv = kFp8PScale / sv_max;
    float m2 = -INFINITY;
    float le[4] = {0.f, 0.f, 0.f, 0.f};
    bool ok = true;
    float c_next = n > 0 ? cq * __ldg(sk) : 0.f;
    float f_next = n > 0 ? fv * __ldg(svs) : 0.f;
    for (int j = 0; j < n; ++j) {
      const float c = c_next, f = f_next;
      if (j + 1 < n) {  // the next tile's scales, loaded ahead
        c_next = cq * __ldg(sk + j + 1);
        f_next = fv * __ldg(svs + j + 1);
      }
      if (!(ok = mbar_wait_warp(bar(Lay::bSF + t), static_cast<uint32_t>(j) & 1u, wc, 2, 8)))
        break;
      tc_fence_after();
      uint32_t u0[32], u1[32], u2[32], u3[32];
      tmem_ld32(s_col + 0, u0);
      tmem_ld32(s_col + 32, u1);
      tmem_ld32(s_col + 64, u2);
      tmem_ld32(s_col + 96, u3);
      tmem_wait_ld_regs(u0);
      tmem_wait_ld_regs(u1);
      tmem_wait_ld_regs(u2);
      tmem_wait_ld_regs(u3);
      float s[128];
      #pragma unroll
      for (int i = 0; i < 32; ++i) {
        s[i] = u2f(u0[i]);
        s[32 + i] = u2f(u1[i]);
        s[64 + i] = u2f(u2[i]);
        s[96 + i] = u2f(u3[i]);
      }
      const int key0 = j * kBN;
      if ((CAUSAL && j == qt) || key0 + kBN > seq_len) {
        const int lim = CAUSAL ? min(seq_len - key0, row - key0 + 1) : (seq_len - key0);
        #pragma unroll
        for (int cc = 0; cc < kBN; ++cc) s[cc] = (cc < lim) ? s[cc] : -INFINITY;
      }
      float mx[8];
      #pragma unroll
      for (int k = 0; k < 8; ++k) mx[k] = s[k];
      #pragma unroll
      for (int cc = 8; cc + 16 <= kBN; cc += 16)  // pairs of 8-key groups: keys 8 .. kBN - 9
        #pragma unroll
        for (int k = 0; k < 8; ++k) mx[k] = fmax3(mx[k], s[cc + k], s[cc + 8 + k]);
      #pragma unroll
      for (int k = 0; k < 8; ++k) mx[k] = fmaxf(mx[k], s[kBN - 8 + k]);  // the last 8 keys
      const float mt = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]),
                             fmaxf(mx[6], mx[7])) * c;
      const float m_new = (mt > m2 + kFp8Tau) ? mt : m2;
      const bool moved = (m_new != m2);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = moved ? ex2_approx(m2 - m_use) : 1.f;
      m2 = m_new;
      if (moved) {
        #pragma unroll
        for (int k = 0; k < 4; ++k) le[k] *= alpha;
      }
      // P = 2^(s c - m); codes of P * f, four keys per 32-bit TMEM column
      // the weights P * f = 2^(s c - m + log2 f) come out of the exponential directly; the row
      // sums take them back to P with one multiplication per tile
      const float lf = log2f(f);
      const float neg_m = lf - m_use;
      uint32_t pk[32];
      float ts[4] = {0.f, 0.f, 0.f, 0.f};
      #pragma unroll
      for (int i = 0; i < 32; ++i) {
        float x0, x1, x2, x3;
        ffma2(x0, x1, s[4 * i], s[4 * i + 1], c, c, neg_m, neg_m);
        ffma2(x2, x3, s[4 * i + 2], s[4 * i + 3], c, c, neg_m, neg_m);
        const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
        const float p2 = ex2_approx(x2), p3 = ex2_approx(x3);
        fadd2(ts[2 * (i & 1)], ts[2 * (i & 1) + 1], p0, p1);
        fadd2(ts[2 * (i & 1)], ts[2 * (i & 1) + 1], p2, p3);
        pk[i] = static_cast<uint32_t>(pack_e4m3x2(p0, p1)) |
                (static_cast<uint32_t>(pack_e4m3x2(p2, p3)) << 16);
      }
      tmem_st32(s_col, pk);
      const float inv_f = ex2_approx(-lf);
      #pragma unroll
      for (int k = 0; k < 4; ++k) le[k] = fmaf(ts[k], inv_f, le[k]);
      if (j > 0 && __any_sync(0xffffffffu, moved)) {
        #pragma unroll
        for (int cc = 0; cc < 128 / 32; ++cc) {
          uint32_t o[32];
          tmem_ld32(o_col + cc * 32, o);
          tmem_wait_ld_regs(o);
          #pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = f2u(u2f(o[i]) * alpha);
          tmem_st32(o_col + cc * 32, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane_id_is_zero()) mbar_arrive(bar(Lay::bPF + t));
    }
    if (n > 0 && ok) ok = mbar_wait_warp(bar(Lay::bOD + t), 0, wc, 2, 9);
    if (n > 0 && ok) {
      // O / l in bf16 through a staging area of this warp's own: 32 rows of 256 bytes, 16-byte
      // chunks XOR-swizzled by row (no bank conflicts); every store instruction of the warp then
      // writes two whole rows (a row per thread would touch 32 separate lines)
      tc_fence_after();
      const float l = (le[0] + le[1]) + (le[2] + le[3]);
      const bool valid = row < seq_len;
      const float mul = 1.f / (fv * l);  // sv_max / (kFp8PScale l)
      const uint32_t stage = sbase + Lay::kOut + static_cast<uint32_t>(warp - 2) * (32 * 256);
      const uint8_t* stage_p = smem + Lay::kOut + (warp - 2) * (32 * 256);
      #pragma unroll
      for (int cc = 0; cc < 4; cc += 2) {
        uint32_t o[2][32];
        tmem_ld32(o_col + cc * 32, o[0]);
        tmem_ld32(o_col + cc * 32 + 32, o[1]);
        tmem_wait_ld_regs(o[0]);
        tmem_wait_ld_regs(o[1]);
        #pragma unroll
        for (int hh = 0; hh < 2; ++hh)
          #pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int chunk = (cc + hh) * 4 + q;
            const uint32_t* w = o[hh] + 8 * q;
            st_shared_v4(stage + lane * 256 + ((chunk ^ (lane & 7)) << 4),
                         pack_bf16x2(u2f(w[0]) * mul, u2f(w[1]) * mul),
                         pack_bf16x2(u2f(w[2]) * mul, u2f(w[3]) * mul),
                         pack_bf16x2(u2f(w[4]) * mul, u2f(w[5]) * mul),
                         pack_bf16x2(u2f(w[6]) * mul, u2f(w[7]) * mul));
          }
      }
      __syncwarp();
      const int row0 = qt * kBM + quarter * 32;  // this warp's first row within the sequence
      __nv_bfloat16* obase =
          p.o + (static_cast<size_t>(z) * static_cast<size_t>(p.N) + static_cast<size_t>(row0)) *
                    128;
      #pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int rr = 2 * i + (lane >> 4), chunk = lane & 15;
        if (row0 + rr < seq_len) {
          const uint4 val =
              *reinterpret_cast<const uint4*>(stage_p + rr * 256 + ((chunk ^ (rr & 7)) << 4));
          *reinterpret_cast<uint4*>(obase + static_cast<size_t>(rr) * 128 + chunk * 8) = val;
        }
      }
      if (valid) {
        const size_t grow = static_cast<size_t>(z) * static_cast<size_t>(p.N) +
                            static_cast<size_t>(row);
        p.lse[grow] = (m2 + log2f(l)) * 0.69314718055994530942f;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace attn
