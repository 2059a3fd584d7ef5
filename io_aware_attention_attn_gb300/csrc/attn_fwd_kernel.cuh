// attn_fwd_kernel.cuh -- fused IO-aware attention forward for sm_103a (GB300).
//
// One CTA owns one 128-row tile of queries of one (sequence, head).  It keeps the Q tile in
// shared memory, streams 128-row K and V tiles through a TMA-fed ring, and never writes the score
// matrix to HBM: the tiled loop and online softmax of the FlashAttention forward (CS336 Lecture 5
// notes, section 6.2; block merge of the CS336 GPU/attention notes, "Online softmax 回顾").
//
// Warp roles (192 threads):
//   warp 0      TMA producer: Q once, then K_j and V_j into two-stage rings (mbarrier tx counts)
//   warp 1      MMA issuer (one elected lane): S_j = Q K_j^T into tensor memory (double buffered),
//               then O += P_j V_j into a tensor-memory accumulator; owns the TMEM allocation
//   warps 2..5  softmax: one query row per thread (the row is the TMEM lane the warp may access);
//               loads S_j, masks diagonal/tail tiles, keeps the running max m and sums l, writes
//               P_j (bf16) to a double-buffered shared tile, rescales O when the max grows, and at
//               the end writes O / l (bf16) and lse = m + ln l (fp32)
//
// Tensor memory (512 columns x 128 lanes, fp32): S buffers at columns 0 and 128, O at column 256.
// Scores stay in the exp2 domain: t = s * scale * log2(e), p = 2^(t - m).  The running max is
// only moved when a tile raises it by more than kTau (in log2 units); O and l always share the
// same reference max, so O / l is unchanged by that choice (the correction factor of the pages'
// algorithm is applied exactly when the reference moves).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "attn_params.h"
#include "sm103_ptx.cuh"

namespace attn {

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }

template <int D, bool CAUSAL, bool VARLEN>
__global__ void __launch_bounds__(kFwdThreads, 1)
    attn_fwd_kernel(const __grid_constant__ FwdParams p) {
  using Lay = FwdLayout<D>;
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
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(Lay::bKF + s), 1);
      mbar_init(bar(Lay::bKE + s), 1);
      mbar_init(bar(Lay::bVF + s), 1);
      mbar_init(bar(Lay::bVE + s), 1);
    }
    mbar_init(bar(Lay::bSF + 0), 1);
    mbar_init(bar(Lay::bSF + 1), 1);
    mbar_init(bar(Lay::bPF), 4 * 32);
    mbar_init(bar(Lay::bOD), 1);
    mbar_init(bar(Lay::bDR), 1);
    fence_barrier_init();
    misc[1] = 0;
  }

  // ---- which tile this CTA owns: (z = head slice of the tensor map, y0 = first row of the
  // sequence along the map's row axis, seq_len, qt = query tile within the sequence)
  int z, y0, seq_len, qt;
  if constexpr (!VARLEN) {
    const int BH = p.B * p.H;
    const int L = blockIdx.x;
    if constexpr (CAUSAL) {  // heaviest tiles (most key tiles) first
      qt = p.n_qt - 1 - L / BH;
      z = L % BH;
    } else {                 // all tiles of a head together: K and V of that head stay in L2
      z = L / p.n_qt;
      qt = L % p.n_qt;
    }
    y0 = 0;
    seq_len = p.N;
  } else {
    if (warp == 0) {
      // tile slot t of head h -> (sequence, tile) by a warp-wide scan of the per-sequence tile
      // counts; cu_seqlens entries are clamped to [0, N] so no write leaves the buffers
      int remaining = blockIdx.x / p.H;
      int f_start = 0, f_len = 0, f_qt = -1;
      for (int base = 0; base < p.B; base += 32) {
        const int s = base + lane;
        int start = 0, len = 0;
        if (s < p.B) {
          int a = __ldg(p.cu_seqlens + s), b = __ldg(p.cu_seqlens + s + 1);
          a = min(max(a, 0), p.N);
          b = min(max(b, a), p.N);
          start = a;
          len = b - a;
        }
        const int nt = (len + kBM - 1) / kBM;
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
          const int src = hit ? __ffs(hit) - 1 : 0;
          const int q_tile = remaining - __shfl_sync(0xffffffffu, excl, src);
          f_start = __shfl_sync(0xffffffffu, start, src);
          f_len = __shfl_sync(0xffffffffu, len, src);
          f_qt = hit ? q_tile : -1;
          break;
        }
        remaining -= total;
      }
      if (lane == 0) {
        misc[2] = static_cast<uint32_t>(f_start);
        misc[3] = static_cast<uint32_t>(f_len);
        misc[4] = static_cast<uint32_t>(f_qt);
      }
    }
  }
  __syncthreads();
  if constexpr (VARLEN) {
    y0 = static_cast<int>(misc[2]);
    seq_len = static_cast<int>(misc[3]);
    qt = static_cast<int>(misc[4]);
    z = blockIdx.x % p.H;
    if (qt < 0) return;  // slot beyond the last tile of the batch (uniform for the CTA)
  }

  if (warp == 1) {
    tmem_alloc(sbase + Lay::kMisc, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  constexpr uint32_t kColS = 0, kColO = 256;

  const int n_kv = CAUSAL ? (qt + 1) : (seq_len + kBN - 1) / kBN;

  if (warp == 0) {
    // ===================================================================== TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      const uint64_t keep = l2_policy_evict_last();   // K/V are re-read by every query tile
      const uint64_t once = l2_policy_evict_first();  // Q is read once
      mbar_arrive_expect_tx(bar(Lay::bQ), Lay::kTile);
      #pragma unroll
      for (int c = 0; c < D / 64; ++c)
        tma_load_3d_hint(sbase + Lay::kQ + c * 16384, &p.tm_q, bar(Lay::bQ), c * 64,
                         y0 + qt * kBM, z, once);
      int nk = 0, nv = 0;
      bool ok = true;
      for (int j = 0; j < n_kv; ++j) {
        const int st = j % kStages;
        const uint32_t ph = static_cast<uint32_t>(j / kStages) & 1u;
        if (j >= kStages && !(ok = mbar_wait(bar(Lay::bKE + st), ph ^ 1u, wc, 0, 1))) break;
        mbar_arrive_expect_tx(bar(Lay::bKF + st), Lay::kTile);
        #pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d_hint(sbase + Lay::kK + st * Lay::kTile + c * 16384, &p.tm_k,
                           bar(Lay::bKF + st), c * 64, y0 + j * kBN, z, keep);
        ++nk;
        if (j >= kStages && !(ok = mbar_wait(bar(Lay::bVE + st), ph ^ 1u, wc, 0, 2))) break;
        mbar_arrive_expect_tx(bar(Lay::bVF + st), Lay::kTile);
        #pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d_hint(sbase + Lay::kV + st * Lay::kTile + c * 16384, &p.tm_v,
                           bar(Lay::bVF + st), c * 64, y0 + j * kBN, z, keep);
        ++nv;
      }
      if (!ok) {  // unwinding: let every copy still in flight land before the CTA exits
        mbar_wait_drain(bar(Lay::bQ), 0);
        for (int j = (nk > kStages ? nk - kStages : 0); j < nk; ++j)
          mbar_wait_drain(bar(Lay::bKF + j % kStages), static_cast<uint32_t>(j / kStages) & 1u);
        for (int j = (nv > kStages ? nv - kStages : 0); j < nv; ++j)
          mbar_wait_drain(bar(Lay::bVF + j % kStages), static_cast<uint32_t>(j / kStages) & 1u);
      }
    }
  } else if (warp == 1) {
    // ===================================================================== MMA issuer
    constexpr uint32_t kIdS = idesc_bf16_f32(kBM, kBN, false, false);  // Q, K both K-major
    constexpr uint32_t kIdO = idesc_bf16_f32(kBM, D, false, true);     // P K-major, V MN-major
    auto issue_s = [&](int j) -> bool {
      const int st = j % kStages;
      if (!mbar_wait_warp(bar(Lay::bKF + st), static_cast<uint32_t>(j / kStages) & 1u, wc, 1, 3))
        return false;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t d_tmem = tmem + kColS + static_cast<uint32_t>(j & 1) * kBN;
        #pragma unroll
        for (int t = 0; t < D / 16; ++t) {  // K = 16 per instruction; 4 steps per 128-byte row
          const uint32_t off = static_cast<uint32_t>((t >> 2) * 16384 + (t & 3) * 32);
          mma_bf16_ss(d_tmem, sdesc_sw128(sbase + Lay::kQ + off, 16, 1024),
                      sdesc_sw128(sbase + Lay::kK + st * Lay::kTile + off, 16, 1024), kIdS,
                      t > 0 ? 1u : 0u);
        }
        mma_commit(bar(Lay::bSF + (j & 1)));
        mma_commit(bar(Lay::bKE + st));
      }
      __syncwarp();
      return true;
    };
    bool ok = mbar_wait_warp(bar(Lay::bQ), 0, wc, 1, 4);
    if (ok) ok = issue_s(0);
    for (int j = 0; ok && j < n_kv; ++j) {
      if (j + 1 < n_kv && !(ok = issue_s(j + 1))) break;
      if (!(ok = mbar_wait_warp(bar(Lay::bPF), static_cast<uint32_t>(j) & 1u, wc, 1, 5))) break;
      const int st = j % kStages;
      if (!(ok = mbar_wait_warp(bar(Lay::bVF + st), static_cast<uint32_t>(j / kStages) & 1u,
                           wc, 1, 6)))
        break;
      if constexpr (VARLEN) {
        // rows of the last V tile past the end of the sequence belong to the next sequence:
        // zero them so that P = 0 there cannot meet a non-finite value
        const int valid = seq_len - j * kBN;
        if (valid < kBN) {
          const uint32_t vbase = sbase + Lay::kV + st * Lay::kTile;
          #pragma unroll
          for (int c = 0; c < D / 64; ++c)
            for (int i = valid * 8 + lane; i < kBN * 8; i += 32)
              st_shared_v4(vbase + c * 16384 + i * 16, 0u, 0u, 0u, 0u);
          fence_proxy_async_smem();
        }
      }
      __syncwarp();
      tc_fence_after();
      if (lane == 0) {
        const uint32_t p_base = sbase + Lay::kP + static_cast<uint32_t>(j & 1) * Lay::kPTile;
        const uint32_t v_base = sbase + Lay::kV + st * Lay::kTile;
        #pragma unroll
        for (int t = 0; t < kBN / 16; ++t) {
          const uint32_t a_off = static_cast<uint32_t>((t >> 2) * 16384 + (t & 3) * 32);
          mma_bf16_ss(tmem + kColO, sdesc_sw128(p_base + a_off, 16, 1024),
                      sdesc_sw128(v_base + t * 2048, 16384, 1024), kIdO,
                      (j > 0 || t > 0) ? 1u : 0u);
        }
        mma_commit(bar(Lay::bOD));
        mma_commit(bar(Lay::bVE + st));
      }
      __syncwarp();
    }
    if (!ok) {  // unwinding: wait for every MMA already issued
      if (lane == 0) mma_commit(bar(Lay::bDR));
      __syncwarp();
      mbar_wait_drain(bar(Lay::bDR), 0);
    }
  } else {
    // ===================================================================== softmax
    const int quarter = warp & 3;  // TMEM lanes this warp may access: 32*quarter .. +31
    const int r = quarter * 32 + lane;  // row of the tile = TMEM lane
    const int row = qt * kBM + r;       // row within the sequence
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float sl2 = p.scale_log2;
    float m2 = -INFINITY;    // reference max of the scaled scores (log2 units)
    float l_exact = 0.f;     // sum of 2^(t - m2) in fp32 (for lse)
    float l_round = 0.f;     // sum of the same values after rounding to bf16 (for O)
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      if (!(ok = mbar_wait_warp(bar(Lay::bSF + (j & 1)), static_cast<uint32_t>(j >> 1) & 1u,
                           wc, 2, 7)))
        break;
      tc_fence_after();
      uint32_t s0[32], s1[32], s2[32], s3[32];
      const uint32_t sa = t_lane + kColS + static_cast<uint32_t>(j & 1) * kBN;
      tmem_ld32(sa + 0, s0);
      tmem_ld32(sa + 32, s1);
      tmem_ld32(sa + 64, s2);
      tmem_ld32(sa + 96, s3);
      tmem_wait_ld_regs(s0);
      tmem_wait_ld_regs(s1);
      tmem_wait_ld_regs(s2);
      tmem_wait_ld_regs(s3);
      float s[128];
      #pragma unroll
      for (int i = 0; i < 32; ++i) {
        s[i] = u2f(s0[i]);
        s[32 + i] = u2f(s1[i]);
        s[64 + i] = u2f(s2[i]);
        s[96 + i] = u2f(s3[i]);
      }
      const int key0 = j * kBN;
      if ((CAUSAL && j == qt) || key0 + kBN > seq_len) {
        const int lim = CAUSAL ? min(seq_len - key0, row - key0 + 1) : (seq_len - key0);
        #pragma unroll
        for (int c = 0; c < kBN; ++c) s[c] = (c < lim) ? s[c] : -INFINITY;
      }
      float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
      #pragma unroll
      for (int c = 4; c < kBN; c += 4) {
        mx0 = fmaxf(mx0, s[c]);
        mx1 = fmaxf(mx1, s[c + 1]);
        mx2 = fmaxf(mx2, s[c + 2]);
        mx3 = fmaxf(mx3, s[c + 3]);
      }
      const float mt = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl2;
      const float m_new = (mt > m2 + kTau) ? mt : m2;
      const bool moved = (m_new != m2);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = moved ? ex2_approx(m2 - m_use) : 1.f;
      m2 = m_new;

      // P_j = 2^(t - m) -> bf16, written into the 128-byte-swizzled K-major tile the PV MMA reads
      const uint32_t prow = sbase + Lay::kP + static_cast<uint32_t>(j & 1) * Lay::kPTile +
                            static_cast<uint32_t>(r) * 128u;
      float se0 = 0.f, se1 = 0.f, sr0 = 0.f, sr1 = 0.f;
      #pragma unroll
      for (int c = 0; c < kBN / 8; ++c) {
        uint32_t pk[4];
        #pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float a = ex2_approx(fmaf(s[8 * c + 2 * e], sl2, -m_use));
          const float b = ex2_approx(fmaf(s[8 * c + 2 * e + 1], sl2, -m_use));
          se0 += a;
          se1 += b;
          pk[e] = pack_bf16x2(a, b);
          sr0 += bf16lo_to_f32(pk[e]);
          sr1 += bf16hi_to_f32(pk[e]);
        }
        const uint32_t chunk = static_cast<uint32_t>(c & 7) ^ static_cast<uint32_t>(r & 7);
        st_shared_v4(prow + static_cast<uint32_t>(c >> 3) * 16384u + (chunk << 4), pk[0], pk[1],
                     pk[2], pk[3]);
      }
      fence_proxy_async_smem();
      l_exact = l_exact * alpha + (se0 + se1);
      l_round = l_round * alpha + (sr0 + sr1);

      if (j > 0) {
        // O must hold P_{j-1} V_{j-1} before it is rescaled for the new reference max
        if (!(ok = mbar_wait_warp(bar(Lay::bOD), static_cast<uint32_t>(j - 1) & 1u, wc, 2, 8)))
          break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, moved)) {
          #pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(t_lane + kColO + c * 32, o);
            tmem_wait_ld_regs(o);
            #pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = f2u(u2f(o[i]) * alpha);
            tmem_st32(t_lane + kColO + c * 32, o);
          }
          tmem_wait_st();
        }
      }
      tc_fence_before();
      mbar_arrive(bar(Lay::bPF));
    }
    if (ok) ok = mbar_wait_warp(bar(Lay::bOD), static_cast<uint32_t>(n_kv - 1) & 1u, wc, 2, 9);
    if (ok) {
      tc_fence_after();
      const bool valid = row < seq_len;
      const float inv_l = 1.f / l_round;
      const size_t grow = static_cast<size_t>(z) * static_cast<size_t>(p.N) +
                          static_cast<size_t>(y0) + static_cast<size_t>(row);
      uint4* orow = reinterpret_cast<uint4*>(p.o + grow * D);
      #pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(t_lane + kColO + c * 32, o);
        tmem_wait_ld_regs(o);
        uint32_t pk[16];
        #pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack_bf16x2(u2f(o[2 * i]) * inv_l, u2f(o[2 * i + 1]) * inv_l);
        if (valid) {
          #pragma unroll
          for (int q = 0; q < 4; ++q)
            orow[c * 4 + q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
      }
      if (valid) p.lse[grow] = (m2 + log2f(l_exact)) * 0.69314718055994530942f;
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
