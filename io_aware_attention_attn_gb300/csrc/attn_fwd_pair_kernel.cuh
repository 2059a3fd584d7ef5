// attn_fwd_pair_kernel.cuh -- fused IO-aware attention forward for sm_103a (GB300), two query
// tiles per CTA.
//
// One CTA owns two adjacent 128-row query tiles (t = 0, 1) of one (sequence, head).  Both tiles
// share every K and V tile the TMA producer streams through shared memory, so K/V traffic per
// FLOP is half that of one tile per CTA.  The score matrix never leaves the chip: the tiled loop
// and online softmax of the FlashAttention forward (CS336 Lecture 5 notes, section 6.2; the block
// merge of the CS336 GPU/attention notes, "Online softmax 回顾").
//
// Warp roles (320 threads):
//   warp 0      TMA producer: Q0 and Q1 once, then K_j and V_j into two-stage rings
//   warp 1      MMA issuer (lane 0) and TMEM owner.  Per key tile j and query tile t:
//               S_t = Q_t K_j^T into tensor memory, then O_t += P_t V_j with P_t read from tensor
//               memory (the A operand of the MMA) and V_j from shared memory
//   warps 2..5  softmax of tile 0, warps 6..9 softmax of tile 1: one query row per thread (the
//               TMEM lane its warp may access).  The two warpgroups work on different tiles at
//               once, so one tile's softmax overlaps the other tile's MMAs.
//
// Tensor memory (512 columns): S_0 at 0, S_1 at 128 (fp32 128 x 128), O_0 at 256, O_1 at 256 + D.
// P_t (bf16, two per column) overwrites the first 64 columns of S_t once the softmax has read S_t.
// The next S_t product rewrites those columns, so the MMA warp waits for the P_t V product to
// complete (a commit barrier) before issuing it: tcgen05 MMAs with different accumulators are not
// ordered with respect to each other.
//
// Softmax in the exp2 domain: t = s * scale * log2(e), p = 2^(t - m).  The reference m is a row
// maximum of some earlier tile; a tile is first exponentiated against it, and the tile's maximum
// is taken (and m moved to it, O and l rescaled) only on the first tile or when the tile's row sum
// exceeds kSumLimit.  O and l always share the reference, so O / l is unchanged.  O is divided by, and lse takes, the fp32 sum of the unrounded P.
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
__global__ void __launch_bounds__(kPairThreads, 1)
    attn_fwd_pair_kernel(const __grid_constant__ FwdParams p) {
  using Lay = PairLayout<D>;
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
    for (int s = 0; s < kPairStagesK; ++s) {
      mbar_init(bar(Lay::bKF + s), 1);
      mbar_init(bar(Lay::bKE + s), 1);
    }
    for (int s = 0; s < kPairStagesV; ++s) {
      mbar_init(bar(Lay::bVF + s), 1);
      mbar_init(bar(Lay::bVE + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(Lay::bSF + t), 1);
      mbar_init(bar(Lay::bPF + t), 4 * 32);
      mbar_init(bar(Lay::bPV + t), 1);
      mbar_init(bar(Lay::bOD + t), 1);
    }
    mbar_init(bar(Lay::bDR), 1);
    fence_barrier_init();
    misc[1] = 0;
  }

  // ---- which pair of query tiles this CTA owns: z = head slice of the tensor maps, y0 = first row
  // of the sequence along the maps' row axis, pt = pair index within the sequence
  int z, y0, seq_len, pt;
  // split-KV (dense only): consecutive CTAs are the slices of one query pair
  const int split = VARLEN ? 0 : static_cast<int>(blockIdx.x) % p.n_splits;
  if constexpr (!VARLEN) {
    const int BH = p.B * p.H;
    const int L = static_cast<int>(blockIdx.x) / p.n_splits;
    if constexpr (CAUSAL) {  // heaviest pairs (most key tiles) first
      pt = p.n_qt - 1 - L / BH;
      z = L % BH;
    } else {                 // all pairs of a head together: its K and V stay in L2
      z = L / p.n_qt;
      pt = L % p.n_qt;
    }
    y0 = 0;
    seq_len = p.N;
  } else {
    if (warp == 0) {
      // slot -> (sequence, pair) by a warp-wide scan of the per-sequence pair counts; entries of
      // cu_seqlens are clamped to [0, N] so no access leaves the buffers
      int remaining = blockIdx.x / p.H;
      int f_start = 0, f_len = 0, f_pt = -1;
      if (blockIdx.x == 0) {
        // one CTA checks that cu_seqlens is a prefix sum from 0 to N (non-decreasing); a bad one
        // is reported through the status word, and every CTA works on offsets clamped into [0, N]
        bool bad = false;
        for (int s = lane; s < p.B; s += 32) {
          const int a = __ldg(p.cu_seqlens + s), b = __ldg(p.cu_seqlens + s + 1);
          bad |= (b < a) || (s == 0 && a != 0) || (s == p.B - 1 && b != p.N);
        }
        if (__any_sync(0xffffffffu, bad) && lane == 0) atomicCAS(p.status, 0, kStatusBadSeqlens);
      }
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
        const int nt = (len + 2 * kBM - 1) / (2 * kBM);
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
          const int pair = remaining - __shfl_sync(0xffffffffu, excl, src);
          f_start = __shfl_sync(0xffffffffu, start, src);
          f_len = __shfl_sync(0xffffffffu, len, src);
          f_pt = hit ? pair : -1;
          break;
        }
        remaining -= total;
      }
      if (lane == 0) {
        misc[2] = static_cast<uint32_t>(f_start);
        misc[3] = static_cast<uint32_t>(f_len);
        misc[4] = static_cast<uint32_t>(f_pt);
      }
    }
  }
  __syncthreads();
  if constexpr (VARLEN) {
    y0 = static_cast<int>(misc[2]);
    seq_len = static_cast<int>(misc[3]);
    pt = static_cast<int>(misc[4]);
    z = blockIdx.x % p.H;
    if (pt < 0) return;  // slot beyond the last pair of the batch (uniform for the CTA)
  }

  // key tiles each query tile visits (0 if the tile starts past the end of the sequence); with
  // split-KV this CTA takes key tiles [kb, kb + chunk) of the pair's range, and n_kv[t] counts
  // the tiles of that slice query tile t visits.  Pipeline bookkeeping runs over j = 0..n_kv-1;
  // key tile kb + j is the data.
  const int n_keytiles = (seq_len + kBN - 1) / kBN;
  int n_full[2];
  #pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int qt = 2 * pt + t;
    n_full[t] = (qt * kBM >= seq_len) ? 0 : (CAUSAL ? qt + 1 : n_keytiles);
  }
  const int n_full_max = n_full[0] > n_full[1] ? n_full[0] : n_full[1];
  const int chunk = (n_full_max + p.n_splits - 1) / p.n_splits;
  const int kb = split * chunk;
  int n_kv[2];
  #pragma unroll
  for (int t = 0; t < 2; ++t) n_kv[t] = max(0, min(kb + chunk, n_full[t]) - kb);
  const int n_max = n_kv[0] > n_kv[1] ? n_kv[0] : n_kv[1];
  if (!VARLEN && p.n_splits > 1 && n_max == 0) {
    // a key slice past the end of this pair's range: nothing to load or multiply; the merge
    // reads max -inf and sums 0 for its rows (uniform for the CTA, before any copy is issued)
    const size_t rows_total = static_cast<size_t>(p.B) * p.H * p.N;
    const size_t plane = static_cast<size_t>(p.n_splits) * rows_total;
    const int row = 2 * pt * kBM + static_cast<int>(threadIdx.x);
    if (threadIdx.x < 2 * kBM && row < seq_len) {
      const size_t slot = static_cast<size_t>(split) * rows_total +
                          static_cast<size_t>(z) * static_cast<size_t>(p.N) + row;
      p.part_stat[slot] = -INFINITY;
      p.part_stat[plane + slot] = 0.f;
    }
    return;
  }

  if (warp == 1) {
    tmem_alloc(sbase + Lay::kMisc, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  constexpr uint32_t kColS[2] = {0, 128};
  constexpr uint32_t kColO[2] = {256, 256 + D};

  // K/V head slice: query head h reads K/V head h / group (grouped-query attention); dense maps
  // are indexed by batch * heads + head, packed maps by head
  const int z_kv = VARLEN ? z / p.group : (z / p.H) * (p.H / p.group) + (z % p.H) / p.group;

  if (warp == 0) {
    // ===================================================================== TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      const uint64_t keep = l2_policy_evict_last();   // K/V are re-read by every query pair
      const uint64_t once = l2_policy_evict_first();  // Q is read once
      mbar_arrive_expect_tx(bar(Lay::bQ), 2 * Lay::kTile);
      #pragma unroll
      for (int t = 0; t < 2; ++t)
        #pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d_hint(sbase + Lay::kQ + t * Lay::kTile + c * 16384, &p.tm_q, bar(Lay::bQ),
                           c * 64, y0 + (2 * pt + t) * kBM, z, once);
      int nk = 0, nv = 0;
      bool ok = true;
      for (int j = 0; j < n_max; ++j) {
        const int sk = j % kPairStagesK, sv = j % kPairStagesV;
        if (j >= kPairStagesK &&
            !(ok = mbar_wait(bar(Lay::bKE + sk),
                             (static_cast<uint32_t>(j / kPairStagesK) & 1u) ^ 1u, wc, 0, 1)))
          break;
        mbar_arrive_expect_tx(bar(Lay::bKF + sk), Lay::kTile);
        #pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d_hint(sbase + Lay::kK + sk * Lay::kTile + c * 16384, &p.tm_k,
                           bar(Lay::bKF + sk), c * 64, y0 + (kb + j) * kBN, z_kv, keep);
        ++nk;
        if (j >= kPairStagesV &&
            !(ok = mbar_wait(bar(Lay::bVE + sv),
                             (static_cast<uint32_t>(j / kPairStagesV) & 1u) ^ 1u, wc, 0, 2)))
          break;
        mbar_arrive_expect_tx(bar(Lay::bVF + sv), Lay::kTile);
        #pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d_hint(sbase + Lay::kV + sv * Lay::kTile + c * 16384, &p.tm_v,
                           bar(Lay::bVF + sv), c * 64, y0 + (kb + j) * kBN, z_kv, keep);
        ++nv;
      }
      if (!ok) {  // unwinding: let every copy still in flight land before the CTA exits
        mbar_wait_drain(bar(Lay::bQ), 0);
        for (int j = (nk > kPairStagesK ? nk - kPairStagesK : 0); j < nk; ++j)
          mbar_wait_drain(bar(Lay::bKF + j % kPairStagesK),
                          static_cast<uint32_t>(j / kPairStagesK) & 1u);
        for (int j = (nv > kPairStagesV ? nv - kPairStagesV : 0); j < nv; ++j)
          mbar_wait_drain(bar(Lay::bVF + j % kPairStagesV),
                          static_cast<uint32_t>(j / kPairStagesV) & 1u);
      }
    }
  } else if (warp == 1) {
    // ===================================================================== MMA issuer
    constexpr uint32_t kIdS = idesc_bf16_f32(kBM, kBN, false, false);  // Q, K both K-major
    constexpr uint32_t kIdO = idesc_bf16_f32(kBM, D, false, true);     // P (TMEM), V MN-major
    // Operand descriptors are built once; every MMA adds a compile-time offset to the 14-bit
    // start-address field (shared addresses stay below 256 KB, so the add never carries out of
    // it).  Recomputing them per instruction made the single issuing thread, not the tensor pipe,
    // the bottleneck.
    constexpr uint64_t kTileD = static_cast<uint64_t>(Lay::kTile >> 4);
    const uint64_t desc_q = sdesc_sw128(sbase + Lay::kQ, 16, 1024);
    const uint64_t desc_k = sdesc_sw128(sbase + Lay::kK, 16, 1024);
    const uint64_t desc_v = sdesc_sw128(sbase + Lay::kV, 16384, 1024);
    auto issue_s = [&](int t, int j) {  // S_t = Q_t K_j^T (lane 0 only)
      const uint64_t a = desc_q + static_cast<uint64_t>(t) * kTileD;
      const uint64_t b = desc_k + static_cast<uint64_t>(j % kPairStagesK) * kTileD;
      const uint32_t d = tmem + kColS[t];
      #pragma unroll
      for (int k = 0; k < D / 16; ++k) {  // K = 16 per instruction; 4 steps per 128-byte row
        const uint64_t off = static_cast<uint64_t>(((k >> 2) * 16384 + (k & 3) * 32) >> 4);
        mma_bf16_ss(d, a + off, b + off, kIdS, k > 0 ? 1u : 0u);
      }
      mma_commit(bar(Lay::bSF + t));
    };
    auto wait_k = [&](int j) {
      return mbar_wait_warp(bar(Lay::bKF + j % kPairStagesK),
                            static_cast<uint32_t>(j / kPairStagesK) & 1u, wc, 1, 3);
    };
    bool ok = mbar_wait_warp(bar(Lay::bQ), 0, wc, 1, 4) && wait_k(0);
    if (ok) {
      tc_fence_after();
      if (lane == 0) {
        if (n_kv[0] > 0) issue_s(0, 0);  // a key slice may hold no tile of query tile 0
        if (n_kv[1] > 0) issue_s(1, 0);
        mma_commit(bar(Lay::bKE + 0));
      }
      __syncwarp();
    }
    for (int j = 0; ok && j < n_max; ++j) {
      const int sv = j % kPairStagesV;
      bool v_ready = false;
      #pragma unroll
      for (int t = 0; t < 2; ++t) {
        if (j >= n_kv[t]) continue;
        if (!(ok = mbar_wait_warp(bar(Lay::bPF + t), static_cast<uint32_t>(j) & 1u, wc, 1, 5)))
          break;
        if (!v_ready) {
          if (!(ok = mbar_wait_warp(bar(Lay::bVF + sv),
                                    static_cast<uint32_t>(j / kPairStagesV) & 1u, wc, 1, 6)))
            break;
          v_ready = true;
          if constexpr (VARLEN) {
            // rows of the last V tile past the end of the sequence belong to the next sequence:
            // zero them so that P = 0 there cannot meet a non-finite value
            const int valid = seq_len - (kb + j) * kBN;
            if (valid < kBN) {
              const uint32_t vbase = sbase + Lay::kV + sv * Lay::kTile;
              #pragma unroll
              for (int c = 0; c < D / 64; ++c)
                for (int i = valid * 8 + lane; i < kBN * 8; i += 32)
                  st_shared_v4(vbase + c * 16384 + i * 16, 0u, 0u, 0u, 0u);
              fence_proxy_async_smem();
            }
            __syncwarp();
          }
        }
        tc_fence_after();
        if (lane == 0) {
          const uint64_t b = desc_v + static_cast<uint64_t>(sv) * kTileD;
          const uint32_t d = tmem + kColO[t], a = tmem + kColS[t];
          #pragma unroll
          for (int k = 0; k < kBN / 16; ++k)  // 16 keys (2048 bytes of V) per instruction
            mma_bf16_ts(d, a + k * 8, b + static_cast<uint64_t>(k * (2048 >> 4)), kIdO,
                        (j > 0 || k > 0) ? 1u : 0u);
          mma_commit(bar(Lay::bPV + t));
          if (j == n_kv[t] - 1) mma_commit(bar(Lay::bOD + t));
        }
        __syncwarp();
        if (j + 1 < n_kv[t]) {
          // S_t for the next key tile rewrites the columns P_t was read from: wait for P_t V_j
          if (!(ok = wait_k(j + 1))) break;
          if (!(ok = mbar_wait_warp(bar(Lay::bPV + t), static_cast<uint32_t>(j) & 1u, wc, 1, 7)))
            break;
          tc_fence_after();
          if (lane == 0) issue_s(t, j + 1);
          __syncwarp();
        }
      }
      if (!ok) break;
      if (lane == 0) {
        mma_commit(bar(Lay::bVE + sv));
        if (j + 1 < n_max) mma_commit(bar(Lay::bKE + (j + 1) % kPairStagesK));
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
    const int t = (warp - 2) >> 2;     // query tile of this warpgroup
    const int quarter = warp & 3;      // TMEM lanes this warp may access: 32*quarter .. +31
    const int r = quarter * 32 + lane; // row of the tile = TMEM lane
    const int qt = 2 * pt + t;
    const int row = qt * kBM + r;      // row within the sequence
    const int n = n_kv[t];
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t s_col = t_lane + kColS[t];
    const uint32_t o_col = t_lane + kColO[t];
    const float sl2 = p.scale_log2;
    float m2 = -INFINITY;            // reference max of the scaled scores (log2 units)
    float le[4] = {0.f, 0.f, 0.f, 0.f};  // sums of 2^(t - m), fp32
    bool ok = true;
    for (int j = 0; j < n; ++j) {
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
      const int key0 = (kb + j) * kBN;
      if ((CAUSAL && kb + j == qt) || key0 + kBN > seq_len) {
        const int lim = CAUSAL ? min(seq_len - key0, row - key0 + 1) : (seq_len - key0);
        #pragma unroll
        for (int c = 0; c < kBN; ++c) s[c] = (c < lim) ? s[c] : -INFINITY;
      }
      // P = 2^(t - m) in bf16, two per 32-bit word, over the first 64 columns of S_t (written in
      // two halves so each half's words are dead once stored); ts = this tile's row sums.
      // Pass 0 exponentiates against the current reference; the row maximum is taken (pass 1)
      // only on the first tile or when a row's tile sum exceeds kSumLimit (every P then stays
      // <= kSumLimit).  Both passes are warp-uniform: the TMEM stores are collective.
      float ts[4];
      bool moved = false;
      float alpha = 1.f;
      bool need = (j == 0);
      #pragma unroll 1
      for (int pass = (j == 0) ? 1 : 0; pass < 2; ++pass) {
        float m_use = m2;
        if (pass == 1) {
          float mx[8];
          #pragma unroll
          for (int k = 0; k < 8; ++k) mx[k] = s[k];
          #pragma unroll
          for (int c = 8; c < kBN; c += 16)
            #pragma unroll
            for (int k = 0; k < 8; ++k) mx[k] = fmax3(mx[k], s[c + k], s[c + 8 + k]);
          const float mt = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]),
                                 fmaxf(mx[6], mx[7])) * sl2;
          const float m_new = need ? fmaxf(mt, m2) : m2;
          moved = (m_new != m2);
          m_use = (m_new == -INFINITY) ? 0.f : m_new;
          alpha = moved ? ex2_approx(m2 - m_use) : 1.f;
          m2 = m_new;
          if (moved) {
            #pragma unroll
            for (int k = 0; k < 4; ++k) le[k] *= alpha;
          }
          tmem_wait_st();  // pass 0's stores land before these overwrite them
        }
        const float neg_m = -m_use;
        #pragma unroll
        for (int k = 0; k < 4; ++k) ts[k] = 0.f;
        #pragma unroll
        for (int h = 0; h < 4; ++h) {  // quarters of 32 keys: 16 packed words each
          uint32_t pk[16];
          #pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int c = 32 * h + 2 * i;
            float x0, x1;
            ffma2(x0, x1, s[c], s[c + 1], sl2, sl2, neg_m, neg_m);
            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
            pk[i] = pack_bf16x2(p0, p1);
            fadd2(ts[2 * (i & 1)], ts[2 * (i & 1) + 1], p0, p1);
          }
          tmem_st16(s_col + 16 * h, pk);
        }
        if (pass == 0) {
          need = !(((ts[0] + ts[1]) + (ts[2] + ts[3])) <= kSumLimit);  // also catches inf, NaN
          if (!__any_sync(0xffffffffu, need)) break;
        }
      }
      #pragma unroll
      for (int k = 0; k < 4; ++k) le[k] += ts[k];

      // O_t holds P_t V up to key tile j-1 (that product completed before S_t was rewritten);
      // bring it to the new reference max before P_t V_j is added
      if (j > 0 && __any_sync(0xffffffffu, moved)) {
        #pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(o_col + c * 32, o);
          tmem_wait_ld_regs(o);
          #pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = f2u(u2f(o[i]) * alpha);
          tmem_st32(o_col + c * 32, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(Lay::bPF + t));
    }
    if (n > 0 && ok) ok = mbar_wait_warp(bar(Lay::bOD + t), 0, wc, 2, 9);
    const float l_exact = (le[0] + le[1]) + (le[2] + le[3]);
    const bool valid = row < seq_len;
    const size_t grow = static_cast<size_t>(z) * static_cast<size_t>(p.N) +
                        static_cast<size_t>(y0) + static_cast<size_t>(row);
    if (p.n_splits > 1) {
      // this key slice's partial result for the merge: unnormalised O, reference max and both
      // row sums (a slice without keys for this tile contributes max -inf and sums 0)
      const size_t rows_total = static_cast<size_t>(p.B) * p.H * p.N;
      const size_t slot = static_cast<size_t>(split) * rows_total + grow;
      const size_t plane = static_cast<size_t>(p.n_splits) * rows_total;
      const bool has = n > 0 && ok;
      if (valid) {
        p.part_stat[slot] = has ? m2 : -INFINITY;
        p.part_stat[plane + slot] = has ? l_exact : 0.f;
      }
      if (has) {
        tc_fence_after();
        float4* prow = reinterpret_cast<float4*>(p.part_o + slot * D);
        #pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(o_col + c * 32, o);
          tmem_wait_ld_regs(o);
          if (valid) {
            #pragma unroll
            for (int q = 0; q < 8; ++q)
              prow[c * 8 + q] = make_float4(u2f(o[4 * q]), u2f(o[4 * q + 1]), u2f(o[4 * q + 2]),
                                            u2f(o[4 * q + 3]));
          }
        }
      }
    } else if (n > 0 && ok) {
      // O / l in bf16 through shared memory: every product that read Q_t has completed, so its
      // tile is free, and each of this tile's warps stages its 32 rows there (16-byte chunks
      // XOR-swizzled by row, no bank conflicts); every store instruction of the warp then writes
      // whole 128-byte lines of consecutive rows (a row per thread would touch 32 lines)
      tc_fence_after();
      const float inv_l = 1.f / l_exact;
      constexpr int kChunks = D / 8;  // 16-byte chunks per row
      const uint32_t stage = sbase + Lay::kQ + t * Lay::kTile + quarter * (32 * D * 2);
      const uint8_t* stage_p = smem + Lay::kQ + t * Lay::kTile + quarter * (32 * D * 2);
      #pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(o_col + c * 32, o);
        tmem_wait_ld_regs(o);
        #pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int chunk = c * 4 + q;
          st_shared_v4(stage + lane * (D * 2) + ((chunk ^ (lane & 7)) << 4),
                       pack_bf16x2(u2f(o[8 * q + 0]) * inv_l, u2f(o[8 * q + 1]) * inv_l),
                       pack_bf16x2(u2f(o[8 * q + 2]) * inv_l, u2f(o[8 * q + 3]) * inv_l),
                       pack_bf16x2(u2f(o[8 * q + 4]) * inv_l, u2f(o[8 * q + 5]) * inv_l),
                       pack_bf16x2(u2f(o[8 * q + 6]) * inv_l, u2f(o[8 * q + 7]) * inv_l));
        }
      }
      __syncwarp();
      const int row0 = qt * kBM + quarter * 32;  // this warp's first row within the sequence
      __nv_bfloat16* obase = p.o + (static_cast<size_t>(z) * static_cast<size_t>(p.N) +
                                    static_cast<size_t>(y0) + static_cast<size_t>(row0)) * D;
      #pragma unroll
      for (int i = 0; i < kChunks; ++i) {
        const int rr = i * (32 / kChunks) + lane / kChunks, chunk = lane % kChunks;
        if (row0 + rr < seq_len) {
          const uint4 val = *reinterpret_cast<const uint4*>(stage_p + rr * (D * 2) +
                                                            ((chunk ^ (rr & 7)) << 4));
          *reinterpret_cast<uint4*>(obase + static_cast<size_t>(rr) * D + chunk * 8) = val;
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
