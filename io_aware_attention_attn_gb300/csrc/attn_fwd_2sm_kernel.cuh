// attn_fwd_2sm_kernel.cuh -- fused IO-aware attention forward for sm_103a (GB300), head dim 64
// or 128, dense or packed batches: one 128-row query tile per SM and one tensor-core product
// across the two SMs of a TPC.
//
// A cluster of two CTAs works on 256 consecutive query rows of one (sequence, head) at a time:
// the CTA of rank r holds rows 128 r .. 128 r + 127 of them.  Each product is a single
// cta_group::2 MMA with M = 256 issued by rank 0: S = Q K_j^T takes A (Q) from each CTA's own rows
// and B (K_j) half from each CTA (keys 64 r .. 64 r + 63 of the tile); O += P V_j takes P from
// each CTA's tensor memory and V_j's value columns 64 r .. 64 r + 63 from CTA r (head dim 64:
// all 64 columns from rank 0, rank 1's V stages zero).  So each SM streams half of every K and V
// tile (the same K/V bytes per FLOP as two query tiles in one CTA) and holds one query tile,
// which leaves tensor memory for three S buffers next to O: S_{j+3} can be issued as soon as
// P_j V_j has completed, while the softmax works on S_{j+1} and S_{j+2}.  The tiled loop and
// online softmax are those of the FlashAttention forward (CS336 Lecture 5 notes, section 6.2;
// the block merge of the CS336 GPU/attention notes, "Online softmax 回顾").
//
// The kernel is persistent: the grid holds as many clusters as fit on the GPU at once, and
// cluster c takes the work units c, 2G - 1 - c, 2G + c, 4G - 1 - c, ... of an order that puts
// heavy units first (causal and packed batches) and keeps a head's units together where that
// keeps its K and V in L2 (see unit_of and Walker below).  Q is double-buffered, and the K/V
// rings, the S buffers and every barrier phase run on across units, so the next unit's Q load
// and first S products overlap the current unit's last tiles and epilogue; only its first P V
// waits, for the epilogue to have read O.
//
// Warp roles (224 threads per CTA):
//   warp 0      TMA producer of this CTA's halves: Q per unit, K_j and V_j into four-stage
//               rings.  Completion is counted on rank 0's barriers.
//   warp 1      tensor memory allocation (both CTAs); on rank 0 lane 0 issues the P V products.
//   warps 2..5  softmax: one query row per thread (the TMEM lane its warp may access), and the
//               epilogue of each unit.
//   warp 6      on rank 0 lane 0 issues the S products, up to three key tiles ahead.
//
// Tensor memory (512 columns in each SM): S buffers at 0, 128, 256 (fp32 128 x 128; the g-th key
// tile the cluster processes, counted across units, uses buffer g % 3), O at 384.  P (bf16, two
// per column) overwrites the first 64 columns of its S buffer once the softmax has read it.
//
// Softmax in the exp2 domain with a sum-triggered reference maximum: a tile is exponentiated
// against the row's reference m first, and its maximum is taken (m moved, O and l rescaled) only
// on the first tile or when the tile's row sum exceeds kSumLimit.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "attn_params.h"
#include "sm103_ptx.cuh"

namespace attn {
namespace fwd2sm {

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }

// Spin for about `ns` nanoseconds (unwinding only: lets copies that signal the peer's barriers
// land before this CTA leaves the cluster barrier).
__device__ __forceinline__ void settle(unsigned long long ns) {
  const unsigned long long t0 = global_timer_ns();
  while (global_timer_ns() - t0 < ns) {
  }
}

// One work unit: 256 query rows of a head and a slice of their key tiles.
struct Unit {
  int z;      // head slice of the tensor maps
  int y0;     // first row of the unit's sequence along the maps' row axis (dense: 0)
  int len;    // rows of that sequence
  int pt;     // query pair within the sequence
  int split;  // key slice
  int kb;     // first key tile of the slice
  int n;      // key tiles of the slice (0: nothing to do)
};

constexpr int kDenseBand = 4;  // pair levels per band of the dense causal order

template <bool CAUSAL>
__device__ __forceinline__ Unit unit_of(const FwdParams& p, int u) {
  Unit w;
  const int BH = p.B * p.H;
  const int L = u / p.n_splits;
  w.split = u % p.n_splits;
  if (CAUSAL && p.n_qt <= 2 * kDenseBand) {
    // heaviest pairs (most key tiles) first, level by level across the heads (short sequences:
    // every head's K and V fit in L2 together, and whole levels balance the clusters best)
    w.pt = p.n_qt - 1 - L / BH;
    w.z = L % BH;
  } else if (CAUSAL) {
    // heaviest pairs (most key tiles) first, in bands of kDenseBand pair levels from the top;
    // inside a band all of a head's pairs sit together, so the clusters that take them at about
    // the same time share that head's K and V tiles in L2
    const int top = (p.n_qt - 1) / kDenseBand;           // highest band
    const int m_top = p.n_qt - kDenseBand * top;         // levels in it (the others are full)
    int b, i, m;
    if (L < BH * m_top) {
      b = top, i = L, m = m_top;
    } else {
      const int L2 = L - BH * m_top;
      b = top - 1 - L2 / (BH * kDenseBand), i = L2 % (BH * kDenseBand), m = kDenseBand;
    }
    w.z = i / m;
    w.pt = kDenseBand * b + m - 1 - i % m;
  } else {                 // all pairs of a head together: its K and V stay in L2
    w.z = L / p.n_qt;
    w.pt = L % p.n_qt;
  }
  w.y0 = 0;
  w.len = p.N;
  // key tiles of the row pair (causal: up to the diagonal of its last row); both CTAs run the
  // same count, rank 0's rows of a tile past their diagonal are fully masked
  const int n_keytiles = (p.N + kBN - 1) / kBN;
  const int n_full = CAUSAL ? min(n_keytiles, 2 * w.pt + 2) : n_keytiles;
  const int chunk = (n_full + p.n_splits - 1) / p.n_splits;
  w.kb = w.split * chunk;
  w.n = max(0, min(w.kb + chunk, n_full) - w.kb);
  return w;
}

// ---- packed variable-length batches: where each unit lies
//
// Sequence s occupies rows [a_s, a_s + len_s) of every head (cu_seqlens clamped into [0, N]) and
// has P_s = ceil(len_s / 256) query pairs.  The H * sum_s P_s units (pair, head, sequence) are
// ordered in bands of kVarBand pair levels, highest band first; inside a band by sequence, then
// head, then pair level from high to low.  Early bands hold the heavy pairs (causal: more key
// tiles the higher the level), so the snake walk of next_unit balances the clusters, and the
// units of one (sequence, head) in a band sit next to each other, so adjacent clusters read the
// same K and V tiles from L2 at about the same time.
constexpr int kVarBand = 4;

__device__ __forceinline__ void seq_span(const FwdParams& p, int s, int& a, int& len) {
  int x = __ldg(p.cu_seqlens + s), y = __ldg(p.cu_seqlens + s + 1);
  x = min(max(x, 0), p.N);
  y = min(max(y, x), p.N);
  a = x;
  len = y - x;
}

// Units of sequence s in band b (warp lanes call it for their own s).
__device__ __forceinline__ int band_units(const FwdParams& p, int s, int b, int& a, int& len) {
  if (s >= p.B) {
    a = len = 0;
    return 0;
  }
  seq_span(p, s, a, len);
  const int pairs = (len + 2 * kBM - 1) / (2 * kBM);
  return min(max(pairs - kVarBand * b, 0), kVarBand);
}

__device__ __forceinline__ int warp_sum(int x) {
  #pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

// Units of band b over all sequences, times the heads (warp-collective).
__device__ __forceinline__ int band_count(const FwdParams& p, int b) {
  const int lane = threadIdx.x & 31;
  int total = 0;
  for (int s0 = 0; s0 < p.B; s0 += 32) {
    int a, len;
    total += warp_sum(band_units(p, s0 + lane, b, a, len));
  }
  return total * p.H;
}

// Walks the units of one cluster in increasing order (next_unit is increasing in k).  Dense
// batches need no state; packed batches keep the current band and the sequence chunk reached
// within it, so each step of the walk costs about one pass over 32 sequences.  Every method is
// warp-collective for packed batches: all 32 lanes call it with the same u and get the same unit.
template <bool CAUSAL, bool VARLEN>
struct Walker {
  int b = 0;     // current band
  int cum = 0;   // units before band b
  int cnt = 0;   // units in band b
  int cs = 0;    // first sequence of the chunk of 32 reached in band b
  int ccum = 0;  // units of band b before sequence cs

  __device__ __forceinline__ void init(const FwdParams& p, int max_pairs) {
    if constexpr (VARLEN) {
      b = (max_pairs + kVarBand - 1) / kVarBand - 1;
      cum = cs = ccum = 0;
      cnt = b >= 0 ? band_count(p, b) : 0;
    }
  }

  __device__ __forceinline__ Unit at(const FwdParams& p, int u) {
    if constexpr (!VARLEN) {
      return unit_of<CAUSAL>(p, u);
    } else {
      const int lane = threadIdx.x & 31;
      while (u >= cum + cnt && b > 0) {
        cum += cnt;
        --b;
        cnt = band_count(p, b);
        cs = ccum = 0;
      }
      const int i = u - cum;  // index within the band
      Unit w;
      w.split = 0;
      w.kb = 0;
      for (;;) {
        int a, len;
        const int m = band_units(p, cs + lane, b, a, len);
        const int wgt = m * p.H;
        int incl = wgt;
        #pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int v = __shfl_up_sync(0xffffffffu, incl, off);
          if (lane >= off) incl += v;
        }
        const int total = __shfl_sync(0xffffffffu, incl, 31);
        if (i < ccum + total || cs + 32 >= p.B) {
          const int r = i - ccum;
          const unsigned hit = __ballot_sync(0xffffffffu, r >= incl - wgt && r < incl);
          const int src = hit ? __ffs(hit) - 1 : 0;
          const int r2 = r - __shfl_sync(0xffffffffu, incl - wgt, src);
          const int ms = max(__shfl_sync(0xffffffffu, m, src), 1);
          w.y0 = __shfl_sync(0xffffffffu, a, src);
          w.len = __shfl_sync(0xffffffffu, len, src);
          w.z = r2 / ms;
          w.pt = kVarBand * b + ms - 1 - r2 % ms;
          const int n_keytiles = (w.len + kBN - 1) / kBN;
          w.n = hit ? (CAUSAL ? min(n_keytiles, 2 * w.pt + 2) : n_keytiles) : 0;
          return w;
        }
        ccum += total;
        cs += 32;
      }
    }
  }
};

// L2 prefetch of the Q tile and the first two key tiles' K and V halves a CTA loads for unit w
// (issued while the CTA sets up, so the first loads find them in L2).
template <int D>
__device__ __forceinline__ void prefetch_first_tiles(const FwdParams& p, const Unit& w, int z_kv,
                                                     int rank) {
  if (w.n == 0) return;
  // only boxes that start inside the tensor's rows
  const int qrow = w.y0 + (2 * w.pt + rank) * kBM;
  #pragma unroll
  for (int c = 0; c < D / 64; ++c) {
    if (qrow < p.N) tma_prefetch_l2_3d(&p.tm_q, c * 64, qrow, w.z);
    for (int j = 0; j < 2 && j < w.n; ++j) {
      const int krow = w.y0 + (w.kb + j) * kBN + 64 * rank;
      if (krow < p.N) tma_prefetch_l2_3d(&p.tm_k, c * 64, krow, z_kv);
    }
  }
  if (D == 128 || rank == 0)
    for (int j = 0; j < 2 && j < w.n; ++j)
      tma_prefetch_l2_3d(&p.tm_v, 64 * rank, w.y0 + (w.kb + j) * kBN, z_kv);
}

// The k-th unit of cluster c among G clusters: rounds of G units, taken forward in even rounds
// and backward in odd ones, so that with units ordered heaviest first every cluster gets a mix.
__device__ __forceinline__ int next_unit(int k, int c, int G) {
  return k * G + ((k & 1) ? G - 1 - c : c);
}

}  // namespace fwd2sm

template <int D, bool CAUSAL, bool VARLEN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(k2smThreads, 1)
    attn_fwd_2sm_kernel(const __grid_constant__ FwdParams p) {
  static_assert(D == 64 || D == 128, "head dim 64 or 128");
  using Lay = Fwd2smLayout<D>;
  using fwd2sm::f2u;
  using fwd2sm::u2f;
  constexpr int SK = k2smStagesK, SV = k2smStagesV, NB = k2smSBufs;
  // P V products are N = 128 wide, 64 value columns from each CTA.  At head dim 64 rank 0 holds
  // all of V's columns and rank 1's V stages stay zero: O's columns 64..127 are zero and unused.
  constexpr bool kVBoth = D == 128;
  constexpr uint32_t kColO = 128u * NB;
  constexpr uint16_t kBoth = 0x3;
  constexpr int kSIssuerWarp = 6;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  const uint32_t sbase = (raw_s + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw_s);
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + Lay::kMisc);
  const WaitCtx wc{reinterpret_cast<volatile int*>(misc + 1), p.status};
  auto bar = [&](int i) -> uint32_t { return sbase + Lay::kBar + 8u * static_cast<uint32_t>(i); };

  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  // rank 0's barrier array in the cluster window (the array is contiguous in both CTAs)
  const uint32_t lbar0 = mapa_shared(sbase + Lay::kBar, 0);
  auto lbar = [&](int i) -> uint32_t { return lbar0 + 8u * static_cast<uint32_t>(i); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = static_cast<int>(gridDim.x) >> 1;  // clusters in the grid
  const int c0 = static_cast<int>(blockIdx.x) >> 1;

  // K/V head slice of a query head slice z: query head h reads K/V head h / group; dense maps are
  // indexed by batch * heads + head, packed maps by head
  auto kv_slice = [&](int z) {
    return VARLEN ? z / p.group : (z / p.H) * (p.H / p.group) + (z % p.H) / p.group;
  };
  if (!VARLEN && warp == 0 && lane == 0) {
    // the tensor maps and this CTA's first tiles start moving while the CTA sets up
    tma_prefetch_desc(&p.tm_q);
    tma_prefetch_desc(&p.tm_k);
    tma_prefetch_desc(&p.tm_v);
    if (c0 < p.n_qt * p.B * p.H * p.n_splits) {
      const fwd2sm::Unit w0 = fwd2sm::unit_of<CAUSAL>(p, c0);
      fwd2sm::prefetch_first_tiles<D>(p, w0, kv_slice(w0.z), static_cast<int>(rank));
    }
  }
  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(Lay::bQF + b), 1);
      mbar_init(bar(Lay::bQE + b), 1);
    }
    for (int s = 0; s < SK; ++s) {
      mbar_init(bar(Lay::bKF + s), 1);
      mbar_init(bar(Lay::bKE + s), 1);
    }
    for (int s = 0; s < SV; ++s) {
      mbar_init(bar(Lay::bVF + s), 1);
      mbar_init(bar(Lay::bVE + s), 1);
    }
    for (int b = 0; b < NB; ++b) {
      mbar_init(bar(Lay::bSF + b), 1);
      mbar_init(bar(Lay::bPF + b), 2 * 4);  // one arrival per softmax warp of both CTAs
      mbar_init(bar(Lay::bPV + b), 1);
    }
    mbar_init(bar(Lay::bOD), 1);
    mbar_init(bar(Lay::bOE), 2 * 4);
    mbar_init(bar(Lay::bDR), 1);
    mbar_init(bar(Lay::bDR + 1), 1);
    fence_barrier_init();
    misc[1] = 0;
  }
  if (VARLEN && warp == 2) {
    // packed batch: the number of units (H * sum of the sequences' query pairs) and the largest
    // pair count, from cu_seqlens clamped into [0, N]; the first CTA also checks that cu_seqlens
    // is a prefix sum from 0 to N (a bad one is reported through the status word)
    int pairs = 0, max_pairs = 0;
    bool bad = false;
    for (int s0 = 0; s0 < p.B; s0 += 32) {
      const int sq = s0 + lane;
      if (sq < p.B) {
        int a, len;
        fwd2sm::seq_span(p, sq, a, len);
        const int np = (len + 2 * kBM - 1) / (2 * kBM);
        pairs += np;
        max_pairs = max(max_pairs, np);
        if (blockIdx.x == 0) {
          const int x = __ldg(p.cu_seqlens + sq), y = __ldg(p.cu_seqlens + sq + 1);
          bad |= (y < x) || (sq == 0 && x != 0) || (sq == p.B - 1 && y != p.N);
        }
      }
    }
    pairs = fwd2sm::warp_sum(pairs);
    #pragma unroll
    for (int off = 16; off > 0; off >>= 1)
      max_pairs = max(max_pairs, __shfl_xor_sync(0xffffffffu, max_pairs, off));
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicCAS(p.status, 0, kStatusBadSeqlens);
    if (lane == 0) {
      misc[2] = static_cast<uint32_t>(pairs * p.H);
      misc[3] = static_cast<uint32_t>(max_pairs);
    }
    if (c0 < pairs * p.H) {
      // this CTA's first tiles start moving while the CTA sets up
      fwd2sm::Walker<CAUSAL, VARLEN> walk;
      walk.init(p, max_pairs);
      const fwd2sm::Unit w0 = walk.at(p, c0);
      if (lane == 0) fwd2sm::prefetch_first_tiles<D>(p, w0, kv_slice(w0.z), static_cast<int>(rank));
    }
  }
  if (!kVBoth && rank == 1) {
    // head dim 64: this CTA's half of every V stage is the zero padding of the P V product
    for (int i = threadIdx.x; i < SV * Lay::kVBytes / 16; i += blockDim.x)
      st_shared_v4(sbase + Lay::kV + i * 16, 0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc_pair(sbase + Lay::kMisc, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // barriers initialised and tensor memory allocated in both CTAs
  tc_fence_after();
  const uint32_t tmem = misc[0];
  const int n_units = VARLEN ? static_cast<int>(misc[2]) : p.n_qt * p.B * p.H * p.n_splits;
  const int max_pairs = VARLEN ? static_cast<int>(misc[3]) : 0;

  // Counters kept by every role: uq = units with work done so far (selects the Q buffer and the
  // per-unit barrier phases), g = key tiles done so far across units (ring stages, S buffers and
  // their phases).
  if (warp == 0) {
    // ===================================================================== TMA producer
    // The whole warp walks the units (the packed-batch walk is warp-collective); lane 0 waits and
    // issues the copies.
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
    }
    const uint64_t keep = l2_policy_evict_last();   // K/V are re-read by every query pair
    const uint64_t once = l2_policy_evict_first();  // Q is read once
    bool ok = true;
    int g = 0, uq = 0;
    fwd2sm::Walker<CAUSAL, VARLEN> walk;
    walk.init(p, max_pairs);
    for (int k = 0, u = c0; ok && u < n_units; u = fwd2sm::next_unit(++k, c0, G)) {
      const fwd2sm::Unit w = walk.at(p, u);
      if (w.n == 0) continue;
      if (lane == 0) {
        const int qb = uq & 1;
        const int z_kv = kv_slice(w.z);
        // the Q buffer was last used by unit uq - 2: its S products have completed
        if (uq >= 2)
          ok = mbar_wait(bar(Lay::bQE + qb), static_cast<uint32_t>((uq - 2) >> 1) & 1u, wc, 0, 3);
        if (ok) {
          if (leader) mbar_arrive_expect_tx(bar(Lay::bQF + qb), 2 * Lay::kQBytes);
          const int qrow0 = w.y0 + (2 * w.pt + static_cast<int>(rank)) * kBM;
          #pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d_pair(sbase + Lay::kQ + qb * Lay::kQBytes + c * 16384, &p.tm_q,
                             lbar(Lay::bQF + qb), c * 64, qrow0, w.z, once);
        }
        for (int j = 0; ok && j < w.n; ++j, ++g) {
          const int sk = g % SK, sv = g % SV;
          const int krow = w.y0 + (w.kb + j) * kBN;
          if (g >= SK &&
              !(ok = mbar_wait(bar(Lay::bKE + sk), (static_cast<uint32_t>(g / SK) & 1u) ^ 1u, wc,
                               0, 1)))
            break;
          if (leader) mbar_arrive_expect_tx(bar(Lay::bKF + sk), 2 * Lay::kKBytes);
          #pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d_pair(sbase + Lay::kK + sk * Lay::kKBytes + c * 8192, &p.tm_k,
                             lbar(Lay::bKF + sk), c * 64, krow + 64 * static_cast<int>(rank),
                             z_kv, keep);
          if (!kVBoth && !leader) continue;  // head dim 64: rank 0 loads all of V's columns
          if (g >= SV &&
              !(ok = mbar_wait(bar(Lay::bVE + sv), (static_cast<uint32_t>(g / SV) & 1u) ^ 1u, wc,
                               0, 2)))
            break;
          if (leader) mbar_arrive_expect_tx(bar(Lay::bVF + sv), (kVBoth ? 2 : 1) * Lay::kVBytes);
          tma_load_3d_pair(sbase + Lay::kV + sv * Lay::kVBytes, &p.tm_v, lbar(Lay::bVF + sv),
                           64 * static_cast<int>(rank), krow, z_kv, keep);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      ++uq;
    }
    // unwinding: copies in flight signal rank 0's barriers and land within microseconds;
    // let them land before the cluster exits
    if (!ok && lane == 0) fwd2sm::settle(100000ull);
  } else if (warp == 1 || warp == kSIssuerWarp) {
    // ========================================= MMA issuers (rank 0): P V on warp 1, S on warp 6
    // Two issuing threads, so that each one's waits overlap the other's products: an MMA issue
    // blocks until the tensor pipe accepts it, so one thread issuing both products leaves the
    // pipe idle during every wait.  S_g needs K_g and the completion of P_{g-3} V_{g-3} (its
    // buffer held P_{g-3}); P_g V_g needs P_g and V_g, and the first P V of a unit also needs the
    // previous unit's epilogue to have read O.
    if (leader) {
      bool ok = true;
      int g = 0, uq = 0;
      if (warp == kSIssuerWarp) {
        constexpr uint32_t kIdS = idesc_bf16_f32(2 * kBM, kBN, false, false);  // Q, K K-major
        const uint64_t desc_k = sdesc_sw128(sbase + Lay::kK, 16, 1024);
        fwd2sm::Walker<CAUSAL, VARLEN> walk;
        walk.init(p, max_pairs);
        for (int k = 0, u = c0; ok && u < n_units; u = fwd2sm::next_unit(++k, c0, G)) {
          const fwd2sm::Unit w = walk.at(p, u);
          if (w.n == 0) continue;
          const int qb = uq & 1;
          const uint64_t desc_q = sdesc_sw128(sbase + Lay::kQ + qb * Lay::kQBytes, 16, 1024);
          if (!(ok = mbar_wait_warp(bar(Lay::bQF + qb), static_cast<uint32_t>(uq >> 1) & 1u, wc,
                                    1, 4)))
            break;
          for (int j = 0; j < w.n; ++j, ++g) {
            // the S issuer runs ahead of the softmax: its waits may suspend (spinning here took
            // issue slots from the softmax warp on the same sub-partition)
            if (g >= NB && !(ok = mbar_wait_warp(bar(Lay::bPV + g % NB),
                                                 static_cast<uint32_t>((g - NB) / NB) & 1u, wc, 1,
                                                 7)))
              break;
            if (!(ok = mbar_wait_warp(bar(Lay::bKF + g % SK), static_cast<uint32_t>(g / SK) & 1u,
                                      wc, 1, 3)))
              break;
            tc_fence_after();
            if (lane == 0) {
              const uint64_t b = desc_k + static_cast<uint64_t>((g % SK) * (Lay::kKBytes >> 4));
              const uint32_t d = tmem + 128u * static_cast<uint32_t>(g % NB);
              #pragma unroll
              for (int k = 0; k < D / 16; ++k) {  // K = 16 per instruction; 4 per 128 bytes
                const uint64_t oq = static_cast<uint64_t>(((k >> 2) * 16384 + (k & 3) * 32) >> 4);
                const uint64_t ok_ = static_cast<uint64_t>(((k >> 2) * 8192 + (k & 3) * 32) >> 4);
                mma_bf16_ss_pair(d, desc_q + oq, b + ok_, kIdS, k > 0 ? 1u : 0u);
              }
              mma_commit_pair(bar(Lay::bSF + g % NB), kBoth);
              mma_commit_pair(bar(Lay::bKE + g % SK), kBoth);
              if (j == w.n - 1) mma_commit_pair(bar(Lay::bQE + qb), kBoth);
            }
            __syncwarp();
          }
          ++uq;
        }
        if (!ok) {  // unwinding: wait for every MMA this thread issued
          if (lane == 0) mma_commit_pair(bar(Lay::bDR), 0x1);
          __syncwarp();
          mbar_wait_drain(bar(Lay::bDR), 0);
        }
      } else {
        constexpr uint32_t kIdO = idesc_bf16_f32(2 * kBM, k2smPVN, false, true);  // P, V MN
        const uint64_t desc_v = sdesc_sw128(sbase + Lay::kV, 16384, 1024);
        fwd2sm::Walker<CAUSAL, VARLEN> walk;
        walk.init(p, max_pairs);
        for (int k = 0, u = c0; ok && u < n_units; u = fwd2sm::next_unit(++k, c0, G)) {
          const fwd2sm::Unit w = walk.at(p, u);
          if (w.n == 0) continue;
          for (int j = 0; j < w.n; ++j, ++g) {
            const int b = g % NB, sv = g % SV;
            if (!(ok = mbar_wait_warp(bar(Lay::bVF + sv),
                                            static_cast<uint32_t>(g / SV) & 1u, wc, 1, 6)))
              break;
            if (!(ok = mbar_wait_warp(bar(Lay::bPF + b), static_cast<uint32_t>(g / NB) & 1u,
                                            wc, 1, 5)))
              break;
            // the first product of a unit overwrites O: the previous unit's epilogue read it
            if (j == 0 && uq > 0 &&
                !(ok = mbar_wait_warp(bar(Lay::bOE), static_cast<uint32_t>(uq - 1) & 1u, wc,
                                            1, 8)))
              break;
            if constexpr (VARLEN) {
              // rows of a sequence's last V tile past its end belong to the next sequence: zero
              // them in both CTAs' halves (the peer's through the cluster window), so that P = 0
              // there cannot meet a non-finite value
              const int valid = w.len - (w.kb + j) * kBN;
              if (valid < kBN) {
                const uint32_t vbase = sbase + Lay::kV + sv * Lay::kVBytes;
                const uint32_t vpeer = mapa_shared(vbase, 1);
                for (int i = max(valid, 0) * 8 + lane; i < kBN * 8; i += 32) {
                  st_shared_v4(vbase + i * 16, 0u, 0u, 0u, 0u);
                  if (kVBoth) st_shared_cluster_v4(vpeer + i * 16, 0u, 0u, 0u, 0u);
                }
                fence_proxy_async_cluster();
              }
              __syncwarp();
            }
            tc_fence_after();
            if (lane == 0) {
              const uint64_t bv = desc_v + static_cast<uint64_t>(sv * (Lay::kVBytes >> 4));
              const uint32_t a = tmem + 128u * static_cast<uint32_t>(b);
              #pragma unroll
              for (int k = 0; k < kBN / 16; ++k)  // 16 keys (2048 bytes of V) per instruction
                mma_bf16_ts_pair(tmem + kColO, a + k * 8,
                                 bv + static_cast<uint64_t>(k * (2048 >> 4)), kIdO,
                                 (j > 0 || k > 0) ? 1u : 0u);
              mma_commit_pair(bar(Lay::bPV + b), kBoth);
              mma_commit_pair(bar(Lay::bVE + sv), kBoth);
              if (j == w.n - 1) mma_commit_pair(bar(Lay::bOD), kBoth);
            }
            __syncwarp();
          }
          if (!ok) break;
          ++uq;
        }
        if (!ok) {
          if (lane == 0) mma_commit_pair(bar(Lay::bDR + 1), 0x1);
          __syncwarp();
          mbar_wait_drain(bar(Lay::bDR + 1), 0);
        }
      }
    }
  } else {
    // ===================================================================== softmax
    const int quarter = warp & 3;       // TMEM lanes this warp may access: 32*quarter .. +31
    const int r = quarter * 32 + lane;  // row of the tile = TMEM lane
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t o_col = t_lane + kColO;
    const float sl2 = p.scale_log2;
    const size_t rows_total = static_cast<size_t>(p.B) * p.H * p.N;
    const size_t plane = static_cast<size_t>(p.n_splits) * rows_total;
    bool ok = true;
    int g = 0, uq = 0;
    fwd2sm::Walker<CAUSAL, VARLEN> walk;
    walk.init(p, max_pairs);
    for (int k = 0, u = c0; ok && u < n_units; u = fwd2sm::next_unit(++k, c0, G)) {
      const fwd2sm::Unit w = walk.at(p, u);
      const int seq_len = w.len;
      const int qrow0 = (2 * w.pt + static_cast<int>(rank)) * kBM;  // first row of this tile
      const int row = qrow0 + r;                                     // row within the sequence
      const bool valid = row < seq_len;
      const size_t grow = static_cast<size_t>(w.z) * static_cast<size_t>(p.N) +
                          static_cast<size_t>(w.y0) + static_cast<size_t>(row);
      if (w.n == 0) {
        if (VARLEN) continue;
        // a key slice past the end of this pair's range: the merge reads max -inf and sum 0
        if (valid) {
          const size_t slot = static_cast<size_t>(w.split) * rows_total + grow;
          p.part_stat[slot] = -INFINITY;
          p.part_stat[plane + slot] = 0.f;
        }
        continue;
      }
      float m2 = -INFINITY;                // reference max of the scaled scores (log2 units)
      float le[4] = {0.f, 0.f, 0.f, 0.f};  // sums of 2^(t - m), fp32
      for (int j = 0; j < w.n; ++j, ++g) {
        const int b = g % NB;
        if (!(ok = mbar_wait_warp(bar(Lay::bSF + b), static_cast<uint32_t>(g / NB) & 1u, wc, 2,
                                  8)))
          break;
        tc_fence_after();
        const uint32_t s_col = t_lane + 128u * static_cast<uint32_t>(b);
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
        const int key0 = (w.kb + j) * kBN;
        if ((CAUSAL && key0 + kBN - 1 > qrow0) || key0 + kBN > seq_len) {
          const int lim = CAUSAL ? min(seq_len - key0, row - key0 + 1) : (seq_len - key0);
          #pragma unroll
          for (int cc = 0; cc < kBN; ++cc) s[cc] = (cc < lim) ? s[cc] : -INFINITY;
        }
        // P = 2^(t - m) in bf16, two per 32-bit word, over the first 64 columns of the buffer;
        // ts = this tile's row sums.  Pass 0 exponentiates against the current reference; the
        // row maximum is taken (pass 1) only on the first tile or when a row's tile sum exceeds
        // kSumLimit.  Both passes are warp-uniform: the TMEM stores are collective.
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
            for (int cc = 8; cc + 16 <= kBN; cc += 16)  // pairs of 8-key groups: keys 8 .. kBN - 9
              #pragma unroll
              for (int k = 0; k < 8; ++k) mx[k] = fmax3(mx[k], s[cc + k], s[cc + 8 + k]);
            #pragma unroll
            for (int k = 0; k < 8; ++k) mx[k] = fmaxf(mx[k], s[kBN - 8 + k]);  // the last 8 keys
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
              const int cc = 32 * h + 2 * i;
              float x0, x1;
              ffma2(x0, x1, s[cc], s[cc + 1], sl2, sl2, neg_m, neg_m);
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

        // O holds P V up to key tile j-1 once that product completes; bring it to the new
        // reference before P_j V_j is added
        if (j > 0 && __any_sync(0xffffffffu, moved)) {
          if (!(ok = mbar_wait_warp(bar(Lay::bPV + (g - 1) % NB),
                                    static_cast<uint32_t>((g - 1) / NB) & 1u, wc, 2, 9)))
            break;
          tc_fence_after();
          #pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
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
        if (lane == 0) mbar_arrive_cluster(lbar(Lay::bPF + b));
      }
      if (!ok) break;
      // ---- epilogue of the unit: O (and the row statistics) out, then O is free again
      if (!(ok = mbar_wait_warp(bar(Lay::bOD), static_cast<uint32_t>(uq) & 1u, wc, 2, 10))) break;
      tc_fence_after();
      const float l_exact = (le[0] + le[1]) + (le[2] + le[3]);
      if (!VARLEN && p.n_splits > 1) {
        // this key slice's partial result for the merge: unnormalised O, reference max, row sum
        const size_t slot = static_cast<size_t>(w.split) * rows_total + grow;
        if (valid) {
          p.part_stat[slot] = m2;
          p.part_stat[plane + slot] = l_exact;
        }
        float4* prow = reinterpret_cast<float4*>(p.part_o + slot * D);
        #pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o[32];
          tmem_ld32(o_col + cc * 32, o);
          tmem_wait_ld_regs(o);
          if (valid) {
            #pragma unroll
            for (int q = 0; q < 8; ++q)
              prow[cc * 8 + q] = make_float4(u2f(o[4 * q]), u2f(o[4 * q + 1]), u2f(o[4 * q + 2]),
                                             u2f(o[4 * q + 3]));
          }
        }
      } else {
        // O / l in bf16, staged in this warp's 8 KB area as D/64 64-column halves of its 32 rows
        // (16-byte chunks XOR-swizzled by row: the tensor map's 128-byte swizzle, and no bank
        // conflicts), then written by D/64 TMA stores that run on while the warp starts the next
        // unit; the map clips rows past the end of the sequence.  The area is rewritten one unit
        // later, once those stores have read it.
        const float inv_l = 1.f / l_exact;
        const uint32_t stage = sbase + Lay::kOut + static_cast<uint32_t>(quarter) * 8192u;
        const int row0 = qrow0 + quarter * 32;  // first row of this warp
        // all of the row's O loads are issued before the first wait
        uint32_t oa[32], ob[32], oc[32], od[32];
        tmem_ld32(o_col + 0, oa);
        tmem_ld32(o_col + 32, ob);
        if constexpr (D == 128) {
          tmem_ld32(o_col + 64, oc);
          tmem_ld32(o_col + 96, od);
        }
        if (lane == 0) bulk_wait_group_read0();  // the previous unit's stores have read the area
        __syncwarp();
        tmem_wait_ld_regs(oa);
        tmem_wait_ld_regs(ob);
        if constexpr (D == 128) {
          tmem_wait_ld_regs(oc);
          tmem_wait_ld_regs(od);
        }
        #pragma unroll
        for (int hcol = 0; hcol < D / 64; ++hcol) {
          #pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const uint32_t* o = hcol == 0 ? (cc == 0 ? oa : ob) : (cc == 0 ? oc : od);
            #pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int chunk = cc * 4 + q;  // 8 bf16 = 16 bytes
              st_shared_v4(stage + hcol * 4096 + lane * 128 + ((chunk ^ (lane & 7)) << 4),
                           pack_bf16x2(u2f(o[8 * q + 0]) * inv_l, u2f(o[8 * q + 1]) * inv_l),
                           pack_bf16x2(u2f(o[8 * q + 2]) * inv_l, u2f(o[8 * q + 3]) * inv_l),
                           pack_bf16x2(u2f(o[8 * q + 4]) * inv_l, u2f(o[8 * q + 5]) * inv_l),
                           pack_bf16x2(u2f(o[8 * q + 6]) * inv_l, u2f(o[8 * q + 7]) * inv_l));
            }
          }
        }
        fence_proxy_async_smem();  // the generic-proxy writes above, before the async-proxy reads
        __syncwarp();
        if (!VARLEN || row0 + 32 <= seq_len) {
          if (lane == 0 && row0 < seq_len) {
            #pragma unroll
            for (int hcol = 0; hcol < D / 64; ++hcol)
              tma_store_3d(&p.tm_o, stage + hcol * 4096, hcol * 64, w.y0 + row0, w.z);
            bulk_commit_group();
          }
        } else if (row0 < seq_len) {
          // the warp's rows run past the end of the sequence, into the next one's rows of the
          // same tensor: write only the rows of this sequence, 16-byte chunks from the staging
          // area (lane = chunk of a row; D/8 chunks per row, 256/D rows per step)
          constexpr int kChunks = D / 8;
          const int nrows = seq_len - row0;
          __nv_bfloat16* obase = p.o + (static_cast<size_t>(w.z) * static_cast<size_t>(p.N) +
                                        static_cast<size_t>(w.y0) + static_cast<size_t>(row0)) *
                                           D;
          const int cq = lane % kChunks;  // 16-byte chunk of the row: half cq / 8, chunk cq % 8
          for (int rr = lane / kChunks; rr < nrows; rr += 32 / kChunks) {
            const uint4 val = *reinterpret_cast<const uint4*>(
                smem + Lay::kOut + quarter * 8192 + (cq >> 3) * 4096 + rr * 128 +
                (((cq & 7) ^ (rr & 7)) << 4));
            *reinterpret_cast<uint4*>(obase + static_cast<size_t>(rr) * D + cq * 8) = val;
          }
        }
        if (valid) p.lse[grow] = (m2 + log2f(l_exact)) * 0.69314718055994530942f;
      }
      // every load of O has completed (wait::ld above); the next unit's first P V may overwrite it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(lbar(Lay::bOE));
      ++uq;
    }
    // this warp's O stores have read the staging area (the writes complete with the grid)
    if (lane == 0) bulk_wait_group_read0();
  }
  tc_fence_before();
  cluster_sync_all();  // no MMA, copy or remote arrival of either CTA is still in flight
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

}  // namespace attn
