// attn_bwd_kernels.cuh -- tcgen05 kernel of the attention backward pass for sm_103a (GB300).
//
// One launch runs two tile passes: CTAs 0 .. n_kv-1 the dK/dV pass, the others the dQ pass.  Each
// CTA keeps one 128-row tile resident, streams the other operand's tiles through TMA-fed
// shared-memory rings, and rebuilds P from the saved logsumexp instead of reading any N x N
// matrix (CS336 Lecture 5 notes, section 6.2, "反向传播怎么办").
//
// Warp roles (384 threads): warp 0 TMA producer; warp 1 TMEM owner and an MMA issuer (lane 0);
// warps 10 and 11 MMA issuers; warps 2..9 compute.  Each pass's products form three streams that
// meet only through barriers (dK/dV: S^T with dK, dP^T, dV; dQ: S, dP, dQ), one per issuing
// thread: an MMA issue blocks until the tensor pipe accepts it, so a thread issuing two streams
// held the second one back behind every issue and every wait of the first.  A compute thread owns
// one row of the resident tile (its TMEM lane: warp w may access lanes 32*(w%4)..+31) and one
// half of the streamed tile's 128 columns: warps 2..5 take columns 0..63, warps 6..9 64..127.
//
// dK/dV pass (rows = 128 keys of tile j, columns = 128 queries of tile i), query tile t in one of
// two 128-column TMEM buffers (t mod 2):
//   S^T  = K_j Q_i^T      (SS MMA into the buffer)
//   P^T  = 2^(S^T scale log2e - lse2_i) per element, kept in fp32 registers
//   dP^T = V_j dO_i^T     (SS MMA over the same buffer, once every compute thread has loaded S^T)
//   P^T as bf16 over the buffer's last 32 columns of each half, then dS^T = P^T * (dP^T - D_i) as
//          bf16 over the first 32 (signalled separately: dV starts while dS is formed)
//   dV  += P^T dO_i       (TS MMA, A = P^T from TMEM, B = dO_i MN-major; TMEM 256..256+D)
//   dK  += dS^T Q_i       (TS MMA, A = dS^T from TMEM, B = Q_i MN-major; TMEM 256+D..)
//   the buffer takes S^T of tile t+2 once dV and dK of tile t have completed
// dQ pass (rows = 128 queries of tile i, columns = 128 keys of tile j), per key tile:
//   S = Q_i K_j^T (TMEM 0..127, rewritten once every compute thread has loaded it),
//   dP = dO_i V_j^T (two buffers at 128 and 384), P and dS as above with per-row lse2 and D,
//   dQ += dS K_j          (TS MMA, B = K_j MN-major; TMEM 256..256+D)
// An SS product into columns that a TS product reads its A operand from waits for that TS
// product to complete (tcgen05 MMAs with different accumulators are not ordered).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "attn_bwd.h"
#include "sm103_ptx.cuh"

namespace attn {
namespace bwd {

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }

// SS product over D/16 K-steps: both operands K-major 128-row tiles (D/64 blocks of 16 KB,
// 128-byte rows, 32 bytes per K-step of 16 elements).
template <int D>
__device__ __forceinline__ void mma_ss_tile(uint32_t d_tmem, uint64_t a, uint64_t b,
                                            uint32_t idesc) {
  #pragma unroll
  for (int k = 0; k < D / 16; ++k) {
    const uint64_t off = static_cast<uint64_t>(((k >> 2) * 16384 + (k & 3) * 32) >> 4);
    mma_bf16_ss(d_tmem, a + off, b + off, idesc, k > 0 ? 1u : 0u);
  }
}

// TS product over 128 rows of K: A = 128 bf16 values per TMEM lane, stored as two halves of 64
// (32 packed columns each) at column offsets 0 and 64; B = a 128-row MN-major tile (16 rows =
// 2048 bytes per K-step).
__device__ __forceinline__ void mma_ts_tile(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                            uint32_t idesc, bool accumulate) {
  #pragma unroll
  for (int k = 0; k < kBN / 16; ++k)
    mma_bf16_ts(d_tmem, a_tmem + (k >> 2) * 64 + (k & 3) * 8,
                b + static_cast<uint64_t>(k * (2048 >> 4)), idesc,
                (accumulate || k > 0) ? 1u : 0u);
}

// Write one row's half of a D-wide fp32 accumulator (TMEM columns col .. col + D/2 - 1) as bf16,
// multiplied by `mul`, to dst[0 .. D/2 - 1] (16-byte aligned).
template <int D>
__device__ __forceinline__ void store_row_half(uint32_t col, float mul, __nv_bfloat16* dst,
                                               bool valid) {
  #pragma unroll
  for (int c = 0; c < D / 64; ++c) {
    uint32_t v[32];
    tmem_ld32(col + 32 * c, v);
    tmem_wait_ld_regs(v);
    if (valid) {
      uint4* out = reinterpret_cast<uint4*>(dst + 32 * c);
      #pragma unroll
      for (int q = 0; q < 4; ++q)
        out[q] = make_uint4(pack_bf16x2(u2f(v[8 * q + 0]) * mul, u2f(v[8 * q + 1]) * mul),
                            pack_bf16x2(u2f(v[8 * q + 2]) * mul, u2f(v[8 * q + 3]) * mul),
                            pack_bf16x2(u2f(v[8 * q + 4]) * mul, u2f(v[8 * q + 5]) * mul),
                            pack_bf16x2(u2f(v[8 * q + 6]) * mul, u2f(v[8 * q + 7]) * mul));
    }
  }
}

// One row's 64-column half of a 128-wide fp32 accumulator (TMEM columns col .. col + 63), times
// `mul`, as bf16 into row `lane` of a warp's 32-row staging tile: 128-byte rows, 16-byte chunks
// XOR-swizzled by row (the output tensor map's 128-byte swizzle, and no bank conflicts).
__device__ __forceinline__ void stage_row_half128(uint32_t col, float mul, uint32_t stage,
                                                  int lane) {
  #pragma unroll
  for (int c = 0; c < 2; ++c) {
    uint32_t v[32];
    tmem_ld32(col + 32 * c, v);
    tmem_wait_ld_regs(v);
    #pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int chunk = 4 * c + q;
      st_shared_v4(stage + lane * 128 + ((chunk ^ (lane & 7)) << 4),
                   pack_bf16x2(u2f(v[8 * q + 0]) * mul, u2f(v[8 * q + 1]) * mul),
                   pack_bf16x2(u2f(v[8 * q + 2]) * mul, u2f(v[8 * q + 3]) * mul),
                   pack_bf16x2(u2f(v[8 * q + 4]) * mul, u2f(v[8 * q + 5]) * mul),
                   pack_bf16x2(u2f(v[8 * q + 6]) * mul, u2f(v[8 * q + 7]) * mul));
    }
  }
}

}  // namespace bwd

// =============================================================================== dK / dV kernel
// One CTA of the dK/dV pass: key tile slot L (see below).
template <int D, bool CAUSAL, bool VARLEN>
__device__ __forceinline__ void bwd_dkdv_cta(const BwdParams& p, const int L, uint8_t* smem_raw) {
  using Lay = BwdKvLayout<D>;
  const uint32_t raw_s = smem_u32(smem_raw);
  const uint32_t sbase = (raw_s + 1023u) & ~1023u;
  if (sbase - raw_s + Lay::kBytes > static_cast<uint32_t>(Lay::kDynBytes)) {
    // the 1024-byte-aligned layout does not fit what the launch gave (uniform for the CTA)
    if (threadIdx.x == 0) atomicCAS(p.status, 0, kStatusSmemLayout);
    return;
  }
  uint8_t* smem = smem_raw + (sbase - raw_s);
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + Lay::kMisc);
  const WaitCtx wc{reinterpret_cast<volatile int*>(misc + 1), p.status};
  auto bar = [&](int i) -> uint32_t { return sbase + Lay::kBar + 8u * static_cast<uint32_t>(i); };
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(bar(Lay::bKV), 1);
    for (int s = 0; s < kBwdStagesQ; ++s) {
      mbar_init(bar(Lay::bQF + s), 1);
      mbar_init(bar(Lay::bQE + s), 1);
    }
    for (int s = 0; s < kBwdStages; ++s) {
      mbar_init(bar(Lay::bOF + s), 1);
      mbar_init(bar(Lay::bOE + s), 1);
    }
    mbar_init(bar(Lay::bS), 1);
    mbar_init(bar(Lay::bS + 1), 1);
    mbar_init(bar(Lay::bSR), 8 * 32);
    mbar_init(bar(Lay::bDP), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(Lay::bP + b), 8 * 32);
      mbar_init(bar(Lay::bDS + b), 8 * 32);
    }
    mbar_init(bar(Lay::bACC), 2);      // a commit of each of the dV and dK issuers
    mbar_init(bar(Lay::bACC + 1), 2);
    mbar_init(bar(Lay::bEND), 2);
    mbar_init(bar(Lay::bVEND), 1);
    for (int d = 0; d < 3; ++d) mbar_init(bar(Lay::bDR + d), 1);
    fence_barrier_init();
    misc[1] = 0;
  }

  // key tile j of K/V head slice z (of B * H_kv); it visits, for each of the `group` query heads
  // that share the K/V head, query tiles j .. n_tiles-1 (causal; the most first) or all of them.
  // dK and dV sum over all of them (grouped-query attention: a shared K/V head's gradient is the
  // sum over its query heads).
  // Packed batches: z is the K/V head, the tile slot L / H_kv names (sequence, j); rows are
  // y0 + .. within the packed tensors and the planes' rows of the sequence start at 128 tbase.
  int z, j, y0 = 0, seq_len = p.N, tbase = 0;
  if constexpr (!VARLEN) {
    const int BHkv = p.B * p.H_kv;
    if constexpr (CAUSAL) {
      j = L / BHkv;
      z = L % BHkv;
    } else {  // the key tiles of a head together: its Q and dO tiles stay in L2
      z = L / p.n_tiles;
      j = L % p.n_tiles;
    }
  } else {
    z = L % p.H_kv;
    if (warp == 0) {
      int start, len, tile, base;
      bwd_locate_tile(p.cu_seqlens, p.n_seqs, p.N, L / p.H_kv, lane, start, len, tile, base);
      if (lane == 0) {
        misc[2] = static_cast<uint32_t>(start);
        misc[3] = static_cast<uint32_t>(len);
        misc[4] = static_cast<uint32_t>(tile);
        misc[5] = static_cast<uint32_t>(base);
      }
    }
  }
  __syncthreads();
  if constexpr (VARLEN) {
    y0 = static_cast<int>(misc[2]);
    seq_len = static_cast<int>(misc[3]);
    j = static_cast<int>(misc[4]);
    tbase = static_cast<int>(misc[5]);
    if (j < 0) return;  // slot past the last tile of the batch (uniform for the CTA)
  }
  const int n_seq_tiles = (seq_len + kBM - 1) / kBM;
  const int i0 = CAUSAL ? j : 0;
  const int n_head = n_seq_tiles - i0;   // query tiles per query head
  const int n_it = n_head * p.group;     // over the group's query heads
  // first query head slice of the group
  const int zq0 = VARLEN ? z * p.group : (z / p.H_kv) * p.H + (z % p.H_kv) * p.group;

  if (warp == 1) {
    tmem_alloc(sbase + Lay::kMisc, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  grid_dependency_wait();  // the row pass's -lse2 / -D planes are complete from here on
  const uint32_t tmem = misc[0];
  // two 128-column buffers: query tile t uses buffer t & 1 for S^T_t, then (once the compute warps
  // have loaded S^T_t) for dP^T_t, then for the bf16 P^T_t and dS^T_t the dV and dK products read
  constexpr uint32_t kColDV = 256, kColDK = 256 + D;
  constexpr uint64_t kTileD = static_cast<uint64_t>(Lay::kTile >> 4);

  if (warp == 0) {
    // ================================================================ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      tma_prefetch_desc(&p.tm_do);
      const uint64_t keep = l2_policy_evict_last();   // Q, dO: re-read by every key tile
      const uint64_t once = l2_policy_evict_first();  // K, V: read once
      mbar_arrive_expect_tx(bar(Lay::bKV), 2 * Lay::kTile);
      #pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        tma_load_3d_hint(sbase + Lay::kK + c * 16384, &p.tm_k, bar(Lay::bKV), c * 64,
                         y0 + j * kBN, z, once);
        tma_load_3d_hint(sbase + Lay::kV + c * 16384, &p.tm_v, bar(Lay::bKV), c * 64,
                         y0 + j * kBN, z, once);
      }
      int nq = 0, no = 0;
      bool ok = true;
      for (int t = 0; t < n_it; ++t) {
        const int sq = t % kBwdStagesQ, so = t % kBwdStages;
        const int i = i0 + t % n_head;
        const int zq = zq0 + t / n_head;
        const size_t vrow =
            static_cast<size_t>(zq) * p.n_pad + static_cast<size_t>(tbase + i) * kBM;
        if (t >= kBwdStagesQ &&
            !(ok = mbar_wait(bar(Lay::bQE + sq),
                             (static_cast<uint32_t>(t / kBwdStagesQ) & 1u) ^ 1u, wc, 0, 1)))
          break;
        mbar_arrive_expect_tx(bar(Lay::bQF + sq), Lay::kTile + 512);
        #pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d_hint(sbase + Lay::kQ + sq * Lay::kTile + c * 16384, &p.tm_q,
                           bar(Lay::bQF + sq), c * 64, y0 + i * kBM, zq, keep);
        bulk_load_1d(sbase + Lay::kLse + sq * 512, p.nlse2 + vrow, 512, bar(Lay::bQF + sq));
        ++nq;
        if (t >= kBwdStages &&
            !(ok = mbar_wait(bar(Lay::bOE + so),
                             (static_cast<uint32_t>(t / kBwdStages) & 1u) ^ 1u, wc, 0, 2)))
          break;
        mbar_arrive_expect_tx(bar(Lay::bOF + so), Lay::kTile + 512);
        #pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d_hint(sbase + Lay::kDO + so * Lay::kTile + c * 16384, &p.tm_do,
                           bar(Lay::bOF + so), c * 64, y0 + i * kBM, zq, keep);
        bulk_load_1d(sbase + Lay::kDvec + so * 512, p.nd + vrow, 512, bar(Lay::bOF + so));
        ++no;
      }
      if (!ok) {  // unwinding: let every copy still in flight land before the CTA exits
        mbar_wait_drain(bar(Lay::bKV), 0);
        for (int t = (nq > kBwdStagesQ ? nq - kBwdStagesQ : 0); t < nq; ++t)
          mbar_wait_drain(bar(Lay::bQF + t % kBwdStagesQ),
                          static_cast<uint32_t>(t / kBwdStagesQ) & 1u);
        for (int t = (no > kBwdStages ? no - kBwdStages : 0); t < no; ++t)
          mbar_wait_drain(bar(Lay::bOF + t % kBwdStages),
                          static_cast<uint32_t>(t / kBwdStages) & 1u);
      }
    }
  } else if (warp == 1 || warp == 10 || warp == 11) {
    // ====================== MMA issuers: S^T and dK on warp 1, dV on warp 10, dP^T on warp 11
    // Query tile t uses buffer t & 1: S^T_t once dV_{t-2} and dK_{t-2} (which read the buffer)
    // have completed; dP^T_t over it once the compute warps have loaded S^T_t; dV_t once they
    // have written P^T_t, dK_t once they have written dS^T_t.  P_{t+1} is formed while dV_t and
    // dP^T_{t+1} run, and S^T_{t+2} runs while the compute warps form dS_{t+1}.  dK_t and S^T_{t+2}
    // sit on the critical path (dS_t written -> dK_t -> S^T_{t+2} -> the compute warps), so they
    // share a warp that is idle when dS_t is written; an MMA issue blocks until the tensor pipe
    // accepts it, and the dV issuer is then often still blocked in dV_t.
    constexpr uint32_t kIdSS = idesc_bf16_f32(kBM, kBN, false, false);
    constexpr uint32_t kIdTS = idesc_bf16_f32(kBM, D, false, true);
    const uint64_t desc_k = sdesc_sw128(sbase + Lay::kK, 16, 1024);
    const uint64_t desc_v = sdesc_sw128(sbase + Lay::kV, 16, 1024);
    const uint64_t desc_q = sdesc_sw128(sbase + Lay::kQ, 16, 1024);         // K-major (S^T)
    const uint64_t desc_do = sdesc_sw128(sbase + Lay::kDO, 16, 1024);       // K-major (dP^T)
    const uint64_t desc_q_mn = sdesc_sw128(sbase + Lay::kQ, 16384, 1024);   // MN-major (dK)
    const uint64_t desc_do_mn = sdesc_sw128(sbase + Lay::kDO, 16384, 1024); // MN-major (dV)
    bool ok = mbar_wait_warp(bar(Lay::bKV), 0, wc, 1, 2);
    if (warp == 1) {
      auto issue_s = [&](int t) -> bool {  // S^T_t = K_j Q_t^T into buffer t & 1
        const int sq = t % kBwdStagesQ;
        if (!mbar_wait_warp(bar(Lay::bQF + sq), static_cast<uint32_t>(t / kBwdStagesQ) & 1u, wc,
                            1, 3))
          return false;
        tc_fence_after();
        if (lane == 0) {
          bwd::mma_ss_tile<D>(tmem + 128u * static_cast<uint32_t>(t & 1), desc_k,
                              desc_q + sq * kTileD, kIdSS);
          mma_commit(bar(Lay::bS + (t & 1)));
        }
        __syncwarp();
        return true;
      };
      if (ok && n_it > 0) ok = issue_s(0);
      if (ok && n_it > 1) ok = issue_s(1);
      for (int t = 0; ok && t < n_it; ++t) {
        const int sq = t % kBwdStagesQ;
        const uint32_t buf = 128u * static_cast<uint32_t>(t & 1);
        if (!(ok = mbar_wait_warp(bar(Lay::bDS + (t & 1)), static_cast<uint32_t>(t >> 1) & 1u, wc, 1,
                                  8)))
          break;
        tc_fence_after();
        if (lane == 0) {  // dK_t += dS^T_t Q_t
          bwd::mma_ts_tile(tmem + kColDK, tmem + buf, desc_q_mn + sq * kTileD, kIdTS, t > 0);
          mma_commit(bar(Lay::bACC + (t & 1)));
          mma_commit(bar(Lay::bQE + sq));
        }
        __syncwarp();
        if (t + 2 < n_it) {
          // the buffer is free once dV_t and dK_t completed (per-buffer barrier: its next
          // completion needs dK_{t+2}, which this warp issues after S^T_{t+2})
          if (!(ok = mbar_wait_warp(bar(Lay::bACC + (t & 1)), static_cast<uint32_t>(t >> 1) & 1u,
                                    wc, 1, 7)))
            break;
          if (!(ok = issue_s(t + 2))) break;
        }
      }
    } else if (warp == 11) {
      for (int t = 0; ok && t < n_it; ++t) {  // dP^T_t = V_j dO_t^T over S^T_t, once it is loaded
        const int so = t % kBwdStages;
        if (!(ok = mbar_wait_warp(bar(Lay::bOF + so), static_cast<uint32_t>(t / kBwdStages) & 1u,
                                  wc, 1, 4)))
          break;
        if (!(ok = mbar_wait_warp(bar(Lay::bSR), static_cast<uint32_t>(t) & 1u, wc, 1, 5))) break;
        tc_fence_after();
        if (lane == 0) {
          bwd::mma_ss_tile<D>(tmem + 128u * static_cast<uint32_t>(t & 1), desc_v,
                              desc_do + so * kTileD, kIdSS);
          mma_commit(bar(Lay::bDP));
        }
        __syncwarp();
      }
    } else {
      for (int t = 0; ok && t < n_it; ++t) {  // dV_t += P^T_t dO_t
        const int so = t % kBwdStages;
        const uint32_t buf = 128u * static_cast<uint32_t>(t & 1);
        if (!(ok = mbar_wait_warp(bar(Lay::bP + (t & 1)), static_cast<uint32_t>(t >> 1) & 1u, wc, 1,
                                  6)))
          break;
        tc_fence_after();
        if (lane == 0) {
          bwd::mma_ts_tile(tmem + kColDV, tmem + buf + 32, desc_do_mn + so * kTileD, kIdTS, t > 0);
          mma_commit(bar(Lay::bACC + (t & 1)));
          mma_commit(bar(Lay::bOE + so));
          if (t == n_it - 1) mma_commit(bar(Lay::bVEND));  // dV final: its epilogue may start
        }
        __syncwarp();
      }
    }
    // every S^T and dP^T product completed before the compute warps wrote the last dS^T, so the
    // commits of the dV and dK issuers after their last products cover every product of the CTA
    if (ok && warp != 11) {
      if (lane == 0) mma_commit(bar(Lay::bEND));
      __syncwarp();
    }
    if (!ok) {  // unwinding: wait for every MMA this thread issued
      const int dr = Lay::bDR + (warp == 1 ? 0 : warp == 10 ? 1 : 2);
      if (lane == 0) mma_commit(bar(dr));
      __syncwarp();
      mbar_wait_drain(bar(dr), 0);
    }
  } else {
    // ================================================================ compute
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int r = quarter * 32 + lane;  // key row within the tile (= TMEM lane)
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float sl2 = p.scale_log2;
    bool ok = true;
    for (int t = 0; t < n_it; ++t) {
      const int sq = t % kBwdStagesQ, so = t % kBwdStages;
      const uint32_t par = static_cast<uint32_t>(t) & 1u;
      const int i = i0 + t % n_head;
      // this half's 64 query columns of buffer t & 1: S^T, then dP^T, then P^T (bf16) over the
      // last 32 columns (written first, for the dV product) and dS^T (bf16) over the first 32
      const uint32_t col = t_lane + 128u * static_cast<uint32_t>(t & 1) + 64 * half;
      if (!(ok = mbar_wait_warp(bar(Lay::bQF + sq), static_cast<uint32_t>(t / kBwdStagesQ) & 1u,
                                wc, 2, 9)))
        break;
      if (!(ok = mbar_wait_warp(bar(Lay::bS + (t & 1)), static_cast<uint32_t>(t >> 1) & 1u, wc, 2,
                                10)))
        break;
      tc_fence_after();
      float pf[64];
      {
        uint32_t u0[32], u1[32];
        tmem_ld32(col, u0);
        tmem_ld32(col + 32, u1);
        tmem_wait_ld_regs(u0);
        tmem_wait_ld_regs(u1);
        #pragma unroll
        for (int c = 0; c < 32; ++c) {
          pf[c] = bwd::u2f(u0[c]);
          pf[32 + c] = bwd::u2f(u1[c]);
        }
      }
      tc_fence_before();
      mbar_arrive(bar(Lay::bSR));  // the buffer may now receive dP^T
      const float* lvec = reinterpret_cast<const float*>(smem + Lay::kLse + sq * 512) + 64 * half;
      #pragma unroll
      for (int c4 = 0; c4 < 16; ++c4) {  // P = 2^(s scale log2e - lse2): packed FMAs, then ex2
        const float4 l = reinterpret_cast<const float4*>(lvec)[c4];  // -lse2 of 4 queries
        float x0, x1, x2, x3;
        ffma2(x0, x1, pf[4 * c4], pf[4 * c4 + 1], sl2, sl2, l.x, l.y);
        ffma2(x2, x3, pf[4 * c4 + 2], pf[4 * c4 + 3], sl2, sl2, l.z, l.w);
        pf[4 * c4 + 0] = ex2_approx(x0);
        pf[4 * c4 + 1] = ex2_approx(x1);
        pf[4 * c4 + 2] = ex2_approx(x2);
        pf[4 * c4 + 3] = ex2_approx(x3);
      }
      if (CAUSAL && i == j) {  // diagonal tile: query 64*half + c precedes key r when < r
        #pragma unroll
        for (int c = 0; c < 64; ++c) pf[c] = (64 * half + c < r) ? 0.f : pf[c];
      }
      if (!(ok = mbar_wait_warp(bar(Lay::bOF + so), static_cast<uint32_t>(t / kBwdStages) & 1u,
                                wc, 2, 11)))
        break;
      if (!(ok = mbar_wait_warp(bar(Lay::bDP), par, wc, 2, 12))) break;
      tc_fence_after();
      {
        // P^T first, over the columns of the second half of dP^T once those are loaded, so the dV
        // product can start while dS is formed.  dS of queries 32..63 packs into columns that
        // still hold dP^T of queries 16..31, so it waits in registers until the first half of
        // dP^T is loaded too.
        const float* dvec =
            reinterpret_cast<const float*>(smem + Lay::kDvec + so * 512) + 64 * half;  // -D
        auto ds_half = [&](const uint32_t (&u)[32], int h, uint32_t (&pk)[16]) {
          #pragma unroll
          for (int q = 0; q < 8; ++q) {  // dS = P (dP - D): packed add and multiply
            const int c4 = 8 * h + q;
            const float4 dl = reinterpret_cast<const float4*>(dvec)[c4];
            float t0, t1, t2, t3, d0, d1, d2, d3;
            fadd2_to(t0, t1, bwd::u2f(u[4 * q]), bwd::u2f(u[4 * q + 1]), dl.x, dl.y);
            fadd2_to(t2, t3, bwd::u2f(u[4 * q + 2]), bwd::u2f(u[4 * q + 3]), dl.z, dl.w);
            fmul2(d0, d1, pf[4 * c4], pf[4 * c4 + 1], t0, t1);
            fmul2(d2, d3, pf[4 * c4 + 2], pf[4 * c4 + 3], t2, t3);
            pk[2 * q] = pack_bf16x2(d0, d1);
            pk[2 * q + 1] = pack_bf16x2(d2, d3);
          }
        };
        uint32_t pk1[16];
        {
          uint32_t u1[32];
          tmem_ld32(col + 32, u1);
          tmem_wait_ld_regs(u1);
          uint32_t pp[32];
          #pragma unroll
          for (int c = 0; c < 32; ++c) pp[c] = pack_bf16x2(pf[2 * c], pf[2 * c + 1]);
          tmem_st32(col + 32, pp);
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(bar(Lay::bP + (t & 1)));
          ds_half(u1, 1, pk1);
        }
        {
          uint32_t u0[32], pk0[16];
          tmem_ld32(col, u0);
          tmem_wait_ld_regs(u0);
          ds_half(u0, 0, pk0);
          tmem_st16(col, pk0);
          tmem_st16(col + 16, pk1);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(Lay::bDS + (t & 1)));
    }
    // epilogue: dV once its last product has completed (the last dK product may still run),
    // then scale dK once every product of the CTA has completed.  Head dim 128: 32-row staging
    // tiles in the dO ring (idle once the last dV product, the last reader of dO, has completed;
    // every load has landed), written by TMA stores; on dense batches the tensor maps clip rows
    // past N, on packed batches only warps whose 32 rows all belong to the sequence take this
    // path (rows past its end are the next sequence's).  Stores from the threads wrote 16 bytes
    // to each of 32 rows per instruction.
    if (ok) ok = mbar_wait_warp(bar(Lay::bVEND), 0, wc, 2, 14);
    const int row0 = j * kBN + quarter * 32;  // this warp's first key row in the sequence
    bool staged = false;
    if constexpr (D == 128) staged = !VARLEN || row0 + 32 <= seq_len;
    const uint32_t stage_v = sbase + Lay::kDO + static_cast<uint32_t>(warp - 2) * 4096u;
    const uint32_t stage_k = stage_v + static_cast<uint32_t>(Lay::kTile);  // the second dO stage
    if (ok && staged) {
      tc_fence_after();
      bwd::stage_row_half128(t_lane + kColDV + half * 64, 1.f, stage_v, lane);
      fence_proxy_async_smem();  // the generic-proxy writes, before the async-proxy reads
      __syncwarp();
      if (lane == 0 && row0 < seq_len) {
        tma_store_3d(&p.tm_dv, stage_v, 64 * half, y0 + row0, z);
        bulk_commit_group();
      }
      __syncwarp();
    }
    if (ok) ok = mbar_wait_warp(bar(Lay::bEND), 0, wc, 2, 13);
    if (ok) {
      tc_fence_after();
      if (staged) {
        bwd::stage_row_half128(t_lane + kColDK + half * 64, p.scale, stage_k, lane);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && row0 < seq_len) {
          tma_store_3d(&p.tm_dk, stage_k, 64 * half, y0 + row0, z);
          bulk_commit_group();
          bulk_wait_group_read0();  // the staging areas stay valid until the stores have read them
        }
        __syncwarp();
      } else {
        const int key = j * kBN + r;
        const bool valid = key < seq_len;
        const size_t row = static_cast<size_t>(z) * p.N + y0 + (valid ? key : 0);
        bwd::store_row_half<D>(t_lane + kColDV + half * (D / 2), 1.f,
                               p.dv + row * D + half * (D / 2), valid);
        bwd::store_row_half<D>(t_lane + kColDK + half * (D / 2), p.scale,
                               p.dk + row * D + half * (D / 2), valid);
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

// =================================================================================== dQ kernel
// One CTA of the dQ pass: query tile slot L (see below).
template <int D, bool CAUSAL, bool VARLEN>
__device__ __forceinline__ void bwd_dq_cta(const BwdParams& p, const int L, uint8_t* smem_raw) {
  using Lay = BwdQLayout<D>;
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
    for (int s = 0; s < kBwdStagesQK; ++s) {
      mbar_init(bar(Lay::bKF + s), 1);
      mbar_init(bar(Lay::bKE + s), 2);  // read by S (warp 1) and dQ (warp 10)
    }
    for (int s = 0; s < kBwdStages; ++s) {
      mbar_init(bar(Lay::bVF + s), 1);
      mbar_init(bar(Lay::bVE + s), 1);
    }
    mbar_init(bar(Lay::bS), 1);
    mbar_init(bar(Lay::bSR), 8 * 32);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(Lay::bDP + b), 1);
      mbar_init(bar(Lay::bDS + b), 8 * 32);
      mbar_init(bar(Lay::bDQ + b), 1);
    }
    for (int d = 0; d < 3; ++d) mbar_init(bar(Lay::bDR + d), 1);
    fence_barrier_init();
    misc[1] = 0;
  }

  // query tile i of head slice z; causal: key tiles 0..i (the heaviest tiles first), else all
  int z, i, y0 = 0, seq_len = p.N, tbase = 0;
  if constexpr (!VARLEN) {
    const int BH = p.B * p.H;
    if constexpr (CAUSAL) {
      i = p.n_tiles - 1 - L / BH;
      z = L % BH;
    } else {  // the query tiles of a head together: its K and V tiles stay in L2
      z = L / p.n_tiles;
      i = L % p.n_tiles;
    }
  } else {  // packed batches: z is the head, the slot L / H names (sequence, i)
    z = L % p.H;
    if (warp == 0) {
      int start, len, tile, base;
      bwd_locate_tile(p.cu_seqlens, p.n_seqs, p.N, L / p.H, lane, start, len, tile, base);
      if (lane == 0) {
        misc[2] = static_cast<uint32_t>(start);
        misc[3] = static_cast<uint32_t>(len);
        misc[4] = static_cast<uint32_t>(tile);
        misc[5] = static_cast<uint32_t>(base);
      }
    }
  }
  __syncthreads();
  if constexpr (VARLEN) {
    y0 = static_cast<int>(misc[2]);
    seq_len = static_cast<int>(misc[3]);
    i = static_cast<int>(misc[4]);
    tbase = static_cast<int>(misc[5]);
    if (i < 0) return;  // slot past the last tile of the batch (uniform for the CTA)
  }
  const int n_kv = CAUSAL ? i + 1 : (seq_len + kBN - 1) / kBN;
  // K/V head slice of query head z
  const int z_kv = VARLEN ? z / p.group : (z / p.H) * p.H_kv + (z % p.H) / p.group;

  if (warp == 1) {
    tmem_alloc(sbase + Lay::kMisc, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  grid_dependency_wait();  // the row pass's -lse2 / -D planes are complete from here on
  const uint32_t tmem = misc[0];
  // S at 0, dQ at 256, dP / dS double-buffered at 128 and 384 (key tile jj uses buffer jj & 1)
  constexpr uint32_t kColS = 0, kColDQ = 256;
  auto dp_col = [](int b) -> uint32_t { return 128u + 256u * static_cast<uint32_t>(b); };
  constexpr uint64_t kTileD = static_cast<uint64_t>(Lay::kTile >> 4);

  if (warp == 0) {
    // ================================================================ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      tma_prefetch_desc(&p.tm_do);
      const uint64_t keep = l2_policy_evict_last();   // K, V: re-read by every query tile
      const uint64_t once = l2_policy_evict_first();  // Q, dO: read once
      mbar_arrive_expect_tx(bar(Lay::bQ), 2 * Lay::kTile);
      #pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        tma_load_3d_hint(sbase + Lay::kQ + c * 16384, &p.tm_q, bar(Lay::bQ), c * 64,
                         y0 + i * kBM, z, once);
        tma_load_3d_hint(sbase + Lay::kDO + c * 16384, &p.tm_do, bar(Lay::bQ), c * 64,
                         y0 + i * kBM, z, once);
      }
      int nk = 0, nv = 0;
      bool ok = true;
      for (int jj = 0; jj < n_kv; ++jj) {
        const int sk = jj % kBwdStagesQK, sv = jj % kBwdStages;
        if (jj >= kBwdStagesQK &&
            !(ok = mbar_wait(bar(Lay::bKE + sk),
                             (static_cast<uint32_t>(jj / kBwdStagesQK) & 1u) ^ 1u, wc, 0, 1)))
          break;
        mbar_arrive_expect_tx(bar(Lay::bKF + sk), Lay::kTile);
        #pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d_hint(sbase + Lay::kK + sk * Lay::kTile + c * 16384, &p.tm_k,
                           bar(Lay::bKF + sk), c * 64, y0 + jj * kBN, z_kv, keep);
        ++nk;
        if (jj >= kBwdStages &&
            !(ok = mbar_wait(bar(Lay::bVE + sv),
                             (static_cast<uint32_t>(jj / kBwdStages) & 1u) ^ 1u, wc, 0, 2)))
          break;
        mbar_arrive_expect_tx(bar(Lay::bVF + sv), Lay::kTile);
        #pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d_hint(sbase + Lay::kV + sv * Lay::kTile + c * 16384, &p.tm_v,
                           bar(Lay::bVF + sv), c * 64, y0 + jj * kBN, z_kv, keep);
        ++nv;
      }
      if (!ok) {  // unwinding: let every copy still in flight land before the CTA exits
        mbar_wait_drain(bar(Lay::bQ), 0);
        for (int t = (nk > kBwdStagesQK ? nk - kBwdStagesQK : 0); t < nk; ++t)
          mbar_wait_drain(bar(Lay::bKF + t % kBwdStagesQK),
                          static_cast<uint32_t>(t / kBwdStagesQK) & 1u);
        for (int t = (nv > kBwdStages ? nv - kBwdStages : 0); t < nv; ++t)
          mbar_wait_drain(bar(Lay::bVF + t % kBwdStages),
                          static_cast<uint32_t>(t / kBwdStages) & 1u);
      }
    }
  } else if (warp == 1 || warp == 10 || warp == 11) {
    // ======================== MMA issuers: S on warp 1, dQ on warp 10, dP on warp 11
    // S and dP run ahead of dQ: dP alternates between two tensor-memory buffers, and a buffer is
    // rewritten once the dQ product that read it (two tiles back) completed; S is rewritten once
    // every compute thread has read the previous one.
    constexpr uint32_t kIdSS = idesc_bf16_f32(kBM, kBN, false, false);
    constexpr uint32_t kIdTS = idesc_bf16_f32(kBM, D, false, true);
    const uint64_t desc_q = sdesc_sw128(sbase + Lay::kQ, 16, 1024);
    const uint64_t desc_do = sdesc_sw128(sbase + Lay::kDO, 16, 1024);
    const uint64_t desc_k = sdesc_sw128(sbase + Lay::kK, 16, 1024);          // K-major use
    const uint64_t desc_v = sdesc_sw128(sbase + Lay::kV, 16, 1024);
    const uint64_t desc_k_mn = sdesc_sw128(sbase + Lay::kK, 16384, 1024);    // MN-major use
    bool ok = mbar_wait_warp(bar(Lay::bQ), 0, wc, 1, 2);
    if (warp == 1) {
      for (int jj = 0; ok && jj < n_kv; ++jj) {  // S = Q_i K_j^T
        const int sk = jj % kBwdStagesQK;
        if (!(ok = mbar_wait_warp(bar(Lay::bKF + sk),
                                  static_cast<uint32_t>(jj / kBwdStagesQK) & 1u, wc, 1, 3)))
          break;
        if (jj > 0 && !(ok = mbar_wait_spin_warp(bar(Lay::bSR), (static_cast<uint32_t>(jj) & 1u) ^ 1u,
                                                 wc, 1, 4)))
          break;
        tc_fence_after();
        if (lane == 0) {
          bwd::mma_ss_tile<D>(tmem + kColS, desc_q, desc_k + sk * kTileD, kIdSS);
          mma_commit(bar(Lay::bS));
          mma_commit(bar(Lay::bKE + sk));
        }
        __syncwarp();
      }
    } else if (warp == 11) {
      for (int jj = 0; ok && jj < n_kv; ++jj) {  // dP = dO_i V_j^T into buffer jj & 1
        const int sv = jj % kBwdStages, b = jj & 1;
        if (!(ok = mbar_wait_warp(bar(Lay::bVF + sv), static_cast<uint32_t>(jj / kBwdStages) & 1u,
                                  wc, 1, 5)))
          break;
        if (jj >= 2 && !(ok = mbar_wait_spin_warp(bar(Lay::bDQ + b),
                                                  (static_cast<uint32_t>(jj >> 1) & 1u) ^ 1u, wc,
                                                  1, 6)))
          break;
        tc_fence_after();
        if (lane == 0) {
          bwd::mma_ss_tile<D>(tmem + dp_col(b), desc_do, desc_v + sv * kTileD, kIdSS);
          mma_commit(bar(Lay::bDP + b));
          mma_commit(bar(Lay::bVE + sv));
        }
        __syncwarp();
      }
    } else {
      for (int jj = 0; ok && jj < n_kv; ++jj) {  // dQ += dS K_j
        const int sk = jj % kBwdStagesQK, b = jj & 1;
        if (!(ok = mbar_wait_spin_warp(bar(Lay::bDS + b), static_cast<uint32_t>(jj >> 1) & 1u, wc,
                                       1, 7)))
          break;
        tc_fence_after();
        if (lane == 0) {
          bwd::mma_ts_tile(tmem + kColDQ, tmem + dp_col(b), desc_k_mn + sk * kTileD, kIdTS,
                           jj > 0);
          mma_commit(bar(Lay::bDQ + b));
          mma_commit(bar(Lay::bKE + sk));
        }
        __syncwarp();
      }
    }
    if (!ok) {  // unwinding: wait for every MMA this thread issued
      const int dr = Lay::bDR + (warp == 1 ? 0 : warp == 10 ? 1 : 2);
      if (lane == 0) mma_commit(bar(dr));
      __syncwarp();
      mbar_wait_drain(bar(dr), 0);
    }
  } else {
    // ================================================================ compute
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int r = quarter * 32 + lane;  // query row within the tile (= TMEM lane)
    const int row = i * kBM + r;        // query row within the sequence (padded rows < n_pad)
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t col_s = t_lane + kColS + 64 * half;
    const float sl2 = p.scale_log2;
    const size_t prow = static_cast<size_t>(z) * p.n_pad + static_cast<size_t>(tbase) * kBM + row;
    const float nlse2 = p.nlse2[prow];  // -lse * log2(e)
    const float nd = p.nd[prow];        // -D
    bool ok = true;
    for (int jj = 0; jj < n_kv; ++jj) {
      const uint32_t par = static_cast<uint32_t>(jj) & 1u;
      if (!(ok = mbar_wait_warp(bar(Lay::bS), par, wc, 2, 8))) break;
      tc_fence_after();
      float pf[64];
      {
        uint32_t u0[32], u1[32];
        tmem_ld32(col_s, u0);
        tmem_ld32(col_s + 32, u1);
        tmem_wait_ld_regs(u0);
        tmem_wait_ld_regs(u1);
        #pragma unroll
        for (int c = 0; c < 32; ++c) {
          pf[c] = bwd::u2f(u0[c]);
          pf[32 + c] = bwd::u2f(u1[c]);
        }
      }
      tc_fence_before();
      mbar_arrive(bar(Lay::bSR));  // S columns may be rewritten
      #pragma unroll
      for (int c = 0; c < 64; c += 2) {
        float x0, x1;
        ffma2(x0, x1, pf[c], pf[c + 1], sl2, sl2, nlse2, nlse2);
        pf[c] = ex2_approx(x0);
        pf[c + 1] = ex2_approx(x1);
      }
      // keys past the end of the sequence, and (diagonal tile) keys after the query, get P = 0
      const int key0 = jj * kBN + 64 * half;
      if ((CAUSAL && jj == i) || key0 + 64 > seq_len) {
        const int lim = CAUSAL ? min(seq_len - key0, row - key0 + 1) : (seq_len - key0);
        #pragma unroll
        for (int c = 0; c < 64; ++c) pf[c] = (c < lim) ? pf[c] : 0.f;
      }
      const int b = jj & 1;
      const uint32_t col_dp = t_lane + dp_col(b) + 64 * half;
      if (!(ok = mbar_wait_warp(bar(Lay::bDP + b), static_cast<uint32_t>(jj >> 1) & 1u, wc, 2, 9)))
        break;
      tc_fence_after();
      {
        uint32_t u0[32], u1[32];
        tmem_ld32(col_dp, u0);
        tmem_ld32(col_dp + 32, u1);
        tmem_wait_ld_regs(u0);
        tmem_wait_ld_regs(u1);
        uint32_t pk[32];
        #pragma unroll
        for (int c = 0; c < 32; ++c) {  // dS = P (dP - D): packed add and multiply
          const uint32_t* u = c < 16 ? u0 : u1;
          const int k = 2 * (c & 15);
          float t0, t1, d0, d1;
          fadd2_to(t0, t1, bwd::u2f(u[k]), bwd::u2f(u[k + 1]), nd, nd);
          fmul2(d0, d1, pf[2 * c], pf[2 * c + 1], t0, t1);
          pk[c] = pack_bf16x2(d0, d1);
        }
        tmem_st32(col_dp, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(Lay::bDS + b));
    }
    // the last dQ commit covers every MMA of the CTA
    if (ok)
      ok = mbar_wait_warp(bar(Lay::bDQ + ((n_kv - 1) & 1)),
                          static_cast<uint32_t>((n_kv - 1) >> 1) & 1u, wc, 2, 10);
    if (ok) {
      tc_fence_after();
      const int row0 = i * kBM + quarter * 32;  // this warp's first query row in the sequence
      bool staged = false;
      if constexpr (D == 128) staged = !VARLEN || row0 + 32 <= seq_len;
      if (staged) {
        // scale dQ through a 32-row staging tile in the idle K ring, written by a TMA store (the
        // conditions of the dK/dV pass's epilogue)
        const uint32_t stage = sbase + Lay::kK + static_cast<uint32_t>(warp - 2) * 4096u;
        bwd::stage_row_half128(t_lane + kColDQ + half * 64, p.scale, stage, lane);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && row0 < seq_len) {
          tma_store_3d(&p.tm_dq, stage, 64 * half, y0 + row0, z);
          bulk_commit_group();
          bulk_wait_group_read0();
        }
        __syncwarp();
      } else {
        const bool valid = row < seq_len;
        const size_t grow = static_cast<size_t>(z) * p.N + y0 + (valid ? row : 0);
        bwd::store_row_half<D>(t_lane + kColDQ + half * (D / 2), p.scale,
                               p.dq + grow * D + half * (D / 2), valid);
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

// Both passes in one launch: CTAs 0 .. n_kv_ctas-1 run the dK/dV pass, the others the dQ pass.
// CTAs start roughly in index order, so the dQ pass fills the SMs the dK/dV pass leaves idle in
// its last, partial wave (two launches each ended in one).
template <int D, bool CAUSAL, bool VARLEN>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_tiles_kernel(const __grid_constant__ BwdParams p, int n_kv_ctas) {
  extern __shared__ uint8_t smem_raw[];
  const int L = static_cast<int>(blockIdx.x);
  if (L < n_kv_ctas)
    bwd_dkdv_cta<D, CAUSAL, VARLEN>(p, L, smem_raw);
  else
    bwd_dq_cta<D, CAUSAL, VARLEN>(p, L - n_kv_ctas, smem_raw);
}

}  // namespace attn
