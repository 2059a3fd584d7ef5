// attn_unfused.cu -- the deliberately unfused "standard attention" comparison path.
//
// Three launches that pass the N x N intermediates through HBM, as in the pages' description of
// standard attention (compute S = Q K^T and write it; read S, softmax, write P; read P and V,
// write O: CS336 GPU/attention notes, "Attention 为什么容易 memory-bound"; CS336 Lecture 5 notes,
// section 6.1, problem 2).  It uses the same tensor-core building blocks as the fused kernel, so
// the difference measured by the bench is the HBM round trip of S and P, not the GEMM quality.
//   1. qk_scores:  S[bh][i][j] = scale * q_i . k_j  (fp32, tiles above the causal diagonal skipped)
//   2. row_softmax: m_i, l_i over the visible keys; P[bh][i][j] = bf16(exp(s_ij - m_i)) (zero for
//                   invisible keys up to the end of the row's last key tile); inv_l_i = 1 / sum of
//                   the rounded P; lse_i = m_i + ln l_i
//   3. pv:          O_i = inv_l_i * sum_j P_ij v_j  (bf16)
#include <cuda_bf16.h>

#include <cmath>

#include "attn_params.h"
#include "attn_host.h"
#include "sm103_ptx.cuh"

namespace attn {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994530942f;

// ------------------------------------------------------------------------------ 1. scores
struct QkParams {
  CUtensorMap tm_q, tm_k;   // {d, N, BH}, box {64, 128, 1}
  CUtensorMap tm_s;         // fp32 {Npad, N, BH}, box {32, 128, 1}
  int* status;
  int n_t, BH;
  float scale;
};

template <int D>
constexpr int qk_smem() {
  return (2 * 128 * D * 2 > 65536 ? 2 * 128 * D * 2 : 65536) + 1024 + 64;
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(128) qk_scores_kernel(const __grid_constant__ QkParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  const uint32_t sbase = (raw_s + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw_s);
  constexpr int kTile = 128 * D * 2;
  constexpr int kOps = (2 * kTile > 65536 ? 2 * kTile : 65536);
  const uint32_t sq = sbase, sk = sbase + kTile, bar_ld = sbase + kOps, bar_mma = bar_ld + 8;
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + kOps + 16);
  const WaitCtx wc{reinterpret_cast<volatile int*>(misc + 1), p.status};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int L = blockIdx.x;
  const int bh = L / (p.n_t * p.n_t);
  const int it = (L / p.n_t) % p.n_t;
  const int jt = L % p.n_t;
  if (CAUSAL && jt > it) return;  // every key of this tile is after every query

  if (threadIdx.x == 0) {
    mbar_init(bar_ld, 1);
    mbar_init(bar_mma, 1);
    fence_barrier_init();
    misc[1] = 0;
  }
  if (warp == 0) {
    tmem_alloc(sbase + kOps + 16, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];

  if (threadIdx.x == 0) {
    bool ok = true;
    mbar_arrive_expect_tx(bar_ld, 2 * kTile);
    #pragma unroll
    for (int c = 0; c < D / 64; ++c) {
      tma_load_3d(sq + c * 16384, &p.tm_q, bar_ld, c * 64, it * 128, bh);
      tma_load_3d(sk + c * 16384, &p.tm_k, bar_ld, c * 64, jt * 128, bh);
    }
    ok = mbar_wait(bar_ld, 0, wc, 4, 1);
    if (ok) {
      tc_fence_after();
      constexpr uint32_t id = idesc_bf16_f32(128, 128, false, false);
      #pragma unroll
      for (int t = 0; t < D / 16; ++t) {
        const uint32_t off = static_cast<uint32_t>((t >> 2) * 16384 + (t & 3) * 32);
        mma_bf16_ss(tmem, sdesc_sw128(sq + off, 16, 1024), sdesc_sw128(sk + off, 16, 1024), id,
                    t > 0 ? 1u : 0u);
      }
      mma_commit(bar_mma);
    } else {
      mbar_wait_drain(bar_ld, 0);
    }
    misc[2] = ok ? 1u : 0u;
  }
  __syncthreads();
  bool ok = misc[2] != 0 && mbar_wait_warp(bar_mma, 0, wc, 4, 2);
  if (ok) {
    tc_fence_after();
    // TMEM row -> scaled fp32 -> 128-byte-swizzled staging (4 blocks of 32 columns), reusing the
    // operand buffers (the MMA has completed)
    const int r = warp * 32 + lane;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    #pragma unroll
    for (int cb = 0; cb < 4; ++cb) {
      uint32_t v[32];
      tmem_ld32(t_lane + cb * 32, v);
      tmem_wait_ld_regs(v);
      #pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint32_t addr = sbase + cb * 16384 + r * 128 +
                              ((static_cast<uint32_t>(c) ^ static_cast<uint32_t>(r & 7)) << 4);
        st_shared_v4(addr, __float_as_uint(__uint_as_float(v[4 * c]) * p.scale),
                     __float_as_uint(__uint_as_float(v[4 * c + 1]) * p.scale),
                     __float_as_uint(__uint_as_float(v[4 * c + 2]) * p.scale),
                     __float_as_uint(__uint_as_float(v[4 * c + 3]) * p.scale));
      }
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  if (ok && threadIdx.x == 0) {
    #pragma unroll
    for (int cb = 0; cb < 4; ++cb)
      tma_store_3d(&p.tm_s, sbase + cb * 16384, jt * 128 + cb * 32, it * 128, bh);
    bulk_commit_group();
    bulk_wait_group_read0();
  }
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

// -------------------------------------------------------------------------- 2. row softmax
template <bool CAUSAL>
__global__ void __launch_bounds__(256) row_softmax_kernel(const float* __restrict__ S,
                                                          __nv_bfloat16* __restrict__ P,
                                                          float* __restrict__ inv_l,
                                                          float* __restrict__ lse, int N,
                                                          int npad, long long rows) {
  const long long g = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (g >= rows) return;
  const int lane = threadIdx.x & 31;
  const int i = static_cast<int>(g % N);
  const int vis = CAUSAL ? i + 1 : N;
  const int end = CAUSAL ? min(npad, (i / 128 + 1) * 128) : npad;
  const float* srow = S + g * npad;
  __nv_bfloat16* prow = P + g * npad;

  // pass 1: running max and sum of 2^(t - m), t = s * log2(e), per lane, then merged
  float m = -INFINITY, l = 0.f;
  for (int j = lane * 4; j < vis; j += 128) {
    const float4 x = *reinterpret_cast<const float4*>(srow + j);
    float t[4] = {x.x * kLog2e, x.y * kLog2e, x.z * kLog2e, x.w * kLog2e};
    #pragma unroll
    for (int e = 0; e < 4; ++e) t[e] = (j + e < vis) ? t[e] : -INFINITY;
    const float mc = fmaxf(fmaxf(t[0], t[1]), fmaxf(t[2], t[3]));
    const float mn = fmaxf(m, mc);
    l = l * ex2_approx(m - mn) + ex2_approx(t[0] - mn) + ex2_approx(t[1] - mn) +
        ex2_approx(t[2] - mn) + ex2_approx(t[3] - mn);
    m = mn;
  }
  #pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float mo = __shfl_xor_sync(0xffffffffu, m, off);
    const float lo = __shfl_xor_sync(0xffffffffu, l, off);
    const float mn = fmaxf(m, mo);
    const float a = (m == -INFINITY) ? 0.f : ex2_approx(m - mn);
    const float b = (mo == -INFINITY) ? 0.f : ex2_approx(mo - mn);
    l = l * a + lo * b;
    m = mn;
  }
  // pass 2: P = bf16(2^(t - m)), zero past the visible keys; sum of the rounded values
  float lr = 0.f;
  for (int j = lane * 4; j < end; j += 128) {
    float pv[4] = {0.f, 0.f, 0.f, 0.f};
    if (j < vis) {
      const float4 x = *reinterpret_cast<const float4*>(srow + j);
      const float xs[4] = {x.x, x.y, x.z, x.w};
      #pragma unroll
      for (int e = 0; e < 4; ++e) pv[e] = (j + e < vis) ? ex2_approx(xs[e] * kLog2e - m) : 0.f;
    }
    const uint32_t a = pack_bf16x2(pv[0], pv[1]), b = pack_bf16x2(pv[2], pv[3]);
    lr += bf16lo_to_f32(a) + bf16hi_to_f32(a) + bf16lo_to_f32(b) + bf16hi_to_f32(b);
    *reinterpret_cast<uint2*>(prow + j) = make_uint2(a, b);
  }
  #pragma unroll
  for (int off = 16; off > 0; off >>= 1) lr += __shfl_xor_sync(0xffffffffu, lr, off);
  if (lane == 0) {
    inv_l[g] = 1.f / lr;
    lse[g] = (m + log2f(l)) * kLn2;
  }
}

// ------------------------------------------------------------------------------------ 3. P V
struct PvParams {
  CUtensorMap tm_p;   // bf16 {Npad, N, BH}, box {64, 128, 1}
  CUtensorMap tm_v;   // bf16 {d, N, BH}
  __nv_bfloat16* o;
  const float* inv_l;
  int* status;
  int N, n_t;
};

constexpr int kPvStages = 2;

template <int D>
constexpr int pv_smem() {
  return kPvStages * (32768 + 128 * D * 2) + 1024 + 128;
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(192, 1) pv_kernel(const __grid_constant__ PvParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  const uint32_t sbase = (raw_s + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw_s);
  constexpr int kVT = 128 * D * 2;
  constexpr int kStage = 32768 + kVT;
  const uint32_t bars = sbase + kPvStages * kStage;
  auto full = [&](int s) { return bars + 8u * s; };
  auto empty = [&](int s) { return bars + 8u * (kPvStages + s); };
  const uint32_t done = bars + 8u * (2 * kPvStages), drain = done + 8;
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + kPvStages * kStage + 8 * (2 * kPvStages + 2));
  const WaitCtx wc{reinterpret_cast<volatile int*>(misc + 1), p.status};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int it = blockIdx.x % p.n_t;
  const int bh = blockIdx.x / p.n_t;
  const int n_j = CAUSAL ? it + 1 : p.n_t;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPvStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    mbar_init(done, 1);
    mbar_init(drain, 1);
    fence_barrier_init();
    misc[1] = 0;
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(misc), 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];

  if (warp == 0) {
    if (lane == 0) {
      bool ok = true;
      int issued = 0;
      for (int j = 0; j < n_j; ++j) {
        const int s = j % kPvStages;
        if (j >= kPvStages &&
            !(ok = mbar_wait(empty(s), (static_cast<uint32_t>(j / kPvStages) & 1u) ^ 1u, wc, 5, 1)))
          break;
        mbar_arrive_expect_tx(full(s), kStage);
        const uint32_t st = sbase + s * kStage;
        tma_load_3d(st, &p.tm_p, full(s), j * 128, it * 128, bh);
        tma_load_3d(st + 16384, &p.tm_p, full(s), j * 128 + 64, it * 128, bh);
        #pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(st + 32768 + c * 16384, &p.tm_v, full(s), c * 64, j * 128, bh);
        ++issued;
      }
      if (!ok)
        for (int j = (issued > kPvStages ? issued - kPvStages : 0); j < issued; ++j)
          mbar_wait_drain(full(j % kPvStages), static_cast<uint32_t>(j / kPvStages) & 1u);
    }
  } else if (warp == 1) {
    constexpr uint32_t id = idesc_bf16_f32(128, D, false, true);
    bool ok = true;
    for (int j = 0; j < n_j; ++j) {
      const int s = j % kPvStages;
      if (!(ok = mbar_wait_warp(full(s), static_cast<uint32_t>(j / kPvStages) & 1u, wc, 5, 2)))
        break;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t st = sbase + s * kStage;
        #pragma unroll
        for (int t = 0; t < 8; ++t) {
          const uint32_t aoff = static_cast<uint32_t>((t >> 2) * 16384 + (t & 3) * 32);
          mma_bf16_ss(tmem, sdesc_sw128(st + aoff, 16, 1024),
                      sdesc_sw128(st + 32768 + t * 2048, 16384, 1024), id,
                      (j > 0 || t > 0) ? 1u : 0u);
        }
        mma_commit(empty(s));
        if (j == n_j - 1) mma_commit(done);
      }
      __syncwarp();
    }
    if (!ok) {
      if (lane == 0) mma_commit(drain);
      __syncwarp();
      mbar_wait_drain(drain, 0);
    }
  } else {
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int row = it * 128 + r;
    if (mbar_wait_warp(done, 0, wc, 5, 3)) {
      tc_fence_after();
      const uint32_t t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
      const bool valid = row < p.N;
      const size_t g = static_cast<size_t>(bh) * p.N + row;
      const float sc = valid ? p.inv_l[g] : 0.f;
      uint4* orow = reinterpret_cast<uint4*>(p.o + g * D);
      #pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(t_lane + c * 32, v);
        tmem_wait_ld_regs(v);
        uint32_t pk[16];
        #pragma unroll
        for (int e = 0; e < 16; ++e)
          pk[e] = pack_bf16x2(__uint_as_float(v[2 * e]) * sc, __uint_as_float(v[2 * e + 1]) * sc);
        if (valid) {
          #pragma unroll
          for (int q = 0; q < 4; ++q)
            orow[c * 4 + q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

template <int D, bool CAUSAL>
cudaError_t launch_all(const UnfusedArgs& a, cudaStream_t stream) {
  const UnfusedLayout L = unfused_workspace_layout(a.B, a.H, a.N);
  const int BH = a.B * a.H;
  const int n_t = static_cast<int>(L.npad / 128);
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  float* S = reinterpret_cast<float*>(ws + L.s_off);
  __nv_bfloat16* P = reinterpret_cast<__nv_bfloat16*>(ws + L.p_off);
  float* inv_l = reinterpret_cast<float*>(ws + L.l_off);

  QkParams qp{};
  if (encode_rows_map(&qp.tm_q, a.q, D, a.N, BH) != CUDA_SUCCESS ||
      encode_rows_map(&qp.tm_k, a.k, D, a.N, BH) != CUDA_SUCCESS ||
      encode_f32_rows_map(&qp.tm_s, S, L.npad, a.N, BH) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  qp.status = a.status;
  qp.n_t = n_t;
  qp.BH = BH;
  qp.scale = a.scale;
  PvParams pp{};
  if (encode_rows_map(&pp.tm_p, P, L.npad, a.N, BH) != CUDA_SUCCESS ||
      encode_rows_map(&pp.tm_v, a.v, D, a.N, BH) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  pp.o = static_cast<__nv_bfloat16*>(a.o);
  pp.inv_l = inv_l;
  pp.status = a.status;
  pp.N = a.N;
  pp.n_t = n_t;

  const long long qk_grid = static_cast<long long>(n_t) * n_t * BH;
  const long long rows = static_cast<long long>(BH) * a.N;
  if (qk_grid > 0x7FFFFFFF || (rows + 7) / 8 > 0x7FFFFFFF) return cudaErrorInvalidValue;

  cudaError_t e;
  auto* k1 = qk_scores_kernel<D, CAUSAL>;
  if ((e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, qk_smem<D>())))
    return e;
  k1<<<static_cast<int>(qk_grid), 128, qk_smem<D>(), stream>>>(qp);
  if ((e = cudaGetLastError())) return e;
  row_softmax_kernel<CAUSAL><<<static_cast<int>((rows + 7) / 8), 256, 0, stream>>>(
      S, P, inv_l, a.lse, a.N, static_cast<int>(L.npad), rows);
  if ((e = cudaGetLastError())) return e;
  auto* k3 = pv_kernel<D, CAUSAL>;
  if ((e = cudaFuncSetAttribute(k3, cudaFuncAttributeMaxDynamicSharedMemorySize, pv_smem<D>())))
    return e;
  k3<<<n_t * BH, 192, pv_smem<D>(), stream>>>(pp);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_unfused(const UnfusedArgs& a, cudaStream_t stream) {
  if (a.d == 64) return a.causal ? launch_all<64, true>(a, stream) : launch_all<64, false>(a, stream);
  return a.causal ? launch_all<128, true>(a, stream) : launch_all<128, false>(a, stream);
}

}  // namespace attn
