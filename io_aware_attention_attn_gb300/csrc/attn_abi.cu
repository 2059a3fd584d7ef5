// attn_abi.cu -- the extern "C" entry points of libattn_gb300: argument validation, TMA map
// encoding and kernel launch.  The arithmetic lives entirely in the CUDA kernels.
#include <atomic>
#include <cmath>
#include <climits>
#include <mutex>

#include <cudaTypedefs.h>

#include "attn_gb300.h"
#include "attn_host.h"
#include "attn_bwd.h"
#include "attn_fp8.h"
#include "attn_params.h"

namespace attn {

__device__ int g_attn_status = 0;

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

constexpr int kMaxDevices = 64;
std::atomic<int> g_dev_ok[kMaxDevices];          // 0 unknown, 1 sm_103, 2 other

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

int encode_rows_map(CUtensorMap* map, const void* base, uint64_t d, uint64_t rows,
                    uint64_t heads, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return CUDA_ERROR_NOT_FOUND;
  const cuuint64_t dims[3] = {d, rows, heads};
  const cuuint64_t strides[2] = {d * 2, d * 2 * rows};  // bytes, dims 1 and 2
  const cuuint32_t box[3] = {64, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

int encode_f32_rows_map(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                        uint64_t heads) {
  auto fn = encode_fn();
  if (!fn) return CUDA_ERROR_NOT_FOUND;
  const cuuint64_t dims[3] = {cols, rows, heads};
  const cuuint64_t strides[2] = {cols * 4, cols * 4 * rows};
  const cuuint32_t box[3] = {32, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// One-byte codes [heads][rows][inner], box 128 x 128 with the 128-byte swizzle.
int encode_u8_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
                  uint64_t heads) {
  auto fn = encode_fn();
  if (!fn) return CUDA_ERROR_NOT_FOUND;
  const cuuint64_t dims[3] = {inner, rows, heads};
  const cuuint64_t strides[2] = {inner, inner * rows};
  const cuuint32_t box[3] = {128, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

int check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_LAUNCH;
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_DEVICE;
  int st = g_dev_ok[dev].load(std::memory_order_acquire);
  if (st == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return ATTN_ERR_LAUNCH;
    st = (major == 10 && minor == 3) ? 1 : 2;
    g_dev_ok[dev].store(st, std::memory_order_release);
  }
  return st == 1 ? 0 : ATTN_ERR_DEVICE;
}

// Device address of the status word in the current context.  Looked up on every call, not cached
// per device: after a device reset or a new context the module may load at another address.
int* status_word() {
  void* addr = nullptr;
  if (cudaGetSymbolAddress(&addr, g_attn_status) != cudaSuccess) return nullptr;
  return static_cast<int*>(addr);
}

// Shared validation of attn_fwd / attn_fwd_unfused.  Sets *empty when there is nothing to do.
static int validate(const void* q, const void* k, const void* v, const void* o, const float* lse,
                    const int32_t* cu, int B, int H, int N, int d, float scale, bool* empty) {
  *empty = false;
  if (B < 0 || H < 0 || N < 0) return ATTN_ERR_SHAPE;
  if (cu != nullptr && B == 0 && N > 0) return ATTN_ERR_SHAPE;  // tokens but no sequences
  if (B == 0 || H == 0 || N == 0) {
    *empty = true;
    return ATTN_OK;
  }
  if (d != 64 && d != 128) return ATTN_ERR_HEAD_DIM;
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return ATTN_ERR_ALIGN;
  if (cu != nullptr && (reinterpret_cast<uintptr_t>(cu) & 3u)) return ATTN_ERR_ALIGN;
  if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_SCALE;
  // grid sizes must fit the kernel's 32-bit indices
  const long long tiles_per_head = (static_cast<long long>(N) + kBM - 1) / kBM;
  const long long grid = cu ? (tiles_per_head + B) * H
                            : tiles_per_head * static_cast<long long>(B) * H;
  if (grid > INT_MAX) return ATTN_ERR_SHAPE;
  if (cu == nullptr && static_cast<long long>(B) * H > INT_MAX) return ATTN_ERR_SHAPE;
  return ATTN_OK;
}

static int fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse,
                    const int32_t* cu_seqlens, int B, int H, int Hkv, int N, int d, int causal,
                    float scale, void* stream, int n_splits = 1, float* part_o = nullptr,
                    float* part_stat = nullptr) {
  bool empty = false;
  int rc = validate(q, k, v, o, lse, cu_seqlens, B, H, N, d, scale, &empty);
  if (rc != ATTN_OK) return rc;
  if (Hkv < 0 || (H > 0 && (Hkv == 0 || H % Hkv != 0))) return ATTN_ERR_SHAPE;
  if (empty) return ATTN_OK;
  if ((rc = check_device()) != 0) return rc;
  FwdParams p{};
  const bool varlen = cu_seqlens != nullptr;
  // every forward runs on CTA pairs (one query tile per SM, each SM loading 64-key halves of the K
  // tiles and writing O in 32-row boxes), packed batches and split-KV slices included
  const uint64_t q_heads = varlen ? static_cast<uint64_t>(H) : static_cast<uint64_t>(B) * H;
  const uint64_t kv_heads = varlen ? static_cast<uint64_t>(Hkv) : static_cast<uint64_t>(B) * Hkv;
  if (encode_rows_map(&p.tm_q, q, d, N, q_heads) != CUDA_SUCCESS ||
      encode_rows_map(&p.tm_k, k, d, N, kv_heads, 64u) != CUDA_SUCCESS ||
      encode_rows_map(&p.tm_v, v, d, N, kv_heads) != CUDA_SUCCESS ||
      encode_rows_map(&p.tm_o, o, d, N, q_heads, 32u) != CUDA_SUCCESS)
    return ATTN_ERR_LAUNCH;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.cu_seqlens = cu_seqlens;
  p.status = status_word();
  if (!p.status) return ATTN_ERR_LAUNCH;
  p.B = B;
  p.H = H;
  p.N = N;
  p.group = H / Hkv;
  p.n_splits = n_splits;
  p.part_o = part_o;
  p.part_stat = part_stat;
  p.n_qt = (N + 2 * kBM - 1) / (2 * kBM);  // pairs of 128-row query tiles per head
  p.scale_log2 = scale * 1.4426950408889634f;
  // work units: (query pair, key slice) per head for dense batches; for packed batches an upper
  // bound on the query pairs of all sequences per head (the kernel counts them exactly); a
  // persistent grid of clusters walks the units
  const long long grid = varlen ? static_cast<long long>(p.n_qt + B) * H
                                 : static_cast<long long>(p.n_qt) * B * H * n_splits;
  if (grid > INT_MAX) return ATTN_ERR_SHAPE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_fwd_2sm(p, d, causal != 0, varlen, static_cast<int>(grid), st);
  if (e == cudaSuccess && n_splits > 1)
    e = launch_splitkv_combine(d, part_o, part_stat, o, lse, static_cast<long long>(B) * H * N,
                               n_splits, st);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

// Split-KV workspace: partial O [S][B H N][d] fp32, then [2][S][B H N] fp32 statistics.
static size_t splitkv_bytes(int B, int H, int N, int d, int S) {
  const size_t rows = static_cast<size_t>(B) * H * N;
  const size_t o_bytes = (static_cast<size_t>(S) * rows * d * 4 + 255) / 256 * 256;
  return o_bytes + (2 * static_cast<size_t>(S) * rows * 4 + 255) / 256 * 256;
}

}  // namespace attn

using namespace attn;

extern "C" int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                        const int32_t* cu_seqlens, int B, int H, int N, int d, int causal,
                        float scale, void* stream) {
  return fwd_impl(q, k, v, o, lse, cu_seqlens, B, H, H, N, d, causal, scale, stream);
}

extern "C" int attn_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse,
                            const int32_t* cu_seqlens, int B, int H, int H_kv, int N, int d,
                            int causal, float scale, void* stream) {
  return fwd_impl(q, k, v, o, lse, cu_seqlens, B, H, H_kv, N, d, causal, scale, stream);
}

extern "C" int attn_fwd_splitkv_slices(int B, int H, int N, int d, int num_splits) {
  if (B <= 0 || H <= 0 || N <= 0 || (d != 64 && d != 128)) return 0;
  return splitkv_pick(B, H, N, d, num_splits);
}

extern "C" size_t attn_fwd_splitkv_workspace_bytes(int B, int H, int N, int d, int num_splits) {
  if (B <= 0 || H <= 0 || N <= 0 || (d != 64 && d != 128)) return 0;
  const int S = splitkv_pick(B, H, N, d, num_splits);
  return S > 1 ? splitkv_bytes(B, H, N, d, S) : 0;
}

extern "C" int attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                                int B, int H, int N, int d, int causal, float scale,
                                int num_splits, void* workspace, size_t workspace_bytes,
                                void* stream) {
  bool empty = false;
  const int rc = validate(q, k, v, o, lse, nullptr, B, H, N, d, scale, &empty);
  if (rc != ATTN_OK || empty) return rc;
  const int S = splitkv_pick(B, H, N, d, num_splits);
  if (S == 1) return fwd_impl(q, k, v, o, lse, nullptr, B, H, H, N, d, causal, scale, stream);
  const size_t need = splitkv_bytes(B, H, N, d, S);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < need)
    return ATTN_ERR_WORKSPACE;
  float* part_o = static_cast<float*>(workspace);
  const size_t rows = static_cast<size_t>(B) * H * N;
  float* part_stat = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                              (static_cast<size_t>(S) * rows * d * 4 + 255) /
                                                  256 * 256);
  return fwd_impl(q, k, v, o, lse, nullptr, B, H, H, N, d, causal, scale, stream, S, part_o,
                  part_stat);
}

// Backward workspace: two fp32 planes [B*H][n_pad] (-lse * log2(e), then -D), each rounded up to
// 256 bytes.
static size_t bwd_plane_bytes(int B, int H, int N) {
  const size_t n_pad = (static_cast<size_t>(N) + kBM - 1) / kBM * kBM;
  return (static_cast<size_t>(B) * H * n_pad * 4 + 255) / 256 * 256;
}

extern "C" size_t attn_bwd_workspace_bytes(int B, int H, int N, int d) {
  if (B <= 0 || H <= 0 || N <= 0 || (d != 64 && d != 128)) return 0;
  return 2 * bwd_plane_bytes(B, H, N);
}

static int bwd_impl(const void* q, const void* k, const void* v, const void* o,
                    const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                    int H, int Hkv, int N, int d, int causal, float scale, void* workspace,
                    size_t workspace_bytes, void* stream) {
  bool empty = false;
  int rc = validate(q, k, v, o, lse, nullptr, B, H, N, d, scale, &empty);
  if (rc != ATTN_OK) return rc;
  if (Hkv < 0 || (H > 0 && (Hkv == 0 || H % Hkv != 0))) return ATTN_ERR_SHAPE;
  if (empty) return ATTN_OK;
  if (!dout || !dq || !dk || !dv) return ATTN_ERR_NULL;
  if (!aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return ATTN_ERR_ALIGN;
  const size_t plane = bwd_plane_bytes(B, H, N);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) ||
      workspace_bytes < 2 * plane)
    return ATTN_ERR_WORKSPACE;
  if ((rc = check_device()) != 0) return rc;
  BwdParams p{};
  const uint64_t heads = static_cast<uint64_t>(B) * H;
  const uint64_t kv_heads = static_cast<uint64_t>(B) * Hkv;
  if (encode_rows_map(&p.tm_q, q, d, N, heads) != CUDA_SUCCESS ||
      encode_rows_map(&p.tm_k, k, d, N, kv_heads) != CUDA_SUCCESS ||
      encode_rows_map(&p.tm_v, v, d, N, kv_heads) != CUDA_SUCCESS ||
      encode_rows_map(&p.tm_do, dout, d, N, heads) != CUDA_SUCCESS)
    return ATTN_ERR_LAUNCH;
  // head dim 128: the tile passes write dQ, dK, dV by TMA stores of 32-row staging tiles
  if (d == 128 && (encode_rows_map(&p.tm_dq, dq, d, N, heads, 32u) != CUDA_SUCCESS ||
                   encode_rows_map(&p.tm_dk, dk, d, N, kv_heads, 32u) != CUDA_SUCCESS ||
                   encode_rows_map(&p.tm_dv, dv, d, N, kv_heads, 32u) != CUDA_SUCCESS))
    return ATTN_ERR_LAUNCH;
  p.H_kv = Hkv;
  p.group = H / Hkv;
  p.dq = static_cast<__nv_bfloat16*>(dq);
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  float* nlse2 = static_cast<float*>(workspace);
  float* nd = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + plane);
  p.nlse2 = nlse2;
  p.nd = nd;
  p.status = status_word();
  if (!p.status) return ATTN_ERR_LAUNCH;
  p.B = B;
  p.H = H;
  p.N = N;
  p.n_tiles = (N + kBM - 1) / kBM;
  p.n_pad = p.n_tiles * kBM;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_bwd_prep(o, dout, lse, nlse2, nd, B * H, N, p.n_pad, d, st);
  if (e == cudaSuccess)
    e = (d == 64) ? launch_bwd_d64(p, causal != 0, st) : launch_bwd_d128(p, causal != 0, st);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

// Packed backward workspace: two fp32 planes of H * 128 * (ceil(T/128) + B) rows (one 128-row
// tile per tile slot of the batch), each rounded up to 256 bytes.
static size_t bwd_varlen_plane_bytes(int B, int H, int T) {
  const size_t slots = (static_cast<size_t>(T) + kBM - 1) / kBM + static_cast<size_t>(B);
  return (static_cast<size_t>(H) * slots * kBM * 4 + 255) / 256 * 256;
}

extern "C" size_t attn_bwd_varlen_workspace_bytes(int B, int H, int T, int d) {
  if (B <= 0 || H <= 0 || T < 0 || (d != 64 && d != 128)) return 0;
  return 2 * bwd_varlen_plane_bytes(B, H, T);
}

extern "C" int attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o,
                               const float* lse, const void* dout, void* dq, void* dk, void* dv,
                               const int32_t* cu_seqlens, int B, int H, int H_kv, int T, int d,
                               int causal, float scale, void* workspace, size_t workspace_bytes,
                               void* stream) {
  if (!cu_seqlens) return ATTN_ERR_NULL;
  bool empty = false;
  int rc = validate(q, k, v, o, lse, cu_seqlens, B, H, T, d, scale, &empty);
  if (rc != ATTN_OK) return rc;
  if (H_kv < 0 || (H > 0 && (H_kv == 0 || H % H_kv != 0))) return ATTN_ERR_SHAPE;
  if (empty) return ATTN_OK;
  if (!dout || !dq || !dk || !dv) return ATTN_ERR_NULL;
  if (!aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return ATTN_ERR_ALIGN;
  const long long slots = (static_cast<long long>(T) + kBM - 1) / kBM + B;
  if (slots * H > INT_MAX) return ATTN_ERR_SHAPE;
  const size_t plane = bwd_varlen_plane_bytes(B, H, T);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) ||
      workspace_bytes < 2 * plane)
    return ATTN_ERR_WORKSPACE;
  if ((rc = check_device()) != 0) return rc;
  BwdParams p{};
  if (encode_rows_map(&p.tm_q, q, d, T, H) != CUDA_SUCCESS ||
      encode_rows_map(&p.tm_k, k, d, T, H_kv) != CUDA_SUCCESS ||
      encode_rows_map(&p.tm_v, v, d, T, H_kv) != CUDA_SUCCESS ||
      encode_rows_map(&p.tm_do, dout, d, T, H) != CUDA_SUCCESS)
    return ATTN_ERR_LAUNCH;
  // head dim 128: warps whose 32 rows lie inside their sequence write by TMA stores
  if (d == 128 && (encode_rows_map(&p.tm_dq, dq, d, T, H, 32u) != CUDA_SUCCESS ||
                   encode_rows_map(&p.tm_dk, dk, d, T, H_kv, 32u) != CUDA_SUCCESS ||
                   encode_rows_map(&p.tm_dv, dv, d, T, H_kv, 32u) != CUDA_SUCCESS))
    return ATTN_ERR_LAUNCH;
  p.dq = static_cast<__nv_bfloat16*>(dq);
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  float* nlse2 = static_cast<float*>(workspace);
  float* nd = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + plane);
  p.nlse2 = nlse2;
  p.nd = nd;
  p.status = status_word();
  if (!p.status) return ATTN_ERR_LAUNCH;
  p.cu_seqlens = cu_seqlens;
  p.n_seqs = B;
  p.B = 1;
  p.H = H;
  p.N = T;
  p.H_kv = H_kv;
  p.group = H / H_kv;
  p.n_tiles = static_cast<int>(slots);
  p.n_pad = p.n_tiles * kBM;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e =
      launch_bwd_prep_varlen(o, dout, lse, nlse2, nd, cu_seqlens, B, H, T, p.n_tiles, d, st);
  if (e == cudaSuccess)
    e = (d == 64) ? launch_bwd_d64(p, causal != 0, st) : launch_bwd_d128(p, causal != 0, st);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

extern "C" int attn_bwd(const void* q, const void* k, const void* v, const void* o,
                        const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                        int H, int N, int d, int causal, float scale, void* workspace,
                        size_t workspace_bytes, void* stream) {
  return bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, B, H, H, N, d, causal, scale, workspace,
                  workspace_bytes, stream);
}

extern "C" int attn_bwd_gqa(const void* q, const void* k, const void* v, const void* o,
                            const float* lse, const void* dout, void* dq, void* dk, void* dv,
                            int B, int H, int H_kv, int N, int d, int causal, float scale,
                            void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, B, H, H_kv, N, d, causal, scale, workspace,
                  workspace_bytes, stream);
}

extern "C" int attn_quantize_fp8(const void* x, void* codes, float* scales, int B, int H, int N,
                                 int d, int transpose, void* stream) {
  if (B < 0 || H < 0 || N < 0) return ATTN_ERR_SHAPE;
  if (B == 0 || H == 0 || N == 0) return ATTN_OK;
  if (d != 64 && d != 128) return ATTN_ERR_HEAD_DIM;
  if (!x || !codes || !scales) return ATTN_ERR_NULL;
  if (!aligned16(x) || !aligned16(codes) || (reinterpret_cast<uintptr_t>(scales) & 3u))
    return ATTN_ERR_ALIGN;
  const long long tiles = (static_cast<long long>(N) + kBM - 1) / kBM;
  if (tiles * B * H > INT_MAX) return ATTN_ERR_SHAPE;
  int rc = check_device();
  if (rc != 0) return rc;
  const cudaError_t e = launch_quantize_fp8(x, codes, scales, B * H, N, d, transpose != 0,
                                            static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

extern "C" int attn_fwd_fp8(const void* q8, const float* sq, const void* k8, const float* sk,
                            const void* vt8, const float* sv, void* o, float* lse, int B, int H,
                            int N, int d, int causal, float scale, void* stream) {
  if (B < 0 || H < 0 || N < 0) return ATTN_ERR_SHAPE;
  if (B == 0 || H == 0 || N == 0) return ATTN_OK;
  if (d != 128) return ATTN_ERR_HEAD_DIM;
  if (!q8 || !sq || !k8 || !sk || !vt8 || !sv || !o || !lse) return ATTN_ERR_NULL;
  if (!aligned16(q8) || !aligned16(k8) || !aligned16(vt8) || !aligned16(o) || !aligned16(lse) ||
      ((reinterpret_cast<uintptr_t>(sq) | reinterpret_cast<uintptr_t>(sk) |
        reinterpret_cast<uintptr_t>(sv)) & 3u))
    return ATTN_ERR_ALIGN;
  if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_SCALE;
  const long long pairs = (static_cast<long long>(N) + 2 * kBM - 1) / (2 * kBM);
  if (pairs * B * H > INT_MAX) return ATTN_ERR_SHAPE;
  int rc = check_device();
  if (rc != 0) return rc;
  Fp8Params p{};
  const uint64_t heads = static_cast<uint64_t>(B) * H;
  const int n_tiles = (N + kBM - 1) / kBM;
  if (encode_u8_map(&p.tm_q, q8, 128, N, heads) != CUDA_SUCCESS ||
      encode_u8_map(&p.tm_k, k8, 128, N, heads) != CUDA_SUCCESS ||
      encode_u8_map(&p.tm_vt, vt8, static_cast<uint64_t>(n_tiles) * kBM, 128, heads) !=
          CUDA_SUCCESS)
    return ATTN_ERR_LAUNCH;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.sq = sq;
  p.sk = sk;
  p.sv = sv;
  p.status = status_word();
  if (!p.status) return ATTN_ERR_LAUNCH;
  p.B = B;
  p.H = H;
  p.N = N;
  p.n_tiles = n_tiles;
  p.n_qt = static_cast<int>(pairs);
  p.scale_log2 = scale * 1.4426950408889634f;
  const cudaError_t e = launch_fwd_fp8(p, causal != 0, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

extern "C" int attn_fwd_unfused(const void* q, const void* k, const void* v, void* o, float* lse,
                                const int32_t* cu_seqlens, int B, int H, int N, int d, int causal,
                                float scale, void* workspace, size_t workspace_bytes,
                                void* stream) {
  if (cu_seqlens != nullptr) return ATTN_ERR_UNSUPPORTED;
  bool empty = false;
  int rc = validate(q, k, v, o, lse, nullptr, B, H, N, d, scale, &empty);
  if (rc != ATTN_OK || empty) return rc;
  const size_t need = attn_fwd_unfused_workspace_bytes(B, H, N, d);
  if (need == 0) return ATTN_ERR_SHAPE;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < need)
    return ATTN_ERR_WORKSPACE;
  if ((rc = check_device()) != 0) return rc;
  UnfusedArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.workspace = workspace;
  a.B = B;
  a.H = H;
  a.N = N;
  a.d = d;
  a.causal = causal != 0;
  a.scale = scale;
  a.status = status_word();
  if (!a.status) return ATTN_ERR_LAUNCH;
  return launch_unfused(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? ATTN_OK
                                                                             : ATTN_ERR_LAUNCH;
}

extern "C" size_t attn_fwd_unfused_workspace_bytes(int B, int H, int N, int d) {
  if (B <= 0 || H <= 0 || N <= 0 || (d != 64 && d != 128)) return 0;
  return unfused_workspace_layout(B, H, N).total;
}

extern "C" int attn_get_last_device_error(void* stream) {
  int* addr = status_word();
  if (!addr) return ATTN_ERR_LAUNCH;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int value = 0;
  if (cudaMemcpyAsync(&value, addr, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return ATTN_ERR_LAUNCH;
  if (value != 0) {
    const int zero = 0;
    if (cudaMemcpyAsync(addr, &zero, sizeof(int), cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
      return ATTN_ERR_LAUNCH;
  }
  return value;
}

extern "C" int attn_version(void) { return 100; }
