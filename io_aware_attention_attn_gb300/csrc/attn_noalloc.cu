// attn_noalloc.cu -- the unfused comparison path with built-in scratch, for callers that cannot
// allocate device memory.
//
// attn_fwd_unfused needs a caller-provided workspace (the score matrix S, the probability matrix P
// and one normaliser per row).  Some callers cannot call cudaMalloc: code running under a memory
// manager that owns every device allocation, or a runtime that forbids allocation once it has
// started (allocation is synchronous and can fail).  attn_fwd_unfused_noalloc takes no workspace:
// its scratch is the file-scope array below, which every GPU that loads this library holds until
// the process exits.
//
// In host code the array's name is only a host-side stand-in, never a device address: its device
// address is looked up with cudaGetSymbolAddress on every call, with the calling device current,
// and passed to the kernels as their workspace pointer.  Nothing is cached between calls, so a
// device reset or a context torn down and re-created in between (which may load the module at
// another address) cannot leave a stale pointer behind.  The first call in a context loads the
// module there; make that first call before any stream capture.
//
// Every call shares the array and it keeps the previous call's contents.  Nothing in it has to
// start at zero: the three kernels write every element of S, P and 1/l that they later read.
// Calls whose work overlaps on the GPU (for example on two streams) race on the array.
#include "attn_gb300.h"
#include "attn_params.h"

namespace attn {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[ATTN_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array in the current context (looked up on every call).
int scratch_address(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
    return ATTN_ERR_LAUNCH;
  *out = p;
  return ATTN_OK;
}

}  // namespace
}  // namespace attn

extern "C" int attn_fwd_unfused_noalloc(const void* q, const void* k, const void* v, void* o,
                                        float* lse, int B, int H, int N, int d, int causal,
                                        float scale, void* stream) {
  // sizes are checked on the host before anything touches the GPU
  if (B < 0 || H < 0 || N < 0) return ATTN_ERR_SHAPE;
  if (B == 0 || H == 0 || N == 0) return ATTN_OK;
  if (d != 64 && d != 128) return ATTN_ERR_HEAD_DIM;
  const size_t need = attn_fwd_unfused_workspace_bytes(B, H, N, d);
  if (need == 0) return ATTN_ERR_SHAPE;
  if (need > static_cast<size_t>(ATTN_NOALLOC_SCRATCH_BYTES)) return ATTN_ERR_SCRATCH_LIMIT;
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_NULL;
  void* scratch = nullptr;
  const int rc = attn::scratch_address(&scratch);
  if (rc != ATTN_OK) return rc;
  return attn_fwd_unfused(q, k, v, o, lse, nullptr, B, H, N, d, causal, scale, scratch,
                          static_cast<size_t>(ATTN_NOALLOC_SCRATCH_BYTES), stream);
}
