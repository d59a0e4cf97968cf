// sparge_mask_noalloc: the block-mask construction of sparge_mask for callers
// that cannot allocate device memory.
//
// Some callers of this library cannot call cudaMalloc: runtimes that hand out
// all device memory through their own pool allocator (a foreign cudaMalloc
// would escape their accounting, or fail because the pool already reserved
// the memory), and latency-critical loops in which an allocation or free may
// synchronise the device.  sparge_mask needs a caller-provided workspace for
// the pooled Q and K (bf16 high / low pairs) and the fp32 pooled logits; this
// variant keeps that scratch in a file-scope device array of fixed size
// instead, so the caller passes only inputs and outputs.
//
// The array exists once per GPU that loads the library and stays allocated
// until the process exits.  Host code cannot use the array's name as a device
// address, so its address is looked up with cudaGetSymbolAddress in the
// current CUDA context and cached under that context's unique id: a device
// reset (which destroys the primary context) or a caller-made context gets a
// lookup of its own instead of a stale address.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>

#include "kernels.h"
#include "sparge.h"

namespace sparge {
namespace {

// Upper bound of the scratch: pooled Q and K (B*H*d*(Mq + Mk)*4 bytes as bf16
// pairs) and the pooled logits (B*H*Mq*Mk*4 bytes) up to 16 MiB, e.g. the 480p
// video shape (B=1, H=12, N=32760, d=128) needs 10.9 MB.
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;

static __device__ __align__(256) unsigned char g_mask_scratch[kNoAllocScratchBytes];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

struct DriverFns {
  CtxGetCurrentFn get_current = nullptr;
  CtxGetIdFn get_id = nullptr;
};

// Driver entry points, resolved once through the runtime (no link-time libcuda).
const DriverFns& driver_fns() {
  static DriverFns fns = []() {
    DriverFns f;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.get_id = reinterpret_cast<CtxGetIdFn>(p);
    return f;
  }();
  return fns;
}

// Unique id of the current context (0 when none is current yet).
int current_context_id(unsigned long long* id) {
  const DriverFns& f = driver_fns();
  if (f.get_current == nullptr || f.get_id == nullptr) return SPARGE_ERR_CUDA;
  CUcontext ctx = nullptr;
  if (f.get_current(&ctx) != CUDA_SUCCESS) return SPARGE_ERR_CUDA;
  *id = 0;
  if (ctx != nullptr && f.get_id(ctx, id) != CUDA_SUCCESS) return SPARGE_ERR_CUDA;
  return SPARGE_OK;
}

constexpr int kCacheSlots = 64;
std::mutex g_scratch_mu;
unsigned long long g_ctx_id[kCacheSlots] = {};
void* g_scratch_addr[kCacheSlots] = {};
int g_cached = 0;

// Device address of g_mask_scratch in the current context.
int scratch_address(void** out) {
  unsigned long long id = 0;
  if (current_context_id(&id) != SPARGE_OK) return SPARGE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  for (int i = 0; i < g_cached && id != 0; ++i) {
    if (g_ctx_id[i] == id) {
      *out = g_scratch_addr[i];
      return SPARGE_OK;
    }
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_mask_scratch) != cudaSuccess || p == nullptr) {
    cudaGetLastError();  // clear it: a later cudaGetLastError must not report it
    return SPARGE_ERR_CUDA;
  }
  // With no context current before the lookup, the runtime has just made the
  // device's primary context current: key the cache by that one.
  if (id == 0 && current_context_id(&id) != SPARGE_OK) return SPARGE_ERR_CUDA;
  if (id != 0 && g_cached < kCacheSlots) {
    g_ctx_id[g_cached] = id;
    g_scratch_addr[g_cached] = p;
    ++g_cached;
  }
  *out = p;
  return SPARGE_OK;
}

}  // namespace
}  // namespace sparge

extern "C" int sparge_mask_noalloc(const sparge_shape* shape, const void* q, const void* k,
                                   float k_frac, float p, float softmax_scale, uint32_t* bitmask,
                                   int32_t* row_idx, int32_t* row_cnt, int32_t* col_idx,
                                   int32_t* col_cnt, float* pooled_prob, float* pooled_logit,
                                   int32_t* status, sparge_stream_t stream) {
  // Every argument is checked before the first CUDA call.
  const int rv = sparge::validate_mask_args(shape, q, k, k_frac, p, softmax_scale, bitmask,
                                            row_idx, row_cnt, col_idx, col_cnt, pooled_prob,
                                            pooled_logit, status);
  if (rv != SPARGE_OK) return rv;
  size_t need = 0;
  const int rc = sparge_mask_workspace_bytes(shape, &need);
  if (rc != SPARGE_OK) return rc;
  if (need > sparge::kNoAllocScratchBytes) return SPARGE_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int rs = sparge::scratch_address(&scratch);
  if (rs != SPARGE_OK) return rs;
  // The pooling kernels overwrite every scratch byte the selection reads, so
  // nothing has to be cleared between calls.
  return sparge_mask(shape, q, k, k_frac, p, softmax_scale, bitmask, row_idx, row_cnt, col_idx,
                     col_cnt, pooled_prob, pooled_logit, scratch, sparge::kNoAllocScratchBytes,
                     status, stream);
}
