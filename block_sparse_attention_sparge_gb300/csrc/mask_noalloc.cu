// sparge_mask_noalloc: the block-mask construction of sparge_mask for callers
// that cannot allocate device memory.
//
// Some callers of this library cannot call cudaMalloc: runtimes that hand out
// all device memory through their own pool allocator (a foreign cudaMalloc
// would escape their accounting, or fail because the pool already reserved
// the memory), and latency-critical loops in which an allocation or free may
// synchronise the device.  sparge_mask needs a caller-provided workspace for
// its fp32 pooled Q and K; this variant instead keeps that scratch in a
// file-scope device array of fixed size, so the caller passes only inputs
// and outputs.
//
// The array exists once per GPU that loads the library and stays allocated
// until the process exits.  Host code cannot use the array's name as a device
// address, so on the first call on each device (with that device current) the
// address is looked up once with cudaGetSymbolAddress and cached.
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>

#include "kernels.h"
#include "sparge.h"

namespace sparge {
namespace {

// Upper bound of the scratch: pooled Q and K (B*H*d*(Mq + Mk)*4 bytes) and
// the pooled logits (B*H*Mq*Mk*4 bytes) up to 16 MiB, e.g. the 480p video
// shape (B=1, H=12, N=32760, d=128) needs 10.9 MB.
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;

static __device__ __align__(256) unsigned char g_mask_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of this GPU's copy of g_mask_scratch (looked up on first use).
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPARGE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SPARGE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_mask_scratch) != cudaSuccess || p == nullptr)
      return SPARGE_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return SPARGE_OK;
}

}  // namespace
}  // namespace sparge

extern "C" int sparge_mask_noalloc(const sparge_shape* shape, const void* q, const void* k,
                                   float k_frac, float p, float softmax_scale, uint32_t* bitmask,
                                   int32_t* row_idx, int32_t* row_cnt, int32_t* col_idx,
                                   int32_t* col_cnt, float* pooled_logit, float* pooled_prob,
                                   int32_t* status, sparge_stream_t stream) {
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
                     col_cnt, pooled_logit, pooled_prob, scratch, sparge::kNoAllocScratchBytes,
                     status, stream);
}
