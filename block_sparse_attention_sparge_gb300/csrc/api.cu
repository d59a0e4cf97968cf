// C ABI of libsparge: argument validation, workspace layout and launches.
// Every check runs before the first CUDA call, so an invalid call returns a
// negative status without touching the device.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "common.cuh"
#include "kernels.h"
#include "sparge.h"

namespace sparge {

Geom make_geom(const sparge_shape& s) {
  Geom g;
  g.B = s.B;
  g.H = s.H;
  g.N = s.N;
  g.d = s.d;
  g.bq = s.block_q;
  g.bk = s.block_kv;
  g.BH = s.B * s.H;
  g.Mq = (s.N + s.block_q - 1) / s.block_q;
  g.Mk = (s.N + s.block_kv - 1) / s.block_kv;
  g.Mkw = (g.Mk + 31) / 32;
  return g;
}

namespace {

constexpr int kMaxN = 524288;  // Mk <= 8192
constexpr size_t kAlign = 256;

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

int check_shape(const sparge_shape* s) {
  if (s == nullptr) return SPARGE_ERR_INVALID_ARG;
  if (s->B < 1 || s->H < 1 || s->N < 1 || s->d < 1 || s->block_q < 1 || s->block_kv < 1)
    return SPARGE_ERR_INVALID_ARG;
  if ((long long)s->B * s->H > 65535LL * 1024LL) return SPARGE_ERR_INVALID_ARG;
  if (s->d != 64 && s->d != 128) return SPARGE_ERR_UNSUPPORTED;
  if (s->block_q != 128 || (s->block_kv != 64 && s->block_kv != 128)) return SPARGE_ERR_UNSUPPORTED;
  if (s->N > kMaxN) return SPARGE_ERR_UNSUPPORTED;
  return SPARGE_OK;
}

int check_tensor(const void* p) {
  if (p == nullptr) return SPARGE_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(p) % 16 != 0) return SPARGE_ERR_MISALIGNED;
  return SPARGE_OK;
}

int check_word(const void* p) {
  if (p == nullptr) return SPARGE_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(p) % 4 != 0) return SPARGE_ERR_MISALIGNED;
  return SPARGE_OK;
}

int check_opt_word(const void* p) { return p == nullptr ? SPARGE_OK : check_word(p); }

#define SPARGE_TRY(expr)          \
  do {                            \
    const int rc_ = (expr);       \
    if (rc_ != SPARGE_OK) return rc_; \
  } while (0)

int cuda_status(cudaError_t e) { return e == cudaSuccess ? SPARGE_OK : SPARGE_ERR_CUDA; }

float resolve_scale(float scale, int d) {
  return scale == 0.f ? 1.0f / sqrtf(static_cast<float>(d)) : scale;
}

int topk_blocks(float k_frac, int Mk) {
  const double k = static_cast<double>(k_frac);
  if (k >= 1.0) return Mk;
  long long c = static_cast<long long>(ceil(k * Mk - 1e-4));
  if (c < 1) c = 1;
  if (c > Mk) c = Mk;
  return static_cast<int>(c);
}

int check_kp(float k_frac, float p) {
  if (!isfinite(k_frac) || !(k_frac > 0.f) || k_frac > 1.f) return SPARGE_ERR_INVALID_ARG;
  if (!isfinite(p) || p < 0.f || p > 1.f) return SPARGE_ERR_INVALID_ARG;
  return SPARGE_OK;
}

// Mask workspace: the Q means [BH, Mq, d] and the K means [BH, Mk, d], each
// as a bf16 pair hi, lo (four arrays), then the pooled logits [BH, Mq, Mk]
// fp32.
size_t mask_ws_bytes(const Geom& g) {
  return 2 * round_up((size_t)g.BH * g.Mq * g.d * 2) + 2 * round_up((size_t)g.BH * g.Mk * g.d * 2) +
         round_up((size_t)g.BH * g.Mq * g.Mk * sizeof(float));
}

size_t bwd_ws_bytes(const Geom& g) { return bwd_workspace_bytes(g); }

// ---------------------------------------------------------------- wait probe
__global__ void wait_probe_kernel(int32_t* status, uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    fence_barrier_init();
  }
  __syncthreads();
  // Nothing arrives on `bar`: the bounded wait must give up and report.
  if (!mbar_wait(b, 0, timeout_ns)) report_error(status, SPARGE_ERR_TIMEOUT);
}

}  // namespace

cudaError_t launch_wait_probe(int32_t* status, uint64_t timeout_ns, cudaStream_t st) {
  wait_probe_kernel<<<1, 32, 0, st>>>(status, timeout_ns);
  return cudaGetLastError();
}

int validate_mask_args(const sparge_shape* shape, const void* q, const void* k, float k_frac,
                       float p, float softmax_scale, const uint32_t* bitmask,
                       const int32_t* row_idx, const int32_t* row_cnt, const int32_t* col_idx,
                       const int32_t* col_cnt, const float* pooled_prob,
                       const float* pooled_logit, const int32_t* status) {
  SPARGE_TRY(check_shape(shape));
  SPARGE_TRY(check_tensor(q));
  SPARGE_TRY(check_tensor(k));
  SPARGE_TRY(check_kp(k_frac, p));
  SPARGE_TRY(check_opt_word(status));
  if (!isfinite(softmax_scale)) return SPARGE_ERR_INVALID_ARG;
  SPARGE_TRY(check_word(bitmask));
  SPARGE_TRY(check_word(row_idx));
  SPARGE_TRY(check_word(row_cnt));
  if ((col_idx == nullptr) != (col_cnt == nullptr)) return SPARGE_ERR_INVALID_ARG;
  SPARGE_TRY(check_opt_word(col_idx));
  SPARGE_TRY(check_opt_word(col_cnt));
  SPARGE_TRY(check_opt_word(pooled_prob));
  SPARGE_TRY(check_opt_word(pooled_logit));
  return SPARGE_OK;
}

}  // namespace sparge

using namespace sparge;

extern "C" {

int sparge_version(void) { return 100; }

const char* sparge_status_string(int status) {
  switch (status) {
    case SPARGE_OK: return "SPARGE_OK";
    case SPARGE_ERR_INVALID_ARG: return "SPARGE_ERR_INVALID_ARG: invalid argument";
    case SPARGE_ERR_UNSUPPORTED: return "SPARGE_ERR_UNSUPPORTED: unsupported head dim or block size";
    case SPARGE_ERR_MISALIGNED: return "SPARGE_ERR_MISALIGNED: pointer not 16-byte aligned";
    case SPARGE_ERR_WORKSPACE: return "SPARGE_ERR_WORKSPACE: workspace missing or too small";
    case SPARGE_ERR_CUDA: return "SPARGE_ERR_CUDA: CUDA call failed";
    case SPARGE_ERR_TIMEOUT: return "SPARGE_ERR_TIMEOUT: device wait gave up";
    default: return "SPARGE_ERR_UNKNOWN";
  }
}

int sparge_pool(const sparge_shape* shape, const void* q, const void* k, float* qbar, float* kbar,
                sparge_stream_t stream) {
  SPARGE_TRY(check_shape(shape));
  if (qbar == nullptr && kbar == nullptr) return SPARGE_ERR_INVALID_ARG;
  if (qbar) SPARGE_TRY(check_tensor(q));
  if (kbar) SPARGE_TRY(check_tensor(k));
  SPARGE_TRY(check_opt_word(qbar));
  SPARGE_TRY(check_opt_word(kbar));
  const Geom g = make_geom(*shape);
  return cuda_status(launch_pool(g, q, k, qbar, kbar, stream));
}

int sparge_mask_workspace_bytes(const sparge_shape* shape, size_t* bytes) {
  SPARGE_TRY(check_shape(shape));
  if (bytes == nullptr) return SPARGE_ERR_INVALID_ARG;
  *bytes = mask_ws_bytes(make_geom(*shape));
  return SPARGE_OK;
}

int sparge_mask(const sparge_shape* shape, const void* q, const void* k, float k_frac, float p,
                float softmax_scale, uint32_t* bitmask, int32_t* row_idx, int32_t* row_cnt,
                int32_t* col_idx, int32_t* col_cnt, float* pooled_prob, float* pooled_logit,
                void* workspace, size_t ws_bytes, int32_t* status, sparge_stream_t stream) {
  SPARGE_TRY(validate_mask_args(shape, q, k, k_frac, p, softmax_scale, bitmask, row_idx, row_cnt,
                                col_idx, col_cnt, pooled_prob, pooled_logit, status));
  const Geom g = make_geom(*shape);
  if (workspace == nullptr || ws_bytes < mask_ws_bytes(g)) return SPARGE_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) % 16 != 0) return SPARGE_ERR_MISALIGNED;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t qb = round_up((size_t)g.BH * g.Mq * g.d * 2);
  const size_t kb = round_up((size_t)g.BH * g.Mk * g.d * 2);
  void* qhi = ws;
  void* qlo = ws + qb;
  void* khi = ws + 2 * qb;
  void* klo = ws + 2 * qb + kb;
  float* logits = reinterpret_cast<float*>(ws + 2 * qb + 2 * kb);
  const float scale = resolve_scale(softmax_scale, g.d);
  return cuda_status(launch_mask_pipeline(g, q, k, qhi, qlo, khi, klo, logits, scale,
                                          topk_blocks(k_frac, g.Mk), p, bitmask, row_idx, row_cnt,
                                          col_idx, col_cnt, pooled_logit, pooled_prob, status,
                                          stream));
}

int sparge_mask_from_prob(const sparge_shape* shape, const float* prob, float k_frac, float p,
                          uint32_t* bitmask, int32_t* row_idx, int32_t* row_cnt,
                          int32_t* col_idx, int32_t* col_cnt, sparge_stream_t stream) {
  SPARGE_TRY(check_shape(shape));
  SPARGE_TRY(check_word(prob));
  SPARGE_TRY(check_kp(k_frac, p));
  SPARGE_TRY(check_word(bitmask));
  SPARGE_TRY(check_word(row_idx));
  SPARGE_TRY(check_word(row_cnt));
  if ((col_idx == nullptr) != (col_cnt == nullptr)) return SPARGE_ERR_INVALID_ARG;
  SPARGE_TRY(check_opt_word(col_idx));
  SPARGE_TRY(check_opt_word(col_cnt));
  const Geom g = make_geom(*shape);
  SPARGE_TRY(cuda_status(launch_select_from_prob(g, prob, topk_blocks(k_frac, g.Mk), p, bitmask,
                                                 row_idx, row_cnt, stream)));
  if (col_idx) SPARGE_TRY(cuda_status(launch_csc(g, bitmask, col_idx, col_cnt, stream)));
  return SPARGE_OK;
}

int sparge_attn_fwd(const sparge_shape* shape, const void* q, const void* k, const void* v,
                    const int32_t* row_idx, const int32_t* row_cnt, float softmax_scale,
                    void* o, float* lse, int32_t* status, sparge_stream_t stream) {
  SPARGE_TRY(check_shape(shape));
  SPARGE_TRY(check_tensor(q));
  SPARGE_TRY(check_tensor(k));
  SPARGE_TRY(check_tensor(v));
  SPARGE_TRY(check_tensor(o));
  SPARGE_TRY(check_word(row_idx));
  SPARGE_TRY(check_word(row_cnt));
  SPARGE_TRY(check_opt_word(lse));
  SPARGE_TRY(check_opt_word(status));
  if (!isfinite(softmax_scale)) return SPARGE_ERR_INVALID_ARG;
  const Geom g = make_geom(*shape);
  return cuda_status(launch_attn_fwd(g, q, k, v, row_idx, row_cnt,
                                     resolve_scale(softmax_scale, g.d), o, lse, status, stream));
}

int sparge_attn_bwd_workspace_bytes(const sparge_shape* shape, size_t* bytes) {
  SPARGE_TRY(check_shape(shape));
  if (bytes == nullptr) return SPARGE_ERR_INVALID_ARG;
  *bytes = bwd_ws_bytes(make_geom(*shape));
  return SPARGE_OK;
}

int sparge_attn_bwd(const sparge_shape* shape, const void* q, const void* k, const void* v,
                    const void* o, const float* lse, const void* dout, const int32_t* row_idx,
                    const int32_t* row_cnt, const int32_t* col_idx, const int32_t* col_cnt,
                    float softmax_scale, void* dq, void* dk, void* dv, void* workspace,
                    size_t ws_bytes, int32_t* status, sparge_stream_t stream) {
  SPARGE_TRY(check_shape(shape));
  SPARGE_TRY(check_tensor(q));
  SPARGE_TRY(check_tensor(k));
  SPARGE_TRY(check_tensor(v));
  SPARGE_TRY(check_tensor(o));
  SPARGE_TRY(check_tensor(dout));
  SPARGE_TRY(check_tensor(dq));
  SPARGE_TRY(check_tensor(dk));
  SPARGE_TRY(check_tensor(dv));
  SPARGE_TRY(check_word(lse));
  SPARGE_TRY(check_word(row_idx));
  SPARGE_TRY(check_word(row_cnt));
  SPARGE_TRY(check_word(col_idx));
  SPARGE_TRY(check_word(col_cnt));
  SPARGE_TRY(check_opt_word(status));
  if (!isfinite(softmax_scale)) return SPARGE_ERR_INVALID_ARG;
  const Geom g = make_geom(*shape);
  if (workspace == nullptr || ws_bytes < bwd_ws_bytes(g)) return SPARGE_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) % 16 != 0) return SPARGE_ERR_MISALIGNED;
  return cuda_status(launch_attn_bwd(g, q, k, v, o, lse, dout, row_idx, row_cnt, col_idx, col_cnt,
                                     resolve_scale(softmax_scale, g.d), dq, dk, dv, workspace,
                                     status, stream));
}

int sparge_status_copy_async(const int32_t* status, int32_t* host_status, sparge_stream_t stream) {
  SPARGE_TRY(check_word(status));
  if (host_status == nullptr) return SPARGE_ERR_INVALID_ARG;
  return cuda_status(cudaMemcpyAsync(host_status, status, sizeof(int32_t), cudaMemcpyDeviceToHost,
                                     stream));
}

int sparge_read_status(const int32_t* status, sparge_stream_t stream, int32_t* host_status) {
  SPARGE_TRY(check_word(status));
  if (host_status == nullptr) return SPARGE_ERR_INVALID_ARG;
  int32_t h = 0;
  if (cudaMemcpyAsync(&h, status, sizeof(int32_t), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return SPARGE_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return SPARGE_ERR_CUDA;
  *host_status = h;
  return SPARGE_OK;
}

int sparge_debug_wait_probe(int32_t* status, uint64_t timeout_ns, sparge_stream_t stream) {
  SPARGE_TRY(check_word(status));
  if (timeout_ns < 1000000ull) timeout_ns = 1000000ull;
  if (timeout_ns > 5000000000ull) timeout_ns = 5000000000ull;
  return cuda_status(launch_wait_probe(status, timeout_ns, stream));
}

}  // extern "C"
