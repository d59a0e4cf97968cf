// Host-side launch functions of the sm_103a kernels (internal to libsparge).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "sparge.h"

namespace sparge {

// Geometry derived from a validated sparge_shape.
struct Geom {
  int B, H, N, d, bq, bk;
  int BH, Mq, Mk, Mkw;  // Mkw = ceil(Mk / 32) bitmask words per row
};

Geom make_geom(const sparge_shape& s);

// Rows of the pooled map one selection CTA handles (fits its logits in smem).
int select_rows_per_cta(int Mk);

// pool.cu / mask.cu
cudaError_t launch_pool(const Geom& g, const void* q, const void* k, float* qbar, float* kbar,
                        cudaStream_t st);
cudaError_t launch_select_from_prob(const Geom& g, const float* prob, int ktop, float p,
                                    uint32_t* bitmask, int32_t* row_idx, int32_t* row_cnt,
                                    cudaStream_t st);
cudaError_t launch_csc(const Geom& g, const uint32_t* bitmask, int32_t* col_idx, int32_t* col_cnt,
                       cudaStream_t st);
// The mask as kernels chained by programmatic dependent launch (mask.cu):
// pooling into qbar [BH, Mq, d] and kbar [BH, Mk, d], tensor-core pooled
// logits into `logits` [BH, Mq, Mk] (fp32), selection, column lists.
cudaError_t launch_mask_pipeline(const Geom& g, const void* q, const void* k, void* qhi,
                                 void* qlo, void* khi, void* klo, float* logits, float scale,
                                 int ktop, float p, uint32_t* bitmask, int32_t* row_idx,
                                 int32_t* row_cnt, int32_t* col_idx, int32_t* col_cnt,
                                 float* logit_out, float* prob_out, int32_t* status,
                                 cudaStream_t st);

// attn_fwd.cu
cudaError_t launch_attn_fwd(const Geom& g, const void* q, const void* k, const void* v,
                            const int32_t* row_idx, const int32_t* row_cnt, float scale, void* o,
                            float* lse, int32_t* status, cudaStream_t st);

// attn_bwd.cu.  Workspace: D = rowsum(dO*O) fp32 [BH, N]; the q-block
// work order [BH*Mq] (long lists first, then the rest in descending index
// order); int32 [4]: the work counters of the persistent gradient kernels
// and the dK/dV item count; five int32 arrays over the dK/dV items
// [<= BH*Mt + 128]: key tile and part word in launch order, then key tile,
// part word and work in tile order; the completion counters of cut tiles
// (int32 [1024]) and their fp32 partial dV | dK slots [128][128][2][d].
// The first kernel of each call rewrites the orders, items and counts and
// zeroes the counters.
struct BwdWorkspace {
  float* delta;
  int32_t* row_order;
  int32_t* work;
  int32_t* seq_tile;
  int32_t* seq_part;
  int32_t* item_tile;
  int32_t* item_part;
  int32_t* item_work;
  int32_t* split_cnt;
  float* split_part;
};
size_t bwd_workspace_bytes(const Geom& g);
BwdWorkspace bwd_workspace_layout(const Geom& g, void* base);
cudaError_t launch_attn_bwd(const Geom& g, const void* q, const void* k, const void* v,
                            const void* o, const float* lse, const void* dout,
                            const int32_t* row_idx, const int32_t* row_cnt,
                            const int32_t* col_idx, const int32_t* col_cnt, float scale, void* dq,
                            void* dk, void* dv, void* workspace, int32_t* status, cudaStream_t st);

// api.cu
cudaError_t launch_wait_probe(int32_t* status, uint64_t timeout_ns, cudaStream_t st);
// Every argument check of sparge_mask (no CUDA call); SPARGE_OK or the error.
int validate_mask_args(const sparge_shape* shape, const void* q, const void* k, float k_frac,
                       float p, float softmax_scale, const uint32_t* bitmask,
                       const int32_t* row_idx, const int32_t* row_cnt, const int32_t* col_idx,
                       const int32_t* col_cnt, const float* pooled_prob,
                       const float* pooled_logit, const int32_t* status);

// tma.cu: 3-D bf16 tensor map over [BH, N, d] with a (64 x box_rows) 128-byte-swizzled box.
int make_tmap_bf16(void* tmap_out, const void* base, int BH, int N, int d, int box_rows);

}  // namespace sparge
