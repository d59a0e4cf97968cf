/*
 * sparge.h -- C ABI of the GB300 (sm_103a) SpargeAttention2 hot path.
 *
 * The method (hybrid Top-k+Top-p block-sparse attention) is described on the
 * mindverse page "Optimierung der Effizienz von Video-Diffusionsmodellen durch
 * SpargeAttention2" (cited below as [P4] with its section name) and in the
 * abstract of "SpargeAttention2: Trainable Sparse Attention via Hybrid
 * Top-k+Top-p Masking and Distillation Fine-Tuning" ([P2] "Abstract").
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Tensors Q, K, V, O, dO, dQ, dK, dV are bf16, shape [B, H, N, d], dense
 *   row-major (d innermost), in device memory, 16-byte aligned.
 * - Blocks: block_q query tokens by block_kv key tokens.  Mq = ceil(N/block_q),
 *   Mk = ceil(N/block_kv).  The last block of each may be partial.
 * - The caller owns every buffer and the stream.  The library allocates,
 *   frees and synchronises nothing, and keeps no global mutable state apart
 *   from the fixed scratch array of sparge_mask_noalloc.  The one blocking
 *   call is sparge_read_status, a convenience that synchronises the given
 *   stream; sparge_status_copy_async reads the same word without blocking.
 * - All launches are asynchronous on `stream` (NULL = the legacy default
 *   stream).  Arguments are validated before any launch; on an error nothing
 *   is launched and a negative status is returned.
 * - `status` (nullable) is a device int32 the caller zeroes before use.  A
 *   kernel that gives up on a bounded internal wait writes SPARGE_ERR_TIMEOUT
 *   there (first error wins) and returns instead of hanging.  Read it with
 *   sparge_status_copy_async (stream-ordered) or sparge_read_status.
 * - softmax_scale 0 means 1/sqrt(d).
 */
#ifndef SPARGE_H_
#define SPARGE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* sparge_stream_t;

/* Status codes returned by every entry point. */
enum sparge_status {
  SPARGE_OK = 0,
  SPARGE_ERR_INVALID_ARG = -1, /* null pointer, bad size, k/p out of range  */
  SPARGE_ERR_UNSUPPORTED = -2, /* d or block size this build does not offer */
  SPARGE_ERR_MISALIGNED = -3,  /* a tensor pointer not 16-byte aligned      */
  SPARGE_ERR_WORKSPACE = -4,   /* workspace null or too small               */
  SPARGE_ERR_CUDA = -5,        /* a CUDA runtime/driver call failed         */
  SPARGE_ERR_TIMEOUT = -6      /* a device-side bounded wait gave up        */
};

/* Problem shape.  Supported: d in {64, 128}; block_q = 128; block_kv in
 * {64, 128}; 1 <= N <= 524288 (so Mk <= 8192); B*H >= 1.  The mask and the
 * attention calls of one problem use the same block sizes. */
typedef struct sparge_shape {
  int32_t B, H, N, d;
  int32_t block_q, block_kv;
} sparge_shape;

/* Library version (major*10000 + minor*100 + patch). */
int sparge_version(void);

/* Human-readable name of a status code (static string, never NULL). */
const char* sparge_status_string(int status);

/*
 * sparge_pool -- step 1 of the mask: per-block mean of Q and of K.
 * [P4 "Maskierungsstrategien: Top-k und Top-p"]: the mask is chosen on a
 * block-pooled attention map; the pooling is the mean over each block's
 * valid tokens.
 *   q, k  : bf16 [B,H,N,d] (device).
 *   qbar  : fp32 [B,H,Mq,d] out (device).  kbar: fp32 [B,H,Mk,d] out (device).
 * Either output may be NULL (then it is not computed).
 */
int sparge_pool(const sparge_shape* shape, const void* q, const void* k, float* qbar,
                float* kbar, sparge_stream_t stream);

/* Workspace bytes sparge_mask needs (pooled Q and K as bf16 high / low
 * pairs, the fp32 pooled logits). */
int sparge_mask_workspace_bytes(const sparge_shape* shape, size_t* bytes);

/*
 * sparge_mask -- block mask construction, steps 1-3 of the hot path.
 * [P4 "Maskierungsstrategien: Top-k und Top-p"], [P4 "Hybride Top-k+Top-p
 * Maskierung"], [P4 "Effiziente Kernel-Implementierung und Modellanpassung"].
 *   1. qbar_i, kbar_j = block means of Q and K (as sparge_pool).
 *   2. L_ij = scale * <qbar_i, kbar_j>;  P_i. = softmax_j(L_i.)  (fp32).
 *   3. Per row i, order blocks by P descending, ties by lower index.
 *      K   = clamp(ceil(k_frac*Mk - 1e-4), 1, Mk)           (Top-k count)
 *      m_p = smallest m with fl64(sum of the first m u_j) >= fl64(p * U),
 *            u_j = floor(P_ij * 2^40), U = sum_j u_j       (Top-p count)
 *            (p <= 0: m_p = 0; p >= 1: m_p = Mk)
 *      keep the first max(K, m_p) blocks (= Top-k set union Top-p set).
 * Arguments:
 *   q, k         : bf16 [B,H,N,d] (device).
 *   k_frac       : in (0, 1]; p in [0, 1] (p = 0 switches Top-p off).
 *   bitmask      : uint32 [B,H,Mq,ceil(Mk/32)] out; block j of row i is bit
 *                  j%32 of word j/32.  Required.
 *   row_idx      : int32 [B,H,Mq,Mk] out; the first row_cnt[i] entries of row
 *                  i are its kept kv-blocks in ascending order; the rest are
 *                  left unwritten.  Required.
 *   row_cnt      : int32 [B,H,Mq] out.  Required.
 *   col_idx/cnt  : int32 [B,H,Mk,Mq] / [B,H,Mk] out; the transposed lists
 *                  (kept q-blocks per kv-block, ascending).  Both NULL or both
 *                  set; needed by sparge_attn_bwd.
 *   pooled_prob  : fp32 [B,H,Mq,Mk] out, P (nullable).
 *   pooled_logit : fp32 [B,H,Mq,Mk] out, L (nullable).
 *   workspace    : device buffer of sparge_mask_workspace_bytes bytes (pooled
 *                  Q and K, pooled logits; no initial contents needed),
 *                  16-byte aligned.
 *   status       : nullable; records SPARGE_ERR_TIMEOUT if a bounded wait of
 *                  the pooled-logit kernel runs out.
 * The mask is a deterministic function of the fp32 P it computes.  The call
 * launches four kernels (three without the column lists) chained by
 * programmatic dependent launch: pooling (each mean written as bf16 high
 * and low parts), pooled logits on the tensor cores (three MMA passes over
 * the parts, operands loaded by TMA), softmax and selection, then the
 * column lists.
 */
int sparge_mask(const sparge_shape* shape, const void* q, const void* k, float k_frac, float p,
                float softmax_scale, uint32_t* bitmask, int32_t* row_idx, int32_t* row_cnt,
                int32_t* col_idx, int32_t* col_cnt, float* pooled_prob, float* pooled_logit,
                void* workspace, size_t ws_bytes, int32_t* status, sparge_stream_t stream);

/*
 * sparge_mask_noalloc -- sparge_mask without a workspace argument, for
 * callers that cannot allocate device memory (a runtime that owns all device
 * memory through its own pool allocator; a latency-critical loop in which an
 * allocation or free may synchronise the device).  The method pages have no
 * counterpart of this call; it is a deployment variant of sparge_mask.
 *   Same arguments, outputs and results as sparge_mask, minus workspace and
 *   ws_bytes.  The pooled Q, K and logits live in a fixed 16 MiB device array inside
 *   the library, one per GPU that loads it, kept until the process exits.
 *   Shapes whose workspace (sparge_mask_workspace_bytes) exceeds 16 MiB return
 *   SPARGE_ERR_WORKSPACE before any launch.
 *   Every argument is checked before any CUDA call.  The first call in a
 *   CUDA context (the current one: normally the primary context of the
 *   current device) looks up the array's device address in that context and
 *   caches it by the context's unique id, so a device reset or another
 *   context gets a fresh lookup; make that first call before any stream
 *   capture.  It allocates nothing: no cudaMalloc, cudaFree or allocating
 *   library routine.
 *   Every call on a device shares the one array, which keeps the last call's
 *   contents (each call overwrites what it reads, so nothing needs clearing).
 *   Calls that overlap on the GPU (different streams, or host threads on the
 *   same device without ordering) race on the array: serialise them.
 */
int sparge_mask_noalloc(const sparge_shape* shape, const void* q, const void* k, float k_frac,
                        float p, float softmax_scale, uint32_t* bitmask, int32_t* row_idx,
                        int32_t* row_cnt, int32_t* col_idx, int32_t* col_cnt,
                        float* pooled_prob, float* pooled_logit, int32_t* status,
                        sparge_stream_t stream);

/*
 * sparge_mask_from_prob -- step 3 alone: the hybrid selection of sparge_mask
 * applied to a caller-supplied pooled probability map.
 *   prob : fp32 [B,H,Mq,Mk] (device), each entry in [0, 1].
 * Other arguments and outputs as in sparge_mask.  Given the same P, the mask
 * equals the one sparge_mask emits.
 */
int sparge_mask_from_prob(const sparge_shape* shape, const float* prob, float k_frac, float p,
                          uint32_t* bitmask, int32_t* row_idx, int32_t* row_cnt,
                          int32_t* col_idx, int32_t* col_cnt, sparge_stream_t stream);

/*
 * sparge_attn_fwd -- block-sparse attention forward, step 4.
 * [P4 "Grundlagen der duennbesetzten Aufmerksamkeit und ihre
 * Herausforderungen"], [P4 "Block-duennbesetzte Aufmerksamkeit"], [P4
 * "Effiziente Kernel-Implementierung und Modellanpassung"]: only the kept
 * (q-block, kv-block) tiles are computed; the softmax of each query token is
 * normalised over the tokens of its kept kv-blocks.  No causal mask.
 *   O_t   = sum_u softmax_u(scale * Q_t.K_u) V_u  over kept tokens u
 *   LSE_t = log sum_u exp(scale * Q_t.K_u)
 * Arguments:
 *   q, k, v          : bf16 [B,H,N,d] (device).
 *   row_idx, row_cnt : the CSR lists of sparge_mask (device); every index in
 *                      [0, Mk), counts in [0, Mk].
 *   o                : bf16 [B,H,N,d] out.  lse: fp32 [B,H,N] out (nullable).
 *   status           : nullable; records SPARGE_ERR_TIMEOUT if a bounded wait
 *                      runs out, SPARGE_ERR_CUDA if a CTA finds its
 *                      shared-memory window misaligned.
 * A q-block with row_cnt 0 gets O = 0 and LSE = -inf.
 */
int sparge_attn_fwd(const sparge_shape* shape, const void* q, const void* k, const void* v,
                    const int32_t* row_idx, const int32_t* row_cnt, float softmax_scale,
                    void* o, float* lse, int32_t* status, sparge_stream_t stream);

/* Workspace bytes sparge_attn_bwd needs: fp32 D = rowsum(dO*O) per token, the
 * work orders of the q-blocks and of the dK/dV work items (int32; items with
 * more than twice the mean work first, then the rest in descending index
 * order), the work counters of the persistent gradient kernels, and room for
 * cutting key tiles with far more than one SM's share of the work into at most
 * 128 parts in all: their int32 completion counters and fp32 partial dK, dV
 * (128 x 128 x 2 x d floats; 16 MiB at d = 128).  Every byte that is read is
 * first written by the call itself (the counters are zeroed by its first
 * kernel), so the buffer needs no initial contents and may be reused by the
 * next call on the same stream. */
int sparge_attn_bwd_workspace_bytes(const sparge_shape* shape, size_t* bytes);

/*
 * sparge_attn_bwd -- gradients of sparge_attn_fwd, step 5.
 * [P2 "Abstract"] (trainable sparse attention), [P4 "Effiziente
 * Kernel-Implementierung und Modellanpassung"] (forward and backward skip
 * masked tiles).  The mask is a constant; for the kept tiles:
 *   P = exp(scale*Q K^T - LSE), D = rowsum(dO * O), dS = P * (dO V^T - D),
 *   dV = P^T dO, dQ = scale * dS K, dK = scale * dS^T Q.
 * Arguments:
 *   q, k, v, o, dout : bf16 [B,H,N,d] (device); o and lse from sparge_attn_fwd.
 *   lse              : fp32 [B,H,N] (device).
 *   row_idx/cnt, col_idx/cnt : CSR and CSC lists from sparge_mask (device).
 *   dq, dk, dv       : bf16 [B,H,N,d] out.  Tokens of kv-blocks no q-block
 *                      keeps get dK = dV = 0.
 *   workspace        : device buffer of sparge_attn_bwd_workspace_bytes bytes,
 *                      16-byte aligned; two calls must not share one buffer
 *                      concurrently (it holds their work counters).
 *   status           : nullable; records SPARGE_ERR_TIMEOUT if a bounded wait
 *                      of a gradient kernel runs out, SPARGE_ERR_CUDA if the
 *                      dK/dV kernel finds its shared-memory window misaligned.
 * The call launches four kernels: the work orders (two CTAs); D, beside them
 * by programmatic dependent launch; dK/dV (one CTA per
 * SM taking 128-key tiles from a work counter; a tile with several times an
 * SM's share of the work, such as an attention-sink block that every q-block
 * keeps when there are few heads, is cut into parts by q-block range whose
 * fp32 partial dK, dV the last part to finish adds in part order); dQ (one CTA
 * per SM taking q-blocks from a second counter, started early by programmatic
 * dependent launch; it does not read dK or dV).  Deterministic: no atomics
 * touch the gradients, each gradient element is accumulated in a fixed order
 * (the counters only decide which CTA does which part), so repeated calls give
 * bitwise identical dQ, dK, dV.
 */
int sparge_attn_bwd(const sparge_shape* shape, const void* q, const void* k, const void* v,
                    const void* o, const float* lse, const void* dout, const int32_t* row_idx,
                    const int32_t* row_cnt, const int32_t* col_idx, const int32_t* col_cnt,
                    float softmax_scale, void* dq, void* dk, void* dv, void* workspace,
                    size_t ws_bytes, int32_t* status, sparge_stream_t stream);

/* Enqueues on `stream` a copy of the device status word into *host_status
 * (caller-owned, page-locked host memory for the copy to be asynchronous) and
 * returns without waiting; the value is valid once the stream has reached the
 * copy (e.g. after an event the caller records behind it completes). */
int sparge_status_copy_async(const int32_t* status, int32_t* host_status, sparge_stream_t stream);

/* Blocking convenience: copies the device status word to *host_status and
 * synchronises `stream` before returning (the library's one blocking call). */
int sparge_read_status(const int32_t* status, sparge_stream_t stream, int32_t* host_status);

/*
 * sparge_debug_wait_probe -- launches one CTA that waits on a barrier nothing
 * ever arrives at, with the given limit (clamped to 1 ms .. 5 s).  It must
 * record SPARGE_ERR_TIMEOUT in `status` and return: a test of the bounded-wait
 * path that never hangs the GPU.
 */
int sparge_debug_wait_probe(int32_t* status, uint64_t timeout_ns, sparge_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPARGE_H_ */
