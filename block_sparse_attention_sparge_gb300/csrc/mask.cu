// Block-mask construction for SpargeAttention2 on sm_103a.
//
// Method: mindverse page "Optimierung der Effizienz von Video-Diffusionsmodellen
// durch SpargeAttention2", sections "Maskierungsstrategien: Top-k und Top-p"
// (block-pooled map; Top-k keeps the k% largest positions of a row; Top-p
// keeps the smallest set whose cumulative probability reaches p) and "Hybride
// Top-k+Top-p Maskierung" (the two rules combined), and section "Effiziente
// Kernel-Implementierung und Modellanpassung" (mask construction in CUDA).
//
// Kernels:
//   pool_kernel          HBM-bound block means of Q and K (16-byte loads).
//   score_select_kernel  pooled logits (fp32 FMA), row softmax, hybrid
//                        selection; emits the bitmask and the CSR lists.
//   select_from_prob_kernel  the selection alone on a given probability map.
//   csc_kernel           transposes the bitmask into per-kv-block q lists.
//
// Selection arithmetic (exact, order-free):
//   u_j = floor(P_j * 2^40) from the fp32 bits of P_j, U = sum u_j (uint64),
//   T = fl64(p * U), Ti = ceil(T); m_p = smallest m with (sum of the m largest
//   u in (P desc, index asc) order) >= Ti.  Since partial sums are integers
//   below 2^53, "fl64(S) >= T" and "S >= ceil(T)" are the same test.
//   The m_p-th element and the max(K, m_p)-th element are found by a 4-pass
//   radix select over the 32-bit keys (fp32 bit patterns of P, which order
//   like the values because P >= 0), with per-warp shared-memory histograms
//   of counts and u-sums; ties at the threshold key go to the lowest indices.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "common.cuh"
#include "kernels.h"

namespace sparge {

namespace {

constexpr int kPoolThreads = 256;
constexpr int kSelThreads = 512;               // 16 warps, one row each
constexpr int kSelMaxRows = kSelThreads / 32;  // rows per CTA upper bound
constexpr int kSelLogitFloats = 20480;         // 80 KB of logits per CTA
constexpr unsigned kFull = 0xffffffffu;

// ---------------------------------------------------------------- pooling
// One CTA per (head, block) unit.  Units [0, BH*Mq) are Q blocks, the rest K
// blocks.  Thread t reads 16-byte chunk (t % CH) of rows t / CH, + RG, ...
template <int D>
__global__ void __launch_bounds__(kPoolThreads) pool_kernel(
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k, int BH, int N,
    int bq, int bk, int Mq, int Mk, int do_q, int do_k, float* __restrict__ qbar,
    float* __restrict__ kbar, float* __restrict__ kbarT) {
  constexpr int CH = D / 8;              // 16-byte chunks per row
  constexpr int RG = kPoolThreads / CH;  // rows read concurrently
  __shared__ float red[RG][D];

  const long long unit = blockIdx.x;
  const long long nq = do_q ? (long long)BH * Mq : 0;
  const bool is_q = unit < nq;
  const long long u = is_q ? unit : unit - nq;
  const int M = is_q ? Mq : Mk;
  const int blk = is_q ? bq : bk;
  const int bh = static_cast<int>(u / M);
  const int i = static_cast<int>(u % M);
  const int r0 = i * blk;
  const int rows = min(blk, N - r0);
  const __nv_bfloat16* src = (is_q ? q : k) + ((long long)bh * N + r0) * D;

  const int c = threadIdx.x % CH;
  const int rg = threadIdx.x / CH;
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  // Up to 128 rows / RG rows per thread; the loads are independent, so the
  // unrolled loop keeps all of them in flight.
#pragma unroll 8
  for (int r = rg; r < rows; r += RG) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(src + (long long)r * D) + c);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(h[e]);
      acc[2 * e] += f.x;
      acc[2 * e + 1] += f.y;
    }
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) red[rg][c * 8 + e] = acc[e];
  __syncthreads();
  if (threadIdx.x < D) {
    float s = 0.f;
#pragma unroll
    for (int g = 0; g < RG; ++g) s += red[g][threadIdx.x];
    const float mean = s / static_cast<float>(rows);
    if (is_q) {
      qbar[((long long)bh * Mq + i) * D + threadIdx.x] = mean;
    } else {
      if (kbar) kbar[((long long)bh * Mk + i) * D + threadIdx.x] = mean;
      if (kbarT) kbarT[((long long)bh * D + threadIdx.x) * Mk + i] = mean;
    }
  }
}

// ---------------------------------------------------------------- selection
__device__ __forceinline__ unsigned long long fixed40(uint32_t bits) {
  // floor(x * 2^40) for a non-negative fp32 x given by its bits (exact).
  const uint32_t e = (bits >> 23) & 0xffu;
  if (e == 0u) return 0ull;  // zero or subnormal: below 2^-126, floor is 0
  const unsigned long long m = (bits & 0x7fffffu) | 0x800000u;
  int sh = static_cast<int>(e) - 150 + 40;  // x * 2^40 = m * 2^sh
  if (sh >= 0) return m << min(sh, 23);     // sh <= 17 for x <= 1
  if (sh <= -24) return 0ull;
  return m >> (-sh);
}

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

template <typename T>
__device__ __forceinline__ T warp_excl_scan(T v) {
  const int lane = threadIdx.x & 31;
  T incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T n = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += n;
  }
  return incl - v;
}

// Radix select over the keys of one row held in shared memory.  With
// use_sum, finds the key tau of the element at which the running u-sum in
// (key desc, index asc) order first reaches `target`; otherwise the key of
// the element at 1-based position `target` by count.  Returns tau and, via
// above_sum / above_cnt, the u-sum and count of all keys strictly above tau.
__device__ uint32_t radix_select(const uint32_t* keys, int Mk, bool use_sum,
                                 unsigned long long target, uint32_t* hcnt,
                                 unsigned long long* hsum, unsigned long long* above_sum,
                                 uint32_t* above_cnt) {
  const int lane = threadIdx.x & 31;
  uint32_t prefix = 0, pmask = 0;
  unsigned long long A = 0;
  uint32_t C = 0;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int b = lane; b < 256; b += 32) {
      hcnt[b] = 0u;
      hsum[b] = 0ull;
    }
    __syncwarp();
    for (int j = lane; j < Mk; j += 32) {
      const uint32_t key = keys[j];
      if ((key & pmask) == prefix) {
        const int dg = (key >> shift) & 0xff;
        atomicAdd(&hcnt[dg], 1u);
        if (use_sum) atomicAdd(&hsum[dg], fixed40(key));
      }
    }
    __syncwarp();
    // Lane L owns digits 255-8L down to 248-8L (descending).
    unsigned long long ls = 0;
    uint32_t lc = 0;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const int b = 255 - 8 * lane - t;
      ls += hsum[b];
      lc += hcnt[b];
    }
    const unsigned long long ex_s = warp_excl_scan<unsigned long long>(ls);
    const uint32_t ex_c = warp_excl_scan<uint32_t>(lc);
    const bool hit = use_sum ? (A + ex_s + ls >= target) : ((unsigned long long)(C + ex_c + lc) >= target);
    const uint32_t hm = __ballot_sync(kFull, hit);
    const int L = hm ? (__ffs(hm) - 1) : 31;  // hm == 0 only for invalid input
    int digit = 0;
    unsigned long long a_new = 0;
    uint32_t c_new = 0;
    if (lane == L) {
      unsigned long long run = A + ex_s;
      uint32_t rc = C + ex_c;
      digit = 248 - 8 * lane;
      for (int t = 0; t < 8; ++t) {
        const int b = 255 - 8 * lane - t;
        const bool reach = use_sum ? (run + hsum[b] >= target)
                                   : ((unsigned long long)(rc + hcnt[b]) >= target);
        if (reach) {
          digit = b;
          break;
        }
        run += hsum[b];
        rc += hcnt[b];
      }
      a_new = run;
      c_new = rc;
    }
    digit = __shfl_sync(kFull, digit, L);
    A = __shfl_sync(kFull, a_new, L);
    C = __shfl_sync(kFull, c_new, L);
    prefix |= static_cast<uint32_t>(digit) << shift;
    pmask |= 0xffu << shift;
    __syncwarp();
  }
  *above_sum = A;
  *above_cnt = C;
  return prefix;
}

// Hybrid Top-k + Top-p selection of one row (one warp).  `prow` holds the
// row's fp32 probabilities in shared memory.
__device__ void select_row(const float* prow, int Mk, int ktop, float p, uint32_t* hcnt,
                           unsigned long long* hsum, uint32_t* __restrict__ bm_row,
                           int32_t* __restrict__ idx_row, int32_t* __restrict__ cnt_out) {
  const int lane = threadIdx.x & 31;
  const uint32_t* keys = reinterpret_cast<const uint32_t*>(prow);
  int m_p;
  if (p >= 1.f) {
    m_p = Mk;
  } else if (!(p > 0.f)) {
    m_p = 0;
  } else {
    unsigned long long U = 0;
    for (int j = lane; j < Mk; j += 32) U += fixed40(keys[j]);
    U = warp_sum_u64(U);
    const double T = __dmul_rn(static_cast<double>(p), static_cast<double>(U));
    const unsigned long long Ti = static_cast<unsigned long long>(ceil(T));
    if (Ti == 0ull) {
      m_p = 0;
    } else {
      unsigned long long A;
      uint32_t C;
      const uint32_t tau = radix_select(keys, Mk, true, Ti, hcnt, hsum, &A, &C);
      const unsigned long long ut = fixed40(tau);
      const unsigned long long need = (ut > 0ull && Ti > A) ? (Ti - A + ut - 1ull) / ut : 1ull;
      m_p = static_cast<int>(min(static_cast<unsigned long long>(Mk), C + need));
    }
  }
  const int c = min(Mk, max(ktop, m_p));
  unsigned long long A2;
  uint32_t c_gt;
  const uint32_t tau_c = radix_select(keys, Mk, false, static_cast<unsigned long long>(c), hcnt,
                                      hsum, &A2, &c_gt);
  const int need_ties = c - static_cast<int>(c_gt);
  const uint32_t lt = (1u << lane) - 1u;
  int ties = 0, kept = 0;
  for (int w0 = 0; w0 < Mk; w0 += 32) {
    const int j = w0 + lane;
    const bool valid = j < Mk;
    const uint32_t key = valid ? keys[j] : 0u;
    const bool gt = valid && key > tau_c;
    const bool eq = valid && key == tau_c;
    const uint32_t em = __ballot_sync(kFull, eq);
    const int rank = ties + __popc(em & lt);
    const bool keep = gt || (eq && rank < need_ties);
    ties += __popc(em);
    const uint32_t km = __ballot_sync(kFull, keep);
    if (lane == 0) bm_row[w0 >> 5] = km;
    if (keep) idx_row[kept + __popc(km & lt)] = j;
    kept += __popc(km);
  }
  if (lane == 0) *cnt_out = kept;
}

struct SelSmem {
  uint32_t hcnt[kSelMaxRows][256];
  unsigned long long hsum[kSelMaxRows][256];
};

// Pooled logits + softmax + selection.  CTA = R consecutive q-block rows of
// one head; grid.x = BH * ceil(Mq / R).
template <int D>
__global__ void __launch_bounds__(kSelThreads) score_select_kernel(
    const float* __restrict__ qbar, const float* __restrict__ kbarT, int Mq, int Mk, int Mkw,
    int R, float scale, int ktop, float p, uint32_t* __restrict__ bitmask,
    int32_t* __restrict__ row_idx, int32_t* __restrict__ row_cnt, float* __restrict__ logit_out,
    float* __restrict__ prob_out) {
  extern __shared__ __align__(16) uint8_t smem[];
  SelSmem* hs = reinterpret_cast<SelSmem*>(smem);
  float* qs = reinterpret_cast<float*>(smem + sizeof(SelSmem));  // [R][D]
  float* ls = qs + kSelMaxRows * D;                                // [R][Mk]

  const int nrb = (Mq + R - 1) / R;
  const int bh = blockIdx.x / nrb;
  const int i0 = (blockIdx.x % nrb) * R;
  const int nrows = min(R, Mq - i0);
  const float* qsrc = qbar + ((long long)bh * Mq + i0) * D;
  for (int t = threadIdx.x; t < kSelMaxRows * D; t += kSelThreads)
    qs[t] = (t < nrows * D) ? qsrc[t] : 0.f;
  __syncthreads();

  // Logits: thread owns columns j, accumulates all R rows over d.
  const float* kt = kbarT + (long long)bh * D * Mk;
  for (int j = threadIdx.x; j < Mk; j += kSelThreads) {
    float acc[kSelMaxRows];
#pragma unroll
    for (int r = 0; r < kSelMaxRows; ++r) acc[r] = 0.f;
#pragma unroll 2
    for (int c = 0; c < D; c += 4) {
      const float k0 = __ldg(kt + (long long)(c + 0) * Mk + j);
      const float k1 = __ldg(kt + (long long)(c + 1) * Mk + j);
      const float k2 = __ldg(kt + (long long)(c + 2) * Mk + j);
      const float k3 = __ldg(kt + (long long)(c + 3) * Mk + j);
#pragma unroll
      for (int r = 0; r < kSelMaxRows; ++r) {
        const float4 qv = *reinterpret_cast<const float4*>(qs + r * D + c);
        acc[r] = fmaf(qv.x, k0, acc[r]);
        acc[r] = fmaf(qv.y, k1, acc[r]);
        acc[r] = fmaf(qv.z, k2, acc[r]);
        acc[r] = fmaf(qv.w, k3, acc[r]);
      }
    }
#pragma unroll
    for (int r = 0; r < kSelMaxRows; ++r)
      if (r < nrows) ls[r * Mk + j] = acc[r] * scale;
  }
  __syncthreads();

  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (w < nrows) {
    float* row = ls + w * Mk;
    const long long grow = (long long)bh * Mq + i0 + w;
    float m = -INFINITY;
    for (int j = lane; j < Mk; j += 32) m = fmaxf(m, row[j]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
    float s = 0.f;
    for (int j = lane; j < Mk; j += 32) {
      const float lg = row[j];
      if (logit_out) logit_out[grow * Mk + j] = lg;
      const float e = expf(lg - m);
      row[j] = e;
      s += e;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(kFull, s, o);
    for (int j = lane; j < Mk; j += 32) {
      const float pj = __fdiv_rn(row[j], s);
      row[j] = pj;
      if (prob_out) prob_out[grow * Mk + j] = pj;
    }
    __syncwarp();
    select_row(row, Mk, ktop, p, hs->hcnt[w], hs->hsum[w], bitmask + grow * Mkw,
               row_idx + grow * Mk, row_cnt + grow);
  }
}

__global__ void __launch_bounds__(kSelThreads) select_from_prob_kernel(
    const float* __restrict__ prob, int Mq, int Mk, int Mkw, int R, int ktop, float p,
    uint32_t* __restrict__ bitmask, int32_t* __restrict__ row_idx, int32_t* __restrict__ row_cnt) {
  extern __shared__ __align__(16) uint8_t smem[];
  SelSmem* hs = reinterpret_cast<SelSmem*>(smem);
  float* ls = reinterpret_cast<float*>(smem + sizeof(SelSmem));
  const int nrb = (Mq + R - 1) / R;
  const int bh = blockIdx.x / nrb;
  const int i0 = (blockIdx.x % nrb) * R;
  const int nrows = min(R, Mq - i0);
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (w < nrows) {
    const long long grow = (long long)bh * Mq + i0 + w;
    float* row = ls + w * Mk;
    for (int j = lane; j < Mk; j += 32) row[j] = __ldg(prob + grow * Mk + j);
    __syncwarp();
    select_row(row, Mk, ktop, p, hs->hcnt[w], hs->hsum[w], bitmask + grow * Mkw,
               row_idx + grow * Mk, row_cnt + grow);
  }
}

// ---------------------------------------------------------------- transpose
// CTA = (head, bitmask word w): stages the Mq words of column group w in
// shared memory, then lane l lists the q-blocks that keep kv-block 32w + l.
constexpr int kCscThreads = 128;
__global__ void __launch_bounds__(kCscThreads) csc_kernel(const uint32_t* __restrict__ bitmask,
                                                          int Mq, int Mk, int Mkw,
                                                          int32_t* __restrict__ col_idx,
                                                          int32_t* __restrict__ col_cnt) {
  extern __shared__ uint32_t words[];  // [Mq]
  const int bh = blockIdx.x / Mkw;
  const int w = blockIdx.x % Mkw;
  const uint32_t* src = bitmask + (long long)bh * Mq * Mkw + w;
  for (int i = threadIdx.x; i < Mq; i += kCscThreads) words[i] = __ldg(src + (long long)i * Mkw);
  __syncthreads();
  if (threadIdx.x < 32) {
    const int j = w * 32 + threadIdx.x;
    if (j < Mk) {
      int32_t* out = col_idx + ((long long)bh * Mk + j) * Mq;
      int cnt = 0;
      for (int i = 0; i < Mq; ++i)
        if ((words[i] >> threadIdx.x) & 1u) out[cnt++] = i;
      col_cnt[(long long)bh * Mk + j] = cnt;
    }
  }
}

size_t select_smem_bytes(int d, int R, int Mk) {
  return sizeof(SelSmem) + (size_t)kSelMaxRows * d * sizeof(float) +
         (size_t)R * Mk * sizeof(float);
}

}  // namespace

int select_rows_per_cta(int Mk) {
  int r = kSelLogitFloats / Mk;
  return r < 1 ? 1 : (r > kSelMaxRows ? kSelMaxRows : r);
}

cudaError_t launch_pool(const Geom& g, const void* q, const void* k, float* qbar, float* kbar,
                        float* kbarT, cudaStream_t st) {
  const int do_q = qbar != nullptr;
  const int do_k = (kbar != nullptr) || (kbarT != nullptr);
  const long long units = (do_q ? (long long)g.BH * g.Mq : 0) + (do_k ? (long long)g.BH * g.Mk : 0);
  if (units == 0) return cudaSuccess;
  const auto* qq = static_cast<const __nv_bfloat16*>(q);
  const auto* kk = static_cast<const __nv_bfloat16*>(k);
  if (g.d == 128)
    pool_kernel<128><<<static_cast<unsigned>(units), kPoolThreads, 0, st>>>(
        qq, kk, g.BH, g.N, g.bq, g.bk, g.Mq, g.Mk, do_q, do_k, qbar, kbar, kbarT);
  else
    pool_kernel<64><<<static_cast<unsigned>(units), kPoolThreads, 0, st>>>(
        qq, kk, g.BH, g.N, g.bq, g.bk, g.Mq, g.Mk, do_q, do_k, qbar, kbar, kbarT);
  return cudaGetLastError();
}

cudaError_t launch_score_select(const Geom& g, const float* qbar, const float* kbarT, float scale,
                                int ktop, float p, uint32_t* bitmask, int32_t* row_idx,
                                int32_t* row_cnt, float* logit_out, float* prob_out,
                                cudaStream_t st) {
  const int R = select_rows_per_cta(g.Mk);
  const int nrb = (g.Mq + R - 1) / R;
  const size_t smem = select_smem_bytes(g.d, R, g.Mk);
  const unsigned grid = static_cast<unsigned>((long long)g.BH * nrb);
  cudaError_t e;
  if (g.d == 128) {
    e = cudaFuncSetAttribute(score_select_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    score_select_kernel<128><<<grid, kSelThreads, smem, st>>>(qbar, kbarT, g.Mq, g.Mk, g.Mkw, R,
                                                               scale, ktop, p, bitmask, row_idx,
                                                               row_cnt, logit_out, prob_out);
  } else {
    e = cudaFuncSetAttribute(score_select_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    score_select_kernel<64><<<grid, kSelThreads, smem, st>>>(qbar, kbarT, g.Mq, g.Mk, g.Mkw, R,
                                                              scale, ktop, p, bitmask, row_idx,
                                                              row_cnt, logit_out, prob_out);
  }
  return cudaGetLastError();
}

cudaError_t launch_select_from_prob(const Geom& g, const float* prob, int ktop, float p,
                                    uint32_t* bitmask, int32_t* row_idx, int32_t* row_cnt,
                                    cudaStream_t st) {
  const int R = select_rows_per_cta(g.Mk);
  const int nrb = (g.Mq + R - 1) / R;
  const size_t smem = sizeof(SelSmem) + (size_t)R * g.Mk * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(select_from_prob_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  select_from_prob_kernel<<<static_cast<unsigned>((long long)g.BH * nrb), kSelThreads, smem, st>>>(
      prob, g.Mq, g.Mk, g.Mkw, R, ktop, p, bitmask, row_idx, row_cnt);
  return cudaGetLastError();
}

cudaError_t launch_csc(const Geom& g, const uint32_t* bitmask, int32_t* col_idx, int32_t* col_cnt,
                       cudaStream_t st) {
  const size_t smem = (size_t)g.Mq * sizeof(uint32_t);
  csc_kernel<<<static_cast<unsigned>((long long)g.BH * g.Mkw), kCscThreads, smem, st>>>(
      bitmask, g.Mq, g.Mk, g.Mkw, col_idx, col_cnt);
  return cudaGetLastError();
}

}  // namespace sparge
