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
//   pool_kernel, logits_kernel, select_logits_reg_kernel (rows up to 512
//                        blocks) or select_logits_kernel, csc_split_kernel
//                        the sparge_mask pipeline (see "mask pipeline"
//                        below); pool_kernel alone also serves sparge_pool.
//   select_from_prob_kernel  the selection alone on a given probability map.
//   csc_kernel           transposes the bitmask into per-kv-block q lists.
//
// Selection arithmetic (exact, order-free):
//   u_j = floor(P_j * 2^40) from the fp32 bits of P_j, U = sum u_j (uint64),
//   T = fl64(p * U), Ti = ceil(T); m_p = smallest m with (sum of the m largest
//   u in (P desc, index asc) order) >= Ti.  Since partial sums are integers
//   below 2^53, "fl64(S) >= T" and "S >= ceil(T)" are the same test.
//   The keys are the fp32 bit patterns of P, which order like the values
//   because P >= 0.  One warp selects one row: the Top-p threshold key is the
//   largest t with (sum of u over keys >= t) >= Ti, and the threshold of the
//   kept count c = max(K, m_p) the largest t with (count of keys >= t) >= c,
//   both found by bisection over the key bits with warp reductions (u sums
//   split into 21-bit halves so the 32-bit reduction is exact), starting
//   below the bits that every key of the row shares; keys equal to a
//   threshold are kept by lowest index.  Rows longer than 2048 blocks
//   use a 4-pass radix select with per-warp shared-memory histograms of
//   counts and u-sums instead.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace sparge {

namespace {

constexpr int kSelThreads = 512;               // 16 warps, one row each
constexpr int kSelMaxRows = kSelThreads / 32;  // rows per CTA upper bound
constexpr int kSelLogitFloats = 20480;         // 80 KB of logits per CTA
constexpr unsigned kFull = 0xffffffffu;

// ---------------------------------------------------------------- pooling
constexpr int kPoolThreads = 256;

// Consecutive rows (tokens) one CTA reads.  128-row units at four CTAs per SM
// (64 registers a thread) keep other CTAs' loads in flight while one reduces;
// measured at 480p: the whole mask 49.4 us against 51.1 us with 256-row
// units at two CTAs per SM.
constexpr int kPoolRows = 128;

// The rows are loaded with ldg_no_l1 (read once: no L1 allocation; measured
// at 480p: the whole mask 47.2 us against 49.6 us with __ldg).  L2 keeps the
// lines, which the forward's Q and K tile loads then partly hit.
// Issues this thread's loads of a run of 128 rows (up to `rows` valid; d = D
// bf16 values per row): 16-byte chunk t % CH of rows t / CH + RG * i
// (i < L), all issued before any is used, so a CTA keeps 32 KB (d = 128) in
// flight.
template <int D>
__device__ __forceinline__ void pool_loads(const __nv_bfloat16* __restrict__ src, int rows,
                                           uint4 (&v)[kPoolRows * D / 8 / kPoolThreads]) {
  constexpr int CH = D / 8;               // 16-byte chunks per row
  constexpr int RG = kPoolThreads / CH;   // rows read concurrently
  constexpr int L = kPoolRows / RG;       // loads per thread
  const int c = threadIdx.x % CH;
  const int rg = threadIdx.x / CH;
#pragma unroll
  for (int i = 0; i < L; ++i) {
    const int r = rg + RG * i;
    v[i] = r < rows ? ldg_no_l1(reinterpret_cast<const uint4*>(src + (long long)r * D) + c)
                    : make_uint4(0u, 0u, 0u, 0u);
  }
}

// Adds the loaded values into per-block partial sums: load i belongs to block
// i * RG / BLK of the run; the sums go to red[row group][block][feature].
template <int D, int BLK>
__device__ __forceinline__ void pool_accumulate(const uint4 (&v)[kPoolRows * D / 8 / kPoolThreads],
                                                float (*red)[kPoolRows / 64][D]) {
  constexpr int CH = D / 8;
  constexpr int RG = kPoolThreads / CH;
  constexpr int L = kPoolRows / RG;
  constexpr int G = kPoolRows / BLK;
  float acc[G][8];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[g][e] = 0.f;
#pragma unroll
  for (int i = 0; i < L; ++i) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v[i]);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(h[e]);
      acc[i * RG / BLK][2 * e] += f.x;
      acc[i * RG / BLK][2 * e + 1] += f.y;
    }
  }
  const int c = threadIdx.x % CH, rg = threadIdx.x / CH;
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < 8; ++e) red[rg][g][c * 8 + e] = acc[g][e];
}

// One CTA per unit: 128 consecutive tokens of one head, i.e. 128 / block
// size blocks.  Units [0, BH*UQ) cover the Q blocks (when do_q), the rest
// the K blocks.  The means are row-major [BH, M, d]: fp32 into qbar / kbar,
// or, when qhi is set, as the bf16 pair hi = bf16(mean), lo = bf16(mean - hi)
// into qhi / qlo and khi / klo (the operands of the pooled-logit MMAs,
// hi*hi + hi*lo + lo*hi).
template <int D>
__global__ void __launch_bounds__(kPoolThreads, 4) pool_kernel(
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k, int BH, int N,
    int bq, int bk, int Mq, int Mk, int do_q, float* __restrict__ qbar,
    float* __restrict__ kbar, __nv_bfloat16* __restrict__ qhi, __nv_bfloat16* __restrict__ qlo,
    __nv_bfloat16* __restrict__ khi, __nv_bfloat16* __restrict__ klo) {
  // Lets a kernel launched with programmatic serialization start early; it
  // waits for this grid's results itself.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  constexpr int CH = D / 8;
  constexpr int RG = kPoolThreads / CH;
  __shared__ float red[RG][kPoolRows / 64][D];
  const int UQ = (N + kPoolRows - 1) / kPoolRows;  // units per head, either tensor
  const long long unit = blockIdx.x;
  const long long nq = do_q ? (long long)BH * UQ : 0;
  const bool is_q = unit < nq;
  const long long u = is_q ? unit : unit - nq;
  const int M = is_q ? Mq : Mk;
  const int blk = is_q ? bq : bk;
  const int G = kPoolRows / blk;
  const int bh = static_cast<int>(u / UQ);
  const int r0 = static_cast<int>(u % UQ) * kPoolRows;
  const __nv_bfloat16* src = (is_q ? q : k) + ((long long)bh * N + r0) * D;
  const int rows = min(kPoolRows, N - r0);
  uint4 v[kPoolRows * D / 8 / kPoolThreads];
  pool_loads<D>(src, rows, v);
  if (blk == 128)
    pool_accumulate<D, 128>(v, red);
  else
    pool_accumulate<D, 64>(v, red);
  __syncthreads();
  for (int o = threadIdx.x; o < G * D; o += kPoolThreads) {
    const int g = o / D, f = o % D;
    const int i = r0 / blk + g;  // block index within the head
    if (i >= M) continue;
    float sum = 0.f;
#pragma unroll
    for (int x = 0; x < RG; ++x) sum += red[x][g][f];
    const float mean = sum / static_cast<float>(min(blk, N - i * blk));
    const long long oi = ((long long)bh * M + i) * D + f;
    if (qhi != nullptr) {
      const __nv_bfloat16 hh = __float2bfloat16_rn(mean);
      const __nv_bfloat16 ll = __float2bfloat16_rn(mean - __bfloat162float(hh));
      (is_q ? qhi : khi)[oi] = hh;
      (is_q ? qlo : klo)[oi] = ll;
    } else {
      (is_q ? qbar : kbar)[oi] = mean;
    }
  }
}

// One CTA per unit of 128 tokens (units = the Q and K runs to pool).
template <int D>
cudaError_t launch_pool_kernel(const Geom& g, const void* q, const void* k, int do_q, int do_k,
                               float* qbar, float* kbar, void* qhi, void* qlo, void* khi,
                               void* klo, cudaStream_t st) {
  const long long uq = (g.N + kPoolRows - 1) / kPoolRows;
  const long long units = (do_q ? (long long)g.BH * uq : 0) + (do_k ? (long long)g.BH * uq : 0);
  if (units == 0) return cudaSuccess;
  pool_kernel<D><<<static_cast<unsigned>(units), kPoolThreads, 0, st>>>(
      static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k), g.BH, g.N, g.bq,
      g.bk, g.Mq, g.Mk, do_q, qbar, kbar, static_cast<__nv_bfloat16*>(qhi),
      static_cast<__nv_bfloat16*>(qlo), static_cast<__nv_bfloat16*>(khi),
      static_cast<__nv_bfloat16*>(klo));
  return cudaGetLastError();
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

// Exact warp sum of per-lane partial sums below 2^46 (u <= 2^40, at most 64
// terms per lane): the three pieces v >> 42, bits 21..41 and bits 0..20 each
// sum over 32 lanes to less than 2^26, exact in 32-bit reductions.
__device__ __forceinline__ unsigned long long warp_sum_u42(unsigned long long v) {
  const uint32_t a = __reduce_add_sync(kFull, static_cast<uint32_t>(v >> 42));
  const uint32_t b = __reduce_add_sync(kFull, static_cast<uint32_t>((v >> 21) & 0x1fffffu));
  const uint32_t c = __reduce_add_sync(kFull, static_cast<uint32_t>(v & 0x1fffffu));
  return (static_cast<unsigned long long>(a) << 42) + (static_cast<unsigned long long>(b) << 21) + c;
}

// Hybrid Top-k + Top-p selection of one row (one warp).  Lane l holds
// elements j = 32 e + l (e < EPL): with kRegs their fp32 keys come in kr[],
// else they are read from `keys` in shared memory.  The thresholds are found
// by a bitwise binary search on the fp32 key: the largest key tau with
// sum_{key >= tau} u >= Ti (Top-p) or #{key >= tau} >= c (Top-k/union);
// absent elements carry key 0, which no candidate (>= 1) admits.  Results
// equal select_row's exactly (same integer rule, same tie order).
template <int EPL, bool kRegs>
__device__ __forceinline__ void select_keys(const uint32_t (&kr)[kRegs ? EPL : 1],
                                            const uint32_t* keys, int Mk, int ktop, float p,
                                            uint32_t* __restrict__ bm_row,
                                            int32_t* __restrict__ idx_row,
                                            int32_t* __restrict__ cnt_out) {
  const int lane = threadIdx.x & 31;
  // Elements per lane actually present (EPL is the compile-time bound).  The
  // loops below unroll fully over EPL so that register arrays stay in
  // registers; in shared-memory mode they stop at ne.
  const int ne = kRegs ? EPL : (Mk + 31) / 32;
  // Element e of this lane (absent elements read as key 0).
  auto key_of = [&](int e) -> uint32_t {
    if (kRegs) return kr[kRegs ? e : 0];
    const int j = e * 32 + lane;
    return j < Mk ? keys[j] : 0u;
  };
  // Bits above `hb` are the same in every present key (`base` holds them):
  // a search candidate that differs from base there admits all keys or none,
  // so both searches below start at bit hb from base (hb = -1: all keys
  // equal, base is the key).
  uint32_t kor = 0u, kand = ~0u;
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    if (!kRegs && e >= ne) break;
    const uint32_t k = key_of(e);
    kor |= k;
    kand &= (e * 32 + lane < Mk) ? k : ~0u;
  }
  kor = __reduce_or_sync(kFull, kor);
  kand = __reduce_and_sync(kFull, kand);
  const uint32_t diff = kor ^ kand;
  const int hb = diff ? 31 - __clz(static_cast<int>(diff)) : -1;
  const uint32_t base = hb >= 0 ? (kand & ~((2u << hb) - 1u)) : kand;
  int m_p;
  if (p >= 1.f) {
    m_p = Mk;
  } else if (!(p > 0.f)) {
    m_p = 0;
  } else {
    // u = floor(P * 2^40) of each element, computed once when the keys are
    // in registers.
    unsigned long long ur[kRegs ? EPL : 1];
    if (kRegs) {
#pragma unroll
      for (int e = 0; e < EPL; ++e) ur[kRegs ? e : 0] = fixed40(key_of(e));
    }
    auto u_of = [&](int e, uint32_t k) -> unsigned long long {
      return kRegs ? ur[kRegs ? e : 0] : fixed40(k);
    };
    unsigned long long part = 0;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      if (!kRegs && e >= ne) break;
      part += u_of(e, key_of(e));
    }
    const unsigned long long U = warp_sum_u42(part);
    const double T = __dmul_rn(static_cast<double>(p), static_cast<double>(U));
    const unsigned long long Ti = static_cast<unsigned long long>(ceil(T));
    if (Ti == 0ull) {
      m_p = 0;
    } else {
      // sum_{key >= base} u = U >= Ti, so base qualifies.
      uint32_t tau = base;
      for (int bit = hb; bit >= 0; --bit) {
        const uint32_t cand = tau | (1u << bit);
        unsigned long long s = 0;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
          if (!kRegs && e >= ne) break;
          const uint32_t k = key_of(e);
          s += k >= cand ? u_of(e, k) : 0ull;
        }
        if (warp_sum_u42(s) >= Ti) tau = cand;
      }
      unsigned long long a = 0;
      uint32_t cgt = 0;
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        if (!kRegs && e >= ne) break;
        const uint32_t k = key_of(e);
        const bool gt = k > tau;
        a += gt ? u_of(e, k) : 0ull;
        cgt += gt ? 1u : 0u;
      }
      const unsigned long long A = warp_sum_u42(a);
      const uint32_t C = __reduce_add_sync(kFull, cgt);
      const unsigned long long ut = fixed40(tau);
      const unsigned long long need = (ut > 0ull && Ti > A) ? (Ti - A + ut - 1ull) / ut : 1ull;
      m_p = static_cast<int>(min(static_cast<unsigned long long>(Mk), C + need));
    }
  }
  const int c = min(Mk, max(ktop, m_p));
  // tau_c: a key with exactly c keys >= it if one exists (the search stops
  // there), else the c-th largest key; either way the kept set below is the
  // c keys >= tau_c, ties at tau_c taken by lower index.  All Mk keys are
  // >= base, so base qualifies for c >= 1 (c = 0 keeps nothing: tau_c stays
  // above every key).
  uint32_t tau_c = c > 0 ? base : 0x7fffffffu;
  bool exact = (c == Mk);  // exactly c keys >= tau_c
  for (int bit = hb; c > 0 && !exact && bit >= 0; --bit) {
    const uint32_t cand = tau_c | (1u << bit);
    uint32_t n = 0;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      if (!kRegs && e >= ne) break;
      n += key_of(e) >= cand ? 1u : 0u;
    }
    const int tot = static_cast<int>(__reduce_add_sync(kFull, n));
    if (tot >= c) {
      tau_c = cand;
      exact = (tot == c);
    }
  }
  // Keys equal to tau_c are real elements or, when tau_c is 0, zero
  // probabilities; absent elements are excluded below by j < Mk.  When
  // exactly c keys are >= tau_c, every tie is kept.
  int need_ties = 0;
  if (!exact) {
    uint32_t ngt = 0;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      if (!kRegs && e >= ne) break;
      ngt += key_of(e) > tau_c ? 1u : 0u;
    }
    need_ties = c - static_cast<int>(__reduce_add_sync(kFull, ngt));
  }
  const uint32_t lt = (1u << lane) - 1u;
  int ties = 0, kept = 0;
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    if (!kRegs && e >= ne) break;
    const int j = e * 32 + lane;
    const bool valid = j < Mk;
    const uint32_t k = key_of(e);
    bool keep;
    if (exact) {
      keep = valid && k >= tau_c;
    } else {
      const bool gt = valid && k > tau_c;
      const bool eq = valid && k == tau_c;
      const uint32_t em = __ballot_sync(kFull, eq);
      const int rank = ties + __popc(em & lt);
      keep = gt || (eq && rank < need_ties);
      ties += __popc(em);
    }
    const uint32_t km = __ballot_sync(kFull, keep);
    if (e * 32 < Mk) {
      if (lane == 0) bm_row[e] = km;
      if (keep) idx_row[kept + __popc(km & lt)] = j;
    }
    kept += __popc(km);
  }
  if (lane == 0) *cnt_out = kept;
}

// select_keys on a row of probabilities in shared memory: copied into
// registers first (kRegs) or read in place.
template <int EPL, bool kRegs>
__device__ void select_row_reg(const float* prow, int Mk, int ktop, float p,
                               uint32_t* __restrict__ bm_row, int32_t* __restrict__ idx_row,
                               int32_t* __restrict__ cnt_out) {
  const int lane = threadIdx.x & 31;
  const uint32_t* keys = reinterpret_cast<const uint32_t*>(prow);
  uint32_t kr[kRegs ? EPL : 1];
  if (kRegs) {
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      const int j = e * 32 + lane;
      kr[kRegs ? e : 0] = j < Mk ? keys[j] : 0u;
    }
  } else {
    kr[0] = 0u;
  }
  select_keys<EPL, kRegs>(kr, keys, Mk, ktop, p, bm_row, idx_row, cnt_out);
}

// Binary search with keys in registers for rows up to 512 blocks, reading
// them from shared memory up to 2048 blocks, else the radix select.
__device__ __forceinline__ void select_row_any(const float* prow, int Mk, int ktop, float p,
                                               uint32_t* hcnt, unsigned long long* hsum,
                                               uint32_t* bm_row, int32_t* idx_row,
                                               int32_t* cnt_out) {
  if (Mk <= 32 * 16)
    select_row_reg<16, true>(prow, Mk, ktop, p, bm_row, idx_row, cnt_out);
  else if (Mk <= 32 * 64)
    select_row_reg<64, false>(prow, Mk, ktop, p, bm_row, idx_row, cnt_out);
  else
    select_row(prow, Mk, ktop, p, hcnt, hsum, bm_row, idx_row, cnt_out);
}

struct SelSmem {
  uint32_t hcnt[kSelMaxRows][256];
  unsigned long long hsum[kSelMaxRows][256];
};

__global__ void __launch_bounds__(kSelThreads, 1) select_from_prob_kernel(
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
    select_row_any(row, Mk, ktop, p, hs->hcnt[w], hs->hsum[w], bitmask + grow * Mkw,
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

// ---------------------------------------------------------------- mask pipeline
// sparge_mask runs four kernels chained by programmatic dependent launch:
//   pool_kernel          Q- and K-block means (HBM-bound, 16-byte loads),
//                        row-major [BH, M, d] as bf16 hi / lo pairs.
//   logits_kernel        L = scale * Qbar Kbar^T per head on the tensor cores,
//                        one CTA per 128 x 128 tile (below).
//   select_logits_reg_kernel  one warp per q-block row, the row's logits in
//                        registers (Mk <= 512): row softmax and hybrid
//                        selection; select_logits_kernel stages longer rows
//                        in shared memory.
//   csc_split_kernel     (when the column lists are wanted) per CTA one head
//                        and 32 kv-blocks: the ascending lists of q-blocks.
// A dependent kernel only launches once every CTA of the previous one has
// started and waits for its results itself, so its waiting CTAs never keep
// the previous kernel from running.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_primary() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Pooled logits on tcgen05: each fp32 mean x is held as bf16 hi = bf16(x)
// and lo = bf16(x - hi) (written so by the pooling kernel); per k-step three
// MMAs accumulate hi.hi + hi.lo + lo.hi in fp32 (the dropped lo.lo term and
// the rounding of lo are about 2^-16 of each product), so the logits agree
// with fp32 arithmetic far inside the map tolerance.  Thread 0 loads the four
// tiles by TMA (128-byte swizzled, K-major, the layout the MMA descriptors
// expect) and issues the MMAs, and warp w reads lanes 32 (w % 4) .. +31,
// columns 32 (w / 4) .. +31 of the accumulator back.
constexpr int kLgThreads = 512;
constexpr int kLgTile = 128;

template <int D>
struct LgCfg {
  static constexpr int KCH = D / 64;                  // 128-byte column chunks per row
  static constexpr uint32_t kTile = kLgTile * D * 2;  // one bf16 [128 x D] tile
  static constexpr uint32_t off_ahi = 0;
  static constexpr uint32_t off_alo = kTile;
  static constexpr uint32_t off_bhi = 2 * kTile;
  static constexpr uint32_t off_blo = 3 * kTile;
  static constexpr uint32_t off_bar = 4 * kTile;      // [0] operands landed, [1] MMAs done
  static constexpr uint32_t off_slot = off_bar + 16;
  static constexpr uint32_t smem_alloc = off_slot + 16 + 1024;
};

// Pooled logits of one 128 x 128 tile (q-blocks mt*128.., k-blocks nt*128..)
// of head bh: scale * (Qhi Khi^T + Qhi Klo^T + Qlo Khi^T) on the tensor
// cores, the split-bf16 means loaded by TMA (rows past Mq / Mk read as zero).
template <int D>
__global__ void __launch_bounds__(kLgThreads, 1) logits_kernel(
    const __grid_constant__ CUtensorMap tmQh, const __grid_constant__ CUtensorMap tmQl,
    const __grid_constant__ CUtensorMap tmKh, const __grid_constant__ CUtensorMap tmKl, int Mq,
    int Mk, int nmt, int nnt, float scale, float* __restrict__ logits,
    int32_t* __restrict__ status) {
  using C = LgCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const uint32_t s0 = smem_u32(sm);
  const uint32_t bar_ld = s0 + C::off_bar, bar_mma = s0 + C::off_bar + 8;
  uint32_t* slot = reinterpret_cast<uint32_t*>(sm + C::off_slot);
  const int warp = threadIdx.x >> 5;
  const int per_head = nmt * nnt;
  const int bh = blockIdx.x / per_head;
  const int mt = (blockIdx.x % per_head) / nnt;
  const int nt = blockIdx.x % nnt;

  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    mbar_init(bar_ld, 1);
    mbar_init(bar_mma, 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(slot), kLgTile);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;
  if (threadIdx.x == 0) {
    pdl_wait_primary();  // the pooled means are complete and visible
    mbar_arrive_expect_tx(bar_ld, 4 * C::kTile);
    for (int c = 0; c < C::KCH; ++c) {
      const uint32_t co = c * (kLgTile * 128);
      tma_load_3d(s0 + C::off_ahi + co, &tmQh, bar_ld, c * 64, mt * kLgTile, bh);
      tma_load_3d(s0 + C::off_alo + co, &tmQl, bar_ld, c * 64, mt * kLgTile, bh);
      tma_load_3d(s0 + C::off_bhi + co, &tmKh, bar_ld, c * 64, nt * kLgTile, bh);
      tma_load_3d(s0 + C::off_blo + co, &tmKl, bar_ld, c * 64, nt * kLgTile, bh);
    }
    if (mbar_wait(bar_ld, 0, kWaitTimeoutNs)) {
      tc_fence_after();
      constexpr uint32_t id = idesc_bf16(kLgTile, kLgTile, false, false);
      const uint64_t ahi = sdesc_sw128(s0 + C::off_ahi, 16, 1024);
      const uint64_t alo = sdesc_sw128(s0 + C::off_alo, 16, 1024);
      const uint64_t bhi = sdesc_sw128(s0 + C::off_bhi, 16, 1024);
      const uint64_t blo = sdesc_sw128(s0 + C::off_blo, 16, 1024);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t ko = (kk >> 2) * (kLgTile * 128) + (kk & 3) * 32;
        tc_mma_bf16(tmem, sdesc_add(ahi, ko), sdesc_add(bhi, ko), id, kk > 0 ? 1u : 0u);
        tc_mma_bf16(tmem, sdesc_add(ahi, ko), sdesc_add(blo, ko), id, 1u);
        tc_mma_bf16(tmem, sdesc_add(alo, ko), sdesc_add(bhi, ko), id, 1u);
      }
    } else {
      report_error(status, SPARGE_ERR_TIMEOUT);
    }
    tc_commit(bar_mma);
  }
  const bool ok = warp_wait(bar_mma, 0);
  if (!ok && (threadIdx.x & 31) == 0) report_error(status, SPARGE_ERR_TIMEOUT);
  tc_fence_after();
  if (ok) {
    const int quarter = warp & 3, cg = warp >> 2;  // lane quarter, column group
    const int i = mt * kLgTile + quarter * 32 + (threadIdx.x & 31);
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    float* dst = logits + ((long long)bh * Mq + min(i, Mq - 1)) * Mk + nt * kLgTile;
    const int ncol = min(kLgTile, Mk - nt * kLgTile);
#pragma unroll 1
    for (int c0 = cg * 32; c0 < cg * 32 + 32; c0 += 16) {
      uint32_t v[16];
      SPARGE_TMEM_LD_X16(lane_base + c0, v);
      SPARGE_TMEM_WAIT_LD16(v);
      if (i < Mq) {
        if ((Mk & 3) == 0 && c0 + 16 <= ncol) {  // rows 16-byte aligned
#pragma unroll
          for (int c = 0; c < 16; c += 4)
            *reinterpret_cast<float4*>(dst + c0 + c) =
                make_float4(__uint_as_float(v[c]) * scale, __uint_as_float(v[c + 1]) * scale,
                            __uint_as_float(v[c + 2]) * scale, __uint_as_float(v[c + 3]) * scale);
        } else {
#pragma unroll
          for (int c = 0; c < 16; ++c)
            if (c0 + c < ncol) dst[c0 + c] = __uint_as_float(v[c]) * scale;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kLgTile);
  }
}

// Row softmax and hybrid selection with the row in registers (Mk <= 32*EPL):
// one warp per q-block row, all of the row's loads in flight at once.
constexpr int kSelrThreads = 256;
template <int EPL>
__global__ void __launch_bounds__(kSelrThreads) select_logits_reg_kernel(
    const float* __restrict__ logits, int rows, int Mk, int Mkw, int ktop, float p,
    uint32_t* __restrict__ bitmask, int32_t* __restrict__ row_idx,
    int32_t* __restrict__ row_cnt, float* __restrict__ logit_out,
    float* __restrict__ prob_out) {
  const int lane = threadIdx.x & 31;
  const long long grow = (long long)blockIdx.x * (kSelrThreads / 32) + (threadIdx.x >> 5);
  pdl_wait_primary();  // logits are complete and visible
  pdl_launch_dependents();
  if (grow >= rows) return;
  const float* src = logits + grow * Mk;
  float x[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    const int j = e * 32 + lane;
    x[e] = j < Mk ? __ldcg(src + j) : -INFINITY;
  }
  float m = -INFINITY;
#pragma unroll
  for (int e = 0; e < EPL; ++e) m = fmaxf(m, x[e]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
  // exp(x - m) = 2^(x log2 e - m log2 e); P = e * (1 / sum), within 2 ulp of
  // the correctly rounded quotient.
  constexpr float kL2e = 1.4426950408889634f;
  const float ml = m * kL2e;
  float sum = 0.f;
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    const int j = e * 32 + lane;
    if (logit_out && j < Mk) logit_out[grow * Mk + j] = x[e];
    x[e] = j < Mk ? ex2_approx(fmaf(x[e], kL2e, -ml)) : 0.f;
    sum += x[e];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(kFull, sum, o);
  const float inv = __frcp_rn(sum);
  uint32_t kr[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    const int j = e * 32 + lane;
    const float pj = x[e] * inv;
    kr[e] = __float_as_uint(pj);  // absent elements: 0 / sum = +0, key 0
    if (prob_out && j < Mk) prob_out[grow * Mk + j] = pj;
  }
  select_keys<EPL, true>(kr, nullptr, Mk, ktop, p, bitmask + grow * Mkw, row_idx + grow * Mk,
                         row_cnt + grow);
}

constexpr int kSelkThreads = 256;                   // 8 warps, one row each
#ifndef SPARGE_SELK_MINB
#define SPARGE_SELK_MINB 3
#endif
constexpr int kSelkRows = kSelkThreads / 32;        // q-blocks per CTA (max)
constexpr int kSelkLogitFloats = 10240;             // 40 KB of rows per CTA

struct SelkSmem {
  uint32_t hcnt[kSelkRows][256];                    // radix fallback (Mk > 2048)
  unsigned long long hsum[kSelkRows][256];
};

__global__ void __launch_bounds__(kSelkThreads, SPARGE_SELK_MINB) select_logits_kernel(
    const float* __restrict__ logits, int Mq, int Mk, int Mkw, int R, int ktop, float p,
    uint32_t* __restrict__ bitmask, int32_t* __restrict__ row_idx,
    int32_t* __restrict__ row_cnt, float* __restrict__ logit_out,
    float* __restrict__ prob_out) {
  extern __shared__ __align__(16) uint8_t smem[];
  SelkSmem* hs = reinterpret_cast<SelkSmem*>(smem);
  float* ls = reinterpret_cast<float*>(smem + sizeof(SelkSmem));  // [R][Mk]
  const int nrb = (Mq + R - 1) / R;
  const int bh = blockIdx.x / nrb;
  const int i0 = (blockIdx.x % nrb) * R;
  const int nrows = min(R, Mq - i0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  pdl_wait_primary();  // logits are complete and visible
  pdl_launch_dependents();
  if (warp < nrows) {
    float* row = ls + warp * Mk;
    const long long grow = (long long)bh * Mq + i0 + warp;
    const float* src = logits + grow * Mk;
    float m = -INFINITY;
    for (int j = lane; j < Mk; j += 32) {
      const float lg = __ldcg(src + j);
      row[j] = lg;
      m = fmaxf(m, lg);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
    float sum = 0.f;
    for (int j = lane; j < Mk; j += 32) {
      const float lg = row[j];
      if (logit_out) logit_out[grow * Mk + j] = lg;
      const float e = expf(lg - m);
      row[j] = e;
      sum += e;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(kFull, sum, o);
    for (int j = lane; j < Mk; j += 32) {
      const float pj = __fdiv_rn(row[j], sum);
      row[j] = pj;
      if (prob_out) prob_out[grow * Mk + j] = pj;
    }
    __syncwarp();
    select_row_any(row, Mk, ktop, p, hs->hcnt[warp], hs->hsum[warp], bitmask + grow * Mkw,
                   row_idx + grow * Mk, row_cnt + grow);
  }
}

// CTA = (head, bitmask word w), 8 warps; the columns are the 32 kv-blocks
// 32w + b.  Rows go in passes of 256, thread t holding the word of row
// pass*256 + t.  Per column b, warp g's 32 rows form the ballot of bit b:
// its popcount is the warp's count, and after an exclusive scan over the
// warps (plus the counts of earlier passes) each set lane writes its row at
// offset + rank, so the column's rows land contiguously in ascending order.
constexpr int kCscSplitThreads = 256;
__global__ void __launch_bounds__(kCscSplitThreads) csc_split_kernel(
    const uint32_t* __restrict__ bitmask, int Mq, int Mk, int Mkw, int32_t* __restrict__ col_idx,
    int32_t* __restrict__ col_cnt) {
  constexpr int W = kCscSplitThreads / 32;
  __shared__ int cnt_w[W][32];
  __shared__ int run[32];
  pdl_wait_primary();
  const int bh = blockIdx.x / Mkw;
  const int w = blockIdx.x % Mkw;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t lt = (1u << lane) - 1u;
  const uint32_t* src = bitmask + (long long)bh * Mq * Mkw + w;
  const int ncol = min(32, Mk - w * 32);
  int32_t* out0 = col_idx + ((long long)bh * Mk + w * 32) * Mq;
  if (threadIdx.x < 32) run[threadIdx.x] = 0;
  for (int r0 = 0; r0 < Mq; r0 += kCscSplitThreads) {
    const int i = r0 + threadIdx.x;
    const uint32_t word = i < Mq ? __ldcg(src + (long long)i * Mkw) : 0u;
    // Lane b keeps this warp's count of column b.
    int mine = 0;
#pragma unroll 8
    for (int b = 0; b < 32; ++b) {
      const int n = __popc(__ballot_sync(kFull, (word >> b) & 1u));
      if (lane == b) mine = n;
    }
    cnt_w[warp][lane] = mine;
    __syncthreads();
    int off = run[lane];
#pragma unroll
    for (int g = 0; g < W; ++g) off += g < warp ? cnt_w[g][lane] : 0;
#pragma unroll 4
    for (int b = 0; b < ncol; ++b) {
      const uint32_t m = __ballot_sync(kFull, (word >> b) & 1u);
      const int ob = __shfl_sync(kFull, off, b);
      if ((word >> b) & 1u) out0[(long long)b * Mq + ob + __popc(m & lt)] = i;
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      int t = 0;
#pragma unroll
      for (int g = 0; g < W; ++g) t += cnt_w[g][threadIdx.x];
      run[threadIdx.x] += t;
    }
    __syncthreads();
  }
  if (threadIdx.x < ncol) col_cnt[(long long)bh * Mk + w * 32 + threadIdx.x] = run[threadIdx.x];
}

}  // namespace

int select_rows_per_cta(int Mk) {
  int r = kSelLogitFloats / Mk;
  return r < 1 ? 1 : (r > kSelMaxRows ? kSelMaxRows : r);
}

cudaError_t launch_pool(const Geom& g, const void* q, const void* k, float* qbar, float* kbar,
                        cudaStream_t st) {
  const int do_q = qbar != nullptr;
  const int do_k = kbar != nullptr;
  if (g.d == 128)
    return launch_pool_kernel<128>(g, q, k, do_q, do_k, qbar, kbar, nullptr, nullptr, nullptr,
                                   nullptr, st);
  return launch_pool_kernel<64>(g, q, k, do_q, do_k, qbar, kbar, nullptr, nullptr, nullptr,
                                nullptr, st);
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

template <typename Kern, typename... Args>
cudaError_t launch_pdl(Kern kern, unsigned grid, unsigned block, size_t smem, cudaStream_t st,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <int D>
cudaError_t launch_mask_pipeline_impl(const Geom& g, const void* q, const void* k, void* qhi,
                                      void* qlo, void* khi, void* klo, float* logits, float scale,
                                      int ktop, float p, uint32_t* bitmask, int32_t* row_idx,
                                      int32_t* row_cnt, int32_t* col_idx, int32_t* col_cnt,
                                      float* logit_out, float* prob_out, int32_t* status,
                                      cudaStream_t st) {
  CUtensorMap tqh, tql, tkh, tkl;
  if (make_tmap_bf16(&tqh, qhi, g.BH, g.Mq, D, kLgTile) != 0 ||
      make_tmap_bf16(&tql, qlo, g.BH, g.Mq, D, kLgTile) != 0 ||
      make_tmap_bf16(&tkh, khi, g.BH, g.Mk, D, kLgTile) != 0 ||
      make_tmap_bf16(&tkl, klo, g.BH, g.Mk, D, kLgTile) != 0)
    return cudaErrorInvalidValue;
  cudaError_t e = launch_pool_kernel<D>(g, q, k, 1, 1, nullptr, nullptr, qhi, qlo, khi, klo, st);
  if (e != cudaSuccess) return e;
  using L = LgCfg<D>;
  const int nmt = (g.Mq + kLgTile - 1) / kLgTile, nnt = (g.Mk + kLgTile - 1) / kLgTile;
  if ((e = cudaFuncSetAttribute(logits_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(L::smem_alloc))) != cudaSuccess)
    return e;
  if ((e = launch_pdl(logits_kernel<D>, static_cast<unsigned>((long long)g.BH * nmt * nnt),
                      kLgThreads, L::smem_alloc, st, tqh, tql, tkh, tkl, g.Mq, g.Mk, nmt, nnt,
                      scale, logits, status)) != cudaSuccess)
    return e;
  if (g.Mk <= 32 * 16) {
    const long long rows = (long long)g.BH * g.Mq;
    constexpr int kRowsPerCta = kSelrThreads / 32;
    if ((e = launch_pdl(select_logits_reg_kernel<16>,
                        static_cast<unsigned>((rows + kRowsPerCta - 1) / kRowsPerCta),
                        kSelrThreads, 0, st, static_cast<const float*>(logits),
                        static_cast<int>(rows), g.Mk, g.Mkw, ktop, p, bitmask, row_idx, row_cnt,
                        logit_out, prob_out)) != cudaSuccess)
      return e;
  } else {
    int R = kSelkLogitFloats / g.Mk;
    R = R < 1 ? 1 : (R > kSelkRows ? kSelkRows : R);
    const int nrb = (g.Mq + R - 1) / R;
    const size_t smem = sizeof(SelkSmem) + (size_t)R * g.Mk * sizeof(float);
    if ((e = cudaFuncSetAttribute(select_logits_kernel,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(smem))) != cudaSuccess)
      return e;
    if ((e = launch_pdl(select_logits_kernel, static_cast<unsigned>((long long)g.BH * nrb),
                        kSelkThreads, smem, st, static_cast<const float*>(logits), g.Mq, g.Mk,
                        g.Mkw, R, ktop, p, bitmask, row_idx, row_cnt, logit_out, prob_out)) !=
        cudaSuccess)
      return e;
  }
  if (col_idx != nullptr) {
    e = launch_pdl(csc_split_kernel, static_cast<unsigned>((long long)g.BH * g.Mkw),
                   kCscSplitThreads, 0, st,
                   static_cast<const uint32_t*>(bitmask), g.Mq, g.Mk, g.Mkw, col_idx, col_cnt);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

cudaError_t launch_mask_pipeline(const Geom& g, const void* q, const void* k, void* qhi,
                                 void* qlo, void* khi, void* klo, float* logits, float scale,
                                 int ktop, float p, uint32_t* bitmask, int32_t* row_idx,
                                 int32_t* row_cnt, int32_t* col_idx, int32_t* col_cnt,
                                 float* logit_out, float* prob_out, int32_t* status,
                                 cudaStream_t st) {
  if (g.d == 128)
    return launch_mask_pipeline_impl<128>(g, q, k, qhi, qlo, khi, klo, logits, scale, ktop, p,
                                          bitmask, row_idx, row_cnt, col_idx, col_cnt, logit_out,
                                          prob_out, status, st);
  return launch_mask_pipeline_impl<64>(g, q, k, qhi, qlo, khi, klo, logits, scale, ktop, p,
                                       bitmask, row_idx, row_cnt, col_idx, col_cnt, logit_out,
                                       prob_out,
                                       status, st);
}

}  // namespace sparge
