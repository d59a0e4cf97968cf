// Block-sparse attention backward on sm_103a (tcgen05 + TMEM + TMA).
//
// Method: "SpargeAttention2: Trainable Sparse Attention via Hybrid Top-k+Top-p
// Masking and Distillation Fine-Tuning", section "Abstract" (the sparse
// attention is trainable), and the mindverse page "Optimierung der Effizienz
// von Video-Diffusionsmodellen durch SpargeAttention2", section "Effiziente
// Kernel-Implementierung und Modellanpassung" (forward and backward skip the
// masked tiles).  The mask is a constant; per kept (q-block i, kv-block j):
//   P = exp(scale*Q_i K_j^T - LSE_i),  dP = dO_i V_j^T,  dS = P * (dP - D_i)
//   dV_j += P^T dO_i,  dK_j += scale * dS^T Q_i,  dQ_i += scale * dS K_j
// with D_t = sum_c dO_tc O_tc.
//
// Kernels, no atomics (deterministic):
//   bwd_delta_kernel  D per token (HBM-bound, 16-byte loads).
//   (two extra CTAs of the delta grid) launch orders of the two gradient
//                     kernels: long lists first, then index order (a stable
//                     partition).
//   bwd_dkdv_kernel   one CTA per kv-block, loops over the q-blocks that keep
//                     it (CSC list).  S and dP are recomputed into TMEM
//                     (M = 128 query rows); dV^T and dK^T accumulate in TMEM
//                     as M = d tiles, dV^T += dO^T P and dK^T += Q^T dS, with
//                     dO, Q, P and dS read in the MN-major smem layout.
//   bwd_dq_kernel     one CTA per q-block, loops over its kept kv-blocks (CSR
//                     list); recomputes S, dP and dS and accumulates
//                     dQ += dS K in TMEM.  Q and dO (reused by every tile)
//                     and dS are MMA A operands read from TMEM.
// Roles per CTA: eight compute warps (two per TMEM lane quarter, each owning
// 32 of a tile's 64 key columns), a TMA producer warp and two MMA-issuing
// warps (S and dP; then the gradient MMAs; two issuers let the gradient MMAs
// of a tile be queued while the next tile's S and dP are issued).  Every wait
// is bounded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "common.cuh"
#include "kernels.h"

namespace sparge {

namespace {

constexpr int kBM = 128;
constexpr int kBN = 64;
constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------- work order
// Launch order of the gradient CTAs: the lists longer than twice the mean
// first, then the others, each group in index order (a stable partition).
// Long lists (attention-sink blocks that nearly every q-block keeps) would
// otherwise run alone at the end of the grid; index order keeps the CTAs of
// one head together, so that head's Q/dO (or K/V) tiles are served from L2.
// One CTA of NT threads partitions the n items.
template <int NT>
__device__ void order_by_count(const int32_t* __restrict__ cnt, int n, int32_t* __restrict__ order) {
  constexpr int W = NT / 32;
  __shared__ long long red[W];
  __shared__ int scan[W];
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int E = (n + NT - 1) / NT;
  const int lo = min(n, tid * E), hi = min(n, lo + E);
  // Total of the counts.
  long long sum = 0;
  for (int it = lo; it < hi; ++it) sum += max(__ldg(cnt + it), 0);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane == 0) red[w] = sum;
  __syncthreads();
  long long total = 0;
#pragma unroll
  for (int i = 0; i < W; ++i) total += red[i];
  // Item `it` is long when cnt * n > 2 * total.
  auto is_long = [&](int it) { return (long long)max(__ldg(cnt + it), 0) * n > 2 * total; };
  int nl = 0;
  for (int it = lo; it < hi; ++it) nl += is_long(it) ? 1 : 0;
  // Exclusive scan of the per-thread long counts.
  int incl = nl;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) scan[w] = incl;
  __syncthreads();
  if (w == 0) {
    int t = lane < W ? scan[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += v;
    }
    if (lane < W) scan[lane] = t;  // inclusive warp totals
  }
  __syncthreads();
  const int before_long = incl - nl + (w > 0 ? scan[w - 1] : 0);
  const int n_long = scan[W - 1];
  int pl = before_long;                // next long position
  int ps = n_long + lo - before_long;  // next short position
  for (int it = lo; it < hi; ++it) order[is_long(it) ? pl++ : ps++] = it;
}

// ---------------------------------------------------------------- D = rowsum(dO * O)
// CTAs [0, ndelta) compute D; the two CTAs after them build the launch orders
// of the kv-blocks and of the q-blocks while the rest of the grid streams O
// and dO.
template <int D>
__global__ void __launch_bounds__(256) bwd_delta_kernel(
    const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout, long long rows,
    float* __restrict__ delta, unsigned ndelta, const int32_t* __restrict__ col_cnt, int ncol,
    int32_t* __restrict__ col_order, const int32_t* __restrict__ row_cnt, int nrow,
    int32_t* __restrict__ row_order) {
  if (blockIdx.x >= ndelta) {
    if (blockIdx.x == ndelta)
      order_by_count<256>(col_cnt, ncol, col_order);
    else
      order_by_count<256>(row_cnt, nrow, row_order);
    return;
  }
  constexpr int CH = D / 8;        // 16-byte chunks per row
  constexpr int RPB = 256 / CH;    // rows per block pass
  const long long r = (long long)blockIdx.x * RPB + threadIdx.x / CH;
  const int c = threadIdx.x % CH;
  float s = 0.f;
  if (r < rows) {
    const uint4 a = __ldg(reinterpret_cast<const uint4*>(o + r * D) + c);
    const uint4 b = __ldg(reinterpret_cast<const uint4*>(dout + r * D) + c);
    const __nv_bfloat162* ha = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* hb = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 fa = __bfloat1622float2(ha[e]);
      const float2 fb = __bfloat1622float2(hb[e]);
      s = fmaf(fa.x, fb.x, s);
      s = fmaf(fa.y, fb.y, s);
    }
  }
#pragma unroll
  for (int off = CH / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (c == 0 && r < rows) delta[r] = s;
}

// Writes 32 bf16 values (half of a 128-byte row: 16-byte chunks 4h .. 4h+3)
// into a 128-byte-swizzled tile.
__device__ __forceinline__ void store_half_row_sw128(uint8_t* tile, int row, int half,
                                                     const uint32_t (&pk)[16]) {
#pragma unroll
  for (int ch = 0; ch < 4; ++ch) {
    uint4 v;
    v.x = pk[4 * ch + 0];
    v.y = pk[4 * ch + 1];
    v.z = pk[4 * ch + 2];
    v.w = pk[4 * ch + 3];
    *reinterpret_cast<uint4*>(tile + sw128_offset(row, (half * 4 + ch) * 16)) = v;
  }
}

// Warp roles of both gradient kernels (352 threads): warps 0-7 compute, with
// query row (or feature) 32*(w % 4) + lane = TMEM lane and score columns
// 32*(w / 4) .. +31 (P comes from the saved LSE, so a row needs no exchange
// between its two warps); warp 8 TMA producer; warp 9 issues the S and dP
// MMAs; warp 10 issues the gradient MMAs.  Two issuers let the MMAs of
// neighbouring tiles overlap.
constexpr int kGradThreads = 352;
constexpr int kComputeWarps = 8;
constexpr int kGProducer = 8;
constexpr int kGIssueA = 9;
constexpr int kGIssueB = 10;

// ---------------------------------------------------------------- dK, dV
template <int D>
struct DkdvCfg {
  static constexpr int NST = 2;
  static constexpr int KCH = D / 64;
  static constexpr uint32_t kKV = kBN * D * 2;  // one K or V tile
  static constexpr uint32_t kQ = kBM * D * 2;   // one Q or dO tile
  static constexpr uint32_t kP = kBM * kBN * 2;
  static constexpr uint32_t off_k = 0;
  static constexpr uint32_t off_v = off_k + kKV;
  static constexpr uint32_t off_q = off_v + kKV;                 // NST stages of Q
  static constexpr uint32_t off_do = off_q + NST * kQ;           // NST stages of dO
  static constexpr uint32_t off_p = off_do + NST * kQ;           // 2 buffers
  static constexpr uint32_t off_ds = off_p + 2 * kP;             // 2 buffers
  static constexpr uint32_t off_bar = off_ds + 2 * kP;
  static constexpr int B_KV = 0;
  static constexpr int B_QF = 1;
  static constexpr int B_QE = B_QF + NST;
  static constexpr int B_SF = B_QE + NST;  // 2
  static constexpr int B_PSF = B_SF + 2;   // 2, count 256
  static constexpr int B_PSE = B_PSF + 2;  // 2
  static constexpr int B_DONE = B_PSE + 2; // count 2
  static constexpr int NBAR = B_DONE + 1;
  static constexpr uint32_t off_slot = off_bar + NBAR * 8;
  static constexpr uint32_t bytes = off_slot + 16;
  static constexpr uint32_t smem_alloc = bytes + 1024;
  static constexpr uint32_t tmem_cols = 512;  // S/dP x2 [0,256), dV^T [256,320), dK^T [320,384)
  static constexpr uint32_t col_dv = 256;
  static constexpr uint32_t col_dk = 320;
};

template <int D>
__global__ void __launch_bounds__(kGradThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                    const float* __restrict__ lse, const float* __restrict__ delta,
                    const int32_t* __restrict__ col_idx, const int32_t* __restrict__ col_cnt,
                    const int32_t* __restrict__ col_order, int N, int Mq, int Mk, float scale,
                    float scale_log2, __nv_bfloat16* __restrict__ dk,
                    __nv_bfloat16* __restrict__ dv, int32_t* __restrict__ status) {
  using C = DkdvCfg<D>;
  // The dQ kernel (independent of this one) may start on SMs this grid's
  // last CTAs leave idle.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const uint32_t s0 = smem_u32(sm);
  auto bar = [&](int i) -> uint32_t { return s0 + C::off_bar + 8u * i; };
  uint32_t* slot = reinterpret_cast<uint32_t*>(sm + C::off_slot);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int item = min(max(__ldg(col_order + blockIdx.x), 0), static_cast<int>(gridDim.x) - 1);
  const int bh = item / Mk;
  const int j = item % Mk;
  const long long col_id = (long long)bh * Mk + j;
  const int n = min(max(__ldg(col_cnt + col_id), 0), Mq);
  const int32_t* list = col_idx + col_id * Mq;
  const int kv_valid = min(kBN, N - j * kBN);

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NBAR; ++i) {
      uint32_t cnt = 1;
      if (i == C::B_PSF || i == C::B_PSF + 1) cnt = 32 * kComputeWarps;
      if (i == C::B_DONE) cnt = 2;
      mbar_init(bar(i), cnt);
    }
    fence_barrier_init();
  }
  if (warp == kGIssueA) {
    tmem_alloc(smem_u32(slot), C::tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;

  if (warp == kGProducer) {
    if (lane == 0 && n > 0) {
      mbar_arrive_expect_tx(bar(C::B_KV), 2 * C::kKV);
      for (int c = 0; c < C::KCH; ++c) {
        tma_load_3d(s0 + C::off_k + c * kBN * 128, &tmK, bar(C::B_KV), c * 64, j * kBN, bh);
        tma_load_3d(s0 + C::off_v + c * kBN * 128, &tmV, bar(C::B_KV), c * 64, j * kBN, bh);
      }
      int issued = 0;
      for (int t = 0; t < n; ++t) {
        const int s = t % C::NST;
        if (t >= C::NST && !mbar_wait(bar(C::B_QE + s), ((t / C::NST) - 1) & 1, kWaitTimeoutNs)) {
          report_error(status, SPARGE_ERR_TIMEOUT);
          break;
        }
        const int i = min(max(__ldg(list + t), 0), Mq - 1);
        mbar_arrive_expect_tx(bar(C::B_QF + s), 2 * C::kQ);
        for (int c = 0; c < C::KCH; ++c) {
          tma_load_3d(s0 + C::off_q + s * C::kQ + c * kBM * 128, &tmQ, bar(C::B_QF + s), c * 64,
                      i * kBM, bh);
          tma_load_3d(s0 + C::off_do + s * C::kQ + c * kBM * 128, &tmDO, bar(C::B_QF + s), c * 64,
                      i * kBM, bh);
        }
        issued = t + 1;
      }
      for (int t = max(0, issued - C::NST); t < issued; ++t)
        mbar_wait(bar(C::B_QF + t % C::NST), (t / C::NST) & 1, kWaitTimeoutNs);
    }
  } else if (warp == kGIssueA) {
    // S_t = Q_t K^T and dP_t = dO_t V^T (M = 128 query rows, N = 64 keys).
    if (lane == 0 && n > 0) {
      constexpr uint32_t idS = idesc_bf16(kBM, kBN, false, false);
      const uint64_t dk0 = sdesc_sw128(s0 + C::off_k, 16, 1024);
      const uint64_t dv0 = sdesc_sw128(s0 + C::off_v, 16, 1024);
      bool ok = mbar_wait(bar(C::B_KV), 0, kWaitTimeoutNs);
      for (int t = 0; ok && t < n; ++t) {
        const int s = t % C::NST;
        // TMEM buffer t & 1 was read by the compute warps of tile t - 2 before
        // they filled P/dS(t - 2).
        if (!mbar_wait(bar(C::B_QF + s), (t / C::NST) & 1, kWaitTimeoutNs) ||
            (t >= 2 && !mbar_wait(bar(C::B_PSF + (t & 1)), ((t - 2) >> 1) & 1, kWaitTimeoutNs))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t dq = sdesc_sw128(s0 + C::off_q + s * C::kQ, 16, 1024);
        const uint64_t ddo = sdesc_sw128(s0 + C::off_do + s * C::kQ, 16, 1024);
        const uint32_t dS = tmem + (t & 1) * 128;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ko = (kk >> 2) * (kBM * 128) + (kk & 3) * 32;
          const uint32_t kko = (kk >> 2) * (kBN * 128) + (kk & 3) * 32;
          tc_mma_bf16(dS, sdesc_add(dq, ko), sdesc_add(dk0, kko), idS, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ko = (kk >> 2) * (kBM * 128) + (kk & 3) * 32;
          const uint32_t kko = (kk >> 2) * (kBN * 128) + (kk & 3) * 32;
          tc_mma_bf16(dS + 64, sdesc_add(ddo, ko), sdesc_add(dv0, kko), idS, kk > 0);
        }
        tc_commit(bar(C::B_SF + (t & 1)));
      }
      if (!ok) report_error(status, SPARGE_ERR_TIMEOUT);
      tc_commit(bar(C::B_DONE));
      mbar_wait(bar(C::B_DONE), 0, kWaitTimeoutNs);
    }
  } else if (warp == kGIssueB) {
    // dV^T += dO_u^T P_u and dK^T += Q_u^T dS_u (M = d, N = 64 keys, K = 16
    // query rows per step; A and B read MN-major).
    if (lane == 0 && n > 0) {
      constexpr uint32_t idG = idesc_bf16(kBM, kBN, true, true);
      bool ok = true;
      for (int u = 0; ok && u < n; ++u) {
        const int su = u % C::NST;
        const int pb = u & 1;
        if (!mbar_wait(bar(C::B_PSF + pb), (u >> 1) & 1, kWaitTimeoutNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t dq = sdesc_sw128(s0 + C::off_q + su * C::kQ, kBM * 128, 1024);
        const uint64_t ddo = sdesc_sw128(s0 + C::off_do + su * C::kQ, kBM * 128, 1024);
        const uint64_t dpb = sdesc_sw128(s0 + C::off_p + pb * C::kP, kBM * 128, 1024);
        const uint64_t dsb = sdesc_sw128(s0 + C::off_ds + pb * C::kP, kBM * 128, 1024);
#pragma unroll
        for (int kk = 0; kk < kBM / 16; ++kk)
          tc_mma_bf16(tmem + C::col_dv, sdesc_add(ddo, kk * 2048), sdesc_add(dpb, kk * 2048), idG,
                      (u > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < kBM / 16; ++kk)
          tc_mma_bf16(tmem + C::col_dk, sdesc_add(dq, kk * 2048), sdesc_add(dsb, kk * 2048), idG,
                      (u > 0 || kk > 0) ? 1u : 0u);
        // S/dP(u) completed before P/dS(u) were written, so the Q/dO stage is
        // free once these MMAs complete.
        tc_commit(bar(C::B_QE + su));
        tc_commit(bar(C::B_PSE + pb));
      }
      if (!ok) report_error(status, SPARGE_ERR_TIMEOUT);
      tc_commit(bar(C::B_DONE));
      mbar_wait(bar(C::B_DONE), 0, kWaitTimeoutNs);
    }
  } else {
    const int quarter = warp & 3, half = warp >> 2;
    const int r = quarter * 32 + lane;
    const int c0 = half * 32;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    bool ok = true;
    // Two-deep prefetch: the q-block index of tile t+2 and the LSE / D of
    // tile t+1 are loaded while tile t is computed.
    const float* lse_h = lse + (long long)bh * N;
    const float* del_h = delta + (long long)bh * N;
    auto row_of = [&](int qi) { return qi * kBM + r; };
    int i_n1 = n > 0 ? min(max(__ldg(list), 0), Mq - 1) : 0;
    int i_n2 = n > 1 ? min(max(__ldg(list + 1), 0), Mq - 1) : 0;
    float lse_n = 0.f, del_n = 0.f;
    if (n > 0 && row_of(i_n1) < N) {
      lse_n = __ldg(lse_h + row_of(i_n1));
      del_n = __ldg(del_h + row_of(i_n1));
    }
    for (int t = 0; t < n; ++t) {
      const bool rv = row_of(i_n1) < N;
      const float lse2 = rv ? lse_n * kLog2e : 0.f;
      const float drow = rv ? del_n : 0.f;
      i_n1 = i_n2;
      if (t + 1 < n && row_of(i_n1) < N) {
        lse_n = __ldg(lse_h + row_of(i_n1));
        del_n = __ldg(del_h + row_of(i_n1));
      }
      if (t + 2 < n) i_n2 = min(max(__ldg(list + t + 2), 0), Mq - 1);
      if (!warp_wait(bar(C::B_SF + (t & 1)), (t >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t pk[16], dk_[16];
      {
        float s[32], dp[32];
        tmem_ld32(lane_base + (t & 1) * 128 + c0, s);
        tmem_ld32(lane_base + (t & 1) * 128 + 64 + c0, dp);
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          float p0 = ex2_approx(fmaf(s[c], scale_log2, -lse2));
          float p1 = ex2_approx(fmaf(s[c + 1], scale_log2, -lse2));
          if (!rv || c0 + c >= kv_valid) p0 = 0.f;
          if (!rv || c0 + c + 1 >= kv_valid) p1 = 0.f;
          pk[c / 2] = pack_bf16x2(p0, p1);
          dk_[c / 2] = pack_bf16x2(p0 * (dp[c] - drow), p1 * (dp[c + 1] - drow));
        }
      }
      // Buffer t & 1 is free once the dV/dK MMAs of tile t-2 have completed.
      if (t >= 2 && !warp_wait(bar(C::B_PSE + (t & 1)), ((t - 2) >> 1) & 1)) {
        ok = false;
        break;
      }
      store_half_row_sw128(sm + C::off_p + (t & 1) * C::kP, r, half, pk);
      store_half_row_sw128(sm + C::off_ds + (t & 1) * C::kP, r, half, dk_);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(C::B_PSF + (t & 1)));
    }
    if (!ok) report_error(status, SPARGE_ERR_TIMEOUT);
    // Epilogue: lane r holds feature r of dV^T / dK^T; this warp writes the 32
    // keys c0 .. c0+31 of it.
    bool have = ok && n > 0;
    if (have) {
      have = warp_wait(bar(C::B_PSE + ((n - 1) & 1)), ((n - 1) >> 1) & 1);
      if (!have) report_error(status, SPARGE_ERR_TIMEOUT);
    }
    tc_fence_after();
    const long long base = ((long long)bh * N + (long long)j * kBN) * D + r;
#pragma unroll 1
    for (int cc = c0; cc < c0 + 32; cc += 16) {
      uint32_t rv_[16], rk_[16];
      if (have) {
        SPARGE_TMEM_LD_X16(lane_base + C::col_dv + cc, rv_);
        SPARGE_TMEM_LD_X16(lane_base + C::col_dk + cc, rk_);
        SPARGE_TMEM_WAIT_LD16(rv_);
        SPARGE_TMEM_WAIT_LD16(rk_);
      } else {
#pragma unroll
        for (int c = 0; c < 16; ++c) rv_[c] = rk_[c] = 0u;
      }
      if (r < D) {
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          if (cc + c < kv_valid) {
            __stcs(dv + base + (long long)(cc + c) * D, __float2bfloat16_rn(__uint_as_float(rv_[c])));
            __stcs(dk + base + (long long)(cc + c) * D,
                   __float2bfloat16_rn(__uint_as_float(rk_[c]) * scale));
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kGIssueA) {
    tc_fence_after();
    tmem_dealloc(tmem, C::tmem_cols);
  }
}

// ---------------------------------------------------------------- dQ
template <int D>
struct DqCfg {
  static constexpr int KCH = D / 64;
  static constexpr uint32_t kKV = kBN * D * 2;
  static constexpr uint32_t kQ = kBM * D * 2;
  static constexpr int NST = 4;
  static constexpr uint32_t off_q = 0;
  static constexpr uint32_t off_do = off_q + kQ;
  static constexpr uint32_t off_k = off_do + kQ;
  static constexpr uint32_t off_v = off_k + NST * kKV;
  static constexpr uint32_t off_bar = off_v + NST * kKV;
  static constexpr int B_Q = 0;
  static constexpr int B_QT = 1;            // Q, dO copied into TMEM (count 256)
  static constexpr int B_KF = 2;
  static constexpr int B_VF = B_KF + NST;
  static constexpr int B_KE = B_VF + NST;   // K slot free (dQ of its tile done)
  static constexpr int B_VE = B_KE + NST;   // V slot free (dP of its tile done)
  static constexpr int B_SF = B_VE + NST;   // 2
  static constexpr int B_DSF = B_SF + 2;    // 2, count 256 (dS written)
  static constexpr int B_DSE = B_DSF + 2;   // 2 (dQ of the tile done: TMEM tile free)
  static constexpr int B_DONE = B_DSE + 2;  // count 2
  static constexpr int NBAR = B_DONE + 1;
  static constexpr uint32_t off_slot = off_bar + NBAR * 8;
  static constexpr uint32_t bytes = off_slot + 16;
  static constexpr uint32_t smem_alloc = bytes + 1024;
  // TMEM: S/dP x2 [0,256) (S_b at 128b, dP_b at 128b + 64), dQ [256, 256+D),
  // Q and dO as MMA A operands (bf16 pairs, D/2 columns each) after it.  dS_t
  // (bf16 pairs, 32 columns) goes over columns 16..47 of S_t's tile: the half
  // of a row that read S columns 0..31 writes 16..31, the other 32..47, so no
  // warp overwrites columns another warp has still to read.  Q and dO in TMEM
  // keep their operand reads (reused by every tile) out of shared memory.
  static constexpr uint32_t tmem_cols = 512;
  static constexpr uint32_t col_dq = 256;
  static constexpr uint32_t col_q = 256 + D;
  static constexpr uint32_t col_do = col_q + D / 2;
  static constexpr uint32_t col_ds = 16;
};

// Copies this thread's half row of a 128-byte-swizzled bf16 tile (rows of D
// values, 64-column chunks 128 * kBM bytes apart) into TMEM lane `lane_addr`
// as bf16 pairs: D/4 columns starting at column half * D/4.
template <int D>
__device__ __forceinline__ void tile_half_row_to_tmem(const uint8_t* tile, int row, int half,
                                                      uint32_t lane_addr) {
  constexpr int W = D / 4;  // 32-bit columns per half row
  uint32_t v[W];
#pragma unroll
  for (int q4 = 0; q4 < W / 4; ++q4) {
    const int byte = half * (D / 2) * 2 + q4 * 16;  // byte offset within the row
    const uint4 u = *reinterpret_cast<const uint4*>(tile + (byte / 128) * (kBM * 128) +
                                                    sw128_offset(row, byte % 128));
    v[4 * q4 + 0] = u.x;
    v[4 * q4 + 1] = u.y;
    v[4 * q4 + 2] = u.z;
    v[4 * q4 + 3] = u.w;
  }
#pragma unroll
  for (int c = 0; c < W; c += 16) SPARGE_TMEM_ST_X16(lane_addr + half * W + c, (v + c));
}

// tcgen05.mma kind::f16 with the A operand in tensor memory (M lanes, K/2
// 32-bit columns holding bf16 pairs, element 2c in the low half of column c).
__device__ __forceinline__ void tc_mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

template <int D>
__global__ void __launch_bounds__(kGradThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                  const float* __restrict__ lse, const float* __restrict__ delta,
                  const int32_t* __restrict__ row_idx, const int32_t* __restrict__ row_cnt,
                  const int32_t* __restrict__ row_order, int N, int Mq, int Mk, float scale,
                  float scale_log2, __nv_bfloat16* __restrict__ dq, int32_t* __restrict__ status) {
  using C = DqCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const uint32_t s0 = smem_u32(sm);
  auto bar = [&](int i) -> uint32_t { return s0 + C::off_bar + 8u * i; };
  uint32_t* slot = reinterpret_cast<uint32_t*>(sm + C::off_slot);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int item = min(max(__ldg(row_order + blockIdx.x), 0), static_cast<int>(gridDim.x) - 1);
  const int bh = item / Mq;
  const int qb = item % Mq;
  const long long row_id = (long long)bh * Mq + qb;
  const int n = min(max(__ldg(row_cnt + row_id), 0), Mk);
  const int32_t* list = row_idx + row_id * Mk;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NBAR; ++i) {
      uint32_t cnt = 1;
      if (i == C::B_DSF || i == C::B_DSF + 1 || i == C::B_QT) cnt = 32 * kComputeWarps;
      if (i == C::B_DONE) cnt = 2;
      mbar_init(bar(i), cnt);
    }
    fence_barrier_init();
  }
  if (warp == kGIssueA) {
    tmem_alloc(smem_u32(slot), C::tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;

  if (warp == kGProducer) {
    if (lane == 0 && n > 0) {
      mbar_arrive_expect_tx(bar(C::B_Q), 2 * C::kQ);
      for (int c = 0; c < C::KCH; ++c) {
        tma_load_3d(s0 + C::off_q + c * kBM * 128, &tmQ, bar(C::B_Q), c * 64, qb * kBM, bh);
        tma_load_3d(s0 + C::off_do + c * kBM * 128, &tmDO, bar(C::B_Q), c * 64, qb * kBM, bh);
      }
      int issued = 0;
      for (int t = 0; t < n; ++t) {
        const int s = t % C::NST;
        if (t >= C::NST && !mbar_wait(bar(C::B_KE + s), ((t / C::NST) - 1) & 1, kWaitTimeoutNs)) {
          report_error(status, SPARGE_ERR_TIMEOUT);
          break;
        }
        const int jj = min(max(__ldg(list + t), 0), Mk - 1);
        mbar_arrive_expect_tx(bar(C::B_KF + s), C::kKV);
        for (int c = 0; c < C::KCH; ++c)
          tma_load_3d(s0 + C::off_k + s * C::kKV + c * kBN * 128, &tmK, bar(C::B_KF + s), c * 64,
                      jj * kBN, bh);
        if (t >= C::NST && !mbar_wait(bar(C::B_VE + s), ((t / C::NST) - 1) & 1, kWaitTimeoutNs)) {
          report_error(status, SPARGE_ERR_TIMEOUT);
          break;
        }
        mbar_arrive_expect_tx(bar(C::B_VF + s), C::kKV);
        for (int c = 0; c < C::KCH; ++c)
          tma_load_3d(s0 + C::off_v + s * C::kKV + c * kBN * 128, &tmV, bar(C::B_VF + s), c * 64,
                      jj * kBN, bh);
        issued = t + 1;
      }
      for (int t = max(0, issued - C::NST); t < issued; ++t) {
        mbar_wait(bar(C::B_KF + t % C::NST), (t / C::NST) & 1, kWaitTimeoutNs);
        mbar_wait(bar(C::B_VF + t % C::NST), (t / C::NST) & 1, kWaitTimeoutNs);
      }
    }
  } else if (warp == kGIssueA) {
    // S_t = Q K_t^T and dP_t = dO V_t^T, with Q and dO read from TMEM.
    if (lane == 0 && n > 0) {
      constexpr uint32_t idS = idesc_bf16(kBM, kBN, false, false);
      bool ok = mbar_wait(bar(C::B_QT), 0, kWaitTimeoutNs);
      for (int t = 0; ok && t < n; ++t) {
        const int s = t % C::NST;
        const uint32_t dS = tmem + (t & 1) * 128;
        // TMEM tile t & 1 holds dS(t - 2) until dQ(t - 2) has completed.
        if (!mbar_wait(bar(C::B_KF + s), (t / C::NST) & 1, kWaitTimeoutNs) ||
            (t >= 2 && !mbar_wait(bar(C::B_DSE + (t & 1)), ((t - 2) >> 1) & 1, kWaitTimeoutNs))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t dk = sdesc_sw128(s0 + C::off_k + s * C::kKV, 16, 1024);
        const uint64_t dv = sdesc_sw128(s0 + C::off_v + s * C::kKV, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t kko = (kk >> 2) * (kBN * 128) + (kk & 3) * 32;
          tc_mma_bf16_ta(dS, tmem + C::col_q + kk * 8, sdesc_add(dk, kko), idS, kk > 0);
        }
        if (!mbar_wait(bar(C::B_VF + s), (t / C::NST) & 1, kWaitTimeoutNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t kko = (kk >> 2) * (kBN * 128) + (kk & 3) * 32;
          tc_mma_bf16_ta(dS + 64, tmem + C::col_do + kk * 8, sdesc_add(dv, kko), idS, kk > 0);
        }
        tc_commit(bar(C::B_SF + (t & 1)));
        tc_commit(bar(C::B_VE + s));
      }
      if (!ok) report_error(status, SPARGE_ERR_TIMEOUT);
      tc_commit(bar(C::B_DONE));
      mbar_wait(bar(C::B_DONE), 0, kWaitTimeoutNs);
    }
  } else if (warp == kGIssueB) {
    // dQ += dS_u K_u (A = dS_u from TMEM, K = 64 keys; B = K_u MN-major, N = d).
    if (lane == 0 && n > 0) {
      constexpr uint32_t idQ = idesc_bf16(kBM, D, false, true);
      bool ok = true;
      for (int u = 0; ok && u < n; ++u) {
        const int su = u % C::NST;
        if (!mbar_wait(bar(C::B_DSF + (u & 1)), (u >> 1) & 1, kWaitTimeoutNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t ads = tmem + (u & 1) * 128 + C::col_ds;
        const uint64_t dk = sdesc_sw128(s0 + C::off_k + su * C::kKV, kBN * 128, 1024);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          tc_mma_bf16_ta(tmem + C::col_dq, ads + kk * 8, sdesc_add(dk, kk * 2048), idQ,
                         (u > 0 || kk > 0) ? 1u : 0u);
        tc_commit(bar(C::B_KE + su));
        tc_commit(bar(C::B_DSE + (u & 1)));
      }
      if (!ok) report_error(status, SPARGE_ERR_TIMEOUT);
      tc_commit(bar(C::B_DONE));
      mbar_wait(bar(C::B_DONE), 0, kWaitTimeoutNs);
    }
  } else {
    const int quarter = warp & 3, half = warp >> 2;
    const int r = quarter * 32 + lane;
    const int c0 = half * 32;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const int row = qb * kBM + r;
    const bool rv = row < N;
    const float lse2 = (rv && n > 0) ? __ldg(lse + (long long)bh * N + row) * kLog2e : 0.f;
    const float drow = rv ? __ldg(delta + (long long)bh * N + row) : 0.f;
    bool ok = true;
    // Q and dO into TMEM (this thread's half row of each), for the S and dP
    // MMAs of every tile.
    if (n > 0) {
      ok = warp_wait(bar(C::B_Q), 0);
      if (ok) {
        tile_half_row_to_tmem<D>(sm + C::off_q, r, half, lane_base + C::col_q);
        tile_half_row_to_tmem<D>(sm + C::off_do, r, half, lane_base + C::col_do);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(C::B_QT));
      }
    }
    int j_next = n > 0 ? min(max(__ldg(list), 0), Mk - 1) : 0;  // one tile ahead
    for (int t = 0; ok && t < n; ++t) {
      const int jj = j_next;
      if (t + 1 < n) j_next = min(max(__ldg(list + t + 1), 0), Mk - 1);
      const int kv_valid = N - jj * kBN;
      if (!warp_wait(bar(C::B_SF + (t & 1)), (t >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t pk[16];
      {
        float s[32], dp[32];
        tmem_ld32(lane_base + (t & 1) * 128 + c0, s);
        tmem_ld32(lane_base + (t & 1) * 128 + 64 + c0, dp);
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          float p0 = ex2_approx(fmaf(s[c], scale_log2, -lse2));
          float p1 = ex2_approx(fmaf(s[c + 1], scale_log2, -lse2));
          if (!rv || c0 + c >= kv_valid) p0 = 0.f;
          if (!rv || c0 + c + 1 >= kv_valid) p1 = 0.f;
          pk[c / 2] = pack_bf16x2(p0 * (dp[c] - drow), p1 * (dp[c + 1] - drow));
        }
      }
      // dS_t over columns col_ds + 16 * half .. + 15 of S_t's tile (this
      // warp's own S columns, already read into registers above).
      {
        const uint32_t da = lane_base + (t & 1) * 128 + C::col_ds + half * 16;
        SPARGE_TMEM_ST_X16(da, pk);
        tmem_st_wait();
      }
      tc_fence_before();
      mbar_arrive(bar(C::B_DSF + (t & 1)));
    }
    if (!ok) report_error(status, SPARGE_ERR_TIMEOUT);
    bool have = ok && n > 0;
    if (have) {
      have = warp_wait(bar(C::B_DSE + ((n - 1) & 1)), ((n - 1) >> 1) & 1);
      if (!have) report_error(status, SPARGE_ERR_TIMEOUT);
    }
    tc_fence_after();
    __nv_bfloat16* qrow = dq + ((long long)bh * N + row) * D;
#pragma unroll 1
    for (int cc = half * (D / 2); cc < (half + 1) * (D / 2); cc += 16) {
      uint32_t ro[16];
      if (have) {
        SPARGE_TMEM_LD_X16(lane_base + C::col_dq + cc, ro);
        SPARGE_TMEM_WAIT_LD16(ro);
      } else {
#pragma unroll
        for (int c = 0; c < 16; ++c) ro[c] = 0u;
      }
      uint4 w0, w1;
      w0.x = pack_bf16x2(__uint_as_float(ro[0]) * scale, __uint_as_float(ro[1]) * scale);
      w0.y = pack_bf16x2(__uint_as_float(ro[2]) * scale, __uint_as_float(ro[3]) * scale);
      w0.z = pack_bf16x2(__uint_as_float(ro[4]) * scale, __uint_as_float(ro[5]) * scale);
      w0.w = pack_bf16x2(__uint_as_float(ro[6]) * scale, __uint_as_float(ro[7]) * scale);
      w1.x = pack_bf16x2(__uint_as_float(ro[8]) * scale, __uint_as_float(ro[9]) * scale);
      w1.y = pack_bf16x2(__uint_as_float(ro[10]) * scale, __uint_as_float(ro[11]) * scale);
      w1.z = pack_bf16x2(__uint_as_float(ro[12]) * scale, __uint_as_float(ro[13]) * scale);
      w1.w = pack_bf16x2(__uint_as_float(ro[14]) * scale, __uint_as_float(ro[15]) * scale);
      if (rv) {
        __stcs(reinterpret_cast<uint4*>(qrow + cc), w0);
        __stcs(reinterpret_cast<uint4*>(qrow + cc + 8), w1);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kGIssueA) {
    tc_fence_after();
    tmem_dealloc(tmem, C::tmem_cols);
    // Started early beside the dK/dV grid: the grid completes only after that
  // one has, so work after this call sees dK and dV written.
  if (blockIdx.x == gridDim.x - 1 && threadIdx.x == 0)
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
}

template <int D>
cudaError_t launch_bwd_impl(const Geom& g, const void* q, const void* k, const void* v,
                            const void* o, const float* lse, const void* dout,
                            const int32_t* row_idx, const int32_t* row_cnt,
                            const int32_t* col_idx, const int32_t* col_cnt, float scale, void* dq,
                            void* dk, void* dv, void* workspace, int32_t* status, cudaStream_t st) {
  const BwdWorkspace ws = bwd_workspace_layout(g, workspace);
  float* delta = ws.delta;
  const long long rows = (long long)g.BH * g.N;
  constexpr int RPB = 256 / (D / 8);
  // D per token, and (two more CTAs) the launch orders of the gradient
  // kernels: longest lists first, kv-blocks by CSC count, q-blocks by CSR count.
  const unsigned ndelta = static_cast<unsigned>((rows + RPB - 1) / RPB);
  bwd_delta_kernel<D><<<ndelta + 2, 256, 0, st>>>(
      static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout), rows, delta,
      ndelta, col_cnt, g.BH * g.Mk, ws.col_order, row_cnt, g.BH * g.Mq, ws.row_order);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  CUtensorMap tq, tk, tv, tdo;
  if (make_tmap_bf16(&tq, q, g.BH, g.N, D, kBM) != 0 || make_tmap_bf16(&tk, k, g.BH, g.N, D, kBN) != 0 ||
      make_tmap_bf16(&tv, v, g.BH, g.N, D, kBN) != 0 ||
      make_tmap_bf16(&tdo, dout, g.BH, g.N, D, kBM) != 0)
    return cudaErrorInvalidValue;
  const float scale_log2 = scale * kLog2e;

  e = cudaFuncSetAttribute(bwd_dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           DkdvCfg<D>::smem_alloc);
  if (e != cudaSuccess) return e;
  bwd_dkdv_kernel<D><<<static_cast<unsigned>((long long)g.BH * g.Mk), kGradThreads,
                       DkdvCfg<D>::smem_alloc, st>>>(
      tq, tk, tv, tdo, lse, delta, col_idx, col_cnt, ws.col_order, g.N, g.Mq, g.Mk, scale,
      scale_log2,
      static_cast<__nv_bfloat16*>(dk), static_cast<__nv_bfloat16*>(dv), status);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  e = cudaFuncSetAttribute(bwd_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           DqCfg<D>::smem_alloc);
  if (e != cudaSuccess) return e;
  // Programmatic dependent launch: the dQ CTAs may start while the last dK/dV
  // CTAs run (D and the launch orders were complete before dK/dV started).
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((long long)g.BH * g.Mq));
  cfg.blockDim = dim3(kGradThreads);
  cfg.dynamicSmemBytes = DqCfg<D>::smem_alloc;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, bwd_dq_kernel<D>, tq, tk, tv, tdo, lse,
                            static_cast<const float*>(delta), row_idx, row_cnt,
                            static_cast<const int32_t*>(ws.row_order), g.N, g.Mq, g.Mk, scale,
                            scale_log2, static_cast<__nv_bfloat16*>(dq), status);
}

}  // namespace

cudaError_t launch_attn_bwd(const Geom& g, const void* q, const void* k, const void* v,
                            const void* o, const float* lse, const void* dout,
                            const int32_t* row_idx, const int32_t* row_cnt,
                            const int32_t* col_idx, const int32_t* col_cnt, float scale, void* dq,
                            void* dk, void* dv, void* workspace, int32_t* status, cudaStream_t st) {
  if (g.d == 128)
    return launch_bwd_impl<128>(g, q, k, v, o, lse, dout, row_idx, row_cnt, col_idx, col_cnt,
                                scale, dq, dk, dv, workspace, status, st);
  return launch_bwd_impl<64>(g, q, k, v, o, lse, dout, row_idx, row_cnt, col_idx, col_cnt, scale,
                             dq, dk, dv, workspace, status, st);
}

namespace {
size_t align256(size_t x) { return (x + 255) / 256 * 256; }
}  // namespace

size_t bwd_workspace_bytes(const Geom& g) {
  return align256((size_t)g.BH * g.N * sizeof(float)) +
         align256((size_t)g.BH * g.Mk * sizeof(int32_t)) +
         align256((size_t)g.BH * g.Mq * sizeof(int32_t));
}

BwdWorkspace bwd_workspace_layout(const Geom& g, void* base) {
  uint8_t* p = static_cast<uint8_t*>(base);
  BwdWorkspace w;
  w.delta = reinterpret_cast<float*>(p);
  p += align256((size_t)g.BH * g.N * sizeof(float));
  w.col_order = reinterpret_cast<int32_t*>(p);
  p += align256((size_t)g.BH * g.Mk * sizeof(int32_t));
  w.row_order = reinterpret_cast<int32_t*>(p);
  return w;
}

}  // namespace sparge
