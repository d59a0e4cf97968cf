// Block-sparse attention forward on sm_103a (tcgen05 + TMEM + TMA).
//
// Method: mindverse page "Optimierung der Effizienz von Video-Diffusionsmodellen
// durch SpargeAttention2", sections "Block-duennbesetzte Aufmerksamkeit" (the
// mask is constant over each tile; a tile is kept whole or dropped whole) and
// "Effiziente Kernel-Implementierung und Modellanpassung" (masked matmuls and
// softmax are skipped).  Each query token's softmax runs over the tokens of
// its q-block's kept kv-blocks only.
//
// One CTA computes one 128-token q-block of one head, looping over its CSR
// list of kept kv-blocks in steps of 64 keys (a 128-key block is two steps);
// two CTAs share an SM so that one CTA's
// latencies (barrier hand-offs, loads, its prologue and epilogue) overlap the
// other's work.  Warp roles (224 threads):
//   warp 4   TMA producer: Q once, then K_j / V_j into a 2-stage K ring and
//            a 3-stage V ring; a K slot is reloaded once S of its tile has
//            completed, a V slot once PV of its tile has.
//   warp 5   S issuer: S_t = Q K_t^T into a double-buffered TMEM tile
//            (128 x 64 fp32).
//   warp 6   PV issuer: O += P_t V_t into a TMEM accumulator (128 x d fp32),
//            with the A operand P_t read from tensor memory.  Separate issuing
//            warps let the S and PV MMAs of neighbouring tiles overlap; each
//            runs its loop as a whole warp and issues every MMA from one
//            elected lane.
//   warps 0-3 softmax: thread r owns query row r (= TMEM lane r).  It reads
//            S_t, masks the ragged kv tail, keeps the running max m and sum l
//            in base 2 and writes P_t (bf16 pairs) over the first 32 columns
//            of S_t's own TMEM tile, where the PV MMA reads it.  Keeping P out
//            of shared memory leaves the shared-memory bandwidth (128 B per
//            clock per SM, which the 128 x 64 x 16 MMAs with both operands in
//            shared memory already use in full) to the operands and loads.
//            O is rescaled in TMEM only when the running max grows by more
//            than 8 (a factor 256); below that the stale max stays exact
//            because l and O share it.  Finally O is scaled by 1/l.
// Every barrier wait is bounded; a timeout records SPARGE_ERR_TIMEOUT.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "common.cuh"
#include "kernels.h"

namespace sparge {

namespace {

constexpr int kBM = 128;           // q-block rows
constexpr int kBN = 64;            // kv-block rows
constexpr int kSoftmaxWarps = 4;
constexpr int kProducerWarp = 4;
constexpr int kSWarp = 5;
constexpr int kPVWarp = 6;
constexpr int kFwdThreads = 224;
constexpr int kFwdCtasPerSm = 2;
constexpr float kRescaleLog2 = 8.0f;

template <int D>
struct FwdCfg {
  // K and V stages of 64 keys.  A K stage is held until S of its step, a V
  // stage until PV.  K tiles were read by the mask's pooling just before and
  // mostly hit L2; V tiles come from DRAM (about 2500 cycles under load), so V
  // gets the deeper ring (measured at 480p: 0.2605 against 0.2656 ms with
  // two stages each).
  static constexpr int NSK = D == 128 ? 2 : 3;
  static constexpr int NSV = D == 128 ? 3 : 4;
  static constexpr int NP = 2;                        // P phases (the S/P TMEM tiles)
  static constexpr int KCH = D / 64;                  // 128-byte chunks per row
  static constexpr uint32_t kQ = kBM * D * 2;
  static constexpr uint32_t kKV = kBN * D * 2;
  static constexpr uint32_t off_q = 0;
  static constexpr uint32_t off_k = off_q + kQ;
  static constexpr uint32_t off_v = off_k + NSK * kKV;
  static constexpr uint32_t off_bar = off_v + NSV * kKV;
  // barriers
  static constexpr int B_Q = 0;
  static constexpr int B_KF = 1;
  static constexpr int B_VF = B_KF + NSK;
  static constexpr int B_KE = B_VF + NSV;   // K slot free (S of its tile done)
  static constexpr int B_VE = B_KE + NSK;   // V slot free (PV of its tile done)
  static constexpr int B_SF = B_VE + NSV;
  static constexpr int B_PF = B_SF + 2;     // count 128 (all softmax threads)
  static constexpr int B_PV = B_PF + NP;
  static constexpr int B_DRAIN = B_PV + 2;  // count 2 (both issuers)
  static constexpr int NBAR = B_DRAIN + 1;
  static constexpr uint32_t off_tmem_slot = off_bar + NBAR * 8;
  static constexpr uint32_t bytes = off_tmem_slot + 16;
  // The dynamic shared-memory window starts 1024-byte aligned on sm_103a
  // (checked at kernel entry), so no alignment pad is allocated: two CTAs
  // with three V stages then fit one SM.
  static constexpr uint32_t smem_alloc = bytes;
  // S0 [0,64) S1 [64,128) O [128,128+D); P_t (bf16 pairs) over the first 32
  // columns of S_(t & 1).
  static constexpr uint32_t tmem_cols = 256;
  static constexpr uint32_t col_s = 0;
  static constexpr uint32_t col_o = 128;
};


template <int D>
__global__ void __launch_bounds__(kFwdThreads, kFwdCtasPerSm)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const int32_t* __restrict__ row_idx,
                    const int32_t* __restrict__ row_cnt, int N, int Mq, int Mk, int bk,
                    float scale_log2,
                    __nv_bfloat16* __restrict__ out, float* __restrict__ lse,
                    int32_t* __restrict__ status) {
  using C = FwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  const uint32_t s0 = smem_u32(sm);
  if ((s0 & 1023u) != 0u) {  // the swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0) report_error(status, SPARGE_ERR_CUDA);
    return;
  }
  auto bar = [&](int i) -> uint32_t { return s0 + C::off_bar + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::off_tmem_slot);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bh = blockIdx.x / Mq;
  const int qb = blockIdx.x % Mq;
  const long long row_id = (long long)bh * Mq + qb;
  const int nkv = min(max(__ldg(row_cnt + row_id), 0), Mk);
  const int32_t* list = row_idx + row_id * Mk;
  // Steps of 64 keys: one per kept block of 64 keys, two per kept block of
  // 128 (its halves).  First key row of step t:
  // bk is 64 or 128 (checked by the host), so a step index splits by a shift.
  const int sub_shift = bk > kBN ? 1 : 0;
  const int n = nkv << sub_shift;
  auto row_of = [&](int t) -> int {
    return min(max(__ldg(list + (t >> sub_shift)), 0), Mk - 1) * bk +
           (t & sub_shift) * kBN;
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NBAR; ++i) {
      uint32_t cnt = 1;
      if (i >= C::B_PF && i < C::B_PF + C::NP) cnt = 32 * kSoftmaxWarps;
      if (i == C::B_DRAIN) cnt = 2;
      mbar_init(bar(i), cnt);
    }
    fence_barrier_init();
  }
  if (warp == kSWarp) {
    tmem_alloc(smem_u32(tmem_slot), C::tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n > 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      mbar_arrive_expect_tx(bar(C::B_Q), C::kQ);
      for (int c = 0; c < C::KCH; ++c)
        tma_load_3d(s0 + C::off_q + c * kBM * 128, &tmQ, bar(C::B_Q), c * 64, qb * kBM, bh);
      int issued = 0;
      for (int t = 0; t < n; ++t) {
        const int sk = t % C::NSK, sv = t % C::NSV;
        if (t >= C::NSK && !mbar_wait(bar(C::B_KE + sk), ((t / C::NSK) - 1) & 1, kWaitTimeoutNs)) {
          report_error(status, SPARGE_ERR_TIMEOUT);
          break;
        }
        const int rw = row_of(t);
        mbar_arrive_expect_tx(bar(C::B_KF + sk), C::kKV);
        for (int c = 0; c < C::KCH; ++c)
          tma_load_3d(s0 + C::off_k + sk * C::kKV + c * kBN * 128, &tmK, bar(C::B_KF + sk), c * 64,
                      rw, bh);
        if (t >= C::NSV && !mbar_wait(bar(C::B_VE + sv), ((t / C::NSV) - 1) & 1, kWaitTimeoutNs)) {
          report_error(status, SPARGE_ERR_TIMEOUT);
          break;
        }
        mbar_arrive_expect_tx(bar(C::B_VF + sv), C::kKV);
        for (int c = 0; c < C::KCH; ++c)
          tma_load_3d(s0 + C::off_v + sv * C::kKV + c * kBN * 128, &tmV, bar(C::B_VF + sv), c * 64,
                      rw, bh);
        issued = t + 1;
      }
      // Let the last loads land before the CTA can exit (they complete on their own).
      for (int t = max(0, issued - C::NSK); t < issued; ++t)
        mbar_wait(bar(C::B_KF + t % C::NSK), (t / C::NSK) & 1, kWaitTimeoutNs);
      for (int t = max(0, issued - C::NSV); t < issued; ++t)
        mbar_wait(bar(C::B_VF + t % C::NSV), (t / C::NSV) & 1, kWaitTimeoutNs);
    }
  } else if (warp == kSWarp) {
    // ------------------------------------------------------------ S issuer
    // The whole warp runs the loop; one elected lane issues each MMA.
    if (n > 0) {
      constexpr uint32_t idS = idesc_bf16(kBM, kBN, false, false);
      const uint64_t dq0 = sdesc_sw128(s0 + C::off_q, 16, 1024);
      const uint64_t dk0 = sdesc_sw128(s0 + C::off_k, 16, 1024);
      bool ok = warp_wait(bar(C::B_Q), 0);
      for (int t = 0; ok && t < n; ++t) {
        const int s = t % C::NSK;
        // TMEM tile t & 1 holds P(t - 2) until PV(t - 2) has completed.
        if (!warp_wait(bar(C::B_KF + s), (t / C::NSK) & 1) ||
            (t >= 2 && !warp_wait(bar(C::B_PV + (t & 1)), ((t - 2) >> 1) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t dk = sdesc_add(dk0, s * C::kKV);
        const uint32_t dS = tmem + C::col_s + (t & 1) * kBN;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk & 3) * 32;
          warp_mma_bf16(dS, sdesc_add(dq0, (kk >> 2) * (kBM * 128) + koff),
                        sdesc_add(dk, (kk >> 2) * (kBN * 128) + koff), idS, kk > 0);
        }
        warp_commit(bar(C::B_SF + (t & 1)));
        warp_commit(bar(C::B_KE + s));
      }
      if (!ok && lane == 0) report_error(status, SPARGE_ERR_TIMEOUT);
      // Drain: every MMA this warp issued has completed once this arrives.
      warp_commit(bar(C::B_DRAIN));
      warp_wait(bar(C::B_DRAIN), 0);
    }
  } else if (warp == kPVWarp) {
    // ------------------------------------------------------------ PV issuer
    if (n > 0) {
      constexpr uint32_t idO = idesc_bf16(kBM, D, false, true);
      bool ok = true;
      for (int u = 0; ok && u < n; ++u) {
        const int su = u % C::NSV;
        if (!warp_wait(bar(C::B_PF + (u % C::NP)), (u / C::NP) & 1) ||
            !warp_wait(bar(C::B_VF + su), (u / C::NSV) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t ap = tmem + C::col_s + (u & 1) * kBN;
        const uint64_t dv = sdesc_sw128(s0 + C::off_v + su * C::kKV, kBN * 128, 1024);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          warp_mma_bf16_ta(tmem + C::col_o, ap + kk * 8, sdesc_add(dv, kk * 16 * 128), idO,
                           (u > 0 || kk > 0) ? 1u : 0u);
        warp_commit(bar(C::B_VE + su));
        warp_commit(bar(C::B_PV + (u & 1)));
      }
      if (!ok && lane == 0) report_error(status, SPARGE_ERR_TIMEOUT);
      warp_commit(bar(C::B_DRAIN));
      warp_wait(bar(C::B_DRAIN), 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int r = threadIdx.x;  // 0..127 == TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const int row = qb * kBM + r;
    float m_used = -INFINITY;
    float l = 0.f;
    bool ok = true;
    // Scores are kept raw; the scale folds into one FFMA before the exp.  The
    // row max is taken on raw scores (the min when the scale is negative).
    const bool pos = scale_log2 > 0.f;
    const float masked = pos ? -INFINITY : INFINITY;
    // The kv-block index of the next tile is loaded one tile ahead.
    int rw_next = n > 0 ? row_of(0) : 0;
    for (int t = 0; t < n; ++t) {
      const int rw = rw_next;
      if (t + 1 < n) rw_next = row_of(t + 1);
      if (!warp_wait(bar(C::B_SF + (t & 1)), (t >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float x[kBN];
      {
        uint32_t ra[16], rb[16], rc[16], rd[16];
        const uint32_t sa = lane_base + C::col_s + (t & 1) * kBN;
        SPARGE_TMEM_LD_X16(sa + 0, ra);
        SPARGE_TMEM_LD_X16(sa + 16, rb);
        SPARGE_TMEM_LD_X16(sa + 32, rc);
        SPARGE_TMEM_LD_X16(sa + 48, rd);
        SPARGE_TMEM_WAIT_LD16(ra);
        SPARGE_TMEM_WAIT_LD16(rb);
        SPARGE_TMEM_WAIT_LD16(rc);
        SPARGE_TMEM_WAIT_LD16(rd);
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          x[c] = __uint_as_float(ra[c]);
          x[16 + c] = __uint_as_float(rb[c]);
          x[32 + c] = __uint_as_float(rc[c]);
          x[48 + c] = __uint_as_float(rd[c]);
        }
      }
      const int valid = N - rw;
      if (valid < kBN) {
#pragma unroll
        for (int c = 0; c < kBN; ++c)
          if (c >= valid) x[c] = masked;
      }
      // Row max as a tree over 8 independent partial maxima, two new
      // columns per three-input max.
      float mp[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) mp[e] = x[e];
      if (pos) {
#pragma unroll
        for (int c = 8; c < 56; c += 16)
#pragma unroll
          for (int e = 0; e < 8; ++e) mp[e] = fmax3(mp[e], x[c + e], x[c + 8 + e]);
#pragma unroll
        for (int e = 0; e < 8; ++e) mp[e] = fmaxf(mp[e], x[56 + e]);
        mp[0] = fmax3(fmax3(mp[0], mp[1], mp[2]), fmax3(mp[3], mp[4], mp[5]), fmaxf(mp[6], mp[7]));
      } else {
#pragma unroll
        for (int c = 8; c < 56; c += 16)
#pragma unroll
          for (int e = 0; e < 8; ++e) mp[e] = fmin3(mp[e], x[c + e], x[c + 8 + e]);
#pragma unroll
        for (int e = 0; e < 8; ++e) mp[e] = fminf(mp[e], x[56 + e]);
        mp[0] = fmin3(fmin3(mp[0], mp[1], mp[2]), fmin3(mp[3], mp[4], mp[5]), fminf(mp[6], mp[7]));
      }
      const float mt = mp[0] * scale_log2;
      const float m_new = fmaxf(m_used, mt);
      // Rescale decision must be warp-uniform (tcgen05.ld/st are warp-wide).
      const bool want = (t > 0) && (m_new - m_used > kRescaleLog2);
      if (t == 0) m_used = m_new;
      if (__any_sync(0xffffffffu, want)) {
        // O holds every PV up to t-1 once that commit has arrived.
        if (!warp_wait(bar(C::B_PV + ((t - 1) & 1)), ((t - 1) >> 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float alpha = want ? exp2f(m_used - m_new) : 1.f;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 16) {
          uint32_t ro[16];
          SPARGE_TMEM_LD_X16(lane_base + C::col_o + c0, ro);
          SPARGE_TMEM_WAIT_LD16(ro);
#pragma unroll
          for (int c = 0; c < 16; ++c) ro[c] = __float_as_uint(__uint_as_float(ro[c]) * alpha);
          SPARGE_TMEM_ST_X16(lane_base + C::col_o + c0, ro);
        }
        tmem_st_wait();
        if (want) {
          l *= alpha;
          m_used = m_new;
        }
      }
      // P_t over the first 32 columns of S_t's tile (this thread's S_t row
      // is already in registers).
      // Eight partial row sums held as four packed pairs; the exponent
      // arguments two columns per packed FMA.
      const uint64_t sl2 = f32x2(scale_log2, scale_log2);
      const uint64_t nm2 = f32x2(-m_used, -m_used);
      uint64_t rs2[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) rs2[e] = f32x2(0.f, 0.f);
      uint32_t pk[32];
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint64_t a = ffma2(f32x2(x[ch * 8 + 2 * e], x[ch * 8 + 2 * e + 1]), sl2, nm2);
          const float p0 = ex2_approx(f32x2_lo(a)), p1 = ex2_approx(f32x2_hi(a));
          rs2[e] = fadd2(rs2[e], f32x2(p0, p1));
          pk[ch * 4 + e] = pack_bf16x2(p0, p1);
        }
      }
      l += ((f32x2_lo(rs2[0]) + f32x2_hi(rs2[0])) + (f32x2_lo(rs2[1]) + f32x2_hi(rs2[1]))) +
           ((f32x2_lo(rs2[2]) + f32x2_hi(rs2[2])) + (f32x2_lo(rs2[3]) + f32x2_hi(rs2[3])));
      {
        const uint32_t pa = lane_base + C::col_s + (t & 1) * kBN;
        SPARGE_TMEM_ST_X16(pa, pk);
        SPARGE_TMEM_ST_X16(pa + 16, (pk + 16));
        tmem_st_wait();
      }
      tc_fence_before();
      mbar_arrive(bar(C::B_PF + (t % C::NP)));
    }
    if (!ok) report_error(status, SPARGE_ERR_TIMEOUT);
    // ---------------------------------------------------------- epilogue
    const bool have = ok && n > 0 && warp_wait(bar(C::B_PV + ((n - 1) & 1)), ((n - 1) >> 1) & 1);
    if (ok && n > 0 && !have) report_error(status, SPARGE_ERR_TIMEOUT);
    tc_fence_after();
    const bool good = have && l > 0.f;
    const float inv_l = good ? 1.f / l : 0.f;
    __nv_bfloat16* orow = out + ((long long)bh * N + row) * D;
    const bool in_range = row < N;
#pragma unroll 1
    for (int c0 = 0; c0 < D; c0 += 16) {
      uint32_t ro[16];
      if (have) {
        SPARGE_TMEM_LD_X16(lane_base + C::col_o + c0, ro);
        SPARGE_TMEM_WAIT_LD16(ro);
      } else {
#pragma unroll
        for (int c = 0; c < 16; ++c) ro[c] = 0u;
      }
      uint4 w0, w1;
      w0.x = pack_bf16x2(__uint_as_float(ro[0]) * inv_l, __uint_as_float(ro[1]) * inv_l);
      w0.y = pack_bf16x2(__uint_as_float(ro[2]) * inv_l, __uint_as_float(ro[3]) * inv_l);
      w0.z = pack_bf16x2(__uint_as_float(ro[4]) * inv_l, __uint_as_float(ro[5]) * inv_l);
      w0.w = pack_bf16x2(__uint_as_float(ro[6]) * inv_l, __uint_as_float(ro[7]) * inv_l);
      w1.x = pack_bf16x2(__uint_as_float(ro[8]) * inv_l, __uint_as_float(ro[9]) * inv_l);
      w1.y = pack_bf16x2(__uint_as_float(ro[10]) * inv_l, __uint_as_float(ro[11]) * inv_l);
      w1.z = pack_bf16x2(__uint_as_float(ro[12]) * inv_l, __uint_as_float(ro[13]) * inv_l);
      w1.w = pack_bf16x2(__uint_as_float(ro[14]) * inv_l, __uint_as_float(ro[15]) * inv_l);
      if (in_range) {
        *reinterpret_cast<uint4*>(orow + c0) = w0;
        *reinterpret_cast<uint4*>(orow + c0 + 8) = w1;
      }
    }
    if (lse != nullptr && in_range)
      lse[(long long)bh * N + row] =
          good ? (m_used + log2f(l)) * 0.69314718055994530942f : -INFINITY;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kSWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::tmem_cols);
  }
}

template <int D>
cudaError_t launch_fwd_impl(const Geom& g, const void* q, const void* k, const void* v,
                            const int32_t* row_idx, const int32_t* row_cnt, float scale, void* o,
                            float* lse, int32_t* status, cudaStream_t st) {
  using C = FwdCfg<D>;
  CUtensorMap tq, tk, tv;
  if (make_tmap_bf16(&tq, q, g.BH, g.N, D, kBM) != 0 || make_tmap_bf16(&tk, k, g.BH, g.N, D, kBN) != 0 ||
      make_tmap_bf16(&tv, v, g.BH, g.N, D, kBN) != 0)
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::smem_alloc);
  if (e != cudaSuccess) return e;
  const float scale_log2 = scale * 1.4426950408889634f;
  const unsigned grid = static_cast<unsigned>((long long)g.BH * g.Mq);
  attn_fwd_kernel<D><<<grid, kFwdThreads, C::smem_alloc, st>>>(
      tq, tk, tv, row_idx, row_cnt, g.N, g.Mq, g.Mk, g.bk, scale_log2,
      static_cast<__nv_bfloat16*>(o), lse, status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_fwd(const Geom& g, const void* q, const void* k, const void* v,
                            const int32_t* row_idx, const int32_t* row_cnt, float scale, void* o,
                            float* lse, int32_t* status, cudaStream_t st) {
  if (g.d == 128) return launch_fwd_impl<128>(g, q, k, v, row_idx, row_cnt, scale, o, lse, status, st);
  return launch_fwd_impl<64>(g, q, k, v, row_idx, row_cnt, scale, o, lse, status, st);
}

}  // namespace sparge
