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
// Kernels, deterministic (no atomics touch a gradient; each gradient element
// is summed in a fixed order):
//   bwd_plan_kernel   two CTAs: the work orders of the gradient kernels (long
//                     work lists first, then the rest in descending index
//                     order), the key tiles with far more than an SM's share
//                     of the work cut into parts, the counters zeroed.
//   bwd_delta_kernel  D per token (HBM-bound, 16-byte loads), launched beside
//                     the plan grid by programmatic dependent launch.
//   bwd_dkdv_kernel   persistent, one CTA per SM taking key tiles of 128 keys
//                     (a pair of adjacent 64-key kv-blocks, or one 128-key
//                     block), or parts of them, from a work counter.  A part
//                     covers a range of q-blocks and leaves fp32 partial dK,
//                     dV; the last part to finish adds them in part order.  The keys are the M = 128
//                     rows of every MMA: S^T = K Q^T and dP^T = V dO^T land in
//                     TMEM with a key per lane, the compute warps turn them
//                     into P^T and dS^T in place (bf16), and those are the A
//                     operands, read from TMEM, of dV += P^T dO and
//                     dK += dS^T Q.  The CTA walks the union of the two
//                     blocks' column lists; a q-block that keeps only one of
//                     the two gets zero P and dS in the other block's rows.
//                     Each q-block is processed as two halves of 64 queries,
//                     so that the S/dP tiles of one half are computed while
//                     the compute warps work on the other half and its
//                     gradients run.
//   bwd_dq_kernel     persistent, one CTA per SM taking q-blocks from a second
//                     counter; a q-block's kept kv-blocks are taken two at a
//                     time (N = 128 keys per MMA): S = Q K^T (double-buffered
//                     in TMEM) and dP = dO V^T with Q and dO in shared memory,
//                     dS written in place over S (bf16), dQ += dS K
//                     accumulated in TMEM.  Launched with programmatic
//                     dependent launch beside the dK/dV grid's last tiles.
// Every MMA is M = 128 with N >= 64 (the 64-query halves of the dK/dV kernel)
// or N = 128, issued from a converged warp (one elected lane per MMA).  Roles
// per CTA: compute warps, a TMA producer warp and two MMA-issuing warps.
// Every wait is bounded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "common.cuh"
#include "kernels.h"

namespace sparge {

namespace {

constexpr int kBM = 128;    // q-block rows
constexpr int kBN = 64;     // rows of one TMA box of K / V (a 64-key kv-block)
constexpr int kPair = 128;  // keys per gradient tile (two 64-key boxes)
constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------- work order
// The planning passes below walk each thread's contiguous range in chunks of
// kChunk items whose loads are issued together: one memory latency per chunk
// rather than per item, so the plan stays shorter than the D pass it runs
// beside.
constexpr int kChunk = 8;

// Exclusive prefix sum over the NT threads of a CTA; *total gets the sum.
template <int NT, typename T>
__device__ T block_exclusive_scan(T v, T* total) {
  constexpr int W = NT / 32;
  __shared__ T wsum[W];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  T incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) wsum[w] = incl;
  __syncthreads();
  T before = 0, all = 0;
#pragma unroll
  for (int i = 0; i < W; ++i) {
    before += i < w ? wsum[i] : 0;
    all += wsum[i];
  }
  __syncthreads();  // wsum may be reused by the next call
  *total = all;
  return before + incl - v;
}

// Work order of the gradient kernels: the items whose work is longer than twice
// the mean first, in index order, then the others in descending index order.
// Long lists (attention-sink blocks that nearly every q-block keeps) would
// otherwise run alone at the end of the grid; index order keeps the items of
// one head together, so that head's tiles are served from L2; descending
// order starts the rest on the last heads, whose dO (read by the delta pass)
// and K/V (read by the dK/dV kernel's last tiles) are still in L2 (measured
// at 480p: 1.060 against 1.067 ms per backward).
// One CTA of NT threads partitions the n items; work[it] is an item's size
// (plain loads: the array may have been written by this CTA), and
// place(pos, load(it)) records item `it` at launch position pos.
template <int NT, typename Load, typename Place>
__device__ void order_by_work(int n, const int32_t* work, Load load, Place place) {
  const int tid = threadIdx.x;
  const int E = (n + NT - 1) / NT;
  const int lo = min(n, tid * E), hi = min(n, lo + E);
  long long sum = 0;
  for (int i0 = lo; i0 < hi; i0 += kChunk) {
    int w[kChunk];
#pragma unroll
    for (int u = 0; u < kChunk; ++u) w[u] = i0 + u < hi ? max(work[i0 + u], 0) : 0;
#pragma unroll
    for (int u = 0; u < kChunk; ++u) sum += w[u];
  }
  long long total = 0;
  block_exclusive_scan<NT>(sum, &total);
  // Item `it` is long when work * n > 2 * total.
  int nl = 0;
  for (int i0 = lo; i0 < hi; i0 += kChunk) {
    int w[kChunk];
#pragma unroll
    for (int u = 0; u < kChunk; ++u) w[u] = i0 + u < hi ? max(work[i0 + u], 0) : 0;
#pragma unroll
    for (int u = 0; u < kChunk; ++u) nl += (long long)w[u] * n > 2 * total ? 1 : 0;
  }
  int n_long = 0;
  const int before_long = block_exclusive_scan<NT>(nl, &n_long);
  int pl = before_long;                // next long position
  int ps = n_long + lo - before_long;  // next short position
  for (int i0 = lo; i0 < hi; i0 += kChunk) {
    int w[kChunk];
    decltype(load(0)) v[kChunk];
#pragma unroll
    for (int u = 0; u < kChunk; ++u) {
      w[u] = i0 + u < hi ? max(work[i0 + u], 0) : 0;
      v[u] = load(min(i0 + u, hi - 1));
    }
#pragma unroll
    for (int u = 0; u < kChunk; ++u) {
      if (i0 + u >= hi) break;
      if ((long long)w[u] * n > 2 * total) place(pl++, v[u]);
      else place(n - 1 - (ps++ - n_long), v[u]);  // short items, descending
    }
  }
}

// The dK/dV kernel's work items in the workspace (see plan_tiles).
struct TileItems {
  int32_t* tile;       // key tile of each item, in tile order
  int32_t* part;       // p | P << 8 | first partial slot << 16
  int32_t* work;       // work of each item
  int32_t* seq_tile;   // the items' key tiles in launch order
  int32_t* seq_part;   // and their part words
  int32_t* n_items;    // item count
  int32_t* split_cnt;  // completion counters of the cut tiles
  float* split_part;   // fp32 partial dV | dK, [slot][128 keys][2][d]
};

// Work items of the dK/dV kernel.  A key tile whose work (the summed length
// of its column lists) is more than an SM's share of the whole, and more
// than kMinPartWork, is cut into P <= kMaxParts parts by q-block range: part
// p takes the q-blocks [Mq p / P, Mq (p + 1) / P) of both lists.  Each part
// runs as its own item and leaves fp32 partial dK, dV in a workspace slot;
// the last part to finish adds the P partials in part order and writes the
// gradients, so the result does not depend on which CTA ran which part.
// Without the cut, one such tile (an attention-sink block that every q-block
// keeps) sets the kernel's length when there are few heads (measured at the
// 480p shape with one head: 0.167 against 0.296 ms per backward).  Parts need
// partial slots; a tile whose slots would pass max_slots stays whole.
// Writes the items in tile order, then in launch order (long items first,
// order_by_work), the item count and zeroed completion counters.
constexpr int kMaxParts = 16;
constexpr int kMinPartWork = 48;
constexpr int kSplitSlots = 128;
constexpr int kSplitCounters = kSplitSlots * 8;  // one per slot and compute warp

template <int NT>
__device__ void plan_tiles(const int32_t* __restrict__ col_cnt, int BH, int Mk, int Mt,
                           int kv_per_tile, int nsm, int Mq, int max_slots, const TileItems& it) {
  const int tid = threadIdx.x;
  for (int i = tid; i < kSplitCounters; i += NT) it.split_cnt[i] = 0;
  const int ntiles = BH * Mt;
  const int E = (ntiles + NT - 1) / NT;
  const int lo = min(ntiles, tid * E), hi = min(ntiles, lo + E);
  // Each tile's work, kept meanwhile in the launch-order tile array (written
  // last), and the items as they are when no tile is cut.
  int32_t* tile_work = it.seq_tile;
  long long sum = 0;
  int wmax = 0;
  for (int t0 = lo; t0 < hi; t0 += kChunk) {
    int w[kChunk];
#pragma unroll
    for (int u = 0; u < kChunk; ++u) {
      const int t = t0 + u;
      int x = 0;
      if (t < hi) {
        const int bh = t / Mt, j0 = (t % Mt) * kv_per_tile;
        const int32_t* c = col_cnt + (long long)bh * Mk + j0;
        x = max(__ldg(c), 0);
        if (kv_per_tile == 2 && j0 + 1 < Mk) x += max(__ldg(c + 1), 0);
      }
      w[u] = x;
    }
#pragma unroll
    for (int u = 0; u < kChunk; ++u) {
      if (t0 + u >= hi) break;
      tile_work[t0 + u] = w[u];
      it.tile[t0 + u] = t0 + u;
      it.part[t0 + u] = 1 << 8;
      it.work[t0 + u] = w[u];
      sum += w[u];
      wmax = max(wmax, w[u]);
    }
  }
  long long total = 0;
  block_exclusive_scan<NT>(sum, &total);
  const long long L = max((long long)kMinPartWork, (total + nsm - 1) / max(nsm, 1));
  if (!__syncthreads_or(wmax > L)) {
    // No tile is cut (every tile within an SM's share: the usual case with
    // many heads); the items are the tiles.
    if (tid == 0) *it.n_items = ntiles;
    order_by_work<NT>(
        ntiles, it.work, [&](int i) { return make_int2(it.tile[i], it.part[i]); },
        [&](int p, int2 v) {
          it.seq_tile[p] = v.x;
          it.seq_part[p] = v.y;
        });
    return;
  }
  auto parts = [&](int w) -> int {
    return w > L ? (int)min((long long)min(kMaxParts, Mq), (w + L - 1) / L) : 1;
  };
  // This thread's tile work, kChunk tiles at a time.
  auto load_work = [&](int t0, int (&w)[kChunk]) {
#pragma unroll
    for (int u = 0; u < kChunk; ++u) w[u] = t0 + u < hi ? tile_work[t0 + u] : 0;
  };
  // Slots requested, then items, each as a prefix over the tiles.
  int req = 0;
  for (int t0 = lo; t0 < hi; t0 += kChunk) {
    int w[kChunk];
    load_work(t0, w);
#pragma unroll
    for (int u = 0; u < kChunk; ++u) {
      const int P = parts(w[u]);
      req += P > 1 ? P : 0;
    }
  }
  int unused = 0;
  const int slot0 = block_exclusive_scan<NT>(req, &unused);
  // Parts of tile t0 + u with its slots (P = 1 where they would not fit).
  auto plan_chunk = [&](int t0, const int (&w)[kChunk], int& slot, int (&P)[kChunk],
                        int (&base)[kChunk]) {
#pragma unroll
    for (int u = 0; u < kChunk; ++u) {
      P[u] = t0 + u < hi ? parts(w[u]) : 0;
      base[u] = 0;
      if (P[u] > 1) {
        const bool fits = slot + P[u] <= max_slots;
        base[u] = slot;
        slot += P[u];
        if (!fits) P[u] = 1, base[u] = 0;
      }
    }
  };
  int nit = 0;
  for (int t0 = lo, slot = slot0; t0 < hi; t0 += kChunk) {
    int w[kChunk], P[kChunk], base[kChunk];
    load_work(t0, w);
    plan_chunk(t0, w, slot, P, base);
#pragma unroll
    for (int u = 0; u < kChunk; ++u) nit += P[u];
  }
  int n = 0;
  int pos = block_exclusive_scan<NT>(nit, &n);
  for (int t0 = lo, slot = slot0; t0 < hi; t0 += kChunk) {
    int w[kChunk], P[kChunk], base[kChunk];
    load_work(t0, w);
    plan_chunk(t0, w, slot, P, base);
#pragma unroll
    for (int u = 0; u < kChunk; ++u) {
      for (int p = 0; p < P[u]; ++p, ++pos) {
        it.tile[pos] = t0 + u;
        it.part[pos] = p | (P[u] << 8) | (base[u] << 16);
        it.work[pos] = (w[u] + P[u] - 1) / P[u];
      }
    }
  }
  if (tid == 0) *it.n_items = n;
  __syncthreads();  // the items are read back by other threads below
  order_by_work<NT>(
      n, it.work, [&](int i) { return make_int2(it.tile[i], it.part[i]); },
      [&](int p, int2 v) {
        it.seq_tile[p] = v.x;
        it.seq_part[p] = v.y;
      });
}

// ---------------------------------------------------------------- plan
// Two CTAs: the first plans the dK/dV work items (key tiles by the summed
// length of their column lists, the longest cut into parts), the second
// orders the q-blocks by row count and zeroes the work counters.  The D pass
// is launched as its programmatic dependent and streams beside them; its last
// CTA waits for this grid before it exits, so the gradient kernels, launched
// after the D pass, see the plan.  In a grid of its own the plan has the
// registers and threads it needs without taking either from the stream
// (measured with the plan in two extra CTAs of the D pass: 39 against 32 us
// per pass at d = 64 and 24 heads, where 6144 key tiles are planned).
// `kv_per_tile` is 2 when a key tile is a pair of 64-key kv-blocks.
constexpr int kPlanThreads = 1024;
__global__ void __launch_bounds__(kPlanThreads, 1) bwd_plan_kernel(
    const int32_t* __restrict__ col_cnt, int BH, int Mk, int Mt, int kv_per_tile,
    const TileItems items, int nsm, int Mq, int max_slots, const int32_t* __restrict__ row_cnt,
    int nrow, int32_t* __restrict__ row_order, int32_t* __restrict__ work) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (blockIdx.x == 0) {
    plan_tiles<kPlanThreads>(col_cnt, BH, Mk, Mt, kv_per_tile, nsm, Mq, max_slots, items);
  } else {
    // The work counters of the persistent gradient kernels start at zero.
    if (threadIdx.x < 2) work[threadIdx.x] = 0;
    order_by_work<kPlanThreads>(
        nrow, row_cnt, [](int i) { return i; }, [&](int p, int i) { row_order[p] = i; });
  }
}

// ---------------------------------------------------------------- D = rowsum(dO * O)
// One 16-thread segment per row, 16-byte streaming loads; launched beside the
// plan grid (above), for which its last CTA waits before exiting.
template <int D>
__global__ void __launch_bounds__(256) bwd_delta_kernel(const __nv_bfloat16* __restrict__ o,
                                                        const __nv_bfloat16* __restrict__ dout,
                                                        long long rows,
                                                        float* __restrict__ delta) {
  constexpr int CH = D / 8;        // 16-byte chunks per row
  constexpr int RPB = 256 / CH;    // rows per block pass
  const long long r = (long long)blockIdx.x * RPB + threadIdx.x / CH;
  const int c = threadIdx.x % CH;
  float s = 0.f;
  if (r < rows) {
    const uint4 a = ldg_no_l1(reinterpret_cast<const uint4*>(o + r * D) + c);
    const uint4 b = ldg_no_l1(reinterpret_cast<const uint4*>(dout + r * D) + c);
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
  if (blockIdx.x == gridDim.x - 1 && threadIdx.x == 0)
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Loads 32 consecutive fp32 TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld32u(uint32_t addr, uint32_t (&a)[16], uint32_t (&b)[16]) {
  SPARGE_TMEM_LD_X16(addr, a);
  SPARGE_TMEM_LD_X16(addr + 16, b);
  SPARGE_TMEM_WAIT_LD16(a);
  SPARGE_TMEM_WAIT_LD16(b);
}

// Warp roles of the gradient kernels: CW compute warps (CW / 4 per TMEM lane
// quarter), then a TMA producer warp, a warp issuing the S and dP MMAs and a
// warp issuing the gradient MMAs.  The dQ kernel runs sixteen compute warps
// (four per SM sub-partition, to hide the tensor-memory and exponential
// latencies of its short per-thread rows); the dK/dV kernel eight, in two
// groups of four that take the two 64-query halves of an entry (measured:
// sixteen warps were slower).
template <int CW>
struct Roles {
  static constexpr int kCompute = CW;
  static constexpr int kThreads = (CW + 3) * 32;
  static constexpr int kProducer = CW;
  static constexpr int kIssueA = CW + 1;
  static constexpr int kIssueB = CW + 2;
};
constexpr int kDkdvWarps = 8;
constexpr int kDqWarps = 16;
static_assert(kSplitCounters == kSplitSlots * kDkdvWarps, "one counter per slot and compute warp");

// ---------------------------------------------------------------- dK, dV
template <int D>
struct DkdvCfg {
  // Q and dO arrive per 64-query half of a q-block: a slot holds Q_h and dO_h
  // (64 rows each) and is released once the gradient MMAs of that half are done.
  static constexpr int NSLOT = D == 128 ? 5 : 8;
  static constexpr int NRING = 4;                    // key tiles handed out ahead
  static constexpr uint32_t kKP = kPair * D * 2;     // K (or V) of the 128 keys
  static constexpr uint32_t kQh = 64 * D * 2;        // one Q (or dO) half tile
  static constexpr uint32_t kChunkK = kPair * 128;   // 64-column chunk of the key tile
  static constexpr uint32_t kChunkH = 64 * 128;      // 64-column chunk of a half tile
  static constexpr uint32_t off_k = 0;
  static constexpr uint32_t off_v = off_k + kKP;
  static constexpr uint32_t off_q = off_v + kKP;               // NSLOT Q halves
  static constexpr uint32_t off_do = off_q + NSLOT * kQh;      // NSLOT dO halves
  static constexpr uint32_t off_row = off_do + NSLOT * kQh;    // NSLOT x {-lse*log2e [64], -D [64]}
  static constexpr uint32_t off_info = off_row + NSLOT * 2 * 64 * 4;  // NSLOT x int32
  static constexpr uint32_t off_ring = off_info + 64;          // NRING x {tile, entries}
  static constexpr uint32_t off_bar = off_ring + 64;
  static constexpr int B_KV = 0;              // K/V of a key tile landed
  static constexpr int B_KVE = 1;             // its S^T and dP^T MMAs done: K/V slots free
  static constexpr int B_QF = 2;              // NSLOT, count 32 (producer lanes) + tx
  static constexpr int B_QE = B_QF + NSLOT;   // NSLOT: the half's gradient MMAs done
  // Per query half h, S^T and dP^T are tracked separately, so that P^T and
  // dV of a half proceed while dP^T and dS^T of it are still in flight.
  static constexpr int B_SSF = B_QE + NSLOT;  // 2: S^T_h in TMEM
  static constexpr int B_DPF = B_SSF + 2;     // 2: dP^T_h in TMEM
  static constexpr int B_PPF = B_DPF + 2;     // 2, half h's compute group: P^T_h written
  static constexpr int B_DSF = B_PPF + 2;     // 2, half h's compute group: dS^T_h written
  static constexpr int B_RVF = B_DSF + 2;     // 2: dV MMAs of half h done (S^T_h region free)
  static constexpr int B_RKF = B_RVF + 2;     // 2: dK MMAs of half h done (dP^T_h region free)
  static constexpr int B_DKE = B_RKF + 2;     // all compute threads: dV, dK read out
  static constexpr int B_IF = B_DKE + 1;      // NRING: key tile handed out
  static constexpr int B_IE = B_IF + NRING;   // NRING: read by both issuers and every compute warp
  static constexpr int B_DONE = B_IE + NRING; // count 2
  static constexpr int NBAR = B_DONE + 1;
  static constexpr uint32_t off_slot = off_bar + NBAR * 8;
  static constexpr uint32_t bytes = off_slot + 16;
  // The dynamic shared-memory window starts 1024-byte aligned on sm_103a
  // (checked at kernel entry), so no alignment pad is allocated: five Q/dO
  // slots at d = 128 then fit.
  static constexpr uint32_t smem_alloc = bytes;
  // TMEM: half h of the queries uses columns [128h, 128h + 128): S^T_h at
  // +0 (64 fp32 columns) and dP^T_h at +64.  P^T_h is written over S^T_h as
  // bf16 pairs in chunks of 32 queries: chunk c (queries 32c .. 32c + 31)
  // goes to columns 32c .. 32c + 15, over columns it had read; dS^T_h
  // likewise over dP^T_h.  dV at 256, dK at 256 + 128.
  static constexpr uint32_t tmem_cols = 512;
  static constexpr uint32_t col_dv = 256;
  static constexpr uint32_t col_dk = 384;
};

// Persistent: one CTA per SM takes work items (key tiles, or parts of cut
// tiles; plan_tiles) from a work counter in the launch order (long column
// lists first).  A key tile is 128 keys: the 64-key
// kv-blocks j0 = 2 * jt and j1 = 2 * jt + 1 (kv_per_tile = 2), or the one
// 128-key block jt (kv_per_tile = 1; then both 64-row halves belong to it).
// The entries of successive tiles share one running entry count t, which
// indexes the Q/dO slot ring and the barrier phases; the next tile's K/V
// load, S^T and P^T overlap the current tile's last entries and epilogue.
template <int D>
__global__ void __launch_bounds__(Roles<kDkdvWarps>::kThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                    const float* __restrict__ lse, const float* __restrict__ delta,
                    const int32_t* __restrict__ col_idx, const int32_t* __restrict__ col_cnt,
                    const TileItems items, int ntiles, int32_t* __restrict__ work,
                    int N, int Mq, int Mk, int Mt, int kv_per_tile, float scale, float scale_log2,
                    __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv,
                    int32_t* __restrict__ status) {
  using C = DkdvCfg<D>;
  using R = Roles<kDkdvWarps>;
  // The dQ kernel (independent of this one) may start on SMs this grid's
  // last CTAs leave idle.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  const uint32_t s0 = smem_u32(sm);
  if ((s0 & 1023u) != 0u) {  // the swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0) report_error(status, SPARGE_ERR_CUDA);
    return;
  }
  auto bar = [&](int i) -> uint32_t { return s0 + C::off_bar + 8u * i; };
  uint32_t* slot = reinterpret_cast<uint32_t*>(sm + C::off_slot);
  int32_t* info = reinterpret_cast<int32_t*>(sm + C::off_info);
  volatile int32_t* ring = reinterpret_cast<volatile int32_t*>(sm + C::off_ring);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool paired = kv_per_tile == 2;
  const int nitems = min(max(__ldg(items.n_items), 0), ntiles + kSplitSlots);

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NBAR; ++i) {
      uint32_t cnt = 1;
      if (i >= C::B_QF && i < C::B_QF + C::NSLOT) cnt = 32;
      if (i >= C::B_PPF && i < C::B_PPF + 4) cnt = 32 * R::kCompute / 2;  // PPF, DSF: one half's group
      if (i == C::B_DKE) cnt = 32 * R::kCompute;
      if (i >= C::B_IE && i < C::B_IE + C::NRING) cnt = 2 + R::kCompute;
      if (i == C::B_DONE) cnt = 2;
      mbar_init(bar(i), cnt);
    }
    fence_barrier_init();
  }
  if (warp == R::kIssueA) {
    tmem_alloc(smem_u32(slot), C::tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = slot[0];

  // The seq-th item of this CTA (its key tile, entry count and part word), as
  // handed out by the producer through the ring (tile -1: no more work, -2:
  // the producer gave up).
  auto next_tile = [&](int seq, bool ok, int* n, int* pw) -> int {
    const int rs = seq % C::NRING;
    if (!ok || !warp_wait(bar(C::B_IF + rs), (seq / C::NRING) & 1)) return -2;
    *n = ring[4 * rs + 1];
    *pw = ring[4 * rs + 2];
    return ring[4 * rs];
  };
  auto release_tile = [&](int seq) { mbar_arrive(bar(C::B_IE + seq % C::NRING)); };
  struct Tile {
    int bh, jt, key0, n0, n1;
    const int32_t *list0, *list1;
  };
  auto tile_info = [&](int it) -> Tile {
    Tile x;
    x.bh = it / Mt;
    x.jt = it % Mt;
    x.key0 = x.jt * kPair;
    const int ja = paired ? 2 * x.jt : x.jt;
    const int jb = paired ? 2 * x.jt + 1 : x.jt;
    x.list0 = col_idx + ((long long)x.bh * Mk + ja) * Mq;
    x.list1 = col_idx + ((long long)x.bh * Mk + min(jb, Mk - 1)) * Mq;
    x.n0 = min(max(__ldg(col_cnt + (long long)x.bh * Mk + ja), 0), Mq);
    x.n1 = (paired && jb < Mk) ? min(max(__ldg(col_cnt + (long long)x.bh * Mk + jb), 0), Mq) : 0;
    return x;
  };

  if (warp == R::kProducer) {
    // ---------------------------------------------------------- producer
    // All 32 lanes: they count the union of a tile's two ascending column
    // lists (list0's entries searched in list1) and load the rows' lse and D;
    // lane 0 issues the TMA copies.
    int t = 0, j = 0;  // running entry count; tiles with work so far
    bool ok = true;
    for (int seq = 0;; ++seq) {
      const int rs = seq % C::NRING;
      if (seq >= C::NRING &&
          !mbar_wait(bar(C::B_IE + rs), ((seq / C::NRING) - 1) & 1, kWaitTimeoutNs))
        ok = false;
      ok = __all_sync(0xffffffffu, ok);
      int it = -1, pw = 0;
      if (ok) {
        int k = 0;
        if (lane == 0) k = atomicAdd(work, 1);
        k = __shfl_sync(0xffffffffu, k, 0);
        if (k < nitems) {
          it = min(max(__ldg(items.seq_tile + k), 0), ntiles - 1);
          pw = __ldg(items.seq_part + k);
        }
      }
      Tile x{};
      int n = 0;
      if (it >= 0) {
        x = tile_info(it);
        const int P = (pw >> 8) & 0xff;
        if (P > 1) {
          // Part p of a cut tile: the entries of q-blocks [Mq p / P, Mq (p + 1) / P).
          const int p = pw & 0xff;
          const int qlo = (int)((long long)Mq * p / P), qhi = (int)((long long)Mq * (p + 1) / P);
          auto lower = [&](const int32_t* l, int cnt, int v) {
            int lo = 0, hi = cnt;
            while (lo < hi) {
              const int mid = (lo + hi) >> 1;
              if (__ldg(l + mid) < v) lo = mid + 1; else hi = mid;
            }
            return lo;
          };
          const int a0 = lower(x.list0, x.n0, qlo), a1 = lower(x.list0, x.n0, qhi);
          const int b0 = lower(x.list1, x.n1, qlo), b1 = lower(x.list1, x.n1, qhi);
          x.list0 += a0;
          x.n0 = a1 - a0;
          x.list1 += b0;
          x.n1 = b1 - b0;
        }
        int common = 0;
        if (paired) {
          for (int e = lane; e < x.n0; e += 32) {
            const int v = __ldg(x.list0 + e);
            int lo = 0, hi = x.n1;
            while (lo < hi) {
              const int mid = (lo + hi) >> 1;
              if (__ldg(x.list1 + mid) < v) lo = mid + 1; else hi = mid;
            }
            common += (lo < x.n1 && __ldg(x.list1 + lo) == v) ? 1 : 0;
          }
          common = __reduce_add_sync(0xffffffffu, common);
        }
        n = paired ? x.n0 + x.n1 - common : x.n0;
      }
      if (lane == 0) {
        ring[4 * rs] = ok ? it : -2;
        ring[4 * rs + 1] = n;
        ring[4 * rs + 2] = pw;
        mbar_arrive(bar(C::B_IF + rs));
      }
      if (it < 0) break;
      if (n == 0) continue;
      if (j >= 1 && !mbar_wait(bar(C::B_KVE), (j - 1) & 1, kWaitTimeoutNs)) ok = false;
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        continue;  // publishes the failure in the next ring slot, then stops
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(C::B_KV), 2 * C::kKP);
        for (int c = 0; c < D / 64; ++c) {
          const uint32_t o = c * C::kChunkK;
          tma_load_3d(s0 + C::off_k + o, &tmK, bar(C::B_KV), c * 64, x.key0, x.bh);
          tma_load_3d(s0 + C::off_k + o + kBN * 128, &tmK, bar(C::B_KV), c * 64, x.key0 + kBN,
                      x.bh);
          tma_load_3d(s0 + C::off_v + o, &tmV, bar(C::B_KV), c * 64, x.key0, x.bh);
          tma_load_3d(s0 + C::off_v + o + kBN * 128, &tmV, bar(C::B_KV), c * 64, x.key0 + kBN,
                      x.bh);
        }
      }
      ++j;
      const float* lse_h = lse + (long long)x.bh * N;
      const float* del_h = delta + (long long)x.bh * N;
      int a = 0, b = 0;
      for (int e = 0; e < n; ++e, ++t) {
        // Next entry of the union (every lane walks the lists identically).
        const int x0 = a < x.n0 ? min(max(__ldg(x.list0 + a), 0), Mq - 1) : Mq;
        const int x1 = b < x.n1 ? min(max(__ldg(x.list1 + b), 0), Mq - 1) : Mq;
        const int i = min(x0, x1);
        int flags = paired ? ((x0 == i ? 1 : 0) | (x1 == i ? 2 : 0)) : 3;
        if (x0 == i) ++a;
        if (x1 == i) ++b;
        if (i >= Mq) flags = 0;  // lists shorter than their counts claim: no work
        const int ic = min(i, Mq - 1);
        for (int h = 0; h < 2; ++h) {
          const int k = 2 * t + h, sl = k % C::NSLOT;
          if (k >= C::NSLOT &&
              !mbar_wait(bar(C::B_QE + sl), ((k / C::NSLOT) - 1) & 1, kWaitTimeoutNs))
            ok = false;
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          const int row0 = ic * kBM + h * 64;
          if (lane == 0) {
            mbar_expect_tx(bar(C::B_QF + sl), 2 * C::kQh);
            for (int c = 0; c < D / 64; ++c) {
              tma_load_3d(s0 + C::off_q + sl * C::kQh + c * C::kChunkH, &tmQ, bar(C::B_QF + sl),
                          c * 64, row0, x.bh);
              tma_load_3d(s0 + C::off_do + sl * C::kQh + c * C::kChunkH, &tmDO,
                          bar(C::B_QF + sl), c * 64, row0, x.bh);
            }
            info[sl] = ic | (flags << 24);
          }
          // -lse * log2(e) and -D of the half's 64 tokens (queries past N get
          // -inf and 0, so that their P and dS are 0).
          float2 l2, d2;
          const int tok = row0 + lane * 2;
          l2.x = tok < N ? -__ldg(lse_h + tok) * kLog2e : -INFINITY;
          l2.y = tok + 1 < N ? -__ldg(lse_h + tok + 1) * kLog2e : -INFINITY;
          d2.x = tok < N ? -__ldg(del_h + tok) : 0.f;
          d2.y = tok + 1 < N ? -__ldg(del_h + tok + 1) : 0.f;
          float* rowv = reinterpret_cast<float*>(sm + C::off_row + sl * (2 * 64 * 4));
          reinterpret_cast<float2*>(rowv)[lane] = l2;
          reinterpret_cast<float2*>(rowv + 64)[lane] = d2;
          mbar_arrive(bar(C::B_QF + sl));
        }
        if (!ok) break;
      }
    }
    if (!ok && lane == 0) report_error(status, SPARGE_ERR_TIMEOUT);
    // Let the last loads land before the CTA can exit.
    if (lane == 0) {
      if (j > 0) mbar_wait(bar(C::B_KV), (j - 1) & 1, kWaitTimeoutNs);
      for (int k = max(0, 2 * t - C::NSLOT); k < 2 * t; ++k)
        mbar_wait(bar(C::B_QF + k % C::NSLOT), (k / C::NSLOT) & 1, kWaitTimeoutNs);
    }
  } else if (warp == R::kIssueA) {
    // ---------------------------------------------------------- S^T, dP^T
    // S^T_h = K Q_h^T and dP^T_h = V dO_h^T (M = 128 keys, N = 64 queries of
    // half h, K = d).  The whole warp runs the loop; one elected lane issues
    // each MMA.
    constexpr uint32_t idS = idesc_bf16(kPair, 64, false, false);
    const uint64_t dk0 = sdesc_sw128(s0 + C::off_k, 16, 1024);
    const uint64_t dv0 = sdesc_sw128(s0 + C::off_v, 16, 1024);
    bool ok = true;
    int t = 0, j = 0;
    for (int seq = 0;; ++seq) {
      int n = 0, pw = 0;
      const int it = next_tile(seq, ok, &n, &pw);
      if (lane == 0) release_tile(seq);
      if (it < 0) {
        if (it == -2) ok = false;
        break;
      }
      if (n == 0) continue;
      if (!warp_wait(bar(C::B_KV), j & 1)) {
        ok = false;
        break;
      }
      ++j;
      for (int e = 0; ok && e < n; ++e, ++t) {
        for (int h = 0; h < 2; ++h) {
          const int k = 2 * t + h, sl = k % C::NSLOT;
          // S^T_h's columns hold P^T_h of entry t - 1 until its dV MMAs are
          // done, dP^T_h's hold dS^T_h until its dK MMAs are.
          if (!warp_wait(bar(C::B_QF + sl), (k / C::NSLOT) & 1) ||
              (t >= 1 && !warp_wait(bar(C::B_RVF + h), (t - 1) & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t dq = sdesc_sw128(s0 + C::off_q + sl * C::kQh, 16, 1024);
          const uint64_t ddo = sdesc_sw128(s0 + C::off_do + sl * C::kQh, 16, 1024);
          const uint32_t dS = tmem + h * 128;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t ka = (kk >> 2) * C::kChunkK + (kk & 3) * 32;
            const uint32_t kb = (kk >> 2) * C::kChunkH + (kk & 3) * 32;
            warp_mma_bf16(dS, sdesc_add(dk0, ka), sdesc_add(dq, kb), idS, kk > 0);
          }
          warp_commit(bar(C::B_SSF + h));
          if (t >= 1 && !warp_wait(bar(C::B_RKF + h), (t - 1) & 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t ka = (kk >> 2) * C::kChunkK + (kk & 3) * 32;
            const uint32_t kb = (kk >> 2) * C::kChunkH + (kk & 3) * 32;
            warp_mma_bf16(dS + 64, sdesc_add(dv0, ka), sdesc_add(ddo, kb), idS, kk > 0);
          }
          warp_commit(bar(C::B_DPF + h));
        }
      }
      if (!ok) break;
      warp_commit(bar(C::B_KVE));  // every S^T and dP^T of this tile issued
    }
    if (!ok && lane == 0) report_error(status, SPARGE_ERR_TIMEOUT);
    warp_commit(bar(C::B_DONE));
    warp_wait(bar(C::B_DONE), 0);
  } else if (warp == R::kIssueB) {
    // ---------------------------------------------------------- dV, dK
    // dV += P^T_h dO_h and dK += dS^T_h Q_h (M = 128 keys, N = d, K = the 64
    // queries of half h); A from TMEM, B = dO_h / Q_h read MN-major.  The
    // first MMAs of a tile overwrite the accumulators, after the compute
    // warps have read out the previous tile's.
    constexpr uint32_t idG = idesc_bf16(kPair, D, false, true);
    constexpr int NC = 32;  // queries per P^T / dS^T chunk in TMEM
    bool ok = true;
    int t = 0, j = 0;
    for (int seq = 0;; ++seq) {
      int n = 0, pw = 0;
      const int it = next_tile(seq, ok, &n, &pw);
      if (lane == 0) release_tile(seq);
      if (it < 0) {
        if (it == -2) ok = false;
        break;
      }
      if (n == 0) continue;
      for (int e = 0; ok && e < n; ++e, ++t) {
        for (int h = 0; h < 2; ++h) {
          const int sl = (2 * t + h) % C::NSLOT;
          const uint64_t dq = sdesc_sw128(s0 + C::off_q + sl * C::kQh, C::kChunkH, 1024);
          const uint64_t ddo = sdesc_sw128(s0 + C::off_do + sl * C::kQh, C::kChunkH, 1024);
          const uint32_t ap = tmem + h * 128;
          const bool first = e == 0 && h == 0;
          if (!warp_wait(bar(C::B_PPF + h), t & 1) ||
              (first && j >= 1 && !warp_wait(bar(C::B_DKE), (j - 1) & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          // Queries 16kk .. 16kk + 15 of the half: the TMEM columns where the
          // compute group wrote their chunk's bf16 pairs.
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            warp_mma_bf16_ta(tmem + C::col_dv, ap + NC * (16 * kk / NC) + (16 * kk % NC) / 2,
                             sdesc_add(ddo, kk * 2048), idG, (!first || kk > 0) ? 1u : 0u);
          warp_commit(bar(C::B_RVF + h));
          if (!warp_wait(bar(C::B_DSF + h), t & 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            warp_mma_bf16_ta(tmem + C::col_dk, ap + 64 + NC * (16 * kk / NC) + (16 * kk % NC) / 2,
                             sdesc_add(dq, kk * 2048), idG, (!first || kk > 0) ? 1u : 0u);
          warp_commit(bar(C::B_RKF + h));
          warp_commit(bar(C::B_QE + sl));
        }
      }
      ++j;
    }
    if (!ok && lane == 0) report_error(status, SPARGE_ERR_TIMEOUT);
    warp_commit(bar(C::B_DONE));
    warp_wait(bar(C::B_DONE), 0);
  } else if (warp < R::kCompute) {
    // ---------------------------------------------------------- compute
    // Thread = key row r (TMEM lane).  Warp group g = warp / 4 takes query
    // half g of every entry (all 64 queries, in two chunks of 32), so the two
    // warps of an SM sub-partition work on different halves and their
    // latencies overlap (measured at 480p: 1.038 against 1.059 ms per
    // backward with both groups on the same half, 32 queries each).
    constexpr int FPW = D / (R::kCompute / 4);  // features per warp in the epilogue
    const int quarter = warp & 3, cg = warp >> 2;
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const int flag_bit = r < kBN ? 1 : 2;  // warp-uniform (quarters 0-1 vs 2-3)
    bool ok = true;
    int t = 0;
    for (int seq = 0;; ++seq) {
      int n = 0, pw = 0;
      const int it = next_tile(seq, ok, &n, &pw);
      __syncwarp();
      if (lane == 0) release_tile(seq);
      if (it < 0) {
        if (it == -2) ok = false;
        break;
      }
      const int bh = it / Mt, key0 = (it % Mt) * kPair;
      const bool key_in = key0 + r < N;
      const long long rowoff = ((long long)bh * N + key0 + r) * D;
      // Part of a cut tile (P > 1): dV and dK of this row go to the part's
      // fp32 slot first (dV at [0, d), dK at [d, 2d)).
      const int P = (pw >> 8) & 0xff, slot0 = (pw >> 16) & 0xffff;
      float* part_row =
          items.split_part + ((long long)(slot0 + (pw & 0xff)) * kPair + r) * (2 * D);
      // Once the part's rows are written: the warp's completion counter of the
      // tile; the warp that completes it adds the P partials in part order
      // (0, 1, ..., P - 1, whichever CTA ran them) and writes bf16 dV, dK.
      auto finish_part = [&]() {
        __threadfence();
        __syncwarp();
        int last = 0;
        if (lane == 0) last = atomicAdd(items.split_cnt + slot0 * kDkdvWarps + warp, 1) == P - 1;
        if (!__shfl_sync(0xffffffffu, last, 0) || !key_in) return;
        __threadfence();
        const float* p0 = items.split_part + ((long long)slot0 * kPair + r) * (2 * D);
#pragma unroll 1
        for (int cc = cg * FPW; cc < (cg + 1) * FPW; cc += 4) {
          float4 sv = make_float4(0.f, 0.f, 0.f, 0.f), sk = sv;
#pragma unroll 1
          for (int q = 0; q < P; ++q) {
            const float4* pr = reinterpret_cast<const float4*>(p0 + (long long)q * kPair * 2 * D);
            const float4 v = __ldcg(pr + cc / 4), w = __ldcg(pr + (D + cc) / 4);
            sv = q == 0 ? v : make_float4(sv.x + v.x, sv.y + v.y, sv.z + v.z, sv.w + v.w);
            sk = q == 0 ? w : make_float4(sk.x + w.x, sk.y + w.y, sk.z + w.z, sk.w + w.w);
          }
          __stcs(reinterpret_cast<uint2*>(dv + rowoff + cc),
                 make_uint2(pack_bf16x2(sv.x, sv.y), pack_bf16x2(sv.z, sv.w)));
          __stcs(reinterpret_cast<uint2*>(dk + rowoff + cc),
                 make_uint2(pack_bf16x2(sk.x * scale, sk.y * scale),
                            pack_bf16x2(sk.z * scale, sk.w * scale)));
        }
      };
      if (n == 0) {
        // Keys no q-block (of this part) keeps: dK = dV = 0.
        if (key_in) {
          const uint4 z = make_uint4(0u, 0u, 0u, 0u);
          for (int cc = cg * FPW; cc < (cg + 1) * FPW; cc += 8) {
            if (P > 1) {
              __stcg(reinterpret_cast<uint4*>(part_row + cc), z);
              __stcg(reinterpret_cast<uint4*>(part_row + cc + 4), z);
              __stcg(reinterpret_cast<uint4*>(part_row + D + cc), z);
              __stcg(reinterpret_cast<uint4*>(part_row + D + cc + 4), z);
            } else {
              __stcs(reinterpret_cast<uint4*>(dv + rowoff + cc), z);
              __stcs(reinterpret_cast<uint4*>(dk + rowoff + cc), z);
            }
          }
        }
        if (P > 1) finish_part();
        continue;
      }
      for (int e = 0; ok && e < n; ++e, ++t) {
        // This warp group's half of the entry: queries 64h .. 64h + 63 of the
        // q-block, taken in two chunks of 32.
        const int h = cg;
        const int k = 2 * t + h, sl = k % C::NSLOT;
        if (!warp_wait(bar(C::B_QF + sl), (k / C::NSLOT) & 1) ||
            !warp_wait(bar(C::B_SSF + h), t & 1)) {
          ok = false;
          break;
        }
        const int flags = info[sl] >> 24;
        const bool live = (flags & flag_bit) != 0;  // warp-uniform
        const float* rowv = reinterpret_cast<const float*>(sm + C::off_row + sl * (2 * 64 * 4));
        tc_fence_after();
        // P^T first (from S^T alone); it is the A operand of dV.  Chunk c's
        // bf16 pairs go over S^T columns 32c .. 32c + 15, which it has read.
        float p[64];
        const uint64_t sl2 = f32x2(scale_log2, scale_log2);
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          const uint32_t sa = lane_base + h * 128 + 32 * c2;
          uint32_t pk[16];
          if (live) {
            uint32_t sr[2][16];
            SPARGE_TMEM_LD_X16(sa, sr[0]);
            SPARGE_TMEM_LD_X16(sa + 16, sr[1]);
            SPARGE_TMEM_WAIT_LD16(sr[0]);
            SPARGE_TMEM_WAIT_LD16(sr[1]);
            // Two queries per packed instruction: P^T = 2^(S^T * scale*log2e - lse*log2e).
            const ulonglong2* l4 = reinterpret_cast<const ulonglong2*>(rowv + 32 * c2);
#pragma unroll
            for (int g = 0; g < 8; ++g) {
              const ulonglong2 lv = l4[g];  // -lse*log2e of queries 4g .. 4g + 3
#pragma unroll
              for (int q2 = 0; q2 < 2; ++q2) {
                const int col = g * 4 + 2 * q2;
                const uint64_t x = ffma2(f32x2(__uint_as_float(sr[col / 16][col % 16]),
                                               __uint_as_float(sr[col / 16][col % 16 + 1])),
                                         sl2, q2 == 0 ? lv.x : lv.y);
                p[32 * c2 + col] = key_in ? ex2_approx(f32x2_lo(x)) : 0.f;
                p[32 * c2 + col + 1] = key_in ? ex2_approx(f32x2_hi(x)) : 0.f;
              }
            }
#pragma unroll
            for (int q4 = 0; q4 < 16; ++q4)
              pk[q4] = pack_bf16x2(p[32 * c2 + 2 * q4], p[32 * c2 + 2 * q4 + 1]);
          } else {
#pragma unroll
            for (int q4 = 0; q4 < 32; ++q4) p[32 * c2 + q4] = 0.f;
#pragma unroll
            for (int q4 = 0; q4 < 16; ++q4) pk[q4] = 0u;
          }
          SPARGE_TMEM_ST_X16(sa, pk);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(C::B_PPF + h));
        // dS^T = P^T * (dP^T - D).
        if (!warp_wait(bar(C::B_DPF + h), t & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          const uint32_t sa = lane_base + h * 128 + 32 * c2;
          uint32_t pk[16];
          if (live) {
            uint32_t dr[2][16];
            SPARGE_TMEM_LD_X16(sa + 64, dr[0]);
            SPARGE_TMEM_LD_X16(sa + 64 + 16, dr[1]);
            SPARGE_TMEM_WAIT_LD16(dr[0]);
            SPARGE_TMEM_WAIT_LD16(dr[1]);
            // Two queries per packed instruction.
            const ulonglong2* d4 = reinterpret_cast<const ulonglong2*>(rowv + 64 + 32 * c2);
#pragma unroll
            for (int g = 0; g < 8; ++g) {
              const ulonglong2 dv4 = d4[g];  // -D of queries 4g .. 4g + 3
#pragma unroll
              for (int q2 = 0; q2 < 2; ++q2) {
                const int col = g * 4 + 2 * q2;
                const uint64_t dd = fadd2(f32x2(__uint_as_float(dr[col / 16][col % 16]),
                                                __uint_as_float(dr[col / 16][col % 16 + 1])),
                                          q2 == 0 ? dv4.x : dv4.y);
                const uint64_t z =
                    fmul2(f32x2(p[32 * c2 + col], p[32 * c2 + col + 1]), dd);
                pk[g * 2 + q2] = pack_bf16x2(f32x2_lo(z), f32x2_hi(z));
              }
            }
          } else {
#pragma unroll
            for (int q4 = 0; q4 < 16; ++q4) pk[q4] = 0u;
          }
          SPARGE_TMEM_ST_X16(sa + 64, pk);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(C::B_DSF + h));
      }
      if (!ok) break;
      // Epilogue: lane r holds key r of dV and dK; warp group cg writes its
      // share of the features, then releases the accumulators to the next
      // tile's first MMAs.  Every gradient MMA of the tile is done once dK of
      // the last entry's second half is (the pipe runs them in order).  The
      // warps of the first half get here as soon as their own last half is
      // done, when that barrier may still be one phase short of the last
      // entry's previous phase (its dP^T had to wait only for the one before),
      // so the wait takes the previous phase first: a parity wait is exact
      // only within one phase of the barrier.
      if ((t >= 2 && !warp_wait(bar(C::B_RKF + 1), (t - 2) & 1)) ||
          !warp_wait(bar(C::B_RKF + 1), (t - 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll 1
      for (int cc = cg * FPW; cc < (cg + 1) * FPW; cc += 16) {
        uint32_t rv_[16], rk_[16];
        SPARGE_TMEM_LD_X16(lane_base + C::col_dv + cc, rv_);
        SPARGE_TMEM_LD_X16(lane_base + C::col_dk + cc, rk_);
        SPARGE_TMEM_WAIT_LD16(rv_);
        SPARGE_TMEM_WAIT_LD16(rk_);
        if (cc + 16 >= (cg + 1) * FPW) {
          tc_fence_before();
          mbar_arrive(bar(C::B_DKE));
        }
        if (key_in && P > 1) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            __stcg(reinterpret_cast<uint4*>(part_row + cc) + i,
                   make_uint4(rv_[4 * i], rv_[4 * i + 1], rv_[4 * i + 2], rv_[4 * i + 3]));
            __stcg(reinterpret_cast<uint4*>(part_row + D + cc) + i,
                   make_uint4(rk_[4 * i], rk_[4 * i + 1], rk_[4 * i + 2], rk_[4 * i + 3]));
          }
        } else if (key_in) {
          uint4 v0, v1, k0, k1;
          v0.x = pack_bf16x2(__uint_as_float(rv_[0]), __uint_as_float(rv_[1]));
          v0.y = pack_bf16x2(__uint_as_float(rv_[2]), __uint_as_float(rv_[3]));
          v0.z = pack_bf16x2(__uint_as_float(rv_[4]), __uint_as_float(rv_[5]));
          v0.w = pack_bf16x2(__uint_as_float(rv_[6]), __uint_as_float(rv_[7]));
          v1.x = pack_bf16x2(__uint_as_float(rv_[8]), __uint_as_float(rv_[9]));
          v1.y = pack_bf16x2(__uint_as_float(rv_[10]), __uint_as_float(rv_[11]));
          v1.z = pack_bf16x2(__uint_as_float(rv_[12]), __uint_as_float(rv_[13]));
          v1.w = pack_bf16x2(__uint_as_float(rv_[14]), __uint_as_float(rv_[15]));
          k0.x = pack_bf16x2(__uint_as_float(rk_[0]) * scale, __uint_as_float(rk_[1]) * scale);
          k0.y = pack_bf16x2(__uint_as_float(rk_[2]) * scale, __uint_as_float(rk_[3]) * scale);
          k0.z = pack_bf16x2(__uint_as_float(rk_[4]) * scale, __uint_as_float(rk_[5]) * scale);
          k0.w = pack_bf16x2(__uint_as_float(rk_[6]) * scale, __uint_as_float(rk_[7]) * scale);
          k1.x = pack_bf16x2(__uint_as_float(rk_[8]) * scale, __uint_as_float(rk_[9]) * scale);
          k1.y = pack_bf16x2(__uint_as_float(rk_[10]) * scale, __uint_as_float(rk_[11]) * scale);
          k1.z = pack_bf16x2(__uint_as_float(rk_[12]) * scale, __uint_as_float(rk_[13]) * scale);
          k1.w = pack_bf16x2(__uint_as_float(rk_[14]) * scale, __uint_as_float(rk_[15]) * scale);
          __stcs(reinterpret_cast<uint4*>(dv + rowoff + cc), v0);
          __stcs(reinterpret_cast<uint4*>(dv + rowoff + cc + 8), v1);
          __stcs(reinterpret_cast<uint4*>(dk + rowoff + cc), k0);
          __stcs(reinterpret_cast<uint4*>(dk + rowoff + cc + 8), k1);
        }
      }
      if (P > 1) finish_part();
    }
    if (!ok) report_error(status, SPARGE_ERR_TIMEOUT);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == R::kIssueA) {
    tc_fence_after();
    tmem_dealloc(tmem, C::tmem_cols);
  }
}

// ---------------------------------------------------------------- dQ
template <int D>
struct DqCfg {
  // K slots outnumber V slots: a K slot is held until dQ of its step, a V
  // slot only until dP.
  static constexpr int NSK = D == 128 ? 3 : 6;
  static constexpr int NSV = D == 128 ? 2 : 4;
  static constexpr int NRING = 4;                   // q-blocks handed out ahead
  static constexpr uint32_t kKP = kPair * D * 2;    // K (or V) of 128 keys
  static constexpr uint32_t kQ = kBM * D * 2;
  static constexpr uint32_t kChunkK = kPair * 128;
  static constexpr uint32_t kChunkQ = kBM * 128;
  static constexpr uint32_t off_q = 0;
  static constexpr uint32_t off_do = off_q + kQ;
  static constexpr uint32_t off_k = off_do + kQ;        // NSK slots of K
  static constexpr uint32_t off_v = off_k + NSK * kKP;  // NSV slots of V
  static constexpr uint32_t off_ring = off_v + NSV * kKP;  // NRING q-block ids
  static constexpr uint32_t off_bar = off_ring + 64;
  static constexpr int B_Q = 0;            // Q, dO of a q-block landed
  static constexpr int B_QE = 1;           // its S and dP MMAs done: Q, dO slots free
  static constexpr int B_KF = 2;           // NSK: K landed
  static constexpr int B_VF = B_KF + NSK;  // NSV: V landed
  static constexpr int B_KE = B_VF + NSV;  // NSK: K slot free (dQ of its step done)
  static constexpr int B_VE = B_KE + NSK;  // NSV: V slot free (dP of its step done)
  static constexpr int B_SF = B_VE + NSV;  // 2: S in TMEM buffer b
  static constexpr int B_SE = B_SF + 2;    // 2: dQ read dS of buffer b (buffer free)
  static constexpr int B_DSF = B_SE + 2;   // 8: dS of key chunk c written into buffer b (4b + c)
  static constexpr int B_DPF = B_DSF + 8;  // dP complete
  static constexpr int B_DPE = B_DPF + 1;  // all compute threads: dP read
  static constexpr int B_DQE = B_DPE + 1;  // all compute threads: dQ accumulator read out
  static constexpr int B_IF = B_DQE + 1;   // NRING: q-block id written
  static constexpr int B_IE = B_IF + NRING;  // NRING: id read by both issuers and every compute warp
  static constexpr int B_DONE = B_IE + NRING;  // count 2
  static constexpr int NBAR = B_DONE + 1;
  static constexpr uint32_t off_slot = off_bar + NBAR * 8;
  static constexpr uint32_t bytes = off_slot + 16;
  static constexpr uint32_t smem_alloc = bytes + 1024;
  // TMEM: dQ [0, D), S of step g in buffer g % 2 at 128 + 128 * (g % 2) (128
  // keys; dS of keys 32c .. 32c + 31 written over its columns 32c .. 32c + 15
  // as bf16 pairs), dP at 384.
  static constexpr uint32_t tmem_cols = 512;
  static constexpr uint32_t col_dq = 0;
  static constexpr uint32_t col_s = 128;
  static constexpr uint32_t col_dp = 384;
};

// Persistent: one CTA per SM takes q-blocks from a work counter, in the
// launch order (long lists first), until all are done.  A q-block's list of
// kept kv-blocks is taken two entries at a time (kv_per_entry = 1: 64-key
// blocks; the second of an odd count is empty), or one 128-key block per step
// (kv_per_entry = 2).  Q and dO stay in shared memory as the A operands of S
// and dP; S is double-buffered in TMEM, so S of the next step is computed
// while the compute warps work on this one, and the loads and first MMAs of
// the next q-block overlap the current one's last steps and epilogue.  The
// steps of successive q-blocks share one running step count g, which indexes
// the slot rings and barrier phases.
template <int D>
__global__ void __launch_bounds__(Roles<kDqWarps>::kThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                  const float* __restrict__ lse, const float* __restrict__ delta,
                  const int32_t* __restrict__ row_idx, const int32_t* __restrict__ row_cnt,
                  const int32_t* __restrict__ row_order, int nitems, int32_t* __restrict__ work,
                  int N, int Mq, int Mk, int kv_per_entry, float scale, float scale_log2,
                  __nv_bfloat16* __restrict__ dq, int32_t* __restrict__ status) {
  using C = DqCfg<D>;
  using R = Roles<kDqWarps>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const uint32_t s0 = smem_u32(sm);
  auto bar = [&](int i) -> uint32_t { return s0 + C::off_bar + 8u * i; };
  uint32_t* slot = reinterpret_cast<uint32_t*>(sm + C::off_slot);
  volatile int32_t* ring = reinterpret_cast<volatile int32_t*>(sm + C::off_ring);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool single = kv_per_entry == 1;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NBAR; ++i) {
      uint32_t cnt = 1;
      if (i == C::B_DPE || i == C::B_DQE) cnt = 32 * R::kCompute;
      if (i >= C::B_DSF && i < C::B_DSF + 8) cnt = 32 * (R::kCompute / 4);
      if (i >= C::B_IE && i < C::B_IE + C::NRING) cnt = 2 + R::kCompute;
      if (i == C::B_DONE) cnt = 2;
      mbar_init(bar(i), cnt);
    }
    fence_barrier_init();
  }
  if (warp == R::kIssueA) {
    tmem_alloc(smem_u32(slot), C::tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;

  // The q-block handed out as the seq-th of this CTA (-1: no more work).  The
  // producer fetches ids from the counter into a ring; the other roles read
  // them from there, in the same order (whole warps: the result is
  // warp-uniform).
  auto next_item = [&](int seq, bool ok) -> int {
    const int rs = seq % C::NRING;
    if (!ok || !warp_wait(bar(C::B_IF + rs), (seq / C::NRING) & 1)) return -2;
    const int it = ring[rs];
    return it;
  };
  auto release_item = [&](int seq) { mbar_arrive(bar(C::B_IE + seq % C::NRING)); };
  struct Item {
    int bh, qb, n, npair;
    const int32_t* list;
  };
  auto item_info = [&](int it) -> Item {
    Item x;
    x.bh = it / Mq;
    x.qb = it % Mq;
    const long long row_id = (long long)x.bh * Mq + x.qb;
    x.n = min(max(__ldg(row_cnt + row_id), 0), Mk);
    x.list = row_idx + row_id * Mk;
    x.npair = single ? (x.n + 1) / 2 : x.n;
    return x;
  };
  // First row (in tokens) of the two 64-key halves of step u; -1 = empty half.
  auto half_row = [&](const Item& x, int u, int half) -> int {
    if (single) {
      const int e = 2 * u + half;
      return e < x.n ? min(max(__ldg(x.list + e), 0), Mk - 1) * kBN : -1;
    }
    return min(max(__ldg(x.list + u), 0), Mk - 1) * kPair + half * kBN;
  };

  if (warp == R::kProducer) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      int g = 0, j = 0;
      bool ok = true;
      for (int seq = 0;; ++seq) {
        const int rs = seq % C::NRING;
        if (seq >= C::NRING &&
            !mbar_wait(bar(C::B_IE + rs), ((seq / C::NRING) - 1) & 1, kWaitTimeoutNs))
          ok = false;
        int it = -1;
        if (ok) {
          const int k = atomicAdd(work, 1);
          it = k < nitems ? min(max(__ldg(row_order + k), 0), nitems - 1) : -1;
        }
        ring[rs] = ok ? it : -2;
        mbar_arrive(bar(C::B_IF + rs));
        if (it < 0) break;
        const Item x = item_info(it);
        if (x.n == 0) continue;
        if (j >= 1 && !mbar_wait(bar(C::B_QE), (j - 1) & 1, kWaitTimeoutNs)) {
          ok = false;
          continue;  // publishes the failure in the next ring slot, then stops
        }
        mbar_arrive_expect_tx(bar(C::B_Q), 2 * C::kQ);
        for (int c = 0; c < D / 64; ++c) {
          tma_load_3d(s0 + C::off_q + c * C::kChunkQ, &tmQ, bar(C::B_Q), c * 64, x.qb * kBM, x.bh);
          tma_load_3d(s0 + C::off_do + c * C::kChunkQ, &tmDO, bar(C::B_Q), c * 64, x.qb * kBM,
                      x.bh);
        }
        ++j;
        for (int u = 0; ok && u < x.npair; ++u, ++g) {
          const int sk = g % C::NSK, sv = g % C::NSV;
          int rw[2];
          for (int half = 0; half < 2; ++half) {
            rw[half] = half_row(x, u, half);
            if (rw[half] < 0) rw[half] = Mk * kBN;  // empty half: rows past N read as zeros
          }
          // K first: S of this step needs it before dP needs V.
          if (g >= C::NSK &&
              !mbar_wait(bar(C::B_KE + sk), ((g / C::NSK) - 1) & 1, kWaitTimeoutNs)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar(C::B_KF + sk), C::kKP);
          for (int half = 0; half < 2; ++half)
            for (int c = 0; c < D / 64; ++c)
              tma_load_3d(s0 + C::off_k + sk * C::kKP + c * C::kChunkK + half * kBN * 128, &tmK,
                          bar(C::B_KF + sk), c * 64, rw[half], x.bh);
          if (g >= C::NSV &&
              !mbar_wait(bar(C::B_VE + sv), ((g / C::NSV) - 1) & 1, kWaitTimeoutNs)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar(C::B_VF + sv), C::kKP);
          for (int half = 0; half < 2; ++half)
            for (int c = 0; c < D / 64; ++c)
              tma_load_3d(s0 + C::off_v + sv * C::kKP + c * C::kChunkK + half * kBN * 128, &tmV,
                          bar(C::B_VF + sv), c * 64, rw[half], x.bh);
        }
      }
      if (!ok) report_error(status, SPARGE_ERR_TIMEOUT);
      // Let the last loads land before the CTA can exit.
      if (j > 0) mbar_wait(bar(C::B_Q), (j - 1) & 1, kWaitTimeoutNs);
      for (int e = max(0, g - C::NSK); e < g; ++e)
        mbar_wait(bar(C::B_KF + e % C::NSK), (e / C::NSK) & 1, kWaitTimeoutNs);
      for (int e = max(0, g - C::NSV); e < g; ++e)
        mbar_wait(bar(C::B_VF + e % C::NSV), (e / C::NSV) & 1, kWaitTimeoutNs);
    }
  } else if (warp == R::kIssueA) {
    // ---------------------------------------------------------- S, dP
    // S_g = Q K_g^T into TMEM buffer g % 2 (free once dQ of step g - 2 has
    // read its dS), then dP_g = dO V_g^T (its region frees once the compute
    // warps have read dP of step g - 1).  M = 128 queries, N = 128 keys.  The
    // whole warp runs the loop; one elected lane issues each MMA.
    constexpr uint32_t idS = idesc_bf16(kBM, kPair, false, false);
    const uint64_t dq0 = sdesc_sw128(s0 + C::off_q, 16, 1024);
    const uint64_t ddo0 = sdesc_sw128(s0 + C::off_do, 16, 1024);
    bool ok = true;
    int g = 0, j = 0;
    for (int seq = 0;; ++seq) {
      const int it = next_item(seq, ok);
      if (lane == 0) release_item(seq);
      if (it < 0) {
        if (it == -2) ok = false;
        break;
      }
      const Item x = item_info(it);
      if (x.n == 0) continue;
      if (!warp_wait(bar(C::B_Q), j & 1)) {
        ok = false;
        break;
      }
      ++j;
      for (int u = 0; ok && u < x.npair; ++u, ++g) {
        const int sk = g % C::NSK, sv = g % C::NSV, b = g & 1;
        if (!warp_wait(bar(C::B_KF + sk), (g / C::NSK) & 1) ||
            (g >= 2 && !warp_wait(bar(C::B_SE + b), ((g >> 1) - 1) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t dkd = sdesc_sw128(s0 + C::off_k + sk * C::kKP, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ka = (kk >> 2) * C::kChunkQ + (kk & 3) * 32;
          const uint32_t kb = (kk >> 2) * C::kChunkK + (kk & 3) * 32;
          warp_mma_bf16(tmem + C::col_s + 128 * b, sdesc_add(dq0, ka), sdesc_add(dkd, kb), idS,
                        kk > 0);
        }
        warp_commit(bar(C::B_SF + b));
        if (!warp_wait(bar(C::B_VF + sv), (g / C::NSV) & 1) ||
            (g >= 1 && !warp_wait(bar(C::B_DPE), (g - 1) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t dvd = sdesc_sw128(s0 + C::off_v + sv * C::kKP, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ka = (kk >> 2) * C::kChunkQ + (kk & 3) * 32;
          const uint32_t kb = (kk >> 2) * C::kChunkK + (kk & 3) * 32;
          warp_mma_bf16(tmem + C::col_dp, sdesc_add(ddo0, ka), sdesc_add(dvd, kb), idS, kk > 0);
        }
        warp_commit(bar(C::B_DPF));
        warp_commit(bar(C::B_VE + sv));
      }
      if (!ok) break;
      warp_commit(bar(C::B_QE));  // every S and dP of this q-block issued
    }
    if (!ok && lane == 0) report_error(status, SPARGE_ERR_TIMEOUT);
    warp_commit(bar(C::B_DONE));
    warp_wait(bar(C::B_DONE), 0);
  } else if (warp == R::kIssueB) {
    // ---------------------------------------------------------- dQ
    // dQ += dS_g K_g (A = dS from TMEM buffer g % 2, K = 128 keys; B = the key
    // tile read MN-major, N = d).  dS of keys 16kk .. 16kk + 15 sits in the
    // buffer's columns 32 (kk / 2) + 8 (kk % 2) .. + 7.  The first step of a
    // q-block waits until the previous one's accumulator has been read out.
    constexpr uint32_t idQ = idesc_bf16(kBM, D, false, true);
    bool ok = true;
    int g = 0, j = 0;
    for (int seq = 0;; ++seq) {
      const int it = next_item(seq, ok);
      if (lane == 0) release_item(seq);
      if (it < 0) {
        if (it == -2) ok = false;
        break;
      }
      const Item x = item_info(it);
      if (x.n == 0) continue;
      for (int u = 0; ok && u < x.npair; ++u, ++g) {
        const int sk = g % C::NSK, b = g & 1;
        if (u == 0 && j >= 1 && !warp_wait(bar(C::B_DQE), (j - 1) & 1)) {
          ok = false;
          break;
        }
        const uint64_t dkd = sdesc_sw128(s0 + C::off_k + sk * C::kKP, C::kChunkK, 1024);
        const uint32_t ads = tmem + C::col_s + 128 * b;
        // Key chunk c (keys 32c .. 32c + 31) is written by the four warps of
        // group c; its two MMAs start as soon as that chunk is there (measured
        // at 480p: 1.038 against 1.044 ms per backward with one barrier for
        // the whole step).
#pragma unroll
        for (int kk = 0; kk < kPair / 16; ++kk) {
          if ((kk & 1) == 0) {
            if (!warp_wait(bar(C::B_DSF + 4 * b + (kk >> 1)), (g >> 1) & 1)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          warp_mma_bf16_ta(tmem + C::col_dq, ads + (kk >> 1) * 32 + (kk & 1) * 8,
                           sdesc_add(dkd, kk * 2048), idQ, (u > 0 || kk > 0) ? 1u : 0u);
        }
        if (!ok) break;
        warp_commit(bar(C::B_SE + b));
        warp_commit(bar(C::B_KE + sk));
      }
      ++j;
    }
    if (!ok && lane == 0) report_error(status, SPARGE_ERR_TIMEOUT);
    warp_commit(bar(C::B_DONE));
    warp_wait(bar(C::B_DONE), 0);
  } else if (warp < R::kCompute) {
    // ---------------------------------------------------------- compute
    // Thread = query row r (TMEM lane); warp group c = warp / 4 takes keys
    // 32c .. 32c + 31 of each step (64-key half c / 2 of it), and features
    // c * D/4 .. (c + 1) * D/4 - 1 of dQ.
    const int quarter = warp & 3, cg = warp >> 2, half = cg >> 1;
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    bool ok = true;
    int g = 0, j = 0;
    for (int seq = 0;; ++seq) {
      const int it = next_item(seq, ok);
      __syncwarp();
      if (lane == 0) release_item(seq);
      if (it < 0) {
        if (it == -2) ok = false;
        break;
      }
      const Item x = item_info(it);
      const int row = x.qb * kBM + r;
      const bool rv = row < N;
      __nv_bfloat16* qrow = dq + ((long long)x.bh * N + row) * D;
      if (x.n == 0) {
        if (rv) {
          const uint4 z = make_uint4(0u, 0u, 0u, 0u);
          for (int cc = cg * (D / 4); cc < (cg + 1) * (D / 4); cc += 8)
            __stcs(reinterpret_cast<uint4*>(qrow + cc), z);
        }
        continue;
      }
      const float lse2 = rv ? __ldg(lse + (long long)x.bh * N + row) * kLog2e : 0.f;
      const float drow = rv ? __ldg(delta + (long long)x.bh * N + row) : 0.f;
      int rw_next = half_row(x, 0, half);  // one step ahead
      for (int u = 0; ok && u < x.npair; ++u, ++g) {
        const int b = g & 1;
        const int rw = rw_next;
        if (u + 1 < x.npair) rw_next = half_row(x, u + 1, half);
        // Valid keys among this thread's 32 (0 for an empty half; warp-uniform).
        const int valid = rw < 0 ? 0 : min(32, max(0, N - rw - 32 * (cg & 1)));
        if (!warp_wait(bar(C::B_SF + b), (g >> 1) & 1) || !warp_wait(bar(C::B_DPF), g & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // dP first, so that its region is released (and dP of the next step
        // computed) while this step's softmax runs.
        uint32_t dr[16], dr2[16], sr[16], sr2[16];
        tmem_ld32u(lane_base + C::col_dp + 32 * cg, dr, dr2);
        tc_fence_before();
        mbar_arrive(bar(C::B_DPE));
        const uint32_t sb = lane_base + C::col_s + 128 * b + 32 * cg;
        tmem_ld32u(sb, sr, sr2);
        uint32_t pk[16];
        if (rv && valid == 32) {
          // Two columns per packed instruction: P = 2^(S * scale*log2e - lse*log2e),
          // dS = P * (dP - D).
          const uint64_t sl2 = f32x2(scale_log2, scale_log2);
          const uint64_t nl2 = f32x2(-lse2, -lse2);
          const uint64_t nd2 = f32x2(-drow, -drow);
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const uint64_t x = ffma2(f32x2(__uint_as_float(e < 16 ? sr[e] : sr2[e - 16]),
                                           __uint_as_float(e < 16 ? sr[e + 1] : sr2[e - 15])),
                                     sl2, nl2);
            const uint64_t pp = f32x2(ex2_approx(f32x2_lo(x)), ex2_approx(f32x2_hi(x)));
            const uint64_t dd = fadd2(f32x2(__uint_as_float(e < 16 ? dr[e] : dr2[e - 16]),
                                            __uint_as_float(e < 16 ? dr[e + 1] : dr2[e - 15])),
                                      nd2);
            const uint64_t z = fmul2(pp, dd);
            pk[e / 2] = pack_bf16x2(f32x2_lo(z), f32x2_hi(z));
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            float p0 = ex2_approx(fmaf(__uint_as_float(e < 16 ? sr[e] : sr2[e - 16]), scale_log2,
                                       -lse2));
            float p1 = ex2_approx(fmaf(__uint_as_float(e < 16 ? sr[e + 1] : sr2[e - 15]),
                                       scale_log2, -lse2));
            if (!rv || e >= valid) p0 = 0.f;
            if (!rv || e + 1 >= valid) p1 = 0.f;
            const float d_a = __uint_as_float(e < 16 ? dr[e] : dr2[e - 16]);
            const float d_b = __uint_as_float(e < 16 ? dr[e + 1] : dr2[e - 15]);
            pk[e / 2] = pack_bf16x2(p0 * (d_a - drow), p1 * (d_b - drow));
          }
        }
        // dS over the first 16 of the 32 S columns this thread read.
        SPARGE_TMEM_ST_X16(sb, pk);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(C::B_DSF + 4 * b + cg));
      }
      if (!ok) break;
      // Epilogue: read this warp's dQ columns, release the accumulator to the
      // next q-block's dQ MMAs, then scale, convert and store.
      const int gl = g - 1;
      if (!warp_wait(bar(C::B_SE + (gl & 1)), (gl >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t ro[D / 4];
#pragma unroll
      for (int c = 0; c < D / 4; c += 16) SPARGE_TMEM_LD_X16(lane_base + C::col_dq + cg * (D / 4) + c, (ro + c));
#pragma unroll
      for (int c = 0; c < D / 4; c += 16) SPARGE_TMEM_WAIT_LD16((ro + c));
      tc_fence_before();
      mbar_arrive(bar(C::B_DQE));
      ++j;
      if (rv) {
#pragma unroll
        for (int c = 0; c < D / 4; c += 8) {
          uint4 w;
          w.x = pack_bf16x2(__uint_as_float(ro[c + 0]) * scale, __uint_as_float(ro[c + 1]) * scale);
          w.y = pack_bf16x2(__uint_as_float(ro[c + 2]) * scale, __uint_as_float(ro[c + 3]) * scale);
          w.z = pack_bf16x2(__uint_as_float(ro[c + 4]) * scale, __uint_as_float(ro[c + 5]) * scale);
          w.w = pack_bf16x2(__uint_as_float(ro[c + 6]) * scale, __uint_as_float(ro[c + 7]) * scale);
          __stcs(reinterpret_cast<uint4*>(qrow + cg * (D / 4) + c), w);
        }
      }
    }
    if (!ok) report_error(status, SPARGE_ERR_TIMEOUT);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == R::kIssueA) {
    tc_fence_after();
    tmem_dealloc(tmem, C::tmem_cols);
    // Started early beside the dK/dV grid: the grid completes only after that
    // one has, so work after this call sees dK and dV written.
    if (blockIdx.x == 0 && threadIdx.x == R::kIssueA * 32)
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
  // Key tiles of 128 keys: pairs of 64-key kv-blocks, or 128-key blocks.
  const int kv_per_tile = g.bk == 64 ? 2 : 1;
  const int Mt = (g.Mk + kv_per_tile - 1) / kv_per_tile;
  const unsigned ndelta = static_cast<unsigned>((rows + RPB - 1) / RPB);
  // Both gradient kernels are persistent: one CTA per SM (or per work item
  // when there are fewer), taking items from their work counters.
  int dev = 0, nsm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const TileItems items{ws.item_tile, ws.item_part, ws.item_work,   ws.seq_tile,
                        ws.seq_part,  ws.work + 2,   ws.split_cnt, ws.split_part};
  bwd_plan_kernel<<<2, kPlanThreads, 0, st>>>(col_cnt, g.BH, g.Mk, Mt, kv_per_tile, items, nsm,
                                               g.Mq, kSplitSlots, row_cnt, g.BH * g.Mq,
                                               ws.row_order, ws.work);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(max(1u, ndelta));
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, bwd_delta_kernel<D>, static_cast<const __nv_bfloat16*>(o),
                           static_cast<const __nv_bfloat16*>(dout), rows, delta);
    if (e != cudaSuccess) return e;
  }

  // Q and dO in 128-row boxes for the dQ kernel, 64-row boxes (query
  // halves) for the dK/dV kernel; K and V in 64-row boxes.
  CUtensorMap tq, tk, tv, tdo, tq64, tdo64;
  if (make_tmap_bf16(&tq, q, g.BH, g.N, D, kBM) != 0 || make_tmap_bf16(&tk, k, g.BH, g.N, D, kBN) != 0 ||
      make_tmap_bf16(&tv, v, g.BH, g.N, D, kBN) != 0 ||
      make_tmap_bf16(&tdo, dout, g.BH, g.N, D, kBM) != 0 ||
      make_tmap_bf16(&tq64, q, g.BH, g.N, D, 64) != 0 ||
      make_tmap_bf16(&tdo64, dout, g.BH, g.N, D, 64) != 0)
    return cudaErrorInvalidValue;
  const float scale_log2 = scale * kLog2e;

  e = cudaFuncSetAttribute(bwd_dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           DkdvCfg<D>::smem_alloc);
  if (e != cudaSuccess) return e;
  // Up to kSplitSlots more items than tiles (the parts of cut tiles).
  const int ntiles = g.BH * Mt;
  bwd_dkdv_kernel<D><<<static_cast<unsigned>(max(1, min(ntiles + kSplitSlots, nsm))),
                       Roles<kDkdvWarps>::kThreads, DkdvCfg<D>::smem_alloc, st>>>(
      tq64, tk, tv, tdo64, lse, delta, col_idx, col_cnt, items, ntiles, ws.work + 1, g.N,
      g.Mq, g.Mk, Mt, kv_per_tile, scale, scale_log2, static_cast<__nv_bfloat16*>(dk),
      static_cast<__nv_bfloat16*>(dv), status);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  e = cudaFuncSetAttribute(bwd_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           DqCfg<D>::smem_alloc);
  if (e != cudaSuccess) return e;
  // Programmatic dependent launch: the dQ CTAs may start while the last dK/dV
  // CTAs run (D and the launch orders were complete before dK/dV started).
  const int nq = g.BH * g.Mq;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(max(1, min(nq, nsm))));
  cfg.blockDim = dim3(Roles<kDqWarps>::kThreads);
  cfg.dynamicSmemBytes = DqCfg<D>::smem_alloc;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, bwd_dq_kernel<D>, tq, tk, tv, tdo, lse,
                            static_cast<const float*>(delta), row_idx, row_cnt,
                            static_cast<const int32_t*>(ws.row_order), nq, ws.work, g.N, g.Mq,
                            g.Mk, g.bk == 64 ? 1 : 2, scale, scale_log2,
                            static_cast<__nv_bfloat16*>(dq), status);
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

// Sizes of the workspace parts, in layout order.
constexpr int kWsParts = 10;
void bwd_workspace_parts(const Geom& g, size_t (&sz)[kWsParts]) {
  const int kv_per_tile = g.bk == 64 ? 2 : 1;
  const size_t nitems = (size_t)g.BH * ((g.Mk + kv_per_tile - 1) / kv_per_tile) + kSplitSlots;
  sz[0] = align256((size_t)g.BH * g.N * sizeof(float));            // delta
  sz[1] = align256((size_t)g.BH * g.Mq * sizeof(int32_t));         // q-block order
  sz[2] = align256(4 * sizeof(int32_t));                             // counters, item count
  for (int i = 3; i < 8; ++i) sz[i] = align256(nitems * sizeof(int32_t));  // item arrays
  sz[8] = align256(kSplitCounters * sizeof(int32_t));                // completion counters
  sz[9] = align256((size_t)kSplitSlots * kPair * 2 * g.d * sizeof(float));  // partials
}
}  // namespace

size_t bwd_workspace_bytes(const Geom& g) {
  size_t sz[kWsParts];
  bwd_workspace_parts(g, sz);
  size_t total = 0;
  for (size_t x : sz) total += x;
  return total;
}

BwdWorkspace bwd_workspace_layout(const Geom& g, void* base) {
  size_t sz[kWsParts];
  bwd_workspace_parts(g, sz);
  uint8_t* p[kWsParts];
  p[0] = static_cast<uint8_t*>(base);
  for (int i = 1; i < kWsParts; ++i) p[i] = p[i - 1] + sz[i - 1];
  BwdWorkspace w;
  w.delta = reinterpret_cast<float*>(p[0]);
  w.row_order = reinterpret_cast<int32_t*>(p[1]);
  w.work = reinterpret_cast<int32_t*>(p[2]);
  w.seq_tile = reinterpret_cast<int32_t*>(p[3]);
  w.seq_part = reinterpret_cast<int32_t*>(p[4]);
  w.item_tile = reinterpret_cast<int32_t*>(p[5]);
  w.item_part = reinterpret_cast<int32_t*>(p[6]);
  w.item_work = reinterpret_cast<int32_t*>(p[7]);
  w.split_cnt = reinterpret_cast<int32_t*>(p[8]);
  w.split_part = reinterpret_cast<float*>(p[9]);
  return w;
}

}  // namespace sparge
