// gqa_decode_umma.cuh — the GQA decode step on the fifth-generation tensor
// core (tcgen05) for units with many query rows: up to 64 query rows share
// one KV head (multi-query attention, wide groups, multi-token causal chunks).
//
// What one launch computes: the same as gqa_decode_kernel (softmax(scale *
// q . K^T) V for every query row over its sequence's cached tokens, query head
// h reading KV head floor(h / G); "Grouped Query Attention (GQA): Efficient
// Multi-Head Attention", Worked example 2 and Two extremes), for 16-bit
// caches with head_dim 128, contiguous or paged.
//
// Why a second kernel: with 32 or 64 query rows per KV head the warp-level
// mma.sync kernel spends more time in its products than HBM needs to deliver
// the tile (multi-query attention: 64 rows, eight times the 70B shape's math
// per byte).  Here one thread issues the products, their operands come
// straight from shared memory and the accumulators live in tensor memory.
//
// Products, transposed so that tensor-memory lanes index tokens and head
// dimensions (M = 128 for both, the lane-per-row layout):
//   S^T[token][row] = K_tile (128 x D, as loaded) . Q^T            M=128 N=NC
//   O^T[d][row]    += V_tile^T (D x 128 tokens) . P^T (128 x rows) M=128 N=64
//   L[any][row]    += ones (128 x 128 tokens) . P^T                 M=128 N=64
// The last one sums the probabilities of every row in every lane: the thread
// that owns O lane d finds its rows' sums beside it, with no reduction across
// threads.  P^T is written by the softmax threads (one thread per token and
// half of the rows: 32 or 16 probabilities) over the K half of the tile's
// ring stage, which the first product has finished reading.
//
// Warp roles (320 threads, one block per SM, persistent over a contiguous
// range of the flat tile list shared with gqa_decode_kernel, 128-token tiles):
//   warp 0     TMA producer: the unit's Q rows (two buffers) and K / V tiles
//              (three-stage ring of 64 KB: 2 x 32 KB, boxes of 64 tokens x
//              64 elements, 128-byte swizzle); L2 evict-first.  A paged cache
//              looks each 64-token box's page up in the block table.
//   warp 1     tensor-memory owner (allocation of all 512 columns) and MMA
//              issuer (one elected thread).
//   warps 2-9  two softmax warpgroups; warpgroup w owns rows [w NC/2,
//              (w+1) NC/2) of the unit, thread t of it tensor-memory lane t:
//              token t of S, head dimension t of O.  Online softmax in the
//              log2 domain with a lazy rescale: a warpgroup's running row
//              maxima m only move (and its O, L columns are rescaled) when a
//              score exceeds m by more than kRescaleLog2, so most tiles need
//              no cross-thread reduction at all; probabilities then stay
//              below 2^8.  The two warpgroups share nothing but the tile
//              barriers.
//   Unit end: O^T / L to the output rows.  A unit split between blocks
//   either leaves a normalised partial and its log2-sum-exp, merged by the
//   last block to arrive (as in gqa_decode_kernel), or — when the launch is
//   a cluster launch and every unit is split evenly over the CTAs of one
//   cluster — the CTAs put their states in shared memory and each merges a
//   slice of the rows from all of them through distributed shared memory:
//   no global partials, counters or fences.
//
// Every mbarrier wait is bounded (DecodeParams::wait_ns); on a give-up the
// block sets kErrWaitTimeout, stops waiting, still drains its bulk copies and
// products and frees its tensor memory before it exits.  The two cluster
// barriers of the shared-memory merge are not bounded waits: every thread of
// every CTA of the cluster takes part in both, and reaches them after
// bounded work only (its loop runs on after a give-up, skipping waits).
#pragma once

#include "gqa_decode_kernel.cuh"

namespace gqa {

constexpr int kUmmaTileTokens = 128;  // tokens per tile: M of every product
constexpr int kUmmaCols = 64;         // query rows per unit, padded: N
constexpr int kUmmaSoftmaxThreads = 256;
constexpr int kUmmaThreads = 64 + kUmmaSoftmaxThreads;
constexpr int kUmmaStages = 3;
constexpr int kUmmaD = 128;
// One 64-element half of head_dim for 128 tokens (rows of 128 bytes).
constexpr int kUmmaHalfBytes = kUmmaTileTokens * 128;       // 16 KB
constexpr int kUmmaTileBytes = 2 * kUmmaHalfBytes;          // K or V: 32 KB
constexpr int kUmmaStageBytes = 2 * kUmmaTileBytes;         // 64 KB
constexpr int kUmmaQBytes = 2 * kUmmaCols * 128;            // 16 KB
constexpr int kUmmaBoxBytes = 64 * 128;                     // one TMA box
constexpr int kUmmaTmemCols = 512;
// Tensor-memory columns: two S buffers, O, L and the all-ones operand.
constexpr int kTmS = 0, kTmO = 128, kTmL = 192, kTmOnes = 256;
constexpr float kRescaleLog2 = 8.f;   // lazy-rescale threshold (log2 units)
// Dynamic shared memory: ring, Q buffers, reduction rows, row vectors,
// barriers (16) and the tensor-memory address, plus alignment slack.
constexpr int kUmmaRingOff = 0;
constexpr int kUmmaQOff = kUmmaStages * kUmmaStageBytes;
constexpr int kUmmaRedOff = kUmmaQOff + 2 * kUmmaQBytes;    // [4][64] fp32
constexpr int kUmmaVecOff = kUmmaRedOff + 4 * 64 * 4;       // m, alpha [64]
constexpr int kUmmaBarOff = kUmmaVecOff + 2 * 64 * 4;
constexpr int kUmmaBars = 17;
constexpr int kUmmaSmemBytes = 1024 + kUmmaBarOff + kUmmaBars * 8 + 16;
static_assert(kUmmaSmemBytes + 256 <= 232448,
              "shared memory of the tensor-core kernel exceeds the limit");
// Named barriers: 1 and 3 the two softmax warpgroups, 4 both of them, 2 the
// MMA warp with both (tensor memory freed after the last read).
constexpr int kBarWg0 = 1, kBarTeardown = 2, kBarWg1 = 3, kBarSoftmax = 4;

// ------------------------------------------------------------- descriptors

enum : uint32_t { kUmmaSwizzle128 = 2 };  // layout-type field value

// Shared-memory matrix descriptor of a tcgen05 operand: start address, the
// leading / stride byte offsets (both >> 4), descriptor version 1 (bits
// 46-47) and the swizzle mode (bits 61-63).  For the K-major operands the
// stride offset is the distance between groups of 8 rows; for the MN-major
// ones the leading offset is the distance between 64-element chunks of M/N
// and the stride offset the distance between groups of 8 rows of K.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo,
                                              uint32_t sbo) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) |
         (1ull << 46) | (static_cast<uint64_t>(kUmmaSwizzle128) << 61);
}

// Instruction descriptor of a kind::f16 product: fp32 accumulator (bits 4-5
// = 1), A and B types (bits 7-9, 10-12: 0 f16, 1 bf16), A / B MN-major
// (bits 15, 16), N >> 3 (bits 17-22), M >> 4 (bits 24-28).
__host__ __device__ constexpr uint32_t umma_idesc(bool bf16, bool a_mn,
                                                  bool b_mn, int M, int N) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// The product with A taken from tensor memory (the all-ones operand).
__device__ __forceinline__ void umma_f16_ts(uint32_t d_tmem, uint32_t a_tmem,
                                            uint64_t b_desc, uint32_t idesc,
                                            bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(
          d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc),
      "r"(static_cast<uint32_t>(accumulate))
      : "memory");
}

// Warp reduce-scatter of NC per-lane values with `op` (NC = 16, 32 or 64):
// afterwards lane L holds the warp-wide result of column L >> 1 (NC = 16), L
// (NC = 32) or of columns 2L and 2L+1 (NC = 64) in v[0] (and v[1]).
// Halving exchanges: NC - 2 (NC = 64) or NC - 1 shuffles instead of NC x 5.
template <int NC, typename Op>
__device__ __forceinline__ void warp_reduce_scatter(float (&v)[NC], Op op) {
  static_assert(NC == 16 || NC == 32 || NC == 64, "16, 32 or 64 columns");
  const int lane = threadIdx.x & 31;
  constexpr int kLast = NC >= 32 ? NC / 32 : 1;
#pragma unroll
  for (int half = NC / 2, off = 16; half >= kLast; half >>= 1, off >>= 1) {
    const bool hi = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float keep = hi ? v[half + i] : v[i];
      const float send = hi ? v[i] : v[half + i];
      v[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, off));
    }
  }
  if constexpr (NC == 16) v[0] = op(v[0], __shfl_xor_sync(0xffffffffu, v[0], 1));
}

// ------------------------------------------------------------------ kernel

template <bool QBF16, int NC, bool PAGED>
__global__ void __launch_bounds__(kUmmaThreads, 1)
    gqa_decode_umma_kernel(const __grid_constant__ CUtensorMap map_k,
                           const __grid_constant__ CUtensorMap map_v,
                           const __grid_constant__ CUtensorMap map_q,
                           const DecodeParams p) {
  static_assert(NC == 32 || NC == 64, "rows per unit padded to 32 or 64");
  constexpr int TT = kUmmaTileTokens;
  constexpr int D = kUmmaD;
  constexpr int NH = NC / 2;  // rows of one softmax warpgroup
  constexpr int kKv = QBF16 ? kKvBF16 : kKvF16;
  constexpr uint32_t kIdescS = umma_idesc(QBF16, false, false, 128, NC);
  constexpr uint32_t kIdescO = umma_idesc(QBF16, true, true, 128, kUmmaCols);
  // the row-sum product: A (all ones) from tensor memory, not transposed
  constexpr uint32_t kIdescL = umma_idesc(QBF16, false, true, 128, kUmmaCols);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem + kUmmaRingOff;
  uint8_t* qbuf = smem + kUmmaQOff;
  float* red = reinterpret_cast<float*>(smem + kUmmaRedOff);   // [4][64]
  float* mrow = reinterpret_cast<float*>(smem + kUmmaVecOff);  // [64]
  float* arow = mrow + 64;                                     // [64]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kUmmaBarOff);
  uint64_t* full = bars;                   // [3]  TMA -> MMA
  uint64_t* empty = full + kUmmaStages;    // [3]  products done -> producer
  uint64_t* qfull = empty + kUmmaStages;   // [2]  Q landed -> MMA
  uint64_t* qempty = qfull + 2;            // [2]  unit's last S done -> producer
  uint64_t* sfull = qempty + 2;            // [2]  S ready -> softmax
  uint64_t* pfull = sfull + 2;             // [2]  P written -> MMA (8 warps)
  uint64_t* oready = pfull + 2;            // [2]  PV of tile i done (i & 1)
  uint64_t* mma_done = oready + 2;         // every product done (teardown)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kUmmaBars);

  __shared__ PlanSmem<kUmmaThreads> s_plan;
  __shared__ volatile int s_abort;
  __shared__ int s_npend;
  __shared__ int s_pend_u[2], s_pend_b[2], s_pend_j[2], s_pend_cf[2],
      s_pend_cl[2];
  __shared__ uint32_t s_pend_t[2];

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int HU = p.Hkv * p.NHC;

  if (warp == 0) {
    if (lane == 0) {
      ptx::prefetch_tensormap(&map_k);
      ptx::prefetch_tensormap(&map_v);
      ptx::prefetch_tensormap(&map_q);
    }
    // (a paged cache's pages are only known from the block table, which the
    // previous kernel may write)
    if constexpr (!PAGED)
      if (!(p.tune & 1))
        prefetch_first_tiles<kKv, D, 4, TT, true>(&map_k, &map_v, p, lane);
  }
  if (tid == 0) {
    for (int s = 0; s < kUmmaStages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&qfull[i], 1);
      ptx::mbar_init(&qempty[i], 1);
      ptx::mbar_init(&sfull[i], 1);
      ptx::mbar_init(&pfull[i], kUmmaSoftmaxThreads / 32);
    }
    ptx::mbar_init(&oready[0], 1);
    ptx::mbar_init(&oready[1], 1);
    ptx::mbar_init(mma_done, 1);
    ptx::fence_barrier_init();
    s_abort = 0;
    s_npend = 0;
    s_plan.found = 0;
    s_plan.b0 = 0;
    s_plan.L0 = 0;
    s_plan.pref0 = 0;
  }
  if (warp == 1) {
    // One block per SM (its shared memory excludes a second), so the whole
    // tensor memory is free.
    ptx::tmem_alloc(tmem_slot, kUmmaTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  prefetch_seq_lens(p, tid);
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();

  long long N, t0, t1;
  int P;
  TileWalkT<TT> w0;
  plan_block<kUmmaThreads, TT>(p, HU, s_plan, N, P, t0, t1, w0);
  // The shared-memory merge: a cluster launch whose block count splits every
  // unit evenly over one cluster's CTAs, and equal tile counts (plan_block
  // took the aligned count).  The same decision in every CTA of a cluster.
  const bool dsm = p.cluster > 1 && p.p_align == p.cluster * HU * p.B &&
                   P == p.p_align;

  if (warp == 0) {
    // =============================== producer ===============================
    if (lane == 0 && t0 < t1) {
      const uint64_t policy = ptx::policy_evict_first();
      TileWalkT<TT> w = w0;
      long long it = 0;
      int nq = 0;  // Q loads issued
      for (long long g = t0; g < t1; ++g, ++it) {
        const int kvh = w.j / p.NHC, hc = w.j % p.NHC;
        const int tok0 = w.ti * TT;
        // the second 64-token half only when it holds a valid token
        const int halves = tok0 + 64 < w.L ? 2 : 1;
        // paged: the boxes' block-table entries before the waits
        int pg[2] = {0, 0};
        if constexpr (PAGED) {
          for (int th = 0; th < halves; ++th)
            pg[th] = __ldg(p.block_table +
                           static_cast<size_t>(w.b) * p.max_pages +
                           (tok0 + th * 64) / p.page_size);
        }
        if (g == t0 || w.ti == 0) {
          // the unit's query rows: 64 rows from its first one (rows past
          // the unit are never used; past the tensor TMA fills zeros)
          const int qb = nq & 1;
          if (!ptx::mbar_wait_bounded(&qempty[qb], ((nq >> 1) & 1) ^ 1u,
                                      p.wait_ns)) {
            atomicOr(p.error, kErrWaitTimeout);
            s_abort = 1;
            break;
          }
          const int row = (w.b * p.Hq + kvh * p.G) * p.T + hc * p.R;
          uint8_t* dq = qbuf + qb * kUmmaQBytes;
          ptx::mbar_arrive_expect_tx(&qfull[qb], kUmmaQBytes);
          ptx::tma_load_2d(dq, &map_q, &qfull[qb], 0, row, policy);
          ptx::tma_load_2d(dq + kUmmaQBytes / 2, &map_q, &qfull[qb], 64, row,
                           policy);
          ++nq;
        }
        const int stage = static_cast<int>(it % kUmmaStages);
        const uint32_t ph = static_cast<uint32_t>((it / kUmmaStages) & 1);
        if (!ptx::mbar_wait_bounded(&empty[stage], ph ^ 1u, p.wait_ns)) {
          atomicOr(p.error, kErrWaitTimeout);
          s_abort = 1;
          break;
        }
        if (s_abort) break;
        ptx::mbar_arrive_expect_tx(&full[stage], halves * 4 * kUmmaBoxBytes);
        uint8_t* ks = ring + stage * kUmmaStageBytes;
        uint8_t* vs = ks + kUmmaTileBytes;
        for (int th = 0; th < halves; ++th) {
          // tile coordinates in the cache view [planes][tokens][D]
          int row = tok0 + th * 64, plane = w.b * p.Hkv + kvh;
          if constexpr (PAGED) {
            int pgv = pg[th];
            if (pgv < 0 || pgv >= p.num_pages) {
              atomicOr(p.error, kErrBadPage);
              pgv = 0;
            }
            row = row % p.page_size;
            plane = pgv * p.Hkv + kvh;
          }
#pragma unroll
          for (int dh = 0; dh < 2; ++dh) {
            const int off = dh * kUmmaHalfBytes + th * kUmmaBoxBytes;
            ptx::tma_load_3d(ks + off, &map_k, &full[stage], dh * 64, row,
                             plane, policy);
            ptx::tma_load_3d(vs + off, &map_v, &full[stage], dh * 64, row,
                             plane, policy);
          }
        }
        w.next(p, HU);
      }
      // Never leave the block with bulk copies still writing its memory.
      const long long issued = it;
      for (int s = 0; s < kUmmaStages; ++s) {
        const long long uses =
            issued > s ? (issued - s + kUmmaStages - 1) / kUmmaStages : 0;
        if (uses > 0)
          ptx::mbar_wait_bounded(&full[s],
                                 static_cast<uint32_t>((uses - 1) & 1),
                                 kDrainLimitNs);
      }
      for (int qb = 0; qb < 2; ++qb) {
        const int uses = (nq + 1 - qb) / 2;
        if (uses > 0)
          ptx::mbar_wait_bounded(&qfull[qb],
                                 static_cast<uint32_t>((uses - 1) & 1),
                                 kDrainLimitNs);
      }
    }
    __syncwarp();
    if (dsm) {
      // every thread of the cluster takes part in its two barriers
      ptx::cluster_sync();
      ptx::cluster_sync();
    }
    return;
  }

  if (warp == 1) {
    // ============================ MMA issuer ================================
    if (lane == 0 && t0 < t1) {
      const uint32_t ring_s = ptx::smem_u32(ring);
      const uint32_t q_s = ptx::smem_u32(qbuf);
      TileWalkT<TT> w = w0;
      long long it = 0;
      int ui = -1;          // unit index within the block
      bool aborted = false;
      bool pv_pending = false, pv_first = false;
      int pv_stage = 0;
      long long pv_it = 0;
      auto fail = [&]() {
        atomicOr(p.error, kErrWaitTimeout);
        s_abort = 1;
        aborted = true;
      };
      // O^T += V^T P^T and L += ones P^T for tile pv_it, once its
      // probabilities are in shared memory; then its stage is free.
      auto issue_pv = [&]() {
        if (!ptx::mbar_wait_bounded(&pfull[pv_it & 1],
                                    static_cast<uint32_t>((pv_it >> 1) & 1),
                                    p.wait_ns)) {
          fail();
          return;
        }
        ptx::tc_fence_after();
        const uint32_t st = ring_s + pv_stage * kUmmaStageBytes;
#pragma unroll
        for (int k = 0; k < TT / 16; ++k) {
          const uint64_t pd = umma_desc(st + k * 2048, kUmmaHalfBytes, 1024);
          const uint64_t vd = umma_desc(st + kUmmaTileBytes + k * 2048,
                                        kUmmaHalfBytes, 1024);
          const bool acc = !(pv_first && k == 0);
          ptx::umma_f16_ss(tmem + kTmO, vd, pd, kIdescO, acc);
          umma_f16_ts(tmem + kTmL, tmem + kTmOnes + 8 * k, pd, kIdescL, acc);
        }
        ptx::umma_commit(&empty[pv_stage]);
        ptx::umma_commit(&oready[pv_it & 1]);
        pv_pending = false;
      };
      for (long long g = t0; g < t1 && !aborted; ++g, ++it) {
        const bool first = (g == t0) || (w.ti == 0);
        const bool last = (w.ti == w.nt - 1) || (g == t1 - 1);
        if (first) {
          ++ui;
          if (!ptx::mbar_wait_bounded(&qfull[ui & 1],
                                      static_cast<uint32_t>((ui >> 1) & 1),
                                      p.wait_ns)) {
            fail();
            break;
          }
        }
        const int stage = static_cast<int>(it % kUmmaStages);
        if (!ptx::mbar_wait_bounded(
                &full[stage],
                static_cast<uint32_t>((it / kUmmaStages) & 1), p.wait_ns)) {
          fail();
          break;
        }
        ptx::tc_fence_after();
        // ---- S^T = K Q^T into S buffer it & 1 (K = head_dim, 8 steps) ----
        const uint32_t st = ring_s + stage * kUmmaStageBytes;
        const uint32_t qs = q_s + (ui & 1) * kUmmaQBytes;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t koff = (k >> 2) * kUmmaHalfBytes + (k & 3) * 32;
          const uint32_t qoff = (k >> 2) * (kUmmaQBytes / 2) + (k & 3) * 32;
          ptx::umma_f16_ss(tmem + kTmS + (it & 1) * 64,
                           umma_desc(st + koff, 16, 1024),
                           umma_desc(qs + qoff, 16, 1024), kIdescS, k > 0);
        }
        ptx::umma_commit(&sfull[it & 1]);
        if (last) ptx::umma_commit(&qempty[ui & 1]);
        // ---- the previous tile's PV (it ran its softmax meanwhile) ----
        if (pv_pending) issue_pv();
        if (aborted) break;
        pv_pending = true;
        pv_first = first;
        pv_stage = stage;
        pv_it = it;
        // the last tile of a unit: its PV now, not behind the next tile
        if (last) issue_pv();
        w.next(p, HU);
      }
      if (pv_pending && !aborted) issue_pv();
      // every product issued has finished before tensor memory is freed
      ptx::umma_commit(mma_done);
      ptx::mbar_wait_bounded(mma_done, 0, kDrainLimitNs);
    }
    __syncwarp();
    if (dsm) {
      // the two cluster barriers of the shared-memory merge
      ptx::cluster_sync();
      ptx::cluster_sync();
    }
    ptx::tc_fence_before();
    ptx::named_bar_sync(kBarTeardown, 32 + kUmmaSoftmaxThreads);
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kUmmaTmemCols);
    return;
  }

  // ============================ softmax warpgroups ==========================
  const int st_id = tid - 64;               // 0 .. 255
  const int wg = st_id >> 7;                // warpgroup: rows [wg NH, +NH)
  const int wt = st_id & 127;               // thread within the warpgroup
  const int cb = wg * NH;                   // first row (column) of it
  const int bar_wg = wg ? kBarWg1 : kBarWg0;
  const int q4 = warp & 3;                  // tensor-memory lane quarter
  const int t = q4 * 32 + lane;             // this thread's lane
  const uint32_t tlane = static_cast<uint32_t>(q4 * 32) << 16;

  // all-ones operand of the row-sum product (every lane, 64 columns; each
  // warpgroup stores 32 of them)
  {
    uint32_t ones[32];
    const uint32_t one2 = QBF16 ? 0x3F803F80u : 0x3C003C00u;
#pragma unroll
    for (int i = 0; i < 32; ++i) ones[i] = one2;
    ptx::tmem_st32(tmem + tlane + kTmOnes + 32 * wg, ones);
    ptx::tmem_wait_st();
  }
  // Sequences with no valid token: all-zero output rows.
  for (int b = blockIdx.x; b < p.B; b += gridDim.x) {
    if (clamp_len(__ldg(p.seq_lens + b), p.Smax) != 0) continue;
    const size_t base = static_cast<size_t>(b) * p.Hq * p.T * D;
    for (int i = st_id; i < p.Hq * p.T * D; i += kUmmaSoftmaxThreads)
      store_out<QBF16>(p.out, base + i, 0.f);
  }
  // (The ones reach tensor memory before the first row-sum product reads
  // them: every softmax warp stores its part before its first pfull
  // arrival, which the MMA thread waits for before that product.)

  // shared-memory merge: this CTA's state (rows x D fp32 over the first 32
  // KB of the ring, row maxima and sums in the reduction rows)
  float* dmp_o = reinterpret_cast<float*>(ring);
  float* dmp_m = red;
  float* dmp_l = red + 64;
  if (dsm && t0 >= t1) {
    // a CTA of the cluster with no tile: an empty state
    if (st_id < kUmmaCols) {
      dmp_m[st_id] = -INFINITY;
      dmp_l[st_id] = 0.f;
    }
  }

  if (st_id == 0 && t0 < t1) prefetch_range_q<D, TT>(p, HU, w0, t0, t1);
  if (t0 < t1) {
    TileWalkT<TT> w = w0;
    long long it = 0;
    long long pv_waited = 0;  // completed PV products consumed (oready phases)
    bool aborted = false;
    const float sl2 = p.scale_log2;
    auto wait_ok = [&](uint64_t* bar, uint32_t parity) {
      if (aborted) return;
      if (!__all_sync(0xffffffffu,
                      ptx::mbar_wait_bounded(bar, parity, p.wait_ns))) {
        atomicOr(p.error, kErrWaitTimeout);
        s_abort = 1;
        aborted = true;
      }
    };
    // PV(i) (block tile index) has completed.  The PV products alternate
    // between two barriers; each barrier's phases are consumed in order and
    // never more than one behind, as parity waits require: PV(i + 2) cannot
    // complete before this thread publishes P(i + 2), and by then PV(i) has
    // been waited for.
    auto wait_pv = [&](long long i) {
      while (pv_waited <= i) {
        wait_ok(&oready[pv_waited & 1],
                static_cast<uint32_t>((pv_waited >> 1) & 1));
        ++pv_waited;
      }
    };

    for (long long g = t0; g < t1; ++g, ++it) {
      const bool first = (g == t0) || (w.ti == 0);
      const bool last = (w.ti == w.nt - 1) || (g == t1 - 1);
      const int kvh = w.j / p.NHC, hc = w.j % p.NHC;
      const int Rv = min(p.R, p.GR - hc * p.R);  // valid rows of the unit
      const int stage = static_cast<int>(it % kUmmaStages);
      const int L = w.L;
      const int tok = w.ti * TT + t;

      // ---- scores of this thread's token for the warpgroup's rows ----
      wait_ok(&sfull[it & 1], static_cast<uint32_t>((it >> 1) & 1));
      ptx::tc_fence_after();
      const bool tail = (w.ti * TT + TT - 1) > L - p.T;
      // x = scale * log2(e) * s, or -inf for keys a row may not see: past
      // the sequence, or (multi-token chunk) past the row's token, t <=
      // L - T + i; padded rows see nothing
      auto load_scores = [&](float (&x)[NH]) {
        uint32_t r[NH];
        ptx::tmem_ld<NH>(tmem + tlane + kTmS + (it & 1) * 64 + cb, r);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < NH; ++c) x[c] = __uint_as_float(r[c]) * sl2;
        if (tail) {
          const int dt = tok - (L - p.T);
          int ic = (hc * p.R + cb) % p.T;
#pragma unroll
          for (int c = 0; c < NH; ++c) {
            if (cb + c >= Rv || dt > ic) x[c] = -INFINITY;
            ic = (ic + 1 == p.T) ? 0 : ic + 1;
          }
        } else if (Rv < cb + NH) {
#pragma unroll
          for (int c = 0; c < NH; ++c)
            if (cb + c >= Rv) x[c] = -INFINITY;
        }
      };
      float x[NH];
      load_scores(x);

      // ---- lazy rescale: only when a score passes m + kRescaleLog2 ----
      bool over = false;
#pragma unroll
      for (int c = 0; c < NH; c += 4) {
        const float4 mv = *reinterpret_cast<const float4*>(mrow + cb + c);
        over |= (x[c] > mv.x + kRescaleLog2) | (x[c + 1] > mv.y + kRescaleLog2) |
                (x[c + 2] > mv.z + kRescaleLog2) |
                (x[c + 3] > mv.w + kRescaleLog2);
      }
      const bool need = ptx::named_bar_or(bar_wg, 128, over) || first;
      if (need) {
        // new row maxima: the tile's column maxima over the 128 tokens (the
        // reduction consumes x; the scores are loaded again afterwards)
        warp_reduce_scatter<NH>(x, [](float a, float b) { return fmaxf(a, b); });
        if constexpr (NH == 32) {
          red[q4 * 64 + cb + lane] = x[0];
        } else {
          if ((lane & 1) == 0) red[q4 * 64 + cb + (lane >> 1)] = x[0];
        }
        ptx::named_bar_sync(bar_wg, 128);
        if (wt < NH) {
          const int col = cb + wt;
          const float tm = fmaxf(fmaxf(red[col], red[64 + col]),
                                 fmaxf(red[128 + col], red[192 + col]));
          const float mo = first ? -INFINITY : mrow[col];
          const float mn = fmaxf(mo, tm);
          arow[col] = mn == -INFINITY ? 1.f : ptx::ex2(mo - mn);
          mrow[col] = mn;
        }
        ptx::named_bar_sync(bar_wg, 128);
        if (!first) {
          // rescale this warpgroup's O and L columns before the tile's PV
          // adds to them (the previous tile's PV must have finished)
          if (it >= 1) wait_pv(it - 1);
          ptx::tc_fence_after();
          uint32_t o[NH], lr[NH];
          const uint32_t oa = tmem + tlane + kTmO + cb;
          const uint32_t la = tmem + tlane + kTmL + cb;
          ptx::tmem_ld<NH>(oa, o);
          ptx::tmem_ld<NH>(la, lr);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < NH; ++c) {
            const float a = arow[cb + c];
            o[c] = __float_as_uint(__uint_as_float(o[c]) * a);
            lr[c] = __float_as_uint(__uint_as_float(lr[c]) * a);
          }
          ptx::tmem_st<NH>(oa, o);
          ptx::tmem_st<NH>(la, lr);
          ptx::tmem_wait_st();
        }
        load_scores(x);
      }
      // The probabilities do not wait for the previous tile's PV (it reads
      // another stage): only PV(it - 2), on the barrier PV(it) completes.
      if (it >= 2) wait_pv(it - 2);

      // ---- probabilities into P^T (this token's row of the stage's K half;
      // the warpgroup's NH rows = NH * 2 bytes)
      uint32_t pw[NH / 2];
#pragma unroll
      for (int c = 0; c < NH; c += 4) {
        const float4 mv = *reinterpret_cast<const float4*>(mrow + cb + c);
        const float m4[4] = {mv.x, mv.y, mv.z, mv.w};
        float pr[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          pr[e] = x[c + e] > -INFINITY ? ptx::ex2(x[c + e] - m4[e]) : 0.f;
        pw[c / 2] = ptx::pack2<QBF16>(pr[0], pr[1]);
        pw[c / 2 + 1] = ptx::pack2<QBF16>(pr[2], pr[3]);
      }
      uint8_t* st_base = ring + stage * kUmmaStageBytes;
      uint8_t* prow = st_base + t * 128;
      constexpr int kChunks = NH / 8;     // 16-byte chunks of this warpgroup
      const int ch0 = cb / 8;
#pragma unroll
      for (int ch = 0; ch < kChunks; ++ch) {
        const uint4 v = make_uint4(pw[4 * ch], pw[4 * ch + 1], pw[4 * ch + 2],
                                   pw[4 * ch + 3]);
        *reinterpret_cast<uint4*>(prow + (((ch0 + ch) ^ (t & 7)) << 4)) = v;
      }
      if constexpr (NC < kUmmaCols) {
        // the rows past NC of the 64-column product: zero probabilities
        // (their output columns are never read; zeros keep them finite)
        const int zc0 = NC / 8 + wg * (kUmmaCols - NC) / 16;
#pragma unroll
        for (int ch = 0; ch < (kUmmaCols - NC) / 16; ++ch)
          *reinterpret_cast<uint4*>(prow + (((zc0 + ch) ^ (t & 7)) << 4)) =
              make_uint4(0u, 0u, 0u, 0u);
      }
      // a V row past the sequence may hold anything (NaN): zero it, so that
      // its zero probability contributes exactly zero (each warpgroup one
      // 64-element half of the row)
      if (tok >= L) {
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
        uint4* vrow = reinterpret_cast<uint4*>(
            st_base + kUmmaTileBytes + wg * kUmmaHalfBytes + t * 128);
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) vrow[ch] = z;
      }
      ptx::fence_proxy_async_shared();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&pfull[it & 1]);

      if (last) {
        // ============== unit end: O^T / L to the output rows ===============
        wait_pv(it);
        ptx::tc_fence_after();
        uint32_t o[NH], lr[NH];
        ptx::tmem_ld<NH>(tmem + tlane + kTmO + cb, o);
        ptx::tmem_ld<NH>(tmem + tlane + kTmL + cb, lr);
        ptx::tmem_wait_ld();
        if (dsm) {
          // this CTA's state for the cluster merge: O^T columns as rows of
          // the dump, the row maxima and sums
#pragma unroll
          for (int c = 0; c < NH; ++c)
            dmp_o[(cb + c) * D + t] = __uint_as_float(o[c]);
          if (wt == 0) {
#pragma unroll
            for (int c = 0; c < NH; ++c) {
              dmp_m[cb + c] = mrow[cb + c];
              dmp_l[cb + c] = __uint_as_float(lr[c]);
            }
          }
        } else {
          const size_t rbase =
              (static_cast<size_t>(w.b) * p.Hq +
               static_cast<size_t>(kvh) * p.G) * p.T +
              static_cast<size_t>(hc) * p.R;
          const long long us = w.pref + static_cast<long long>(w.j) * w.nt;
          const int u = w.b * HU + w.j;
          const int cf = block_of_tile(us, N, P);
          const int cl = block_of_tile(us + w.nt - 1, N, P);
          const bool whole = cf == cl;
          const size_t slot = static_cast<size_t>(blockIdx.x) + u;
#pragma unroll
          for (int c = 0; c < NH; ++c) {
            const int row = cb + c;
            if (row >= Rv) continue;
            const float lv = __uint_as_float(lr[c]);
            const float val =
                lv > 0.f ? __uint_as_float(o[c]) * __fdividef(1.f, lv) : 0.f;
            if (whole)
              store_out<QBF16>(p.out, (rbase + row) * D + t, val);
            else
              p.part_o[(slot * kUmmaCols + row) * D + t] = val;
          }
          if (!whole && q4 == 0 && lane < NH) {
            // log2-sum-exp of row cb + lane
            float lv = 0.f;
#pragma unroll
            for (int c = 0; c < NH; ++c)
              lv = (c == lane) ? __uint_as_float(lr[c]) : lv;
            const int row = cb + lane;
            p.part_lse[slot * kUmmaCols + row] =
                lv > 0.f ? mrow[row] + ptx::lg2(lv) : -INFINITY;
          }
          // partial stores before the arrival (released by it)
          ptx::named_bar_sync(kBarSoftmax, kUmmaSoftmaxThreads);
          if (!whole && st_id == 0 && s_npend < 2) {
            const int k = s_npend;
            s_pend_t[k] = arrive_unit(p, u, cl - cf + 1);
            s_pend_u[k] = u;
            s_pend_b[k] = w.b;
            s_pend_j[k] = w.j;
            s_pend_cf[k] = cf;
            s_pend_cl[k] = cl;
            s_npend = k + 1;
          }
        }
      }
      w.next(p, HU);
    }

    // ---- split combines of the units whose last arrival was this block's
    // (the acquire side of the arrivals: st_id 0's swap, then the barrier) --
    ptx::named_bar_sync(kBarSoftmax, kUmmaSoftmaxThreads);
    for (int i = 0; i < s_npend; ++i)
      if (s_pend_t[i] == static_cast<uint32_t>(s_pend_cl[i] - s_pend_cf[i]))
        combine_unit<kKv, QBF16, D, 4, kUmmaSoftmaxThreads>(
            st_id, p, s_pend_u[i], s_pend_b[i], s_pend_j[i], s_pend_cf[i],
            s_pend_cl[i]);
  }

  if (dsm) {
    // ======= cluster merge: CTA r of the unit's k writes rows [r R/k, ...)
    ptx::cluster_sync();  // every CTA's state is in its shared memory
    const int k = p.cluster;
    const uint32_t rank = ptx::cluster_ctarank();
    const int u = static_cast<int>(blockIdx.x) / k;  // the cluster's unit
    const int b = u / HU, j = u % HU;
    const int kvh = j / p.NHC, hc = j % p.NHC;
    const int Rv = min(p.R, p.GR - hc * p.R);
    const int rpc = NC / k;                          // rows per CTA
    const size_t rbase =
        (static_cast<size_t>(b) * p.Hq + static_cast<size_t>(kvh) * p.G) *
            p.T + static_cast<size_t>(hc) * p.R;
    const uint32_t o_s = ptx::smem_u32(dmp_o), m_s = ptx::smem_u32(dmp_m),
                   l_s = ptx::smem_u32(dmp_l);
    constexpr int kG = D / 8;                        // 8-column items per row
    for (int i = st_id; i < rpc * kG; i += kUmmaSoftmaxThreads) {
      const int row = static_cast<int>(rank) * rpc + i / kG;
      const int n = i % kG;
      if (row >= Rv) continue;
      // every CTA's values first (independent loads in flight together),
      // then the arithmetic
      float mv[4], lv[4];
      float4 ov[4][2];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        if (r < k) {
          const uint32_t a =
              ptx::mapa_shared(o_s + (row * D + 8 * n) * 4, r);
          mv[r] = ptx::ld_dsmem_f32(ptx::mapa_shared(m_s + row * 4, r));
          lv[r] = ptx::ld_dsmem_f32(ptx::mapa_shared(l_s + row * 4, r));
          ov[r][0] = ptx::ld_dsmem_f4(a);
          ov[r][1] = ptx::ld_dsmem_f4(a + 16);
        } else {
          mv[r] = -INFINITY;
          lv[r] = 0.f;
          ov[r][0] = ov[r][1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      float M = -INFINITY;
#pragma unroll
      for (int r = 0; r < 4; ++r) M = fmaxf(M, mv[r]);
      float acc[8];
#pragma unroll
      for (int x = 0; x < 8; ++x) acc[x] = 0.f;
      float lt = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          if (mv[r] == -INFINITY) continue;
          const float f = ptx::ex2(mv[r] - M);
          lt += f * lv[r];
          acc[0] += f * ov[r][0].x;
          acc[1] += f * ov[r][0].y;
          acc[2] += f * ov[r][0].z;
          acc[3] += f * ov[r][0].w;
          acc[4] += f * ov[r][1].x;
          acc[5] += f * ov[r][1].y;
          acc[6] += f * ov[r][1].z;
          acc[7] += f * ov[r][1].w;
        }
      }
      store_out8<QBF16>(p.out, (rbase + row) * D + 8 * n, acc,
                        lt > 0.f ? 1.f / lt : 0.f);
    }
    ptx::cluster_sync();  // no CTA leaves while another reads its state
  }
  // tensor memory is freed by warp 1 once every softmax thread is done with it
  ptx::tc_fence_before();
  ptx::named_bar_sync(kBarTeardown, 32 + kUmmaSoftmaxThreads);
}

}  // namespace gqa
