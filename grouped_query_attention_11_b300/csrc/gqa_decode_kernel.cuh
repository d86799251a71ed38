// gqa_decode_kernel.cuh — the split-sequence GQA decode kernel for sm_103a.
//
// What one launch computes: for every sequence b, KV head j and query head h
// of j's group (h = j*G .. j*G+G-1), softmax(scale * q[b,h] . K[b,j,t]) over
// the t < seq_lens[b] cached tokens, applied to V[b,j,t] ("Grouped Query
// Attention (GQA): Efficient Multi-Head Attention", Worked example 2 and Two
// extremes; the head-to-KV-head mapping of "Llama-2 70B uses 64 query heads
// ...", What the choice does to attention).
//
// How (design for B300, not taken from the pages):
//
//  * Work units.  A unit is (sequence b, KV head j, chunk of <= 64 query heads
//    of j's group).  Its tokens are cut into 64-token tiles.  All tiles of all
//    units form one flat list (sequence-major), computed on the device from
//    seq_lens by every block: no host sync, ragged lengths cost nothing extra.
//  * Persistent blocks.  The grid is one wave of blocks; block c takes the
//    contiguous tile range [c*N/P, (c+1)*N/P).  Every block streams the same
//    number of KV bytes (+-1 tile), whatever the length mix.  A unit cut by a
//    range boundary is finished by the fused split combine below.  When all
//    sequences have the same tile count, P is a host-chosen count that puts
//    the range boundaries on unit boundaries (see DecodeParams::p_align).
//  * Warp roles.  A block is three warpgroups.  Warpgroup 0: one producer
//    warp and three merge warps; warpgroups 1 and 2: eight consumer warps.
//    setmaxnreg moves registers from warpgroup 0 (56 per thread) to the
//    consumers (224) for their mma fragments, accumulators and query rows.
//  * Launch overlap.  Launched as a programmatic dependent: before
//    griddepcontrol.wait a block only initialises barriers and asks L2 for
//    seq_lens, its first tiles (cp.async.bulk.prefetch.tensor) and its first
//    unit's query rows, which overlaps the previous kernel's last blocks;
//    every global read comes after the wait.
//  * KV stream.  The producer warp issues TMA tensor loads (128-byte
//    swizzle, L2 evict-first) of the K and V tiles into a multi-stage shared
//    memory ring guarded by mbarriers.  Each KV byte is read from HBM once and
//    serves all query heads of its group from shared memory.
//  * Group-batched math.  Consumer warps hold the group's query rows as mma
//    A fragments (16 rows per head block; G < 16 pads with zero rows) and run
//    QK^T and PV through mma.sync m16n8k16 with fp32 accumulation.  The online
//    softmax (running row max, rescale, row sum) lives in registers; row
//    reductions are two quad shuffles.  Narrow rows (NR: 8-bit caches with at
//    most 8 query rows a unit) swap the operands: keys and head dimensions
//    on the mma rows, the unit's rows on its 8 columns (S^T = K Q^T, O^T +=
//    V^T P^T with P^T from movmatrix), halving the padded mma work.
//  * Consumer groups.  The consumer warps form groups (two of four warps, or
//    four of two for the 8-bit caches with one head block) that take the
//    ring's stages in turn, each with its own softmax state, so that one
//    group's dependent mma / exp chains overlap the others'.
//  * Asynchronous unit epilogue.  At the end of a unit every consumer warp
//    only dumps its softmax state to shared memory (its rows normalised,
//    row-major) and signals an mbarrier; it goes straight on with the next
//    unit, whose query rows it has already started loading.  The merge warps combine the eight
//    states, write the output rows or a split partial, and publish the
//    block's arrival, off the consumers' critical path.
//  * FP8 cache (E4M3 or E5M2).  Bytes are turned into exact f16 pairs in
//    registers (cvt.rn.f16x2.e4m3x2; an E5M2 byte is the upper byte of its
//    f16); q is moved into f16 with a per-warp power of two so no value can
//    overflow; k_scale and the power of two fold into the score multiplier
//    and v_scale into the output.
//  * Split combine.  A unit covered by one block is written out directly;
//    otherwise each block writes a normalised partial (O, log2-sum-exp) and
//    bumps a per-unit counter; the block that arrives last merges all
//    partials of the unit (after its own last unit) and writes the output,
//    then resets the counter.  A block that finds, while it merges its last
//    unit, that the unit's other blocks have all arrived combines at once
//    without an arrival of its own.  No block ever waits on another block.  The
//    counters carry the launch's generation, so a count that a launch left
//    behind (because one of its waits gave up) is never taken for this one's.
//  * Paged cache (PAGED).  Only the producer changes: each tile's page comes
//    from the block table and the TMA load addresses (row in page, page x
//    Hkv + KV head) of the page pool [pages x Hkv][page_size][D].
//  * Every mbarrier wait gives up after a time limit, sets an error flag the
//    host can query, and lets the block finish without hanging the GPU.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <type_traits>

#include "ptx.cuh"

namespace gqa {

constexpr int kTileTokens = 64;   // tokens per pipeline stage
// Eight consumer warps, split into groups that take the ring's tiles in turn
// (per variant: two groups of four warps, or four of two; see Cfg).
constexpr int kConsumerWarps = 8;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kMergeWarps = 3;     // warps 1..3 of warpgroup 0
constexpr int kMergeThreads = kMergeWarps * 32;
constexpr int kFirstConsumerWarp = 4;
constexpr int kThreads = 3 * 128;  // three warpgroups
// Registers per thread after the setmaxnreg split: warpgroup 0 gives up
// registers to the two consumer warpgroups.  The sum equals the launch's
// total (384 threads x 168, the __launch_bounds__(384, 1) allocation):
// 128 x 56 + 256 x 224 = 64512.
constexpr int kRegsSmall = 56;
constexpr int kRegsBig = 224;
static_assert(128 * kRegsSmall + 256 * kRegsBig <= kThreads * 168,
              "register split exceeds the launch allocation");
constexpr int kMaxUnitRows = 64;  // query heads per unit (4 head blocks)
constexpr int kPrefetchTiles = 12; // tiles per block warmed in L2 at launch
// Default time limit of a pipeline wait (DecodeParams::wait_ns); the drain of
// a block's own bulk copies before it exits always uses kDrainLimitNs.
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s per wait
constexpr uint64_t kDrainLimitNs = 200000000ull;   // 0.2 s per final drain
// Retries of the compare-and-swap that counts a block's arrival at a unit
// (each failure means another block's arrival succeeded, so a few suffice).
constexpr int kMaxArrivalTries = 1 << 16;
constexpr int kQPrefetchUnits = 8;   // later units whose q rows are warmed
// A split-combine ticket not yet returned by the arrival (never a count).
constexpr uint32_t kTicketPending = 0xfffffffeu;
// Dynamic shared memory per block: the sm_100-family opt-in maximum (227 KB)
// less 512 bytes left for the kernel's static shared variables.
constexpr int kSmemBudget = 232448 - 512;

enum KvKind : int { kKvF16 = 0, kKvBF16 = 1, kKvE4M3 = 2, kKvE5M2 = 3 };

// 8-bit cache element kinds (E4M3, E5M2); the others are 16-bit.
__host__ __device__ constexpr bool is_fp8(int kv) {
  return kv == kKvE4M3 || kv == kKvE5M2;
}

enum ErrorBits : uint32_t {
  kErrWaitTimeout = 1u,  // a pipeline wait gave up after its time limit
  kErrBadPage = 2u,      // a block-table entry outside [0, num_pages)
  kErrCacheFull = 4u,    // an append found a sequence's cache full
};

struct DecodeParams {
  const void* q;            // [B, Hq, D] f16 / bf16
  // the caches' base addresses (contiguous caches only; they are read
  // through the tensor maps, these only warm L2)
  const void* kc;
  const void* vc;
  void* out;                // [B, Hq, D] same dtype as q
  const int32_t* seq_lens;  // [B]
  const float* k_scale;     // [B, Hkv] (E4M3 only)
  const float* v_scale;     // [B, Hkv] (E4M3 only)
  float* part_o;            // [slots, rows_pad, D]  normalised partial outputs
  float* part_lse;          // [slots, rows_pad]     log2-sum-exp of partials
  // [units] arrivals per unit: (launch generation << 32) | blocks arrived;
  // a value that carries another launch's generation counts as zero
  unsigned long long* counters;
  uint32_t* error;          // fault flags
  uint32_t gen;             // this launch's generation (never 0)
  uint64_t wait_ns;         // time limit of a pipeline wait (0: give up at once)
  // paged cache only: block_table[b * max_pages + i] is the page holding
  // tokens [i * page_size, (i + 1) * page_size) of sequence b
  const int32_t* block_table;
  int max_pages, page_size, num_pages;
  float scale_log2;         // softmax scale * log2(e)
  int B, Hq, Hkv, Smax, G;
  // Query rows: T new tokens per sequence (1 for the decode step), so every
  // KV head serves GR = G * T rows, ordered (head in group, token); q and out
  // are [B, Hq, T, D], in which a KV head's rows are contiguous.
  int T, GR;
  int NHC;                  // row chunks per KV head
  int R;                    // query rows per chunk (<= 64)
  // Blocks to use when every sequence has the same number of tiles, chosen
  // by the host so that block ranges line up with unit boundaries (0: none;
  // then min(grid, tiles) blocks take part).
  int p_align;
  // Tensor-core kernel only: the launch's cluster size when p_align splits
  // every unit evenly over the CTAs of one thread-block cluster (2 or 4);
  // their states are then merged through distributed shared memory.  0 or
  // 1: no cluster launch.
  int cluster;
  // Design choices turned off for A/B measurements (bit 0: no L2 warm-up
  // before the dependent-launch wait).
  int tune;
};

// ------------------------------------------------------------ compile-time

// NR: the narrow-row path for 8-bit caches whose units have at most 8 query
// rows.  Keys are the 16-row A operand and the group's rows the 8 columns of
// each mma (S^T = K Q^T, O^T = V^T P^T), which halves the mma work of the
// 16-row padding and the O registers.
template <int KV, int D, int HB, bool NR = false>
struct Cfg {
  static constexpr int kElemBytes = is_fp8(KV) ? 1 : 2;
  static constexpr int kRowBytes = D * kElemBytes;            // one token
  static constexpr int kTileBytes = kTileTokens * kRowBytes;  // K or V tile
  static constexpr int kStageBytes = 2 * kTileBytes;
  // TMA box: 128-byte rows for 16-bit (D=128 needs two boxes), the whole row
  // for E4M3 (128 B at D=128 -> 128B swizzle, 64 B at D=64 -> 64B swizzle).
  static constexpr int kBoxElems = is_fp8(KV) ? D : 64;
  static constexpr int kBoxBytes = kTileTokens * kBoxElems * kElemBytes;
  static constexpr int kBoxesPerTile = D / kBoxElems;
  // Consumer groups: four of two warps for the 8-bit caches with one head
  // block, whose warps are bound by their dequantising arithmetic (32 tokens
  // a warp per tile: more independent work per softmax round); otherwise two
  // of four warps.
  static constexpr int kGroups = (is_fp8(KV) && HB == 1) ? 4 : 2;
  static constexpr int kGroupWarps = kConsumerWarps / kGroups;
  static constexpr int kWarpsPerBlock = kGroupWarps / HB;  // per head block
  static constexpr int kWarpTokens = kTileTokens / kWarpsPerBlock;
  static constexpr int kSTiles = kWarpTokens / 8;   // S n-tiles per warp
  static constexpr int kPSteps = kWarpTokens / 16;  // PV k-steps per warp
  static constexpr int kOTiles = D / 8;             // O n-tiles
  static constexpr int kQSteps = D / 16;            // QK k-steps
  static constexpr int kMTiles = kWarpTokens / 16;  // NR: key m-tiles per warp
  // mma accumulator tiles of O per warp: O n-tiles, or (NR) O^T m-tiles
  static constexpr int kOAcc = NR ? D / 16 : D / 8;
  static constexpr int kRowsPad = HB * 16;
  // Unit dump: per consumer warp its 16 rows of normalised O, row-major, in
  // f16 for the 8-bit caches (values bounded by the code range) and fp32
  // otherwise; then the row maxima and row sums.
  using DumpT = typename std::conditional<is_fp8(KV), __half, float>::type;
  static constexpr int kDumpRowBytes = D * static_cast<int>(sizeof(DumpT));
  static constexpr int kDumpWarpBytes = 16 * kDumpRowBytes;
  static constexpr int kMergeBytes =
      kConsumerWarps * kDumpWarpBytes + 2 * kConsumerWarps * 16 * 4;
  static constexpr int kStagesRaw = (kSmemBudget - kMergeBytes - 1024 - 256) /
                                    kStageBytes;
  // A multiple of the group count, so that stage s is always consumed by
  // group s % kGroups: each group then waits on the phases of its stages
  // strictly in order, which the mbarrier parity test requires.
  static constexpr int kStages =
      (kStagesRaw > 16 ? 16 : kStagesRaw) / kGroups * kGroups;
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kSmemBytes = 1024 /*alignment slack*/ + kRingBytes +
                                    kMergeBytes + 2 * kStages * 8 + 64;
  static_assert(kStages >= 2 * kGroups && kStages % kGroups == 0,
                "pipeline needs two stages per group");
  static_assert(kWarpsPerBlock >= 1, "a head block needs a warp per group");
  static_assert(!NR || (is_fp8(KV) && HB == 1 && kMTiles >= 1),
                "the narrow-row path serves 8-bit caches with one head block");
  static_assert(kSTiles % 2 == 0 && kPSteps >= 1, "warp tile shape");
  static_assert(kQSteps % 2 == 0, "QK k-steps are split into two chains");
  // Short accumulator chains: with two S tiles per warp the QK k-loop is
  // split over two accumulator sets (even / odd k-steps) and summed.  With
  // four, the second set's registers push the warp into local-memory spills
  // at D = 128 (32-row units: 54.3 us split against 50.4 us unsplit on the
  // 70B shape's 4-token chunk), so those keep one chain per S tile.
  static constexpr bool kSplitQK = kSTiles <= 2;
};

__device__ __forceinline__ int clamp_len(int L, int Smax) {
  return L < 0 ? 0 : (L > Smax ? Smax : L);
}

template <int TT>
__device__ __forceinline__ int tiles_of_t(int L) {
  return (L + TT - 1) / TT;
}

// Position of a block in the flat tile list (tiles of TT tokens), advanced
// one tile at a time.
template <int TT>
struct TileWalkT {
  int b;          // sequence
  int L;          // its valid length
  int nt;         // its tiles per unit
  int j;          // unit within the sequence: kv_head * NHC + head_chunk
  int ti;         // tile within the unit
  long long pref; // global index of the sequence's first tile

  __device__ __forceinline__ void next(const DecodeParams& p, int HU) {
    if (++ti < nt) return;
    ti = 0;
    if (++j < HU) return;
    j = 0;
    pref += static_cast<long long>(nt) * HU;
    do {
      ++b;
      if (b >= p.B) return;
      L = clamp_len(__ldg(p.seq_lens + b), p.Smax);
      nt = tiles_of_t<TT>(L);
    } while (nt == 0);
  }
};
using TileWalk = TileWalkT<kTileTokens>;

// Index of the block whose tile range holds global tile x.
__device__ __forceinline__ int block_of_tile(long long x, long long N, int P) {
  return static_cast<int>(((x + 1) * P - 1) / N);
}

// 16-bit tile: D/64 boxes of [64 tokens][128 B], 128-byte swizzle.
__device__ __forceinline__ uint32_t swz16(int t, int chunk) {
  const int box = chunk >> 3, c = chunk & 7;
  return static_cast<uint32_t>(box * (kTileTokens * 128) + t * 128 +
                               ((c ^ (t & 7)) << 4));
}

// E4M3 tile: [64 tokens][D bytes]; 128-byte swizzle at D=128, 64-byte at 64.
template <int D>
__device__ __forceinline__ uint32_t swz8(int t, int chunk) {
  if constexpr (D == 128) {
    return static_cast<uint32_t>(t * 128 + ((chunk ^ (t & 7)) << 4));
  } else {
    return static_cast<uint32_t>(t * 64 + ((chunk ^ ((t >> 1) & 3)) << 4));
  }
}

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<__half>(__half x) {
  return __half2float(x);
}
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}

template <bool kBF16>
__device__ __forceinline__ void store_out(void* out, size_t idx, float v) {
  if constexpr (kBF16) {
    reinterpret_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
  } else {
    reinterpret_cast<__half*>(out)[idx] = __float2half_rn(v);
  }
}

// Eight consecutive output elements from v * mult, one 16-byte store (idx is
// a multiple of 8 and out 16-byte aligned).
template <bool kBF16>
__device__ __forceinline__ void store_out8(void* out, size_t idx,
                                           const float (&v)[8], float mult) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (kBF16) {
      const __nv_bfloat162 h =
          __floats2bfloat162_rn(v[2 * i] * mult, v[2 * i + 1] * mult);
      memcpy(&w[i], &h, 4);
    } else {
      const __half2 h = __floats2half2_rn(v[2 * i] * mult, v[2 * i + 1] * mult);
      memcpy(&w[i], &h, 4);
    }
  }
  *reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + idx) =
      make_uint4(w[0], w[1], w[2], w[3]);
}

// Block-wide int64 sum over all NT threads (uses `red` scratch).
template <int NT>
__device__ __forceinline__ long long block_sum(long long v, long long* red) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  long long s = 0;
  for (int w = 0; w < NT / 32; ++w) s += red[w];
  __syncthreads();
  return s;
}

// Block-wide inclusive scan of int64 over NT threads (uses `red` scratch).
// Returns the inclusive prefix; *total receives the block sum.
template <int NT>
__device__ __forceinline__ long long block_incl_scan(long long v,
                                                     long long* red,
                                                     long long* total) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  long long x = v;
  for (int o = 1; o < 32; o <<= 1) {
    long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();
  if (lane == 31) red[warp] = x;
  __syncthreads();
  long long before = 0, all = 0;
  for (int w = 0; w < NT / 32; ++w) {
    if (w < warp) before += red[w];
    all += red[w];
  }
  __syncthreads();
  *total = all;
  return before + x;
}

// Issues the global loads of one unit's query rows into the mma A-fragment
// registers qf (raw 16-bit pairs).  row0 / row1 are this thread's two fragment
// rows; invalid rows read as zero.
//
// 16-bit cache: k-step ks uses d = 16ks + 2cq + {0,1} (+8), the layout of an
// m16n8k16 A fragment.  FP8 cache: the k index is permuted so that each
// thread's K bytes are one contiguous run of its token row: thread column cq
// owns d in [cq*D/4, (cq+1)*D/4) and k-step ks uses d = cq*D/4 + 4ks + {0..3};
// the raw pairs then go through fp8_finish_q.
template <bool kFp8, int D, typename QT>
__device__ __forceinline__ void load_q_raw(uint32_t (&qf)[D / 16][4],
                                           const QT* q0, const QT* q1,
                                           bool ok0, bool ok1, int cq) {
  if constexpr (!kFp8) {
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const int d0 = 16 * ks + 2 * cq;
      qf[ks][0] = ok0 ? __ldg(reinterpret_cast<const uint32_t*>(q0 + d0)) : 0u;
      qf[ks][1] = ok1 ? __ldg(reinterpret_cast<const uint32_t*>(q1 + d0)) : 0u;
      qf[ks][2] = ok0 ? __ldg(reinterpret_cast<const uint32_t*>(q0 + d0 + 8)) : 0u;
      qf[ks][3] = ok1 ? __ldg(reinterpret_cast<const uint32_t*>(q1 + d0 + 8)) : 0u;
    }
  } else {
    // run of D/4 elements = D/2 bytes = D/32 16-byte vectors per row
    const uint4* a = reinterpret_cast<const uint4*>(q0 + cq * (D / 4));
    const uint4* b = reinterpret_cast<const uint4*>(q1 + cq * (D / 4));
#pragma unroll
    for (int i = 0; i < D / 32; ++i) {
      const uint4 va = ok0 ? __ldg(a + i) : make_uint4(0u, 0u, 0u, 0u);
      const uint4 vb = ok1 ? __ldg(b + i) : make_uint4(0u, 0u, 0u, 0u);
      // words 4i..4i+3 of the run: pairs (d, d+1) for d = 8i + {0, 2, 4, 6},
      // i.e. k-steps 2i (words 4i, 4i+1) and 2i+1 (words 4i+2, 4i+3)
      qf[2 * i][0] = va.x;
      qf[2 * i][2] = va.y;
      qf[2 * i + 1][0] = va.z;
      qf[2 * i + 1][2] = va.w;
      qf[2 * i][1] = vb.x;
      qf[2 * i][3] = vb.y;
      qf[2 * i + 1][1] = vb.z;
      qf[2 * i + 1][3] = vb.w;
    }
  }
}

template <bool QBF16>
__device__ __forceinline__ float2 unpack_q2(uint32_t w) {
  if constexpr (QBF16) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
  } else {
    return __half22float2(*reinterpret_cast<const __half2*>(&w));
  }
}

// FP8 cache: turns the raw q pairs into f16 mma operands scaled by a power of
// two that puts the largest |q| of the warp's rows in [2^14, 2^15) (exact, and
// no q value can overflow f16).  Returns the exponent e of that power.
template <bool QBF16, int D>
__device__ __forceinline__ int fp8_finish_q(uint32_t (&qf)[D / 16][4]) {
  float amax = 0.f;
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 v = unpack_q2<QBF16>(qf[ks][i]);
      amax = fmaxf(amax, fmaxf(fabsf(v.x), fabsf(v.y)));
    }
  for (int off = 16; off > 0; off >>= 1)
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  int e = 0;
  if (amax > 0.f) {
    int ex;
    frexpf(amax, &ex);  // amax = f * 2^ex, f in [0.5, 1)
    e = 15 - ex;
    e = e > 100 ? 100 : (e < -100 ? -100 : e);
  }
  const float up = ldexpf(1.f, e);
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 v = unpack_q2<QBF16>(qf[ks][i]);
      qf[ks][i] = ptx::pack2<false>(v.x * up, v.y * up);
    }
  return e;
}

// Two 8-bit cache elements (bytes 0 and 1, or bytes 2 and 3, of w) -> two
// exact f16 values packed low/high.  E4M3: the hardware conversion.  E5M2 is
// the upper byte of an IEEE binary16, so its f16 is the byte moved up.
template <int KV>
__device__ __forceinline__ uint32_t fp8_lo(uint32_t w) {
  if constexpr (KV == kKvE5M2) {
    return __byte_perm(w, 0u, 0x1404);
  } else {
    return ptx::e4m3x2_to_f16x2(w & 0xffffu);
  }
}

template <int KV>
__device__ __forceinline__ uint32_t fp8_hi(uint32_t w) {
  if constexpr (KV == kKvE5M2) {
    return __byte_perm(w, 0u, 0x3424);
  } else {
    return ptx::e4m3x2_to_f16x2(w >> 16);
  }
}

// 8-bit cache: the K bytes of token row t (in the tile) that thread column cq
// owns, d in [cq*D/4, (cq+1)*D/4): word ks holds d = cq*D/4 + 4ks + {0..3},
// i.e. the k slots (2cq, 2cq+1) and (2cq+8, 2cq+9) of QK k-step ks.
template <int D>
__device__ __forceinline__ void fp8_key_words(uint32_t kbase, int t, int cq,
                                              uint32_t (&kw)[D / 16]) {
  if constexpr (D == 128) {
    const uint4 a = ptx::lds128(kbase + swz8<D>(t, 2 * cq));
    const uint4 b = ptx::lds128(kbase + swz8<D>(t, 2 * cq + 1));
    kw[0] = a.x; kw[1] = a.y; kw[2] = a.z; kw[3] = a.w;
    kw[4] = b.x; kw[5] = b.y; kw[6] = b.z; kw[7] = b.w;
  } else {
    const uint4 a = ptx::lds128(kbase + swz8<D>(t, cq));
    kw[0] = a.x; kw[1] = a.y; kw[2] = a.z; kw[3] = a.w;
  }
}

// Byte offset of the 16-byte chunk c of dump row `row` (row-major rows of
// kRowBytes; chunks XOR-swizzled by row & 7 so that the eight rows a warp
// writes or reads together fall in different banks).
template <int kRowBytes>
__device__ __forceinline__ int dump_off(int row, int c) {
  return row * kRowBytes + ((c ^ (row & 7)) << 4);
}

// Eight consecutive values (columns 8n .. 8n+7) of dump row `row`.
template <typename DumpT, int D>
__device__ __forceinline__ void dump_load8(const uint8_t* w, int row, int n,
                                          float (&v)[8]) {
  constexpr int kRowBytes = D * static_cast<int>(sizeof(DumpT));
  if constexpr (std::is_same<DumpT, float>::value) {
    const float4 a =
        *reinterpret_cast<const float4*>(w + dump_off<kRowBytes>(row, 2 * n));
    const float4 b = *reinterpret_cast<const float4*>(
        w + dump_off<kRowBytes>(row, 2 * n + 1));
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  } else {
    const uint4 a =
        *reinterpret_cast<const uint4*>(w + dump_off<kRowBytes>(row, n));
    const uint32_t x[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __half2 h;
      memcpy(&h, &x[i], 4);
      const float2 f = __half22float2(h);
      v[2 * i] = f.x;
      v[2 * i + 1] = f.y;
    }
  }
}

// Merges the eight consumer warps' dumped softmax states of one unit
// (warps of head block hbk: both groups' warps with that head block) and
// writes the unit's output rows (whole: the unit lies in this block alone) or
// its normalised partial (row-major fp32 + log2-sum-exp per row).  Run by
// kNT threads (t = 0 .. kNT-1) that synchronise on named barrier kBar.
template <int KV, bool QBF16, int D, int HB, int kNT, int kBar>
__device__ __forceinline__ void merge_unit(int t, const uint8_t* dmp_o,
                                           float* dmp_m, const float* dmp_l,
                                           float* s_rowlse,
                                           const DecodeParams& p, int u,
                                           int bq, int j, bool whole, int cta) {
  using C = Cfg<KV, D, HB>;
  constexpr bool kFp8 = is_fp8(KV);
  constexpr int kW = C::kGroups * C::kWarpsPerBlock;  // warps per head block
  const int kvh = j / p.NHC, hc = j % p.NHC;
  const float o_mult = kFp8 ? __ldg(p.v_scale + bq * p.Hkv + kvh) : 1.f;
  // the k-th warp of head block hbk
  auto warp_of = [](int hbk, int k) {
    return (k / C::kWarpsPerBlock) * C::kGroupWarps + hbk * C::kWarpsPerBlock +
           k % C::kWarpsPerBlock;
  };

  // 1) per merged row: the max over the head block's warps, the total, and
  //    each warp's weight exp2(m_w - M) * l_w / total (written over m_w; the
  //    dumped rows are normalised by their own sums l_w).  One
  //    thread per (row, warp); the kW threads of a row are adjacent lanes and
  //    reduce with shuffles.
  static_assert(32 % kW == 0, "a row's warps must share a warp of threads");
  for (int i = t; i < HB * 16 * kW; i += kNT) {  // warp-uniform bounds
    const int row = i / kW, k = i % kW;
    const int hbk = row >> 4, rr = row & 15;
    const int wk = warp_of(hbk, k);
    const float mv = dmp_m[wk * 16 + rr], lv = dmp_l[wk * 16 + rr];
    float M = mv;
#pragma unroll
    for (int o = 1; o < kW; o <<= 1)
      M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float Mb = (M == -INFINITY) ? 0.f : M;
    const float f = ptx::ex2(mv - Mb);
    float lt = lv * f;
#pragma unroll
    for (int o = 1; o < kW; o <<= 1) lt += __shfl_xor_sync(0xffffffffu, lt, o);
    dmp_m[wk * 16 + rr] = lt > 0.f ? f * lv / lt : 0.f;
    if (k == 0) s_rowlse[row] = lt > 0.f ? Mb + ptx::lg2(lt) : -INFINITY;
  }
  ptx::named_bar_sync(kBar, kNT);

  // 2) merge item by item (eight columns of one row): the head block's
  //    warps' dump values weighted and summed, one 16-byte output store or
  //    two float4 partial stores.  Rows past the chunk (never dumped when a
  //    head block has at most 8 rows) are skipped.
  const int slot = whole ? 0 : cta + u;
  // the unit's first query row in q / out, in rows of D elements
  const size_t rbase =
      (static_cast<size_t>(bq) * p.Hq + static_cast<size_t>(j / p.NHC) * p.G) *
          p.T + static_cast<size_t>(hc) * p.R;
  constexpr int kItems = 2 * D;  // per head block: 16 rows x D/8 columns
  for (int i = t; i < HB * kItems; i += kNT) {  // warp-uniform bounds
    const int hbk = i / kItems;
    const int rr = i & 15, n = (i % kItems) >> 4;  // row fastest: no conflicts
    const int row = hbk * 16 + rr;
    if (row >= p.R || hc * p.R + row >= p.GR) continue;
    float acc[8];
#pragma unroll
    for (int x = 0; x < 8; ++x) acc[x] = 0.f;
    // the consumer threads (registers to spare after their tile loop) keep
    // every warp's loads in flight together; the merge warps, one at a time
#pragma unroll (kNT >= 256 ? 8 : 1)
    for (int k = 0; k < kW; ++k) {
      const int wk = warp_of(hbk, k);
      const float wt = dmp_m[wk * 16 + rr];
      float v[8];
      dump_load8<typename C::DumpT, D>(dmp_o + wk * C::kDumpWarpBytes, rr, n,
                                       v);
#pragma unroll
      for (int x = 0; x < 8; ++x) acc[x] += wt * v[x];
    }
    if (whole) {
      store_out8<QBF16>(p.out, (rbase + row) * D + 8 * n, acc, o_mult);
    } else {
      float4* dst = reinterpret_cast<float4*>(
          p.part_o + (static_cast<size_t>(slot) * C::kRowsPad + row) * D +
          8 * n);
      dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
  }
  if (!whole)
    for (int row = t; row < HB * 16; row += kNT)
      p.part_lse[static_cast<size_t>(slot) * C::kRowsPad + row] =
          s_rowlse[row];
  ptx::named_bar_sync(kBar, kNT);
}

// Split combine of unit u (covered by blocks cf..cl): the output rows from
// all partials, one pass with a running maximum.  A thread takes kI items of
// eight columns (two float4 of a row) and loads them from kB partials at a
// time, all in flight together.  Run by kNT threads.
template <int KV, bool QBF16, int D, int HB, int kNT>
__device__ __forceinline__ void combine_unit(int t, const DecodeParams& p,
                                             int u, int b, int j, int cf,
                                             int cl) {
  using C = Cfg<KV, D, HB>;
  constexpr bool kFp8 = is_fp8(KV);
  constexpr int kB = 4;       // partials per batch
  constexpr int kI = 2;       // items per thread per pass
  constexpr int kG = D / 8;   // items per row
  const int kvh = j / p.NHC, hc = j % p.NHC;
  const float om = kFp8 ? __ldg(p.v_scale + b * p.Hkv + kvh) : 1.f;
  const int n_items = min(p.R, p.GR - hc * p.R) * kG;  // valid rows only
  const size_t h_base =
      ((static_cast<size_t>(b) * p.Hq + static_cast<size_t>(kvh) * p.G) * p.T +
       static_cast<size_t>(hc) * p.R) * D;
  for (int i0 = t; i0 < n_items; i0 += kI * kNT) {
    float M[kI], lt[kI], acc[kI][8];
#pragma unroll
    for (int x = 0; x < kI; ++x) {
      M[x] = -INFINITY;
      lt[x] = 0.f;
#pragma unroll
      for (int y = 0; y < 8; ++y) acc[x][y] = 0.f;
    }
    for (int c0 = cf; c0 <= cl; c0 += kB) {
      float ls[kB][kI];
      float4 ov[kB][kI][2];
#pragma unroll
      for (int k = 0; k < kB; ++k)
#pragma unroll
        for (int x = 0; x < kI; ++x) {
          const int it = i0 + x * kNT;
          const bool ok = c0 + k <= cl && it < n_items;
          const size_t row =
              static_cast<size_t>(c0 + k + u) * C::kRowsPad + it / kG;
          const float4* src = reinterpret_cast<const float4*>(
              p.part_o + row * D + (it % kG) * 8);
          ls[k][x] = ok ? __ldcg(p.part_lse + row) : -INFINITY;
          ov[k][x][0] = ok ? __ldcg(src) : make_float4(0.f, 0.f, 0.f, 0.f);
          ov[k][x][1] = ok ? __ldcg(src + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
      for (int x = 0; x < kI; ++x) {
        float Mn = M[x];
#pragma unroll
        for (int k = 0; k < kB; ++k) Mn = fmaxf(Mn, ls[k][x]);
        if (Mn == -INFINITY) continue;
        const float a = ptx::ex2(M[x] - Mn);  // 0 while M is -inf
        lt[x] *= a;
#pragma unroll
        for (int y = 0; y < 8; ++y) acc[x][y] *= a;
#pragma unroll
        for (int k = 0; k < kB; ++k) {
          const float f = ptx::ex2(ls[k][x] - Mn);
          lt[x] += f;
          acc[x][0] += f * ov[k][x][0].x;
          acc[x][1] += f * ov[k][x][0].y;
          acc[x][2] += f * ov[k][x][0].z;
          acc[x][3] += f * ov[k][x][0].w;
          acc[x][4] += f * ov[k][x][1].x;
          acc[x][5] += f * ov[k][x][1].y;
          acc[x][6] += f * ov[k][x][1].z;
          acc[x][7] += f * ov[k][x][1].w;
        }
        M[x] = Mn;
      }
    }
#pragma unroll
    for (int x = 0; x < kI; ++x) {
      const int it = i0 + x * kNT;
      if (it < n_items)
        store_out8<QBF16>(p.out, h_base + static_cast<size_t>(it / kG) * D +
                                     (it % kG) * 8,
                          acc[x], (lt[x] > 0.f ? 1.f / lt[x] : 0.f) * om);
    }
  }
  if (t == 0) p.counters[u] = 0ull;
}

// Counts this block's arrival at unit u (after its partial is stored) and
// returns how many blocks of this launch arrived before it.  The counter
// carries the launch generation in its upper half: a value another launch
// left behind (one whose waits gave up before all its blocks arrived) counts
// as no arrival, so such a launch cannot shift the tickets of later ones.
// The swap has acquire-release semantics: the caller's partial stores (and
// those ordered before it by a barrier) are released, and the last arriver
// sees every other block's.  The first swap guesses that this block is the
// last of the unit's `expect` blocks (one round trip for the block that then
// combines, which is the one on the kernel's critical path); a wrong guess
// returns the counter's value for the next try.  Sets kErrWaitTimeout and
// returns a ticket that matches no arrival count if the swap keeps failing.
__device__ __forceinline__ uint32_t arrive_unit(const DecodeParams& p, int u,
                                                int expect) {
  unsigned long long* c = p.counters + u;
  const unsigned long long tag = static_cast<unsigned long long>(p.gen) << 32;
  unsigned long long cur =
      tag | static_cast<uint32_t>(expect > 0 ? expect - 1 : 0);
  for (int i = 0; i < kMaxArrivalTries; ++i) {
    const uint32_t n =
        (cur >> 32) == p.gen ? static_cast<uint32_t>(cur) : 0u;
    const unsigned long long want = tag | (n + 1u);
    const unsigned long long seen = ptx::atom_cas_acq_rel_gpu(c, cur, want);
    if (seen == cur) return n;
    cur = seen;
  }
  atomicOr(p.error, kErrWaitTimeout);
  return 0xffffffffu;
}

// Warms L2 with the lines of seq_lens (read first after the wait for the
// previous kernel; an L2 prefetch returns nothing to the thread, so it may be
// issued before that wait).  Threads 0..31 of the block.
__device__ __forceinline__ void prefetch_seq_lens(const DecodeParams& p,
                                                  int tid) {
  if (tid < 32 && tid * 32 < p.B) ptx::prefetch_l2(p.seq_lens + tid * 32);
}

template <int NT>
struct PlanSmem {
  long long red[NT / 32];
  int nt_min[NT / 32], nt_max[NT / 32];
  long long pref0;
  int b0;
  int L0;
  int found;
};

// floor(N * c / P) for the block-range edges: 32-bit unsigned division when
// the product fits (the common case), else 64-bit.
__device__ __forceinline__ long long range_edge(long long N, int c, int P) {
  const unsigned long long x = static_cast<unsigned long long>(N) *
                               static_cast<unsigned>(c);
  if (x <= 0xffffffffull)
    return static_cast<long long>(static_cast<unsigned>(x) /
                                  static_cast<unsigned>(P));
  return static_cast<long long>(x / static_cast<unsigned long long>(P));
}

// The flat tile list (tiles of TT tokens, units sequence-major): its length
// N, the number of blocks that take part P, this block's range [t0, t1) and
// the walk position of its first tile.  Called by all NT threads of the
// block.  Blocks that take part: at most one per tile (P = min(grid, N)), so
// that every block in a unit's covering range [c_first, c_last] owns at least
// one of its tiles (the arrival count of the split combine relies on it);
// when every sequence has the same tile count, the host's unit-aligned count
// p.p_align replaces it.
//
// Batches of at most NT sequences: one seq_lens load per thread, a warp scan
// and two block barriers (the warps' totals and tile-count extremes, then the
// block's start position).
template <int NT, int TT>
__device__ __forceinline__ void plan_block(const DecodeParams& p, int HU,
                                           PlanSmem<NT>& sm, long long& N,
                                           int& P, long long& t0,
                                           long long& t1, TileWalkT<TT>& w0) {
  const int tid = threadIdx.x;
  const int cta = blockIdx.x;
  t0 = 0;
  t1 = 0;
  if (p.B <= NT) {
    const int b = tid;
    const int warp = tid >> 5, lane = tid & 31;
    const int Lb = b < p.B ? clamp_len(__ldg(p.seq_lens + b), p.Smax) : 0;
    const int nt_b = tiles_of_t<TT>(Lb);
    const long long v = static_cast<long long>(nt_b) * HU;
    long long x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    const int wmin = __reduce_min_sync(0xffffffffu, b < p.B ? nt_b : INT_MAX);
    const int wmax = __reduce_max_sync(0xffffffffu, b < p.B ? nt_b : 0);
    if (lane == 31) {
      sm.red[warp] = x;
      sm.nt_min[warp] = wmin;
      sm.nt_max[warp] = wmax;
    }
    __syncthreads();
    long long before = 0;
    N = 0;
    int mn = INT_MAX, mx = 0;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) {
      const long long r = sm.red[w];
      before += w < warp ? r : 0;
      N += r;
      mn = min(mn, sm.nt_min[w]);
      mx = max(mx, sm.nt_max[w]);
    }
    const long long incl = before + x;
    // equal tile counts: the host's unit-aligned block count applies
    const bool uniform = mn == mx;
    P = static_cast<int>(N < gridDim.x ? N : gridDim.x);
    if (uniform && p.p_align > 0 && N >= p.p_align) P = p.p_align;
    if (cta < P) {
      t0 = range_edge(N, cta, P);
      t1 = range_edge(N, cta + 1, P);
    }
    if (t0 < t1 && v > 0 && incl - v <= t0 && t0 < incl) {
      sm.b0 = b;
      sm.pref0 = incl - v;
      sm.L0 = Lb;
    }
  } else {
    long long mine = 0;
    for (int b = tid; b < p.B; b += NT)
      mine += static_cast<long long>(tiles_of_t<TT>(
                  clamp_len(__ldg(p.seq_lens + b), p.Smax))) * HU;
    N = block_sum<NT>(mine, sm.red);
    P = static_cast<int>(N < gridDim.x ? N : gridDim.x);
    if (cta < P) {
      t0 = range_edge(N, cta, P);
      t1 = range_edge(N, cta + 1, P);
    }
    if (t0 < t1) {
      long long run = 0;
      for (int base = 0; base < p.B; base += NT) {
        const int b = base + tid;
        long long v = 0;
        int Lb = 0;
        if (b < p.B) {
          Lb = clamp_len(__ldg(p.seq_lens + b), p.Smax);
          v = static_cast<long long>(tiles_of_t<TT>(Lb)) * HU;
        }
        long long tot;
        const long long incl = block_incl_scan<NT>(v, sm.red, &tot);
        const long long excl = incl - v;
        if (v > 0 && run + excl <= t0 && t0 < run + incl) {
          sm.b0 = b;
          sm.pref0 = run + excl;
          sm.L0 = Lb;
          sm.found = 1;
        }
        run += tot;
        __syncthreads();
        if (sm.found) break;
      }
    }
  }
  __syncthreads();
  if (t0 < t1) {
    w0.b = sm.b0;
    w0.L = sm.L0;
    w0.nt = tiles_of_t<TT>(w0.L);
    w0.pref = sm.pref0;
    const long long off = t0 - w0.pref;
    if (off <= 0x7fffffffll) {
      const unsigned uo = static_cast<unsigned>(off);
      const unsigned jj = uo / static_cast<unsigned>(w0.nt);
      w0.j = static_cast<int>(jj);
      w0.ti = static_cast<int>(uo - jj * static_cast<unsigned>(w0.nt));
    } else {
      w0.j = static_cast<int>(off / w0.nt);
      w0.ti = static_cast<int>(off % w0.nt);
    }
  }
}

// Warms L2 with the query rows of unit (b, kvh, hc): one bulk prefetch of
// the unit's contiguous rows of q [B, Hq, T, D] (16-bit).
template <int D>
__device__ __forceinline__ void prefetch_unit_q(const DecodeParams& p, int b,
                                                int kvh, int hc) {
  const int rows = min(p.R, p.GR - hc * p.R);
  if (rows <= 0) return;
  const size_t row0 =
      (static_cast<size_t>(b) * p.Hq + static_cast<size_t>(kvh) * p.G) * p.T +
      static_cast<size_t>(hc) * p.R;
  ptx::bulk_prefetch_l2(static_cast<const uint16_t*>(p.q) + row0 * D,
                        static_cast<uint32_t>(rows * D * 2));
}

// Warms L2 with the query rows of the units that start inside this block's
// tile range [t0, t1) after its first one (at most kQPrefetchUnits), so that
// a change of unit late in the range does not wait for them in HBM.  One
// thread; w is the walk position of tile t0.
template <int D, int TT>
__device__ __forceinline__ void prefetch_range_q(const DecodeParams& p, int HU,
                                                 TileWalkT<TT> w, long long t0,
                                                 long long t1) {
  long long g = t0;
  for (int k = 0; k < kQPrefetchUnits; ++k) {
    g += w.nt - w.ti;  // the next unit's first tile
    if (g >= t1) return;
    w.ti = w.nt - 1;
    w.next(p, HU);
    prefetch_unit_q<D>(p, w.b, w.j / p.NHC, w.j % p.NHC);
  }
}

// Warms L2 with this block's first tiles, guessing that every sequence fills
// its cache (exact for uniform lengths; a wrong guess only costs bandwidth).
// Uses kernel parameters only, so it may run before the previous kernel in
// the stream has finished.  32-bit integer arithmetic and a fast approximate
// divide only: a 64-bit or IEEE division here compiles to a called routine
// that costs the whole kernel registers.  The start tile only needs to be
// close; problems with more than 2^31 tiles skip the prefetch.
template <int KV, int D, int HB, int TT = kTileTokens, bool BULK = false>
__device__ __forceinline__ void prefetch_first_tiles(const CUtensorMap* map_k,
                                                     const CUtensorMap* map_v,
                                                     const DecodeParams& p,
                                                     int lane) {
  using C = Cfg<KV, D, HB>;
  const int B = p.B, Hkv = p.Hkv, NHC = p.NHC, Smax = p.Smax;
  const int p_align = p.p_align;
  // the same bytes whatever the tile length: kPrefetchTiles 64-token tiles
  constexpr int kTiles = kPrefetchTiles * kTileTokens / TT;
  const unsigned nt = (static_cast<unsigned>(Smax) + TT - 1) / TT;
  const unsigned long long n64 =
      static_cast<unsigned long long>(nt) * Hkv * NHC * B;
  if (n64 == 0ull || n64 > 0x7fffffffull) return;
  const unsigned per_seq = nt * Hkv * NHC;
  const unsigned ng = static_cast<unsigned>(n64);
  unsigned pg = ng < gridDim.x ? ng : gridDim.x;
  if (p_align > 0 && ng >= static_cast<unsigned>(p_align)) pg = p_align;
  if (blockIdx.x >= pg) return;
  // approximate start tile (no IEEE division: its slow path is a call)
  unsigned x0 = static_cast<unsigned>(
      __fdividef(static_cast<float>(ng), static_cast<float>(pg)) * blockIdx.x);
  if (BULK && NHC == 1 && p.kc != nullptr) {
    // one KV head per unit: the guessed range is contiguous in each cache
    // ([B*Hkv][Smax][D], plane x / nt): one bulk prefetch of K and one of V
    // instead of one per box and tile, which the TMA unit issues one at a
    // time at the block's start (measured: faster for the tensor-core
    // kernel's multi-query steps, slower for the warp-level kernel's)
    if (lane == 0 && x0 < ng) {
      const unsigned plane = x0 / nt;
      const unsigned long long row = static_cast<unsigned long long>(D) *
                                     C::kElemBytes;
      const unsigned long long start =
          (static_cast<unsigned long long>(plane) * Smax + (x0 % nt) * TT) *
          row;
      const unsigned long long total =
          static_cast<unsigned long long>(B) * Hkv * Smax * row;
      unsigned long long len =
          static_cast<unsigned long long>(kPrefetchTiles) * kTileTokens * row;
      if (start < total) {
        if (len > total - start) len = total - start;
        ptx::bulk_prefetch_l2(static_cast<const uint8_t*>(p.kc) + start,
                              static_cast<uint32_t>(len));
        ptx::bulk_prefetch_l2(static_cast<const uint8_t*>(p.vc) + start,
                              static_cast<uint32_t>(len));
      }
      prefetch_unit_q<D>(p, static_cast<int>(plane) / Hkv,
                         static_cast<int>(plane) % Hkv, 0);
    }
    return;
  }
  // lane k prefetches tile k of the range (one warp, no divergence in the
  // arithmetic)
  x0 += lane;
  if (lane < kTiles && x0 < ng) {
    const unsigned bq = x0 / per_seq, rem = x0 % per_seq;
    const int plane = static_cast<int>(bq) * Hkv +
                      static_cast<int>(rem / nt) / NHC;
    const int tok = static_cast<int>(rem % nt) * TT;
    if (lane == 0) {
      // the query rows of the first unit
      const int jj = static_cast<int>(rem / nt);
      prefetch_unit_q<D>(p, static_cast<int>(bq), jj / NHC, jj % NHC);
    }
#pragma unroll
    for (int th = 0; th < TT / kTileTokens; ++th)
#pragma unroll
      for (int bx = 0; bx < C::kBoxesPerTile; ++bx) {
        ptx::tma_prefetch_3d(map_k, bx * C::kBoxElems, tok + th * kTileTokens,
                             plane);
        ptx::tma_prefetch_3d(map_v, bx * C::kBoxElems, tok + th * kTileTokens,
                             plane);
      }
  }
}

template <int KV, bool QBF16, int D, int HB, bool PAGED, bool NR = false>
__global__ void __launch_bounds__(kThreads, 1)
    gqa_decode_kernel(const __grid_constant__ CUtensorMap map_k,
                      const __grid_constant__ CUtensorMap map_v,
                      const DecodeParams p) {
  using C = Cfg<KV, D, HB, NR>;
  constexpr bool kFp8 = is_fp8(KV);
  constexpr bool kMmaBF16 = !kFp8 && QBF16;
  using QT = typename std::conditional<QBF16, __nv_bfloat16, __half>::type;
  constexpr int kPos = C::kOTiles * 4 * 32;  // fragment positions per warp

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  // Dump area of the unit epilogue: per consumer warp its 16 normalised O
  // rows (row-major, chunks swizzled as in dump_off), then the row maxima and
  // row sums of all warps.
  uint8_t* dmp_o = ring + C::kRingBytes;
  float* dmp_m =
      reinterpret_cast<float*>(dmp_o + kConsumerWarps * C::kDumpWarpBytes);
  float* dmp_l = dmp_m + kConsumerWarps * 16;
  uint64_t* full = reinterpret_cast<uint64_t*>(dmp_l + kConsumerWarps * 16);
  uint64_t* empty = full + C::kStages;
  uint64_t* dump_full = empty + C::kStages;   // 8 consumer warps arrive
  uint64_t* dump_empty = dump_full + 1;       // the merge warps arrive
  __shared__ PlanSmem<kThreads> s_plan;
  __shared__ volatile int s_abort;
  // the flat list's tile count and the blocks taking part, re-read at unit
  // ends (volatile: not held in registers through the tile loop)
  __shared__ volatile long long s_N;
  __shared__ volatile int s_P;
  __shared__ float s_rowlse[HB * 16];   // log2-sum-exp per merged row
  // descriptor of the unit whose states are in the dump area; s_dstop marks
  // the block's last unit, which the consumers merge themselves
  __shared__ int s_du, s_db, s_dj, s_dcf, s_dcl, s_dstop;
  // Units this block covers only in part (at most the first and the last of
  // its range), with the block's arrival ticket; their split combine runs
  // after the block's last unit.
  __shared__ int s_npend;
  __shared__ int s_pend_u[2], s_pend_b[2], s_pend_j[2], s_pend_cf[2],
      s_pend_cl[2], s_pend_last[2];
  __shared__ volatile uint32_t s_pend_t[2];

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int cta = blockIdx.x;
  const int HU = p.Hkv * p.NHC;  // units per sequence

  if (warp == 0) {
    if (lane == 0) {
      // descriptor fetch overlaps the scheduler prologue
      ptx::prefetch_tensormap(&map_k);
      ptx::prefetch_tensormap(&map_v);
    }
    if constexpr (!PAGED)
      if (!(p.tune & 1))
        prefetch_first_tiles<KV, D, HB>(&map_k, &map_v, p, lane);
  }
  if (tid == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], C::kGroupWarps);
    }
    ptx::mbar_init(dump_full, kConsumerWarps);
    ptx::mbar_init(dump_empty, 1);
    ptx::fence_barrier_init();
    s_abort = 0;
    s_npend = 0;
    s_plan.found = 0;
    s_plan.b0 = 0;
    s_plan.L0 = 0;
    s_plan.pref0 = 0;
  }
  // Launched as a programmatic dependent of the previous kernel in the
  // stream: everything above overlapped its tail; nothing before this point
  // reads global memory (q, the caches and seq_lens may be written by it).
  // seq_lens is only warmed in L2, which stays coherent with those writes.
  prefetch_seq_lens(p, tid);
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();

  // ---- flat tile list: total N, this block's range, its first sequence ----
  long long N, t0, t1;
  int P;
  TileWalk w0;
  plan_block<kThreads, kTileTokens>(p, HU, s_plan, N, P, t0, t1, w0);
  if (tid == 0) {
    s_N = N;
    s_P = P;
  }
  __syncthreads();

  if (warp < 4) {
    ptx::setmaxnreg_dec<kRegsSmall>();
  } else {
    ptx::setmaxnreg_inc<kRegsBig>();
  }

  if (warp == 0) {
    // =============================== producer ===============================
    if (lane == 0 && t0 < t1) {
      const uint64_t policy = ptx::policy_evict_first();
      TileWalk w = w0;
      long long it = 0;
      for (long long g = t0; g < t1; ++g, ++it) {
        const int stage = static_cast<int>(it % C::kStages);
        const uint32_t ph = static_cast<uint32_t>((it / C::kStages) & 1);
        const int kvh = w.j / p.NHC;
        const int tok = w.ti * kTileTokens;
        // paged: the tile's block-table entry is loaded before the wait for
        // its ring slot, so that the load's latency hides behind the wait
        // (a tile lies inside one page: page_size is a multiple of it)
        int pg = 0;
        if constexpr (PAGED)
          pg = __ldg(p.block_table + static_cast<size_t>(w.b) * p.max_pages +
                     tok / p.page_size);
        if (!ptx::mbar_wait_bounded(&empty[stage], ph ^ 1u, p.wait_ns)) {
          atomicOr(p.error, kErrWaitTimeout);
          s_abort = 1;
          break;
        }
        if (s_abort) break;
        ptx::mbar_arrive_expect_tx(&full[stage], C::kStageBytes);
        // tile coordinates in the cache view [planes][tokens][D]
        int row = tok, plane = w.b * p.Hkv + kvh;
        if constexpr (PAGED) {
          if (pg < 0 || pg >= p.num_pages) {
            atomicOr(p.error, kErrBadPage);
            pg = 0;
          }
          row = tok % p.page_size;
          plane = pg * p.Hkv + kvh;
        }
        uint8_t* ks = ring + stage * C::kStageBytes;
        uint8_t* vs = ks + C::kTileBytes;
#pragma unroll
        for (int bx = 0; bx < C::kBoxesPerTile; ++bx) {
          ptx::tma_load_3d(ks + bx * C::kBoxBytes, &map_k, &full[stage],
                           bx * C::kBoxElems, row, plane, policy);
          ptx::tma_load_3d(vs + bx * C::kBoxBytes, &map_v, &full[stage],
                           bx * C::kBoxElems, row, plane, policy);
        }
        w.next(p, HU);
      }
      // Never leave the block with bulk copies still writing its memory.
      const long long issued = it;
      for (int s = 0; s < C::kStages; ++s) {
        const long long uses =
            issued > s ? (issued - s + C::kStages - 1) / C::kStages : 0;
        if (uses > 0)
          ptx::mbar_wait_bounded(&full[s],
                                 static_cast<uint32_t>((uses - 1) & 1),
                                 kDrainLimitNs);
      }
    }
    return;
  }

  if (warp < 4) {
    // ================================= merge =================================
    const int mt = tid - 32;  // 0 .. kMergeThreads-1
    if (mt == 0 && t0 < t1) prefetch_range_q<D, kTileTokens>(p, HU, w0, t0, t1);
    // Sequences with no valid token: all-zero output rows.
    for (int b = cta; b < p.B; b += gridDim.x) {
      if (clamp_len(__ldg(p.seq_lens + b), p.Smax) != 0) continue;
      const size_t base = static_cast<size_t>(b) * p.Hq * p.T * D;
      for (int i = mt; i < p.Hq * p.T * D; i += kMergeThreads)
        store_out<QBF16>(p.out, base + i, 0.f);
    }
    if (t0 >= t1) return;

    // Units that end inside this block's range, in order; the block's last
    // unit is merged by the consumers themselves (descriptor s_dstop).
    uint32_t kph = 0;  // parity of the dump being waited for
    while (true) {
      // Every merge thread waits; the give-up decision is taken together
      // (barrier with an OR of the outcomes), so that all merge warps either
      // go on to merge_unit's barriers or leave.
      const bool ok = ptx::mbar_wait_bounded(dump_full, kph, p.wait_ns);
      if (ptx::named_bar_or(2, kMergeThreads, !ok)) {
        if (mt == 0) {
          atomicOr(p.error, kErrWaitTimeout);
          s_abort = 1;
        }
        return;
      }
      kph ^= 1u;
      if (s_dstop) return;
      const int u = s_du, bq = s_db, j = s_dj;
      const int c_first = s_dcf, c_last = s_dcl;
      const bool whole = (c_first == c_last);
      merge_unit<KV, QBF16, D, HB, kMergeThreads, 2>(
          mt, dmp_o, dmp_m, dmp_l, s_rowlse, p, u, bq, j, whole, cta);
      // A partial also counts this block's arrival (acquire-release add: the
      // merge warps' partial stores are ordered before it by their barrier);
      // the ticket is kept for the combine after the block's last unit.  The
      // dump area is handed back first (merge_unit's last barrier: no merge
      // thread reads it any more), so that the consumers' next dump does not
      // wait for the arrival's release of the partial stores.
      if (mt == 0) {
        // the slot first (its ticket marked pending), then the dump area,
        // then the arrival and its ticket
        int k = -1;
        if (!whole && s_npend < 2) {
          k = s_npend;
          s_pend_t[k] = kTicketPending;
          s_pend_u[k] = u;
          s_pend_b[k] = bq;
          s_pend_j[k] = j;
          s_pend_cf[k] = c_first;
          s_pend_cl[k] = c_last;
          s_npend = k + 1;
        }
        ptx::mbar_arrive(dump_empty);
        if (k >= 0) {
          const uint32_t tk = arrive_unit(p, u, c_last - c_first + 1);
          __threadfence_block();
          s_pend_t[k] = tk;
        }
      }
    }
  }

  // =============================== consumers ================================
  const int cw = warp - kFirstConsumerWarp;  // consumer warp 0..7
  const int grp = cw / C::kGroupWarps;       // consumer group
  const int lw = cw % C::kGroupWarps;        // warp within the group
  const int hb = lw / C::kWarpsPerBlock;     // head block of this warp
  const int wsl = lw % C::kWarpsPerBlock;    // token slice of this warp
  const int r = lane >> 2, cq = lane & 3;    // mma fragment coordinates
  if (t0 >= t1) return;

  TileWalk w = w0;
  uint32_t qf[C::kQSteps][4];
  float o[C::kOAcc][4];
  float m[2], l[2];
  float s_mult = 0.f;
  bool fresh = true;
  bool aborted = false;  // this warp gave up on a wait: skip further waits
  // Last key each of this thread's two rows may see: new token i of a chunk
  // attends causally to keys t <= L - T + i (T = 1: every key t < L).  The
  // 8-bit cache kernels serve one token per sequence only (T = 1 at compile
  // time), which keeps their register budget.
  const int T = kFp8 ? 1 : p.T;
  int lim0 = 0, lim1 = 0;

  // This thread's two fragment rows within its head block, and their query
  // rows for unit (kvh, hc) of sequence b.
  const int row0 = hb * 16 + r, row1 = row0 + 8;
  // 8-bit caches: the unit's K scale, loaded with its query rows (it is
  // needed at the unit's first tile, where a load's latency would stall)
  float k_scale_next = 1.f;
  auto issue_q = [&](int b, int kvh, int hc) {
    if constexpr (kFp8) k_scale_next = __ldg(p.k_scale + b * p.Hkv + kvh);
    const bool ok0 = row0 < p.R && hc * p.R + row0 < p.GR;
    const bool ok1 = row1 < p.R && hc * p.R + row1 < p.GR;
    const size_t r0 =
        (static_cast<size_t>(b) * p.Hq + static_cast<size_t>(kvh) * p.G) *
            T + static_cast<size_t>(hc) * p.R + row0;
    const QT* q0 = reinterpret_cast<const QT*>(p.q) + (ok0 ? r0 : 0) * D;
    const QT* q1 = reinterpret_cast<const QT*>(p.q) + (ok1 ? r0 + 8 : 0) * D;
    load_q_raw<kFp8, D, QT>(qf, q0, q1, ok0, ok1, cq);
  };
  issue_q(w.b, w.j / p.NHC, w.j % p.NHC);

  int stage = 0;     // ring stage of tile g: (g - t0) % kStages
  uint32_t ph = 0;   // its phase parity: ((g - t0) / kStages) & 1
  int par = 0;       // (g - t0) % kGroups: the group that computes tile g
  uint32_t dph = 0;  // parity of this block's unit epilogues so far
  for (long long g = t0; g < t1; ++g) {
    if (fresh) {
      // ---- new unit: softmax state and multipliers (q already issued) ----
      fresh = false;
      if constexpr (!kFp8) {
        s_mult = p.scale_log2;
      } else {
        const int e = fp8_finish_q<QBF16, D>(qf);
        s_mult = p.scale_log2 * k_scale_next * ldexpf(1.f, -e);
      }
#pragma unroll
      for (int n = 0; n < C::kOAcc; ++n)
        o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
      m[0] = m[1] = -INFINITY;
      l[0] = l[1] = 0.f;
      const int hc = w.j % p.NHC;
      lim0 = w.L - T + (hc * p.R + row0) % T;
      lim1 = kFp8 ? lim0 : w.L - T + (hc * p.R + row1) % T;
    }

    if (par == grp) {
    // ---- wait for the stage (the groups take the tiles in turn) ----
    // the warp decides together (a lane-divergent give-up would leave its
    // lanes on different paths)
    if (!aborted &&
        !__all_sync(0xffffffffu,
                    ptx::mbar_wait_bounded(&full[stage], ph, p.wait_ns))) {
      atomicOr(p.error, kErrWaitTimeout);
      aborted = true;
      s_abort = 1;  // stops the producer
    }
    const uint32_t kbase = ptx::smem_u32(ring + stage * C::kStageBytes);
    const uint32_t vbase = kbase + C::kTileBytes;
    const int L = w.L;
    const int tok0 = w.ti * kTileTokens + wsl * C::kWarpTokens;  // in-seq
    const int trow0 = wsl * C::kWarpTokens;                      // in-tile
    // tiles that may hold keys a row must not see: the last one (tokens
    // beyond L) and, for a multi-token chunk, those reaching past L - T
    const bool tail = (w.ti == w.nt - 1) ||
                      (w.ti * kTileTokens + kTileTokens - 1 > L - T);

    if constexpr (NR) {
    // ==== narrow rows: S^T = K Q^T, O^T += V^T P^T (keys / d on the mma
    // rows, this unit's <= 8 query rows on its 8 columns) ====
    // S^T m-tile mt: tokens trow0 + 16mt + r (+8) on the rows, query rows
    // 2cq, 2cq+1 on the columns: entries 0/1 (token r), 2/3 (token r + 8).
    float st[C::kMTiles][4];
#pragma unroll
    for (int mt = 0; mt < C::kMTiles; ++mt) {
      uint32_t ka[D / 16], kb[D / 16];
      fp8_key_words<D>(kbase, trow0 + mt * 16 + r, cq, ka);
      fp8_key_words<D>(kbase, trow0 + mt * 16 + r + 8, cq, kb);
      float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ks = 0; ks < C::kQSteps; ++ks) {
        // A: keys (rows r, r+8) at the k slots of q's permuted d (B: row r)
        const uint32_t a[4] = {fp8_lo<KV>(ka[ks]), fp8_lo<KV>(kb[ks]),
                               fp8_hi<KV>(ka[ks]), fp8_hi<KV>(kb[ks])};
        if (ks & 1)
          ptx::mma16816<false>(sb, a, qf[ks][0], qf[ks][2]);
        else
          ptx::mma16816<false>(sa, a, qf[ks][0], qf[ks][2]);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) st[mt][e] = sa[e] + sb[e];
    }
    // online softmax of rows 2cq (entries 0, 2) and 2cq+1 (entries 1, 3);
    // a column's 8 lanes (r = 0..7) reduce with three shuffles
    {
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int mt = 0; mt < C::kMTiles; ++mt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float v = st[mt][e] * s_mult;
          if (tail && tok0 + mt * 16 + r + 8 * (e >> 1) > lim0) v = -INFINITY;
          st[mt][e] = v;
        }
        mx0 = fmaxf(mx0, fmaxf(st[mt][0], st[mt][2]));
        mx1 = fmaxf(mx1, fmaxf(st[mt][1], st[mt][3]));
      }
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
      }
      const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
      const float base0 = (mn0 == -INFINITY) ? 0.f : mn0;
      const float base1 = (mn1 == -INFINITY) ? 0.f : mn1;
      const float al0 = ptx::ex2(m[0] - base0);
      const float al1 = ptx::ex2(m[1] - base1);
      m[0] = mn0;
      m[1] = mn1;
      float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
      for (int mt = 0; mt < C::kMTiles; ++mt) {
        st[mt][0] = ptx::ex2(st[mt][0] - base0);
        st[mt][2] = ptx::ex2(st[mt][2] - base0);
        st[mt][1] = ptx::ex2(st[mt][1] - base1);
        st[mt][3] = ptx::ex2(st[mt][3] - base1);
        rs0 += st[mt][0] + st[mt][2];
        rs1 += st[mt][1] + st[mt][3];
      }
      l[0] = l[0] * al0 + rs0;
      l[1] = l[1] * al1 + rs1;
      if (al0 != 1.f || al1 != 1.f) {
#pragma unroll
        for (int n = 0; n < C::kOAcc; ++n) {
          o[n][0] *= al0;
          o[n][2] *= al0;
          o[n][1] *= al1;
          o[n][3] *= al1;
        }
      }
    }
    // O^T m-tile mt_d holds d = (D/8) r + 2 mt_d (rows r) and + 1 (rows
    // r + 8): each thread row owns one contiguous run of D/8 V bytes.
#pragma unroll
    for (int kk = 0; kk < C::kMTiles; ++kk) {
      // P^T as the B operand: the (token x row) 8x8 blocks transposed
      const uint32_t b0 =
          ptx::movmatrix_trans(ptx::pack2<false>(st[kk][0], st[kk][1]));
      const uint32_t b1 =
          ptx::movmatrix_trans(ptx::pack2<false>(st[kk][2], st[kk][3]));
      const int tk = tok0 + kk * 16 + 2 * cq;  // tokens tk, tk+1, tk+8, tk+9
      const int ta = trow0 + kk * 16 + 2 * cq;
      constexpr int kW = D / 32;  // 32-bit words per thread per token row
      uint32_t xa[kW], xb[kW], xc[kW], xd[kW];
      if constexpr (D == 128) {
        const uint4 a = ptx::lds128(vbase + swz8<D>(ta, r));
        const uint4 b = ptx::lds128(vbase + swz8<D>(ta + 1, r));
        const uint4 c = ptx::lds128(vbase + swz8<D>(ta + 8, r));
        const uint4 d = ptx::lds128(vbase + swz8<D>(ta + 9, r));
        xa[0] = a.x; xa[1] = a.y; xa[2] = a.z; xa[3] = a.w;
        xb[0] = b.x; xb[1] = b.y; xb[2] = b.z; xb[3] = b.w;
        xc[0] = c.x; xc[1] = c.y; xc[2] = c.z; xc[3] = c.w;
        xd[0] = d.x; xd[1] = d.y; xd[2] = d.z; xd[3] = d.w;
      } else {
        const int half = (r & 1) * 8;
        const uint2 a = ptx::lds64(vbase + swz8<D>(ta, r >> 1) + half);
        const uint2 b = ptx::lds64(vbase + swz8<D>(ta + 1, r >> 1) + half);
        const uint2 c = ptx::lds64(vbase + swz8<D>(ta + 8, r >> 1) + half);
        const uint2 d = ptx::lds64(vbase + swz8<D>(ta + 9, r >> 1) + half);
        xa[0] = a.x; xa[1] = a.y;
        xb[0] = b.x; xb[1] = b.y;
        xc[0] = c.x; xc[1] = c.y;
        xd[0] = d.x; xd[1] = d.y;
      }
      if (tail) {  // bytes of tokens past the end may hold anything
        const uint32_t ka = tk < L ? ~0u : 0u, kb = tk + 1 < L ? ~0u : 0u;
        const uint32_t kc = tk + 8 < L ? ~0u : 0u, kd = tk + 9 < L ? ~0u : 0u;
#pragma unroll
        for (int i = 0; i < kW; ++i) {
          xa[i] &= ka;
          xb[i] &= kb;
          xc[i] &= kc;
          xd[i] &= kd;
        }
      }
#pragma unroll
      for (int wi = 0; wi < kW; ++wi) {
        // byte j of word wi: d = (D/8) r + 4wi + j -> m-tile 2wi + j/2, row
        // r + 8 (j & 1); pair up tokens (tk, tk+1) and (tk+8, tk+9)
        const uint32_t p01 = __byte_perm(xa[wi], xb[wi], 0x5140);
        const uint32_t p23 = __byte_perm(xa[wi], xb[wi], 0x7362);
        const uint32_t q01 = __byte_perm(xc[wi], xd[wi], 0x5140);
        const uint32_t q23 = __byte_perm(xc[wi], xd[wi], 0x7362);
        const uint32_t a0[4] = {fp8_lo<KV>(p01), fp8_hi<KV>(p01),
                                fp8_lo<KV>(q01), fp8_hi<KV>(q01)};
        const uint32_t a1[4] = {fp8_lo<KV>(p23), fp8_hi<KV>(p23),
                                fp8_lo<KV>(q23), fp8_hi<KV>(q23)};
        ptx::mma16816<false>(o[2 * wi], a0, b0, b1);
        ptx::mma16816<false>(o[2 * wi + 1], a1, b0, b1);
      }
    }
    } else {
    // ---- S = Q K^T for this warp's tokens ----
    float s[C::kSTiles][4];
    float s2[C::kSplitQK ? C::kSTiles : 1][4];  // odd k-steps when split
#pragma unroll
    for (int n = 0; n < C::kSTiles; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
    for (int n = 0; n < (C::kSplitQK ? C::kSTiles : 1); ++n)
      s2[n][0] = s2[n][1] = s2[n][2] = s2[n][3] = 0.f;

    if constexpr (!kFp8) {
      const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
      for (int ks = 0; ks < C::kQSteps; ++ks) {
#pragma unroll
        for (int np = 0; np < C::kSTiles / 2; ++np) {
          const int t = trow0 + np * 16 + (mi >> 1) * 8 + rr;
          const int chunk = 2 * ks + (mi & 1);
          uint32_t b0, b1, b2, b3;
          ptx::ldsm_x4(kbase + swz16(t, chunk), b0, b1, b2, b3);
          if (C::kSplitQK && (ks & 1)) {
            ptx::mma16816<kMmaBF16>(s2[2 * np], qf[ks], b0, b1);
            ptx::mma16816<kMmaBF16>(s2[2 * np + 1], qf[ks], b2, b3);
          } else {
            ptx::mma16816<kMmaBF16>(s[2 * np], qf[ks], b0, b1);
            ptx::mma16816<kMmaBF16>(s[2 * np + 1], qf[ks], b2, b3);
          }
        }
      }
    } else {
#pragma unroll
      for (int n = 0; n < C::kSTiles; ++n) {
        const int t = trow0 + n * 8 + r;
        uint32_t kw[D / 16];
        fp8_key_words<D>(kbase, t, cq, kw);
#pragma unroll
        for (int ks = 0; ks < C::kQSteps; ++ks) {
          const uint32_t b0 = fp8_lo<KV>(kw[ks]);
          const uint32_t b1 = fp8_hi<KV>(kw[ks]);
          if (C::kSplitQK && (ks & 1))
            ptx::mma16816<false>(s2[n], qf[ks], b0, b1);
          else
            ptx::mma16816<false>(s[n], qf[ks], b0, b1);
        }
      }
    }
    if constexpr (C::kSplitQK) {
#pragma unroll
      for (int n = 0; n < C::kSTiles; ++n) {
        s[n][0] += s2[n][0];
        s[n][1] += s2[n][1];
        s[n][2] += s2[n][2];
        s[n][3] += s2[n][3];
      }
    }

    // ---- online softmax (log2 domain) ----
    // kHi: rows r + 8 of this warp's head block are real.  When a head block
    // has at most 8 rows they are padding: their probabilities are set to 0
    // and their max / exp / sum work is skipped (warp-uniform choice).
    auto softmax = [&](auto hi_c) {
      constexpr bool kHi = decltype(hi_c)::value;
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int n = 0; n < C::kSTiles; ++n) {
#pragma unroll
        for (int e = 0; e < (kHi ? 4 : 2); ++e) {
          float v = s[n][e] * s_mult;
          if (tail) {
            const int tk = tok0 + n * 8 + 2 * cq + (e & 1);
            if (tk > ((e & 2) ? lim1 : lim0)) v = -INFINITY;
          }
          s[n][e] = v;
        }
        mx0 = fmaxf(mx0, fmaxf(s[n][0], s[n][1]));
        if (kHi) mx1 = fmaxf(mx1, fmaxf(s[n][2], s[n][3]));
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      if (kHi) {
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      }
      const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
      const float base0 = (mn0 == -INFINITY) ? 0.f : mn0;
      const float base1 = (mn1 == -INFINITY) ? 0.f : mn1;
      const float al0 = ptx::ex2(m[0] - base0);
      const float al1 = kHi ? ptx::ex2(m[1] - base1) : 1.f;
      m[0] = mn0;
      m[1] = mn1;
      float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
      for (int n = 0; n < C::kSTiles; ++n) {
        s[n][0] = ptx::ex2(s[n][0] - base0);
        s[n][1] = ptx::ex2(s[n][1] - base0);
        if (kHi) {
          s[n][2] = ptx::ex2(s[n][2] - base1);
          s[n][3] = ptx::ex2(s[n][3] - base1);
          rs1 += s[n][2] + s[n][3];
        } else {
          s[n][2] = s[n][3] = 0.f;
        }
        rs0 += s[n][0] + s[n][1];
      }
      l[0] = l[0] * al0 + rs0;
      if (kHi) l[1] = l[1] * al1 + rs1;
      if (al0 != 1.f || al1 != 1.f) {
#pragma unroll
        for (int n = 0; n < C::kOTiles; ++n) {
          o[n][0] *= al0;
          o[n][1] *= al0;
          if (kHi) {
            o[n][2] *= al1;
            o[n][3] *= al1;
          }
        }
      }
    };
    if (hb * 16 + 8 < p.R)
      softmax(std::integral_constant<bool, true>{});
    else
      softmax(std::integral_constant<bool, false>{});

    // ---- O += P V ----
    constexpr bool kPBF16 = kMmaBF16;
#pragma unroll
    for (int kk = 0; kk < C::kPSteps; ++kk) {
      uint32_t pa[4];
      pa[0] = ptx::pack2<kPBF16>(s[2 * kk][0], s[2 * kk][1]);
      pa[1] = ptx::pack2<kPBF16>(s[2 * kk][2], s[2 * kk][3]);
      pa[2] = ptx::pack2<kPBF16>(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      pa[3] = ptx::pack2<kPBF16>(s[2 * kk + 1][2], s[2 * kk + 1][3]);
      // tokens (in sequence) of this thread's B-fragment k slots
      const int tk = tok0 + kk * 16 + 2 * cq;
      if constexpr (!kFp8) {
        uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
        if (tail) {
          mlo = (tk < L ? 0x0000ffffu : 0u) | (tk + 1 < L ? 0xffff0000u : 0u);
          mhi = (tk + 8 < L ? 0x0000ffffu : 0u) |
                (tk + 9 < L ? 0xffff0000u : 0u);
        }
        const int mi = lane >> 3, rr = lane & 7;
        const int t = trow0 + kk * 16 + (mi & 1) * 8 + rr;
#pragma unroll
        for (int jp = 0; jp < C::kOTiles / 2; ++jp) {
          uint32_t b0, b1, b2, b3;
          ptx::ldsm_x4_trans(vbase + swz16(t, 2 * jp + (mi >> 1)), b0, b1, b2,
                             b3);
          b0 &= mlo;
          b2 &= mlo;
          b1 &= mhi;
          b3 &= mhi;
          ptx::mma16816<kMmaBF16>(o[2 * jp], pa, b0, b1);
          ptx::mma16816<kMmaBF16>(o[2 * jp + 1], pa, b2, b3);
        }
      } else {
        // Output columns are permuted too: thread row r owns d in
        // [r*D/8, (r+1)*D/8); n-tile jn holds d = r*D/8 + jn.
        const int ta = trow0 + kk * 16 + 2 * cq;
        constexpr int kW = D / 32;  // 32-bit words per thread per token row
        uint32_t xa[kW], xb[kW], xc[kW], xd[kW];
        if constexpr (D == 128) {
          const uint4 a = ptx::lds128(kbase + C::kTileBytes + swz8<D>(ta, r));
          const uint4 b = ptx::lds128(kbase + C::kTileBytes + swz8<D>(ta + 1, r));
          const uint4 c = ptx::lds128(kbase + C::kTileBytes + swz8<D>(ta + 8, r));
          const uint4 d = ptx::lds128(kbase + C::kTileBytes + swz8<D>(ta + 9, r));
          xa[0] = a.x; xa[1] = a.y; xa[2] = a.z; xa[3] = a.w;
          xb[0] = b.x; xb[1] = b.y; xb[2] = b.z; xb[3] = b.w;
          xc[0] = c.x; xc[1] = c.y; xc[2] = c.z; xc[3] = c.w;
          xd[0] = d.x; xd[1] = d.y; xd[2] = d.z; xd[3] = d.w;
        } else {
          const int half = (r & 1) * 8;
          const uint2 a = ptx::lds64(vbase + swz8<D>(ta, r >> 1) + half);
          const uint2 b = ptx::lds64(vbase + swz8<D>(ta + 1, r >> 1) + half);
          const uint2 c = ptx::lds64(vbase + swz8<D>(ta + 8, r >> 1) + half);
          const uint2 d = ptx::lds64(vbase + swz8<D>(ta + 9, r >> 1) + half);
          xa[0] = a.x; xa[1] = a.y;
          xb[0] = b.x; xb[1] = b.y;
          xc[0] = c.x; xc[1] = c.y;
          xd[0] = d.x; xd[1] = d.y;
        }
        if (tail) {
          const uint32_t ka = tk < L ? ~0u : 0u, kb = tk + 1 < L ? ~0u : 0u;
          const uint32_t kc = tk + 8 < L ? ~0u : 0u, kd = tk + 9 < L ? ~0u : 0u;
#pragma unroll
          for (int i = 0; i < kW; ++i) {
            xa[i] &= ka;
            xb[i] &= kb;
            xc[i] &= kc;
            xd[i] &= kd;
          }
        }
#pragma unroll
        for (int wi = 0; wi < kW; ++wi) {
          const uint32_t p01 = __byte_perm(xa[wi], xb[wi], 0x5140);
          const uint32_t p23 = __byte_perm(xa[wi], xb[wi], 0x7362);
          const uint32_t q01 = __byte_perm(xc[wi], xd[wi], 0x5140);
          const uint32_t q23 = __byte_perm(xc[wi], xd[wi], 0x7362);
          ptx::mma16816<false>(o[4 * wi + 0], pa,
                               fp8_lo<KV>(p01),
                               fp8_lo<KV>(q01));
          ptx::mma16816<false>(o[4 * wi + 1], pa,
                               fp8_hi<KV>(p01),
                               fp8_hi<KV>(q01));
          ptx::mma16816<false>(o[4 * wi + 2], pa,
                               fp8_lo<KV>(p23),
                               fp8_lo<KV>(q23));
          ptx::mma16816<false>(o[4 * wi + 3], pa,
                               fp8_hi<KV>(p23),
                               fp8_hi<KV>(q23));
        }
      }
    }

    }  // NR / wide rows

    // ---- release the stage ----
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(&empty[stage]);
    }  // this group's tile

    const bool unit_end = (w.ti == w.nt - 1) || (g == t1 - 1);
    if (unit_end) {
      // ============ unit epilogue: hand the state to the merge warps ========
      // wait until the merge warps have finished with the previous dump
      if (!aborted &&
          !__all_sync(0xffffffffu,
                      ptx::mbar_wait_bounded(dump_empty, dph ^ 1u,
                                             p.wait_ns))) {
        atomicOr(p.error, kErrWaitTimeout);
        aborted = true;
        s_abort = 1;
      }
      dph ^= 1u;
      uint8_t* mo = dmp_o + cw * C::kDumpWarpBytes;
      if constexpr (NR) {
        // rows 2cq, 2cq+1: sums over the column's 8 lanes; this thread's run
        // d = (D/8) r + j of each row holds O^T entries 0 / 1 (j even) and
        // 2 / 3 (j odd) of m-tile j / 2
        float lt0 = l[0], lt1 = l[1];
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          lt0 += __shfl_xor_sync(0xffffffffu, lt0, off);
          lt1 += __shfl_xor_sync(0xffffffffu, lt1, off);
        }
        const float inv0 = lt0 > 0.f ? __fdividef(1.f, lt0) : 0.f;
        const float inv1 = lt1 > 0.f ? __fdividef(1.f, lt1) : 0.f;
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
          uint32_t w0[4], w1[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const __half2 h0 = __floats2half2_rn(o[4 * h + i][0] * inv0,
                                                 o[4 * h + i][2] * inv0);
            const __half2 h1 = __floats2half2_rn(o[4 * h + i][1] * inv1,
                                                 o[4 * h + i][3] * inv1);
            memcpy(&w0[i], &h0, 4);
            memcpy(&w1[i], &h1, 4);
          }
          const int c = r * (D / 64) + h;
          if (2 * cq < p.R)
            *reinterpret_cast<uint4*>(
                mo + dump_off<C::kDumpRowBytes>(2 * cq, c)) =
                make_uint4(w0[0], w0[1], w0[2], w0[3]);
          if (2 * cq + 1 < p.R)
            *reinterpret_cast<uint4*>(
                mo + dump_off<C::kDumpRowBytes>(2 * cq + 1, c)) =
                make_uint4(w1[0], w1[1], w1[2], w1[3]);
        }
        if (r == 0) {
          dmp_m[cw * 16 + 2 * cq] = m[0];
          dmp_m[cw * 16 + 2 * cq + 1] = m[1];
          dmp_l[cw * 16 + 2 * cq] = lt0;
          dmp_l[cw * 16 + 2 * cq + 1] = lt1;
        }
      } else {
      float lt0 = l[0], lt1 = l[1];
      lt0 += __shfl_xor_sync(0xffffffffu, lt0, 1);
      lt0 += __shfl_xor_sync(0xffffffffu, lt0, 2);
      lt1 += __shfl_xor_sync(0xffffffffu, lt1, 1);
      lt1 += __shfl_xor_sync(0xffffffffu, lt1, 2);
      const bool hi_rows = hb * 16 + 8 < p.R;  // rows r+8 exist (uniform)
      // rows normalised by their sums, into this warp's row-major dump
      const float inv0 = lt0 > 0.f ? __fdividef(1.f, lt0) : 0.f;
      const float inv1 = lt1 > 0.f ? __fdividef(1.f, lt1) : 0.f;
      if constexpr (!kFp8) {
        // fragment element e of n-tile n: column 8n + 2cq + (e & 1)
#pragma unroll
        for (int n = 0; n < C::kOTiles; ++n) {
          const int c = 2 * n + (cq >> 1), off = (cq & 1) * 8;
          *reinterpret_cast<float2*>(
              mo + dump_off<C::kDumpRowBytes>(r, c) + off) =
              make_float2(o[n][0] * inv0, o[n][1] * inv0);
          if (hi_rows)
            *reinterpret_cast<float2*>(
                mo + dump_off<C::kDumpRowBytes>(r + 8, c) + off) =
                make_float2(o[n][2] * inv1, o[n][3] * inv1);
        }
      } else {
        // permuted columns: element e of n-tile n is column
        // (2cq + (e & 1)) * D/8 + n, so n-tiles 8c' .. 8c'+7 fill one chunk
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (e >= 2 && !hi_rows) break;
          const float inv = e < 2 ? inv0 : inv1;
#pragma unroll
          for (int ng = 0; ng < D / 64; ++ng) {
            uint32_t wv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const __half2 h = __floats2half2_rn(o[8 * ng + 2 * i][e] * inv,
                                                  o[8 * ng + 2 * i + 1][e] * inv);
              memcpy(&wv[i], &h, 4);
            }
            const int c = (2 * cq + (e & 1)) * (D / 64) + ng;
            *reinterpret_cast<uint4*>(
                mo + dump_off<C::kDumpRowBytes>(r + 8 * (e >> 1), c)) =
                make_uint4(wv[0], wv[1], wv[2], wv[3]);
          }
        }
      }
      if (cq == 0) {
        dmp_m[cw * 16 + r] = m[0];
        dmp_m[cw * 16 + r + 8] = m[1];
        dmp_l[cw * 16 + r] = lt0;
        dmp_l[cw * 16 + r + 8] = lt1;
      }
      }  // NR / wide rows
      const bool last = (g == t1 - 1);
      const long long us = w.pref + static_cast<long long>(w.j) * w.nt;
      const int u = w.b * HU + w.j;
      const long long Nv = s_N;
      const int Pv = s_P;
      const int c_first = block_of_tile(us, Nv, Pv);
      const int c_last = block_of_tile(us + w.nt - 1, Nv, Pv);
      if (cw == 0 && lane == 0) {
        s_du = u;
        s_db = w.b;
        s_dj = w.j;
        s_dcf = c_first;
        s_dcl = c_last;
        s_dstop = last ? 1 : 0;
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(dump_full);
      if (!last) {
        // the next unit's query rows load while the merge warps work
        TileWalk wn = w;
        wn.next(p, HU);
        issue_q(wn.b, wn.j / p.NHC, wn.j % p.NHC);
        fresh = true;
      } else {
        break;  // g == t1 - 1: the block's range is done
      }
    }
    if (++par == C::kGroups) par = 0;
    if (++stage == C::kStages) {
      stage = 0;
      ph ^= 1u;
    }
    w.next(p, HU);
  }

  // ---- the block's last unit: all consumer threads merge it, then run the
  // split combines of the units whose last arrival was this block's.  After
  // the tile loop, so that none of its registers are live; the unit's
  // descriptor is in shared memory (written before the dump's arrival). ----
  const int ct = tid - kFirstConsumerWarp * 32;  // 0 .. 255
  ptx::named_bar_sync(1, kConsumerThreads);  // every warp's dump
  {
    const int u = s_du, c_first = s_dcf, c_last = s_dcl;
    const bool whole = (c_first == c_last);
    const int expect = c_last - c_first + 1;  // blocks of a split unit
    // Have the unit's other blocks all arrived?  Read (with acquire) while
    // the merge runs.  If so this block is the last one: it combines at once,
    // with no arrival of its own and so without waiting for its partial
    // stores to be released (its own threads see them through the barrier).
    unsigned long long seen = 0ull;
    if (ct == 0 && !whole) seen = ptx::ld_acquire_gpu(p.counters + u);
    merge_unit<KV, QBF16, D, HB, kConsumerThreads, 1>(
        ct, dmp_o, dmp_m, dmp_l, s_rowlse, p, u, s_db, s_dj, whole, cta);
    if (ct == 0) {
      if (!whole && s_npend < 2) {
        const int k = s_npend;
        const unsigned long long all_others =
            (static_cast<unsigned long long>(p.gen) << 32) |
            static_cast<uint32_t>(expect - 1);
        s_pend_t[k] = seen == all_others ? static_cast<uint32_t>(expect - 1)
                                         : arrive_unit(p, u, expect);
        s_pend_u[k] = u;
        s_pend_b[k] = s_db;
        s_pend_j[k] = s_dj;
        s_pend_cf[k] = c_first;
        s_pend_cl[k] = c_last;
        s_npend = k + 1;
      }
      // A merge warp's ticket may still be on its way (its arrival runs
      // after it handed the dump area back): wait for it (bounded).
      const uint64_t t_start = ptx::globaltimer_ns();
      for (int i = 0; i < s_npend; ++i)
        while (s_pend_t[i] == kTicketPending) {
          if (ptx::globaltimer_ns() - t_start > p.wait_ns) {
            atomicOr(p.error, kErrWaitTimeout);
            s_pend_t[i] = 0xffffffffu;  // matches no arrival count
          }
        }
      __threadfence_block();
      // last arrival of a unit: this block combines its partials
      // (the acquire side of both adds: what the other blocks released
      // before their arrivals is visible to this thread, and to the
      // others through the barrier below)
      for (int i = 0; i < 2; ++i)
        s_pend_last[i] =
            i < s_npend && s_pend_t[i] == static_cast<uint32_t>(
                                              s_pend_cl[i] - s_pend_cf[i]);
    }
    ptx::named_bar_sync(1, kConsumerThreads);
  }
  for (int i = 0; i < 2; ++i)
    if (s_pend_last[i])  // uniform
      combine_unit<KV, QBF16, D, HB, kConsumerThreads>(
          ct, p, s_pend_u[i], s_pend_b[i], s_pend_j[i], s_pend_cf[i],
          s_pend_cl[i]);
}

}  // namespace gqa
