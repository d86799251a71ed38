// gqa_api.cu — host side of libgqa_b300.so: the C ABI declared in
// include/gqa.h (argument checks, TMA descriptors, per-stream scratch,
// kernel selection and launch).  All GPU work is in gqa_decode_kernel.cuh
// (warp-level mma kernel) and gqa_decode_umma.cuh (tensor-core kernel).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <map>
#include <tuple>
#include <mutex>
#include <utility>

#include "gqa.h"
#include "gqa_append_kernel.cuh"
#include "gqa_decode_kernel.cuh"
#include "gqa_umma.h"

namespace gqa {
namespace {

// ------------------------------------------------------------ driver entry

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = []() {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      ptr = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }();
  return fn;
}

// Rank-3 view [B*Hkv][Smax][D] of a cache, box = one pipeline tile.
bool make_cache_map(CUtensorMap* map, const void* base, int elem_bytes,
                    int B, int Hkv, int Smax, int D) {
  auto enc = encode_fn();
  if (!enc) return false;
  const int box_elems = (elem_bytes == 1) ? D : 64;
  const int box_bytes = box_elems * elem_bytes;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D),
                        static_cast<cuuint64_t>(Smax),
                        static_cast<cuuint64_t>(B) * Hkv};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * elem_bytes,
                           static_cast<cuuint64_t>(Smax) * D * elem_bytes};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(box_elems),
                       static_cast<cuuint32_t>(kTileTokens), 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUtensorMapSwizzle sw = box_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                                 : CU_TENSOR_MAP_SWIZZLE_64B;
  const CUresult r = enc(
      map, elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                           : CU_TENSOR_MAP_DATA_TYPE_UINT16,
      3, const_cast<void*>(base), dims, strides, box, estr,
      CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Rank-2 view [rows][D] of the 16-bit queries [B, Hq, T, D] for the
// tensor-core kernel: box = 64 rows x 64 elements (128-byte rows, 128-byte
// swizzle), the K-major operand layout of its first product.
bool make_q_map(CUtensorMap* map, const void* base, long long rows, int D) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(D),
                        static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * 2};
  cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(kUmmaCols)};
  cuuint32_t estr[2] = {1u, 1u};
  const CUresult r = enc(
      map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(base), dims,
      strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Encoded descriptors of recently used caches and queries: a descriptor only
// records the base address, shape and strides, so it stays valid for any
// later call on the same (pointer, shape).  Bounded; cleared when full.
// Guarded by g_mu.  kind 0: a cache view, 1: a query view.
struct MapKey {
  const void* base;
  int kind, elem_bytes, B, Hkv, Smax, D;
  bool operator<(const MapKey& o) const {
    return std::tie(base, kind, elem_bytes, B, Hkv, Smax, D) <
           std::tie(o.base, o.kind, o.elem_bytes, o.B, o.Hkv, o.Smax, o.D);
  }
};
std::map<MapKey, CUtensorMap> g_maps;
constexpr size_t kMaxCachedMaps = 256;

bool cached_cache_map(CUtensorMap* map, const void* base, int elem_bytes,
                      int B, int Hkv, int Smax, int D) {
  const MapKey key{base, 0, elem_bytes, B, Hkv, Smax, D};
  auto it = g_maps.find(key);
  if (it != g_maps.end()) {
    *map = it->second;
    return true;
  }
  if (!make_cache_map(map, base, elem_bytes, B, Hkv, Smax, D)) return false;
  if (g_maps.size() >= kMaxCachedMaps) g_maps.clear();
  g_maps.emplace(key, *map);
  return true;
}

bool cached_q_map(CUtensorMap* map, const void* base, int rows, int D) {
  const MapKey key{base, 1, 2, rows, 0, 0, D};
  auto it = g_maps.find(key);
  if (it != g_maps.end()) {
    *map = it->second;
    return true;
  }
  if (!make_q_map(map, base, rows, D)) return false;
  if (g_maps.size() >= kMaxCachedMaps) g_maps.clear();
  g_maps.emplace(key, *map);
  return true;
}

// ----------------------------------------------------------- kernel table

using KernelFn = void (*)(const CUtensorMap, const CUtensorMap,
                          const DecodeParams);

struct Variant {
  KernelFn fn;
  int smem;
};

template <int KV, bool QB, int D, int HB, bool PG, bool NR = false>
Variant variant() {
  return {&gqa_decode_kernel<KV, QB, D, HB, PG, NR>,
          Cfg<KV, D, HB, NR>::kSmemBytes};
}

// 8-bit caches whose units have at most 8 query rows: the narrow-row path.
template <int KV>
Variant pick_nr(bool q_bf16, int D) {
  if (D == 64)
    return q_bf16 ? variant<KV, true, 64, 1, false, true>()
                  : variant<KV, false, 64, 1, false, true>();
  return q_bf16 ? variant<KV, true, 128, 1, false, true>()
                : variant<KV, false, 128, 1, false, true>();
}

template <int KV, bool QB, int D, bool PG>
Variant pick_hb(int hb) {
  switch (hb) {
    case 1: return variant<KV, QB, D, 1, PG>();
    case 2: return variant<KV, QB, D, 2, PG>();
    default: return variant<KV, QB, D, 4, PG>();
  }
}

template <int KV, bool QB, bool PG = false>
Variant pick_d(int D, int hb) {
  return D == 64 ? pick_hb<KV, QB, 64, PG>(hb) : pick_hb<KV, QB, 128, PG>(hb);
}

// Paged caches are instantiated for the 16-bit element types.  rows: query
// rows per unit (R).
Variant pick(int kv, bool q_bf16, int D, int hb, int rows, bool paged = false,
             bool narrow = true) {
  if (is_fp8(kv) && rows <= 8 && narrow)
    return kv == kKvE5M2 ? pick_nr<kKvE5M2>(q_bf16, D)
                         : pick_nr<kKvE4M3>(q_bf16, D);
  if (paged)
    return kv == kKvBF16 ? pick_d<kKvBF16, true, true>(D, hb)
                         : pick_d<kKvF16, false, true>(D, hb);
  if (kv == kKvF16) return pick_d<kKvF16, false>(D, hb);
  if (kv == kKvBF16) return pick_d<kKvBF16, true>(D, hb);
  if (kv == kKvE5M2)
    return q_bf16 ? pick_d<kKvE5M2, true>(D, hb) : pick_d<kKvE5M2, false>(D, hb);
  return q_bf16 ? pick_d<kKvE4M3, true>(D, hb) : pick_d<kKvE4M3, false>(D, hb);
}

// ------------------------------------------------------- per-device state

std::mutex g_mu;

struct DeviceInfo {
  int sms = 0;
  std::map<const void*, int> blocks_per_sm;  // configured kernels
};
std::map<int, DeviceInfo> g_dev;

// Scratch per (device, stream), in two allocations:
//  * ctl  = [error flags (kHeaderBytes) | arrival counters, 8 bytes per unit].
//    Zeroed once when allocated and never re-initialised between calls: each
//    launch tags its counts with its own generation (DecodeParams::gen), and
//    a launch that completes leaves every counter at zero, so whatever an
//    earlier launch left behind is never read as an arrival of this one.  It
//    is never shared with the partials.
//  * part = [partial log2-sum-exp | partial O], fully written before it is
//    read within one call; no initial value needed.
struct Scratch {
  void* ctl = nullptr;
  size_t ctl_units = 0;  // counter capacity
  void* part = nullptr;
  size_t part_bytes = 0;
  uint32_t gen = 0;      // generation of the last launch on this stream
};

constexpr size_t kCounterBytes = 8;

// Next launch generation after `g` (0 is never used: zeroed counters carry
// no generation).
uint32_t next_gen(uint32_t g) { return g + 1u == 0u ? 1u : g + 1u; }
std::map<std::pair<int, cudaStream_t>, Scratch> g_scratch;

int g_num_ctas_override = 0;
uint64_t g_wait_ns = kWaitLimitNs;
// Kernel choice: 0 automatic (the tensor-core kernel for units of more than
// kUmmaMinRows query rows with a 16-bit cache and head_dim 128), 1 the
// warp-level mma kernel everywhere, 2 the tensor-core kernel wherever it
// applies (also for units of fewer rows).
int g_kernel_path = 0;
// Units of more rows than this go to the tensor-core kernel by default.
// Measured (back-to-back steps): 64-row units (multi-query attention) 22.8
// us against 32.1 us on the warp-level kernel; 32-row units (the 70B
// shape's 4-token chunk) 55.2 us against 54.0 us, so they stay there.
constexpr int kUmmaMinRows = 32;
int g_tuning = 0;  // GQA_TUNE_* bits: design choices turned off
thread_local int t_last_launches = 0;

constexpr size_t kHeaderBytes = 256;  // error word(s)

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Sets a kernel's dynamic shared memory once per device; returns its
// occupancy (blocks per SM) and the device's SM count.
cudaError_t configure(int dev, const void* fn, int smem, int threads, int* sms,
                      int* per_sm) {
  DeviceInfo& di = g_dev[dev];
  if (di.sms == 0) {
    cudaError_t e =
        cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
  }
  auto it = di.blocks_per_sm.find(fn);
  if (it == di.blocks_per_sm.end()) {
    cudaError_t e = cudaFuncSetAttribute(
        fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, smem);
    if (e != cudaSuccess) return e;
    if (n < 1) return cudaErrorInvalidConfiguration;
    it = di.blocks_per_sm.emplace(fn, n).first;
  }
  *sms = di.sms;
  *per_sm = it->second;
  return cudaSuccess;
}

// How many clusters of k blocks of kernel `fn` can run at the same time on
// the device (cached per kernel and k; 0 when the query fails).
long long max_clusters(int dev, const void* fn, int smem, int threads, int k) {
  static std::map<std::tuple<int, const void*, int>, long long> cache;
  const auto key = std::make_tuple(dev, fn, k);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(k));
  cfg.blockDim = dim3(static_cast<unsigned>(threads));
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(k);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    n = 0;
  }
  cache.emplace(key, n);
  return n;
}

cudaError_t configure(int dev, const Variant& v, int* sms, int* per_sm) {
  return configure(dev, reinterpret_cast<const void*>(v.fn), v.smem, kThreads,
                   sms, per_sm);
}

// Grows the stream's scratch to hold `units` counters and `part_need` bytes of
// partials.  Allocation is stream-ordered (the device's default pool).
cudaError_t scratch_for(int dev, cudaStream_t stream, size_t units,
                        size_t part_need, Scratch** out) {
  Scratch& s = g_scratch[{dev, stream}];
  if (s.ctl_units < units || !s.ctl) {
    const size_t cap = align_up(units + units / 4 + 1024, 1024);
    void* ctl = nullptr;
    cudaError_t e =
        cudaMallocAsync(&ctl, kHeaderBytes + cap * kCounterBytes, stream);
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(ctl, 0, kHeaderBytes + cap * kCounterBytes, stream);
    if (e != cudaSuccess) return e;
    if (s.ctl) {
      // carry the error flags over to the new, zeroed region
      e = cudaMemcpyAsync(ctl, s.ctl, sizeof(uint32_t),
                          cudaMemcpyDeviceToDevice, stream);
      if (e != cudaSuccess) return e;
      e = cudaFreeAsync(s.ctl, stream);
      if (e != cudaSuccess) return e;
    }
    s.ctl = ctl;
    s.ctl_units = cap;
  }
  if (s.part_bytes < part_need || !s.part) {
    if (s.part) {
      cudaError_t e = cudaFreeAsync(s.part, stream);
      s.part = nullptr;
      s.part_bytes = 0;
      if (e != cudaSuccess) return e;
    }
    const size_t bytes = align_up(part_need + part_need / 4 + 1, 1 << 20);
    cudaError_t e = cudaMallocAsync(&s.part, bytes, stream);
    if (e != cudaSuccess) {
      s.part = nullptr;
      return e;
    }
    s.part_bytes = bytes;
  }
  *out = &s;
  return cudaSuccess;
}

bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

gqa_status check_common(const void* q, const void* k, const void* v,
                        const int32_t* seq_lens, float scale, const void* out,
                        int B, int Hq, int Hkv, int Smax, int D) {
  if (!q || !k || !v || !seq_lens || !out) return GQA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) ||
      !aligned(out, 16) || !aligned(seq_lens, 4))
    return GQA_ERR_INVALID_ARG;
  if (B < 1 || Hq < 1 || Hkv < 1 || Smax < 1 || D < 1)
    return GQA_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return GQA_ERR_INVALID_ARG;
  if (!(std::isfinite(scale) && scale > 0.f)) return GQA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return GQA_ERR_UNSUPPORTED;
  // TMA coordinates and the unit index are 32-bit.
  if (static_cast<long long>(B) * Hq > INT32_MAX) return GQA_ERR_UNSUPPORTED;
  return GQA_OK;
}

// Block count that lines block ranges up with unit boundaries when every
// sequence has the same number of tiles (the kernel checks that on the
// device): the largest P of at least 5/6 of the grid that is a multiple of
// the unit count or divides it.  Fewer blocks stream more bytes each, so
// this pays where the cuts it removes are a large share of a block's work:
//  * P = units (one unit per block) or P = units / k for k <= 4;
//  * P = k * units for k > 1 (every unit split over k blocks) only for
//    64-row units (hb == 4), whose partials are the costliest to merge when
//    the cuts fall anywhere.
// 0: no such P.
int aligned_blocks(long long units, int grid, int hb) {
  const int min_p = grid - grid / 6;
  if (units <= grid) {
    const int k = grid / static_cast<int>(units);
    const int pa = k * static_cast<int>(units);
    return (pa >= min_p && (k == 1 || hb == 4)) ? pa : 0;
  }
  for (int d = grid; d >= min_p; --d)
    if (units % d == 0) return units / d <= 4 ? d : 0;
  return 0;
}

// Smax: the cache's token capacity per sequence.  A paged cache passes its
// block table, page size and page count (Smax = max_pages * page_size);
// block_table == nullptr is a contiguous cache.
gqa_status launch(const void* q, const void* k, const void* v,
                  const float* k_scale, const float* v_scale,
                  const int32_t* seq_lens, float scale, void* out, int B,
                  int Hq, int Hkv, int Smax, int D, int kv_kind, bool q_bf16,
                  void* stream_ptr, const int32_t* block_table = nullptr,
                  int page_size = 0, int num_pages = 0, int T = 1) {
  const bool paged = block_table != nullptr;
  t_last_launches = 0;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  const int G = Hq / Hkv;
  const int GR = G * T;  // query rows per KV head
  const int NHC = (GR + kMaxUnitRows - 1) / kMaxUnitRows;
  const int R = (GR + NHC - 1) / NHC;
  const int hb = R <= 16 ? 1 : (R <= 32 ? 2 : 4);
  const long long units = static_cast<long long>(B) * Hkv * NHC;
  if (units > INT32_MAX / 2) return GQA_ERR_UNSUPPORTED;

  // the tensor-core kernel: 16-bit caches, head_dim 128
  const bool umma = !is_fp8(kv_kind) && D == kUmmaD &&
                    (g_kernel_path == 2 ||
                     (g_kernel_path == 0 && R > kUmmaMinRows));
  const int tile_tokens = umma ? kUmmaTileTokens : kTileTokens;
  const int rows_pad = umma ? kUmmaCols : hb * 16;
  const Variant var = pick(kv_kind, q_bf16, D, hb, R, paged,
                           !(g_tuning & GQA_TUNE_NO_NARROW_ROWS));
  const UmmaVariant uvar = umma ? umma_variant(q_bf16, R, paged)
                                : UmmaVariant{};
  const int elem_bytes = is_fp8(kv_kind) ? 1 : 2;
  // the TMA view [planes][rows][D]: (B*Hkv, Smax) or (num_pages*Hkv,
  // page_size)
  const int planes_outer = paged ? num_pages : B;
  const int rows = paged ? page_size : Smax;

  std::lock_guard<std::mutex> lock(g_mu);
  CUtensorMap map_k, map_v, map_q;
  if (!cached_cache_map(&map_k, k, elem_bytes, planes_outer, Hkv, rows, D) ||
      !cached_cache_map(&map_v, v, elem_bytes, planes_outer, Hkv, rows, D))
    return GQA_ERR_CUDA;
  if (umma && !cached_q_map(&map_q, q, B * Hq * T, D)) return GQA_ERR_CUDA;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GQA_ERR_CUDA;
  int sms = 0, per_sm = 0;
  const cudaError_t ce =
      umma ? configure(dev, reinterpret_cast<const void*>(uvar.fn), uvar.smem,
                       kUmmaThreads, &sms, &per_sm)
           : configure(dev, var, &sms, &per_sm);
  if (ce != cudaSuccess) return GQA_ERR_CUDA;
  // Default: one full wave, but never more blocks than the largest possible
  // number of tiles (seq_lens stay on the device; Smax bounds them).
  const long long max_tiles =
      units * ((static_cast<long long>(Smax) + tile_tokens - 1) / tile_tokens);
  const long long wave = static_cast<long long>(sms) * per_sm;
  int grid = g_num_ctas_override > 0
                 ? g_num_ctas_override
                 : static_cast<int>(max_tiles < wave ? max_tiles : wave);
  const int p_align = g_num_ctas_override > 0
                          ? 0
                          : aligned_blocks(units, grid, umma ? 4 : hb);
  // Tensor-core kernel, every unit split evenly over k = 2 or 4 blocks:
  // launch those blocks as thread-block clusters, which merge their states
  // through distributed shared memory, when every cluster fits at once.
  int cluster = 0;
  if (umma && p_align > units && p_align % units == 0 &&
      !(g_tuning & GQA_TUNE_NO_CLUSTER)) {
    const int k = static_cast<int>(p_align / units);
    if ((k == 2 || k == 4) &&
        max_clusters(dev, reinterpret_cast<const void*>(uvar.fn), uvar.smem,
                     kUmmaThreads, k) >= units) {
      cluster = k;
      grid = p_align;
    }
  }

  const size_t slots = static_cast<size_t>(grid) + static_cast<size_t>(units);
  const size_t lse_bytes = align_up(slots * rows_pad * 4, 256);
  const size_t o_bytes = slots * rows_pad * static_cast<size_t>(D) * 4;
  Scratch* sc = nullptr;
  if (scratch_for(dev, stream, static_cast<size_t>(units), lse_bytes + o_bytes,
                  &sc) != cudaSuccess)
    return GQA_ERR_CUDA;
  uint8_t* ctl = static_cast<uint8_t*>(sc->ctl);
  uint8_t* part = static_cast<uint8_t*>(sc->part);

  DecodeParams p = {};
  p.q = q;
  p.kc = paged ? nullptr : k;
  p.vc = paged ? nullptr : v;
  p.out = out;
  p.seq_lens = seq_lens;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.error = reinterpret_cast<uint32_t*>(ctl);
  p.counters = reinterpret_cast<unsigned long long*>(ctl + kHeaderBytes);
  sc->gen = next_gen(sc->gen);
  p.gen = sc->gen;
  p.wait_ns = g_wait_ns;
  p.part_lse = reinterpret_cast<float*>(part);
  p.part_o = reinterpret_cast<float*>(part + lse_bytes);
  p.scale_log2 = scale * 1.4426950408889634f;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Smax = Smax;
  p.G = G;
  p.T = T;
  p.GR = GR;
  p.NHC = NHC;
  p.R = R;
  p.p_align = p_align;
  p.cluster = cluster;
  p.tune = g_tuning;
  p.block_table = block_table;
  p.max_pages = paged ? Smax / page_size : 0;
  p.page_size = page_size;
  p.num_pages = num_pages;

  // Programmatic dependent launch: the kernel may start launching while the
  // previous kernel in the stream finishes; it waits (griddepcontrol.wait)
  // for that kernel's completion before it reads any global memory.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(umma ? kUmmaThreads : kThreads);
  cfg.dynamicSmemBytes = umma ? uvar.smem : var.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cluster > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  const cudaError_t le =
      umma ? cudaLaunchKernelEx(&cfg, uvar.fn, map_k, map_v, map_q, p)
           : cudaLaunchKernelEx(&cfg, var.fn, map_k, map_v, p);
  if (le != cudaSuccess) {
    (void)cudaGetLastError();
    return GQA_ERR_CUDA;
  }
  t_last_launches = 1;
  return GQA_OK;
}

}  // namespace
}  // namespace gqa

// ------------------------------------------------- fixed-scratch variant
//
// Scratch of gqa_decode_static: one array per GPU in the library's static
// device memory, [error word | arrival counters | partial log2-sum-exp |
// partial O].  It exists on every device that loads the library until the
// process exits, so its size is kept modest.
constexpr size_t kStaticScratchBytes = size_t(16) << 20;  // 16 MiB
static __device__ __align__(256) uint8_t gqa_static_scratch[kStaticScratchBytes];

namespace gqa {
namespace {

// Device address of gqa_static_scratch, looked up once per device (with
// that device current).  The host-side name of the array is only a stand-in:
// a kernel must be given this address instead.
std::map<int, void*> g_static_addr;
std::map<int, uint32_t> g_static_gen;  // last launch generation per device

cudaError_t static_scratch_addr(int dev, void** out) {
  auto it = g_static_addr.find(dev);
  if (it != g_static_addr.end()) {
    *out = it->second;
    return cudaSuccess;
  }
  void* ptr = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&ptr, gqa_static_scratch);
  if (e != cudaSuccess) return e;
  g_static_addr.emplace(dev, ptr);
  *out = ptr;
  return cudaSuccess;
}

// Same plan and kernel as launch(), with the scratch carved out of
// gqa_static_scratch instead of the per-stream allocation.
gqa_status launch_static(const void* q, const void* k, const void* v,
                         const int32_t* seq_lens, float scale, void* out,
                         int B, int Hq, int Hkv, int Smax, int D, int kv_kind,
                         bool q_bf16, void* stream_ptr) {
  t_last_launches = 0;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  const int G = Hq / Hkv;
  const int NHC = (G + kMaxUnitRows - 1) / kMaxUnitRows;
  const int R = (G + NHC - 1) / NHC;
  const int GR = G, T = 1;
  const int hb = R <= 16 ? 1 : (R <= 32 ? 2 : 4);
  const int rows_pad = hb * 16;
  const long long units = static_cast<long long>(B) * Hkv * NHC;
  if (units > INT32_MAX / 2) return GQA_ERR_UNSUPPORTED;

  const Variant var = pick(kv_kind, q_bf16, D, hb, R);
  CUtensorMap map_k, map_v;
  if (!make_cache_map(&map_k, k, 2, B, Hkv, Smax, D) ||
      !make_cache_map(&map_v, v, 2, B, Hkv, Smax, D))
    return GQA_ERR_CUDA;

  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GQA_ERR_CUDA;
  int sms = 0, per_sm = 0;
  if (configure(dev, var, &sms, &per_sm) != cudaSuccess) return GQA_ERR_CUDA;
  const long long max_tiles =
      units * ((static_cast<long long>(Smax) + kTileTokens - 1) / kTileTokens);
  const long long wave = static_cast<long long>(sms) * per_sm;
  const int grid = g_num_ctas_override > 0
                       ? g_num_ctas_override
                       : static_cast<int>(max_tiles < wave ? max_tiles : wave);

  const size_t slots = static_cast<size_t>(grid) + static_cast<size_t>(units);
  const size_t cnt_bytes =
      align_up(static_cast<size_t>(units) * kCounterBytes, 256);
  const size_t lse_bytes = align_up(slots * rows_pad * 4, 256);
  const size_t o_bytes = slots * rows_pad * static_cast<size_t>(D) * 4;
  const size_t need = kHeaderBytes + cnt_bytes + lse_bytes + o_bytes;
  if (need > kStaticScratchBytes) return GQA_ERR_UNSUPPORTED;

  void* base = nullptr;
  if (static_scratch_addr(dev, &base) != cudaSuccess) return GQA_ERR_CUDA;
  uint8_t* wb = static_cast<uint8_t*>(base);
  // The array keeps whatever the previous call left: the error word and the
  // arrival counters must start at zero.
  if (cudaMemsetAsync(wb, 0, kHeaderBytes + cnt_bytes, stream) != cudaSuccess)
    return GQA_ERR_CUDA;

  DecodeParams p = {};
  p.q = q;
  p.kc = k;
  p.vc = v;
  p.out = out;
  p.seq_lens = seq_lens;
  p.k_scale = nullptr;
  p.v_scale = nullptr;
  p.error = reinterpret_cast<uint32_t*>(wb);
  p.counters = reinterpret_cast<unsigned long long*>(wb + kHeaderBytes);
  uint32_t& gen = g_static_gen[dev];
  gen = next_gen(gen);
  p.gen = gen;
  p.wait_ns = g_wait_ns;
  p.part_lse = reinterpret_cast<float*>(wb + kHeaderBytes + cnt_bytes);
  p.part_o =
      reinterpret_cast<float*>(wb + kHeaderBytes + cnt_bytes + lse_bytes);
  p.scale_log2 = scale * 1.4426950408889634f;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Smax = Smax;
  p.G = G;
  p.T = T;
  p.GR = GR;
  p.NHC = NHC;
  p.R = R;
  p.p_align = g_num_ctas_override > 0 ? 0 : aligned_blocks(units, grid, hb);

  var.fn<<<grid, kThreads, var.smem, stream>>>(map_k, map_v, p);
  if (cudaGetLastError() != cudaSuccess) return GQA_ERR_CUDA;
  t_last_launches = 1;
  return GQA_OK;
}

}  // namespace
}  // namespace gqa

extern "C" {

gqa_status gqa_decode(const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* seq_lens, float scale, void* out, int B,
                      int Hq, int Hkv, int Smax, int D, gqa_dtype dtype,
                      void* stream) {
  gqa::t_last_launches = 0;
  if (dtype != GQA_F16 && dtype != GQA_BF16) return GQA_ERR_INVALID_ARG;
  const gqa_status st = gqa::check_common(q, k_cache, v_cache, seq_lens, scale,
                                          out, B, Hq, Hkv, Smax, D);
  if (st != GQA_OK) return st;
  try {
    return gqa::launch(q, k_cache, v_cache, nullptr, nullptr, seq_lens, scale,
                       out, B, Hq, Hkv, Smax, D,
                       dtype == GQA_BF16 ? gqa::kKvBF16 : gqa::kKvF16,
                       dtype == GQA_BF16, stream);
  } catch (...) {
    return GQA_ERR_CUDA;
  }
}

gqa_status gqa_decode_fp8(const void* q, const void* k_cache,
                          const void* v_cache, const float* k_scale,
                          const float* v_scale, const int32_t* seq_lens,
                          float scale, void* out, int B, int Hq, int Hkv,
                          int Smax, int D, gqa_dtype kv_dtype,
                          gqa_dtype qo_dtype, void* stream) {
  gqa::t_last_launches = 0;
  if (qo_dtype != GQA_F16 && qo_dtype != GQA_BF16) return GQA_ERR_INVALID_ARG;
  if (kv_dtype != GQA_E4M3 && kv_dtype != GQA_E5M2) return GQA_ERR_INVALID_ARG;
  if (!k_scale || !v_scale || !gqa::aligned(k_scale, 4) ||
      !gqa::aligned(v_scale, 4))
    return GQA_ERR_INVALID_ARG;
  const gqa_status st = gqa::check_common(q, k_cache, v_cache, seq_lens, scale,
                                          out, B, Hq, Hkv, Smax, D);
  if (st != GQA_OK) return st;
  try {
    return gqa::launch(q, k_cache, v_cache, k_scale, v_scale, seq_lens, scale,
                       out, B, Hq, Hkv, Smax, D,
                       kv_dtype == GQA_E5M2 ? gqa::kKvE5M2 : gqa::kKvE4M3,
                       qo_dtype == GQA_BF16, stream);
  } catch (...) {
    return GQA_ERR_CUDA;
  }
}

size_t gqa_kv_bytes_per_token(int layers, int kv_heads, int head_dim,
                              int bytes_per_elem) {
  if (layers <= 0 || kv_heads <= 0 || head_dim <= 0 || bytes_per_elem <= 0)
    return 0;
  return static_cast<size_t>(2) * static_cast<size_t>(layers) *
         static_cast<size_t>(kv_heads) * static_cast<size_t>(head_dim) *
         static_cast<size_t>(bytes_per_elem);
}

const char* gqa_status_string(gqa_status status) {
  switch (status) {
    case GQA_OK: return "ok";
    case GQA_ERR_INVALID_ARG: return "invalid argument";
    case GQA_ERR_UNSUPPORTED: return "unsupported configuration";
    case GQA_ERR_CUDA: return "CUDA error";
    case GQA_ERR_DEVICE: return "device-side fault reported by a kernel";
  }
  return "unknown status";
}

gqa_status gqa_device_errors(void* stream_ptr, uint32_t* flags) {
  if (!flags) return GQA_ERR_INVALID_ARG;
  *flags = 0;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  if (cudaStreamSynchronize(stream) != cudaSuccess) return GQA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(gqa::g_mu);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GQA_ERR_CUDA;
  auto it = gqa::g_scratch.find({dev, stream});
  if (it == gqa::g_scratch.end() || !it->second.ctl) return GQA_OK;
  uint32_t v = 0;
  if (cudaMemcpy(&v, it->second.ctl, 4, cudaMemcpyDeviceToHost) != cudaSuccess)
    return GQA_ERR_CUDA;
  if (v != 0 && cudaMemset(it->second.ctl, 0, 4) != cudaSuccess)
    return GQA_ERR_CUDA;
  // After a wait gave up some arrival counters may be left non-zero.  Later
  // launches ignore them (their generation differs), except replays of one
  // captured launch, which reuse its generation: clear them.
  if ((v & gqa::kErrWaitTimeout) &&
      cudaMemset(static_cast<uint8_t*>(it->second.ctl) + gqa::kHeaderBytes, 0,
                 it->second.ctl_units * gqa::kCounterBytes) != cudaSuccess)
    return GQA_ERR_CUDA;
  *flags = v;
  return GQA_OK;
}

void gqa_set_kernel_path(int path) {
  std::lock_guard<std::mutex> lock(gqa::g_mu);
  gqa::g_kernel_path = (path == 1 || path == 2) ? path : 0;
}

void gqa_set_tuning(int flags) {
  std::lock_guard<std::mutex> lock(gqa::g_mu);
  gqa::g_tuning = flags & (GQA_TUNE_NO_L2_WARMUP | GQA_TUNE_NO_CLUSTER |
                           GQA_TUNE_NO_NARROW_ROWS);
}

void gqa_set_wait_limit_ns(long long ns) {
  std::lock_guard<std::mutex> lock(gqa::g_mu);
  gqa::g_wait_ns = ns < 0 ? gqa::kWaitLimitNs : static_cast<uint64_t>(ns);
}

void gqa_set_num_ctas(int num_ctas) {
  std::lock_guard<std::mutex> lock(gqa::g_mu);
  gqa::g_num_ctas_override = num_ctas > 0 ? num_ctas : 0;
}

gqa_status gqa_append_kv(const void* k_new, const void* v_new, void* k_cache,
                         void* v_cache, float* k_scale, float* v_scale,
                         int32_t* seq_lens, int B, int Hkv, int Smax, int D,
                         gqa_dtype in_dtype, gqa_dtype cache_dtype,
                         void* stream_ptr) {
  using namespace gqa;
  t_last_launches = 0;
  if (in_dtype != GQA_F16 && in_dtype != GQA_BF16) return GQA_ERR_INVALID_ARG;
  const bool fp8 = cache_dtype == GQA_E4M3 || cache_dtype == GQA_E5M2;
  if (!fp8 && cache_dtype != in_dtype) return GQA_ERR_INVALID_ARG;
  if (!k_new || !v_new || !k_cache || !v_cache || !seq_lens)
    return GQA_ERR_INVALID_ARG;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) ||
      !aligned(v_cache, 16) || !aligned(seq_lens, 4))
    return GQA_ERR_INVALID_ARG;
  if (fp8 && (!k_scale || !v_scale || !aligned(k_scale, 4) ||
              !aligned(v_scale, 4)))
    return GQA_ERR_INVALID_ARG;
  if (B < 1 || Hkv < 1 || Smax < 1) return GQA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return GQA_ERR_UNSUPPORTED;
  try {
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    std::lock_guard<std::mutex> lock(g_mu);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GQA_ERR_CUDA;
    Scratch* sc = nullptr;  // only its error word is used
    if (scratch_for(dev, stream, 1, 1, &sc) != cudaSuccess) return GQA_ERR_CUDA;
    AppendParams p = {};
    p.k_new = k_new;
    p.v_new = v_new;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    p.seq_lens = seq_lens;
    p.error = static_cast<uint32_t*>(sc->ctl);
    p.B = B;
    p.Hkv = Hkv;
    p.Smax = Smax;
    p.D = D;
    const bool bf16 = in_dtype == GQA_BF16;
    void (*fn)(const AppendParams) =
        cache_dtype == GQA_E4M3
            ? (bf16 ? gqa_append_kernel<true, kKvE4M3>
                    : gqa_append_kernel<false, kKvE4M3>)
        : cache_dtype == GQA_E5M2
            ? (bf16 ? gqa_append_kernel<true, kKvE5M2>
                    : gqa_append_kernel<false, kKvE5M2>)
            : (bf16 ? gqa_append_kernel<true, kKvBF16>
                    : gqa_append_kernel<false, kKvF16>);
    fn<<<B, kAppendThreads, 0, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return GQA_ERR_CUDA;
    t_last_launches = 1;
    return GQA_OK;
  } catch (...) {
    return GQA_ERR_CUDA;
  }
}

gqa_status gqa_decode_chunk(const void* q, const void* k_cache,
                            const void* v_cache, const int32_t* seq_lens,
                            float scale, void* out, int B, int Hq, int Hkv,
                            int T, int Smax, int D, gqa_dtype dtype,
                            void* stream) {
  gqa::t_last_launches = 0;
  if (dtype != GQA_F16 && dtype != GQA_BF16) return GQA_ERR_INVALID_ARG;
  if (T < 1) return GQA_ERR_INVALID_ARG;
  const gqa_status st = gqa::check_common(q, k_cache, v_cache, seq_lens, scale,
                                          out, B, Hq, Hkv, Smax, D);
  if (st != GQA_OK) return st;
  if (static_cast<long long>(B) * Hq * T > INT32_MAX ||
      static_cast<long long>(Hq / Hkv) * T > INT32_MAX / 2)
    return GQA_ERR_UNSUPPORTED;
  try {
    return gqa::launch(q, k_cache, v_cache, nullptr, nullptr, seq_lens, scale,
                       out, B, Hq, Hkv, Smax, D,
                       dtype == GQA_BF16 ? gqa::kKvBF16 : gqa::kKvF16,
                       dtype == GQA_BF16, stream, nullptr, 0, 0, T);
  } catch (...) {
    return GQA_ERR_CUDA;
  }
}

gqa_status gqa_decode_paged(const void* q, const void* k_pages,
                            const void* v_pages, const int32_t* block_table,
                            const int32_t* seq_lens, float scale, void* out,
                            int B, int Hq, int Hkv, int num_pages,
                            int page_size, int max_pages, int D,
                            gqa_dtype dtype, void* stream) {
  gqa::t_last_launches = 0;
  if (dtype != GQA_F16 && dtype != GQA_BF16) return GQA_ERR_INVALID_ARG;
  if (!block_table || !gqa::aligned(block_table, 4)) return GQA_ERR_INVALID_ARG;
  if (num_pages < 1 || max_pages < 1 || page_size < 1)
    return GQA_ERR_INVALID_ARG;
  if (page_size % gqa::kTileTokens != 0) return GQA_ERR_UNSUPPORTED;
  const long long smax = static_cast<long long>(max_pages) * page_size;
  if (smax > INT32_MAX ||
      static_cast<long long>(num_pages) * Hkv > INT32_MAX)
    return GQA_ERR_UNSUPPORTED;
  const gqa_status st =
      gqa::check_common(q, k_pages, v_pages, seq_lens, scale, out, B, Hq, Hkv,
                        static_cast<int>(smax), D);
  if (st != GQA_OK) return st;
  try {
    return gqa::launch(q, k_pages, v_pages, nullptr, nullptr, seq_lens, scale,
                       out, B, Hq, Hkv, static_cast<int>(smax), D,
                       dtype == GQA_BF16 ? gqa::kKvBF16 : gqa::kKvF16,
                       dtype == GQA_BF16, stream, block_table, page_size,
                       num_pages);
  } catch (...) {
    return GQA_ERR_CUDA;
  }
}

gqa_status gqa_decode_static(const void* q, const void* k_cache,
                             const void* v_cache, const int32_t* seq_lens,
                             float scale, void* out, int B, int Hq, int Hkv,
                             int Smax, int D, gqa_dtype dtype, void* stream) {
  gqa::t_last_launches = 0;
  if (dtype != GQA_F16 && dtype != GQA_BF16) return GQA_ERR_INVALID_ARG;
  const gqa_status st = gqa::check_common(q, k_cache, v_cache, seq_lens, scale,
                                          out, B, Hq, Hkv, Smax, D);
  if (st != GQA_OK) return st;
  try {
    return gqa::launch_static(q, k_cache, v_cache, seq_lens, scale, out, B, Hq,
                              Hkv, Smax, D,
                              dtype == GQA_BF16 ? gqa::kKvBF16 : gqa::kKvF16,
                              dtype == GQA_BF16, stream);
  } catch (...) {
    return GQA_ERR_CUDA;
  }
}

int gqa_last_launch_count(void) { return gqa::t_last_launches; }

gqa_status gqa_release_stream(void* stream_ptr) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  std::lock_guard<std::mutex> lock(gqa::g_mu);
  if (gqa::g_scratch.empty()) return GQA_OK;  // nothing held: no CUDA call
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GQA_ERR_CUDA;
  auto it = gqa::g_scratch.find({dev, stream});
  if (it == gqa::g_scratch.end()) return GQA_OK;
  gqa::Scratch& s = it->second;
  gqa_status st = GQA_OK;
  if (s.ctl && cudaFreeAsync(s.ctl, stream) != cudaSuccess) st = GQA_ERR_CUDA;
  if (s.part && cudaFreeAsync(s.part, stream) != cudaSuccess)
    st = GQA_ERR_CUDA;
  gqa::g_scratch.erase(it);
  if (st != GQA_OK) (void)cudaGetLastError();
  return st;
}

}  // extern "C"
