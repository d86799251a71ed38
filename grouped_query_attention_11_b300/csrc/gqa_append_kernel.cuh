// gqa_append_kernel.cuh — the cache-append step before the decode step, for
// sm_103a.
//
// What one launch computes: for every sequence b with L_b = seq_lens[b] <
// Smax, the new token's K and V rows of every KV head are written at cache
// position L_b and seq_lens[b] becomes L_b + 1 ("Grouped Query Attention
// (GQA): Efficient Multi-Head Attention", The bottleneck: the cache grows by
// one token's K and V per decoding step).  16-bit caches receive the rows as
// they are.  8-bit caches ("Grouped-Query Attention: How Sharing KV Heads
// Shrinks Inference Memory", FP8 KV cache: codes with scaling factors) keep
// one fp32 scale per (sequence, KV head) and tensor, and decide every code in
// fp32 with IEEE division and round-to-nearest-even:
//   a = max_d |x_d|;
//   an unset scale (<= 0) becomes a / MAX (1 when a == 0);
//   otherwise the scale doubles until a / scale <= MAX, and when it grew the
//   earlier codes of that (sequence, KV head) are re-encoded with the ratio
//   old / new, a power of two, so they change only where they fall below the
//   format's normal range;
//   the new row's codes are x_d / scale.
// A sequence whose cache is full is left unchanged and raises an error bit.
//
// One block per sequence; the block reads L_b once, writes every head (16-bit
// pieces all at once; one warp per 8-bit row), then bumps seq_lens[b], so the
// heads of a sequence never race on its length.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>
#include <cstring>
#include <type_traits>

#include "gqa_decode_kernel.cuh"

namespace gqa {

constexpr int kAppendThreads = 128;

struct AppendParams {
  const void* k_new;   // [B, Hkv, D] f16 / bf16
  const void* v_new;
  void* k_cache;       // [B, Hkv, Smax, D] 16-bit or 8-bit codes
  void* v_cache;
  float* k_scale;      // [B, Hkv] (8-bit caches), updated in place
  float* v_scale;
  int32_t* seq_lens;   // [B], read then incremented
  uint32_t* error;     // fault flags
  int B, Hkv, Smax, D;
};

template <int KV>
__device__ __forceinline__ float fp8_max_value() {
  return KV == kKvE5M2 ? 57344.f : 448.f;
}

// Two fp32 values -> two 8-bit codes, round to nearest even, clamped to the
// largest finite value; x0 lands in the low byte.
template <int KV>
__device__ __forceinline__ uint32_t encode2(float x0, float x1) {
  uint16_t r;
  if constexpr (KV == kKvE5M2) {
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(x1), "f"(x0));
  } else {
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(x1), "f"(x0));
  }
  return r;
}

__device__ __forceinline__ float2 f16x2_to_float2(uint32_t w) {
  __half2 h;
  memcpy(&h, &w, sizeof(h));
  return __half22float2(h);
}

template <bool IN_BF16, int KV>
__global__ void __launch_bounds__(kAppendThreads)
    gqa_append_kernel(const AppendParams p) {
  using QT = typename std::conditional<IN_BF16, __nv_bfloat16, __half>::type;
  constexpr int kWarps = kAppendThreads / 32;

  const int b = blockIdx.x, tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  int L = __ldg(p.seq_lens + b);
  L = L < 0 ? 0 : L;
  if (L >= p.Smax) {
    if (tid == 0) atomicOr(p.error, kErrCacheFull);
    return;
  }
  const int D = p.D;
  if constexpr (!is_fp8(KV)) {
    // 16-bit cache: every 16-byte piece of every row is independent
    const int per_row = D / 8;
    const int n = p.Hkv * 2 * per_row;
    for (int i = tid; i < n; i += kAppendThreads) {
      const int which = i / (p.Hkv * per_row);
      const int rem = i % (p.Hkv * per_row);
      const size_t row = static_cast<size_t>(b) * p.Hkv + rem / per_row;
      const int c = rem % per_row;
      const QT* src = static_cast<const QT*>(which ? p.v_new : p.k_new);
      QT* dst = static_cast<QT*>(which ? p.v_cache : p.k_cache);
      reinterpret_cast<uint4*>(dst + (row * p.Smax + L) * D)[c] =
          reinterpret_cast<const uint4*>(src + row * D)[c];
    }
  } else {
    // 8-bit cache: one warp per (KV head, tensor) row; lane l holds the
    // D/32 consecutive elements l*D/32 ..
    const float M = fp8_max_value<KV>();
    constexpr int kMaxPer = 4;  // D / 32 for D = 128
    const int per = D / 32;
    for (int rw = warp; rw < p.Hkv * 2; rw += kWarps) {
      const int which = rw / p.Hkv;
      const size_t row = static_cast<size_t>(b) * p.Hkv + rw % p.Hkv;
      const QT* src = static_cast<const QT*>(which ? p.v_new : p.k_new);
      uint8_t* codes = static_cast<uint8_t*>(which ? p.v_cache : p.k_cache);
      float* scales = which ? p.v_scale : p.k_scale;
      float x[kMaxPer];
      float a = 0.f;
#pragma unroll
      for (int i = 0; i < kMaxPer; ++i) {
        x[i] = i < per ? to_f32<QT>(src[row * D + lane * per + i]) : 0.f;
        a = fmaxf(a, fabsf(x[i]));
      }
      for (int o = 16; o > 0; o >>= 1)
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
      float s = 0.f, s2 = 0.f;
      if (lane == 0) {
        s = scales[row];
        if (!(s > 0.f)) {
          s2 = a > 0.f ? __fdiv_rn(a, M) : 1.f;
        } else {
          s2 = s;
          for (int it = 0; it < 256 && __fdiv_rn(a, s2) > M; ++it)
            s2 = s2 * 2.f;
        }
        scales[row] = s2;
      }
      s = __shfl_sync(0xffffffffu, s, 0);
      s2 = __shfl_sync(0xffffffffu, s2, 0);
      if (s > 0.f && s2 != s) {
        // the scale grew: re-encode the L earlier tokens, 4 codes a lane
        const float ratio = __fdiv_rn(s, s2);
        uint32_t* w4 = reinterpret_cast<uint32_t*>(codes + row * p.Smax * D);
        const int n4 = L * D / 4;
        for (int i = lane; i < n4; i += 32) {
          const uint32_t c = w4[i];
          const float2 lo = f16x2_to_float2(fp8_lo<KV>(c));
          const float2 hi = f16x2_to_float2(fp8_hi<KV>(c));
          w4[i] = encode2<KV>(lo.x * ratio, lo.y * ratio) |
                  (encode2<KV>(hi.x * ratio, hi.y * ratio) << 16);
        }
      }
      uint8_t* dst = codes + (row * p.Smax + L) * D + lane * per;
      if (per == 4) {
        *reinterpret_cast<uint32_t*>(dst) =
            encode2<KV>(__fdiv_rn(x[0], s2), __fdiv_rn(x[1], s2)) |
            (encode2<KV>(__fdiv_rn(x[2], s2), __fdiv_rn(x[3], s2)) << 16);
      } else {
        *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(
            encode2<KV>(__fdiv_rn(x[0], s2), __fdiv_rn(x[1], s2)));
      }
    }
  }
  __syncthreads();
  if (tid == 0) p.seq_lens[b] = L + 1;
}

}  // namespace gqa
