// gqa_umma.h — entry of the tensor-core (tcgen05) decode kernel for the host
// code in gqa_api.cu.  The kernel is compiled in its own translation unit
// (gqa_umma.cu); this header gives its launch signature, its constants and
// the instantiation for a launch.
#pragma once

#include <cuda.h>

#include "gqa_decode_umma.cuh"

namespace gqa {

using UmmaKernelFn = void (*)(const CUtensorMap, const CUtensorMap,
                              const CUtensorMap, const DecodeParams);

struct UmmaVariant {
  UmmaKernelFn fn;
  int smem;  // dynamic shared memory per block
};

// The instantiation for q / out in bf16 (else f16), units of `rows` query
// rows (17 .. 64; up to 32 use the 32-column softmax) and a contiguous or
// paged cache.
UmmaVariant umma_variant(bool q_bf16, int rows, bool paged);

}  // namespace gqa
