// gqa_umma.cu — instantiations of the tensor-core (tcgen05) decode kernel
// (gqa_decode_umma.cuh), in a translation unit of their own.
#include "gqa_umma.h"

namespace gqa {

UmmaVariant umma_variant(bool q_bf16, int rows) {
  if (q_bf16)
    return rows <= 32 ? UmmaVariant{&gqa_decode_umma_kernel<true, 32>,
                                    kUmmaSmemBytes}
                      : UmmaVariant{&gqa_decode_umma_kernel<true, 64>,
                                    kUmmaSmemBytes};
  return rows <= 32
             ? UmmaVariant{&gqa_decode_umma_kernel<false, 32>, kUmmaSmemBytes}
             : UmmaVariant{&gqa_decode_umma_kernel<false, 64>, kUmmaSmemBytes};
}

}  // namespace gqa
