// gqa_umma.cu — instantiations of the tensor-core (tcgen05) decode kernel
// (gqa_decode_umma.cuh), in a translation unit of their own.
#include "gqa_umma.h"

namespace gqa {

namespace {

template <bool QBF16, bool PAGED>
UmmaVariant pick_cols(int rows) {
  return rows <= 32
             ? UmmaVariant{&gqa_decode_umma_kernel<QBF16, 32, PAGED>,
                           kUmmaSmemBytes}
             : UmmaVariant{&gqa_decode_umma_kernel<QBF16, 64, PAGED>,
                           kUmmaSmemBytes};
}

}  // namespace

UmmaVariant umma_variant(bool q_bf16, int rows, bool paged) {
  if (q_bf16)
    return paged ? pick_cols<true, true>(rows) : pick_cols<true, false>(rows);
  return paged ? pick_cols<false, true>(rows) : pick_cols<false, false>(rows);
}

}  // namespace gqa
