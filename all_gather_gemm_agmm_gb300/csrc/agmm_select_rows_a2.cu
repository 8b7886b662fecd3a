// agmm_select_rows_a2.cu -- the row-tile variants of the fused kernel with
// two k blocks per pipeline stage.
#include "agmm_fused_kernel.cuh"

namespace agmm {

KernelFn select_rows_kernel_a2(const KernelKey& k) {
#define AGMM_PICK_ROWS(BN, CM, PAIR) \
  (k.store ? AGMM_FUSED_PICK(kPathRows, BN, CM, PAIR, 2, true) : AGMM_FUSED_PICK(kPathRows, BN, CM, PAIR, 2, false))
  if (k.path != kPathRows || k.atoms != 2) return nullptr;
  if (k.cm == 1 && !k.pair) {
    if (k.bn == 256) return AGMM_PICK_ROWS(256, 1, false);
    if (k.bn == 128) return AGMM_PICK_ROWS(128, 1, false);
  } else if (k.cm == 2 && k.pair) {
    if (k.bn == 256) return AGMM_PICK_ROWS(256, 2, true);
    if (k.bn == 128) return AGMM_PICK_ROWS(128, 2, true);
  }
  return nullptr;
#undef AGMM_PICK_ROWS
}

}  // namespace agmm
