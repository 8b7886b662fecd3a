// agmm_select_swap.cu -- the swapped-tile variants of the fused kernel.
#include "agmm_fused_kernel.cuh"

namespace agmm {

KernelFn select_swap_kernel(const KernelKey& k) {
  if (k.path != kPathSwap || k.cm != 1 || k.pair || k.store) return nullptr;
  return k.atoms == 2 ? AGMM_FUSED_PICK(kPathSwap, 128, 1, false, 2, false)
                      : AGMM_FUSED_PICK(kPathSwap, 128, 1, false, 1, false);
}

}  // namespace agmm
