// k_fused_ftz.cu -- the flush-to-zero instantiations of the single-pass kernel
// (k_fused.cuh) for R = 4 and 8, compiled as a translation unit of their own so that the
// variants build in parallel.
#include "k_fused.cuh"

namespace repstep {

FusedKernelFn pick_fused_ftz(const FusedShape &s) { return pick_fused<1, 0>(s); }

}  // namespace repstep
