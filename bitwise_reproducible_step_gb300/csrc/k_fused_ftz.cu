// k_fused_ftz.cu -- the flush-to-zero instantiations of the single-pass kernel
// (k_fused.cuh), compiled as a translation unit of their own so that the two arithmetic
// modes build in parallel.
#include "k_fused.cuh"

namespace repstep {

FusedKernelFn pick_fused_ftz(const FusedShape &s) { return pick_fused<1>(s); }

}  // namespace repstep
