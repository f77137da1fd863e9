// k_adamw_ftz.cu -- the flush-to-zero instantiations of the AdamW / leaf kernel
// (k_adamw.cuh), a translation unit of their own so that the two arithmetic modes build
// in parallel.
#include "k_adamw.cuh"

namespace repstep {

AdamwKernelFn pick_adamw_ftz(const AdamwShape &s) { return pick_adamw<1>(s); }

}  // namespace repstep
