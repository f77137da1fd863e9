// k_reduce_ftz.cu -- the flush-to-zero instantiations of the replica-reduce
// kernel (k_reduce.cuh), compiled as a translation unit of their own so that the two
// arithmetic modes build in parallel.
#include "k_reduce.cuh"

namespace repstep {

ReduceKernelFn pick_reduce_ftz(const ReduceShape &s) { return pick_reduce<1>(s); }

}  // namespace repstep
