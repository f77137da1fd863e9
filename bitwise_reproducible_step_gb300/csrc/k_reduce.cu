// k_reduce.cu -- the IEEE instantiations of the replica-reduce kernel (k_reduce.cuh) and
// the host-side helpers that size, prepare and launch any reduce variant.
#include "k_reduce.cuh"

namespace repstep {

ReduceKernelFn pick_reduce_ieee(const ReduceShape &s) { return pick_reduce<0>(s); }

namespace {

ReduceKernelFn pick(const ReduceShape &s)
{
    return s.fz ? pick_reduce_ftz(s) : pick_reduce_ieee(s);
}

}  // namespace

size_t reduce_smem_bytes(const ReduceShape &s, ReduceArgs &args)
{
    const uint32_t esz = s.dtype == 1 ? 2u : 4u;
    const uint32_t te = 4u * uint32_t(s.nt);
    const uint32_t per_stage = (args.R < uint32_t(s.rg) ? args.R : uint32_t(s.rg));
    const uint32_t stride = (s.mode != 0 ? 8u : per_stage) * te * esz;
    uint32_t stages = kRingBytes / stride;
    if (stages > kMaxStages) stages = kMaxStages;
    if (stages < 2) stages = 2;
    args.stages = stages;
    args.stage_stride = stride;
    return size_t(kRingOffset) + size_t(stages) * stride;
}

cudaError_t reduce_prepare(const ReduceShape &s, size_t smem)
{
    ReduceKernelFn f = pick(s);
    if (!f) return cudaErrorInvalidValue;
    return cudaFuncSetAttribute(reinterpret_cast<const void *>(f),
                                cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
}

cudaError_t reduce_occupancy(const ReduceShape &s, size_t smem, int *blocks_per_sm)
{
    ReduceKernelFn f = pick(s);
    if (!f) return cudaErrorInvalidValue;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        blocks_per_sm, reinterpret_cast<const void *>(f), s.nt + 32, smem);
}

cudaError_t launch_reduce(const ReduceShape &s, const ReduceArgs &args, int grid, size_t smem,
                          cudaStream_t st)
{
    ReduceKernelFn f = pick(s);
    if (!f) return cudaErrorInvalidValue;
    // the kernel hands out chunks from this counter
    cudaError_t e = cudaMemsetAsync(&args.sc->next_chunk, 0, sizeof(uint32_t), st);
    if (e != cudaSuccess) return e;
    void *params[] = {const_cast<ReduceArgs *>(&args)};
    return cudaLaunchKernel(reinterpret_cast<const void *>(f), dim3(grid), dim3(s.nt + 32),
                            params, smem, st);
}

}  // namespace repstep
