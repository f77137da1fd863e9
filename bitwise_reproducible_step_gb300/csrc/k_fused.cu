// k_fused.cu -- the IEEE instantiations of the single-pass kernel (k_fused.cuh) for R = 4
// and 8, and the host-side helpers that size, prepare and launch any of its variants.
#include "k_fused.cuh"

namespace repstep {

FusedKernelFn pick_fused_ieee(const FusedShape &s) { return pick_fused<0, 0>(s); }

namespace {

FusedKernelFn pick_any(const FusedShape &s)
{
    if (s.rg == 16) return s.fz ? pick_fused_wide_ftz(s) : pick_fused_wide_ieee(s);
    return s.fz ? pick_fused_ftz(s) : pick_fused_ieee(s);
}

}  // namespace

size_t fused_smem_bytes(const FusedShape &s, FusedArgs &args)
{
    constexpr uint32_t TE = 4u * kFusedNT;
    const uint32_t es = s.dtype == 1 ? 2u : 4u;
    // as the kernel's GS: gradient stages of at most 64 KB
    const uint32_t per = TE * es;
    const uint32_t gs_bytes = 64u * 1024u / per;
    const uint32_t gs = s.rg < 8 ? uint32_t(s.rg) : (gs_bytes < 8u ? gs_bytes : 8u);
    const uint32_t grad_stage = gs * per;
    const uint32_t state_stage = 3u * TE * 4u + (s.mk ? TE / 8u : 0u);   // w, m, v, mask bits
    const uint32_t big = grad_stage > state_stage ? grad_stage : state_stage;
    const uint32_t stride = (big + 1023) / 1024 * 1024;
    uint32_t stages = kFusedRing / stride;
    if (stages > kFusedMaxStages) stages = kFusedMaxStages;
    if (stages < 2) stages = 2;
    args.adam.stages = stages;
    args.adam.stage_stride = stride;
    return size_t(fused_ring_offset<kFusedNT, int(kChunk / TE)>()) + size_t(stages) * stride;
}

cudaError_t fused_prepare(const FusedShape &s, size_t smem)
{
    FusedKernelFn f = pick_any(s);
    if (!f) return cudaErrorInvalidValue;
    return cudaFuncSetAttribute(reinterpret_cast<const void *>(f),
                                cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
}

cudaError_t fused_occupancy(const FusedShape &s, size_t smem, int *blocks_per_sm)
{
    FusedKernelFn f = pick_any(s);
    if (!f) return cudaErrorInvalidValue;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, reinterpret_cast<const void *>(f),
                                                         kFusedNT + 64, smem);
}

cudaError_t launch_fused(const FusedShape &s, const FusedArgs &args, int grid, size_t smem,
                         cudaStream_t st, cudaEvent_t ev_begin, cudaEvent_t ev_end)
{
    FusedKernelFn f = pick_any(s);
    if (!f) return cudaErrorInvalidValue;
    // the kernel hands out chunks from this counter
    cudaError_t e = cudaMemsetAsync(&args.adam.sc->next_chunk, 0, sizeof(uint32_t), st);
    if (e == cudaSuccess && ev_begin) e = cudaEventRecord(ev_begin, st);
    if (e != cudaSuccess) return e;
    void *params[] = {const_cast<FusedArgs *>(&args)};
    e = cudaLaunchKernel(reinterpret_cast<const void *>(f), dim3(grid), dim3(kFusedNT + 64),
                         params, smem, st);
    if (e == cudaSuccess && ev_end) e = cudaEventRecord(ev_end, st);
    return e;
}

}  // namespace repstep
