// k_adamw.cu -- the IEEE instantiations of the AdamW / leaf kernel (k_adamw.cuh), the
// self-test of its fixed-divisor division, and the host-side helpers that size, prepare
// and launch any AdamW variant.
#include "k_adamw.cuh"

namespace repstep {

AdamwKernelFn pick_adamw_ieee(const AdamwShape &s) { return pick_adamw<0>(s); }

namespace {

// Self-test of div_fast: every significand pair x, b in [1, 2) (2^23 x 2^23), with y the
// correctly rounded reciprocal of b, against the IEEE division.  Exponents only scale the
// operands and results by powers of two, exactly, inside the guarded range, so this
// covers every x and b the fast path accepts.
__global__ void __launch_bounds__(256) k_selftest_div(uint32_t b_begin, uint32_t b_count,
                                                      unsigned long long *mismatches)
{
    unsigned long long bad = 0;
    for (uint32_t bi = blockIdx.x; bi < b_count; bi += gridDim.x) {
        const float b = __uint_as_float(0x3F800000u | ((b_begin + bi) & 0x7FFFFFu));
        const float y = __frcp_rn(b);
        for (uint32_t xs = threadIdx.x; xs < (1u << 23); xs += blockDim.x) {
            const float x = __uint_as_float(0x3F800000u | xs);
            bad += __float_as_uint(div_fast(x, b, y)) != __float_as_uint(__fdiv_rn(x, b));
        }
    }
    if (bad) atomicAdd(mismatches, bad);
}

// Self-test of the branch-free square root, reciprocal and division against the IEEE
// operations.  which 0: sqrt_rn_fast(x) for the float bit patterns [begin, begin + count);
// 1: rcp_rn_fast(b) for those patterns; 2: div_rn_fast(a, b) for count x 1024 pseudo-random
// pairs from `seed`: b in [2^-41, 2^41), a = +-0 or |a| in [2^-85, 2^81), either sign.
__device__ __forceinline__ uint64_t st_mix(uint64_t z)
{
    z += 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

__global__ void __launch_bounds__(256) k_selftest_fast_math(int which, uint32_t begin,
                                                            uint32_t count, uint64_t seed,
                                                            unsigned long long *mismatches)
{
    unsigned long long bad = 0;
    const uint64_t total = which == 2 ? uint64_t(count) * 1024u : uint64_t(count);
    const uint64_t stride = uint64_t(gridDim.x) * blockDim.x;
    for (uint64_t i = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
        if (which == 0) {
            const float x = __uint_as_float(begin + uint32_t(i));
            bad += __float_as_uint(sqrt_rn_fast(x)) != __float_as_uint(__fsqrt_rn(x));
        } else if (which == 1) {
            const float b = __uint_as_float(begin + uint32_t(i));
            bad += __float_as_uint(rcp_rn_fast(b)) != __float_as_uint(__frcp_rn(b));
        } else {
            const uint64_t r = st_mix(seed ^ (i * 0xD1B54A32D192ED03ull));
            const uint32_t b_lo = 0x2B000000u, b_hi = 0x54000000u;     // 2^-41, 2^41
            const uint32_t a_lo = 0x15000000u, a_hi = 0x68000000u;     // 2^-85, 2^81
            const float b = __uint_as_float(b_lo + uint32_t(r % (b_hi - b_lo)));
            uint32_t ab = a_lo + uint32_t((r >> 32) % (a_hi - a_lo));
            if (((r >> 58) & 63u) == 0u) ab = 0u;                       // zeros now and then
            const float a = __uint_as_float(ab | (uint32_t(r >> 57) & 1u) << 31);
            bad += __float_as_uint(div_rn_fast(a, b)) != __float_as_uint(__fdiv_rn(a, b));
        }
    }
    if (bad) atomicAdd(mismatches, bad);
}

// The leaves-only mode has one (IEEE) instantiation; the others follow the arithmetic mode.
AdamwKernelFn pick(const AdamwShape &s)
{
    return (s.fz && s.mode != 1) ? pick_adamw_ftz(s) : pick_adamw_ieee(s);
}

uint32_t ring_off(int nt)
{
    return nt == 128 ? ring_offset<128>() : (nt == 256 ? ring_offset<256>() : ring_offset<512>());
}

uint32_t ring_bytes(int nt)
{
    return nt == 128 ? Shape<128>::ring : (nt == 256 ? Shape<256>::ring : Shape<512>::ring);
}

}  // namespace

size_t adamw_smem_bytes(const AdamwShape &s, AdamwArgs &args)
{
    const uint32_t ns = s.mode == 1 ? 3u : 4u;
    const uint32_t per_elem = 4u * ns - (s.pt ? 2u : 0u);     // w is 2 bytes when bf16
    const uint32_t te = uint32_t(kEPT) * uint32_t(s.nt);
    // a stage holds the streams' tiles, plus the tile's decay bits when a mask is set
    const uint32_t mask_bytes = (s.mode != 1 && s.mk) ? te / 8u : 0u;
    const uint32_t stride = per_elem * te + mask_bytes;
    uint32_t stages = ring_bytes(s.nt) / (per_elem * te);
    if (stages > kMaxStages) stages = kMaxStages;
    if (stages < 2) stages = 2;
    args.stages = stages;
    args.stage_stride = stride;
    return size_t(ring_off(s.nt)) + size_t(stages) * stride;
}

cudaError_t adamw_prepare(const AdamwShape &s, size_t smem)
{
    AdamwKernelFn f = pick(s);
    if (!f) return cudaErrorInvalidValue;
    return cudaFuncSetAttribute(reinterpret_cast<const void *>(f),
                                cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
}

cudaError_t adamw_occupancy(const AdamwShape &s, size_t smem, int *blocks_per_sm)
{
    AdamwKernelFn f = pick(s);
    if (!f) return cudaErrorInvalidValue;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        blocks_per_sm, reinterpret_cast<const void *>(f), s.nt + 64, smem);
}

cudaError_t launch_selftest_div(uint32_t b_begin, uint32_t b_count, unsigned long long *mismatches,
                               cudaStream_t st)
{
    k_selftest_div<<<152 * 8, 256, 0, st>>>(b_begin, b_count, mismatches);
    return cudaGetLastError();
}

cudaError_t launch_selftest_fast_math(int which, uint32_t begin, uint32_t count, uint64_t seed,
                                      unsigned long long *mismatches, cudaStream_t st)
{
    k_selftest_fast_math<<<152 * 8, 256, 0, st>>>(which, begin, count, seed, mismatches);
    return cudaGetLastError();
}

cudaError_t launch_adamw(const AdamwShape &s, const AdamwArgs &args, int grid, size_t smem,
                         cudaStream_t st)
{
    AdamwKernelFn f = pick(s);
    if (!f) return cudaErrorInvalidValue;
    // the kernel hands out chunks from this counter
    cudaError_t e = cudaMemsetAsync(&args.sc->next_chunk, 0, sizeof(uint32_t), st);
    if (e != cudaSuccess) return e;
    void *params[] = {const_cast<AdamwArgs *>(&args)};
    return cudaLaunchKernel(reinterpret_cast<const void *>(f), dim3(grid), dim3(s.nt + 64),
                            params, smem, st);
}

}  // namespace repstep
