// k_blake2b.cu -- audit-mode leaf digests: BLAKE2b-64 (RFC 7693) of each leaf's bytes in
// the checkpoint image.  Leaf 0 is the 8-byte header [LE int32 step][LE uint32 n]; leaf
// 1 + a*c + k is chunk k (4096 elements, the last one short) of array a in (w, m, v), as
// little-endian fp32 bytes.  ("OPEN-1B: A Fully Auditable Training Run", App. B: every step
// is hashed with blake2b; this mode uses it for the leaves as well as the Merkle nodes.)
//
// BLAKE2b is a sequential chain over 128-byte blocks, so each leaf is one thread's chain of
// 128 compressions; the 1 + 3c leaves give the parallelism.  The work is ALU-bound (about
// 2,200 integer instructions per 128 bytes), far from the HBM bound of the PF61 leaves.
// A bf16 w is digested as its exactly widened fp32 words (the image's layout).
#include "common.cuh"
#include "kernels.h"

namespace repstep {

namespace {

// 32-bit word e of array a: fp32 bits, or a bf16 w widened.
__device__ __forceinline__ uint32_t word_of(const void *arr, bool narrow, uint64_t e)
{
    return narrow ? uint32_t(__ldg(static_cast<const unsigned short *>(arr) + e)) << 16
                  : __ldg(static_cast<const uint32_t *>(arr) + e);
}

__global__ void __launch_bounds__(256) k_leaves_b2(const void *w, int w_bf16, const float *m,
                                                   const float *v, uint64_t n, uint64_t c,
                                                   uint64_t *leaves, uint32_t step)
{
    const uint64_t total = 1 + 3 * c;
    const uint64_t stride = uint64_t(gridDim.x) * blockDim.x;
    for (uint64_t L = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x; L < total; L += stride) {
        uint64_t h[8];
        b2_init64(h);
        if (L == 0) {
            uint64_t msg[16] = {};
            msg[0] = uint64_t(step) | (uint64_t(uint32_t(n)) << 32);
            b2_compress(h, msg, 8, true);
            leaves[0] = h[0];
            continue;
        }
        const uint64_t a = (L - 1) / c, k = (L - 1) % c;
        const void *arr = a == 0 ? w : (a == 1 ? static_cast<const void *>(m) : v);
        const bool narrow = a == 0 && w_bf16;
        const uint64_t lo = k * kChunk;
        const uint32_t words = uint32_t(n - lo < kChunk ? n - lo : kChunk);
        const uint32_t bytes = 4u * words;
        const uint32_t blocks = (bytes + 127u) / 128u;
        // chunk starts are 4096-element aligned, so both the fp32 and the bf16 rows are
        // 16-byte aligned
        for (uint32_t j = 0; j < blocks; ++j) {
            uint64_t msg[16];
            const bool last = j + 1 == blocks;
            if ((!last || bytes == 128u * blocks) && !narrow) {
                const uint4 *p = static_cast<const uint4 *>(arr) + (lo / 4) + j * 8;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const uint4 u = __ldg(p + q);
                    msg[2 * q] = uint64_t(u.x) | (uint64_t(u.y) << 32);
                    msg[2 * q + 1] = uint64_t(u.z) | (uint64_t(u.w) << 32);
                }
            } else if (!last || bytes == 128u * blocks) {
                // 32 bf16 values = four 16-byte loads, widened to 32 words
                const uint4 *p = static_cast<const uint4 *>(arr) + (lo / 8) + j * 4;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 u = __ldg(p + q);
                    const uint32_t h[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        msg[4 * q + i] = uint64_t(h[i] << 16) | (uint64_t(h[i] & 0xFFFF0000u) << 32);
                }
            } else {
                // a short final block: the words that exist, zero padding after them
                const uint64_t w0 = lo + uint64_t(j) * 32u;
                const uint32_t have = words - j * 32u;
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    const uint32_t lo32 = uint32_t(2 * q) < have ? word_of(arr, narrow, w0 + 2 * q) : 0u;
                    const uint32_t hi32 =
                        uint32_t(2 * q + 1) < have ? word_of(arr, narrow, w0 + 2 * q + 1) : 0u;
                    msg[q] = uint64_t(lo32) | (uint64_t(hi32) << 32);
                }
            }
            const uint64_t t = last ? uint64_t(bytes) : uint64_t(128u) * (j + 1);
            b2_compress(h, msg, t, last);
        }
        leaves[L] = h[0];
    }
}

}  // namespace

cudaError_t leaves_b2_prepare()
{
    // On the hash stream the leaves run beside the next step's single pass: their blocks
    // must not leave an SM configured with less shared memory than its CTAs need.
    return cudaFuncSetAttribute(reinterpret_cast<const void *>(k_leaves_b2),
                                cudaFuncAttributePreferredSharedMemoryCarveout,
                                int(cudaSharedmemCarveoutMaxShared));
}

cudaError_t launch_leaves_b2(const void *w, int w_bf16, const float *m, const float *v, uint64_t n,
                             uint64_t c, uint64_t *leaves, uint32_t step, int sm_count,
                             cudaStream_t st)
{
    const uint64_t total = 1 + 3 * c;
    uint64_t blocks = (total + 255) / 256;
    const uint64_t cap = uint64_t(sm_count > 0 ? sm_count : 1) * 8;
    if (blocks > cap) blocks = cap;
    k_leaves_b2<<<unsigned(blocks), 256, 0, st>>>(w, w_bf16, m, v, n, c, leaves, step);
    return cudaGetLastError();
}

}  // namespace repstep
