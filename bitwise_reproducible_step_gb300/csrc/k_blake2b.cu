// k_blake2b.cu -- audit-mode leaf digests: BLAKE2b-64 (RFC 7693) of each leaf's bytes in
// the checkpoint image.  Leaf 0 is the 8-byte header [LE int32 step][LE uint32 n]; leaf
// 1 + a*c + k is chunk k (4096 elements, the last one short) of array a in (w, m, v), as
// little-endian fp32 bytes.  ("OPEN-1B: A Fully Auditable Training Run", App. B: every step
// is hashed with blake2b; this mode uses it for the leaves as well as the Merkle nodes.)
//
// BLAKE2b is a sequential chain over 128-byte blocks, so each leaf is one thread's chain of
// 128 compressions; the 1 + 3c leaves give the parallelism.  The work is ALU-bound (about
// 2,200 integer instructions per 128 bytes), far from the HBM bound of the PF61 leaves.
#include "common.cuh"
#include "kernels.h"

namespace repstep {

namespace {

__global__ void __launch_bounds__(256) k_leaves_b2(const float *w, const float *m, const float *v,
                                                   uint64_t n, uint64_t c, uint64_t *leaves,
                                                   uint32_t step)
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
        const float *arr = a == 0 ? w : (a == 1 ? m : v);
        const uint64_t lo = k * kChunk;
        const uint32_t words = uint32_t(n - lo < kChunk ? n - lo : kChunk);
        const uint32_t bytes = 4u * words;
        const uint32_t blocks = (bytes + 127u) / 128u;
        const uint4 *p = reinterpret_cast<const uint4 *>(arr + lo);   // 16-byte aligned
        for (uint32_t j = 0; j < blocks; ++j) {
            uint64_t msg[16];
            const bool last = j + 1 == blocks;
            if (!last || bytes == 128u * blocks) {
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const uint4 u = __ldg(p + j * 8 + q);
                    msg[2 * q] = uint64_t(u.x) | (uint64_t(u.y) << 32);
                    msg[2 * q + 1] = uint64_t(u.z) | (uint64_t(u.w) << 32);
                }
            } else {
                // a short final block: the words that exist, zero padding after them
                const uint32_t *pw = reinterpret_cast<const uint32_t *>(arr + lo) + j * 32u;
                const uint32_t have = words - j * 32u;
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    const uint32_t lo32 = uint32_t(2 * q) < have ? __ldg(pw + 2 * q) : 0u;
                    const uint32_t hi32 = uint32_t(2 * q + 1) < have ? __ldg(pw + 2 * q + 1) : 0u;
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

cudaError_t launch_leaves_b2(const float *w, const float *m, const float *v, uint64_t n,
                             uint64_t c, uint64_t *leaves, uint32_t step, int sm_count,
                             cudaStream_t st)
{
    const uint64_t total = 1 + 3 * c;
    uint64_t blocks = (total + 255) / 256;
    const uint64_t cap = uint64_t(sm_count > 0 ? sm_count : 1) * 8;
    if (blocks > cap) blocks = cap;
    k_leaves_b2<<<unsigned(blocks), 256, 0, st>>>(w, m, v, n, c, leaves, step);
    return cudaGetLastError();
}

}  // namespace repstep
