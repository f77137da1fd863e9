// k_small.cu -- the short kernels of the step: PF61 power table, global norm and clip
// scale, Merkle levels, image header, and the fix-ups for chunks cut by range boundaries.
#include "common.cuh"
#include "kernels.h"
#include "merkle.h"

namespace repstep {

namespace {

// K^(i+1) mod p for i < 4096, by square-and-multiply.
__global__ void k_init_powers(uint64_t *powers)
{
    const uint32_t i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= kChunk) return;
    uint32_t e = i + 1;
    uint64_t r = 1, b = kK61;
    while (e) {
        if (e & 1u) r = pf_mul(r, b);
        b = pf_mul(b, b);
        e >>= 1;
    }
    powers[i] = r;
}

struct ChunkList {
    uint64_t idx[kFixMax];
    int count;
};

// Sum of squares of whole chunks of g, for chunks a range boundary cut during reduce.
// 256 threads per chunk, the same fixed tree as the reduce kernel (common.cuh), in the
// arithmetic mode FZ.
template <int FZ>
__global__ void __launch_bounds__(256) k_chunk_fix(const float *g, uint64_t n, float *chunk_sq,
                                                   const ChunkList L)
{
    __shared__ float red[4 * 8];
    const uint64_t k = L.idx[blockIdx.x];
    const int tid = threadIdx.x;
    float part[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float q[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint64_t e = k * kChunk + uint64_t(j) * 1024 + 4u * tid + i;
            const float x = e < n ? g[e] : 0.0f;
            q[i] = e < n ? Ar<FZ>::mul(x, x) : 0.0f;
        }
        part[j] = sum4<FZ>(q[0], q[1], q[2], q[3]);
    }
    const float total = chunk_tree<256, 4, FZ>(part, red, tid, [] { __syncthreads(); });
    if (tid == 0) chunk_sq[k] = total;
}

// Leaf digests of whole chunks of w, m, v, for chunks a range boundary cut during AdamW.
// A bf16 w is digested as its exactly widened fp32 words.
__global__ void __launch_bounds__(256) k_leaf_fix(const void *w, int w_bf16, const float *m,
                                                  const float *v, uint64_t n, uint64_t c,
                                                  uint64_t *leaves, const uint64_t *powers,
                                                  const ChunkList L)
{
    __shared__ uint64_t pb[3][256];
    const uint64_t k = L.idx[blockIdx.x];
    const int tid = threadIdx.x;
    const float *arr[3] = {static_cast<const float *>(w), m, v};
    const unsigned short *w16 = static_cast<const unsigned short *>(w);
    uint32_t acc[3][4];
#pragma unroll
    for (int s = 0; s < 3; ++s)
#pragma unroll
        for (int t = 0; t < 4; ++t) acc[s][t] = 0u;
    for (uint32_t p = tid; p < kChunk; p += 256) {
        const uint64_t e = k * kChunk + p;
        if (e >= n) break;
        const uint64_t pk = powers[p];
        const uint32_t p0 = uint32_t(pk), p1 = uint32_t(pk >> 32);
        const uint32_t w0 = w_bf16 ? uint32_t(w16[e]) << 16 : __float_as_uint(arr[0][e]);
        pf_mac(acc[0], w0, p0, p1);
#pragma unroll
        for (int s = 1; s < 3; ++s) pf_mac(acc[s], __float_as_uint(arr[s][e]), p0, p1);
    }
#pragma unroll
    for (int s = 0; s < 3; ++s) pb[s][tid] = pf_fold128(acc[s]);
    __syncthreads();
    const int warp = tid >> 5, lane = tid & 31;
    if (warp < 3) {
        uint64_t sum = 0;
        for (int t = lane; t < 256; t += 32) sum = pf_add(sum, pb[warp][t]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            sum = pf_add(sum, __shfl_xor_sync(0xffffffffu, sum, off));
        if (lane == 0) {
            const uint64_t c0 = k * kChunk;
            const uint64_t c1 = c0 + kChunk < n ? c0 + kChunk : n;
            leaves[1 + uint64_t(warp) * c + k] = pf_add(c1 - c0, sum);
        }
    }
}

// Global norm.  Block b reduces in[4096 b .. 4096 b + 4096) (zero past `count`) in the
// fixed tree; with final_pass the single block's total S gives norm = sqrt(S) and the
// clip scale, otherwise it writes the block partial.  Zero padding leaves the canonical
// tree of non-negative sums unchanged, so two passes equal one tree over all chunks.
template <int FZ>
__global__ void __launch_bounds__(256) k_norm(const float *in, uint64_t count, float *out,
                                              Scalars *sc, int final_pass, float clip,
                                              float *norm_out, float *scale_out,
                                              volatile uint32_t *clip_flag)
{
    __shared__ float red[4 * 8];
    const int tid = threadIdx.x;
    const uint64_t base = uint64_t(blockIdx.x) * kChunk;
    float part[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float q[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint64_t e = base + uint64_t(j) * 1024 + 4u * tid + i;
            q[i] = e < count ? in[e] : 0.0f;        // results of .ftz operations already
        }
        part[j] = sum4<FZ>(q[0], q[1], q[2], q[3]);
    }
    const float S = chunk_tree<256, 4, FZ>(part, red, tid, [] { __syncthreads(); });
    if (tid != 0) return;
    if (!final_pass) {
        out[blockIdx.x] = S;
        return;
    }
    const float norm = Ar<FZ>::sqrt(S);
    // OPEN-1B §3.2 clips gradients by their global l2 norm; the formula is not given.
    // Reading: scale = clip / norm when the norm exceeds the threshold, else 1 (a NaN norm
    // compares false).
    const float scale = norm > clip ? Ar<FZ>::div(clip, norm) : 1.0f;
    const bool finite = isfinite(norm);
    sc->norm = norm;
    sc->scale = scale;
    if (clip_flag) *clip_flag = __float_as_uint(scale) != 0x3F800000u ? 1u : 0u;
    sc->flags = (sc->flags & ~kFlagNonfinite) | (finite ? 0u : kFlagNonfinite);
    if (norm_out) *norm_out = norm;
    if (scale_out) *scale_out = scale;
}

// PF61 of the header words {step, n}: (2 + step K + n K^2) mod p.
__device__ __forceinline__ uint64_t header_leaf(uint32_t step, uint32_t n32, const uint64_t *powers)
{
    return pf_add(pf_add(2, pf_mul(step, powers[0])), pf_mul(n32, powers[1]));
}

// One Merkle block: the canonical tree over up to kMerkleBlock consecutive digests, level by
// level (pair neighbours, carry an odd last node up unchanged), which is the same tree as
// the recursive split T = T(first 2^k) + T(rest).  Aligned power-of-two blocks are complete
// subtrees of the whole tree (a short last block included), so further passes over the
// block roots finish it.  1024-digest blocks give the leaf pass of a 1.2e9-parameter state
// 859 blocks, about 5.7 per SM, where 4096-digest blocks gave 215 and left the SMs that
// held two of them as the tail.  Block 0 of the leaf pass computes the header leaf
// PF61({step, n}) itself.
__global__ void __launch_bounds__(256) k_merkle(const uint64_t *in, uint64_t count, uint64_t *out,
                                                int header_mode, uint64_t *leaves_rw,
                                                uint32_t step, uint32_t n32,
                                                const uint64_t *powers, Scalars *sc,
                                                uint64_t *root_out, int final_pass)
{
    __shared__ uint64_t mk[2][kMerkleBlock];
    uint64_t *buf0 = mk[0], *buf1 = mk[1];
    const int tid = threadIdx.x;
    const uint64_t base = uint64_t(blockIdx.x) * kMerkleBlock;
    uint32_t cnt = uint32_t(count - base < kMerkleBlock ? count - base : kMerkleBlock);
    for (uint32_t i = tid; i < cnt; i += blockDim.x) buf0[i] = in[base + i];
    __syncthreads();
    if (header_mode && blockIdx.x == 0 && tid == 0) {
        const uint64_t h = header_leaf(step, n32, powers);
        buf0[0] = h;
        leaves_rw[0] = h;
    }
    __syncthreads();
    while (cnt > 1) {
        const uint32_t half = cnt >> 1;
        for (uint32_t i = tid; i < half; i += blockDim.x) buf1[i] = b2_node(buf0[2 * i], buf0[2 * i + 1]);
        if ((cnt & 1u) && tid == 0) buf1[half] = buf0[cnt - 1];
        __syncthreads();
        uint64_t *t = buf0;
        buf0 = buf1;
        buf1 = t;
        cnt = half + (cnt & 1u);
    }
    if (tid == 0) {
        if (final_pass) {
            sc->root = buf0[0];
            if (root_out) *root_out = buf0[0];
        } else {
            out[blockIdx.x] = buf0[0];
        }
    }
}

// The PF61 header leaf alone (the standalone leaves call; the Merkle pass computes it
// otherwise).
__global__ void k_header_leaf(uint64_t *leaves, uint32_t step, uint32_t n32,
                              const uint64_t *powers)
{
    leaves[0] = header_leaf(step, n32, powers);
}

__global__ void k_write_header(void *dst, int32_t step, uint32_t n32)
{
    uint32_t *p = static_cast<uint32_t *>(dst);
    p[0] = uint32_t(step);
    p[1] = n32;
}

}  // namespace

cudaError_t launch_init_powers(uint64_t *powers, cudaStream_t st)
{
    k_init_powers<<<kChunk / 256, 256, 0, st>>>(powers);
    return cudaGetLastError();
}

cudaError_t launch_chunk_fix(const float *g, uint64_t n, float *chunk_sq, const uint64_t *chunks,
                             int count, int fz, cudaStream_t st)
{
    ChunkList L{};
    for (int i = 0; i < count; ++i) L.idx[i] = chunks[i];
    L.count = count;
    if (fz) k_chunk_fix<1><<<count, 256, 0, st>>>(g, n, chunk_sq, L);
    else k_chunk_fix<0><<<count, 256, 0, st>>>(g, n, chunk_sq, L);
    return cudaGetLastError();
}

cudaError_t launch_leaf_fix(const void *w, int w_bf16, const float *m, const float *v, uint64_t n,
                            uint64_t c, uint64_t *leaves, const uint64_t *powers,
                            const uint64_t *chunks, int count, cudaStream_t st)
{
    ChunkList L{};
    for (int i = 0; i < count; ++i) L.idx[i] = chunks[i];
    L.count = count;
    k_leaf_fix<<<count, 256, 0, st>>>(w, w_bf16, m, v, n, c, leaves, powers, L);
    return cudaGetLastError();
}

cudaError_t launch_norm(const float *in, uint64_t count, float *out, Scalars *sc, int final_pass,
                        float clip, float *norm_out, float *scale_out, int blocks, int fz,
                        cudaStream_t st, uint32_t *clip_flag)
{
    if (fz)
        k_norm<1><<<blocks, 256, 0, st>>>(in, count, out, sc, final_pass, clip, norm_out, scale_out,
                                         clip_flag);
    else
        k_norm<0><<<blocks, 256, 0, st>>>(in, count, out, sc, final_pass, clip, norm_out, scale_out,
                                         clip_flag);
    return cudaGetLastError();
}

cudaError_t merkle_prepare()
{
    // The root passes may run on a second stream beside the next reduce, whose persistent
    // CTAs need most of an SM's shared memory.  An SM whose L1/shared split was set for a
    // small kernel cannot take such a CTA until it drains, so these kernels ask for the
    // largest shared-memory carveout too: then a reduce CTA fits beside their blocks
    // (registers: 544 x 96 + 256 x 48 <= 65536).
    cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void *>(k_merkle),
                                         cudaFuncAttributePreferredSharedMemoryCarveout,
                                         int(cudaSharedmemCarveoutMaxShared));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(reinterpret_cast<const void *>(k_leaf_fix),
                                 cudaFuncAttributePreferredSharedMemoryCarveout,
                                 int(cudaSharedmemCarveoutMaxShared));
    return e;
}

cudaError_t launch_merkle(const uint64_t *in, uint64_t count, uint64_t *out, int header_mode,
                          uint64_t *leaves_rw, uint32_t step, uint32_t n32, const uint64_t *powers,
                          Scalars *sc, uint64_t *root_out, int blocks, cudaStream_t st)
{
    k_merkle<<<blocks, 256, 0, st>>>(in, count, out, header_mode, leaves_rw, step, n32, powers,
                                     sc, root_out, blocks == 1 ? 1 : 0);
    return cudaGetLastError();
}

cudaError_t launch_header_leaf(uint64_t *leaves, int32_t step, uint32_t n32, const uint64_t *powers,
                               cudaStream_t st)
{
    k_header_leaf<<<1, 1, 0, st>>>(leaves, uint32_t(step), n32, powers);
    return cudaGetLastError();
}

cudaError_t launch_write_header(void *dst, int32_t step, uint32_t n32, cudaStream_t st)
{
    k_write_header<<<1, 1, 0, st>>>(dst, step, n32);
    return cudaGetLastError();
}

namespace {

// bf16 -> fp32 is exact: the bf16 bits are the top half of the fp32 word.
__global__ void __launch_bounds__(256) k_widen_bf16(float *dst, const unsigned short *src,
                                                    uint64_t n)
{
    const uint64_t stride = uint64_t(gridDim.x) * blockDim.x;
    for (uint64_t e = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x; e < n; e += stride)
        dst[e] = __uint_as_float(uint32_t(src[e]) << 16);
}

// fp32 -> bf16 by dropping the low half, valid only when that half is zero (the value is a
// bf16 exactly).  With dst null it only checks; any other word sets *bad.
__global__ void __launch_bounds__(256) k_narrow_bf16(unsigned short *dst, const float *src,
                                                     uint64_t n, uint32_t *bad)
{
    const uint64_t stride = uint64_t(gridDim.x) * blockDim.x;
    uint32_t mine = 0;
    for (uint64_t e = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x; e < n; e += stride) {
        const uint32_t u = __float_as_uint(src[e]);
        mine |= u & 0xFFFFu;
        if (dst) dst[e] = (unsigned short)(u >> 16);
    }
    if (mine && bad) atomicOr(bad, 1u);
}

unsigned elementwise_blocks(uint64_t n)
{
    uint64_t b = (n + 255) / 256;
    if (b > 152u * 16u) b = 152u * 16u;
    return unsigned(b > 0 ? b : 1);
}

}  // namespace

cudaError_t launch_widen_bf16(float *dst, const unsigned short *src, uint64_t n, cudaStream_t st)
{
    if (n == 0) return cudaSuccess;
    k_widen_bf16<<<elementwise_blocks(n), 256, 0, st>>>(dst, src, n);
    return cudaGetLastError();
}

cudaError_t launch_narrow_bf16(unsigned short *dst, const float *src, uint64_t n, uint32_t *bad,
                               cudaStream_t st)
{
    if (n == 0) return cudaSuccess;
    k_narrow_bf16<<<elementwise_blocks(n), 256, 0, st>>>(dst, src, n, bad);
    return cudaGetLastError();
}

}  // namespace repstep
