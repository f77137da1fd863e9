// k_adamw.cu -- clipped AdamW fused with the state-hash leaf digests (one HBM pass), and a
// leaves-only mode for the standalone hash.
//
// MODE 0 (AdamW): for every element of the active range, in this fixed order
//     gc = g*scale;  m' = b1*m + (1-b1)*gc;  v' = b2*v + (1-b2)*(gc*gc)
//     u = (m'/bc1) / (sqrt(v'/bc2) + eps);   w' = w*(1 - lr*wd) - lr*u
// ("OPEN-1B: A Fully Auditable Training Run", §3.2: AdamW with decoupled weight decay and
// global-norm clipping; §3.2 paragraph on optimizer-state precision: moments and update in
// FP32), writing w', m', v' in place; then the PF61 digest of every
// 4096-element chunk of the NEW w', m', v' that lies wholly inside the range.
// MODE 1 (leaves): the PF61 digests of the chunks of the given w, m, v, nothing written.
//
// PF61 of a chunk of W 32-bit words x_i is (W + sum x_i K^(i+1)) mod (2^61 - 1): the
// per-word terms are exact integers, so each thread accumulates its words' products in a
// 128-bit register sum and the chunk total is an exact integer sum in any order -- the
// digest cannot depend on the launch shape.  (App. B of the same paper anchors every
// step with a hash of parameters and optimizer state; this is its on-device form.)
//
// GB300 design: as the reduce kernel -- a persistent grid, one producer lane streaming
// 4 (or 3) arrays tile by tile into a shared-memory ring with 1-D bulk TMA copies on
// mbarriers, NT compute threads taking one 16-byte group per array per tile, 16-byte
// stores of the results.  Every fp32 operation is an explicitly rounded intrinsic.
#include "common.cuh"
#include "kernels.h"

namespace repstep {

namespace {

constexpr uint32_t kRingBytes = 128 * 1024;
constexpr uint32_t kMaxStages = 12;

template <int NT>
__host__ __device__ constexpr uint32_t ring_offset()
{
    // barriers (2 x kMaxStages x 8) | abort flags (8) | leaf partials 2 x 3 x NT u64
    return ((16 * kMaxStages + 16 + 2 * 3 * NT * 8) + 1023) / 1024 * 1024;
}

__device__ __forceinline__ void adamw_elem(float g, float &w, float &m, float &v, float scale,
                                           const AdamwArgs &A)
{
    const float gc = __fmul_rn(g, scale);
    const float m_new = __fadd_rn(__fmul_rn(A.beta1, m), __fmul_rn(A.om1, gc));
    const float gsq = __fmul_rn(gc, gc);
    const float v_new = __fadd_rn(__fmul_rn(A.beta2, v), __fmul_rn(A.om2, gsq));
    const float mhat = __fdiv_rn(m_new, A.bc1);
    const float vhat = __fdiv_rn(v_new, A.bc2);
    const float denom = __fadd_rn(__fsqrt_rn(vhat), A.eps);
    const float u = __fdiv_rn(mhat, denom);
    w = __fsub_rn(__fmul_rn(w, A.delta), __fmul_rn(A.lr, u));
    m = m_new;
    v = v_new;
}

template <int NT, int MODE>
__global__ void __launch_bounds__(NT + 32, 1) k_adamw(const __grid_constant__ AdamwArgs A)
{
    constexpr int NS = MODE == 0 ? 4 : 3;        // streamed arrays
    constexpr uint32_t TE = 4u * NT;
    constexpr int TPC = int(kChunk / TE);
    constexpr int W = NT / 32;
    static_assert(W >= 3, "three warps finish the three leaves of a chunk");

    extern __shared__ __align__(1024) unsigned char smem[];
    const uint32_t S = A.stages;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + kMaxStages;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + 16 * kMaxStages);
    volatile int *never_flag = abort_flag + 1;
    uint64_t *pfbuf = reinterpret_cast<uint64_t *>(smem + 16 * kMaxStages + 16);
    unsigned char *ring = smem + ring_offset<NT>();

    const int tid = threadIdx.x;
    if (tid == 0) {
        for (uint32_t s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), W);
        }
        *abort_flag = 0;
        *never_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    const uint32_t flag_bit = MODE == 0 ? kFlagTimeoutAdamw : kFlagTimeoutLeaves;

    if (tid >= NT) {
        // ------------------------------ producer warp ------------------------------
        if (tid != NT) return;
        const void *src[4];
        if (MODE == 0) {
            src[0] = A.g; src[1] = A.w; src[2] = A.m; src[3] = A.v;
        } else {
            src[0] = A.w; src[1] = A.m; src[2] = A.v; src[3] = nullptr;
        }
        const uint64_t pol = l2_evict_first();
        uint32_t it = 0;
        bool ok = true;
        for (uint64_t k = A.chunk_lo + blockIdx.x; ok && k < A.chunk_hi; k += gridDim.x) {
            for (int j = 0; j < TPC; ++j) {
                const TileRange tr =
                    tile_range(k * kChunk + uint64_t(j) * TE, TE, A.begin, A.end, 4);
                const uint32_t bytes = uint32_t(tr.b16 - tr.a16) * 4u;
                const uint32_t soff = uint32_t(tr.a16 - tr.base) * 4u;
                const uint32_t slot = it % S, round = it / S;
                if (!mbar_wait_bounded(smem_u32(&empty[slot]), (round & 1u) ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = smem_u32(&full[slot]);
                mbar_arrive_expect_tx(fb, bytes * NS);
                if (bytes) {
                    const uint32_t dst = smem_u32(ring + slot * A.stage_stride) + soff;
#pragma unroll
                    for (int s = 0; s < NS; ++s)
                        bulk_g2s(dst + s * TE * 4u,
                                 static_cast<const float *>(src[s]) + tr.a16, bytes, fb, pol);
                }
                ++it;
            }
        }
        if (!ok) {
            atomicOr(&A.sc->flags, flag_bit);
            *abort_flag = 1;
        }
        const uint32_t last = it < S ? it : S;
        for (uint32_t d = 0; d < last; ++d) {
            const uint32_t idx = it - 1 - d;
            mbar_wait_bounded(smem_u32(&full[idx % S]), (idx / S) & 1u, never_flag);
        }
        return;
    }

    // ------------------------------ compute threads -------------------------------
    const int lane = tid & 31, warp = tid >> 5;
    const float scale = MODE == 0 ? A.sc->scale : 1.0f;
    uint32_t it = 0;
    int cb = 0;
    bool aborted = false;
    for (uint64_t k = A.chunk_lo + blockIdx.x; k < A.chunk_hi; k += gridDim.x) {
        uint32_t acc[3][4];
#pragma unroll
        for (int s = 0; s < 3; ++s)
#pragma unroll
            for (int t = 0; t < 4; ++t) acc[s][t] = 0u;
#pragma unroll
        for (int j = 0; j < TPC; ++j) {
            const TileRange tr = tile_range(k * kChunk + uint64_t(j) * TE, TE, A.begin, A.end, 4);
            const uint32_t off = 4u * tid;
            const uint64_t e0 = tr.base + off;
            const bool in_bulk = e0 >= tr.a16 && e0 + 4 <= tr.b16;
            const uint32_t slot = it % S, round = it / S;
            if (!aborted && !mbar_wait_bounded(smem_u32(&full[slot]), round & 1u, abort_flag)) {
                aborted = true;
                if (lane == 0) {
                    atomicOr(&A.sc->flags, flag_bit);
                    *abort_flag = 1;
                }
            }
            const unsigned char *sb = ring + slot * A.stage_stride;
            float4 x[NS];
            uint32_t inmask = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i)
                inmask |= (e0 + i >= tr.a && e0 + i < tr.b) ? (1u << i) : 0u;
            if (in_bulk) {
#pragma unroll
                for (int s = 0; s < NS; ++s)
                    x[s] = *reinterpret_cast<const float4 *>(sb + s * TE * 4u + off * 4u);
            } else {
                const float *srcs[4];
                if (MODE == 0) {
                    srcs[0] = A.g; srcs[1] = A.w; srcs[2] = A.m; srcs[3] = A.v;
                } else {
                    srcs[0] = A.w; srcs[1] = A.m; srcs[2] = A.v; srcs[3] = nullptr;
                }
#pragma unroll
                for (int s = 0; s < NS; ++s) {
                    float r[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        r[i] = (inmask >> i) & 1u ? __ldg(srcs[s] + e0 + i) : 0.0f;
                    x[s] = make_float4(r[0], r[1], r[2], r[3]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty[slot]));
            ++it;

            float4 ow, om, ov;   // the words hashed: new state (MODE 0) or given state
            if (MODE == 0) {
                ow = x[1]; om = x[2]; ov = x[3];
                adamw_elem(x[0].x, ow.x, om.x, ov.x, scale, A);
                adamw_elem(x[0].y, ow.y, om.y, ov.y, scale, A);
                adamw_elem(x[0].z, ow.z, om.z, ov.z, scale, A);
                adamw_elem(x[0].w, ow.w, om.w, ov.w, scale, A);
                if (inmask == 0xFu) {
                    *reinterpret_cast<float4 *>(A.w + e0) = ow;
                    *reinterpret_cast<float4 *>(A.m + e0) = om;
                    *reinterpret_cast<float4 *>(A.v + e0) = ov;
                } else {
                    const float aw[4] = {ow.x, ow.y, ow.z, ow.w};
                    const float am[4] = {om.x, om.y, om.z, om.w};
                    const float av[4] = {ov.x, ov.y, ov.z, ov.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        if ((inmask >> i) & 1u) {
                            A.w[e0 + i] = aw[i];
                            A.m[e0 + i] = am[i];
                            A.v[e0 + i] = av[i];
                        }
                    }
                }
            } else {
                ow = x[0]; om = x[1]; ov = x[2];
            }

            // PF61 terms x * K^(p+1) for word positions p = j*TE + off + i of the chunk
            const ulonglong2 *pw =
                reinterpret_cast<const ulonglong2 *>(A.powers + uint32_t(j) * TE + off);
            const ulonglong2 p01 = __ldg(pw), p23 = __ldg(pw + 1);
            const uint64_t pk[4] = {p01.x, p01.y, p23.x, p23.y};
            const uint32_t wb[4] = {__float_as_uint(ow.x), __float_as_uint(ow.y),
                                    __float_as_uint(ow.z), __float_as_uint(ow.w)};
            const uint32_t mb[4] = {__float_as_uint(om.x), __float_as_uint(om.y),
                                    __float_as_uint(om.z), __float_as_uint(om.w)};
            const uint32_t vb[4] = {__float_as_uint(ov.x), __float_as_uint(ov.y),
                                    __float_as_uint(ov.z), __float_as_uint(ov.w)};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t p0 = uint32_t(pk[i]), p1 = uint32_t(pk[i] >> 32);
                const uint32_t on = (inmask >> i) & 1u ? 0xFFFFFFFFu : 0u;
                pf_mac(acc[0], wb[i] & on, p0, p1);
                pf_mac(acc[1], mb[i] & on, p0, p1);
                pf_mac(acc[2], vb[i] & on, p0, p1);
            }
        }

        // chunk leaves: exact integer sum of every thread's partial, then + W mod p
        uint64_t *pb = pfbuf + cb * 3 * NT;
#pragma unroll
        for (int s = 0; s < 3; ++s) pb[s * NT + tid] = pf_fold128(acc[s]);
        named_barrier(1, NT);
        if (warp < 3) {
            uint64_t sum = 0;
            for (int t = lane; t < NT; t += 32) sum = pf_add(sum, pb[warp * NT + t]);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                sum = pf_add(sum, __shfl_xor_sync(0xffffffffu, sum, off));
            if (lane == 0) {
                const uint64_t c0 = k * kChunk;
                const uint64_t c1 = c0 + kChunk < A.n ? c0 + kChunk : A.n;
                if (c0 >= A.begin && c1 <= A.end)
                    A.leaves[1 + uint64_t(warp) * A.c + k] = pf_add(c1 - c0, sum);
            }
        }
        cb ^= 1;
    }
}

using KernelFn = void (*)(AdamwArgs);

KernelFn pick(int nt, int mode)
{
    switch (nt) {
    case 128: return mode ? k_adamw<128, 1> : k_adamw<128, 0>;
    case 256: return mode ? k_adamw<256, 1> : k_adamw<256, 0>;
    case 512: return mode ? k_adamw<512, 1> : k_adamw<512, 0>;
    default: return nullptr;
    }
}

uint32_t ring_off(int nt)
{
    return nt == 128 ? ring_offset<128>() : (nt == 256 ? ring_offset<256>() : ring_offset<512>());
}

}  // namespace

size_t adamw_smem_bytes(int nt, int mode, AdamwArgs &args)
{
    const uint32_t ns = mode == 0 ? 4u : 3u;
    const uint32_t stride = ns * 4u * uint32_t(nt) * 4u;
    uint32_t stages = kRingBytes / stride;
    if (stages > kMaxStages) stages = kMaxStages;
    if (stages < 2) stages = 2;
    args.stages = stages;
    args.stage_stride = stride;
    return size_t(ring_off(nt)) + size_t(stages) * stride;
}

cudaError_t adamw_prepare(int nt, int mode, size_t smem)
{
    KernelFn f = pick(nt, mode);
    if (!f) return cudaErrorInvalidValue;
    return cudaFuncSetAttribute(reinterpret_cast<const void *>(f),
                                cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
}

cudaError_t adamw_occupancy(int nt, int mode, size_t smem, int *blocks_per_sm)
{
    KernelFn f = pick(nt, mode);
    if (!f) return cudaErrorInvalidValue;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        blocks_per_sm, reinterpret_cast<const void *>(f), nt + 32, smem);
}

cudaError_t launch_adamw(int nt, int mode, const AdamwArgs &args, int grid, size_t smem,
                         cudaStream_t st)
{
    KernelFn f = pick(nt, mode);
    if (!f) return cudaErrorInvalidValue;
    void *params[] = {const_cast<AdamwArgs *>(&args)};
    return cudaLaunchKernel(reinterpret_cast<const void *>(f), dim3(grid), dim3(nt + 32),
                            params, smem, st);
}

}  // namespace repstep
