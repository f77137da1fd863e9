// k_fused.cuh -- the speculative single-pass step (kernel template; k_fused.cu holds the
// IEEE instantiations for R = 4 and 8 and the host helpers, k_fused_ftz.cu the
// flush-to-zero ones, k_fused_wide.cu and k_fused_wide_ftz.cu those for R = 16).
//
// One HBM pass computes, for every element i and every 4096-element chunk k:
//     g_i = T_{r<R}(G_r[i]) * fp32(1/R)                      (the replica reduce)
//     s_k = T(g_i * g_i over chunk k)                          (the chunk sums of squares)
//     m', v', w' = AdamW(w, m, v, gc = g * 1)                  (clip scale taken as 1)
//     the PF61 digests of chunk k of the new w', m', v'
// (w' rounded once to bf16 with bf16 parameters, per-element decay with a decay mask,
// .rn.ftz operations in the flush-to-zero mode, as the two-pass kernels do)
// reading the R gradients and the state (w, m, v) once and writing the new state to a
// second buffer (wo, mo, vo); g itself never goes to HBM.  ("OPEN-1B: A Fully Auditable
// Training Run", App. A.1 and A.3 for the reduce, §3.2 for the clipped AdamW, App. B for
// the state hash.)  After it, the norm passes compute the global norm and the true clip
// scale from the chunk sums.  The scale is exactly 1 whenever norm <= clip (and for a
// non-finite norm), and then every bit written here is the step's: gc = g * 1 is the
// same operation with the same operands as the two-pass step's gc = g * scale.  When the
// scale is not 1, the reduce and AdamW kernels run again (gate kGateIfClipped) from the
// untouched (w, m, v) and overwrite (wo, mo, vo) and the leaves; otherwise they return at
// once.  The host launches the pass only when the last clip outcome it can see did not
// clip; after one that did, the step takes the two passes directly.
//
// The arithmetic is the two-pass kernels' own, element for element: the same kind of
// element-to-thread mapping as k_reduce (a thread holds 4 consecutive elements of each
// 4*NT-element tile), the canonical replica tree (group_tree over a group of RG = R <= 8
// replicas, or over two groups of 8 for R = 16), the same chunk tree (chunk_tree, defined
// over element indices), the AdamW of adamw_math.cuh and the same PF61 limb sums, so every
// bit equals theirs.
//
// GB300 design: a persistent grid of two CTAs per SM, each with NT = 256 compute threads.
// Each CTA's producer lane streams, for each 1024-element tile, a stage with the R gradient
// tiles (32 KB for R = 8 fp32) and a stage with the w, m, v tiles (12 KB) into a 96 KB
// shared-memory ring (1-D bulk TMA copies, L2 evict-first, mbarrier completion); chunks are
// handed out at run time from a counter.  Two CTAs, each with its own producer and ring,
// kept the SM's memory pipe fuller than one CTA of 512 threads with a 192 KB ring (measured
// at 1.2e9 parameters: 10.22 -> 10.02 ms per pass).  The compute threads do the arithmetic
// and store the new state with vector stores; one leaf warp finishes the chunk digests
// from the compute warps' per-warp piece sums.  Every wait is bounded; a timeout sets a
// flag.
#pragma once
#include <cuda_bf16.h>

#include "adamw_math.cuh"
#include "common.cuh"
#include "kernels.h"

namespace repstep {

namespace {

constexpr uint32_t kFusedRing = 96 * 1024;     // per CTA; two CTAs per SM
constexpr uint32_t kFusedMaxStages = 12;
constexpr int kFusedLeafBufs = 4;
constexpr int kFusedPieces = 27;     // 3 arrays x 3 limbs x 3 pieces of 27 bits
constexpr int kFusedNT = 256;

// Shared-memory header: ring barriers | leaf barriers | chunk-tree scratch | abort flags |
// per-warp leaf pieces | the chunk of each ring slot and of each leaf buffer; then the ring.
template <int NT, int TPC>
__host__ __device__ constexpr uint32_t fused_ring_offset()
{
    return ((16 * kFusedMaxStages + 16 * kFusedLeafBufs + 2 * TPC * (NT / 32) * 4 + 16 +
             kFusedLeafBufs * (NT / 32) * kFusedPieces * 4 + 8 * kFusedMaxStages +
             8 * kFusedLeafBufs) + 1023) / 1024 * 1024;
}

template <int FZ>
__device__ __forceinline__ float4 fadd4(float4 a, float4 b)
{
    return make_float4(Ar<FZ>::add(a.x, b.x), Ar<FZ>::add(a.y, b.y), Ar<FZ>::add(a.z, b.z),
                       Ar<FZ>::add(a.w, b.w));
}

// The canonical tree of one full group of RG replicas: pairs, then pairs of pairs, the
// lower replicas on the left.
template <int RG, int FZ>
__device__ __forceinline__ float4 group_tree(float4 (&x)[RG])
{
#pragma unroll
    for (int s = 1; s < RG; s <<= 1) {
#pragma unroll
        for (int i = 0; i < RG; i += 2 * s) x[i] = fadd4<FZ>(x[i], x[i + s]);
    }
    return x[0];
}

template <int DT>
__device__ __forceinline__ float grad_elem(const void *p, uint64_t e)
{
    if (DT == 0) return __ldg(static_cast<const float *>(p) + e);
    return __uint_as_float(uint32_t(__ldg(static_cast<const unsigned short *>(p) + e)) << 16);
}

// A 4-element group: from the staged tile when it lies in the bulk-copied interior, else
// element by element from global memory, zero outside [a, b).  ES: bytes per element of
// the staged stream (4, or 2 for bf16 gradients, widened exactly).
template <int ES>
__device__ __forceinline__ float4 group_of(const unsigned char *tile, uint32_t off, bool in_bulk,
                                           const void *src, uint64_t e0, uint64_t a, uint64_t b)
{
    if (in_bulk) {
        if (ES == 4) return *reinterpret_cast<const float4 *>(tile + off * 4u);
        const uint2 u = *reinterpret_cast<const uint2 *>(tile + off * 2u);
        return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                           __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
    }
    float r[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint64_t e = e0 + i;
        r[i] = (e >= a && e < b) ? grad_elem<ES == 4 ? 0 : 1>(src, e) : 0.0f;
    }
    return make_float4(r[0], r[1], r[2], r[3]);
}

// DT: gradients fp32 (0) or bf16 (1).  RG: R, one full replica group of 4 or 8.  LEAVES:
// the PF61 leaves fused (1) or none (the audit mode).  PT: parameters fp32 (0) or bf16 (1).
// FZ: IEEE (0) or flush-to-zero (1) arithmetic.  MK: a per-element decay mask (1).
template <int NT, int DT, int RG, int LEAVES, int PT, int FZ, int MK>
__global__ void __launch_bounds__(NT + 64, 2) k_fused(const __grid_constant__ FusedArgs F)
{
    constexpr int W = NT / 32;
    constexpr uint32_t TE = 4u * NT;
    constexpr int TPC = int(kChunk / TE);
    constexpr uint32_t ESZ = DT == 0 ? 4u : 2u;
    constexpr uint32_t WSZ = PT == 0 ? 4u : 2u;  // bytes per parameter
    // elements per 16 bytes of the narrowest stream: bulk copies start and end there
    constexpr uint32_t VEC = 16u / (ESZ < WSZ ? ESZ : WSZ);
    // replicas per gradient stage: at most 64 KB of gradients per stage (all R replicas of
    // a tile for R <= 8)
    // replicas per gradient stage: at most 8 (the registers of one group) and 64 KB
    constexpr int GS_BYTES = 64 * 1024 / int(TE * ESZ);
    constexpr int GS = RG < 8 ? RG : (GS_BYTES < 8 ? GS_BYTES : 8);
    constexpr int NGS = RG / GS;                 // gradient stages per tile
    static_assert(GS * NGS == RG && (NGS & (NGS - 1)) == 0,
                  "gradient stages hold whole groups, a power of two of them");
    static_assert(TPC * TE == kChunk && TPC * 4 <= 32, "tiles divide the chunk; limb bound");
    const AdamwArgs &A = F.adam;

    extern __shared__ __align__(1024) unsigned char smem[];
    const uint32_t S = A.stages;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + kFusedMaxStages;
    uint64_t *leaf_full = empty + kFusedMaxStages;
    uint64_t *leaf_empty = leaf_full + kFusedLeafBufs;
    float *red = reinterpret_cast<float *>(leaf_empty + kFusedLeafBufs);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(red + 2 * TPC * W);
    volatile int *never_flag = abort_flag + 1;
    uint32_t *pieces_buf = reinterpret_cast<uint32_t *>(red + 2 * TPC * W) + 4;
    uint64_t *stage_chunk = reinterpret_cast<uint64_t *>(pieces_buf + kFusedLeafBufs * W * kFusedPieces);
    uint64_t *leaf_chunk = stage_chunk + kFusedMaxStages;
    unsigned char *ring = smem + fused_ring_offset<NT, TPC>();

    const int tid = threadIdx.x;
    if (tid == 0) {
        for (uint32_t s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), W);
        }
        for (int b = 0; b < kFusedLeafBufs; ++b) {
            mbar_init(smem_u32(&leaf_full[b]), W);
            mbar_init(smem_u32(&leaf_empty[b]), 1);
        }
        *abort_flag = 0;
        *never_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (tid >= NT + 32) {
        // -------------------------------- leaf warp --------------------------------
        if (!LEAVES) return;
        const int lane = tid - NT - 32;
        const int ls = lane / 9, ll = (lane / 3) % 3, lj = lane % 3;
        const int shift = (21 * ll + 27 * lj) % 61;
        for (uint32_t ci = 0;; ++ci) {
            const uint32_t b = ci % kFusedLeafBufs, round = ci / kFusedLeafBufs;
            const bool got = __all_sync(
                0xFFFFFFFFu, mbar_wait_bounded(smem_u32(&leaf_full[b]), round & 1u, abort_flag));
            if (!got) {
                if (lane == 0) {
                    atomicOr(&A.sc->flags, kFlagTimeoutAdamw);
                    *abort_flag = 1;
                }
                break;
            }
            const uint64_t k = leaf_chunk[b];
            if (k == kNoChunk) break;
            uint64_t sum = 0;
            if (lane < kFusedPieces) {
                const uint32_t *pb = pieces_buf + b * W * kFusedPieces + lane;
#pragma unroll
                for (int w = 0; w < W; ++w) sum += pb[w * kFusedPieces];
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&leaf_empty[b]));
            uint64_t term = lane < kFusedPieces ? pf_shl(pf_reduce64(sum), shift) : 0;
#pragma unroll
            for (int d = 1; d < 9; ++d) {
                const uint64_t o = __shfl_sync(0xFFFFFFFFu, term, (lane + d) & 31);
                if (lane % 9 == 0 && lane < kFusedPieces) term = pf_add(term, o);
            }
            if (lane % 9 == 0 && lane < kFusedPieces) {
                const uint64_t c0 = k * kChunk;
                const uint64_t c1 = c0 + kChunk < A.n ? c0 + kChunk : A.n;
                A.leaves[1 + uint64_t(ls) * A.c + k] = pf_add(c1 - c0, term);
            }
        }
        return;
    }

    if (tid >= NT) {
        // ------------------------------ producer warp ------------------------------
        if (tid != NT) return;
        const uint64_t pol = l2_evict_first();
        uint32_t it = 0;
        RingPos pos;
        bool ok = true;
        const void *state[3] = {A.w, A.m, A.v};
        uint64_t k_next = atomicAdd(&A.sc->next_chunk, 1u);
        while (ok && k_next < A.c) {
            const uint64_t k = k_next;
            k_next = atomicAdd(&A.sc->next_chunk, 1u);
            const bool whole = k * kChunk + kChunk <= A.n;
            for (int j = 0; ok && j < TPC; ++j) {
                const uint64_t tb = k * kChunk + uint64_t(j) * TE;
                const TileRange tr = whole ? whole_tile(tb, TE) : tile_range(tb, TE, 0, A.n, VEC);
                const uint32_t elems = uint32_t(tr.b16 - tr.a16);
                const uint32_t skip = uint32_t(tr.a16 - tr.base);
                // stages 0 .. NGS-1: the gradient tiles, GS replicas each; stage NGS: the
                // w, m, v tiles
                for (int part = 0; ok && part <= NGS; ++part) {
                    const uint32_t slot = pos.slot;
                    if (!mbar_wait_bounded(smem_u32(&empty[slot]), pos.phase ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    fence_reads_before_refill();
                    const uint32_t fb = smem_u32(&full[slot]);
                    const uint32_t dst = smem_u32(ring + slot * A.stage_stride);
                    if (j == 0 && part == 0) stage_chunk[slot] = k;   // published by the arrive
                    if (part < NGS) {
                        mbar_arrive_expect_tx(fb, elems * ESZ * uint32_t(GS));
                        if (elems)
                            for (int i = 0; i < GS; ++i)
                                bulk_g2s(dst + i * TE * ESZ + skip * ESZ,
                                         static_cast<const unsigned char *>(F.grads[part * GS + i]) +
                                             tr.a16 * ESZ,
                                         elems * ESZ, fb, pol);
                    } else {
                        // w (WSZ bytes per element), m and v, each in a 4*TE-byte part; with
                        // a decay mask, the tile's TE/8 mask bytes after them (whole tiles)
                        const bool stage_mask = MK != 0 && tr.a == tr.base && tr.b == tr.base + TE;
                        mbar_arrive_expect_tx(fb, elems * (WSZ + 8u) + (stage_mask ? TE / 8u : 0u));
                        if (stage_mask)
                            bulk_g2s(dst + 3u * TE * 4u,
                                     reinterpret_cast<const unsigned char *>(A.decay_mask) + tr.base / 8u,
                                     TE / 8u, fb, pol);
                        if (elems) {
                            if constexpr (PT != 0)
                                bulk_g2s(dst + skip * 2u,
                                         static_cast<const unsigned char *>(state[0]) + tr.a16 * 2u,
                                         elems * 2u, fb, pol);
                            for (int s = PT != 0 ? 1 : 0; s < 3; ++s)
                                bulk_g2s(dst + s * TE * 4u + skip * 4u,
                                         static_cast<const unsigned char *>(state[s]) + tr.a16 * 4u,
                                         elems * 4u, fb, pol);
                        }
                    }
                    ++it;
                    pos.advance(S);
                }
            }
        }
        // one more stage, without data, carries the end marker
        if (ok) {
            const uint32_t slot = pos.slot;
            if (mbar_wait_bounded(smem_u32(&empty[slot]), pos.phase ^ 1u, abort_flag)) {
                stage_chunk[slot] = kNoChunk;
                mbar_arrive(smem_u32(&full[slot]));
                ++it;
                pos.advance(S);
            } else {
                ok = false;
            }
        }
        if (!ok) {
            atomicOr(&A.sc->flags, kFlagTimeoutReduce);
            *abort_flag = 1;
        }
        // never leave while copies into the ring may be in flight (bounded waits)
        const uint32_t last = it < S ? it : S;
        for (uint32_t d = 0; d < last; ++d) {
            const uint32_t idx = it - 1 - d;
            mbar_wait_bounded(smem_u32(&full[idx % S]), (idx / S) & 1u, never_flag);
        }
        return;
    }

    // ------------------------------ compute threads -------------------------------
    const int lane = tid & 31, warp = tid >> 5;
    const float rho = F.rho;
    const uint32_t off = 4u * uint32_t(tid);

    RingPos pos;
    int cb = 0;
    bool aborted = false;
    auto fail = [&](uint32_t bit) {
        aborted = true;
        if (lane == 0) {
            atomicOr(&A.sc->flags, bit);
            *abort_flag = 1;
        }
    };
    for (uint32_t ci = 0;; ++ci) {
        // the stage that opens the next chunk carries its index, or the end marker; one
        // barrier vote makes the decision uniform over the compute threads
        const uint32_t slot0 = pos.slot;
        bool got = false;
        if (!aborted) {
            got = mbar_wait_bounded(smem_u32(&full[slot0]), pos.phase, abort_flag);
            if (!got) fail(kFlagTimeoutReduce);
        }
        const uint64_t k = got ? stage_chunk[slot0] : kNoChunk;
        if (named_barrier_or(2, NT, k == kNoChunk)) {
            // pass the end on to the leaf warp through the next leaf buffer
            if (LEAVES && got && lane == 0) {
                const uint32_t b = ci % kFusedLeafBufs, round = ci / kFusedLeafBufs;
                if (mbar_wait_bounded(smem_u32(&leaf_empty[b]), (round & 1u) ^ 1u, abort_flag)) {
                    leaf_chunk[b] = kNoChunk;
                    mbar_arrive(smem_u32(&leaf_full[b]));
                }
            }
            break;
        }
        const bool whole = k * kChunk + kChunk <= A.n;
        float part[TPC];
        Acc3 acc[3] = {{0, 0, 0}, {0, 0, 0}, {0, 0, 0}};
#pragma unroll
        for (int j = 0; j < TPC; ++j) {
            const uint64_t tb = k * kChunk + uint64_t(j) * TE;
            const TileRange tr = whole ? whole_tile(tb, TE) : tile_range(tb, TE, 0, A.n, VEC);
            const uint64_t e0 = tr.base + off;
            const bool in_bulk = e0 >= tr.a16 && e0 + 4 <= tr.b16;
            const bool all_in = e0 >= tr.a && e0 + 4 <= tr.b;

            // the replica reduce of this thread's 4 elements: each stage's group of GS
            // replicas is a perfect subtree of the canonical tree, and the NGS (a power of
            // two) group sums combine pairwise, the lower replicas on the left
            float4 grp[NGS];
            uint32_t slot;
            const unsigned char *sb;
#pragma unroll
            for (int q = 0; q < NGS; ++q) {
                slot = pos.slot;
                if ((j > 0 || q > 0) && !aborted &&
                    !mbar_wait_bounded(smem_u32(&full[slot]), pos.phase, abort_flag))
                    fail(kFlagTimeoutReduce);
                sb = ring + slot * A.stage_stride;
                float4 x[GS];
#pragma unroll
                for (int i = 0; i < GS; ++i)
                    x[i] = whole ? group_of<ESZ>(sb + i * TE * ESZ, off, true, nullptr, 0, 0, 0)
                                 : group_of<ESZ>(sb + i * TE * ESZ, off, in_bulk,
                                                 F.grads[q * GS + i], e0, tr.a, tr.b);
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&empty[slot]));
                pos.advance(S);
                grp[q] = group_tree<GS, FZ>(x);
            }
            const float4 s4 = group_tree<NGS, FZ>(grp);
            const float4 gv = make_float4(Ar<FZ>::mul(s4.x, rho), Ar<FZ>::mul(s4.y, rho),
                                          Ar<FZ>::mul(s4.z, rho), Ar<FZ>::mul(s4.w, rho));
            float q4[4];
            {
                const float gg[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint64_t e = e0 + i;
                    q4[i] = (all_in || (e >= tr.a && e < tr.b)) ? Ar<FZ>::mul(gg[i], gg[i]) : 0.0f;
                }
            }
            part[j] = sum4<FZ>(q4[0], q4[1], q4[2], q4[3]);

            // the state of the same elements
            slot = pos.slot;
            if (!aborted && !mbar_wait_bounded(smem_u32(&full[slot]), pos.phase, abort_flag))
                fail(kFlagTimeoutAdamw);
            sb = ring + slot * A.stage_stride;
            // the decay bits of the 4 elements (e0 is a multiple of 4: one mask word), from
            // the stage in a whole tile
            uint32_t dmask = 0xFu;
            if constexpr (MK != 0) {
                uint32_t word = 0;
                if (tr.a == tr.base && tr.b == tr.base + TE)
                    word = reinterpret_cast<const uint32_t *>(sb + 3u * TE * 4u)[off >> 5];
                else if (e0 < A.n)
                    word = __ldg(A.decay_mask + (e0 >> 5));
                dmask = (word >> (uint32_t(e0) & 31u)) & 0xFu;
            }
            const float4 w4 = whole ? group_of<WSZ>(sb, off, true, nullptr, 0, 0, 0)
                                    : group_of<WSZ>(sb, off, in_bulk, A.w, e0, tr.a, tr.b);
            const float4 m4 = whole ? group_of<4>(sb + TE * 4u, off, true, nullptr, 0, 0, 0)
                                    : group_of<4>(sb + TE * 4u, off, in_bulk, A.m, e0, tr.a, tr.b);
            const float4 v4 = whole ? group_of<4>(sb + 2u * TE * 4u, off, true, nullptr, 0, 0, 0)
                                    : group_of<4>(sb + 2u * TE * 4u, off, in_bulk, A.v, e0, tr.a, tr.b);
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty[slot]));
            pos.advance(S);

            // AdamW with the clip scale taken as 1
            float g[4] = {gv.x, gv.y, gv.z, gv.w};
            float w[4] = {w4.x, w4.y, w4.z, w4.w};
            float m[4] = {m4.x, m4.y, m4.z, m4.w};
            float v[4] = {v4.x, v4.y, v4.z, v4.w};
            adamw_n<MK != 0, FZ, 4>(g, w, m, v, 1.0f, dmask, A);
            uint32_t wpk[2] = {0u, 0u};
            if constexpr (PT != 0) {
                // one rounding of the fp32 result to bf16 (a pair per conversion); the hash
                // sees the rounded parameter, widened exactly
#pragma unroll
                for (int p2 = 0; p2 < 2; ++p2) {
                    const __nv_bfloat162 b2 = __floats2bfloat162_rn(w[2 * p2], w[2 * p2 + 1]);
                    wpk[p2] = *reinterpret_cast<const uint32_t *>(&b2);
                    w[2 * p2] = __uint_as_float(wpk[p2] << 16);
                    w[2 * p2 + 1] = __uint_as_float(wpk[p2] & 0xFFFF0000u);
                }
            }
            float *WO = static_cast<float *>(A.wo);
            unsigned short *WO16 = static_cast<unsigned short *>(A.wo);
            if (all_in) {
                if constexpr (PT != 0)
                    *reinterpret_cast<uint2 *>(WO16 + e0) = make_uint2(wpk[0], wpk[1]);
                else
                    *reinterpret_cast<float4 *>(WO + e0) = make_float4(w[0], w[1], w[2], w[3]);
                *reinterpret_cast<float4 *>(A.mo + e0) = make_float4(m[0], m[1], m[2], m[3]);
                *reinterpret_cast<float4 *>(A.vo + e0) = make_float4(v[0], v[1], v[2], v[3]);
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint64_t e = e0 + i;
                    const bool in = e >= tr.a && e < tr.b;
                    if (in) {
                        if constexpr (PT != 0)
                            WO16[e] = (unsigned short)(__float_as_uint(w[i]) >> 16);
                        else
                            WO[e] = w[i];
                        A.mo[e] = m[i];
                        A.vo[e] = v[i];
                    } else {
                        w[i] = m[i] = v[i] = 0.0f;    // words outside the range add nothing
                    }
                }
            }
            if (LEAVES) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const Limbs pw = limbs_of(__ldg(A.powers + uint32_t(j) * TE + off + i));
                    acc_word(acc[0], __float_as_uint(w[i]), pw);
                    acc_word(acc[1], __float_as_uint(m[i]), pw);
                    acc_word(acc[2], __float_as_uint(v[i]), pw);
                }
            }
        }

        // the chunk's sum of squares: the fixed tree of chunk_tree, as in k_reduce
        float *redb = red + cb * TPC * W;
        const float total = chunk_tree<NT, TPC, FZ>(part, redb, tid, [] { named_barrier(1, NT); });
        if (tid == 0) F.chunk_sq[k] = total;
        cb ^= 1;

        // the chunk's leaves: each warp sums its lanes' limb sums exactly (27-bit pieces)
        // and hands the piece sums to the leaf warp
        if (LEAVES) {
            uint32_t pc[kFusedPieces];
#pragma unroll
            for (int st = 0; st < 3; ++st) {
                const uint64_t limb[3] = {acc[st].a0, acc[st].a1, acc[st].a2};
#pragma unroll
                for (int l = 0; l < 3; ++l) {
                    pc[(st * 3 + l) * 3 + 0] = uint32_t(limb[l]) & ((1u << 27) - 1);
                    pc[(st * 3 + l) * 3 + 1] = uint32_t(limb[l] >> 27) & ((1u << 27) - 1);
                    pc[(st * 3 + l) * 3 + 2] = uint32_t(limb[l] >> 54);
                }
            }
#pragma unroll
            for (int i = 0; i < kFusedPieces; ++i) pc[i] = __reduce_add_sync(0xFFFFFFFFu, pc[i]);
            if (lane == 0) {
                const uint32_t b = ci % kFusedLeafBufs, round = ci / kFusedLeafBufs;
                if (!aborted &&
                    !mbar_wait_bounded(smem_u32(&leaf_empty[b]), (round & 1u) ^ 1u, abort_flag)) {
                    aborted = true;
                    atomicOr(&A.sc->flags, kFlagTimeoutAdamw);
                    *abort_flag = 1;
                }
                uint32_t *pb = pieces_buf + (b * W + warp) * kFusedPieces;
#pragma unroll
                for (int i = 0; i < kFusedPieces; ++i) pb[i] = pc[i];
                leaf_chunk[b] = k;                     // every warp writes the same index
                mbar_arrive(smem_u32(&leaf_full[b]));
            }
        }
    }
}

template <int FZ, int DT, int RG, int LEAVES>
FusedKernelFn pick_fused_pm(const FusedShape &s)
{
    if (s.pt) return s.mk ? k_fused<kFusedNT, DT, RG, LEAVES, 1, FZ, 1> : k_fused<kFusedNT, DT, RG, LEAVES, 1, FZ, 0>;
    return s.mk ? k_fused<kFusedNT, DT, RG, LEAVES, 0, FZ, 1> : k_fused<kFusedNT, DT, RG, LEAVES, 0, FZ, 0>;
}

template <int FZ, int DT, int RG>
FusedKernelFn pick_fused_l(const FusedShape &s)
{
    return s.leaves ? pick_fused_pm<FZ, DT, RG, 1>(s) : pick_fused_pm<FZ, DT, RG, 0>(s);
}

// WIDE 0: R = 4 or 8 (one replica stage per tile); WIDE 1: R = 16 (two).  R = 32 (four
// replica stages per tile, then the state's, in a ring of three slots) was measured slower
// than the two passes at 268M parameters (7.62 against 6.06 ms) and is left to them.
template <int FZ, int DT, int WIDE>
FusedKernelFn pick_fused_r(const FusedShape &s)
{
    if constexpr (WIDE == 0) {
        if (s.rg == 4) return pick_fused_l<FZ, DT, 4>(s);
        if (s.rg == 8) return pick_fused_l<FZ, DT, 8>(s);
    } else {
        if (s.rg == 16) return pick_fused_l<FZ, DT, 16>(s);
    }
    return nullptr;
}

// The variant of a launch in one arithmetic mode and replica-count class; null for a shape
// the kernel does not cover.  The four classes compile as translation units of their own
// (k_fused.cu, k_fused_ftz.cu, k_fused_wide.cu, k_fused_wide_ftz.cu), in parallel.
template <int FZ, int WIDE>
FusedKernelFn pick_fused(const FusedShape &s)
{
    if (s.dtype == 0) return pick_fused_r<FZ, 0, WIDE>(s);
    if (s.dtype == 1) return pick_fused_r<FZ, 1, WIDE>(s);
    return nullptr;
}

}  // namespace

}  // namespace repstep
