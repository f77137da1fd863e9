// k_reduce.cuh -- replica reduce + per-chunk sum of squares (one HBM pass over R gradients).
// The kernel template; k_reduce.cu instantiates the IEEE variants (FZ = 0) and holds the
// host-side launch helpers, k_reduce_ftz.cu the flush-to-zero variants (FZ = 1).
//
// Computes, for every element i of the active range,
//     g_i = T_{r<R}(G_r[i]) * fp32(1/R)
// with T the canonical tree over global replica index ("OPEN-1B: A Fully Auditable
// Training Run", App. A.1: replicas paired, pairs paired again, lower replica on the
// left; §5: a non-power-of-two count is split into its largest power-of-two block and
// the rest; App. A.3: the average is a multiply by the reciprocal, never a divide),
// and, for every 4096-element chunk lying wholly inside the range, the chunk's sum of
// squares s_k = T(g_i * g_i) in the fixed perfect tree of common.cuh.
//
// GB300 design: a persistent grid of one CTA per SM (192 KB ring).  The last warp is the
// producer: one lane streams tiles of TE = 4*NT elements of up to RG replicas at a time
// from HBM into a shared-memory ring with 1-D bulk TMA copies (cp.async.bulk, L2
// evict-first), completing on an mbarrier per stage.  The NT compute threads each take
// one 4-element group (a 16-byte float4, or 8 bytes of bf16) per replica per tile, sum
// the replicas in registers with a binary-carry stack that reproduces the canonical tree
// for any R, multiply by fp32(1/R), store g with 16-byte stores and fold g*g into the
// chunk tree.  With fp32 gradients the chunks are handed out at run time from a counter
// (the kernel's only atomic, on an index, never on data); with bf16 gradients by CTA
// index.  Every sum has one fixed order: the grid size, NT and the chunk order change
// which CTA does which chunk, never any rounding.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace repstep {

namespace {

constexpr uint32_t kRingBytes = 192 * 1024;
constexpr uint32_t kMaxStages = 12;
constexpr uint32_t kRingOffset = 1024;   // barriers, chunk-tree scratch and abort flag first

template <int FZ>
__device__ __forceinline__ float4 add4(float4 a, float4 b)
{
    return make_float4(Ar<FZ>::add(a.x, b.x), Ar<FZ>::add(a.y, b.y), Ar<FZ>::add(a.z, b.z),
                       Ar<FZ>::add(a.w, b.w));
}

template <int FZ>
__device__ __forceinline__ float4 mul4(float4 a, float b)
{
    return make_float4(Ar<FZ>::mul(a.x, b), Ar<FZ>::mul(a.y, b), Ar<FZ>::mul(a.z, b),
                       Ar<FZ>::mul(a.w, b));
}

// Push a complete block of 2^BASE replicas, the `cnt`-th such block, onto the carry
// stack: while the stack holds a block of the same size, combine (lower block on the
// left) and move up a level -- binary counting, as in TreeFold.
template <int MAXLEV, int BASE, int FZ>
__device__ __forceinline__ void push_block(float4 (&st)[MAXLEV], uint32_t cnt, float4 a)
{
    bool carry = true;
#pragma unroll
    for (int L = BASE; L < MAXLEV; ++L) {
        if (carry) {
            if ((cnt >> (L - BASE)) & 1u) {
                a = add4<FZ>(st[L], a);
            } else {
                st[L] = a;
                carry = false;
            }
        }
    }
}

// The same push for the paper-exact mode, where every virtual rank's partial is pushed on
// its own.  The number of carries is the number of trailing one bits of cnt, the same for
// every thread of the warp, so a switch runs exactly those folds as straight-line code
// instead of a predicated pass over every level.  fold_carries<L0, K> computes
// a = st[L0] + a, then st[L0+1] + a, ... K times, and stores the result at level L0 + K:
// the order of push_block.  (The other modes keep push_block: with two stacks live, as in
// the staged mode, the switch's code raises register spills.)
template <int L0, int K, int MAXLEV, int FZ>
__device__ __forceinline__ void fold_carries(float4 (&st)[MAXLEV], float4 a)
{
    if constexpr (K == 0) st[L0] = a;
    else fold_carries<L0 + 1, K - 1, MAXLEV, FZ>(st, add4<FZ>(st[L0], a));
}

#define REPSTEP_PUSH_CASE(K)                                                              \
    case K:                                                                               \
        if constexpr (K < MAXLEV) fold_carries<0, K, MAXLEV, FZ>(st, a);                   \
        break;

template <int MAXLEV, int FZ>
__device__ __forceinline__ void push_one_switched(float4 (&st)[MAXLEV], uint32_t cnt, float4 a)
{
    const uint32_t carries = uint32_t(__ffs(int(~cnt))) - 1u;   // trailing ones of cnt
    switch (carries) {
        REPSTEP_PUSH_CASE(0)
        REPSTEP_PUSH_CASE(1)
        REPSTEP_PUSH_CASE(2)
        REPSTEP_PUSH_CASE(3)
        REPSTEP_PUSH_CASE(4)
        REPSTEP_PUSH_CASE(5)
        REPSTEP_PUSH_CASE(6)
        REPSTEP_PUSH_CASE(7)
        REPSTEP_PUSH_CASE(8)
    default: break;
    }
}

#undef REPSTEP_PUSH_CASE

// Canonical-tree result of `count` pushed items: the stack holds one block per set bit
// of count (largest block = lowest replicas at the highest level).  The recursive split
// T = T(first 2^k) + T(rest) combines them from the smallest block upward, each larger
// (lower-replica) block on the left.
template <int MAXLEV, int FZ>
__device__ __forceinline__ float4 stack_result(const float4 (&st)[MAXLEV], uint32_t count)
{
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    bool have = false;
#pragma unroll
    for (int L = 0; L < MAXLEV; ++L) {
        if ((count >> L) & 1u) {
            if (have) {
                acc = add4<FZ>(st[L], acc);
            } else {
                acc = st[L];
                have = true;
            }
        }
    }
    return acc;
}

// TreeFold's Result in the paper-exact mode: the leftover blocks, one per set bit of
// `count`, combined starting from the largest (lowest replicas, highest level), each later
// block added on the right.
template <int MAXLEV, int FZ>
__device__ __forceinline__ float4 stack_result_leftfold(const float4 (&st)[MAXLEV], uint32_t count)
{
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    bool have = false;
#pragma unroll
    for (int L = MAXLEV - 1; L >= 0; --L) {
        if ((count >> L) & 1u) {
            if (have) {
                acc = add4<FZ>(acc, st[L]);
            } else {
                acc = st[L];
                have = true;
            }
        }
    }
    return acc;
}

template <int RG, int FZ>
__device__ __forceinline__ float4 tree_group(float4 (&x)[RG])
{
#pragma unroll
    for (int s = 1; s < RG; s <<= 1) {
#pragma unroll
        for (int i = 0; i < RG; i += 2 * s) x[i] = add4<FZ>(x[i], x[i + s]);
    }
    return x[0];
}

template <int DT>
__device__ __forceinline__ float load_elem(const void *p, uint64_t e)
{
    if (DT == 0) return __ldg(static_cast<const float *>(p) + e);
    const uint16_t b = __ldg(static_cast<const unsigned short *>(p) + e);
    return __uint_as_float(uint32_t(b) << 16);   // bf16 -> fp32 exactly
}

template <int DT>
__device__ __forceinline__ float4 load_group_raw(const unsigned char *tile, uint32_t off,
                                                 bool in_bulk, const void *src, uint64_t e0,
                                                 uint64_t a, uint64_t b)
{
    if (in_bulk) {
        if (DT == 0) return *reinterpret_cast<const float4 *>(tile + off * 4u);
        const uint2 u = *reinterpret_cast<const uint2 *>(tile + off * 2u);
        return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                           __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
    }
    float r[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint64_t e = e0 + i;
        r[i] = (e >= a && e < b) ? load_elem<DT>(src, e) : 0.0f;
    }
    return make_float4(r[0], r[1], r[2], r[3]);
}

// One 4-element group of one replica: from the staged tile when the group lies in the
// bulk-copied interior, else element by element from global memory (zero outside [a, b)).
// The flush-to-zero mode needs no flush here: every value read reaches g only through
// .ftz additions and the final multiply by rho, which treat a subnormal operand as zero.
template <int DT, int FZ>
__device__ __forceinline__ float4 load_group(const unsigned char *tile, uint32_t off,
                                             bool in_bulk, const void *src, uint64_t e0,
                                             uint64_t a, uint64_t b)
{
    return load_group_raw<DT>(tile, off, in_bulk, src, e0, a, b);
}

// MODE 0: the canonical tree over all R replicas.  MODE 1: the same tree staged as a
// cluster would run it (each node's replicas, then the node partials).  MODE 2: the
// paper-exact order of OPEN-1B §6 Algorithm 1 (ascending shard sums times fp32(1/dp_shard),
// TreeFold over replicas, Result times fp32(1/dp_replicate)); A.gpn = dp_shard,
// A.nodes = dp_replicate, A.rho2 = fp32(1/dp_shard), A.rho = fp32(1/dp_replicate).  With
// A.accum > 0 the R inputs are microbatch gradients, A.accum per virtual rank in order,
// and each rank's gradient is the accumulation +0 + x_1*rho3 + x_2*rho3 + ... (the
// algorithm's inner loop; rho3 = fp32(1/accum)).
template <int NT, int DT, int MODE, int RG, int MAXLEV, int FZ>
__global__ void __launch_bounds__(NT + 32, 1) k_reduce(const __grid_constant__ ReduceArgs A)
{
    constexpr int W = NT / 32;
    constexpr uint32_t TE = 4u * NT;
    constexpr int TPC = int(kChunk / TE);
    constexpr uint32_t ESZ = DT == 0 ? 4u : 2u;
    constexpr uint32_t VEC = 16u / ESZ;
    constexpr int LOG2RG = RG == 8 ? 3 : (RG == 4 ? 2 : (RG == 2 ? 1 : 0));
    // Chunks handed out at run time (fp32 gradients) or by CTA index (bf16 gradients).
    // The run-time order lets CTAs on faster or earlier-free SMs take more chunks
    // (measured: fp32 reduce 6.34 -> 6.02 ms at 1.2e9 parameters); its per-chunk vote and
    // index read cost the instruction-heavier bf16 reduce more than it gains (3e9 bf16
    // gradients: 9.12 -> 9.75 ms).
    constexpr bool DYN = DT == 0;
    static_assert(16 * kMaxStages + 2 * TPC * W * 4 + 8 + 8 * kMaxStages <= kRingOffset,
                  "smem header");
    // the second pass of the single-pass step: nothing to do when the clip scale is 1
    if (!gate_open(A.gate, A.sc)) return;

    extern __shared__ __align__(1024) unsigned char smem[];
    const uint32_t S = A.stages;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + kMaxStages;
    float *red = reinterpret_cast<float *>(smem + 16 * kMaxStages);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(red + 2 * TPC * W);
    volatile int *never_flag = abort_flag + 1;   // stays 0: drain waits ignore the abort
    // the chunk index each ring slot's stage opens (kNoChunk: the end of the work)
    uint64_t *stage_chunk = reinterpret_cast<uint64_t *>(smem + 16 * kMaxStages + 2 * TPC * W * 4 + 8);
    unsigned char *ring = smem + kRingOffset;

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

    const uint32_t R = A.R;
    const uint32_t NG = (R + RG - 1) / RG;

    if (tid >= NT) {
        // ------------------------------ producer warp ------------------------------
        if (tid != NT) return;
        const uint64_t pol = l2_evict_first();
        uint32_t it = 0;
        RingPos pos;
        bool ok = true;
        // Chunks are handed out one at a time from a counter zeroed before the launch, so
        // a CTA that starts late (its SM still busy with another stream's kernel) takes
        // fewer and no SM idles while work is left.  Which CTA sums a chunk changes no bit.
        // The next index is fetched one chunk ahead.
        uint64_t k_next = A.chunk_lo + (DYN ? atomicAdd(&A.sc->next_chunk, 1u) : blockIdx.x);
        while (ok && k_next < A.chunk_hi) {
            const uint64_t k = k_next;
            k_next = DYN ? A.chunk_lo + atomicAdd(&A.sc->next_chunk, 1u) : k + gridDim.x;
            const bool whole = k * kChunk >= A.begin && k * kChunk + kChunk <= A.end;
            for (int j = 0; ok && j < TPC; ++j) {
                const uint64_t tb = k * kChunk + uint64_t(j) * TE;
                const TileRange tr = whole ? whole_tile(tb, TE)
                                           : tile_range(tb, TE, A.begin, A.end, VEC);
                const uint32_t bytes = uint32_t(tr.b16 - tr.a16) * ESZ;
                const uint32_t soff = uint32_t(tr.a16 - tr.base) * ESZ;
                for (uint32_t q = 0; q < NG; ++q) {
                    const uint32_t slot = pos.slot;
                    if (!mbar_wait_bounded(smem_u32(&empty[slot]), pos.phase ^ 1u,
                                           abort_flag)) {
                        ok = false;
                        break;
                    }
                    fence_reads_before_refill();
                    const uint32_t nr = min(uint32_t(RG), R - q * RG);
                    const uint32_t fb = smem_u32(&full[slot]);
                    if (DYN && j == 0 && q == 0) stage_chunk[slot] = k;   // published by the arrive
                    mbar_arrive_expect_tx(fb, bytes * nr);
                    if (bytes) {
                        const uint32_t dst = smem_u32(ring + slot * A.stage_stride) + soff;
                        for (uint32_t i = 0; i < nr; ++i) {
                            const unsigned char *src =
                                static_cast<const unsigned char *>(A.grads[q * RG + i]) +
                                tr.a16 * ESZ;
                            bulk_g2s(dst + i * TE * ESZ, src, bytes, fb, pol);
                        }
                    }
                    ++it;
                    pos.advance(S);
                }
            }
        }
        // with run-time chunks, one more stage, without data, carries the end marker
        if (DYN && ok) {
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
        // Never leave the CTA while copies into its ring may be in flight: wait (bounded)
        // for the most recent stage issued into every slot.
        const uint32_t last = it < S ? it : S;
        for (uint32_t d = 0; d < last; ++d) {
            const uint32_t idx = it - 1 - d;
            mbar_wait_bounded(smem_u32(&full[idx % S]), (idx / S) & 1u, never_flag);
        }
        return;
    }

    // ------------------------------ compute threads -------------------------------
    const int lane = tid & 31;
    const float rho = A.rho;
    RingPos pos;
    int cb = 0;
    bool aborted = false;
    for (uint32_t ci = 0;; ++ci) {
        uint64_t k = A.chunk_lo + blockIdx.x + uint64_t(ci) * gridDim.x;
        if (!DYN && k >= A.chunk_hi) break;
        if (DYN) {
            // The stage that opens the next chunk carries its index, or the end marker.
            // Every compute thread reads it and one barrier vote makes the decision
            // uniform, so all warps run the same number of chunks through the chunk-tree
            // barriers below (a failed wait votes for the end too).  The chunk's first
            // wait below then returns at once.
            const uint32_t slot0 = pos.slot;
            bool got = false;
            if (!aborted) {
                got = mbar_wait_bounded(smem_u32(&full[slot0]), pos.phase, abort_flag);
                if (!got) {
                    aborted = true;
                    if (lane == 0) {
                        atomicOr(&A.sc->flags, kFlagTimeoutReduce);
                        *abort_flag = 1;
                    }
                }
            }
            k = got ? stage_chunk[slot0] : kNoChunk;
            if (named_barrier_or(2, NT, k == kNoChunk)) break;
        }
        float part[TPC];
        const bool whole = k * kChunk >= A.begin && k * kChunk + kChunk <= A.end;
#pragma unroll
        for (int j = 0; j < TPC; ++j) {
            const uint64_t tb = k * kChunk + uint64_t(j) * TE;
            const TileRange tr = whole ? whole_tile(tb, TE) : tile_range(tb, TE, A.begin, A.end, VEC);
            const uint32_t off = 4u * tid;
            const uint64_t e0 = tr.base + off;
            const bool in_bulk = e0 >= tr.a16 && e0 + 4 <= tr.b16;
            float4 st[MAXLEV];
            float4 sto[MAXLEV];   // node partials (staged sum only)
            float4 inner = make_float4(0.f, 0.f, 0.f, 0.f);   // running shard sum (MODE 2)
            float4 macc = make_float4(0.f, 0.f, 0.f, 0.f);    // microbatch sum (MODE 2)
            uint32_t c_in = 0, c_out = 0;   // position within a node / replica, and its index
            uint32_t c_mb = 0;              // microbatch within the virtual rank (MODE 2)
            for (uint32_t q = 0; q < NG; ++q) {
                const uint32_t slot = pos.slot;
                if (!aborted &&
                    !mbar_wait_bounded(smem_u32(&full[slot]), pos.phase, abort_flag)) {
                    aborted = true;
                    if (lane == 0) {
                        atomicOr(&A.sc->flags, kFlagTimeoutReduce);
                        *abort_flag = 1;
                    }
                }
                const unsigned char *sb = ring + slot * A.stage_stride;
                const uint32_t nr = min(uint32_t(RG), R - q * RG);
                if constexpr (MODE == 0) {
                    float4 x[RG];
                    if (whole && nr == uint32_t(RG)) {
                        // a whole tile of a full group: every value is in the staged tile
#pragma unroll
                        for (int i = 0; i < RG; ++i)
                            x[i] = load_group<DT, FZ>(sb + i * TE * ESZ, off, true, nullptr, 0,
                                                      0, 0);
                    } else {
#pragma unroll
                        for (int i = 0; i < RG; ++i) {
                            if (uint32_t(i) < nr)
                                x[i] = load_group<DT, FZ>(sb + i * TE * ESZ, off, in_bulk,
                                                          A.grads[q * RG + i], e0, tr.a, tr.b);
                        }
                    }
                            __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&empty[slot]));
                    pos.advance(S);
                    if (R == uint32_t(RG)) {
                        // one full group: the carry stack would hold exactly this block at
                        // level log2(RG) and return it
                        st[LOG2RG] = tree_group<RG, FZ>(x);
                    } else if (nr == uint32_t(RG)) {
                        push_block<MAXLEV, LOG2RG, FZ>(st, q, tree_group<RG, FZ>(x));
                    } else {
#pragma unroll
                        for (int i = 0; i < RG; ++i)
                            if (uint32_t(i) < nr) push_block<MAXLEV, 0, FZ>(st, q * RG + i, x[i]);
                    }
                } else {
                    // one replica at a time straight from the staged tile
#pragma unroll 1
                    for (uint32_t i = 0; i < nr; ++i) {
                        const float4 xi = load_group<DT, FZ>(sb + i * TE * ESZ, off, in_bulk,
                                                         A.grads[q * RG + i], e0, tr.a, tr.b);
                        if constexpr (MODE == 2) {
                            // microbatches of a virtual rank: g_r <- g_r + x * fp32(1/accum)
                            // from g_r = +0 (an explicit add, so -0 becomes +0)
                            float4 xr = xi;
                            bool rank_ready = true;
                            if (A.accum) {
                                const float4 t = mul4<FZ>(xi, A.rho3);
                                macc = add4<FZ>(c_mb == 0 ? make_float4(0.f, 0.f, 0.f, 0.f) : macc, t);
                                rank_ready = ++c_mb == A.accum;
                                if (rank_ready) {
                                    c_mb = 0;
                                    xr = macc;
                                }
                            }
                            // virtual ranks in mesh order: ascending sum over a replica's
                            // shards, times fp32(1/dp_shard), then into the TreeFold
                            if (rank_ready) inner = c_in == 0 ? xr : add4<FZ>(inner, xr);
                            if (rank_ready && ++c_in == A.gpn) {
                                const float4 p = mul4<FZ>(inner, A.rho2);
                                push_one_switched<MAXLEV, FZ>(st, c_out++, p);
                                c_in = 0;
                            }
                        } else {
                            // per node first, then over nodes (a two-level cluster reduction)
                            push_block<MAXLEV, 0, FZ>(st, c_in, xi);
                            if (++c_in == A.gpn) {
                                const float4 p = stack_result<MAXLEV, FZ>(st, A.gpn);
                                push_block<MAXLEV, 0, FZ>(sto, c_out++, p);
                                c_in = 0;
                            }
                        }
                    }
                            __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&empty[slot]));
                    pos.advance(S);
                }
            }
            float4 s;
            if constexpr (MODE == 2) s = stack_result_leftfold<MAXLEV, FZ>(st, A.nodes);
            else if constexpr (MODE == 1) s = stack_result<MAXLEV, FZ>(sto, A.nodes);
            else s = R == uint32_t(RG) ? st[LOG2RG] : stack_result<MAXLEV, FZ>(st, R);
            const float4 gv = mul4<FZ>(s, rho);
            const bool all_in = e0 >= tr.a && e0 + 4 <= tr.b;
            float q4[4];
            if (all_in) {
                *reinterpret_cast<float4 *>(A.g + e0) = gv;
                q4[0] = Ar<FZ>::mul(gv.x, gv.x);
                q4[1] = Ar<FZ>::mul(gv.y, gv.y);
                q4[2] = Ar<FZ>::mul(gv.z, gv.z);
                q4[3] = Ar<FZ>::mul(gv.w, gv.w);
            } else {
                const float gg[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint64_t e = e0 + i;
                    const bool in = e >= tr.a && e < tr.b;
                    if (in) A.g[e] = gg[i];
                    q4[i] = in ? Ar<FZ>::mul(gg[i], gg[i]) : 0.0f;
                }
            }
            part[j] = sum4<FZ>(q4[0], q4[1], q4[2], q4[3]);
        }
        float *redb = red + cb * TPC * W;
        const float total =
            chunk_tree<NT, TPC, FZ>(part, redb, tid, [] { named_barrier(1, NT); });
        if (tid == 0) {
            const uint64_t c0 = k * kChunk;
            const uint64_t c1 = c0 + kChunk < A.n ? c0 + kChunk : A.n;
            if (c0 >= A.begin && c1 <= A.end) A.chunk_sq[k] = total;
        }
        cb ^= 1;
    }
}

template <int NT, int DT, int FZ>
ReduceKernelFn pick_dt(const ReduceShape &s)
{
    if (s.mode == 2)
        return s.maxlev == 6 ? k_reduce<NT, DT, 2, 8, 6, FZ> : k_reduce<NT, DT, 2, 8, 9, FZ>;
    if (s.mode == 1)
        return s.maxlev == 6 ? k_reduce<NT, DT, 1, 8, 6, FZ> : k_reduce<NT, DT, 1, 8, 9, FZ>;
    if (s.rg == 4) return k_reduce<NT, DT, 0, 4, 6, FZ>;
    if (s.maxlev == 6) return k_reduce<NT, DT, 0, 8, 6, FZ>;
    return k_reduce<NT, DT, 0, 8, 9, FZ>;
}

template <int FZ>
ReduceKernelFn pick_reduce(const ReduceShape &s)
{
    const bool bf = s.dtype == 1;
    switch (s.nt) {
    case 128: return bf ? pick_dt<128, 1, FZ>(s) : pick_dt<128, 0, FZ>(s);
    case 256: return bf ? pick_dt<256, 1, FZ>(s) : pick_dt<256, 0, FZ>(s);
    case 512: return bf ? pick_dt<512, 1, FZ>(s) : pick_dt<512, 0, FZ>(s);
    default: return nullptr;
    }
}

}  // namespace

}  // namespace repstep
