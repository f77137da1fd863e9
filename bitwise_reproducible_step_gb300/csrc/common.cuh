// common.cuh -- device helpers shared by the repstep kernels (sm_103a).
//
// * mbarrier + 1-D bulk TMA (cp.async.bulk) staging of HBM tiles into shared memory,
//   with bounded waits: no wait in this library can spin forever.  A wait that runs
//   past its limit sets a device flag and the kernel winds down without touching its
//   ring again (the host reads the flag with repstep_sync()).
// * The fixed chunk tree: the perfect pairwise tree over one 4096-element chunk, whose
//   rounding sequence is independent of grid size and of the compute-thread count.
// * PF61 arithmetic modulo 2^61 - 1 and the BLAKE2b compression (RFC 7693) used for
//   Merkle nodes.
//
// All fp32 arithmetic of the step goes through Ar<FZ> below: the explicitly rounded
// intrinsics (__fadd_rn, __fmul_rn, __fdiv_rn, __fsqrt_rn), which the compiler never
// contracts into FMA ("OPEN-1B: A Fully Auditable Training Run", §2.1 "Fused multiply-add":
// explicitly unfused multiply and add on the GPU), optionally followed by a software
// flush of subnormal results (§2.1 "Subnormals").  The library is built with -fmad=false.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace repstep {

constexpr uint32_t kChunk = 4096;
constexpr int kMaxReplicas = 256;
constexpr uint32_t kFlagNonfinite = 0x1u;
constexpr uint32_t kFlagTimeoutReduce = 0x2u;
constexpr uint32_t kFlagTimeoutAdamw = 0x4u;
constexpr uint32_t kFlagTimeoutLeaves = 0x8u;
constexpr uint64_t kNoChunk = ~0ull;     // ring-stage marker of the persistent kernels: no chunk follows

// PF61 modulus p = 2^61 - 1 and multiplier K = floor(2^61 (sqrt5 - 1)/2).
constexpr uint64_t kP61 = 0x1FFFFFFFFFFFFFFFull;
constexpr uint64_t kK61 = 0x13C6EF372FE94F82ull;

// ----------------------------------------------------------------------------------
// Arithmetic policy.  FZ = 0: IEEE binary32 with gradual underflow.  FZ = 1:
// flush-to-zero ("OPEN-1B", §2.1 "Subnormals": FTZ zeroes a subnormal result, DAZ a
// subnormal input), read as: every operation treats a subnormal operand as a zero of the
// same sign, and zeroes (keeping the sign) a result that is tiny in IEEE 754's sense with
// tininess detected after rounding -- the exact result rounded to 24 bits as though the
// exponent were unbounded lies below 2^-126.  The .rn.ftz forms of add, sub, mul, div and
// sqrt do exactly this, one instruction each: a sum below 2^-126 is exact, a square root
// of a normal value is normal, and for products and quotients the flush decision was
// checked against that rule on operands built to land within a few units of 2^-126.
// So no operand needs a separate flush; flush_subnormal (a .ftz multiply by 1.0: any
// other value times 1.0 is exact, NaN stays NaN) remains for the few values that leave
// the kernels without passing through an operation.
// ----------------------------------------------------------------------------------
__device__ __forceinline__ float flush_subnormal(float x)
{
    float r;
    asm("mul.rn.ftz.f32 %0, %1, 0f3F800000;" : "=f"(r) : "f"(x));
    return r;
}

template <int FZ>
struct Ar {
    static __device__ __forceinline__ float in(float x)
    {
        if constexpr (FZ != 0) return flush_subnormal(x);
        else return x;
    }
    static __device__ __forceinline__ float add(float a, float b)
    {
        if constexpr (FZ == 0) return __fadd_rn(a, b);
        float r;
        asm("add.rn.ftz.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
        return r;
    }
    static __device__ __forceinline__ float sub(float a, float b)
    {
        if constexpr (FZ == 0) return __fsub_rn(a, b);
        float r;
        asm("sub.rn.ftz.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
        return r;
    }
    static __device__ __forceinline__ float mul(float a, float b)
    {
        if constexpr (FZ == 0) return __fmul_rn(a, b);
        float r;
        asm("mul.rn.ftz.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
        return r;
    }
    static __device__ __forceinline__ float div(float a, float b)
    {
        if constexpr (FZ == 0) return __fdiv_rn(a, b);
        float r;
        asm("div.rn.ftz.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
        return r;
    }
    static __device__ __forceinline__ float sqrt(float a)
    {
        if constexpr (FZ == 0) return __fsqrt_rn(a);
        float r;
        asm("sqrt.rn.ftz.f32 %0, %1;" : "=f"(r) : "f"(a));
        return r;
    }
};

// Device-side scalars kept in the workspace.
struct Scalars {
    float norm;           // pre-clip global norm of the last clip
    float scale;          // clip scale of the last clip
    uint32_t flags;       // REPSTEP_FLAG_* bits
    uint32_t aux;         // scratch flag of host-driven checks (image narrowing)
    uint64_t root;        // last Merkle root
    uint32_t next_chunk;  // work counter of the running reduce (zeroed before each launch)
    uint32_t spare;
};

// Whether a launch runs: always, or only when the last clip's scale is not exactly 1 (the
// second pass of the single-pass step, after it speculated that the step would not clip).
// A closed gate returns before any access.
enum : int {
    kGateAlways = 0,
    kGateIfClipped = 1,
};

__device__ __forceinline__ bool gate_open(int gate, const Scalars *sc)
{
    return gate == kGateAlways || __float_as_uint(sc->scale) != 0x3F800000u;
}

// ----------------------------------------------------------------------------------
// PTX wrappers: shared-memory addresses, mbarriers, bulk copies, timers
// ----------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Longest any single wait may take before it is declared stuck.
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s
constexpr uint32_t kWaitLimitSpins = 1u << 28;

// Wait for the phase of parity `parity` of barrier `bar` to complete.  Returns false if
// *abort_flag becomes non-zero or the time / spin limit passes.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  const volatile int *abort_flag)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t spin = 0; spin < kWaitLimitSpins; ++spin) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
    return false;
}

// Before the producer refills a ring slot: the consumers' reads of the slot are generic-
// proxy loads, the refill is an async-proxy (bulk-copy) write, and only a proxy fence
// orders the two.  The producer lane runs it after the slot's empty barrier completes
// (which makes every consumer read happen before it) and before it issues the copies.
// Without it a refill overtook a read still in flight: about 1 run in 80 of a 268M-
// parameter step with 256-thread AdamW CTAs had a warp read part of the next tile.
__device__ __forceinline__ void fence_reads_before_refill()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// L2 policy for data read exactly once (replica gradients, optimizer state).
__device__ __forceinline__ uint64_t l2_evict_first()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 1-D bulk copy global -> this CTA's shared memory, completing on `bar` as tx bytes.
// dst and src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar, uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(pol)
        : "memory");
}

__device__ __forceinline__ void named_barrier(uint32_t id, uint32_t nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier that also returns, to every participating thread, the OR of `pred` over
// all of them (whole warps only, like bar.sync).
__device__ __forceinline__ bool named_barrier_or(uint32_t id, uint32_t nthreads, bool pred)
{
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\t"
                 "setp.ne.u32 p, %1, 0;\n\t"
                 "bar.red.or.pred q, %2, %3, p;\n\t"
                 "selp.u32 %0, 1, 0, q;\n\t}"
                 : "=r"(r)
                 : "r"(pred ? 1u : 0u), "r"(id), "r"(nthreads)
                 : "memory");
    return r != 0;
}

// ----------------------------------------------------------------------------------
// Tile geometry.  A tile is TE consecutive elements starting at `base`; the part inside
// the active range [lo, hi) is [a, b); its 16-byte-aligned interior [a16, b16) is staged
// by bulk copy, the (< vec element) head and tail are read with plain loads.
// ----------------------------------------------------------------------------------
struct TileRange {
    uint64_t base, a, b, a16, b16;
};

// The range of a tile that lies wholly inside the active range (every chunk of the range
// but the two at its ends).
__device__ __forceinline__ TileRange whole_tile(uint64_t base, uint32_t te)
{
    return TileRange{base, base, base + te, base, base + te};
}

// Position in a ring of S stages: the slot and the parity of its current round, advanced
// without the division that it % S and it / S would cost per stage.
struct RingPos {
    uint32_t slot = 0, phase = 0;
    __device__ __forceinline__ void advance(uint32_t S)
    {
        if (++slot == S) {
            slot = 0;
            phase ^= 1u;
        }
    }
};

__device__ __forceinline__ TileRange tile_range(uint64_t base, uint32_t te, uint64_t lo,
                                                uint64_t hi, uint32_t vec)
{
    TileRange t;
    t.base = base;
    t.a = base > lo ? base : lo;
    uint64_t e = base + te;
    t.b = e < hi ? e : hi;
    if (t.b < t.a) t.b = t.a;
    t.a16 = (t.a + vec - 1) / vec * vec;
    t.b16 = t.b / vec * vec;
    if (t.b16 < t.a16) t.b16 = t.a16;
    return t;
}

// ----------------------------------------------------------------------------------
// Fixed chunk tree (sum of non-negative squares over one 4096-element chunk).
// Compute thread t owns elements {j*4*NT + 4t + i : i < 4, j < TPC} of the chunk
// (TPC = 4096 / (4*NT)), so that:
//   levels 1-2     the thread's 4 consecutive elements        ((q0+q1)+(q2+q3))
//   levels 3-7     the 32 lanes of a warp, xor butterfly      (adjacent 4-groups)
//   levels 8..     the NT/32 warps of the block, in shared memory
//   last levels    the TPC tiles of the chunk
// -- exactly the perfect pairwise tree over the chunk in index order.  Addition is
// commutative in IEEE arithmetic, so both butterfly partners hold the same bits.
// Elements past n contribute +0, which equals the canonical tree over the short chunk
// because every term is >= +0.
// ----------------------------------------------------------------------------------
template <int W, int FZ>
__device__ __forceinline__ float tree_pow2(float *x)
{
#pragma unroll
    for (int s = 1; s < W; s <<= 1) {
#pragma unroll
        for (int i = 0; i < W; i += 2 * s) x[i] = Ar<FZ>::add(x[i], x[i + s]);
    }
    return x[0];
}

template <int FZ>
__device__ __forceinline__ float sum4(float a, float b, float c, float d)
{
    return Ar<FZ>::add(Ar<FZ>::add(a, b), Ar<FZ>::add(c, d));
}

// red: shared scratch of TPC * (NT/32) floats.  All NT compute threads call this; the
// chunk total is returned in thread 0.  `sync` synchronises exactly the NT threads.
template <int NT, int TPC, int FZ, typename Sync>
__device__ __forceinline__ float chunk_tree(float (&part)[TPC], float *red, int tid, Sync sync)
{
    constexpr int W = NT / 32;
#pragma unroll
    for (int j = 0; j < TPC; ++j) {
        float v = part[j];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1)
            v = Ar<FZ>::add(v, __shfl_xor_sync(0xffffffffu, v, off));
        part[j] = v;
    }
    const int warp = tid >> 5;
    if ((tid & 31) == 0) {
#pragma unroll
        for (int j = 0; j < TPC; ++j) red[j * W + warp] = part[j];
    }
    sync();
    float total = 0.0f;
    if (tid == 0) {
        float tiles[TPC];
#pragma unroll
        for (int j = 0; j < TPC; ++j) {
            float w[W];
#pragma unroll
            for (int i = 0; i < W; ++i) w[i] = red[j * W + i];
            tiles[j] = tree_pow2<W, FZ>(w);
        }
        total = tree_pow2<TPC, FZ>(tiles);
    }
    return total;
}

// ----------------------------------------------------------------------------------
// PF61: arithmetic modulo p = 2^61 - 1 (2^61 == 1 mod p)
// ----------------------------------------------------------------------------------
__device__ __forceinline__ uint64_t pf_reduce64(uint64_t x)
{
    x = (x & kP61) + (x >> 61);
    return x >= kP61 ? x - kP61 : x;
}

__device__ __forceinline__ uint64_t pf_add(uint64_t a, uint64_t b)   // a, b < p
{
    return pf_reduce64(a + b);
}

__device__ __forceinline__ uint64_t pf_mul(uint64_t a, uint64_t b)   // a, b < p
{
    const uint64_t lo = a * b;
    const uint64_t hi = __umul64hi(a, b);          // product < 2^122, so hi < 2^58
    // hi * 2^64 == hi * 8 (mod p)
    uint64_t s = (lo & kP61) + (lo >> 61) + (hi << 3);
    return pf_reduce64(s);
}

// a (128-bit as four 32-bit limbs) += x * P where P = p1 * 2^32 + p0 (P < 2^61).
__device__ __forceinline__ void pf_mac(uint32_t (&a)[4], uint32_t x, uint32_t p0, uint32_t p1)
{
    asm("mad.lo.cc.u32  %0, %4, %5, %0;\n\t"
        "madc.hi.cc.u32 %1, %4, %5, %1;\n\t"
        "addc.cc.u32    %2, %2, 0;\n\t"
        "addc.u32       %3, %3, 0;\n\t"
        "mad.lo.cc.u32  %1, %4, %6, %1;\n\t"
        "madc.hi.cc.u32 %2, %4, %6, %2;\n\t"
        "addc.u32       %3, %3, 0;"
        : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3])
        : "r"(x), "r"(p0), "r"(p1));
}

// 128-bit value mod p.
__device__ __forceinline__ uint64_t pf_fold128(const uint32_t (&a)[4])
{
    const uint64_t lo = (uint64_t(a[1]) << 32) | a[0];
    const uint64_t hi = (uint64_t(a[3]) << 32) | a[2];
    // hi * 2^64 == hi * 8; write hi = h1 * 2^58 + h0, then hi * 8 == h1 + h0 * 8.
    const uint64_t h0 = hi & ((1ull << 58) - 1), h1 = hi >> 58;
    uint64_t s = (lo & kP61) + (lo >> 61) + (h0 << 3) + h1;   // < 2^62 + 2^7
    return pf_reduce64(pf_reduce64(s));
}

// ----------------------------------------------------------------------------------
// BLAKE2b (RFC 7693) specialised to one 16-byte message LE64(a) || LE64(b), unkeyed,
// 8-byte digest: the Merkle node function N(a, b).
// ----------------------------------------------------------------------------------
__device__ __forceinline__ uint64_t rotr64(uint64_t x, int s)
{
    return (x >> s) | (x << (64 - s));
}

#define REPSTEP_B2_G(a, b, c, d, x, y)        \
    do {                                      \
        v[a] = v[a] + v[b] + (x);             \
        v[d] = rotr64(v[d] ^ v[a], 32);       \
        v[c] = v[c] + v[d];                   \
        v[b] = rotr64(v[b] ^ v[c], 24);       \
        v[a] = v[a] + v[b] + (y);             \
        v[d] = rotr64(v[d] ^ v[a], 16);       \
        v[c] = v[c] + v[d];                   \
        v[b] = rotr64(v[b] ^ v[c], 63);       \
    } while (0)

// m(i): message word i (only words 0 and 1 are non-zero).
#define REPSTEP_B2_M(i) ((i) == 0 ? ma : ((i) == 1 ? mb : 0ull))

#define REPSTEP_B2_ROUND(s0, s1, s2, s3, s4, s5, s6, s7, s8, s9, s10, s11, s12, s13, s14, s15) \
    do {                                                                                   \
        REPSTEP_B2_G(0, 4, 8, 12, REPSTEP_B2_M(s0), REPSTEP_B2_M(s1));                    \
        REPSTEP_B2_G(1, 5, 9, 13, REPSTEP_B2_M(s2), REPSTEP_B2_M(s3));                    \
        REPSTEP_B2_G(2, 6, 10, 14, REPSTEP_B2_M(s4), REPSTEP_B2_M(s5));                   \
        REPSTEP_B2_G(3, 7, 11, 15, REPSTEP_B2_M(s6), REPSTEP_B2_M(s7));                   \
        REPSTEP_B2_G(0, 5, 10, 15, REPSTEP_B2_M(s8), REPSTEP_B2_M(s9));                   \
        REPSTEP_B2_G(1, 6, 11, 12, REPSTEP_B2_M(s10), REPSTEP_B2_M(s11));                 \
        REPSTEP_B2_G(2, 7, 8, 13, REPSTEP_B2_M(s12), REPSTEP_B2_M(s13));                  \
        REPSTEP_B2_G(3, 4, 9, 14, REPSTEP_B2_M(s14), REPSTEP_B2_M(s15));                  \
    } while (0)

__device__ __forceinline__ uint64_t b2_node(uint64_t ma, uint64_t mb)
{
    // initialisation vector (RFC 7693 §2.6) and parameter block: digest length 8, no key
    const uint64_t iv0 = 0x6A09E667F3BCC908ull, iv1 = 0xBB67AE8584CAA73Bull,
                   iv2 = 0x3C6EF372FE94F82Bull, iv3 = 0xA54FF53A5F1D36F1ull,
                   iv4 = 0x510E527FADE682D1ull, iv5 = 0x9B05688C2B3E6C1Full,
                   iv6 = 0x1F83D9ABFB41BD6Bull, iv7 = 0x5BE0CD19137E2179ull;
    const uint64_t h0 = iv0 ^ 0x01010008ull;
    uint64_t v[16] = {h0,  iv1, iv2, iv3, iv4, iv5, iv6, iv7,
                      iv0, iv1, iv2, iv3, iv4 ^ 16ull, iv5, ~iv6, iv7};
    // message schedule SIGMA (RFC 7693 §2.7); rounds 10 and 11 repeat rounds 0 and 1
    REPSTEP_B2_ROUND(0, 1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12, 13, 14, 15);
    REPSTEP_B2_ROUND(14, 10, 4, 8, 9, 15, 13, 6, 1, 12, 0, 2, 11, 7, 5, 3);
    REPSTEP_B2_ROUND(11, 8, 12, 0, 5, 2, 15, 13, 10, 14, 3, 6, 7, 1, 9, 4);
    REPSTEP_B2_ROUND(7, 9, 3, 1, 13, 12, 11, 14, 2, 6, 5, 10, 4, 0, 15, 8);
    REPSTEP_B2_ROUND(9, 0, 5, 7, 2, 4, 10, 15, 14, 1, 11, 12, 6, 8, 3, 13);
    REPSTEP_B2_ROUND(2, 12, 6, 10, 0, 11, 8, 3, 4, 13, 7, 5, 15, 14, 1, 9);
    REPSTEP_B2_ROUND(12, 5, 1, 15, 14, 13, 4, 10, 0, 7, 6, 3, 9, 2, 8, 11);
    REPSTEP_B2_ROUND(13, 11, 7, 14, 12, 1, 3, 9, 5, 0, 15, 4, 8, 6, 2, 10);
    REPSTEP_B2_ROUND(6, 15, 14, 9, 11, 3, 0, 8, 12, 2, 13, 7, 1, 4, 10, 5);
    REPSTEP_B2_ROUND(10, 2, 8, 4, 7, 6, 1, 5, 15, 11, 9, 14, 3, 12, 13, 0);
    REPSTEP_B2_ROUND(0, 1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12, 13, 14, 15);
    REPSTEP_B2_ROUND(14, 10, 4, 8, 9, 15, 13, 6, 1, 12, 0, 2, 11, 7, 5, 3);
    return h0 ^ v[0] ^ v[8];
}

#undef REPSTEP_B2_ROUND
#undef REPSTEP_B2_M

// The full BLAKE2b compression F(h, m, t, last) of RFC 7693 §3.2 on one 128-byte block.
#define REPSTEP_B2_RF(s0, s1, s2, s3, s4, s5, s6, s7, s8, s9, s10, s11, s12, s13, s14, s15) \
    do {                                                                                \
        REPSTEP_B2_G(0, 4, 8, 12, m[s0], m[s1]);                                        \
        REPSTEP_B2_G(1, 5, 9, 13, m[s2], m[s3]);                                        \
        REPSTEP_B2_G(2, 6, 10, 14, m[s4], m[s5]);                                       \
        REPSTEP_B2_G(3, 7, 11, 15, m[s6], m[s7]);                                       \
        REPSTEP_B2_G(0, 5, 10, 15, m[s8], m[s9]);                                       \
        REPSTEP_B2_G(1, 6, 11, 12, m[s10], m[s11]);                                     \
        REPSTEP_B2_G(2, 7, 8, 13, m[s12], m[s13]);                                      \
        REPSTEP_B2_G(3, 4, 9, 14, m[s14], m[s15]);                                      \
    } while (0)

__device__ __forceinline__ void b2_compress(uint64_t (&h)[8], const uint64_t (&m)[16],
                                            uint64_t t, bool last)
{
    uint64_t v[16] = {h[0], h[1], h[2], h[3], h[4], h[5], h[6], h[7],
                      0x6A09E667F3BCC908ull, 0xBB67AE8584CAA73Bull, 0x3C6EF372FE94F82Bull,
                      0xA54FF53A5F1D36F1ull, 0x510E527FADE682D1ull ^ t, 0x9B05688C2B3E6C1Full,
                      0x1F83D9ABFB41BD6Bull, 0x5BE0CD19137E2179ull};
    if (last) v[14] = ~v[14];
    REPSTEP_B2_RF(0, 1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12, 13, 14, 15);
    REPSTEP_B2_RF(14, 10, 4, 8, 9, 15, 13, 6, 1, 12, 0, 2, 11, 7, 5, 3);
    REPSTEP_B2_RF(11, 8, 12, 0, 5, 2, 15, 13, 10, 14, 3, 6, 7, 1, 9, 4);
    REPSTEP_B2_RF(7, 9, 3, 1, 13, 12, 11, 14, 2, 6, 5, 10, 4, 0, 15, 8);
    REPSTEP_B2_RF(9, 0, 5, 7, 2, 4, 10, 15, 14, 1, 11, 12, 6, 8, 3, 13);
    REPSTEP_B2_RF(2, 12, 6, 10, 0, 11, 8, 3, 4, 13, 7, 5, 15, 14, 1, 9);
    REPSTEP_B2_RF(12, 5, 1, 15, 14, 13, 4, 10, 0, 7, 6, 3, 9, 2, 8, 11);
    REPSTEP_B2_RF(13, 11, 7, 14, 12, 1, 3, 9, 5, 0, 15, 4, 8, 6, 2, 10);
    REPSTEP_B2_RF(6, 15, 14, 9, 11, 3, 0, 8, 12, 2, 13, 7, 1, 4, 10, 5);
    REPSTEP_B2_RF(10, 2, 8, 4, 7, 6, 1, 5, 15, 11, 9, 14, 3, 12, 13, 0);
    REPSTEP_B2_RF(0, 1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12, 13, 14, 15);
    REPSTEP_B2_RF(14, 10, 4, 8, 9, 15, 13, 6, 1, 12, 0, 2, 11, 7, 5, 3);
#pragma unroll
    for (int i = 0; i < 8; ++i) h[i] ^= v[i] ^ v[i + 8];
}

// Unkeyed BLAKE2b-64 initial state (digest length 8 in the parameter block).
__device__ __forceinline__ void b2_init64(uint64_t (&h)[8])
{
    h[0] = 0x6A09E667F3BCC908ull ^ 0x01010008ull;
    h[1] = 0xBB67AE8584CAA73Bull;
    h[2] = 0x3C6EF372FE94F82Bull;
    h[3] = 0xA54FF53A5F1D36F1ull;
    h[4] = 0x510E527FADE682D1ull;
    h[5] = 0x9B05688C2B3E6C1Full;
    h[6] = 0x1F83D9ABFB41BD6Bull;
    h[7] = 0x5BE0CD19137E2179ull;
}

#undef REPSTEP_B2_RF
#undef REPSTEP_B2_G

}  // namespace repstep
