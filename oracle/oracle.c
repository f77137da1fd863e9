/*
 * oracle.c -- plain, slow, single-threaded CPU oracle for the bitwise-reproducible
 * optimizer step (replica reduce, global-norm clip, AdamW, chunked state hash).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark load this file's library.  The product path (the CUDA library
 * and its Python binding) never calls, links or imports it, and this file includes
 * nothing from the product path.
 *
 * Every function below is the plain definition written out: loops over element index,
 * recursion for trees, no blocking, no vectorisation, no threads.  Build with
 *     gcc -std=c11 -O2 -ffp-contract=off -fno-fast-math -fPIC -shared
 * so that a*b+c is never fused into one rounding (aarch64 GCC fuses by default in
 * GNU mode) and subnormals are kept (gradual underflow).
 *
 * Sources (cited by page title and section):
 *   [OPEN-1B]  "OPEN-1B: A Fully Auditable Training Run" -- §2.1 Reproducible Operations
 *              (reduction order, fused multiply-add, subnormals), §3.2 Training Recipe
 *              (AdamW, global-norm clipping at 1.0), §3.4.2 (pre-clip norm), App. A.1
 *              (TreeFold, lower-replica operand on the left), App. A.3 (average via
 *              reciprocal multiply), App. B (per-step state hash), §5 (for a count that
 *              is not a power of two, the butterfly splits off its largest power-of-two
 *              block and handles the rest separately).
 *   [CKPT]     "grow_a_language_model_checkpoints" -- Format / Total size sections:
 *              [int32 step][int32 n_params][w][m][v], total = 8 + 12 n bytes,
 *              beta1 = 0.9 for m and beta2 = 0.999 for v.
 *   [OLMO12]   OLMo-core MoE §12 "Topology-agnostic checkpoint saving and loading",
 *              Table 27: FP32 main weights + first moment + second moment = 12P bytes;
 *              §12.1 canonical element order independent of topology.
 *   [RFC7693]  BLAKE2b as specified in RFC 7693 (used for Merkle nodes).
 *
 * Where the pages leave a step open, the reading taken is stated at the function.
 *
 * Parity status: every exported function is pinned by a CPU test against something
 * other than itself (closed forms, hand-derived golden values, hashlib, exact
 * rationals, invariants); see the tests directory.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <float.h>

#define ORACLE_CHUNK 4096u          /* fixed chunk length for norm and hash leaves */

/* ------------------------------------------------------------------------------ */
/* Arithmetic model: IEEE binary32, round-to-nearest-even, one rounding per op, no  */
/* contraction, subnormals kept.  [OPEN-1B] §2.1 "Fused multiply-add": fusion is    */
/* disabled in the processor build.  The subnormal flush of §2.1 exists only to     */
/* match Apple GPUs; this oracle keeps IEEE gradual underflow (reading).            */
/* ------------------------------------------------------------------------------ */

/* Returns a*b+c exactly as written (two roundings).  Used by a test to prove the
 * library was built without contraction. */
float oracle_probe_mul_add(float a, float b, float c)
{
    float p = a * b;
    float s = p + c;
    return s;
}

/* 1 if subnormal arithmetic works in this thread (no FTZ/DAZ), else 0. */
int oracle_probe_subnormals(void)
{
    volatile float tiny = FLT_MIN;
    volatile float half = 0.5f;
    float s = tiny * half;          /* 2^-127: subnormal, exact */
    volatile float back = s * 2.0f; /* back to FLT_MIN if s was kept */
    return (s != 0.0f && back == FLT_MIN) ? 1 : 0;
}

/* Largest power of two strictly below L (L >= 2). */
static uint64_t split_point(uint64_t L)
{
    uint64_t k = 1;
    while (k * 2 < L) k *= 2;
    return k;
}

/* ------------------------------------------------------------------------------ */
/* Canonical tree T(x_0..x_{L-1}) for float addition.                               */
/* L == 1: x_0.  Otherwise k = largest power of two < L and                          */
/* T = T(x_0..x_{k-1}) + T(x_k..x_{L-1}), lower indices always the left operand.    */
/* [OPEN-1B] App. A.1 pairs replicas, pairs the pairs, and keeps the lower-replica  */
/* operand on the left; §5 splits a non-power-of-two count into its largest        */
/* power-of-two block and the rest.  For power-of-two L this is the perfect         */
/* pairwise tree, identical to the App. A.1 TreeFold.  For counts with three or     */
/* more set bits App. A.1's Result and this recursion group the leftover blocks     */
/* differently; the recursive split is the reading taken here.                      */
/* Empty input (L == 0) is the empty sum, +0.                                       */
/* ------------------------------------------------------------------------------ */
static float tree_sum_rec(const float *x, uint64_t L)
{
    if (L == 1) return x[0];
    uint64_t k = split_point(L);
    float left = tree_sum_rec(x, k);
    float right = tree_sum_rec(x + k, L - k);
    return left + right;
}

float oracle_tree_sum(const float *x, uint64_t L)
{
    if (L == 0) return 0.0f;
    return tree_sum_rec(x, L);
}

/* Widen a bfloat16 bit pattern to binary32 (exact: the 16 bits become the top half). */
static float bf16_to_f32(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* dtype codes: 0 = fp32 gradients, 1 = bf16 gradients (bit patterns). */
static float load_grad(const void *buf, int dtype, uint64_t i)
{
    if (dtype == 1) return bf16_to_f32(((const uint16_t *)buf)[i]);
    return ((const float *)buf)[i];
}

/* ------------------------------------------------------------------------------ */
/* Replica reduce.  g_i = T_{r<R}(G_r[i]) * fp32(1/R).                               */
/* Sum over replicas in the canonical tree over global replica index ([OPEN-1B]     */
/* App. A.1), then the average as a multiply by the fp32 reciprocal of R computed   */
/* once, never a division ([OPEN-1B] App. A.3).                                     */
/* grads: array of R pointers to n elements each, in global replica order.          */
/* Returns 0 on success, -1 on bad arguments.                                       */
/* ------------------------------------------------------------------------------ */
int oracle_reduce(const void *const *grads, int dtype, uint32_t R, uint64_t n, float *g)
{
    if (R == 0 || (dtype != 0 && dtype != 1)) return -1;
    float rho = 1.0f / (float)R;
    float *vals = (float *)malloc(sizeof(float) * R);
    if (!vals) return -1;
    for (uint64_t i = 0; i < n; ++i) {
        for (uint32_t r = 0; r < R; ++r) vals[r] = load_grad(grads[r], dtype, i);
        float s = tree_sum_rec(vals, R);
        g[i] = s * rho;
    }
    free(vals);
    return 0;
}

/* ------------------------------------------------------------------------------ */
/* Topology-staged replica reduce (a cluster of `nodes` nodes with `gpus_per_node`   */
/* replicas each, replica r = node * gpus_per_node + gpu).  Each node first sums its */
/* own replicas in the canonical tree; the node partials are then summed in the     */
/* canonical tree over node index; then the reciprocal multiply.  This is how a     */
/* two-level cluster reduction ([OPEN-1B] App. A: intra-node then inter-node) runs. */
/* It equals oracle_reduce bit for bit iff gpus_per_node is a power of two or       */
/* nodes == 1; other shapes are rejected (-2) because they would break the single   */
/* canonical order.                                                                  */
/* ------------------------------------------------------------------------------ */
int oracle_reduce_topology(const void *const *grads, int dtype, uint32_t nodes,
                           uint32_t gpus_per_node, uint64_t n, float *g)
{
    if (nodes == 0 || gpus_per_node == 0 || (dtype != 0 && dtype != 1)) return -1;
    if (nodes > 1 && (gpus_per_node & (gpus_per_node - 1)) != 0) return -2;
    uint32_t R = nodes * gpus_per_node;
    float rho = 1.0f / (float)R;
    float *inner = (float *)malloc(sizeof(float) * gpus_per_node);
    float *outer = (float *)malloc(sizeof(float) * nodes);
    if (!inner || !outer) { free(inner); free(outer); return -1; }
    for (uint64_t i = 0; i < n; ++i) {
        for (uint32_t nd = 0; nd < nodes; ++nd) {
            for (uint32_t q = 0; q < gpus_per_node; ++q)
                inner[q] = load_grad(grads[nd * gpus_per_node + q], dtype, i);
            outer[nd] = tree_sum_rec(inner, gpus_per_node);
        }
        float s = tree_sum_rec(outer, nodes);
        g[i] = s * rho;
    }
    free(inner);
    free(outer);
    return 0;
}

/* ------------------------------------------------------------------------------ */
/* Paper-exact reduction: [OPEN-1B] §6 Algorithm 1 with App. A.1-A.3.  The R inputs   */
/* are the gradients of the virtual ranks in mesh order r = rep * dp_shard + shard.  */
/* For each replica, its dp_shard shard gradients are summed in ascending shard     */
/* order (App. A.2: the deterministic reduce-scatter's local sum) and multiplied by  */
/* fp32(1/dp_shard) (App. A.3); the result is pushed into the TreeFold of App. A.1: */
/* a binary-carry stack of (level, partial) where equal levels combine with the      */
/* lower-replica partial on the left.  Result: the leftover blocks (one per set bit  */
/* of dp_replicate) are combined starting from the largest block, each later block   */
/* added on the right -- the reading that keeps both of App. A.1's stated rules      */
/* (largest block first; lower-replica block on the left), whose level wording       */
/* contradicts itself.  Finally g = Result * fp32(1/dp_replicate).                   */
/* ------------------------------------------------------------------------------ */
/* The gradient of virtual rank r at element i.  accum == 0: the rank's gradient as  */
/* given (one input per rank).  accum >= 1: [OPEN-1B] §6 Algorithm 1's microbatch    */
/* accumulation on a single device, taken literally -- g_r starts at +0 and each of  */
/* the rank's accum microbatch gradients (inputs r*accum .. r*accum + accum - 1, in  */
/* order) is added after multiplying by fp32(1/accum) (App. A.3: every average is a   */
/* reciprocal multiply).                                                             */
static float rank_grad(const void *const *grads, int dtype, uint32_t r, uint32_t accum,
                       float rho_acc, uint64_t i)
{
    if (accum == 0) return load_grad(grads[r], dtype, i);
    float gr = 0.0f;
    for (uint32_t k = 0; k < accum; ++k) {
        float term = load_grad(grads[(uint64_t)r * accum + k], dtype, i) * rho_acc;
        gr = gr + term;
    }
    return gr;
}

static int reduce_alg1(const void *const *grads, int dtype, uint32_t R, uint32_t dp_shard,
                       uint32_t accum, uint64_t n, float *g)
{
    if (R == 0 || dp_shard == 0 || R % dp_shard != 0 || (dtype != 0 && dtype != 1)) return -1;
    uint32_t dp_rep = R / dp_shard;
    float rho_shard = 1.0f / (float)dp_shard;
    float rho_rep = 1.0f / (float)dp_rep;
    float rho_acc = accum ? 1.0f / (float)accum : 1.0f;
    /* the stack: at most one entry per level, 64 levels is more than any R */
    float part[64];
    int level[64];
    for (uint64_t i = 0; i < n; ++i) {
        int depth = 0;
        float inner = 0.0f;
        for (uint32_t r = 0; r < R; ++r) {
            uint32_t shard = r % dp_shard;
            float x = rank_grad(grads, dtype, r, accum, rho_acc, i);
            if (shard == 0) inner = x;
            else inner = inner + x;
            if (shard == dp_shard - 1) {
                float p = inner * rho_shard;
                int lv = 0;
                while (depth > 0 && level[depth - 1] == lv) {
                    float lower = part[depth - 1];
                    --depth;
                    p = lower + p;        /* lower-replica operand on the left */
                    ++lv;
                }
                part[depth] = p;
                level[depth] = lv;
                ++depth;
            }
        }
        /* stack bottom = largest (earliest) block; left fold upward in the stack */
        float acc = part[0];
        for (int d = 1; d < depth; ++d) acc = acc + part[d];
        g[i] = acc * rho_rep;
    }
    return 0;
}

int oracle_reduce_alg1(const void *const *grads, int dtype, uint32_t R, uint32_t dp_shard,
                       uint64_t n, float *g)
{
    return reduce_alg1(grads, dtype, R, dp_shard, 0, n, g);
}

/* The same with the microbatch accumulation of Algorithm 1's inner loop: grads holds  */
/* R * accum microbatch gradients, rank-major (input r*accum + k is microbatch k of    */
/* virtual rank r).  accum >= 1.                                                     */
int oracle_reduce_alg1_accum(const void *const *grads, int dtype, uint32_t R, uint32_t dp_shard,
                             uint32_t accum, uint64_t n, float *g)
{
    if (accum == 0) return -1;
    return reduce_alg1(grads, dtype, R, dp_shard, accum, n, g);
}

/* ------------------------------------------------------------------------------ */
/* Global gradient norm over fixed 4096-element chunks.                              */
/* q_i = g_i * g_i; s_k = T(q over chunk k in index order); S = T(s_0..s_{c-1});     */
/* norm = sqrt(S).  Chunk k = [4096k, min(4096k + 4096, n)); the last chunk uses its */
/* true length.  [OPEN-1B] §3.2: gradients are clipped to a global l2 norm; §2.1:   */
/* one fixed reduction order on every backend.  The fixed chunking makes the bits   */
/* independent of any launch shape.                                                  */
/* chunk_sums (nullable) receives s_0..s_{c-1}.                                      */
/* ------------------------------------------------------------------------------ */
float oracle_norm(const float *g, uint64_t n, float *chunk_sums)
{
    uint64_t c = (n + ORACLE_CHUNK - 1) / ORACLE_CHUNK;
    if (c == 0) return 0.0f;
    float *s = (float *)malloc(sizeof(float) * c);
    float *q = (float *)malloc(sizeof(float) * ORACLE_CHUNK);
    if (!s || !q) { free(s); free(q); return NAN; }
    for (uint64_t k = 0; k < c; ++k) {
        uint64_t lo = k * ORACLE_CHUNK;
        uint64_t hi = lo + ORACLE_CHUNK < n ? lo + ORACLE_CHUNK : n;
        for (uint64_t i = lo; i < hi; ++i) q[i - lo] = g[i] * g[i];
        s[k] = tree_sum_rec(q, hi - lo);
        if (chunk_sums) chunk_sums[k] = s[k];
    }
    float S = tree_sum_rec(s, c);
    float norm = sqrtf(S);
    free(s);
    free(q);
    return norm;
}

/* ------------------------------------------------------------------------------ */
/* Clip scale.  [OPEN-1B] §3.2: clipped to a global l2 norm of 1.0.  The pages do   */
/* not give the formula; reading: scale = clip / norm when norm > clip, else 1.     */
/* A NaN norm compares false and gives scale 1.                                      */
/* ------------------------------------------------------------------------------ */
float oracle_clip_scale(float norm, float clip)
{
    if (norm > clip) return clip / norm;
    return 1.0f;
}

/* ------------------------------------------------------------------------------ */
/* Bias corrections.  p_j(0) = 1, p_j(t) = p_j(t-1) * beta_j in fp32, and           */
/* bc_j(t) = 1 - p_j(t).  [OPEN-1B] §3.2 uses AdamW (Loshchilov and Hutter); the    */
/* pages do not say how beta^t is formed; repeated fp32 products are the reading.  */
/* ------------------------------------------------------------------------------ */
void oracle_bias_corrections(float beta1, float beta2, int32_t t, float *bc1, float *bc2)
{
    float p1 = 1.0f, p2 = 1.0f;
    for (int32_t j = 0; j < t; ++j) {
        p1 = p1 * beta1;
        p2 = p2 * beta2;
    }
    *bc1 = 1.0f - p1;
    *bc2 = 1.0f - p2;
}

/* ------------------------------------------------------------------------------ */
/* AdamW with decoupled weight decay, one element at a time, in this fixed order:   */
/*   gc = g * scale                                                                  */
/*   m' = (beta1 * m) + ((1 - beta1) * gc)                                           */
/*   v' = (beta2 * v) + ((1 - beta2) * (gc * gc))                                    */
/*   mhat = m' / bc1 ;  vhat = v' / bc2                                              */
/*   u = mhat / (sqrt(vhat) + eps)                                                   */
/*   w' = (w * (1 - lr * wd)) - (lr * u)                                             */
/* [OPEN-1B] §3.2 (AdamW, decoupled weight decay 0.1) and "Optimizer-state          */
/* precision" (entire moment and parameter update in FP32); [CKPT] (m is the EMA of */
/* gradients with beta1, v of squared gradients with beta2).  The op order, the     */
/* bias-correction form and where the decay is applied are not on the pages; this   */
/* is the textbook Adam moment form with the decay as a multiply by (1 - lr*wd).    */
/* The three constants 1-beta1, 1-beta2 and 1-lr*wd are each rounded to fp32 once.  */
/* ------------------------------------------------------------------------------ */
void oracle_adamw(float *w, float *m, float *v, const float *g, uint64_t n, float scale,
                  float lr, float beta1, float beta2, float eps, float wd,
                  float bc1, float bc2)
{
    float omega1 = 1.0f - beta1;
    float omega2 = 1.0f - beta2;
    float lrwd = lr * wd;
    float delta = 1.0f - lrwd;
    for (uint64_t i = 0; i < n; ++i) {
        float gc = g[i] * scale;
        float m_old = beta1 * m[i];
        float m_new_term = omega1 * gc;
        float m_new = m_old + m_new_term;
        float gsq = gc * gc;
        float v_old = beta2 * v[i];
        float v_new_term = omega2 * gsq;
        float v_new = v_old + v_new_term;
        float mhat = m_new / bc1;
        float vhat = v_new / bc2;
        float root = sqrtf(vhat);
        float denom = root + eps;
        float u = mhat / denom;
        float w_decayed = w[i] * delta;
        float step = lr * u;
        w[i] = w_decayed - step;
        m[i] = m_new;
        v[i] = v_new;
    }
}

/* ------------------------------------------------------------------------------ */
/* bf16 parameters ([OPEN-1B] §3.2, paragraph on optimizer-state precision: the      */
/* parameters are held in BF16, the fused optimizer step widens parameter and        */
/* gradient to FP32, does the whole moment and parameter update in FP32, and rounds  */
/* the result back to BF16 once per step; m and v stay FP32).                         */
/* Rounding fp32 -> bf16 to nearest, ties to even, on the bit pattern: keep the top   */
/* 16 bits after adding half of the dropped range plus the kept lowest bit.  NaN      */
/* stays a NaN (its payload is outside the contract).                                */
/* ------------------------------------------------------------------------------ */
uint16_t oracle_f32_to_bf16(float x)
{
    uint32_t u;
    memcpy(&u, &x, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u);          /* quiet NaN */
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

/* AdamW with bf16 parameters: w16 in place, m and v fp32; the update of oracle_adamw  */
/* on the widened parameter, rounded once back to bf16.                               */
void oracle_adamw_bf16w(uint16_t *w16, float *m, float *v, const float *g, uint64_t n,
                        float scale, float lr, float beta1, float beta2, float eps, float wd,
                        float bc1, float bc2)
{
    for (uint64_t i = 0; i < n; ++i) {
        float w32 = bf16_to_f32(w16[i]);
        oracle_adamw(&w32, m + i, v + i, g + i, 1, scale, lr, beta1, beta2, eps, wd, bc1, bc2);
        w16[i] = oracle_f32_to_bf16(w32);
    }
}

/* ------------------------------------------------------------------------------ */
/* Per-segment weight decay ([OPEN-1B] §3.2, optimizer paragraph: no weight decay on  */
/* the embeddings, the normalisation gains or RoPE).  The flat parameter vector is   */
/* cut into `count` segments: segment s covers [seg_begin[s], seg_begin[s+1]), the   */
/* last one ends at n; seg_begin[0] is 0 and the starts increase strictly.  An       */
/* element of a segment with decay[s] != 0 takes the update with weight decay wd,    */
/* any other element the same update with weight decay 0.                            */
/* Returns 0, or -1 on a bad segment list.                                           */
/* ------------------------------------------------------------------------------ */
static int segments_ok(uint64_t n, const uint64_t *seg_begin, uint32_t count)
{
    if (count == 0) return n == 0;
    if (seg_begin[0] != 0) return 0;
    for (uint32_t s = 1; s < count; ++s)
        if (seg_begin[s] <= seg_begin[s - 1] || seg_begin[s] >= n) return 0;
    return 1;
}

static float segment_wd(uint64_t i, const uint64_t *seg_begin, const uint8_t *decay,
                        uint32_t count, float wd)
{
    uint32_t s = 0;
    while (s + 1 < count && seg_begin[s + 1] <= i) ++s;
    return decay[s] ? wd : 0.0f;
}

int oracle_adamw_segments(float *w, float *m, float *v, const float *g, uint64_t n, float scale,
                          float lr, float beta1, float beta2, float eps, float wd, float bc1,
                          float bc2, const uint64_t *seg_begin, const uint8_t *decay,
                          uint32_t count)
{
    if (!segments_ok(n, seg_begin, count)) return -1;
    for (uint64_t i = 0; i < n; ++i)
        oracle_adamw(w + i, m + i, v + i, g + i, 1, scale, lr, beta1, beta2, eps,
                     segment_wd(i, seg_begin, decay, count, wd), bc1, bc2);
    return 0;
}

int oracle_adamw_bf16w_segments(uint16_t *w16, float *m, float *v, const float *g, uint64_t n,
                                float scale, float lr, float beta1, float beta2, float eps,
                                float wd, float bc1, float bc2, const uint64_t *seg_begin,
                                const uint8_t *decay, uint32_t count)
{
    if (!segments_ok(n, seg_begin, count)) return -1;
    for (uint64_t i = 0; i < n; ++i)
        oracle_adamw_bf16w(w16 + i, m + i, v + i, g + i, 1, scale, lr, beta1, beta2, eps,
                           segment_wd(i, seg_begin, decay, count, wd), bc1, bc2);
    return 0;
}

/* ------------------------------------------------------------------------------ */
/* Software flush-to-zero mode ([OPEN-1B] §2.1 "Subnormals": two modes discard       */
/* subnormals -- FTZ zeroes a subnormal result, DAZ a subnormal input -- and RepOps  */
/* applies both on every backend to match the least permissive one).  Readings:     */
/*   - every fp32 operation of the step flushes its operands and its result;        */
/*   - a flushed value becomes a zero of the same sign;                              */
/*   - "subnormal result" means a tiny result in IEEE 754's sense with tininess      */
/*     detected after rounding (IEEE 754-2008 §7.5): the exact result, rounded to    */
/*     24 significant bits as though the exponent range were unbounded, is nonzero   */
/*     and below 2^-126 in magnitude.  Such a result is zeroed; every other result   */
/*     is the IEEE result.  So a product whose exact value lies just below 2^-126    */
/*     but rounds (unbounded) to 2^-126 is kept, and one that rounds (unbounded) to  */
/*     2^-126 - 2^-150 is zeroed although the binary32 rounding would give 2^-126;   */
/*   - a sum or difference below 2^-126 is exact (both operands are multiples of     */
/*     2^-149), and a square root of a normal value is normal, so for these the rule */
/*     is the plain flush of the IEEE result;                                       */
/*   - the rounding of a bf16 parameter is an operation too, but its input is then  */
/*     zero or at least the smallest normal, so it never yields a subnormal.          */
/* The functions below repeat the IEEE-mode definitions above with every operation  */
/* written through these helpers, in the same order.                                */
/* ------------------------------------------------------------------------------ */
static float flush(float x)
{
    if (fpclassify(x) == FP_SUBNORMAL) return copysignf(0.0f, x);
    return x;
}

/* Tininess of a product or quotient r = IEEE(a op b) of two flushed operands.  Only
   |r| <= 2^-126 can be tiny.  Then a is at most about 4 in magnitude (b is zero or
   at least 2^-126 for a product; the quotient is at most 2^-126 for a division), so
   a * 2^64 is exact and the same operation on it rounds the exact result times 2^64
   to 24 bits in the normal range -- the unbounded-exponent rounding, scaled.  The
   result is tiny when that is below 2^-62.  (Exact results below 2^-190 leave the
   scaled rounding subnormal or zero, and are tiny either way.) */
static float fz_mul(float a, float b)
{
    a = flush(a);
    b = flush(b);
    float r = a * b;
    if (!(fabsf(r) <= 0x1p-126f)) return r;          /* normal, infinite or NaN */
    float s = (a * 0x1p64f) * b;
    return fabsf(s) < 0x1p-62f ? copysignf(0.0f, r) : r;
}

static float fz_div(float a, float b)
{
    a = flush(a);
    b = flush(b);
    float r = a / b;
    if (!(fabsf(r) <= 0x1p-126f)) return r;
    float s = (a * 0x1p64f) / b;
    return fabsf(s) < 0x1p-62f ? copysignf(0.0f, r) : r;
}

static float fz_add(float a, float b) { return flush(flush(a) + flush(b)); }
static float fz_sub(float a, float b) { return flush(flush(a) - flush(b)); }
static float fz_sqrt(float a) { return flush(sqrtf(flush(a))); }

float oracle_flush(float x) { return flush(x); }
float oracle_mul_ftz(float a, float b) { return fz_mul(a, b); }
float oracle_div_ftz(float a, float b) { return fz_div(a, b); }

static float fz_tree_sum_rec(const float *x, uint64_t L)
{
    if (L == 1) return flush(x[0]);
    uint64_t k = split_point(L);
    float left = fz_tree_sum_rec(x, k);
    float right = fz_tree_sum_rec(x + k, L - k);
    return fz_add(left, right);
}

float oracle_tree_sum_ftz(const float *x, uint64_t L)
{
    if (L == 0) return 0.0f;
    return fz_tree_sum_rec(x, L);
}

/* Replica reduce in FTZ mode: g_i = T_{r<R}(G_r[i]) * fp32(1/R), every op flushed.   */
int oracle_reduce_ftz(const void *const *grads, int dtype, uint32_t R, uint64_t n, float *g)
{
    if (R == 0 || (dtype != 0 && dtype != 1)) return -1;
    float rho = fz_div(1.0f, (float)R);
    float *vals = (float *)malloc(sizeof(float) * R);
    if (!vals) return -1;
    for (uint64_t i = 0; i < n; ++i) {
        for (uint32_t r = 0; r < R; ++r) vals[r] = load_grad(grads[r], dtype, i);
        g[i] = fz_mul(fz_tree_sum_rec(vals, R), rho);
    }
    free(vals);
    return 0;
}

/* Paper-exact reduction (Algorithm 1, accum 0 = rank gradients given) in FTZ mode. */
int oracle_reduce_alg1_ftz(const void *const *grads, int dtype, uint32_t R, uint32_t dp_shard,
                           uint32_t accum, uint64_t n, float *g)
{
    if (R == 0 || dp_shard == 0 || R % dp_shard != 0 || (dtype != 0 && dtype != 1)) return -1;
    uint32_t dp_rep = R / dp_shard;
    float rho_shard = fz_div(1.0f, (float)dp_shard);
    float rho_rep = fz_div(1.0f, (float)dp_rep);
    float rho_acc = accum ? fz_div(1.0f, (float)accum) : 1.0f;
    float part[64];
    int level[64];
    for (uint64_t i = 0; i < n; ++i) {
        int depth = 0;
        float inner = 0.0f;
        for (uint32_t r = 0; r < R; ++r) {
            uint32_t shard = r % dp_shard;
            float x;
            if (accum == 0) {
                x = flush(load_grad(grads[r], dtype, i));
            } else {
                x = 0.0f;
                for (uint32_t k = 0; k < accum; ++k)
                    x = fz_add(x, fz_mul(load_grad(grads[(uint64_t)r * accum + k], dtype, i),
                                         rho_acc));
            }
            if (shard == 0) inner = x;
            else inner = fz_add(inner, x);
            if (shard == dp_shard - 1) {
                float p = fz_mul(inner, rho_shard);
                int lv = 0;
                while (depth > 0 && level[depth - 1] == lv) {
                    float lower = part[depth - 1];
                    --depth;
                    p = fz_add(lower, p);
                    ++lv;
                }
                part[depth] = p;
                level[depth] = lv;
                ++depth;
            }
        }
        float acc = part[0];
        for (int d = 1; d < depth; ++d) acc = fz_add(acc, part[d]);
        g[i] = fz_mul(acc, rho_rep);
    }
    return 0;
}

/* Global norm in FTZ mode: squares, chunk trees, the tree over chunks, sqrt.         */
float oracle_norm_ftz(const float *g, uint64_t n, float *chunk_sums)
{
    uint64_t c = (n + ORACLE_CHUNK - 1) / ORACLE_CHUNK;
    if (c == 0) return 0.0f;
    float *s = (float *)malloc(sizeof(float) * c);
    float *q = (float *)malloc(sizeof(float) * ORACLE_CHUNK);
    if (!s || !q) { free(s); free(q); return NAN; }
    for (uint64_t k = 0; k < c; ++k) {
        uint64_t lo = k * ORACLE_CHUNK;
        uint64_t hi = lo + ORACLE_CHUNK < n ? lo + ORACLE_CHUNK : n;
        for (uint64_t i = lo; i < hi; ++i) q[i - lo] = fz_mul(g[i], g[i]);
        s[k] = fz_tree_sum_rec(q, hi - lo);
        if (chunk_sums) chunk_sums[k] = s[k];
    }
    float norm = fz_sqrt(fz_tree_sum_rec(s, c));
    free(s);
    free(q);
    return norm;
}

float oracle_clip_scale_ftz(float norm, float clip)
{
    if (flush(norm) > flush(clip)) return fz_div(clip, norm);
    return 1.0f;
}

void oracle_bias_corrections_ftz(float beta1, float beta2, int32_t t, float *bc1, float *bc2)
{
    float p1 = 1.0f, p2 = 1.0f;
    for (int32_t j = 0; j < t; ++j) {
        p1 = fz_mul(p1, beta1);
        p2 = fz_mul(p2, beta2);
    }
    *bc1 = fz_sub(1.0f, p1);
    *bc2 = fz_sub(1.0f, p2);
}

/* AdamW in FTZ mode, same op order as oracle_adamw; w is fp32 (w_bf16 == 0) or bf16  */
/* bit patterns (widened, updated, rounded once to nearest even); optional            */
/* decay segments as in oracle_adamw_segments (count 0: every element decays).       */
int oracle_adamw_ftz(void *w, int w_bf16, float *m, float *v, const float *g, uint64_t n,
                     float scale, float lr, float beta1, float beta2, float eps, float wd,
                     float bc1, float bc2, const uint64_t *seg_begin, const uint8_t *decay,
                     uint32_t count)
{
    if (count > 0 && !segments_ok(n, seg_begin, count)) return -1;
    float omega1 = fz_sub(1.0f, beta1);
    float omega2 = fz_sub(1.0f, beta2);
    for (uint64_t i = 0; i < n; ++i) {
        float wd_i = count > 0 ? segment_wd(i, seg_begin, decay, count, wd) : wd;
        float delta = fz_sub(1.0f, fz_mul(lr, wd_i));
        float wi = w_bf16 ? bf16_to_f32(((uint16_t *)w)[i]) : ((float *)w)[i];
        float gc = fz_mul(g[i], scale);
        float m_new = fz_add(fz_mul(beta1, m[i]), fz_mul(omega1, gc));
        float v_new = fz_add(fz_mul(beta2, v[i]), fz_mul(omega2, fz_mul(gc, gc)));
        float mhat = fz_div(m_new, bc1);
        float vhat = fz_div(v_new, bc2);
        float u = fz_div(mhat, fz_add(fz_sqrt(vhat), eps));
        float w_new = fz_sub(fz_mul(wi, delta), fz_mul(lr, u));
        if (w_bf16) {
            /* w_new is zero or at least 2^-126 in magnitude, a bf16 value itself, so the
               rounding cannot produce a bf16 subnormal and needs no flush */
            ((uint16_t *)w)[i] = oracle_f32_to_bf16(w_new);
        } else {
            ((float *)w)[i] = w_new;
        }
        m[i] = m_new;
        v[i] = v_new;
    }
    return 0;
}

/* ------------------------------------------------------------------------------ */
/* PF61 leaf digest over a sequence of 32-bit words:                                 */
/*   F(x_0..x_{W-1}) = (W + sum_{i<W} x_i * K^(i+1)) mod p,  p = 2^61 - 1,          */
/*   K = (isqrt(5 * 2^122) - 2^61) >> 1 (floor of 2^61 (sqrt5 - 1)/2).               */
/* [OPEN-1B] App. B anchors every step with a canonical hash of parameters and      */
/* optimizer state; the pages do not fix the leaf function.  Reading: a polynomial  */
/* fingerprint modulo a Mersenne prime, whose per-word terms can be summed in any   */
/* order, so a parallel kernel reproduces it exactly.                                */
/* ------------------------------------------------------------------------------ */
#define PF61_P ((uint64_t)0x1FFFFFFFFFFFFFFFull)
#define PF61_K ((uint64_t)0x13C6EF372FE94F82ull)

uint64_t oracle_pf61_constant(void) { return PF61_K; }

static uint64_t mod61(unsigned __int128 x)
{
    /* 2^61 == 1 (mod p): fold 61-bit digits until below p. */
    while (x >> 61) x = (x & PF61_P) + (x >> 61);
    uint64_t r = (uint64_t)x;
    if (r >= PF61_P) r -= PF61_P;
    return r;
}

static uint64_t mulmod61(uint64_t a, uint64_t b)
{
    return mod61((unsigned __int128)a * (unsigned __int128)b);
}

uint64_t oracle_pf61(const uint32_t *x, uint64_t W)
{
    uint64_t acc = mod61((unsigned __int128)W);
    uint64_t power = PF61_K;                 /* K^(i+1) for i = 0 */
    for (uint64_t i = 0; i < W; ++i) {
        uint64_t term = mulmod61((uint64_t)x[i], power);
        acc = mod61((unsigned __int128)acc + term);
        power = mulmod61(power, PF61_K);
    }
    return acc;
}

/* ------------------------------------------------------------------------------ */
/* BLAKE2b, written from RFC 7693 (sections 2 and 3): 12 rounds of the G mixing      */
/* function over a 16-word state, 128-byte blocks, little-endian words.  No key.    */
/* ------------------------------------------------------------------------------ */
static const uint64_t B2_IV[8] = {
    0x6A09E667F3BCC908ull, 0xBB67AE8584CAA73Bull, 0x3C6EF372FE94F82Bull, 0xA54FF53A5F1D36F1ull,
    0x510E527FADE682D1ull, 0x9B05688C2B3E6C1Full, 0x1F83D9ABFB41BD6Bull, 0x5BE0CD19137E2179ull,
};

static const uint8_t B2_SIGMA[12][16] = {
    { 0, 1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12, 13, 14, 15 },
    { 14, 10, 4, 8, 9, 15, 13, 6, 1, 12, 0, 2, 11, 7, 5, 3 },
    { 11, 8, 12, 0, 5, 2, 15, 13, 10, 14, 3, 6, 7, 1, 9, 4 },
    { 7, 9, 3, 1, 13, 12, 11, 14, 2, 6, 5, 10, 4, 0, 15, 8 },
    { 9, 0, 5, 7, 2, 4, 10, 15, 14, 1, 11, 12, 6, 8, 3, 13 },
    { 2, 12, 6, 10, 0, 11, 8, 3, 4, 13, 7, 5, 15, 14, 1, 9 },
    { 12, 5, 1, 15, 14, 13, 4, 10, 0, 7, 6, 3, 9, 2, 8, 11 },
    { 13, 11, 7, 14, 12, 1, 3, 9, 5, 0, 15, 4, 8, 6, 2, 10 },
    { 6, 15, 14, 9, 11, 3, 0, 8, 12, 2, 13, 7, 1, 4, 10, 5 },
    { 10, 2, 8, 4, 7, 6, 1, 5, 15, 11, 9, 14, 3, 12, 13, 0 },
    { 0, 1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12, 13, 14, 15 },
    { 14, 10, 4, 8, 9, 15, 13, 6, 1, 12, 0, 2, 11, 7, 5, 3 },
};

static uint64_t rotr64(uint64_t x, unsigned s) { return (x >> s) | (x << (64 - s)); }

static uint64_t load64_le(const uint8_t *p)
{
    uint64_t v = 0;
    for (int i = 7; i >= 0; --i) v = (v << 8) | p[i];
    return v;
}

static void b2_mix(uint64_t v[16], int a, int b, int c, int d, uint64_t x, uint64_t y)
{
    v[a] = v[a] + v[b] + x;
    v[d] = rotr64(v[d] ^ v[a], 32);
    v[c] = v[c] + v[d];
    v[b] = rotr64(v[b] ^ v[c], 24);
    v[a] = v[a] + v[b] + y;
    v[d] = rotr64(v[d] ^ v[a], 16);
    v[c] = v[c] + v[d];
    v[b] = rotr64(v[b] ^ v[c], 63);
}

static void b2_compress(uint64_t h[8], const uint8_t block[128], uint64_t t_lo, uint64_t t_hi,
                        int last)
{
    uint64_t v[16], m[16];
    for (int i = 0; i < 16; ++i) m[i] = load64_le(block + 8 * i);
    for (int i = 0; i < 8; ++i) { v[i] = h[i]; v[i + 8] = B2_IV[i]; }
    v[12] ^= t_lo;
    v[13] ^= t_hi;
    if (last) v[14] = ~v[14];
    for (int r = 0; r < 12; ++r) {
        const uint8_t *s = B2_SIGMA[r];
        b2_mix(v, 0, 4, 8, 12, m[s[0]], m[s[1]]);
        b2_mix(v, 1, 5, 9, 13, m[s[2]], m[s[3]]);
        b2_mix(v, 2, 6, 10, 14, m[s[4]], m[s[5]]);
        b2_mix(v, 3, 7, 11, 15, m[s[6]], m[s[7]]);
        b2_mix(v, 0, 5, 10, 15, m[s[8]], m[s[9]]);
        b2_mix(v, 1, 6, 11, 12, m[s[10]], m[s[11]]);
        b2_mix(v, 2, 7, 8, 13, m[s[12]], m[s[13]]);
        b2_mix(v, 3, 4, 9, 14, m[s[14]], m[s[15]]);
    }
    for (int i = 0; i < 8; ++i) h[i] ^= v[i] ^ v[i + 8];
}

/* Unkeyed BLAKE2b of `len` bytes into `outlen` (1..64) bytes.  Returns 0 or -1. */
int oracle_blake2b(const uint8_t *in, uint64_t len, uint8_t *out, uint32_t outlen)
{
    if (outlen == 0 || outlen > 64) return -1;
    uint64_t h[8];
    for (int i = 0; i < 8; ++i) h[i] = B2_IV[i];
    h[0] ^= 0x01010000ull ^ (uint64_t)outlen;
    uint8_t block[128];
    uint64_t done = 0;
    /* every full block except the last one */
    while (len - done > 128) {
        memcpy(block, in + done, 128);
        done += 128;
        b2_compress(h, block, done, 0, 0);
    }
    /* final block (possibly empty), zero padded */
    memset(block, 0, sizeof block);
    memcpy(block, in + done, (size_t)(len - done));
    b2_compress(h, block, len, 0, 1);
    for (uint32_t i = 0; i < outlen; ++i) out[i] = (uint8_t)(h[i / 8] >> (8 * (i % 8)));
    return 0;
}

/* Merkle node: N(a, b) = LE-u64 of BLAKE2b-64(LE64(a) || LE64(b)).  The pages hash  */
/* with blake2b on the host ([OPEN-1B] App. B, Figure 11); here it combines digests. */
uint64_t oracle_node(uint64_t a, uint64_t b)
{
    uint8_t msg[16], out[8];
    for (int i = 0; i < 8; ++i) {
        msg[i] = (uint8_t)(a >> (8 * i));
        msg[8 + i] = (uint8_t)(b >> (8 * i));
    }
    oracle_blake2b(msg, 16, out, 8);
    uint64_t r = 0;
    for (int i = 7; i >= 0; --i) r = (r << 8) | out[i];
    return r;
}

/* Merkle root: the canonical tree (same recursive split as oracle_tree_sum) over the */
/* leaf digests with node function N, lower index on the left.  L >= 1.              */
static uint64_t merkle_rec(const uint64_t *x, uint64_t L)
{
    if (L == 1) return x[0];
    uint64_t k = split_point(L);
    uint64_t left = merkle_rec(x, k);
    uint64_t right = merkle_rec(x + k, L - k);
    return oracle_node(left, right);
}

uint64_t oracle_merkle_root(const uint64_t *leaves, uint64_t L)
{
    if (L == 0) return 0;
    return merkle_rec(leaves, L);
}

/* ------------------------------------------------------------------------------ */
/* Checkpoint image and its leaves.                                                  */
/* [CKPT] Format: [int32 step][int32 n_params][n x f32 w][n x f32 m][n x f32 v],     */
/* total 8 + 12 n bytes ([OLMO12] Table 27: ~12P).  Little-endian.  n is stored as   */
/* the same 32 bits read unsigned (reading: the pages' int32 cannot hold n >= 2^31). */
/* Leaves in layout order: the 8-byte header (2 words), then the 4096-element chunks */
/* of w, then of m, then of v (last chunk of each short).  L = 1 + 3c.               */
/* ------------------------------------------------------------------------------ */
uint64_t oracle_image_bytes(uint64_t n) { return 8 + 12 * n; }

int oracle_image(int32_t step, uint64_t n, const float *w, const float *m, const float *v,
                 uint8_t *out)
{
    if (n > 0xFFFFFFFFull) return -1;
    uint32_t s = (uint32_t)step, nn = (uint32_t)n;
    for (int i = 0; i < 4; ++i) {
        out[i] = (uint8_t)(s >> (8 * i));
        out[4 + i] = (uint8_t)(nn >> (8 * i));
    }
    const float *arrs[3] = { w, m, v };
    uint64_t off = 8;
    for (int a = 0; a < 3; ++a) {
        for (uint64_t i = 0; i < n; ++i) {
            uint32_t u;
            memcpy(&u, &arrs[a][i], 4);
            for (int b = 0; b < 4; ++b) out[off + 4 * i + b] = (uint8_t)(u >> (8 * b));
        }
        off += 4 * n;
    }
    return 0;
}

uint64_t oracle_num_leaves(uint64_t n) { return 1 + 3 * ((n + ORACLE_CHUNK - 1) / ORACLE_CHUNK); }

int oracle_leaves(int32_t step, uint64_t n, const float *w, const float *m, const float *v,
                  uint64_t *leaves)
{
    if (n > 0xFFFFFFFFull) return -1;
    uint64_t c = (n + ORACLE_CHUNK - 1) / ORACLE_CHUNK;
    uint32_t header[2] = { (uint32_t)step, (uint32_t)n };
    leaves[0] = oracle_pf61(header, 2);
    const float *arrs[3] = { w, m, v };
    uint32_t *words = (uint32_t *)malloc(sizeof(uint32_t) * ORACLE_CHUNK);
    if (!words) return -1;
    for (int a = 0; a < 3; ++a) {
        for (uint64_t k = 0; k < c; ++k) {
            uint64_t lo = k * ORACLE_CHUNK;
            uint64_t hi = lo + ORACLE_CHUNK < n ? lo + ORACLE_CHUNK : n;
            memcpy(words, arrs[a] + lo, sizeof(uint32_t) * (size_t)(hi - lo));
            leaves[1 + (uint64_t)a * c + k] = oracle_pf61(words, hi - lo);
        }
    }
    free(words);
    return 0;
}

/* ------------------------------------------------------------------------------ */
/* Audit-mode leaves: each leaf is BLAKE2b-64 of its bytes in the image -- the      */
/* 8-byte header, then each 4096-element chunk of w, of m, of v as little-endian     */
/* fp32 (the last chunk short).  [OPEN-1B] App. B hashes every step with host       */
/* blake2b; this mode uses that function for the leaves as well as the nodes.       */
/* hash_mode 0 = PF61 leaves (oracle_leaves), 1 = BLAKE2b-64 leaves.                */
/* ------------------------------------------------------------------------------ */
static uint64_t b2_64(const uint8_t *bytes, uint64_t len)
{
    uint8_t out[8];
    oracle_blake2b(bytes, len, out, 8);
    uint64_t r = 0;
    for (int i = 7; i >= 0; --i) r = (r << 8) | out[i];
    return r;
}

int oracle_leaves_mode(int32_t step, uint64_t n, const float *w, const float *m, const float *v,
                       int hash_mode, uint64_t *leaves)
{
    if (hash_mode == 0) return oracle_leaves(step, n, w, m, v, leaves);
    if (hash_mode != 1 || n > 0xFFFFFFFFull) return -1;
    uint64_t c = (n + ORACLE_CHUNK - 1) / ORACLE_CHUNK;
    uint8_t header[8];
    uint32_t s = (uint32_t)step, nn = (uint32_t)n;
    for (int i = 0; i < 4; ++i) {
        header[i] = (uint8_t)(s >> (8 * i));
        header[4 + i] = (uint8_t)(nn >> (8 * i));
    }
    leaves[0] = b2_64(header, 8);
    const float *arrs[3] = { w, m, v };
    uint8_t *buf = (uint8_t *)malloc(4 * ORACLE_CHUNK);
    if (!buf) return -1;
    for (int a = 0; a < 3; ++a) {
        for (uint64_t k = 0; k < c; ++k) {
            uint64_t lo = k * ORACLE_CHUNK;
            uint64_t hi = lo + ORACLE_CHUNK < n ? lo + ORACLE_CHUNK : n;
            for (uint64_t i = lo; i < hi; ++i) {
                uint32_t u;
                memcpy(&u, &arrs[a][i], 4);
                for (int b = 0; b < 4; ++b) buf[4 * (i - lo) + b] = (uint8_t)(u >> (8 * b));
            }
            leaves[1 + (uint64_t)a * c + k] = b2_64(buf, 4 * (hi - lo));
        }
    }
    free(buf);
    return 0;
}

int oracle_state_hash_mode(int32_t step, uint64_t n, const float *w, const float *m,
                           const float *v, int hash_mode, uint64_t *root)
{
    uint64_t L = oracle_num_leaves(n);
    uint64_t *leaves = (uint64_t *)malloc(sizeof(uint64_t) * L);
    if (!leaves) return -1;
    if (oracle_leaves_mode(step, n, w, m, v, hash_mode, leaves) != 0) { free(leaves); return -1; }
    *root = oracle_merkle_root(leaves, L);
    free(leaves);
    return 0;
}

/* State hash of (step, w, m, v): the Merkle root over oracle_leaves. */
int oracle_state_hash(int32_t step, uint64_t n, const float *w, const float *m, const float *v,
                      uint64_t *root)
{
    uint64_t L = oracle_num_leaves(n);
    uint64_t *leaves = (uint64_t *)malloc(sizeof(uint64_t) * L);
    if (!leaves) return -1;
    if (oracle_leaves(step, n, w, m, v, leaves) != 0) { free(leaves); return -1; }
    *root = oracle_merkle_root(leaves, L);
    free(leaves);
    return 0;
}

/* ------------------------------------------------------------------------------ */
/* One full optimizer step: reduce -> norm -> clip scale -> AdamW -> state hash.     */
/* w, m, v are updated in place; the image header carries step t after the update.  */
/* nodes/gpus_per_node select the staged reduction (nodes == 1: flat).              */
/* Outputs: pre-clip norm ([OPEN-1B] §3.4.2 logs the pre-clip norm), clip scale and  */
/* Merkle root.  Returns 0, -1 (bad argument) or -2 (unsupported topology).          */
/* ------------------------------------------------------------------------------ */
int oracle_step_mode(const void *const *grads, int dtype, uint32_t nodes, uint32_t gpus_per_node,
                     uint64_t n, float *w, float *m, float *v,
                     float lr, float beta1, float beta2, float eps, float wd, float clip,
                     int32_t t, int hash_mode, float *norm_out, float *scale_out,
                     uint64_t *root_out);

int oracle_step(const void *const *grads, int dtype, uint32_t nodes, uint32_t gpus_per_node,
                uint64_t n, float *w, float *m, float *v,
                float lr, float beta1, float beta2, float eps, float wd, float clip,
                int32_t t, float *norm_out, float *scale_out, uint64_t *root_out)
{
    return oracle_step_mode(grads, dtype, nodes, gpus_per_node, n, w, m, v, lr, beta1, beta2,
                            eps, wd, clip, t, 0, norm_out, scale_out, root_out);
}

int oracle_step_mode(const void *const *grads, int dtype, uint32_t nodes, uint32_t gpus_per_node,
                     uint64_t n, float *w, float *m, float *v,
                     float lr, float beta1, float beta2, float eps, float wd, float clip,
                     int32_t t, int hash_mode, float *norm_out, float *scale_out,
                     uint64_t *root_out)
{
    float *g = (float *)malloc(sizeof(float) * (n ? n : 1));
    if (!g) return -1;
    int rc = oracle_reduce_topology(grads, dtype, nodes, gpus_per_node, n, g);
    if (rc != 0) { free(g); return rc; }
    float norm = oracle_norm(g, n, NULL);
    float scale = oracle_clip_scale(norm, clip);
    float bc1, bc2;
    oracle_bias_corrections(beta1, beta2, t, &bc1, &bc2);
    oracle_adamw(w, m, v, g, n, scale, lr, beta1, beta2, eps, wd, bc1, bc2);
    free(g);
    if (norm_out) *norm_out = norm;
    if (scale_out) *scale_out = scale;
    if (root_out) return oracle_state_hash_mode(t, n, w, m, v, hash_mode, root_out);
    return 0;
}
