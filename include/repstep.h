/*
 * repstep.h -- C ABI of the bitwise-reproducible optimizer step for one GB300 (sm_103a).
 *
 * One optimizer step is: sum R replica gradients in one canonical tree and average them by
 * a reciprocal multiply; compute the global l2 norm over fixed 4096-element chunks; clip;
 * apply AdamW to flat weights (fp32, or bf16 updated in fp32) and fp32 Adam moments; hash
 * the checkpoint image [int32 step][uint32 n][w][m][v] with per-chunk digests combined in
 * a Merkle tree.  Every output bit is fixed by the definition below, independent of the
 * launch configuration, of how replicas are grouped into nodes, and of how the parameter
 * range is split.  Options: per-segment weight decay, a flush-to-zero mode, the
 * paper-exact reduction order of OPEN-1B's audit replay, and the hash on a second stream.
 *
 * Sources, by page title and section:
 *   "OPEN-1B: A Fully Auditable Training Run" (Gensyn): §2.1 Reproducible Operations
 *     (one fixed reduction order, no implicit fused multiply-add); §3.2 Training Recipe
 *     (AdamW, decoupled weight decay, global-norm clipping at 1.0); §3.4.2 (pre-clip
 *     gradient norm); App. A (deterministic gradient reduction: TreeFold over replicas
 *     with the lower replica on the left, reduce-scatter over shards, App. A.3 average
 *     via reciprocal multiply); App. B (per-step state hash).
 *   "grow_a_language_model_checkpoints": Format and Total size (8 + 12 n bytes).
 *   OLMo-core MoE §12 "Topology-agnostic checkpoint saving and loading" (FP32 weights and
 *     both moments, canonical element order independent of topology).
 *
 * Definitions (every fp32 operation is IEEE binary32 round-to-nearest-even, rounded once,
 * never contracted into a fused multiply-add; subnormals are kept, unless the context's
 * subnormal mode is REPSTEP_SUBNORMALS_FTZ, which flushes every operand and result):
 *   T(x_0..x_{L-1})  canonical tree: x_0 if L == 1, else T(x_0..x_{k-1}) + T(x_k..x_{L-1})
 *                    with k the largest power of two below L; lower indices on the left.
 *   reduce           g_i = T_{r<R}(G_r[i]) * fp32(1/R); bf16 gradients widened exactly.
 *   norm             s_k = T(g_i*g_i over chunk k = [4096k, min(4096k+4096, n)));
 *                    S = T(s_0..s_{c-1}), c = ceil(n/4096); norm = sqrt(S)  (pre-clip).
 *   clip             scale = norm > clip ? clip / norm : 1.
 *   AdamW            gc = g*scale; m' = b1*m + (1-b1)*gc; v' = b2*v + (1-b2)*(gc*gc);
 *                    u = (m'/bc1) / (sqrt(v'/bc2) + eps); w' = w*(1 - lr*wd) - lr*u,
 *                    with 1-b1, 1-b2 and 1-lr*wd each rounded to fp32 once; wd = 0 for
 *                    elements a decay mask excludes; a bf16 w is widened first and w'
 *                    rounded to bf16 (nearest even) once.
 *   hash             leaves: PF61(header words {step, n}), then PF61 of each 4096-element
 *                    chunk of w, of m, of v (as 32-bit words); PF61(x_0..x_{W-1}) =
 *                    (W + sum x_i K^(i+1)) mod (2^61-1), K = floor(2^61 (sqrt5 - 1) / 2).
 *                    In audit mode (REPSTEP_HASH_BLAKE2B) each leaf is instead the LE u64
 *                    BLAKE2b-64 of the same bytes: the 8-byte header, then each chunk.
 *                    Root = T(leaves) with node N(a,b) = LE64 of BLAKE2b-64(LE64 a||LE64 b).
 *
 * Conventions for every call:
 *   - Device pointers are plain addresses in the current CUDA device's memory, owned by
 *     the caller (for example PyTorch allocations).  The library allocates no device
 *     memory: the caller provides one workspace of repstep_workspace_bytes() bytes.
 *   - All device work is enqueued asynchronously on the context's stream (a cudaStream_t
 *     passed as void*; NULL is the legacy default stream).  A returned REPSTEP_OK means
 *     the arguments were valid and the kernels were launched; a fault inside a kernel
 *     shows up at the next synchronisation, and repstep_sync() reports it.
 *   - Gradient, weight and moment buffers must be 16-byte aligned; the workspace 256-byte
 *     aligned.  Misalignment returns REPSTEP_ERR_ALIGN and launches nothing.
 *   - No call throws; every call returns a status code (repstep_strerror names it).
 *   - A context is not thread-safe; use one context per host thread or serialise.
 */
#ifndef REPSTEP_H
#define REPSTEP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define REPSTEP_CHUNK 4096u          /* fixed chunk length of the norm and of the hash   */
#define REPSTEP_MAX_REPLICAS 256u    /* largest R a single reduce accepts                */

enum repstep_status {
    REPSTEP_OK = 0,
    REPSTEP_ERR_ARG = 1,       /* null pointer, R == 0, bad range, non-finite hyperparameter */
    REPSTEP_ERR_ALIGN = 2,     /* a device pointer is not aligned as required               */
    REPSTEP_ERR_SIZE = 3,      /* n >= 2^32, R > REPSTEP_MAX_REPLICAS, workspace too small   */
    REPSTEP_ERR_TOPOLOGY = 4,  /* nodes*gpus_per_node != R, or gpus_per_node not a power of
                                  two while nodes > 1 (the staged sum would leave the
                                  canonical tree)                                         */
    REPSTEP_ERR_CUDA = 5,      /* a CUDA runtime call failed; repstep_last_cuda_error()     */
    REPSTEP_ERR_TIMEOUT = 6,   /* a kernel's bounded wait expired (reported by repstep_sync) */
    REPSTEP_ERR_STATE = 7,     /* call order: clip before the whole range was reduced, AdamW
                                  before clip, root before the whole range was updated      */
    REPSTEP_ERR_FORMAT = 8     /* checkpoint image: wrong size or header                     */
};

enum repstep_dtype { REPSTEP_F32 = 0, REPSTEP_BF16 = 1 };

enum repstep_subnormals { REPSTEP_SUBNORMALS_IEEE = 0, REPSTEP_SUBNORMALS_FTZ = 1 };

/* Leaf digest of the state hash.  PF61 (default) is fused into the AdamW pass and stays
 * under the HBM bound.  BLAKE2B ("audit mode") digests each leaf's image bytes with
 * BLAKE2b-64 -- the function the OPEN-1B paper hashes its steps with (App. B) -- in a
 * separate ALU-bound pass over the new state.  The Merkle tree and its BLAKE2b-64 nodes
 * are the same in both modes. */
enum repstep_hash_mode { REPSTEP_HASH_PF61 = 0, REPSTEP_HASH_BLAKE2B = 1 };

/* Device flag bits reported by repstep_sync(). */
#define REPSTEP_FLAG_NONFINITE_NORM  0x1u  /* the pre-clip norm is NaN or infinite        */
#define REPSTEP_FLAG_TIMEOUT_REDUCE  0x2u  /* a bounded wait expired in the reduce kernel  */
#define REPSTEP_FLAG_TIMEOUT_ADAMW   0x4u  /* ... in the AdamW / leaf kernel               */
#define REPSTEP_FLAG_TIMEOUT_LEAVES  0x8u  /* ... in the standalone leaf kernel            */

typedef struct repstep_ctx repstep_ctx;   /* opaque, host-side only */

typedef struct {
    uint64_t n;              /* number of fp32 parameters; n < 2^32 (0 is allowed)        */
    int32_t grad_dtype;      /* enum repstep_dtype of the replica gradients                */
    int32_t grid_blocks;     /* 0: persistent grid (SM count x resident CTAs); otherwise
                                the CTA count of the streaming kernels.  Never changes bits. */
    int32_t block_threads;   /* 0: default; else 128, 256 or 512 compute threads per CTA of
                                the streaming kernels.  Never changes bits.                */
    int32_t hash_mode;       /* enum repstep_hash_mode (0 = PF61 leaves)                   */
    int32_t param_dtype;     /* enum repstep_dtype of the parameters w.  REPSTEP_BF16: w is
                                bf16, widened exactly for the update, which runs in fp32,
                                and rounded back to bf16 once, to nearest even (OPEN-1B
                                §3.2, optimizer-state precision).  m and v are fp32 either
                                way; the image and the hash hold w widened to fp32.        */
    int32_t subnormals;      /* enum repstep_subnormals: 0 IEEE gradual underflow (default);
                                1 flush-to-zero -- every fp32 operation of the step treats
                                a subnormal operand as a zero of the same sign, and zeroes
                                a tiny result, keeping its sign (OPEN-1B §2.1 "Subnormals",
                                FTZ + DAZ).  Tiny means IEEE 754's tininess after rounding:
                                the exact result rounded to 24 bits with an unbounded
                                exponent is below 2^-126 -- the rule of the device's .ftz
                                instructions.  Also the hyperparameters and the constants
                                derived from them on the host.  Never changes the hash
                                function, only the values hashed.                          */
} repstep_config;

typedef struct {
    float lr, beta1, beta2, eps, weight_decay;
    float clip;              /* clip threshold (> 0; +inf disables clipping)               */
    float bc1, bc2;          /* bias corrections of this step, see repstep_bias_corrections */
} repstep_hparams;

/* Bytes of device workspace a context with this configuration needs (0 on a bad config).
 * Layout: g[n] fp32 | chunk sums fp32[c] | norm partials | leaf digests u64[1+3c] |
 * Merkle partials | PF61 power table u64[4096] | device scalars.  The norm and Merkle
 * partials are sized for the largest n (about 26 KB), so that the gathered calls of a
 * sharded step can run over every range's chunk sums and leaves. */
size_t repstep_workspace_bytes(const repstep_config *cfg);

/* Byte offsets of the workspace regions (for inspection and tests): g fp32[n], chunk sums
 * fp32[c], norm partials, leaf digests u64[1+3c] (header leaf first, then the w, m, v
 * chunks), Merkle partials, PF61 power table u64[4096], device scalars (pre-clip norm fp32,
 * clip scale fp32, flags u32, aux u32, root u64).  Returns REPSTEP_ERR_ARG on a bad config. */
typedef struct {
    uint64_t g, chunk_sums, norm_partials, leaves, merkle_partials, pow_table, scalars, total;
} repstep_layout;
int repstep_workspace_layout(const repstep_config *cfg, repstep_layout *out);

/* Create a context over a caller-owned workspace (256-byte aligned, at least
 * repstep_workspace_bytes(cfg) bytes) on `stream`.  Enqueues the initialisation of the
 * PF61 power table on the stream.  The workspace must outlive the context. */
int repstep_create(const repstep_config *cfg, void *d_workspace, size_t workspace_bytes,
                   void *stream, repstep_ctx **out);

/* Destroy the context: its host resources, after the work queued on its stream has
 * finished (a norm pass there may still store the last clip outcome into the context's
 * one word of mapped pinned host memory).  The workspace is the caller's. */
int repstep_destroy(repstep_ctx *ctx);

/* Change the stream later calls enqueue on. */
int repstep_set_stream(repstep_ctx *ctx, void *stream);

/* Optional second stream for the state hash (NULL, the default: none).  When set,
 * repstep_root (and the root of repstep_step and repstep_step_fused) runs its Merkle
 * passes on the hash stream, after the work already on the context's stream, which does
 * not wait for them: the next step overlaps them, the ALU-bound hash beside HBM-bound
 * kernels.  The bits are the same either way.
 * - PF61 mode: the call first completes the leaf array on the context's stream (the leaf
 *   fix-ups of cut chunks and the header leaf) and copies it to a snapshot in the
 *   workspace, which the Merkle passes read.  The next update (repstep_adamw,
 *   repstep_step, repstep_step_fused) therefore runs beside them.
 * - Audit mode: the BLAKE2b leaves are computed from w, m, v on the hash stream too, so an
 *   update that writes those arrays waits for them; repstep_step_fused's update into the
 *   other state buffer runs beside them.
 * Ordering, handled by the library: repstep_root, repstep_hash, repstep_leaves,
 * repstep_root_gathered, repstep_image_read and repstep_checkpoint_load (and, in the audit
 * mode, an update whose outputs share a byte with the hashed state) first make the
 * context's stream wait for the pending passes.
 * Ordering left to the caller: d_root_out is complete when the hash stream reaches the
 * end of the passes -- order a stream after them with repstep_wait_hash, or call
 * repstep_sync, which waits for both streams -- and in the audit mode w, m, v must not be
 * written by other code until then, because the leaf kernel reads them.
 * Creates two CUDA events on first use (host resources; no device memory). */
int repstep_set_hash_stream(repstep_ctx *ctx, void *hash_stream);

/* Profiling: while set, repstep_step_fused records ev_begin on the context's stream just
 * before its single pass and ev_end just after it, so that the caller can time that one
 * kernel (cudaEventElapsedTime).  Both are cudaEvent_t handles the caller created and
 * keeps alive while set; both null clears (one null and one not: REPSTEP_ERR_ARG).  The
 * events are recorded whenever the single pass is launched, also when its gate skips it;
 * configurations without the single pass record nothing. */
int repstep_set_pass_events(repstep_ctx *ctx, void *ev_begin, void *ev_end);

/* Make `stream` wait for the root passes last enqueued on the hash stream (no-op when none
 * is pending). */
int repstep_wait_hash(repstep_ctx *ctx, void *stream);

/* Replica reduce (OPEN-1B App. A.1 and A.3) over the element range [begin, begin+count):
 * g_i = T_{r<R}(G_r[i]) * fp32(1/R) into the workspace, plus the sum of squares of every
 * 4096-chunk lying wholly inside the range.  d_grads is a HOST array of R device pointers
 * to full-length gradient buffers (n elements of grad_dtype), in global replica order.
 * nodes x gpus_per_node (replica r = node*gpus_per_node + gpu) selects a staged sum: each
 * node's replicas first, then the node partials -- the same bits as the flat tree, which
 * the call guarantees by rejecting shapes that would differ (REPSTEP_ERR_TOPOLOGY).
 * Pass nodes = 1, gpus_per_node = R for the flat tree.  With count = 0 nothing is read, and
 * the R pointers may be NULL.  Ranges of one step may be reduced
 * in separate calls (reduce-scatter into shards, OPEN-1B App. A.2); chunks cut by a range
 * boundary are summed at clip time from the complete g. */
int repstep_reduce(repstep_ctx *ctx, const void *const *d_grads, uint32_t R, uint32_t nodes,
                   uint32_t gpus_per_node, uint64_t begin, uint64_t count);

/* Paper-exact replica reduce: the order of OPEN-1B §6 Algorithm 1 (App. A), for replaying
 * a cluster run bit for bit.  d_grads holds the R = dp_replicate * dp_shard virtual-rank
 * gradients in mesh order (r = replica * dp_shard + shard).  Per replica: its dp_shard
 * gradients summed in ascending shard order (App. A.2), times fp32(1/dp_shard) (App. A.3);
 * the replica partials folded by TreeFold (App. A.1: binary carry, lower replica on the
 * left; Result combines the leftover blocks from the largest, each later block on the
 * right -- the reading taken of App. A.1's self-contradictory level wording); times
 * fp32(1/dp_replicate).  Any dp_shard dividing R (REPSTEP_ERR_TOPOLOGY otherwise);
 * dp_replicate <= 256.  It writes the same workspace as repstep_reduce (g and the chunk sums)
 * and is followed by repstep_clip / repstep_adamw / repstep_root as usual.  For dp_shard = 1
 * and a power-of-two R it equals repstep_reduce bit for bit. */
int repstep_reduce_paper(repstep_ctx *ctx, const void *const *d_grads, uint32_t R,
                         uint32_t dp_shard, uint64_t begin, uint64_t count);

/* Paper-exact reduce with the microbatch accumulation of OPEN-1B §6 Algorithm 1's inner
 * loop: d_grads holds R * accum microbatch gradients, rank-major (pointer r*accum + k is
 * microbatch k of virtual rank r, r in mesh order as above); R * accum <= 256.  Each
 * virtual rank's gradient starts at +0 and adds its microbatches in order, each times
 * fp32(1/accum) (App. A.3) -- an explicit add, so with accum = 1 a -0 gradient element
 * becomes +0, the only difference from repstep_reduce_paper on the same pointers.  Then as
 * repstep_reduce_paper.  accum = 0 is REPSTEP_ERR_ARG. */
int repstep_reduce_paper_accum(repstep_ctx *ctx, const void *const *d_grads, uint32_t R,
                               uint32_t dp_shard, uint32_t accum, uint64_t begin,
                               uint64_t count);

/* Global norm and clip scale (OPEN-1B §3.2, §3.4.2) from the chunk sums of the reduced g.
 * Requires the reduce calls since the previous clip to have covered exactly n elements
 * (else REPSTEP_ERR_STATE).  Writes the pre-clip norm and the scale to the optional device
 * outputs (fp32, 4-byte aligned) and keeps them in the workspace for repstep_adamw.
 * clip must be > 0 (+inf: never clip). */
int repstep_clip(repstep_ctx *ctx, float clip, float *d_norm_out, float *d_scale_out);

/* Clipped AdamW over [begin, begin+count) of the full-length arrays w (param_dtype), m, v
 * (fp32), updated in place, using g and the scale from the last reduce/clip.  All three
 * pointers 16-byte aligned, and non-NULL unless the context's n is 0.  Also writes the
 * PF61 leaf digest of every new w, m and v chunk lying wholly inside the range;
 * repstep_root() completes the others.  All calls of one step must pass the same w, m, v
 * base pointers.  Requires repstep_clip() since the last reduce (else REPSTEP_ERR_STATE). */
int repstep_adamw(repstep_ctx *ctx, void *d_w, float *d_m, float *d_v,
                  const repstep_hparams *hp, uint64_t begin, uint64_t count);

/* Sharded steps ("OPEN-1B: A Fully Auditable Training Run", App. A.2: reduce-scatter over
 * shards -- each shard owner receives every replica's slice of its range and sums it in a
 * fixed order).  Each GPU owns one chunk-aligned range of the flat parameters and a context
 * whose n is that range's length; the exchanges between GPUs are the caller's collective
 * library, and carry data only: a routing of gradient slices before repstep_reduce, an
 * all-gather of the ranges' chunk sums before repstep_clip_gathered, an all-gather of
 * their leaf digests before repstep_root_gathered.  Every floating-point sum stays in this
 * library's canonical trees, so the bits equal the unsharded step's.
 *
 * repstep_clip_gathered: the global pre-clip norm and clip scale from d_chunk_sums, the
 * c_total = ceil(n_total/4096) chunk sums of every range in chunk order (fp32, 4-byte
 * aligned; this context's own are at repstep_layout.chunk_sums after its reduce).  Takes
 * the place of repstep_clip: the reduce calls since the last clip must have covered this
 * context's n along the chunk grid (REPSTEP_ERR_STATE otherwise), and the scale is kept for
 * repstep_adamw.  c_total below this context's chunk count is REPSTEP_ERR_ARG, above 2^20
 * REPSTEP_ERR_SIZE. */
int repstep_clip_gathered(repstep_ctx *ctx, const float *d_chunk_sums, uint64_t c_total,
                          float clip, float *d_norm_out, float *d_scale_out);

/* repstep_root_gathered: the Merkle root of the whole sharded state.  d_leaves (u64,
 * 8-byte aligned) holds 1 + 3 c_total slots: slots 1 .. 3 c_total the chunk leaf digests of
 * every range, gathered by the caller in image order (all w chunks, then all m chunks,
 * then all v chunks; this context's own are at repstep_layout.leaves + 1 after
 * repstep_adamw, or after repstep_leaves in audit mode); slot 0 receives the header leaf
 * of (step, n_total).  Requires the AdamW calls since the clip to have covered this
 * context's n along the chunk grid (REPSTEP_ERR_STATE).  Writes the root to d_root_out
 * (nullable) and to the context's scalars.  n_total below this context's n is
 * REPSTEP_ERR_ARG, at or above 2^32 REPSTEP_ERR_SIZE. */
int repstep_root_gathered(repstep_ctx *ctx, int32_t step, uint64_t n_total, uint64_t *d_leaves,
                          uint64_t *d_root_out);

/* Per-segment weight decay (OPEN-1B §3.2, optimizer paragraph: the embeddings, the
 * normalisation gains and RoPE take no weight decay).  d_mask is a device bitmask of
 * ceil(n/32) uint32 words (16-byte aligned, caller-owned, read by every later repstep_adamw
 * and repstep_step until replaced): bit e % 32 of word e / 32 set means element e decays,
 * w * (1 - lr*wd); clear means it does not, w * 1 (the update with wd = 0, bit for bit).
 * NULL (the default) makes every element decay.  Costs n/8 bytes of extra reads: the bits
 * of each whole tile are bulk-copied into shared memory with the tile. */
int repstep_set_decay_mask(repstep_ctx *ctx, const uint32_t *d_mask);

/* Host helper (no device access): the bitmask above from a segment list.  Segment s covers
 * [seg_begin[s], seg_begin[s+1]), the last one ends at n; seg_begin[0] must be 0 and the
 * starts strictly increasing and below n (REPSTEP_ERR_ARG otherwise; count 0 only for
 * n = 0).  decay[s] != 0 sets the segment's bits.  Writes all ceil(n/32) words of h_mask,
 * bits past n zero. */
int repstep_decay_mask_from_segments(uint64_t n, const uint64_t *seg_begin, const uint8_t *decay,
                                     uint32_t count, uint32_t *h_mask);

/* Merkle root of the state left by the repstep_adamw calls since the last clip, whose
 * ranges must total n elements (else REPSTEP_ERR_STATE); the header carries `step`.
 * Chunks cut by a range boundary get their leaves recomputed from the final w, m, v.
 * Writes the u64 root to d_root_out (8-byte aligned device pointer). */
int repstep_root(repstep_ctx *ctx, int32_t step, uint64_t *d_root_out);

/* Standalone state hash (OPEN-1B App. B) of an arbitrary (step, w, m, v): every leaf is
 * computed from the arrays (w of param_dtype, hashed as its fp32 image words), then the
 * Merkle root.  Equals repstep_root() after a step.  The arrays must be non-null and
 * 16-byte aligned (REPSTEP_ERR_ARG, REPSTEP_ERR_ALIGN) unless n = 0, where only the header
 * is hashed. */
int repstep_hash(repstep_ctx *ctx, int32_t step, const void *d_w, const float *d_m,
                 const float *d_v, uint64_t *d_root_out);

/* The leaves of repstep_hash without the Merkle passes: the 1 + 3c digests of (step, w, m,
 * v) -- header leaf first, then the chunks of w, of m, of v -- written as LE u64 words to
 * the workspace's leaf array (repstep_layout.leaves), where they stay until the next call
 * that hashes.  Comparing two states' leaf arrays locates the chunks where they differ.
 * Same arguments, alignment rules and errors as repstep_hash. */
int repstep_leaves(repstep_ctx *ctx, int32_t step, const void *d_w, const float *d_m,
                   const float *d_v);

/* One whole step: reduce over [0, n) -> clip -> AdamW over [0, n) -> root, bit-identical
 * to the four separate calls.  `step` is the header's step counter after the update; the
 * caller sets hp->bc1/bc2 for it (repstep_bias_corrections).  d_norm_out (nullable)
 * receives the pre-clip norm, d_root_out (nullable) the root. */
int repstep_step(repstep_ctx *ctx, const void *const *d_grads, uint32_t R, uint32_t nodes,
                 uint32_t gpus_per_node, void *d_w, float *d_m, float *d_v,
                 const repstep_hparams *hp, int32_t step, float *d_norm_out,
                 uint64_t *d_root_out);

/* One whole step in a single HBM pass when it does not clip, from the state (d_w, d_m, d_v)
 * into a second state buffer (d_w_out, d_m_out, d_v_out); the inputs are left untouched
 * (d_w and d_w_out of param_dtype, the others fp32; all 16-byte aligned, and no output may
 * share a byte with an input -- REPSTEP_ERR_ARG).  A caller alternates the two buffers
 * from step to step.
 * - The pass reduces the R gradients, forms the chunk sums of squares, applies AdamW with
 *   the clip scale taken as 1 and writes the new state and its PF61 leaves, reading the
 *   gradients and the state once and never writing g.  Then the norm passes compute the
 *   true scale.  Whenever the pre-clip norm does not exceed the clip threshold the scale
 *   is exactly 1 and those bits are the step's ("OPEN-1B: A Fully Auditable Training
 *   Run", §3.2: clipping to a global norm); otherwise the reduce and AdamW run again from
 *   the untouched inputs and overwrite the outputs.
 * - The context predicts from the last clip outcome (by any call) that has run by the time
 *   of the call: every final norm pass stores it into a word of mapped pinned host
 *   memory, which the call reads without waiting.  After a clip whose scale was not 1, the
 *   step takes the two passes of repstep_step at once (into the output buffers), and the
 *   single pass is not launched.  A right prediction costs one pass over R*b_g + 24 bytes
 *   per parameter without clipping, or the two passes' R*b_g + 32 with it; a wrong one
 *   costs the two passes, or the single pass and then the two.  A late outcome (the GPU
 *   behind the host) can only cost time.
 * - The result is bit for bit repstep_step's on the same inputs either way; only the
 *   time differs.
 * - The single pass covers R = 4, 8 or 16 with the default launch shape, in every gradient
 *   and parameter dtype, arithmetic mode, decay mask and hash mode; any other replica count
 *   or launch shape runs the two passes of repstep_step, writing the output buffers.
 * - `step`, hp, d_norm_out and d_root_out as repstep_step; the root is the output state's. */
int repstep_step_fused(repstep_ctx *ctx, const void *const *d_grads, uint32_t R,
                       const void *d_w, const float *d_m, const float *d_v, void *d_w_out,
                       float *d_m_out, float *d_v_out, const repstep_hparams *hp, int32_t step,
                       float *d_norm_out, uint64_t *d_root_out);

/* The two halves of repstep_step_fused, for a step whose clip runs between them -- the
 * sharded step, where the norm comes from every range's chunk sums (repstep_clip_gathered):
 *   repstep_fused_begin -> repstep_clip or repstep_clip_gathered -> repstep_fused_end ->
 *   repstep_root, or the leaves' gather and repstep_root_gathered.
 * repstep_fused_begin launches the single pass over [0, n) (or, after a clip that clipped,
 * the reduce of the two passes), which leaves the chunk sums at repstep_layout.chunk_sums;
 * with it the context counts as reduced over [0, n).  repstep_fused_end launches the
 * second pass where the clip needs one, and the AdamW of the two passes, into the output
 * buffers.  Both take the same arguments as repstep_step_fused (same rules, same errors);
 * repstep_fused_end must get exactly the buffers repstep_fused_begin got, after a clip
 * (REPSTEP_ERR_STATE otherwise).  The three calls together give repstep_step_fused's
 * bits. */
int repstep_fused_begin(repstep_ctx *ctx, const void *const *d_grads, uint32_t R,
                        const void *d_w, const float *d_m, const float *d_v, void *d_w_out,
                        float *d_m_out, float *d_v_out, const repstep_hparams *hp);
int repstep_fused_end(repstep_ctx *ctx, const void *const *d_grads, uint32_t R,
                      const void *d_w, const float *d_m, const float *d_v, void *d_w_out,
                      float *d_m_out, float *d_v_out, const repstep_hparams *hp);

/* One whole step whose R replica gradients start in HOST memory, with the norm and the
 * root returned to host memory: the end-to-end form of repstep_step for a caller whose
 * gradients arrive on the host side ("OPEN-1B: A Fully Auditable Training Run", §5: the
 * paper's step moves state to the host to hash it; here only the gradients cross the host
 * link, once, and everything after them runs on the device).
 * - h_grads: host array of R host pointers, each to n gradient elements of grad_dtype, in
 *   global replica order.  Page-locked memory (cudaHostAlloc, cudaHostRegister) lets the
 *   copies run asynchronously; pageable memory works, but each copy then blocks the host.
 * - d_staging: host array of R device pointers to caller-owned buffers of n elements
 *   (16-byte aligned) that the gradients are copied into and reduced from.  They must not
 *   be written by other code while the call's work runs.
 * - pieces: the parameter range is cut into this many chunk-aligned ranges (0: 8; at most
 *   64); range p of every replica is copied, and its reduce starts as soon as those copies
 *   are done, while later ranges are still being copied.
 * - copy_streams: the copies of a range are spread over this many streams, replica r on
 *   stream r mod copy_streams (0: 2; at most 8; at most R are used).  The streams and
 *   their events are created on the first call (host resources; no device memory) and
 *   wait for the work already on the context's stream before overwriting the staging.
 * - d_w, d_m, d_v, hp, step: as repstep_step.  The state stays on the device.
 * - h_norm_out (fp32), h_root_out (u64): host outputs, nullable.  When either is given,
 *   the call copies the pre-clip norm and the root there and returns after the step has
 *   finished (it synchronises the context's stream, after joining a pending root on the
 *   hash stream).  With both NULL it returns once everything is enqueued.
 * Bits: identical to repstep_step on the same gradients (a reduce split along the chunk
 * grid gives the bits of one reduce).  Errors: REPSTEP_ERR_ARG (null pointer, R == 0,
 * pieces > 64, copy_streams > 8, bad hyperparameter), REPSTEP_ERR_SIZE (R > 256),
 * REPSTEP_ERR_ALIGN, REPSTEP_ERR_CUDA; nothing is enqueued on an argument error. */
int repstep_step_from_host(repstep_ctx *ctx, const void *const *h_grads, uint32_t R,
                           void *const *d_staging, uint32_t pieces, uint32_t copy_streams,
                           void *d_w, float *d_m, float *d_v, const repstep_hparams *hp,
                           int32_t step, float *h_norm_out, uint64_t *h_root_out);

/* Checkpoint image ("grow_a_language_model_checkpoints", Format):
 * [LE int32 step][LE uint32 n][n fp32 w][n fp32 m][n fp32 v], 8 + 12n bytes, written to
 * dst (device memory, 4-byte aligned, or host memory when dst_is_host != 0) on the
 * context's stream.  bf16 parameters are written widened to fp32 (exact); to a host dst
 * that part is synchronous. */
uint64_t repstep_image_bytes(uint64_t n);
int repstep_image_write(repstep_ctx *ctx, int32_t step, const void *d_w, const float *d_m,
                        const float *d_v, void *dst, uint64_t dst_bytes, int dst_is_host);

/* Load an image into w, m, v (device arrays of the context's n).  Rejects (with
 * REPSTEP_ERR_FORMAT, before copying anything) a buffer whose size is not 8 + 12n, whose
 * header n differs from the context's n, or -- with bf16 parameters -- whose w holds a
 * word that is not a bf16 value exactly (low 16 bits not zero).  *step_out receives the
 * header step. */
int repstep_image_read(repstep_ctx *ctx, const void *src, uint64_t src_bytes, int src_is_host,
                       int32_t *step_out, void *d_w, float *d_m, float *d_v);

/* Checkpoint files ("grow_a_language_model_checkpoints", step_NNNNNN.bin): the image above,
 * streamed between the device arrays w, m, v (the context's n) and `path` through one
 * pinned host buffer of 64 MiB (host memory only; no device allocation).  Synchronous on
 * the context's stream.  Save writes `path`.tmp and renames it over `path` only when every
 * byte was written, so a crash never leaves a truncated file under the final name.  Load
 * rejects, before copying anything, a file whose size is not 8 + 12n or whose header n
 * differs (REPSTEP_ERR_FORMAT) -- a check that cannot fail is not a check, so the tests
 * feed it truncated, oversized and mismatched files.  bf16 parameters are widened on save;
 * load first reads the file's w words once and rejects (REPSTEP_ERR_FORMAT) a file with
 * any word that is not a bf16 value exactly.  REPSTEP_ERR_ARG if the file cannot be opened
 * or written. */
int repstep_checkpoint_save(repstep_ctx *ctx, const char *path, int32_t step, const void *d_w,
                            const float *d_m, const float *d_v);
int repstep_checkpoint_load(repstep_ctx *ctx, const char *path, int32_t *step_out, void *d_w,
                            float *d_m, float *d_v);

/* Bias corrections for step t >= 1: p_j = beta_j^t as t repeated fp32 products,
 * bc_j = 1 - p_j (the reading taken for AdamW's bias correction; computed on the host). */
void repstep_bias_corrections(float beta1, float beta2, int32_t t, float *bc1, float *bc2);

/* Synchronise the context's stream (and the pending root passes of the hash stream, if
 * any) and read the device flags (REPSTEP_FLAG_*; nullable output).  Returns
 * REPSTEP_ERR_CUDA if the stream reported an error, REPSTEP_ERR_TIMEOUT if a kernel's
 * bounded wait expired, else REPSTEP_OK.  Clears the timeout flags. */
int repstep_sync(repstep_ctx *ctx, uint32_t *flags_out);

/* Self-test of the fixed-divisor division inside the AdamW kernel.  The bias corrections
 * bc1 and bc2 are the same for every element of a step, so the kernel divides by them as
 * q = RN(x*y), r = x - q*b, RN(q + r*y) with y = RN(1/b) (Markstein's correction, two fused
 * multiply-adds) instead of a full IEEE division, for b in [2^-40, 2] and |x| in
 * [2^-100, 2^60]; other operands take the IEEE division.  This entry point compares that
 * code with the IEEE division for every x significand in [1, 2) and every b significand in
 * [1 + b_sig_begin 2^-23, 1 + (b_sig_begin + b_sig_count) 2^-23), adding the number of
 * differing results to *d_mismatches (a device u64 the caller zeroes).  The whole range
 * (begin 0, count 2^23; 2^46 pairs) takes well under a minute on a GB300 and finds none.
 * Returns REPSTEP_ERR_ARG for a range outside [0, 2^23). */
int repstep_selftest_fixed_division(uint32_t b_sig_begin, uint32_t b_sig_count,
                                    uint64_t *d_mismatches, void *stream);

/* Self-test of the branch-free square root, reciprocal and division of the AdamW kernel's
 * fast path (Newton iterations from the hardware approximations, then Markstein's
 * correction).  The kernel takes that path when every lane of a warp has m' zero or of
 * magnitude in [2^-84, 2^40] and v' zero or in [2^-100, 2^40], and the bias corrections
 * are in [2^-40, 2] and eps in [2^-40, 2^20]; then sqrt(v'/bc2) has an argument in
 * [2^-101, 2^80] and the update divides a numerator in [2^-85, 2^80] by a denominator in
 * [2^-40, 2^41).  which = 0: the square root of every float whose bit pattern is in
 * [begin, begin+count); 1: the reciprocal of every such float; 2: count x 1024
 * pseudo-random divisions drawn from `seed`, with divisor in [2^-41, 2^41) and dividend 0
 * or of magnitude in [2^-85, 2^81), either sign.  Each result is compared with the IEEE
 * operation, and the number that differ is added to *d_mismatches (a device u64 the
 * caller zeroes).  The whole square-root range 0x0C800000..0x68000000 ([2^-102, 2^81)) and
 * reciprocal range 0x2A800000..0x54800000 ([2^-42, 2^42)) find none.  Returns
 * REPSTEP_ERR_ARG for which outside 0..2 or a bit range past 2^32. */
int repstep_selftest_fast_math(int which, uint32_t begin, uint32_t count, uint64_t seed,
                               uint64_t *d_mismatches, void *stream);

/* Kernels this context has launched so far. */
uint64_t repstep_launch_count(const repstep_ctx *ctx);

/* The cudaError_t of the last failed CUDA call (0 if none). */
int repstep_last_cuda_error(const repstep_ctx *ctx);

/* Static name of a status code. */
const char *repstep_strerror(int code);

/* ---------------------------------------------------------------------------------------
 * Replica reduce + global norm WITHOUT ANY DEVICE ALLOCATION.  The paper has no counterpart
 * to this entry point; it serves callers that may not allocate device memory when they need
 * the averaged gradient and its norm -- for example an audit replay running beside a
 * training job that already holds almost all device memory through its own allocator, or
 * an error path entered after an out-of-memory condition.  Such callers cannot provide the
 * workspace the other entry points need.
 *
 * Computes g[i] = T_{r<R}(G_r[i]) * fp32(1/R) into d_g (n fp32, 16-byte aligned) and writes
 * the pre-clip norm to *d_norm_out and, if d_scale_out is not NULL, the clip scale for
 * `clip` -- bit for bit what repstep_reduce (flat tree) + repstep_clip produce with the
 * default launch configuration.  d_grads is a host array of R device pointers, as for
 * repstep_reduce.  Work is enqueued on `stream` (a cudaStream_t as void*).
 *
 * Scratch: one fixed array inside the library (about 1 MiB, held on every GPU that loads
 * the library until the process exits), so n is limited to REPSTEP_NOALLOC_MAX_N; larger n
 * returns REPSTEP_ERR_SIZE before any work is enqueued.  The call allocates nothing: no
 * cudaMalloc, cudaFree or allocating library routine.  Every call on a device shares the
 * same array and leaves its contents behind (each call clears what must start at zero), so
 * calls whose GPU work overlaps -- on different streams or host threads -- race and give
 * undefined results: serialise them.  The first call on each device, with that device
 * current, looks up the array's device address (cudaGetSymbolAddress) and -- since CUDA
 * loads device code lazily by default -- may load the library's device code and this array
 * onto the device, which does take device memory.  So make that first call at start-up,
 * before the device's memory is taken and before any stream capture; from then until the
 * process exits the array stays held and later calls allocate nothing.  Returns
 * REPSTEP_OK, REPSTEP_ERR_ARG, REPSTEP_ERR_ALIGN, REPSTEP_ERR_SIZE or REPSTEP_ERR_CUDA. */
#define REPSTEP_NOALLOC_MAX_N (1ull << 30)
int repstep_reduce_norm_noalloc(const void *const *d_grads, uint32_t R, int32_t grad_dtype,
                                uint64_t n, float clip, float *d_g, float *d_norm_out,
                                float *d_scale_out, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* REPSTEP_H */
