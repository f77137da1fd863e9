// kernels.h -- host-side launch interface between the C ABI (repstep.cu) and the kernel
// translation units.  Internal; not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace repstep {

struct Scalars;

// Replica reduce + chunk sums of squares (k_reduce.cu).
struct ReduceArgs {
    const void *grads[256];   // R device pointers, global replica order
    float *g;                 // workspace g[n]
    float *chunk_sq;          // workspace fp32[c]
    Scalars *sc;              // device scalars (flags)
    uint64_t n, begin, end;   // active range [begin, end)
    uint64_t chunk_lo, chunk_hi;
    uint32_t R, nodes, gpn;
    uint32_t stages;          // ring depth
    uint32_t stage_stride;    // bytes per stage
    float rho;                // fp32(1/R); fp32(1/dp_replicate) in the paper-exact mode
    float rho2;               // fp32(1/dp_shard) in the paper-exact mode
    uint32_t accum;           // paper-exact mode: 0 = one gradient per virtual rank; else
                              // microbatches per rank, accumulated from +0
    float rho3;               // fp32(1/accum)
    int gate;                 // kGateAlways, or kGateIfClipped (repstep_step_fused)
};

struct ReduceShape {
    int nt;          // compute threads (128, 256, 512)
    int dtype;       // 0 fp32, 1 bf16
    int mode;        // 0 canonical tree, 1 topology-staged, 2 paper-exact (Algorithm 1)
    int rg;          // replicas per stage group (4 or 8)
    int maxlev;      // carry-stack depth (6 or 9)
    int fz;          // 0 IEEE, 1 flush-to-zero (.ftz arithmetic)
};

using ReduceKernelFn = void (*)(ReduceArgs);
// The instantiation for a shape, from the translation unit of its arithmetic mode.
ReduceKernelFn pick_reduce_ieee(const ReduceShape &s);
ReduceKernelFn pick_reduce_ftz(const ReduceShape &s);

// Chooses the kernel instantiation and ring depth for a reduce; returns the dynamic
// shared-memory bytes and fills args.stages / args.stage_stride.
size_t reduce_smem_bytes(const ReduceShape &s, ReduceArgs &args);
cudaError_t reduce_prepare(const ReduceShape &s, size_t smem);   // raise the smem limit
cudaError_t reduce_occupancy(const ReduceShape &s, size_t smem, int *blocks_per_sm);
cudaError_t launch_reduce(const ReduceShape &s, const ReduceArgs &args, int grid, size_t smem,
                          cudaStream_t st);

// AdamW + leaf digests, or leaves only (k_adamw.cu).
struct AdamwArgs {
    const float *g;           // MODE adamw: workspace g
    void *w;                  // parameters: fp32, or bf16 when the kernel's PT is 1
    float *m, *v;             // Adam moments (fp32), read
    void *wo;                 // where the AdamW modes write w', m', v': w, m, v themselves
    float *mo, *vo;           // (in place), or a second state buffer (repstep_step_fused)
    int gate;                 // kGateAlways, or kGateIfClipped (repstep_step_fused)
    uint64_t *leaves;         // workspace u64[1 + 3c]
    const uint64_t *powers;   // workspace K^1..K^4096 mod p
    Scalars *sc;              // device scalars (scale, flags)
    uint64_t n, c, begin, end;
    uint64_t chunk_lo, chunk_hi;
    uint32_t stages, stage_stride;
    float lr, beta1, beta2, eps, bc1, bc2, om1, om2, delta;
    float rbc1, rbc2;         // RN(1/bc1), RN(1/bc2): divisors fixed for the launch
    int fastdiv;              // bias corrections in [2^-40, 2], eps in [2^-40, 2^20]
    const uint32_t *decay_mask;   // null: every element decays; else bit e%32 of word e/32
};

// The AdamW / leaf kernel variant of a launch.
struct AdamwShape {
    int nt;     // compute threads (128, 256, 512)
    int mode;   // 0 AdamW + PF61 leaves, 1 leaves only, 2 AdamW only
    int pt;     // 1: bf16 parameters
    int fz;     // 1: flush-to-zero (.ftz) arithmetic
    int mk;     // 1: per-element weight-decay mask (args.decay_mask)
};
size_t adamw_smem_bytes(const AdamwShape &s, AdamwArgs &args);
cudaError_t adamw_prepare(const AdamwShape &s, size_t smem);
cudaError_t adamw_occupancy(const AdamwShape &s, size_t smem, int *blocks_per_sm);
cudaError_t launch_adamw(const AdamwShape &s, const AdamwArgs &args, int grid, size_t smem,
                         cudaStream_t st);
using AdamwKernelFn = void (*)(AdamwArgs);
AdamwKernelFn pick_adamw_ieee(const AdamwShape &s);
AdamwKernelFn pick_adamw_ftz(const AdamwShape &s);
// The speculative single-pass step (k_fused.cuh): replica reduce, chunk sums of squares,
// AdamW with clip scale 1 from (w, m, v) into (wo, mo, vo), and the PF61 leaves of the new
// state.  R is 4, 8 or 16.
struct FusedArgs {
    const void *grads[16];    // the R replica gradients, global replica order
    float *chunk_sq;          // workspace fp32[c]
    uint32_t R;
    float rho;                // fp32(1/R)
    AdamwArgs adam;           // state in and out, leaves, powers, scalars, n, c, constants,
                              // ring depth and stage size
};

struct FusedShape {
    int dtype;    // gradients: 0 fp32, 1 bf16
    int rg;       // R: 4, 8 or 16
    int leaves;   // 1: PF61 leaves fused (hash mode PF61); 0: none (audit mode)
    int pt;       // 1: bf16 parameters
    int fz;       // 1: flush-to-zero (.ftz) arithmetic
    int mk;       // 1: per-element weight-decay mask (adam.decay_mask)
};
using FusedKernelFn = void (*)(FusedArgs);
FusedKernelFn pick_fused_ieee(const FusedShape &s);       // R = 4, 8
FusedKernelFn pick_fused_ftz(const FusedShape &s);
FusedKernelFn pick_fused_wide_ieee(const FusedShape &s);  // R = 16
FusedKernelFn pick_fused_wide_ftz(const FusedShape &s);
size_t fused_smem_bytes(const FusedShape &s, FusedArgs &args);
cudaError_t fused_prepare(const FusedShape &s, size_t smem);
cudaError_t fused_occupancy(const FusedShape &s, size_t smem, int *blocks_per_sm);
// ev_begin / ev_end (both or neither): recorded on st just before and after the kernel
cudaError_t launch_fused(const FusedShape &s, const FusedArgs &args, int grid, size_t smem,
                         cudaStream_t st, cudaEvent_t ev_begin = nullptr,
                         cudaEvent_t ev_end = nullptr);

cudaError_t launch_selftest_div(uint32_t b_begin, uint32_t b_count, unsigned long long *mismatches,
                               cudaStream_t st);
cudaError_t launch_selftest_fast_math(int which, uint32_t begin, uint32_t count, uint64_t seed,
                                      unsigned long long *mismatches, cudaStream_t st);

// Small kernels (k_small.cu).
cudaError_t launch_init_powers(uint64_t *powers, cudaStream_t st);
cudaError_t launch_chunk_fix(const float *g, uint64_t n, float *chunk_sq, const uint64_t *chunks,
                             int count, int fz, cudaStream_t st);
cudaError_t launch_leaf_fix(const void *w, int w_bf16, const float *m, const float *v, uint64_t n,
                            uint64_t c, uint64_t *leaves, const uint64_t *powers,
                            const uint64_t *chunks, int count, cudaStream_t st);
// clip_flag (nullable, a host-mapped word): the final pass stores 1 there when the scale
// is not 1, else 0
cudaError_t launch_norm(const float *in, uint64_t count, float *out, Scalars *sc, int final_pass,
                        float clip, float *norm_out, float *scale_out, int blocks, int fz,
                        cudaStream_t st, uint32_t *clip_flag = nullptr);
cudaError_t merkle_prepare();
cudaError_t launch_merkle(const uint64_t *in, uint64_t count, uint64_t *out, int header_mode,
                          uint64_t *leaves_rw, uint32_t step, uint32_t n32, const uint64_t *powers,
                          Scalars *sc, uint64_t *root_out, int blocks, cudaStream_t st);
cudaError_t launch_header_leaf(uint64_t *leaves, int32_t step, uint32_t n32, const uint64_t *powers,
                               cudaStream_t st);
cudaError_t launch_write_header(void *dst, int32_t step, uint32_t n32, cudaStream_t st);
// bf16 -> fp32 (exact) into an image's w region.  fp32 -> bf16 by dropping the low half
// (dst nullable: check only); a word whose low half is not zero sets *bad (nullable) to 1.
cudaError_t launch_widen_bf16(float *dst, const unsigned short *src, uint64_t n, cudaStream_t st);
cudaError_t launch_narrow_bf16(unsigned short *dst, const float *src, uint64_t n, uint32_t *bad,
                               cudaStream_t st);

// Audit-mode leaves: BLAKE2b-64 of the header and of every chunk of w, m, v (k_blake2b.cu).
cudaError_t launch_leaves_b2(const void *w, int w_bf16, const float *m, const float *v, uint64_t n,
                             uint64_t c, uint64_t *leaves, uint32_t step, int sm_count,
                             cudaStream_t st);
cudaError_t leaves_b2_prepare();   // shared-memory carveout (run beside the single pass)

constexpr int kFixMax = 64;   // chunk indices per fix-up launch

}  // namespace repstep
