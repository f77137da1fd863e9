// repstep.cu -- host side of the C ABI declared in include/repstep.h: argument validation,
// workspace layout, host-computed fp32 constants, call-order state, and the sequence of
// kernel launches on the caller's stream.  No device memory is allocated here.
//
// Host fp32 constants are computed with plain IEEE single operations, one rounding each
// (the library is built with -ffp-contract=off for host code too):
//   rho = 1/R   ("OPEN-1B: A Fully Auditable Training Run", App. A.3: every average is a
//                multiply by a host-computed reciprocal)
//   1 - b1, 1 - b2, 1 - lr*wd, and the bias corrections 1 - b^t (t repeated products).
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "../../include/repstep.h"
#include "common.cuh"
#include "kernels.h"
#include "merkle.h"

using namespace repstep;

namespace {

constexpr uint32_t kMaxCopyStreams = 8;   // repstep_step_from_host: copy streams
constexpr uint32_t kMaxPieces = 64;        // ... and pipelined ranges

struct Layout {
    uint64_t g, chunk_sq, norm_part, leaves, merkle_part, leaf_snap, powers, scalars, total;
};

// An NVTX range over one public call, for timeline tools (a no-op when none is attached).
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};

constexpr uint64_t kAlign = 256;

uint64_t align_up(uint64_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool valid_config(const repstep_config *cfg)
{
    if (!cfg) return false;
    if (cfg->n > 0xFFFFFFFFull) return false;
    if (cfg->grad_dtype != REPSTEP_F32 && cfg->grad_dtype != REPSTEP_BF16) return false;
    if (cfg->param_dtype != REPSTEP_F32 && cfg->param_dtype != REPSTEP_BF16) return false;
    if (cfg->subnormals != REPSTEP_SUBNORMALS_IEEE && cfg->subnormals != REPSTEP_SUBNORMALS_FTZ)
        return false;
    if (cfg->grid_blocks < 0) return false;
    if (cfg->block_threads != 0 && cfg->block_threads != 128 && cfg->block_threads != 256 &&
        cfg->block_threads != 512)
        return false;
    return cfg->hash_mode == REPSTEP_HASH_PF61 || cfg->hash_mode == REPSTEP_HASH_BLAKE2B;
}

Layout layout_of(uint64_t n)
{
    const uint64_t c = (n + kChunk - 1) / kChunk;
    // The norm and Merkle partials are sized for the largest n (2^32 - 1, c = 2^20 chunks),
    // not for this context's: repstep_clip_gathered and repstep_root_gathered run the same
    // passes over all shards' chunk sums and leaves (about 26 KB in all).
    const uint64_t c_max = ((uint64_t(1) << 32) - 1 + kChunk - 1) / kChunk;
    const uint64_t nb2 = (c_max + kChunk - 1) / kChunk;
    const uint64_t L_max = 1 + 3 * c_max;
    // Merkle partials, ping-pong: the first pass's block roots, then the second pass's
    const uint64_t mb1 = (L_max + kMerkleBlock - 1) / kMerkleBlock;
    const uint64_t mb2 = (mb1 + kMerkleBlock - 1) / kMerkleBlock;
    Layout l{};
    uint64_t off = 0;
    l.g = off;           off = align_up(off + 4 * (n ? n : 1));
    l.chunk_sq = off;    off = align_up(off + 4 * (c ? c : 1));
    l.norm_part = off;   off = align_up(off + 4 * nb2);
    l.leaves = off;      off = align_up(off + 8 * (1 + 3 * c));
    l.merkle_part = off; off = align_up(off + 8 * (mb1 + mb2));
    l.leaf_snap = off;   off = align_up(off + 8 * (1 + 3 * c));
    l.powers = off;      off = align_up(off + 8 * kChunk);
    l.scalars = off;     off = align_up(off + sizeof(Scalars));
    l.total = off;
    return l;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool finite_f(float x) { return std::isfinite(x); }

// Host side of the flush-to-zero mode: a subnormal becomes a zero of the same sign
// (fz != 0); used for the hyperparameters and the constants derived from them.
float hflush(int fz, float x)
{
    return (fz && std::fpclassify(x) == FP_SUBNORMAL) ? std::copysign(0.0f, x) : x;
}

// A product in the flush-to-zero mode, as the device's mul.rn.ftz computes it: operands
// flushed, and a tiny result -- the exact product rounded to 24 bits as though the
// exponent were unbounded is below 2^-126 -- becomes a zero of the product's sign.  The
// double product of two floats is exact; below 2^-126 it is rounded to 24 bits by hand.
float hmul(int fz, float a, float b)
{
    if (!fz) return a * b;
    a = hflush(1, a);
    b = hflush(1, b);
    const double p = double(a) * double(b);
    const float r = float(p);
    if (!(std::fabs(p) < 0x1p-126) || p == 0.0) return r;
    int e = 0;
    const double frac = std::frexp(std::fabs(p), &e);                // in [0.5, 1)
    const double rounded = std::ldexp(std::nearbyint(std::ldexp(frac, 24)), e - 24);
    return rounded < 0x1p-126 ? std::copysign(0.0f, r) : r;
}

}  // namespace

struct repstep_ctx {
    repstep_config cfg;
    Layout lay;
    unsigned char *ws;
    cudaStream_t stream;
    uint64_t n, c;
    int sm_count;
    int nt_reduce, nt_adamw;
    uint64_t launches;
    int last_err;
    // call-order state of the current step
    uint64_t reduced;        // elements reduced since the last clip
    bool scale_ready;        // a clip followed the last reduce
    uint64_t updated;        // elements updated by AdamW since the last clip
    const void *sw;
    const float *sm, *sv;
    const uint32_t *decay_mask = nullptr;     // per-element weight-decay bits (caller-owned)
    // optional second stream for the root passes (repstep_set_hash_stream): ev_state marks
    // the state they read, ev_hash their end, which later writers of that state wait for
    cudaStream_t hash_stream = nullptr;
    cudaEvent_t ev_state = nullptr, ev_hash = nullptr;
    // caller's events recorded around the single pass (repstep_set_pass_events)
    cudaEvent_t pass_ev[2] = {nullptr, nullptr};
    // the outcome of the last clip that has run, as the host sees it: a word of mapped
    // pinned host memory (clip_flag_h) that every final norm pass stores 1 (clipped) or 0
    // into through its device address (clip_flag_d); null where the device maps no host
    // memory, and then the single-pass step always speculates
    uint32_t *clip_flag_h = nullptr, *clip_flag_d = nullptr;
    // the single-pass step between its halves (repstep_fused_begin .. repstep_fused_end):
    // the buffers the second half must be given (the state and, of the gradients, the
    // first 16, all the single pass takes), and whether the single pass was launched
    struct FusedCall {
        bool open = false, single = false;
        uint32_t R = 0;
        const void *g[16] = {};
        const void *st[6] = {};
    } fused;
    bool hash_pending = false;
    // the pending root passes read the state (the audit mode: hash_st, the three arrays
    // and their bytes); otherwise they read only the leaf snapshot and the Merkle partials
    bool hash_reads_live = false;
    const void *hash_st[3] = {nullptr, nullptr, nullptr};
    uint64_t hash_st_bytes[3] = {0, 0, 0};
    std::vector<uint64_t> cut_norm, cut_leaf;   // chunks cut by range boundaries

    // repstep_step_from_host: copy streams and events, created on first use (host resources
    // only).  ev_free orders the copies after earlier readers of the staging buffers on the
    // context's stream; copy_ev[p * kMaxCopyStreams + k] marks the end of range p's copies on
    // copy stream k, which the reduce of range p waits for.
    cudaStream_t copy_st[kMaxCopyStreams] = {};
    std::vector<cudaEvent_t> copy_ev;
    cudaEvent_t ev_free = nullptr;

    float *g() const { return reinterpret_cast<float *>(ws + lay.g); }
    float *chunk_sq() const { return reinterpret_cast<float *>(ws + lay.chunk_sq); }
    float *norm_part() const { return reinterpret_cast<float *>(ws + lay.norm_part); }
    uint64_t *leaves() const { return reinterpret_cast<uint64_t *>(ws + lay.leaves); }
    uint64_t *merkle_part() const { return reinterpret_cast<uint64_t *>(ws + lay.merkle_part); }
    // the leaves the Merkle passes read on the hash stream in the PF61 mode (repstep_root)
    uint64_t *leaf_snap() const { return reinterpret_cast<uint64_t *>(ws + lay.leaf_snap); }
    uint64_t *powers() const { return reinterpret_cast<uint64_t *>(ws + lay.powers); }
    Scalars *sc() const { return reinterpret_cast<Scalars *>(ws + lay.scalars); }
    int w_bf16() const { return cfg.param_dtype == REPSTEP_BF16 ? 1 : 0; }
    int fz() const { return cfg.subnormals == REPSTEP_SUBNORMALS_FTZ ? 1 : 0; }
    uint64_t w_bytes() const { return n * (w_bf16() ? 2 : 4); }

    int cuda_fail(cudaError_t e)
    {
        last_err = int(e);
        return REPSTEP_ERR_CUDA;
    }
};

namespace {

// Order the context's stream after a root still running on the hash stream: called before
// anything that writes the leaves, the leaf snapshot, the Merkle partials or the state the
// root passes read.
int join_hash(repstep_ctx *x)
{
    if (!x->hash_pending) return REPSTEP_OK;
    const cudaError_t e = cudaStreamWaitEvent(x->stream, x->ev_hash, 0);
    if (e != cudaSuccess) return x->cuda_fail(e);
    x->hash_pending = false;
    return REPSTEP_OK;
}

bool overlaps(const void *a, uint64_t na, const void *b, uint64_t nb);

// Before an update writes (wo, mo, vo): only a pending root that reads what it writes
// must end first.  A PF61 root reads the leaf snapshot its call took; an audit-mode root
// reads the state it hashes, which an update into the other state buffer of the
// single-pass step leaves alone.  So both run beside such an update.
int join_hash_for_update(repstep_ctx *x, const void *wo, const void *mo, const void *vo)
{
    if (!x->hash_pending || !x->hash_reads_live) return REPSTEP_OK;
    const void *outs[3] = {wo, mo, vo};
    const uint64_t out_bytes[3] = {x->w_bytes(), 4 * x->n, 4 * x->n};
    for (int i = 0; i < 3; ++i)
        for (int j = 0; j < 3; ++j)
            if (overlaps(outs[i], out_bytes[i], x->hash_st[j], x->hash_st_bytes[j]))
                return join_hash(x);
    return REPSTEP_OK;
}

// Persistent grid: SM count x resident CTAs, never more CTAs than chunks to process.
int grid_for(repstep_ctx *x, int blocks_per_sm, uint64_t chunks)
{
    uint64_t g = x->cfg.grid_blocks > 0 ? uint64_t(x->cfg.grid_blocks)
                                        : uint64_t(x->sm_count) * uint64_t(blocks_per_sm > 0 ? blocks_per_sm : 1);
    if (g > chunks) g = chunks;
    if (g < 1) g = 1;
    return int(g);
}

// Record the chunks a range [b, e) cuts (partly covered, so not summed in the kernel).
void note_cut_chunks(std::vector<uint64_t> &v, uint64_t b, uint64_t e, uint64_t n)
{
    if (b >= e) return;
    const uint64_t k0 = b / kChunk, k1 = (e - 1) / kChunk;
    auto cut = [&](uint64_t k) {
        const uint64_t c0 = k * kChunk, c1 = c0 + kChunk < n ? c0 + kChunk : n;
        return !(c0 >= b && c1 <= e);
    };
    if (cut(k0)) v.push_back(k0);
    if (k1 != k0 && cut(k1)) v.push_back(k1);
}

// Each cut chunk once, in ascending order (a step reduced in many ranges lists many).
void unique_sort(std::vector<uint64_t> &v)
{
    std::sort(v.begin(), v.end());
    v.erase(std::unique(v.begin(), v.end()), v.end());
}

int check_hparams(const repstep_hparams *hp)
{
    if (!hp) return REPSTEP_ERR_ARG;
    if (!finite_f(hp->lr) || !finite_f(hp->beta1) || !finite_f(hp->beta2) ||
        !finite_f(hp->eps) || !finite_f(hp->weight_decay) || !finite_f(hp->bc1) ||
        !finite_f(hp->bc2) || hp->bc1 == 0.0f || hp->bc2 == 0.0f)
        return REPSTEP_ERR_ARG;
    return REPSTEP_OK;
}

// mode 0: canonical tree (nodes x gpn staged when nodes > 1); mode 2: paper-exact order of
// OPEN-1B Algorithm 1 with dp_replicate = nodes and dp_shard = gpn.
// R replicas (virtual ranks) = nodes x gpn; with accum > 0 (paper mode only) `grads`
// holds R * accum microbatch gradients, rank-major.
// gate: kGateIfClipped for the second pass of the single-pass step, which returns at once
// when the clip scale is 1; the call-order state is left as the caller set it.
int do_reduce(repstep_ctx *x, const void *const *grads, uint32_t R, uint32_t nodes,
              uint32_t gpn, uint64_t begin, uint64_t count, int paper = 0, uint32_t accum = 0,
              int gate = kGateAlways)
{
    if (!grads || R == 0) return REPSTEP_ERR_ARG;
    const uint64_t inputs = uint64_t(R) * (accum ? accum : 1);
    if (inputs > kMaxReplicas) return REPSTEP_ERR_SIZE;
    if (nodes == 0 || gpn == 0 || uint64_t(nodes) * gpn != R) return REPSTEP_ERR_TOPOLOGY;
    if (!paper && nodes > 1 && (gpn & (gpn - 1)) != 0) return REPSTEP_ERR_TOPOLOGY;
    if (begin > x->n || count > x->n - begin) return REPSTEP_ERR_ARG;
    R = uint32_t(inputs);     // the kernel streams every input
    for (uint32_t r = 0; r < R && count > 0; ++r) {   // an empty range reads no buffer
        if (!grads[r]) return REPSTEP_ERR_ARG;
        if (!aligned(grads[r], 16)) return REPSTEP_ERR_ALIGN;
    }
    if (gate == kGateAlways) {
        x->fused.open = false;                // a single-pass step left between its halves
        if (x->scale_ready || x->updated) {   // a new step starts
            x->scale_ready = false;
            x->updated = 0;
            x->cut_leaf.clear();
        }
        x->reduced += count;
    }
    if (count == 0) return REPSTEP_OK;
    // The bf16-gradient reduce hands out chunks by CTA index, so CTAs held back by the
    // Merkle blocks of a pending root finish late and the whole launch waits for them:
    // it starts after the root instead (measured at 3e9 parameters: 21.7 -> 21.5 ms).
    if (x->cfg.grad_dtype == REPSTEP_BF16) {
        const int jr = join_hash(x);
        if (jr) return jr;
    }

    const uint64_t end = begin + count;
    ReduceArgs a{};
    for (uint32_t r = 0; r < R; ++r) a.grads[r] = grads[r];
    a.g = x->g();
    a.chunk_sq = x->chunk_sq();
    a.sc = x->sc();
    a.n = x->n;
    a.begin = begin;
    a.end = end;
    a.chunk_lo = begin / kChunk;
    a.chunk_hi = (end + kChunk - 1) / kChunk;
    a.R = R;
    a.nodes = nodes;
    a.gpn = gpn;
    const float one = 1.0f;
    const int fz = x->fz();
    a.rho = hflush(fz, paper ? one / float(nodes) : one / float(R));
    a.rho2 = hflush(fz, paper ? one / float(gpn) : one);
    a.accum = paper ? accum : 0;
    a.rho3 = hflush(fz, accum ? one / float(accum) : one);
    a.gate = gate;
    ReduceShape s{};
    s.nt = x->nt_reduce;
    s.dtype = x->cfg.grad_dtype;
    s.mode = paper ? 2 : (nodes > 1 ? 1 : 0);
    s.rg = R >= 8 ? 8 : 4;
    s.maxlev = R <= 32 ? 6 : 9;
    s.fz = fz;
    const size_t smem = reduce_smem_bytes(s, a);
    cudaError_t e = reduce_prepare(s, smem);
    if (e != cudaSuccess) return x->cuda_fail(e);
    int bps = 1;
    e = reduce_occupancy(s, smem, &bps);
    if (e != cudaSuccess) return x->cuda_fail(e);
    const int grid = grid_for(x, bps, a.chunk_hi - a.chunk_lo);
    e = launch_reduce(s, a, grid, smem, x->stream);
    if (e != cudaSuccess) return x->cuda_fail(e);
    ++x->launches;
    if (gate == kGateAlways) note_cut_chunks(x->cut_norm, begin, end, x->n);
    return REPSTEP_OK;
}

// The canonical tree over `c` chunk sums, its square root and the clip scale (one or two
// passes), into the context's scalars and the optional outputs.
int norm_passes(repstep_ctx *x, const float *sums, uint64_t c, float clip, float *norm_out,
                float *scale_out)
{
    const int fz = x->fz();
    cudaError_t e;
    if (c > kChunk) {
        const int nb = int((c + kChunk - 1) / kChunk);
        e = launch_norm(sums, c, x->norm_part(), x->sc(), 0, clip, nullptr, nullptr, nb, fz,
                        x->stream);
        if (e != cudaSuccess) return x->cuda_fail(e);
        ++x->launches;
        e = launch_norm(x->norm_part(), uint64_t(nb), nullptr, x->sc(), 1, clip, norm_out,
                        scale_out, 1, fz, x->stream, x->clip_flag_d);
    } else {
        e = launch_norm(sums, c, nullptr, x->sc(), 1, clip, norm_out, scale_out, 1, fz,
                        x->stream, x->clip_flag_d);
    }
    if (e != cudaSuccess) return x->cuda_fail(e);
    ++x->launches;
    return REPSTEP_OK;
}

int do_clip(repstep_ctx *x, float clip, float *norm_out, float *scale_out)
{
    if (!(clip > 0.0f)) return REPSTEP_ERR_ARG;   // also rejects NaN; +inf is allowed
    if (norm_out && !aligned(norm_out, 4)) return REPSTEP_ERR_ALIGN;
    if (scale_out && !aligned(scale_out, 4)) return REPSTEP_ERR_ALIGN;
    if (x->reduced != x->n) return REPSTEP_ERR_STATE;
    const int fz = x->fz();
    clip = hflush(fz, clip);
    cudaError_t e;
    unique_sort(x->cut_norm);
    for (size_t i = 0; i < x->cut_norm.size(); i += kFixMax) {
        const int cnt = int(x->cut_norm.size() - i < size_t(kFixMax) ? x->cut_norm.size() - i : kFixMax);
        e = launch_chunk_fix(x->g(), x->n, x->chunk_sq(), x->cut_norm.data() + i, cnt, fz,
                             x->stream);
        if (e != cudaSuccess) return x->cuda_fail(e);
        ++x->launches;
    }
    x->cut_norm.clear();
    const int rc = norm_passes(x, x->chunk_sq(), x->c, clip, norm_out, scale_out);
    if (rc) return rc;
    x->reduced = 0;
    x->scale_ready = true;
    x->updated = 0;
    x->cut_leaf.clear();
    x->sw = x->sm = x->sv = nullptr;
    return REPSTEP_OK;
}

// The hyperparameters of an AdamW launch and the constants derived from them, each
// operation flushed in the flush-to-zero mode like every device operation.
void adamw_hparams(const repstep_ctx *x, const repstep_hparams *hp, AdamwArgs &a)
{
    const int fz = x->fz();
    a.lr = hflush(fz, hp->lr);
    a.beta1 = hflush(fz, hp->beta1);
    a.beta2 = hflush(fz, hp->beta2);
    a.eps = hflush(fz, hp->eps);
    a.bc1 = hflush(fz, hp->bc1);
    a.bc2 = hflush(fz, hp->bc2);
    const float one = 1.0f;
    a.om1 = hflush(fz, one - a.beta1);
    a.om2 = hflush(fz, one - a.beta2);
    const float lrwd = hmul(fz, a.lr, hflush(fz, hp->weight_decay));
    a.delta = hflush(fz, one - lrwd);
    // reciprocals of the bias corrections for the fixed-divisor division in k_adamw
    a.rbc1 = one / a.bc1;
    a.rbc2 = one / a.bc2;
    // the branch-free divisions and square roots of k_adamw hold for bias corrections in
    // [2^-40, 2] and eps in [2^-40, 2^20]; otherwise every element takes the IEEE path
    const float lo = std::ldexp(1.0f, -40), hi = 2.0f, eps_hi = std::ldexp(1.0f, 20);
    a.fastdiv = (a.bc1 >= lo && a.bc1 <= hi && a.bc2 >= lo && a.bc2 <= hi && a.eps >= lo &&
                 a.eps <= eps_hi) ? 1 : 0;
}

// AdamW over [begin, begin+count): reads w, m, v and writes w', m', v' to wo, mo, vo (the
// same arrays for the in-place update).  gate: kGateIfClipped in the single-pass step,
// where the kernel returns at once when the pass already wrote the update; the call-order
// state moves on either way.
int do_adamw_to(repstep_ctx *x, void *w, float *m, float *v, void *wo, float *mo, float *vo,
                const repstep_hparams *hp, uint64_t begin, uint64_t count,
                int gate = kGateAlways)
{
    if (x->n > 0 && (!w || !m || !v || !wo || !mo || !vo)) return REPSTEP_ERR_ARG;
    if (!aligned(w, 16) || !aligned(m, 16) || !aligned(v, 16) || !aligned(wo, 16) ||
        !aligned(mo, 16) || !aligned(vo, 16))
        return REPSTEP_ERR_ALIGN;
    int rc = check_hparams(hp);
    if (rc) return rc;
    if (begin > x->n || count > x->n - begin) return REPSTEP_ERR_ARG;
    if (!x->scale_ready) return REPSTEP_ERR_STATE;
    // a pending audit-mode root reads the state; the bf16-parameter kernel hands out
    // chunks by CTA index (see do_reduce)
    rc = x->w_bf16() ? join_hash(x) : join_hash_for_update(x, wo, mo, vo);
    if (rc) return rc;
    // the state the root hashes is the one written
    if (x->sw && (x->sw != wo || x->sm != mo || x->sv != vo)) return REPSTEP_ERR_ARG;
    x->sw = wo;
    x->sm = mo;
    x->sv = vo;
    x->updated += count;
    if (count == 0) return REPSTEP_OK;
    const uint64_t end = begin + count;
    AdamwArgs a{};
    a.g = x->g();
    a.w = w;
    a.m = m;
    a.v = v;
    a.wo = wo;
    a.mo = mo;
    a.vo = vo;
    a.gate = gate;
    a.leaves = x->leaves();
    a.powers = x->powers();
    a.sc = x->sc();
    a.n = x->n;
    a.c = x->c;
    a.begin = begin;
    a.end = end;
    a.chunk_lo = begin / kChunk;
    a.chunk_hi = (end + kChunk - 1) / kChunk;
    adamw_hparams(x, hp, a);
    a.decay_mask = x->decay_mask;
    const int nt = x->nt_adamw;
    // PF61 mode: AdamW fused with the leaf digests; audit mode: AdamW alone (the BLAKE2b
    // leaves are computed from the final state by repstep_root)
    const int mode = x->cfg.hash_mode == REPSTEP_HASH_BLAKE2B ? 2 : 0;
    const AdamwShape shape{nt, mode, x->w_bf16(), x->fz(), a.decay_mask ? 1 : 0};
    const size_t smem = adamw_smem_bytes(shape, a);
    cudaError_t e = adamw_prepare(shape, smem);
    if (e != cudaSuccess) return x->cuda_fail(e);
    int bps = 1;
    e = adamw_occupancy(shape, smem, &bps);
    if (e != cudaSuccess) return x->cuda_fail(e);
    const int grid = grid_for(x, bps, a.chunk_hi - a.chunk_lo);
    e = launch_adamw(shape, a, grid, smem, x->stream);
    if (e != cudaSuccess) return x->cuda_fail(e);
    ++x->launches;
    if (mode == 0) note_cut_chunks(x->cut_leaf, begin, end, x->n);
    return REPSTEP_OK;
}

int do_adamw(repstep_ctx *x, void *w, float *m, float *v, const repstep_hparams *hp,
             uint64_t begin, uint64_t count)
{
    return do_adamw_to(x, w, m, v, w, m, v, hp, begin, count);
}

// Merkle root over the leaves.  In the PF61 mode the first Merkle pass computes the header
// leaf itself; in the audit mode the leaf kernel has already written it.
// The Merkle passes over L leaves (the first pass also writes the PF61 header leaf of
// {step, n32} to leaves[0] in the PF61 mode) until one block remains: its root goes to the
// context's scalars and to root_out.
int merkle_over(repstep_ctx *x, uint64_t *leaves, uint64_t L, int32_t step, uint32_t n32,
                uint64_t *root_out, cudaStream_t st, int header = -1)
{
    const uint64_t mb1 = (L + kMerkleBlock - 1) / kMerkleBlock;
    // passes until one block remains; the block roots alternate between two regions (the
    // second pass's roots fit the second region, and every later pass's fit either)
    uint64_t *part[2] = {x->merkle_part(), x->merkle_part() + mb1};
    const uint64_t *in = leaves;
    uint64_t count = L;
    if (header < 0) header = x->cfg.hash_mode == REPSTEP_HASH_PF61 ? 1 : 0;
    for (int pass = 0;; ++pass) {
        const uint64_t nb = (count + kMerkleBlock - 1) / kMerkleBlock;
        const bool last = nb == 1;
        uint64_t *out = last ? nullptr : part[pass & 1];
        cudaError_t e = launch_merkle(in, count, out, header, leaves, uint32_t(step), n32,
                                      x->powers(), x->sc(), last ? root_out : nullptr, int(nb),
                                      st);
        if (e != cudaSuccess) return x->cuda_fail(e);
        ++x->launches;
        if (last) return REPSTEP_OK;
        in = out;
        count = nb;
        header = 0;
    }
}

int merkle(repstep_ctx *x, int32_t step, uint64_t *root_out, cudaStream_t st)
{
    return merkle_over(x, x->leaves(), 1 + 3 * x->c, step, uint32_t(x->n), root_out, st);
}

// Audit mode: BLAKE2b-64 leaves of the whole state (header included).
int audit_leaves(repstep_ctx *x, int32_t step, const void *w, const float *m, const float *v,
                 cudaStream_t st)
{
    cudaError_t e = launch_leaves_b2(w, x->w_bf16(), m, v, x->n, x->c, x->leaves(), uint32_t(step),
                                     x->sm_count, st);
    if (e != cudaSuccess) return x->cuda_fail(e);
    ++x->launches;
    return REPSTEP_OK;
}

int root_passes(repstep_ctx *x, int32_t step, uint64_t *root_out, cudaStream_t st);
int leaf_fixups(repstep_ctx *x, cudaStream_t st);

int do_root(repstep_ctx *x, int32_t step, uint64_t *root_out)
{
    if (root_out && !aligned(root_out, 8)) return REPSTEP_ERR_ALIGN;
    if (!x->scale_ready || x->updated != x->n) return REPSTEP_ERR_STATE;
    int rc = join_hash(x);
    if (rc) return rc;
    if (!x->hash_stream) return root_passes(x, step, root_out, x->stream);
    const bool pf61 = x->cfg.hash_mode == REPSTEP_HASH_PF61;
    if (pf61) {
        // the leaf array is completed on the context's stream (leaf fix-ups, header leaf)
        // and copied; the Merkle passes read the copy, so the next update, which rewrites
        // the leaves, need not wait for them
        rc = leaf_fixups(x, x->stream);
        if (rc) return rc;
        cudaError_t e = launch_header_leaf(x->leaves(), step, uint32_t(x->n), x->powers(),
                                           x->stream);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(x->leaf_snap(), x->leaves(), 8 * (1 + 3 * x->c),
                                cudaMemcpyDeviceToDevice, x->stream);
        if (e != cudaSuccess) return x->cuda_fail(e);
        ++x->launches;
    }
    // the passes wait for the work on the context's stream, then run on the hash stream;
    // the context's stream goes on without them (join_hash orders later writers)
    cudaError_t e = cudaEventRecord(x->ev_state, x->stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(x->hash_stream, x->ev_state, 0);
    if (e != cudaSuccess) return x->cuda_fail(e);
    if (!pf61) {          // the state the audit-mode leaves read
        x->hash_st[0] = x->sw;
        x->hash_st[1] = x->sm;
        x->hash_st[2] = x->sv;
        x->hash_st_bytes[0] = x->w_bytes();
        x->hash_st_bytes[1] = x->hash_st_bytes[2] = 4 * x->n;
    }
    rc = pf61 ? merkle_over(x, x->leaf_snap(), 1 + 3 * x->c, step, uint32_t(x->n), root_out,
                            x->hash_stream, 0)
              : root_passes(x, step, root_out, x->hash_stream);
    if (rc) return rc;
    e = cudaEventRecord(x->ev_hash, x->hash_stream);
    if (e != cudaSuccess) return x->cuda_fail(e);
    x->hash_pending = true;
    x->hash_reads_live = !pf61;
    return REPSTEP_OK;
}

// The leaf fix-ups (or the audit-mode leaves) and the Merkle passes of repstep_root, on st.
int root_passes(repstep_ctx *x, int32_t step, uint64_t *root_out, cudaStream_t st)
{
    if (x->cfg.hash_mode == REPSTEP_HASH_BLAKE2B) {
        x->cut_leaf.clear();
        int rc = audit_leaves(x, step, x->sw, x->sm, x->sv, st);
        if (rc) return rc;
        return merkle(x, step, root_out, st);
    }
    const int rc = leaf_fixups(x, st);
    return rc ? rc : merkle(x, step, root_out, st);
}

// PF61 mode: recompute the leaves of the chunks the AdamW ranges cut, on st.
int leaf_fixups(repstep_ctx *x, cudaStream_t st)
{
    unique_sort(x->cut_leaf);
    for (size_t i = 0; i < x->cut_leaf.size(); i += kFixMax) {
        const int cnt = int(x->cut_leaf.size() - i < size_t(kFixMax) ? x->cut_leaf.size() - i : kFixMax);
        cudaError_t e = launch_leaf_fix(x->sw, x->w_bf16(), x->sm, x->sv, x->n, x->c, x->leaves(),
                                        x->powers(),
                                        x->cut_leaf.data() + i, cnt, st);
        if (e != cudaSuccess) return x->cuda_fail(e);
        ++x->launches;
    }
    x->cut_leaf.clear();
    return REPSTEP_OK;
}

// The leaves of (step, w, m, v) into the workspace, on the context's stream: all 1 + 3c in
// the audit mode; in the PF61 mode the chunk leaves only (the header leaf is the first
// Merkle pass's, or the caller's to add).
int hash_leaves(repstep_ctx *x, int32_t step, const void *w, const float *m, const float *v)
{
    if (x->n > 0 && (!w || !m || !v)) return REPSTEP_ERR_ARG;   // n = 0 reads no array
    if (!aligned(w, 16) || !aligned(m, 16) || !aligned(v, 16)) return REPSTEP_ERR_ALIGN;
    int rc = join_hash(x);
    if (rc) return rc;
    if (x->cfg.hash_mode == REPSTEP_HASH_BLAKE2B) return audit_leaves(x, step, w, m, v, x->stream);
    if (x->n > 0) {
        AdamwArgs a{};
        a.w = a.wo = const_cast<void *>(w);
        a.m = a.mo = const_cast<float *>(m);
        a.v = a.vo = const_cast<float *>(v);
        a.leaves = x->leaves();
        a.powers = x->powers();
        a.sc = x->sc();
        a.n = x->n;
        a.c = x->c;
        a.begin = 0;
        a.end = x->n;
        a.chunk_lo = 0;
        a.chunk_hi = x->c;
        // the leaves-only mode reads bits and does no float arithmetic: one variant
        const AdamwShape shape{x->nt_adamw, 1, x->w_bf16(), 0, 0};
        const size_t smem = adamw_smem_bytes(shape, a);
        cudaError_t e = adamw_prepare(shape, smem);
        if (e != cudaSuccess) return x->cuda_fail(e);
        int bps = 1;
        e = adamw_occupancy(shape, smem, &bps);
        if (e != cudaSuccess) return x->cuda_fail(e);
        e = launch_adamw(shape, a, grid_for(x, bps, x->c), smem, x->stream);
        if (e != cudaSuccess) return x->cuda_fail(e);
        ++x->launches;
    }
    return REPSTEP_OK;
}

int do_hash(repstep_ctx *x, int32_t step, const void *w, const float *m, const float *v,
            uint64_t *root_out)
{
    if (root_out && !aligned(root_out, 8)) return REPSTEP_ERR_ALIGN;
    const int rc = hash_leaves(x, step, w, m, v);
    if (rc) return rc;
    return merkle(x, step, root_out, x->stream);
}

int do_leaves(repstep_ctx *x, int32_t step, const void *w, const float *m, const float *v)
{
    const int rc = hash_leaves(x, step, w, m, v);
    if (rc || x->cfg.hash_mode == REPSTEP_HASH_BLAKE2B) return rc;
    const cudaError_t e = launch_header_leaf(x->leaves(), step, uint32_t(x->n), x->powers(), x->stream);
    if (e != cudaSuccess) return x->cuda_fail(e);
    ++x->launches;
    return REPSTEP_OK;
}

// ---- bf16 parameters in the fp32 image -------------------------------------------------
// The image always holds w as fp32 words.  A bf16 value widens exactly (its bits are the
// top half of the fp32 word); an fp32 word narrows back only when its low half is zero.

// n bf16 values sit at p + 2n; widen them into the fp32 words at p, in place.  Going
// upward, word i overwrites bytes [4i, 4i+4), which hold only bf16 values of index <= i,
// all of them read already.
void widen_bf16_in_place(unsigned char *p, uint64_t n)
{
    for (uint64_t i = 0; i < n; ++i) {
        uint16_t h;
        std::memcpy(&h, p + 2 * n + 2 * i, 2);
        const uint32_t u = uint32_t(h) << 16;
        std::memcpy(p + 4 * i, &u, 4);
    }
}

// fp32 words at p narrowed to bf16 at p, in place (value i moves from 4i to 2i, below it).
void narrow_bf16_in_place(unsigned char *p, uint64_t n)
{
    for (uint64_t i = 0; i < n; ++i) {
        uint32_t u;
        std::memcpy(&u, p + 4 * i, 4);
        const uint16_t h = uint16_t(u >> 16);
        std::memcpy(p + 2 * i, &h, 2);
    }
}

bool all_bf16_exact(const unsigned char *p, uint64_t n)
{
    for (uint64_t i = 0; i < n; ++i) {
        uint32_t u;
        std::memcpy(&u, p + 4 * i, 4);
        if (u & 0xFFFFu) return false;
    }
    return true;
}

constexpr uint64_t kIoChunk = 64ull << 20;   // bytes per staged host transfer

struct PinnedBuf {
    void *p = nullptr;
    ~PinnedBuf()
    {
        if (p) cudaFreeHost(p);
    }
};

// Host fp32 words (checked exact by the caller) -> device bf16, through a pinned buffer;
// synchronous on the context's stream.
cudaError_t narrow_host_to_device(repstep_ctx *x, unsigned short *d_w, const unsigned char *src,
                                  uint64_t n)
{
    PinnedBuf buf;
    cudaError_t e = cudaMallocHost(&buf.p, kIoChunk);
    if (e != cudaSuccess) return e;
    unsigned char *b = static_cast<unsigned char *>(buf.p);
    const uint64_t per = kIoChunk / 4;
    for (uint64_t i = 0; i < n; i += per) {
        const uint64_t cnt = n - i < per ? n - i : per;
        std::memcpy(b, src + 4 * i, 4 * cnt);
        narrow_bf16_in_place(b, cnt);
        e = cudaMemcpyAsync(d_w + i, b, 2 * cnt, cudaMemcpyHostToDevice, x->stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(x->stream);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// One whole step: validate everything, then reduce -> clip -> AdamW -> root.
int do_step(repstep_ctx *x, const void *const *grads, uint32_t R, uint32_t nodes, uint32_t gpn,
            void *w, float *m, float *v, const repstep_hparams *hp, int32_t step,
            float *norm_out, uint64_t *root_out)
{
    // validate everything before launching anything
    if (x->n > 0 && (!w || !m || !v)) return REPSTEP_ERR_ARG;
    if (!aligned(w, 16) || !aligned(m, 16) || !aligned(v, 16)) return REPSTEP_ERR_ALIGN;
    int rc = check_hparams(hp);
    if (rc) return rc;
    if (!(hp->clip > 0.0f)) return REPSTEP_ERR_ARG;
    if (norm_out && !aligned(norm_out, 4)) return REPSTEP_ERR_ALIGN;
    if (root_out && !aligned(root_out, 8)) return REPSTEP_ERR_ALIGN;
    x->reduced = 0;
    x->cut_norm.clear();
    rc = do_reduce(x, grads, R, nodes, gpn, 0, x->n);
    if (rc) return rc;
    rc = do_clip(x, hp->clip, norm_out, nullptr);
    if (rc) return rc;
    rc = do_adamw(x, w, m, v, hp, 0, x->n);
    if (rc) return rc;
    return do_root(x, step, root_out);
}

// Copy streams and events of repstep_step_from_host, created once per context.
int ensure_copy_resources(repstep_ctx *x)
{
    cudaError_t e = cudaSuccess;
    if (!x->ev_free) e = cudaEventCreateWithFlags(&x->ev_free, cudaEventDisableTiming);
    for (uint32_t k = 0; e == cudaSuccess && k < kMaxCopyStreams; ++k)
        if (!x->copy_st[k]) e = cudaStreamCreateWithFlags(&x->copy_st[k], cudaStreamNonBlocking);
    if (e == cudaSuccess && x->copy_ev.empty()) {
        x->copy_ev.assign(size_t(kMaxPieces) * kMaxCopyStreams, nullptr);
        for (cudaEvent_t &ev : x->copy_ev) {
            e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
            if (e != cudaSuccess) break;
        }
    }
    return e == cudaSuccess ? REPSTEP_OK : x->cuda_fail(e);
}

// One step whose gradients start in host memory: the parameter range is cut into `pieces`
// chunk-aligned ranges; range p of replica r is copied host-to-device into d_staging[r] on
// copy stream r mod K, and the reduce of range p waits for exactly those copies, so it runs
// while later ranges are still crossing the host link.  Then clip, AdamW and the root, as
// in do_step.  A range split that follows the chunk grid gives the bits of one reduce.
int step_from_host(repstep_ctx *x, const void *const *h_grads, uint32_t R,
                   void *const *d_staging, uint32_t pieces, uint32_t copy_streams, void *w,
                   float *m, float *v, const repstep_hparams *hp, int32_t step,
                   float *h_norm_out, uint64_t *h_root_out)
{
    // validate everything before enqueuing anything
    if (!h_grads || !d_staging || R == 0) return REPSTEP_ERR_ARG;
    if (R > kMaxReplicas) return REPSTEP_ERR_SIZE;
    if (pieces > kMaxPieces || copy_streams > kMaxCopyStreams) return REPSTEP_ERR_ARG;
    if (!w || !m || !v) return REPSTEP_ERR_ARG;
    if (!aligned(w, 16) || !aligned(m, 16) || !aligned(v, 16)) return REPSTEP_ERR_ALIGN;
    for (uint32_t r = 0; r < R; ++r) {
        if (!h_grads[r] || !d_staging[r]) return REPSTEP_ERR_ARG;
        if (!aligned(d_staging[r], 16)) return REPSTEP_ERR_ALIGN;
    }
    int rc = check_hparams(hp);
    if (rc) return rc;
    if (!(hp->clip > 0.0f)) return REPSTEP_ERR_ARG;
    rc = ensure_copy_resources(x);
    if (rc) return rc;
    const uint32_t P = pieces ? pieces : 8;
    uint32_t K = copy_streams ? copy_streams : 2;
    if (K > R) K = R;
    const uint64_t esz = x->cfg.grad_dtype == REPSTEP_BF16 ? 2 : 4;
    uint64_t per = (x->n + P - 1) / P;
    per = (per + kChunk - 1) / kChunk * kChunk;
    if (per == 0) per = kChunk;

    // the copies overwrite the staging buffers: after the work already on the context's
    // stream (an earlier step's reduce reads them)
    cudaError_t e = cudaEventRecord(x->ev_free, x->stream);
    for (uint32_t k = 0; e == cudaSuccess && k < K; ++k)
        e = cudaStreamWaitEvent(x->copy_st[k], x->ev_free, 0);
    if (e != cudaSuccess) return x->cuda_fail(e);
    x->reduced = 0;
    x->cut_norm.clear();
    if (x->n == 0) {
        rc = do_reduce(x, d_staging, R, 1, R, 0, 0);
        if (rc) return rc;
    }
    uint32_t p = 0;
    for (uint64_t lo = 0; lo < x->n; lo += per, ++p) {
        const uint64_t hi = lo + per < x->n ? lo + per : x->n;
        for (uint32_t r = 0; r < R; ++r) {
            e = cudaMemcpyAsync(static_cast<unsigned char *>(d_staging[r]) + lo * esz,
                                static_cast<const unsigned char *>(h_grads[r]) + lo * esz,
                                (hi - lo) * esz, cudaMemcpyHostToDevice, x->copy_st[r % K]);
            if (e != cudaSuccess) return x->cuda_fail(e);
        }
        for (uint32_t k = 0; k < K; ++k) {
            cudaEvent_t ev = x->copy_ev[size_t(p) * kMaxCopyStreams + k];
            e = cudaEventRecord(ev, x->copy_st[k]);
            if (e == cudaSuccess) e = cudaStreamWaitEvent(x->stream, ev, 0);
            if (e != cudaSuccess) return x->cuda_fail(e);
        }
        rc = do_reduce(x, d_staging, R, 1, R, lo, hi - lo);
        if (rc) return rc;
    }
    rc = do_clip(x, hp->clip, nullptr, nullptr);
    if (rc) return rc;
    rc = do_adamw(x, w, m, v, hp, 0, x->n);
    if (rc) return rc;
    rc = do_root(x, step, nullptr);
    if (rc) return rc;
    if (!h_norm_out && !h_root_out) return REPSTEP_OK;
    // the results to the host: the root may still be running on the hash stream
    rc = join_hash(x);
    if (rc) return rc;
    if (h_norm_out) e = cudaMemcpyAsync(h_norm_out, &x->sc()->norm, sizeof(float),
                                        cudaMemcpyDeviceToHost, x->stream);
    if (e == cudaSuccess && h_root_out)
        e = cudaMemcpyAsync(h_root_out, &x->sc()->root, sizeof(uint64_t), cudaMemcpyDeviceToHost,
                            x->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(x->stream);
    return e == cudaSuccess ? REPSTEP_OK : x->cuda_fail(e);
}

// Whether [a, a+na) and [b, b+nb) share a byte.
bool overlaps(const void *a, uint64_t na, const void *b, uint64_t nb)
{
    const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return na && nb && pa < pb + nb && pb < pa + na;
}

// The speculative single-pass step (k_fused.cuh) where its kernel covers the configuration:
// R = 4, 8 or 16 and the default launch shape (any gradient and parameter dtype,
// arithmetic mode, decay mask and hash mode).  Elsewhere the same result
// comes from the ordinary passes, with AdamW writing the second state buffer.
bool fused_supported(const repstep_ctx *x, uint32_t R)
{
    return (R == 4 || R == 8 || R == 16) && x->cfg.grid_blocks == 0 &&
           (x->cfg.block_threads == 0 || x->cfg.block_threads == 512) && x->n > 0;
}

// Arguments of the single-pass step, checked before anything is launched.
int check_fused_args(const repstep_ctx *x, const void *const *grads, uint32_t R,
                     const void *w, const float *m, const float *v, const void *wo,
                     const float *mo, const float *vo, const repstep_hparams *hp)
{
    if (!grads || R == 0) return REPSTEP_ERR_ARG;
    if (R > uint32_t(kMaxReplicas)) return REPSTEP_ERR_SIZE;
    if (x->n > 0 && (!w || !m || !v || !wo || !mo || !vo)) return REPSTEP_ERR_ARG;
    if (!aligned(w, 16) || !aligned(m, 16) || !aligned(v, 16) || !aligned(wo, 16) ||
        !aligned(mo, 16) || !aligned(vo, 16))
        return REPSTEP_ERR_ALIGN;
    for (uint32_t r = 0; r < R && x->n > 0; ++r) {
        if (!grads[r]) return REPSTEP_ERR_ARG;
        if (!aligned(grads[r], 16)) return REPSTEP_ERR_ALIGN;
    }
    // the input state must survive the first pass: no output may share a byte with it
    const uint64_t wb = x->w_bytes(), fb = 4 * x->n;
    const void *ins[3] = {w, m, v};
    const uint64_t in_bytes[3] = {wb, fb, fb};
    const void *outs[3] = {wo, mo, vo};
    for (int i = 0; i < 3; ++i)
        for (int j = 0; j < 3; ++j)
            if (overlaps(ins[i], in_bytes[i], outs[j], in_bytes[j])) return REPSTEP_ERR_ARG;
    const int rc = check_hparams(hp);
    if (rc) return rc;
    return hp->clip > 0.0f ? REPSTEP_OK : REPSTEP_ERR_ARG;
}

// The first half of the single-pass step: the single pass when the last clip outcome the
// host can see did not clip, else the reduce of the two passes; either leaves the chunk
// sums for a clip (repstep_clip, or repstep_clip_gathered over every shard's).  The
// outcome is read without waiting: when the GPU is behind, it is an older step's, which
// only costs time, never bits.  Configurations the single pass does not cover run the
// reduce.
int fused_begin(repstep_ctx *x, const void *const *grads, uint32_t R, const void *w,
                const float *m, const float *v, void *wo, float *mo, float *vo,
                const repstep_hparams *hp)
{
    int rc = check_fused_args(x, grads, R, w, m, v, wo, mo, vo, hp);
    if (rc) return rc;
    const bool predict_clip = x->clip_flag_h && *static_cast<volatile uint32_t *>(x->clip_flag_h);
    const bool single = fused_supported(x, R) && !predict_clip;
    x->fused = repstep_ctx::FusedCall{};
    if (!single) {
        x->reduced = 0;
        x->cut_norm.clear();
        rc = do_reduce(x, grads, R, 1, R, 0, x->n);
        if (rc) return rc;
    } else {
        rc = join_hash_for_update(x, wo, mo, vo);   // an audit-mode root reads its state
        if (rc) return rc;
        FusedArgs f{};
        for (uint32_t r = 0; r < R; ++r) f.grads[r] = grads[r];
        f.chunk_sq = x->chunk_sq();
        f.R = R;
        const float one = 1.0f;
        f.rho = hflush(x->fz(), one / float(R));
        AdamwArgs &a = f.adam;
        a.w = const_cast<void *>(w);
        a.m = const_cast<float *>(m);
        a.v = const_cast<float *>(v);
        a.wo = wo;
        a.mo = mo;
        a.vo = vo;
        a.leaves = x->leaves();
        a.powers = x->powers();
        a.sc = x->sc();
        a.n = x->n;
        a.c = x->c;
        a.begin = 0;
        a.end = x->n;
        a.chunk_lo = 0;
        a.chunk_hi = x->c;
        adamw_hparams(x, hp, a);
        a.decay_mask = x->decay_mask;
        const FusedShape shape{x->cfg.grad_dtype == REPSTEP_BF16 ? 1 : 0, int(R),
                               x->cfg.hash_mode == REPSTEP_HASH_PF61 ? 1 : 0, x->w_bf16(),
                               x->fz(), x->decay_mask ? 1 : 0};
        const size_t smem = fused_smem_bytes(shape, f);
        cudaError_t e = fused_prepare(shape, smem);
        if (e != cudaSuccess) return x->cuda_fail(e);
        int bps = 1;
        e = fused_occupancy(shape, smem, &bps);
        if (e != cudaSuccess) return x->cuda_fail(e);
        e = launch_fused(shape, f, grid_for(x, bps, x->c), smem, x->stream, x->pass_ev[0],
                         x->pass_ev[1]);
        if (e != cudaSuccess) return x->cuda_fail(e);
        ++x->launches;
        // the call-order state of a finished reduce over [0, n)
        x->reduced = x->n;
        x->cut_norm.clear();
        x->scale_ready = false;
        x->updated = 0;
        x->cut_leaf.clear();
    }
    // what the second half must be called with
    x->fused.open = true;
    x->fused.single = single;
    x->fused.R = R;
    for (uint32_t r = 0; r < R && r < 16; ++r) x->fused.g[r] = grads[r];
    x->fused.st[0] = w;
    x->fused.st[1] = m;
    x->fused.st[2] = v;
    x->fused.st[3] = wo;
    x->fused.st[4] = mo;
    x->fused.st[5] = vo;
    return REPSTEP_OK;
}

// The second half, after the clip: when the single pass ran and the scale is not 1, g
// again from the gradients; then, unless the single pass wrote the update, AdamW from the
// untouched input state into the output state, with its leaves.
int fused_end(repstep_ctx *x, const void *const *grads, uint32_t R, const void *w,
              const float *m, const float *v, void *wo, float *mo, float *vo,
              const repstep_hparams *hp)
{
    int rc = check_fused_args(x, grads, R, w, m, v, wo, mo, vo, hp);
    if (rc) return rc;
    const repstep_ctx::FusedCall &fc = x->fused;
    bool same = fc.open && fc.R == R && fc.st[0] == w && fc.st[1] == m && fc.st[2] == v &&
                fc.st[3] == wo && fc.st[4] == mo && fc.st[5] == vo;
    for (uint32_t r = 0; same && r < R && r < 16; ++r) same = fc.g[r] == grads[r];
    if (!same || !x->scale_ready) return REPSTEP_ERR_STATE;
    void *w_in = const_cast<void *>(w);
    float *m_in = const_cast<float *>(m), *v_in = const_cast<float *>(v);
    x->fused.open = false;
    if (!fc.single) return do_adamw_to(x, w_in, m_in, v_in, wo, mo, vo, hp, 0, x->n);
    rc = do_reduce(x, grads, R, 1, R, 0, x->n, 0, 0, kGateIfClipped);
    if (rc) return rc;
    return do_adamw_to(x, w_in, m_in, v_in, wo, mo, vo, hp, 0, x->n, kGateIfClipped);
}

int step_fused(repstep_ctx *x, const void *const *grads, uint32_t R, const void *w,
               const float *m, const float *v, void *wo, float *mo, float *vo,
               const repstep_hparams *hp, int32_t step, float *norm_out, uint64_t *root_out)
{
    // validate everything before launching anything
    int rc = check_fused_args(x, grads, R, w, m, v, wo, mo, vo, hp);
    if (rc) return rc;
    if (norm_out && !aligned(norm_out, 4)) return REPSTEP_ERR_ALIGN;
    if (root_out && !aligned(root_out, 8)) return REPSTEP_ERR_ALIGN;
    rc = fused_begin(x, grads, R, w, m, v, wo, mo, vo, hp);
    if (!rc) rc = do_clip(x, hp->clip, norm_out, nullptr);
    if (!rc) rc = fused_end(x, grads, R, w, m, v, wo, mo, vo, hp);
    return rc ? rc : do_root(x, step, root_out);
}

// Sharded steps.  The norm and clip scale from the chunk sums of every shard, gathered by
// the caller into one array in chunk order; the local reduce must have covered this
// context's range along the chunk grid (its own chunk sums complete).
int clip_gathered(repstep_ctx *x, const float *sums, uint64_t c_total, float clip,
                  float *norm_out, float *scale_out)
{
    if (!(clip > 0.0f)) return REPSTEP_ERR_ARG;
    if (!sums && c_total > 0) return REPSTEP_ERR_ARG;
    if (c_total > (uint64_t(1) << 20)) return REPSTEP_ERR_SIZE;
    if (c_total < x->c) return REPSTEP_ERR_ARG;
    if (!aligned(sums, 4)) return REPSTEP_ERR_ALIGN;
    if (norm_out && !aligned(norm_out, 4)) return REPSTEP_ERR_ALIGN;
    if (scale_out && !aligned(scale_out, 4)) return REPSTEP_ERR_ALIGN;
    if (x->reduced != x->n || !x->cut_norm.empty()) return REPSTEP_ERR_STATE;
    const int rc = norm_passes(x, sums, c_total, hflush(x->fz(), clip), norm_out, scale_out);
    if (rc) return rc;
    x->reduced = 0;
    x->scale_ready = true;
    x->updated = 0;
    x->cut_leaf.clear();
    x->sw = x->sm = x->sv = nullptr;
    return REPSTEP_OK;
}

// The Merkle root over the leaves of every shard, gathered by the caller into
// leaves[1 .. 3 c_total] in image order; leaves[0] receives the header leaf of
// (step, n_total).  The local AdamW must have covered this context's range along the chunk
// grid (so its own chunk leaves were complete when they were gathered).
int root_gathered(repstep_ctx *x, int32_t step, uint64_t n_total, uint64_t *leaves,
                  uint64_t *root_out)
{
    if (!leaves) return REPSTEP_ERR_ARG;
    if (!aligned(leaves, 8) || (root_out && !aligned(root_out, 8))) return REPSTEP_ERR_ALIGN;
    if (n_total > 0xFFFFFFFFull) return REPSTEP_ERR_SIZE;
    if (n_total < x->n) return REPSTEP_ERR_ARG;
    if (!x->scale_ready || x->updated != x->n || !x->cut_leaf.empty()) return REPSTEP_ERR_STATE;
    int rc = join_hash(x);
    if (rc) return rc;
    const uint64_t c_total = (n_total + kChunk - 1) / kChunk;
    if (x->cfg.hash_mode == REPSTEP_HASH_BLAKE2B) {
        // the BLAKE2b-64 header leaf alone: the leaf kernel with no chunks
        const cudaError_t e = launch_leaves_b2(nullptr, 0, nullptr, nullptr, n_total, 0, leaves,
                                               uint32_t(step), x->sm_count, x->stream);
        if (e != cudaSuccess) return x->cuda_fail(e);
        ++x->launches;
    }
    return merkle_over(x, leaves, 1 + 3 * c_total, step, uint32_t(n_total), root_out,
                       x->stream);
}

}  // namespace

extern "C" {

size_t repstep_workspace_bytes(const repstep_config *cfg)
{
    if (!valid_config(cfg)) return 0;
    return size_t(layout_of(cfg->n).total);
}

int repstep_workspace_layout(const repstep_config *cfg, repstep_layout *out)
{
    if (!valid_config(cfg) || !out) return REPSTEP_ERR_ARG;
    const Layout l = layout_of(cfg->n);
    out->g = l.g;
    out->chunk_sums = l.chunk_sq;
    out->norm_partials = l.norm_part;
    out->leaves = l.leaves;
    out->merkle_partials = l.merkle_part;
    out->pow_table = l.powers;
    out->scalars = l.scalars;
    out->total = l.total;
    return REPSTEP_OK;
}

int repstep_create(const repstep_config *cfg, void *d_workspace, size_t workspace_bytes,
                   void *stream, repstep_ctx **out)
{
    if (!out) return REPSTEP_ERR_ARG;
    *out = nullptr;
    if (!cfg || !d_workspace) return REPSTEP_ERR_ARG;
    if (!valid_config(cfg)) return cfg->n > 0xFFFFFFFFull ? REPSTEP_ERR_SIZE : REPSTEP_ERR_ARG;
    if (!aligned(d_workspace, kAlign)) return REPSTEP_ERR_ALIGN;
    const Layout lay = layout_of(cfg->n);
    if (workspace_bytes < lay.total) return REPSTEP_ERR_SIZE;
    repstep_ctx *x = new (std::nothrow) repstep_ctx();
    if (!x) return REPSTEP_ERR_ARG;
    x->cfg = *cfg;
    x->lay = lay;
    x->ws = static_cast<unsigned char *>(d_workspace);
    x->stream = static_cast<cudaStream_t>(stream);
    x->n = cfg->n;
    x->c = (cfg->n + kChunk - 1) / kChunk;
    x->nt_reduce = cfg->block_threads ? cfg->block_threads : 512;
    x->nt_adamw = cfg->block_threads ? cfg->block_threads : 512;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&x->sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = merkle_prepare();
    if (e == cudaSuccess) e = leaves_b2_prepare();
    if (e == cudaSuccess) {
        // the host-visible clip outcome (pinned host memory: no device allocation)
        void *h = nullptr;
        if (cudaHostAlloc(&h, sizeof(uint32_t), cudaHostAllocMapped) == cudaSuccess) {
            *static_cast<volatile uint32_t *>(h) = 0;
            void *d = nullptr;
            if (cudaHostGetDevicePointer(&d, h, 0) == cudaSuccess) {
                x->clip_flag_h = static_cast<uint32_t *>(h);
                x->clip_flag_d = static_cast<uint32_t *>(d);
            } else {
                cudaFreeHost(h);
            }
        }
        cudaGetLastError();   // a device without mapped host memory: no prediction
    }
    if (e == cudaSuccess) e = cudaMemsetAsync(x->ws + lay.scalars, 0, sizeof(Scalars), x->stream);
    if (e == cudaSuccess) e = launch_init_powers(x->powers(), x->stream);
    if (e != cudaSuccess) {
        delete x;
        return REPSTEP_ERR_CUDA;
    }
    x->launches = 1;
    *out = x;
    return REPSTEP_OK;
}

int repstep_destroy(repstep_ctx *ctx)
{
    if (!ctx) return REPSTEP_ERR_ARG;
    if (ctx->clip_flag_h) {
        // a norm pass still queued may store the clip outcome into the mapped word
        cudaStreamSynchronize(ctx->stream);
        cudaFreeHost(ctx->clip_flag_h);
    }
    if (ctx->ev_state) cudaEventDestroy(ctx->ev_state);
    if (ctx->ev_hash) cudaEventDestroy(ctx->ev_hash);
    if (ctx->ev_free) cudaEventDestroy(ctx->ev_free);
    for (cudaEvent_t ev : ctx->copy_ev)
        if (ev) cudaEventDestroy(ev);
    for (cudaStream_t st : ctx->copy_st)
        if (st) cudaStreamDestroy(st);
    delete ctx;
    return REPSTEP_OK;
}

int repstep_set_hash_stream(repstep_ctx *ctx, void *hash_stream)
{
    if (!ctx) return REPSTEP_ERR_ARG;
    if (hash_stream && !ctx->ev_state) {
        cudaError_t e = cudaEventCreateWithFlags(&ctx->ev_state, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ctx->ev_hash, cudaEventDisableTiming);
        if (e != cudaSuccess) return ctx->cuda_fail(e);
    }
    ctx->hash_stream = static_cast<cudaStream_t>(hash_stream);
    return REPSTEP_OK;
}

int repstep_set_pass_events(repstep_ctx *ctx, void *ev_begin, void *ev_end)
{
    if (!ctx || (!ev_begin) != (!ev_end)) return REPSTEP_ERR_ARG;
    ctx->pass_ev[0] = static_cast<cudaEvent_t>(ev_begin);
    ctx->pass_ev[1] = static_cast<cudaEvent_t>(ev_end);
    return REPSTEP_OK;
}

int repstep_wait_hash(repstep_ctx *ctx, void *stream)
{
    if (!ctx) return REPSTEP_ERR_ARG;
    if (!ctx->hash_pending) return REPSTEP_OK;
    const cudaError_t e = cudaStreamWaitEvent(static_cast<cudaStream_t>(stream), ctx->ev_hash, 0);
    return e == cudaSuccess ? REPSTEP_OK : ctx->cuda_fail(e);
}

int repstep_set_stream(repstep_ctx *ctx, void *stream)
{
    if (!ctx) return REPSTEP_ERR_ARG;
    ctx->stream = static_cast<cudaStream_t>(stream);
    return REPSTEP_OK;
}

int repstep_reduce(repstep_ctx *ctx, const void *const *d_grads, uint32_t R, uint32_t nodes,
                   uint32_t gpus_per_node, uint64_t begin, uint64_t count)
{
    const NvtxRange nvtx_("repstep_reduce");
    if (!ctx) return REPSTEP_ERR_ARG;
    return do_reduce(ctx, d_grads, R, nodes, gpus_per_node, begin, count);
}

int repstep_reduce_paper(repstep_ctx *ctx, const void *const *d_grads, uint32_t R,
                         uint32_t dp_shard, uint64_t begin, uint64_t count)
{
    const NvtxRange nvtx_("repstep_reduce_paper");
    if (!ctx) return REPSTEP_ERR_ARG;
    if (dp_shard == 0 || R % dp_shard != 0) return REPSTEP_ERR_TOPOLOGY;
    return do_reduce(ctx, d_grads, R, R / dp_shard, dp_shard, begin, count, 1);
}

int repstep_reduce_paper_accum(repstep_ctx *ctx, const void *const *d_grads, uint32_t R,
                               uint32_t dp_shard, uint32_t accum, uint64_t begin, uint64_t count)
{
    const NvtxRange nvtx_("repstep_reduce_paper_accum");
    if (!ctx) return REPSTEP_ERR_ARG;
    if (accum == 0) return REPSTEP_ERR_ARG;
    if (dp_shard == 0 || R % dp_shard != 0) return REPSTEP_ERR_TOPOLOGY;
    return do_reduce(ctx, d_grads, R, R / dp_shard, dp_shard, begin, count, 1, accum);
}

int repstep_clip(repstep_ctx *ctx, float clip, float *d_norm_out, float *d_scale_out)
{
    const NvtxRange nvtx_("repstep_clip");
    if (!ctx) return REPSTEP_ERR_ARG;
    return do_clip(ctx, clip, d_norm_out, d_scale_out);
}

int repstep_adamw(repstep_ctx *ctx, void *d_w, float *d_m, float *d_v, const repstep_hparams *hp,
                  uint64_t begin, uint64_t count)
{
    const NvtxRange nvtx_("repstep_adamw");
    if (!ctx) return REPSTEP_ERR_ARG;
    return do_adamw(ctx, d_w, d_m, d_v, hp, begin, count);
}

int repstep_root(repstep_ctx *ctx, int32_t step, uint64_t *d_root_out)
{
    const NvtxRange nvtx_("repstep_root");
    if (!ctx) return REPSTEP_ERR_ARG;
    return do_root(ctx, step, d_root_out);
}

int repstep_leaves(repstep_ctx *ctx, int32_t step, const void *d_w, const float *d_m,
                   const float *d_v)
{
    const NvtxRange nvtx_("repstep_leaves");
    if (!ctx) return REPSTEP_ERR_ARG;
    return do_leaves(ctx, step, d_w, d_m, d_v);
}

int repstep_hash(repstep_ctx *ctx, int32_t step, const void *d_w, const float *d_m,
                 const float *d_v, uint64_t *d_root_out)
{
    const NvtxRange nvtx_("repstep_hash");
    if (!ctx) return REPSTEP_ERR_ARG;
    return do_hash(ctx, step, d_w, d_m, d_v, d_root_out);
}

int repstep_step(repstep_ctx *ctx, const void *const *d_grads, uint32_t R, uint32_t nodes,
                 uint32_t gpus_per_node, void *d_w, float *d_m, float *d_v,
                 const repstep_hparams *hp, int32_t step, float *d_norm_out, uint64_t *d_root_out)
{
    const NvtxRange nvtx_("repstep_step");
    if (!ctx) return REPSTEP_ERR_ARG;
    return do_step(ctx, d_grads, R, nodes, gpus_per_node, d_w, d_m, d_v, hp, step, d_norm_out,
                   d_root_out);
}

int repstep_step_from_host(repstep_ctx *ctx, const void *const *h_grads, uint32_t R,
                           void *const *d_staging, uint32_t pieces, uint32_t copy_streams,
                           void *d_w, float *d_m, float *d_v, const repstep_hparams *hp,
                           int32_t step, float *h_norm_out, uint64_t *h_root_out)
{
    const NvtxRange nvtx_("repstep_step_from_host");
    if (!ctx) return REPSTEP_ERR_ARG;
    return step_from_host(ctx, h_grads, R, d_staging, pieces, copy_streams, d_w, d_m, d_v, hp,
                          step, h_norm_out, h_root_out);
}

int repstep_step_fused(repstep_ctx *ctx, const void *const *d_grads, uint32_t R,
                       const void *d_w, const float *d_m, const float *d_v, void *d_w_out,
                       float *d_m_out, float *d_v_out, const repstep_hparams *hp, int32_t step,
                       float *d_norm_out, uint64_t *d_root_out)
{
    const NvtxRange nvtx_("repstep_step_fused");
    if (!ctx) return REPSTEP_ERR_ARG;
    return step_fused(ctx, d_grads, R, d_w, d_m, d_v, d_w_out, d_m_out, d_v_out, hp, step,
                      d_norm_out, d_root_out);
}

int repstep_fused_begin(repstep_ctx *ctx, const void *const *d_grads, uint32_t R,
                        const void *d_w, const float *d_m, const float *d_v, void *d_w_out,
                        float *d_m_out, float *d_v_out, const repstep_hparams *hp)
{
    const NvtxRange nvtx_("repstep_fused_begin");
    if (!ctx) return REPSTEP_ERR_ARG;
    return fused_begin(ctx, d_grads, R, d_w, d_m, d_v, d_w_out, d_m_out, d_v_out, hp);
}

int repstep_fused_end(repstep_ctx *ctx, const void *const *d_grads, uint32_t R,
                      const void *d_w, const float *d_m, const float *d_v, void *d_w_out,
                      float *d_m_out, float *d_v_out, const repstep_hparams *hp)
{
    const NvtxRange nvtx_("repstep_fused_end");
    if (!ctx) return REPSTEP_ERR_ARG;
    return fused_end(ctx, d_grads, R, d_w, d_m, d_v, d_w_out, d_m_out, d_v_out, hp);
}

int repstep_clip_gathered(repstep_ctx *ctx, const float *d_chunk_sums, uint64_t c_total,
                          float clip, float *d_norm_out, float *d_scale_out)
{
    const NvtxRange nvtx_("repstep_clip_gathered");
    if (!ctx) return REPSTEP_ERR_ARG;
    return clip_gathered(ctx, d_chunk_sums, c_total, clip, d_norm_out, d_scale_out);
}

int repstep_root_gathered(repstep_ctx *ctx, int32_t step, uint64_t n_total, uint64_t *d_leaves,
                          uint64_t *d_root_out)
{
    const NvtxRange nvtx_("repstep_root_gathered");
    if (!ctx) return REPSTEP_ERR_ARG;
    return root_gathered(ctx, step, n_total, d_leaves, d_root_out);
}

int repstep_set_decay_mask(repstep_ctx *ctx, const uint32_t *d_mask)
{
    if (!ctx) return REPSTEP_ERR_ARG;
    if (d_mask && !aligned(d_mask, 16)) return REPSTEP_ERR_ALIGN;
    ctx->decay_mask = d_mask;
    return REPSTEP_OK;
}

int repstep_decay_mask_from_segments(uint64_t n, const uint64_t *seg_begin, const uint8_t *decay,
                                     uint32_t count, uint32_t *h_mask)
{
    if (count > 0 && (!seg_begin || !decay)) return REPSTEP_ERR_ARG;
    if (n > 0 && !h_mask) return REPSTEP_ERR_ARG;
    if (count == 0) return n == 0 ? REPSTEP_OK : REPSTEP_ERR_ARG;
    if (seg_begin[0] != 0) return REPSTEP_ERR_ARG;
    for (uint32_t s = 1; s < count; ++s)
        if (seg_begin[s] <= seg_begin[s - 1] || seg_begin[s] >= n) return REPSTEP_ERR_ARG;
    const uint64_t words = (n + 31) / 32;
    std::memset(h_mask, 0, words * sizeof(uint32_t));
    for (uint32_t s = 0; s < count; ++s) {
        if (!decay[s]) continue;
        const uint64_t lo = seg_begin[s], hi = s + 1 < count ? seg_begin[s + 1] : n;
        uint64_t e = lo;
        for (; e < hi && (e & 31); ++e) h_mask[e >> 5] |= 1u << (e & 31);      // head bits
        for (; e + 32 <= hi; e += 32) h_mask[e >> 5] = 0xFFFFFFFFu;             // whole words
        for (; e < hi; ++e) h_mask[e >> 5] |= 1u << (e & 31);                  // tail bits
    }
    return REPSTEP_OK;
}

uint64_t repstep_image_bytes(uint64_t n) { return 8 + 12 * n; }

int repstep_image_write(repstep_ctx *ctx, int32_t step, const void *d_w, const float *d_m,
                        const float *d_v, void *dst, uint64_t dst_bytes, int dst_is_host)
{
    const NvtxRange nvtx_("repstep_image_write");
    if (!ctx || !d_w || !d_m || !d_v || !dst) return REPSTEP_ERR_ARG;
    const uint64_t n = ctx->n;
    if (dst_bytes < repstep_image_bytes(n)) return REPSTEP_ERR_SIZE;
    unsigned char *d = static_cast<unsigned char *>(dst);
    cudaError_t e;
    const cudaMemcpyKind kind = dst_is_host ? cudaMemcpyDeviceToHost : cudaMemcpyDeviceToDevice;
    if (dst_is_host) {
        const uint32_t h[2] = {uint32_t(step), uint32_t(n)};
        std::memcpy(d, h, 8);   // the header is little-endian on every supported host
    } else {
        if (!aligned(dst, 4)) return REPSTEP_ERR_ALIGN;
        e = launch_write_header(dst, step, uint32_t(n), ctx->stream);
        if (e != cudaSuccess) return ctx->cuda_fail(e);
        ++ctx->launches;
    }
    if (n == 0) return REPSTEP_OK;
    // w: fp32 bytes as they are, or bf16 widened exactly to fp32
    if (!ctx->w_bf16()) {
        e = cudaMemcpyAsync(d + 8, d_w, 4 * n, kind, ctx->stream);
    } else if (!dst_is_host) {
        e = launch_widen_bf16(reinterpret_cast<float *>(d + 8),
                              static_cast<const unsigned short *>(d_w), n, ctx->stream);
        ++ctx->launches;
    } else {
        // the bf16 values land in the upper half of the image's w region and are widened in
        // place on the host (synchronous)
        e = cudaMemcpyAsync(d + 8 + 2 * n, d_w, 2 * n, cudaMemcpyDeviceToHost, ctx->stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(ctx->stream);
        if (e == cudaSuccess) widen_bf16_in_place(d + 8, n);
    }
    if (e != cudaSuccess) return ctx->cuda_fail(e);
    const float *arrs[2] = {d_m, d_v};
    for (int a = 0; a < 2; ++a) {
        e = cudaMemcpyAsync(d + 8 + uint64_t(a + 1) * 4 * n, arrs[a], 4 * n, kind, ctx->stream);
        if (e != cudaSuccess) return ctx->cuda_fail(e);
    }
    return REPSTEP_OK;
}

int repstep_image_read(repstep_ctx *ctx, const void *src, uint64_t src_bytes, int src_is_host,
                       int32_t *step_out, void *d_w, float *d_m, float *d_v)
{
    const NvtxRange nvtx_("repstep_image_read");
    if (!ctx || !src || !d_w || !d_m || !d_v) return REPSTEP_ERR_ARG;
    const uint64_t n = ctx->n;
    if (src_bytes != repstep_image_bytes(n)) return REPSTEP_ERR_FORMAT;
    uint32_t h[2];
    cudaError_t e;
    if (src_is_host) {
        std::memcpy(h, src, 8);
    } else {
        e = cudaMemcpyAsync(h, src, 8, cudaMemcpyDeviceToHost, ctx->stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(ctx->stream);
        if (e != cudaSuccess) return ctx->cuda_fail(e);
    }
    if (uint64_t(h[1]) != n) return REPSTEP_ERR_FORMAT;
    int rc = join_hash(ctx);      // a pending root may still read the state
    if (rc) return rc;
    const unsigned char *s = static_cast<const unsigned char *>(src);
    // bf16 parameters: every w word of the image must be a bf16 value exactly; checked
    // before anything is copied
    if (ctx->w_bf16() && n > 0) {
        bool exact = true;
        if (src_is_host) {
            exact = all_bf16_exact(s + 8, n);
        } else {
            if (!aligned(src, 4)) return REPSTEP_ERR_ALIGN;
            uint32_t bad = 0;
            Scalars *sc = ctx->sc();
            e = cudaMemsetAsync(&sc->aux, 0, sizeof(uint32_t), ctx->stream);
            if (e == cudaSuccess)
                e = launch_narrow_bf16(nullptr, reinterpret_cast<const float *>(s + 8), n, &sc->aux,
                                       ctx->stream);
            if (e == cudaSuccess)
                e = cudaMemcpyAsync(&bad, &sc->aux, sizeof bad, cudaMemcpyDeviceToHost, ctx->stream);
            if (e == cudaSuccess) e = cudaStreamSynchronize(ctx->stream);
            if (e != cudaSuccess) return ctx->cuda_fail(e);
            ++ctx->launches;
            exact = bad == 0;
        }
        if (!exact) return REPSTEP_ERR_FORMAT;
    }
    if (step_out) *step_out = int32_t(h[0]);
    if (n == 0) return REPSTEP_OK;
    const cudaMemcpyKind kind = src_is_host ? cudaMemcpyHostToDevice : cudaMemcpyDeviceToDevice;
    if (!ctx->w_bf16()) {
        e = cudaMemcpyAsync(d_w, s + 8, 4 * n, kind, ctx->stream);
    } else if (!src_is_host) {
        e = launch_narrow_bf16(static_cast<unsigned short *>(d_w),
                               reinterpret_cast<const float *>(s + 8), n, nullptr, ctx->stream);
        ++ctx->launches;
    } else {
        e = narrow_host_to_device(ctx, static_cast<unsigned short *>(d_w), s + 8, n);
    }
    if (e != cudaSuccess) return ctx->cuda_fail(e);
    float *arrs[2] = {d_m, d_v};
    for (int a = 0; a < 2; ++a) {
        e = cudaMemcpyAsync(arrs[a], s + 8 + uint64_t(a + 1) * 4 * n, 4 * n, kind, ctx->stream);
        if (e != cudaSuccess) return ctx->cuda_fail(e);
    }
    return REPSTEP_OK;
}

// ----------------------------------------------------------------------------------------
// Checkpoint files: the image streamed between the device arrays and a file through one
// reusable pinned host buffer ("grow_a_language_model_checkpoints": step_NNNNNN.bin).
// ----------------------------------------------------------------------------------------
int repstep_checkpoint_save(repstep_ctx *ctx, const char *path, int32_t step, const void *d_w,
                            const float *d_m, const float *d_v)
{
    const NvtxRange nvtx_("repstep_checkpoint_save");
    if (!ctx || !path || !d_w || !d_m || !d_v) return REPSTEP_ERR_ARG;
    const uint64_t n = ctx->n;
    const std::string tmp = std::string(path) + ".tmp";
    FILE *f = std::fopen(tmp.c_str(), "wb");
    if (!f) return REPSTEP_ERR_ARG;
    int rc = REPSTEP_OK;
    const uint32_t header[2] = {uint32_t(step), uint32_t(n)};   // little-endian hosts
    if (std::fwrite(header, 4, 2, f) != 2) rc = REPSTEP_ERR_ARG;
    PinnedBuf buf;
    if (rc == REPSTEP_OK && n > 0) {
        cudaError_t e = cudaMallocHost(&buf.p, kIoChunk);
        if (e != cudaSuccess) rc = ctx->cuda_fail(e);
    }
    if (ctx->w_bf16() && rc == REPSTEP_OK) {
        // bf16 w: each piece lands in the upper half of the buffer and is widened in place
        unsigned char *b = static_cast<unsigned char *>(buf.p);
        const unsigned short *w16 = static_cast<const unsigned short *>(d_w);
        const uint64_t per = kIoChunk / 4;
        for (uint64_t i = 0; i < n && rc == REPSTEP_OK; i += per) {
            const uint64_t cnt = n - i < per ? n - i : per;
            cudaError_t e = cudaMemcpyAsync(b + 2 * cnt, w16 + i, 2 * cnt, cudaMemcpyDeviceToHost,
                                            ctx->stream);
            if (e == cudaSuccess) e = cudaStreamSynchronize(ctx->stream);
            if (e != cudaSuccess) {
                rc = ctx->cuda_fail(e);
                break;
            }
            widen_bf16_in_place(b, cnt);
            if (std::fwrite(b, 1, 4 * cnt, f) != 4 * cnt) rc = REPSTEP_ERR_ARG;
        }
    }
    const void *arrs[3] = {d_w, d_m, d_v};
    for (int a = ctx->w_bf16() ? 1 : 0; a < 3 && rc == REPSTEP_OK; ++a) {
        const unsigned char *src = static_cast<const unsigned char *>(arrs[a]);
        for (uint64_t off = 0; off < 4 * n && rc == REPSTEP_OK; off += kIoChunk) {
            const uint64_t len = 4 * n - off < kIoChunk ? 4 * n - off : kIoChunk;
            cudaError_t e = cudaMemcpyAsync(buf.p, src + off, len, cudaMemcpyDeviceToHost,
                                            ctx->stream);
            if (e == cudaSuccess) e = cudaStreamSynchronize(ctx->stream);
            if (e != cudaSuccess) rc = ctx->cuda_fail(e);
            else if (std::fwrite(buf.p, 1, len, f) != len) rc = REPSTEP_ERR_ARG;
        }
    }
    if (std::fclose(f) != 0 && rc == REPSTEP_OK) rc = REPSTEP_ERR_ARG;
    if (rc == REPSTEP_OK && std::rename(tmp.c_str(), path) != 0) rc = REPSTEP_ERR_ARG;
    if (rc != REPSTEP_OK) std::remove(tmp.c_str());
    return rc;
}

int repstep_checkpoint_load(repstep_ctx *ctx, const char *path, int32_t *step_out, void *d_w,
                            float *d_m, float *d_v)
{
    const NvtxRange nvtx_("repstep_checkpoint_load");
    if (!ctx || !path || !d_w || !d_m || !d_v) return REPSTEP_ERR_ARG;
    const uint64_t n = ctx->n;
    FILE *f = std::fopen(path, "rb");
    if (!f) return REPSTEP_ERR_ARG;
    // guards first, before anything is copied: exact size, then the header's n
    int rc = REPSTEP_OK;
    if (std::fseek(f, 0, SEEK_END) != 0) rc = REPSTEP_ERR_FORMAT;
    const long long size = rc == REPSTEP_OK ? std::ftell(f) : -1;
    if (size < 0 || uint64_t(size) != repstep_image_bytes(n)) rc = REPSTEP_ERR_FORMAT;
    uint32_t header[2] = {0, 0};
    if (rc == REPSTEP_OK && (std::fseek(f, 0, SEEK_SET) != 0 || std::fread(header, 4, 2, f) != 2))
        rc = REPSTEP_ERR_FORMAT;
    if (rc == REPSTEP_OK && uint64_t(header[1]) != n) rc = REPSTEP_ERR_FORMAT;
    if (rc == REPSTEP_OK) rc = join_hash(ctx);      // a pending root may still read the state
    PinnedBuf buf;
    if (rc == REPSTEP_OK && n > 0) {
        cudaError_t e = cudaMallocHost(&buf.p, kIoChunk);
        if (e != cudaSuccess) rc = ctx->cuda_fail(e);
    }
    unsigned char *b = static_cast<unsigned char *>(buf.p);
    if (ctx->w_bf16() && rc == REPSTEP_OK && n > 0) {
        // bf16 parameters: first a pass over the file's w words -- each must be a bf16
        // value exactly -- so that nothing is copied from an image that cannot be loaded
        for (uint64_t off = 0; off < 4 * n && rc == REPSTEP_OK; off += kIoChunk) {
            const uint64_t len = 4 * n - off < kIoChunk ? 4 * n - off : kIoChunk;
            if (std::fread(b, 1, len, f) != len || !all_bf16_exact(b, len / 4))
                rc = REPSTEP_ERR_FORMAT;
        }
        if (rc == REPSTEP_OK && std::fseek(f, 8, SEEK_SET) != 0) rc = REPSTEP_ERR_FORMAT;
        unsigned short *w16 = static_cast<unsigned short *>(d_w);
        const uint64_t per = kIoChunk / 4;
        for (uint64_t i = 0; i < n && rc == REPSTEP_OK; i += per) {
            const uint64_t cnt = n - i < per ? n - i : per;
            if (std::fread(b, 1, 4 * cnt, f) != 4 * cnt) {
                rc = REPSTEP_ERR_FORMAT;
                break;
            }
            narrow_bf16_in_place(b, cnt);
            cudaError_t e = cudaMemcpyAsync(w16 + i, b, 2 * cnt, cudaMemcpyHostToDevice,
                                            ctx->stream);
            if (e == cudaSuccess) e = cudaStreamSynchronize(ctx->stream);
            if (e != cudaSuccess) rc = ctx->cuda_fail(e);
        }
    }
    void *arrs[3] = {d_w, d_m, d_v};
    for (int a = ctx->w_bf16() ? 1 : 0; a < 3 && rc == REPSTEP_OK; ++a) {
        unsigned char *dst = static_cast<unsigned char *>(arrs[a]);
        for (uint64_t off = 0; off < 4 * n && rc == REPSTEP_OK; off += kIoChunk) {
            const uint64_t len = 4 * n - off < kIoChunk ? 4 * n - off : kIoChunk;
            if (std::fread(buf.p, 1, len, f) != len) {
                rc = REPSTEP_ERR_FORMAT;
                break;
            }
            cudaError_t e = cudaMemcpyAsync(dst + off, buf.p, len, cudaMemcpyHostToDevice,
                                            ctx->stream);
            if (e == cudaSuccess) e = cudaStreamSynchronize(ctx->stream);
            if (e != cudaSuccess) rc = ctx->cuda_fail(e);
        }
    }
    std::fclose(f);
    if (rc == REPSTEP_OK && step_out) *step_out = int32_t(header[0]);
    return rc;
}

void repstep_bias_corrections(float beta1, float beta2, int32_t t, float *bc1, float *bc2)
{
    float p1 = 1.0f, p2 = 1.0f;
    for (int32_t j = 0; j < t; ++j) {
        p1 = p1 * beta1;
        p2 = p2 * beta2;
    }
    const float one = 1.0f;
    if (bc1) *bc1 = one - p1;
    if (bc2) *bc2 = one - p2;
}

int repstep_sync(repstep_ctx *ctx, uint32_t *flags_out)
{
    if (!ctx) return REPSTEP_ERR_ARG;
    cudaError_t e = cudaStreamSynchronize(ctx->stream);
    if (e == cudaSuccess && ctx->hash_pending) e = cudaEventSynchronize(ctx->ev_hash);
    if (e != cudaSuccess) return ctx->cuda_fail(e);
    ctx->hash_pending = false;
    Scalars s;
    e = cudaMemcpy(&s, ctx->sc(), sizeof s, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return ctx->cuda_fail(e);
    if (flags_out) *flags_out = s.flags;
    const uint32_t timeouts = kFlagTimeoutReduce | kFlagTimeoutAdamw | kFlagTimeoutLeaves;
    if (s.flags & timeouts) {
        const uint32_t keep = s.flags & ~timeouts;
        e = cudaMemcpy(&ctx->sc()->flags, &keep, sizeof keep, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return ctx->cuda_fail(e);
        return REPSTEP_ERR_TIMEOUT;
    }
    return REPSTEP_OK;
}

int repstep_selftest_fixed_division(uint32_t b_sig_begin, uint32_t b_sig_count,
                                    uint64_t *d_mismatches, void *stream)
{
    if (!d_mismatches || !aligned(d_mismatches, 8)) return REPSTEP_ERR_ARG;
    if (b_sig_begin > (1u << 23) || b_sig_count > (1u << 23) - b_sig_begin) return REPSTEP_ERR_ARG;
    if (b_sig_count == 0) return REPSTEP_OK;
    const cudaError_t e = launch_selftest_div(b_sig_begin, b_sig_count,
                                              reinterpret_cast<unsigned long long *>(d_mismatches),
                                              static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? REPSTEP_OK : REPSTEP_ERR_CUDA;
}

uint64_t repstep_launch_count(const repstep_ctx *ctx) { return ctx ? ctx->launches : 0; }

int repstep_selftest_fast_math(int which, uint32_t begin, uint32_t count, uint64_t seed,
                               uint64_t *d_mismatches, void *stream)
{
    if (!d_mismatches || !aligned(d_mismatches, 8)) return REPSTEP_ERR_ARG;
    if (which < 0 || which > 2) return REPSTEP_ERR_ARG;
    if (which < 2 && uint64_t(begin) + count > (1ull << 32)) return REPSTEP_ERR_ARG;
    if (count == 0) return REPSTEP_OK;
    const cudaError_t e = launch_selftest_fast_math(
        which, begin, count, seed, reinterpret_cast<unsigned long long *>(d_mismatches),
        static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? REPSTEP_OK : REPSTEP_ERR_CUDA;
}

int repstep_last_cuda_error(const repstep_ctx *ctx) { return ctx ? ctx->last_err : 0; }

const char *repstep_strerror(int code)
{
    switch (code) {
    case REPSTEP_OK: return "ok";
    case REPSTEP_ERR_ARG: return "invalid argument";
    case REPSTEP_ERR_ALIGN: return "misaligned device pointer";
    case REPSTEP_ERR_SIZE: return "size out of range";
    case REPSTEP_ERR_TOPOLOGY: return "replica topology breaks the canonical tree";
    case REPSTEP_ERR_CUDA: return "CUDA runtime error";
    case REPSTEP_ERR_TIMEOUT: return "a kernel wait timed out";
    case REPSTEP_ERR_STATE: return "call order violated";
    case REPSTEP_ERR_FORMAT: return "bad checkpoint image";
    default: return "unknown status";
    }
}

}  // extern "C"
