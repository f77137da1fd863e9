// noalloc.cu -- replica reduce + global norm for callers that cannot allocate device memory.
//
// Who needs this: a process that must compute the averaged gradient and its pre-clip norm
// but is not allowed to allocate device memory at that point.  Examples: an audit replay
// that runs beside a training job whose caching allocator has already reserved nearly all
// of the GPU's memory; a checkpoint-on-signal or error path entered after an out-of-memory
// condition; a host framework that forbids cudaMalloc after start-up.  The normal entry
// points need a caller-provided workspace; this one needs none.
//
// How: the scratch the reduce and norm kernels need beyond their inputs and outputs -- the
// per-chunk sums of squares, the norm partials and the device scalars -- lives in one
// file-scope __device__ array of fixed size, part of the loaded library.  Every GPU that
// loads the library holds it (about 1 MiB) until the process exits.  The kernels are the
// same ones repstep_reduce / repstep_clip launch, so the bits are the same.
#include <cstdint>
#include <mutex>

#include "../../include/repstep.h"
#include "common.cuh"
#include "kernels.h"

using namespace repstep;

namespace {

constexpr uint64_t kStaticMaxChunks = REPSTEP_NOALLOC_MAX_N / kChunk;    // 262,144
constexpr size_t kChunkSumBytes = kStaticMaxChunks * sizeof(float);      // 1 MiB
constexpr size_t kPartialOff = kChunkSumBytes;                           // norm partials
constexpr size_t kPartialBytes = 256;                                    // 64 floats
constexpr size_t kScalarOff = kPartialOff + kPartialBytes;               // device scalars
constexpr size_t kScratchBytes = kScalarOff + 256;
static_assert(kStaticMaxChunks / kChunk * sizeof(float) <= kPartialBytes, "partials fit");
static_assert(sizeof(Scalars) <= 256, "scalars fit");

// The shared scratch.  In host code this name is only a host-side stand-in, never a device
// address: host code must use the address cudaGetSymbolAddress returns for the device.
static __device__ __align__(256) unsigned char noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per device.
cudaError_t scratch_address(unsigned char **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, noalloc_scratch);
        if (e != cudaSuccess) return e;
        if (!p) return cudaErrorInvalidSymbol;
        g_scratch_addr[dev] = p;
    }
    *out = static_cast<unsigned char *>(g_scratch_addr[dev]);
    return cudaSuccess;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" int repstep_reduce_norm_noalloc(const void *const *d_grads, uint32_t R,
                                           int32_t grad_dtype, uint64_t n, float clip,
                                           float *d_g, float *d_norm_out, float *d_scale_out,
                                           void *stream)
{
    // host-side checks first: nothing is launched on a bad argument
    if (!d_grads || R == 0 || !d_g || !d_norm_out) return REPSTEP_ERR_ARG;
    if (grad_dtype != REPSTEP_F32 && grad_dtype != REPSTEP_BF16) return REPSTEP_ERR_ARG;
    if (!(clip > 0.0f)) return REPSTEP_ERR_ARG;
    if (R > REPSTEP_MAX_REPLICAS) return REPSTEP_ERR_SIZE;
    if (n > REPSTEP_NOALLOC_MAX_N) return REPSTEP_ERR_SIZE;
    if (!aligned(d_g, 16) || !aligned(d_norm_out, 4) || (d_scale_out && !aligned(d_scale_out, 4)))
        return REPSTEP_ERR_ALIGN;
    for (uint32_t r = 0; r < R; ++r) {
        if (!d_grads[r]) return REPSTEP_ERR_ARG;
        if (!aligned(d_grads[r], 16)) return REPSTEP_ERR_ALIGN;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned char *scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return REPSTEP_ERR_CUDA;
    float *chunk_sums = reinterpret_cast<float *>(scratch);
    float *partials = reinterpret_cast<float *>(scratch + kPartialOff);
    Scalars *sc = reinterpret_cast<Scalars *>(scratch + kScalarOff);

    // the scalars keep the previous call's contents: the flags must start at zero
    if (cudaMemsetAsync(sc, 0, sizeof(Scalars), st) != cudaSuccess) return REPSTEP_ERR_CUDA;

    const uint64_t c = (n + kChunk - 1) / kChunk;
    if (n > 0) {
        ReduceArgs a{};
        for (uint32_t r = 0; r < R; ++r) a.grads[r] = d_grads[r];
        a.g = d_g;
        a.chunk_sq = chunk_sums;   // every chunk of [0, n) is written: no clearing needed
        a.sc = sc;
        a.n = n;
        a.begin = 0;
        a.end = n;
        a.chunk_lo = 0;
        a.chunk_hi = c;
        a.R = R;
        a.nodes = 1;
        a.gpn = R;
        const float one = 1.0f;
        a.rho = one / float(R);
        ReduceShape s{};
        s.nt = 512;
        s.dtype = grad_dtype;
        s.mode = 0;
        s.rg = R >= 8 ? 8 : 4;
        s.maxlev = R <= 32 ? 6 : 9;
        s.fz = 0;
        const size_t smem = reduce_smem_bytes(s, a);
        if (reduce_prepare(s, smem) != cudaSuccess) return REPSTEP_ERR_CUDA;
        int bps = 1, dev = 0, sms = 1;
        if (reduce_occupancy(s, smem, &bps) != cudaSuccess) return REPSTEP_ERR_CUDA;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return REPSTEP_ERR_CUDA;
        uint64_t grid = uint64_t(sms) * uint64_t(bps > 0 ? bps : 1);
        if (grid > c) grid = c;
        if (launch_reduce(s, a, int(grid), smem, st) != cudaSuccess) return REPSTEP_ERR_CUDA;
    }
    cudaError_t e;
    if (c > kChunk) {
        const int nb = int((c + kChunk - 1) / kChunk);
        e = launch_norm(chunk_sums, c, partials, sc, 0, clip, nullptr, nullptr, nb, 0, st);
        if (e == cudaSuccess)
            e = launch_norm(partials, uint64_t(nb), nullptr, sc, 1, clip, d_norm_out, d_scale_out,
                            1, 0, st);
    } else {
        e = launch_norm(chunk_sums, c, nullptr, sc, 1, clip, d_norm_out, d_scale_out, 1, 0, st);
    }
    return e == cudaSuccess ? REPSTEP_OK : REPSTEP_ERR_CUDA;
}
