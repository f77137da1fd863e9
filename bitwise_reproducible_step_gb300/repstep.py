"""Python binding of librepstep.so (include/repstep.h): ctypes argument marshalling only.

Every step of the optimizer step runs in the library's CUDA kernels; this module checks
tensor devices, dtypes and sizes, passes raw device pointers and the current torch stream,
and turns status codes into exceptions.  There is no CPU fallback: if the library is not
built, importing the binding's functions raises.

Typical use:
    ctx = Repstep(n)                        # workspace allocated by torch on the device
    hp = hparams(lr=..., beta1=..., beta2=..., eps=..., weight_decay=..., clip=1.0, t=1)
    ctx.step(grads, w, m, v, hp, step=1, norm_out=norm, root_out=root)
"""
from __future__ import annotations

import ctypes as C
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "librepstep.so")

REPSTEP_F32 = 0
REPSTEP_BF16 = 1
CHUNK = 4096
MAX_REPLICAS = 256

FLAG_NONFINITE_NORM = 0x1
FLAG_TIMEOUT_REDUCE = 0x2
FLAG_TIMEOUT_ADAMW = 0x4
FLAG_TIMEOUT_LEAVES = 0x8

STATUS = {0: "REPSTEP_OK", 1: "REPSTEP_ERR_ARG", 2: "REPSTEP_ERR_ALIGN", 3: "REPSTEP_ERR_SIZE",
          4: "REPSTEP_ERR_TOPOLOGY", 5: "REPSTEP_ERR_CUDA", 6: "REPSTEP_ERR_TIMEOUT",
          7: "REPSTEP_ERR_STATE", 8: "REPSTEP_ERR_FORMAT"}


class Config(C.Structure):
    _fields_ = [("n", C.c_uint64), ("grad_dtype", C.c_int32), ("grid_blocks", C.c_int32),
                ("block_threads", C.c_int32), ("hash_mode", C.c_int32),
                ("param_dtype", C.c_int32), ("subnormals", C.c_int32)]


HASH_PF61 = 0
HASH_BLAKE2B = 1
SUBNORMALS_IEEE = 0
SUBNORMALS_FTZ = 1


class HParams(C.Structure):
    _fields_ = [(k, C.c_float) for k in
                ("lr", "beta1", "beta2", "eps", "weight_decay", "clip", "bc1", "bc2")]


class Layout(C.Structure):
    _fields_ = [(k, C.c_uint64) for k in
                ("g", "chunk_sums", "norm_partials", "leaves", "merkle_partials", "pow_table",
                 "scalars", "total")]


class RepstepError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        super().__init__(f"{STATUS.get(code, code)}: {strerror(code)}{(' -- ' + what) if what else ''}")


EXPORTS = [
    "repstep_workspace_bytes", "repstep_workspace_layout", "repstep_create", "repstep_destroy",
    "repstep_set_stream", "repstep_reduce", "repstep_clip", "repstep_adamw", "repstep_root",
    "repstep_hash", "repstep_step", "repstep_image_bytes", "repstep_image_write",
    "repstep_image_read", "repstep_bias_corrections", "repstep_sync", "repstep_launch_count",
    "repstep_last_cuda_error", "repstep_strerror", "repstep_reduce_norm_noalloc",
    "repstep_selftest_fixed_division", "repstep_reduce_paper", "repstep_checkpoint_save",
    "repstep_checkpoint_load", "repstep_set_decay_mask", "repstep_decay_mask_from_segments",
    "repstep_reduce_paper_accum", "repstep_set_hash_stream", "repstep_wait_hash",
    "repstep_leaves", "repstep_selftest_fast_math", "repstep_step_from_host",
    "repstep_clip_gathered", "repstep_step_fused",
    "repstep_root_gathered", "repstep_set_pass_events", "repstep_fused_begin",
    "repstep_fused_end",
]
NOALLOC_MAX_N = 1 << 30

_lib = None


def lib():
    """Load librepstep.so (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -c \"import "
                           "__graft_entry__ as g; g.build()\"` (needs nvcc)")
    L = C.CDLL(LIB_PATH)
    vp, u64, u32, i32 = C.c_void_p, C.c_uint64, C.c_uint32, C.c_int32
    L.repstep_workspace_bytes.argtypes = [C.POINTER(Config)]
    L.repstep_workspace_bytes.restype = C.c_size_t
    L.repstep_workspace_layout.argtypes = [C.POINTER(Config), C.POINTER(Layout)]
    L.repstep_create.argtypes = [C.POINTER(Config), vp, C.c_size_t, vp, C.POINTER(vp)]
    L.repstep_destroy.argtypes = [vp]
    L.repstep_set_stream.argtypes = [vp, vp]
    L.repstep_reduce.argtypes = [vp, C.POINTER(vp), u32, u32, u32, u64, u64]
    L.repstep_clip.argtypes = [vp, C.c_float, vp, vp]
    L.repstep_adamw.argtypes = [vp, vp, vp, vp, C.POINTER(HParams), u64, u64]
    L.repstep_root.argtypes = [vp, i32, vp]
    L.repstep_hash.argtypes = [vp, i32, vp, vp, vp, vp]
    L.repstep_leaves.argtypes = [vp, i32, vp, vp, vp]
    L.repstep_step.argtypes = [vp, C.POINTER(vp), u32, u32, u32, vp, vp, vp, C.POINTER(HParams),
                               i32, vp, vp]
    L.repstep_clip_gathered.argtypes = [vp, vp, u64, C.c_float, vp, vp]
    L.repstep_step_fused.argtypes = [vp, C.POINTER(vp), u32, vp, vp, vp, vp, vp, vp,
                                     C.POINTER(HParams), i32, vp, vp]
    L.repstep_root_gathered.argtypes = [vp, i32, u64, vp, vp]
    for fn in (L.repstep_fused_begin, L.repstep_fused_end):
        fn.argtypes = [vp, C.POINTER(vp), u32, vp, vp, vp, vp, vp, vp, C.POINTER(HParams)]
    L.repstep_step_from_host.argtypes = [vp, C.POINTER(vp), u32, C.POINTER(vp), u32, u32, vp, vp,
                                         vp, C.POINTER(HParams), i32, vp, vp]
    L.repstep_image_bytes.argtypes = [u64]
    L.repstep_image_bytes.restype = u64
    L.repstep_image_write.argtypes = [vp, i32, vp, vp, vp, vp, u64, C.c_int]
    L.repstep_image_read.argtypes = [vp, vp, u64, C.c_int, C.POINTER(i32), vp, vp, vp]
    L.repstep_bias_corrections.argtypes = [C.c_float, C.c_float, i32, C.POINTER(C.c_float),
                                           C.POINTER(C.c_float)]
    L.repstep_bias_corrections.restype = None
    L.repstep_sync.argtypes = [vp, C.POINTER(u32)]
    L.repstep_launch_count.argtypes = [vp]
    L.repstep_launch_count.restype = u64
    L.repstep_last_cuda_error.argtypes = [vp]
    L.repstep_strerror.argtypes = [C.c_int]
    L.repstep_strerror.restype = C.c_char_p
    L.repstep_selftest_fixed_division.argtypes = [u32, u32, vp, vp]
    L.repstep_selftest_fast_math.argtypes = [C.c_int, u32, u32, u64, vp, vp]
    L.repstep_reduce_paper.argtypes = [vp, C.POINTER(vp), u32, u32, u64, u64]
    L.repstep_checkpoint_save.argtypes = [vp, C.c_char_p, i32, vp, vp, vp]
    L.repstep_checkpoint_load.argtypes = [vp, C.c_char_p, C.POINTER(i32), vp, vp, vp]
    L.repstep_reduce_norm_noalloc.argtypes = [C.POINTER(vp), u32, i32, u64, C.c_float, vp, vp,
                                              vp, vp]
    L.repstep_set_decay_mask.argtypes = [vp, vp]
    L.repstep_set_hash_stream.argtypes = [vp, vp]
    L.repstep_set_pass_events.argtypes = [vp, vp, vp]
    L.repstep_wait_hash.argtypes = [vp, vp]
    L.repstep_reduce_paper_accum.argtypes = [vp, C.POINTER(vp), u32, u32, u32, u64, u64]
    L.repstep_decay_mask_from_segments.argtypes = [u64, vp, vp, u32, vp]
    _lib = L
    return L


def strerror(code: int) -> str:
    return lib().repstep_strerror(int(code)).decode()


def _check(rc: int, what: str = ""):
    if rc != 0:
        raise RepstepError(rc, what)


def bias_corrections(beta1: float, beta2: float, t: int):
    b1, b2 = C.c_float(), C.c_float()
    lib().repstep_bias_corrections(beta1, beta2, int(t), C.byref(b1), C.byref(b2))
    return b1.value, b2.value


def hparams(*, lr, beta1, beta2, eps, weight_decay, clip, t) -> HParams:
    """AdamW hyperparameters for step t (bias corrections from the library's host recipe)."""
    bc1, bc2 = bias_corrections(beta1, beta2, t)
    return HParams(lr, beta1, beta2, eps, weight_decay, clip, bc1, bc2)


def checkpoint_name(step: int) -> str:
    """File name of the checkpoint written after `step` ("grow_a_language_model_checkpoints":
    step_NNNNNN.bin, six digits, zero padded)."""
    if step < 0:
        raise ValueError("step must be >= 0")
    return f"step_{step:06d}.bin"


def image_bytes(n: int) -> int:
    return int(lib().repstep_image_bytes(n))


def workspace_bytes(n: int, grad_dtype=torch.float32, grid_blocks=0, block_threads=0) -> int:
    cfg = Config(n, _dtype_code(grad_dtype), grid_blocks, block_threads, 0, REPSTEP_F32, 0)
    return int(lib().repstep_workspace_bytes(C.byref(cfg)))


def _dtype_code(dt) -> int:
    if dt == torch.float32:
        return REPSTEP_F32
    if dt == torch.bfloat16:
        return REPSTEP_BF16
    raise TypeError(f"dtype {dt}: float32 or bfloat16")


def reduce_norm_noalloc(grads, clip: float, g_out: torch.Tensor, norm_out: torch.Tensor,
                        scale_out: torch.Tensor | None = None, stream=None):
    """repstep_reduce_norm_noalloc: averaged gradient and pre-clip norm using the library's
    fixed scratch array instead of a workspace (for callers that may not allocate device
    memory; n <= NOALLOC_MAX_N).  Calls whose GPU work overlaps must be serialised."""
    grads = list(grads)
    n = g_out.numel()
    dt = grads[0].dtype
    for t in grads:
        if t.dtype != dt or not t.is_cuda or not t.is_contiguous() or t.numel() < n:
            raise ValueError("gradients: contiguous CUDA tensors of one dtype, >= n elements")
    for t, want in ((g_out, torch.float32), (norm_out, torch.float32), (scale_out, torch.float32)):
        if t is not None and (t.dtype != want or not t.is_cuda):
            raise ValueError("outputs: CUDA float32 tensors")
    arr = (C.c_void_p * len(grads))(*[t.data_ptr() for t in grads])
    st = stream or torch.cuda.current_stream(g_out.device)
    _check(lib().repstep_reduce_norm_noalloc(arr, len(grads), _dtype_code(dt), n, clip,
                                             _ptr(g_out), _ptr(norm_out), _ptr(scale_out),
                                             C.c_void_p(st.cuda_stream)), "reduce_norm_noalloc")


def selftest_fixed_division(b_sig_begin: int = 0, b_sig_count: int = 1 << 23) -> int:
    """Mismatches between the AdamW kernel's fixed-divisor division and IEEE division over
    all x significands and the given b significands (see repstep_selftest_fixed_division)."""
    out = torch.zeros(1, dtype=torch.int64, device="cuda")
    _check(lib().repstep_selftest_fixed_division(b_sig_begin, b_sig_count, _ptr(out),
                                                 C.c_void_p(torch.cuda.current_stream().cuda_stream)),
           "selftest_fixed_division")
    return int(out.item())


SQRT_FAST_BITS = (0x0C800000, 0x68000000)     # [2^-102, 2^81): the fast square root's range
RCP_FAST_BITS = (0x2A800000, 0x54800000)      # [2^-42, 2^42): the fast reciprocal's range


def selftest_fast_math(which: int, begin: int = 0, count: int = 0, seed: int = 0) -> int:
    """Mismatches between the AdamW kernel's branch-free square root (which=0),
    reciprocal (1) or division (2, count x 1024 random pairs) and the IEEE operations (see
    repstep_selftest_fast_math)."""
    out = torch.zeros(1, dtype=torch.int64, device="cuda")
    _check(lib().repstep_selftest_fast_math(int(which), int(begin), int(count), int(seed),
                                            _ptr(out),
                                            C.c_void_p(torch.cuda.current_stream().cuda_stream)),
           "selftest_fast_math")
    return int(out.item())


def decay_mask_from_segments(n: int, segments) -> torch.Tensor:
    """Host int32 tensor of ceil(n/32) words: the weight-decay bitmask of a segment list
    [(begin, decays), ...] cutting [0, n) in increasing order from 0 (see
    repstep_decay_mask_from_segments).  Upload it and pass it to Repstep.set_decay_mask."""
    import numpy as np
    b = np.ascontiguousarray([int(s[0]) for s in segments] or [0], dtype=np.uint64)
    d = np.ascontiguousarray([1 if s[1] else 0 for s in segments] or [0], dtype=np.uint8)
    out = torch.zeros(max((n + 31) // 32, 1), dtype=torch.int32)
    _check(lib().repstep_decay_mask_from_segments(n, C.c_void_p(b.ctypes.data),
                                                  C.c_void_p(d.ctypes.data), len(segments),
                                                  C.c_void_p(out.data_ptr())),
           "decay_mask_from_segments")
    return out[:(n + 31) // 32]


def _ptr(t: torch.Tensor | None):
    return None if t is None else C.c_void_p(t.data_ptr())


class Repstep:
    """One context over a torch-allocated device workspace (see repstep_create)."""

    def __init__(self, n: int, grad_dtype=torch.float32, device=None, grid_blocks: int = 0,
                 block_threads: int = 0, stream: torch.cuda.Stream | None = None,
                 hash_mode: int = HASH_PF61, param_dtype=torch.float32,
                 subnormals: int = SUBNORMALS_IEEE, workspace: torch.Tensor | None = None):
        """workspace: an optional caller-owned uint8 device tensor of at least
        workspace_bytes() bytes (256-byte aligned); by default one is allocated here."""
        L = lib()
        self.n = int(n)
        self.grad_dtype = grad_dtype
        self.param_dtype = param_dtype
        self.device = torch.device("cuda", torch.cuda.current_device()) if device is None \
            else torch.device(device)
        self._fixed_stream = stream
        self.hash_mode = hash_mode
        self.subnormals = subnormals
        self.cfg = Config(self.n, _dtype_code(grad_dtype), grid_blocks, block_threads, hash_mode,
                          _dtype_code(param_dtype), subnormals)
        nbytes = int(L.repstep_workspace_bytes(C.byref(self.cfg)))
        if nbytes == 0:
            raise RepstepError(1, "bad configuration")
        self.layout = Layout()
        _check(L.repstep_workspace_layout(C.byref(self.cfg), C.byref(self.layout)))
        if workspace is None:
            workspace = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        elif (workspace.dtype != torch.uint8 or workspace.device != self.device
              or not workspace.is_contiguous() or workspace.numel() < nbytes):
            raise ValueError(f"workspace: contiguous uint8 on the context's device, at least "
                             f"{nbytes} bytes")
        self.workspace = workspace
        self._decay_mask = None
        self._hash_stream = None
        self._streams_used = {}          # cuda_stream handle -> stream, see _used_on
        self._ctx = C.c_void_p()
        _check(L.repstep_create(C.byref(self.cfg), _ptr(self.workspace), nbytes,
                                C.c_void_p(self._stream().cuda_stream), C.byref(self._ctx)))
        self._used_on(self._stream())    # the create's initialisation runs there
        self.c = (self.n + CHUNK - 1) // CHUNK

    # ---------------------------------------------------------------- plumbing
    def _stream(self):
        return self._fixed_stream or torch.cuda.current_stream(self.device)

    def _bind(self):
        if not self._ctx:
            raise RuntimeError("context destroyed")
        st = self._stream()
        self._used_on(st)
        lib().repstep_set_stream(self._ctx, C.c_void_p(st.cuda_stream))

    def _used_on(self, st):
        """Tell PyTorch's caching allocator that the device memory the library reads and
        writes for this context (the workspace, the decay mask) is used on stream `st`.
        Freeing a tensor then waits for the work enqueued on every such stream, so that a
        root still running on the hash stream, or a step on another stream than the one
        the workspace was allocated on, never writes memory handed to a new tensor."""
        if st.cuda_stream in self._streams_used:
            return
        self._streams_used[st.cuda_stream] = st
        self.workspace.record_stream(st)
        if self._decay_mask is not None:
            self._decay_mask.record_stream(st)

    def _state(self, w, m, v):
        for t, want in ((w, self.param_dtype), (m, torch.float32), (v, torch.float32)):
            if t.device != self.device or t.dtype != want or not t.is_contiguous() \
                    or t.numel() < self.n:
                raise ValueError(f"state arrays: contiguous {want} on the context's device, "
                                 f"at least n={self.n} elements")

    def _grads(self, grads):
        grads = list(grads)
        for t in grads:
            if t.device != self.device or t.dtype != self.grad_dtype or not t.is_contiguous() \
                    or t.numel() < self.n:
                raise ValueError(f"gradients: contiguous {self.grad_dtype} on the context's "
                                 f"device, at least n={self.n} elements")
        arr = (C.c_void_p * max(len(grads), 1))(*[t.data_ptr() for t in grads])
        return arr, len(grads)

    @staticmethod
    def _out(t, dtype, numel=1):
        if t is not None and (t.dtype != dtype or t.numel() < numel or not t.is_cuda):
            raise ValueError(f"output must be a CUDA {dtype} tensor")
        return _ptr(t)

    # ---------------------------------------------------------------- the C ABI
    def reduce(self, grads, nodes: int = 1, gpus_per_node: int | None = None, begin: int = 0,
               count: int | None = None):
        arr, R = self._grads(grads)
        gpn = R // max(nodes, 1) if gpus_per_node is None else gpus_per_node
        count = self.n - begin if count is None else count
        self._bind()
        _check(lib().repstep_reduce(self._ctx, arr, R, nodes, gpn, begin, count), "reduce")

    def reduce_paper(self, grads, dp_shard: int, begin: int = 0, count: int | None = None,
                     accum: int | None = None):
        """Paper-exact reduce (OPEN-1B Algorithm 1): grads are the virtual-rank gradients
        in mesh order, R = dp_replicate * dp_shard (see repstep_reduce_paper).  With
        `accum`, grads are R * accum microbatch gradients, rank-major, accumulated first
        (repstep_reduce_paper_accum)."""
        arr, R = self._grads(grads)
        count = self.n - begin if count is None else count
        self._bind()
        if accum is None:
            _check(lib().repstep_reduce_paper(self._ctx, arr, R, dp_shard, begin, count),
                   "reduce_paper")
            return
        if accum < 1 or R % accum:
            raise ValueError("the gradient count must be a multiple of accum >= 1")
        _check(lib().repstep_reduce_paper_accum(self._ctx, arr, R // accum, dp_shard, accum,
                                                begin, count), "reduce_paper_accum")

    def clip(self, clip: float, norm_out=None, scale_out=None):
        self._bind()
        _check(lib().repstep_clip(self._ctx, clip, self._out(norm_out, torch.float32),
                                  self._out(scale_out, torch.float32)), "clip")

    def clip_gathered(self, chunk_sums, clip: float, norm_out=None, scale_out=None):
        """Norm and clip scale from every range's chunk sums, gathered in chunk order (a
        CUDA fp32 tensor of ceil(n_total/4096) slots), in place of clip() in a sharded step
        (repstep_clip_gathered)."""
        if not chunk_sums.is_cuda or chunk_sums.dtype != torch.float32 \
                or not chunk_sums.is_contiguous():
            raise ValueError("chunk sums: a contiguous CUDA fp32 tensor")
        self._bind()
        _check(lib().repstep_clip_gathered(self._ctx, _ptr(chunk_sums), chunk_sums.numel(),
                                           clip, self._out(norm_out, torch.float32),
                                           self._out(scale_out, torch.float32)),
               "clip_gathered")

    def root_gathered(self, step: int, n_total: int, leaves, root_out=None):
        """Merkle root of a sharded state from every range's leaves gathered in image order
        into leaves[1:] (a CUDA int64 tensor of 1 + 3 ceil(n_total/4096) slots; slot 0
        receives the header leaf) (repstep_root_gathered)."""
        c_total = (n_total + CHUNK - 1) // CHUNK
        if not leaves.is_cuda or leaves.dtype != torch.int64 or not leaves.is_contiguous() \
                or leaves.numel() < 1 + 3 * c_total:
            raise ValueError("leaves: a contiguous CUDA int64 tensor of 1 + 3c slots")
        self._bind()
        _check(lib().repstep_root_gathered(self._ctx, int(step), n_total, _ptr(leaves),
                                           self._out(root_out, torch.int64)), "root_gathered")

    def adamw(self, w, m, v, hp: HParams, begin: int = 0, count: int | None = None):
        self._state(w, m, v)
        count = self.n - begin if count is None else count
        self._bind()
        _check(lib().repstep_adamw(self._ctx, _ptr(w), _ptr(m), _ptr(v), C.byref(hp), begin,
                                   count), "adamw")

    def root(self, step: int, root_out=None):
        self._bind()
        _check(lib().repstep_root(self._ctx, int(step), self._out(root_out, torch.int64)), "root")

    def hash(self, step: int, w, m, v, root_out=None):
        self._state(w, m, v)
        self._bind()
        _check(lib().repstep_hash(self._ctx, int(step), _ptr(w), _ptr(m), _ptr(v),
                                  self._out(root_out, torch.int64)), "hash")

    def leaves(self, step: int, w, m, v) -> torch.Tensor:
        """The hash's 1 + 3c leaf digests of (step, w, m, v), without the Merkle passes: a
        view of the workspace's leaf array (int64 bits of the u64 digests), valid until the
        next call that hashes."""
        self._state(w, m, v)
        self._bind()
        _check(lib().repstep_leaves(self._ctx, int(step), _ptr(w), _ptr(m), _ptr(v)), "leaves")
        return self.leaves_view()

    def step(self, grads, w, m, v, hp: HParams, step: int, norm_out=None, root_out=None,
             nodes: int = 1, gpus_per_node: int | None = None):
        arr, R = self._grads(grads)
        self._state(w, m, v)
        gpn = R // max(nodes, 1) if gpus_per_node is None else gpus_per_node
        self._bind()
        _check(lib().repstep_step(self._ctx, arr, R, nodes, gpn, _ptr(w), _ptr(m), _ptr(v),
                                  C.byref(hp), int(step), self._out(norm_out, torch.float32),
                                  self._out(root_out, torch.int64)), "step")

    def step_fused(self, grads, w, m, v, w_out, m_out, v_out, hp: HParams, step: int,
                   norm_out=None, root_out=None):
        """One step from (w, m, v) into (w_out, m_out, v_out), in a single HBM pass when it
        does not clip (repstep_step_fused); after a clip that clipped, in the two passes at
        once.  The inputs are left untouched and the bits equal step()'s.  Alternate the
        two state buffers from step to step."""
        arr, R = self._grads(grads)
        self._state(w, m, v)
        self._state(w_out, m_out, v_out)
        self._bind()
        _check(lib().repstep_step_fused(self._ctx, arr, R, _ptr(w), _ptr(m), _ptr(v),
                                        _ptr(w_out), _ptr(m_out), _ptr(v_out), C.byref(hp),
                                        int(step), self._out(norm_out, torch.float32),
                                        self._out(root_out, torch.int64)), "step_fused")

    def fused_begin(self, grads, w, m, v, w_out, m_out, v_out, hp: HParams):
        """The first half of step_fused (repstep_fused_begin): the single pass, or after a
        clip that clipped the reduce of the two passes; then clip() or clip_gathered(),
        then fused_end() with the same arguments."""
        arr, R = self._grads(grads)
        self._state(w, m, v)
        self._state(w_out, m_out, v_out)
        self._bind()
        _check(lib().repstep_fused_begin(self._ctx, arr, R, _ptr(w), _ptr(m), _ptr(v),
                                         _ptr(w_out), _ptr(m_out), _ptr(v_out), C.byref(hp)),
               "fused_begin")

    def fused_end(self, grads, w, m, v, w_out, m_out, v_out, hp: HParams):
        """The second half of step_fused after the clip (repstep_fused_end): the second
        pass where the clip needs one, and the AdamW of the two passes."""
        arr, R = self._grads(grads)
        self._state(w, m, v)
        self._state(w_out, m_out, v_out)
        self._bind()
        _check(lib().repstep_fused_end(self._ctx, arr, R, _ptr(w), _ptr(m), _ptr(v),
                                       _ptr(w_out), _ptr(m_out), _ptr(v_out), C.byref(hp)),
               "fused_end")

    def step_from_host(self, host_grads, staging, w, m, v, hp: HParams, step: int,
                       pieces: int = 8, copy_streams: int = 2):
        """One step whose replica gradients start in host memory (repstep_step_from_host):
        host_grads are R contiguous CPU tensors of the gradient dtype (pinned for
        asynchronous copies), staging R device buffers of n elements they are copied into.
        The library pipelines the copies over `pieces` chunk-aligned ranges and
        `copy_streams` streams, reducing each range as it lands; then clip, AdamW and the
        root.  Returns (pre-clip norm, root) read back to the host; the call returns after
        the step has finished.  Bit-identical to step() on the same gradients."""
        host_grads, staging = list(host_grads), list(staging)
        if len(host_grads) != len(staging):
            raise ValueError("one staging buffer per replica")
        for h in host_grads:
            if h.is_cuda or h.dtype != self.grad_dtype or not h.is_contiguous() \
                    or h.numel() < self.n:
                raise ValueError(f"host gradients: contiguous CPU {self.grad_dtype} tensors of "
                                 f"at least n={self.n} elements")
        arr, R = self._grads(staging)
        self._state(w, m, v)
        harr = (C.c_void_p * max(R, 1))(*[h.data_ptr() for h in host_grads])
        nrm, root = C.c_float(), C.c_uint64()
        self._bind()
        _check(lib().repstep_step_from_host(self._ctx, harr, R, arr, pieces, copy_streams,
                                            _ptr(w), _ptr(m), _ptr(v), C.byref(hp), int(step),
                                            C.byref(nrm), C.byref(root)), "step_from_host")
        return float(nrm.value), int(root.value)

    def set_hash_stream(self, stream: torch.cuda.Stream | None):
        """Run the root passes on `stream`, beside the next step's work on the context's
        stream (see repstep_set_hash_stream); None returns to one stream.  The root output
        is complete after wait_hash() or sync()."""
        _check(lib().repstep_set_hash_stream(
            self._ctx, None if stream is None else C.c_void_p(stream.cuda_stream)),
            "set_hash_stream")
        if stream is not None:
            self._used_on(stream)
        self._hash_stream = stream

    def set_pass_events(self, begin: torch.cuda.Event | None, end: torch.cuda.Event | None):
        """Record these timing events around the single pass of every step_fused() call
        while set (repstep_set_pass_events); None, None clears.  The events must have been
        recorded once, so that they exist."""
        def handle(ev):
            if ev is None:
                return None
            h = ev.cuda_event
            if not h:
                raise RepstepError(1, "record the event once before passing it")
            return C.c_void_p(h)
        _check(lib().repstep_set_pass_events(self._ctx, handle(begin), handle(end)),
               "set_pass_events")

    def wait_hash(self, stream: torch.cuda.Stream | None = None):
        """Make `stream` (default: the current stream) wait for the pending root passes."""
        st = stream or torch.cuda.current_stream(self.device)
        _check(lib().repstep_wait_hash(self._ctx, C.c_void_p(st.cuda_stream)), "wait_hash")

    def set_decay_mask(self, mask: torch.Tensor | None):
        """Per-element weight decay for later adamw/step calls: a CUDA int32 tensor of
        ceil(n/32) words from decay_mask_from_segments (bit set = decays), or None for
        decay everywhere.  The context keeps a reference to the tensor."""
        if mask is not None and (not mask.is_cuda or mask.dtype != torch.int32
                                 or not mask.is_contiguous() or mask.numel() < (self.n + 31) // 32
                                 or mask.device != self.device):
            raise ValueError("decay mask: contiguous CUDA int32 on the context's device, "
                             "ceil(n/32) words")
        _check(lib().repstep_set_decay_mask(self._ctx, _ptr(mask)), "set_decay_mask")
        if mask is not None:
            for st in self._streams_used.values():
                mask.record_stream(st)
        self._decay_mask = mask

    def image_write(self, step: int, w, m, v, dst: torch.Tensor):
        self._state(w, m, v)
        if dst.dtype != torch.uint8 or not dst.is_contiguous():
            raise ValueError("image buffer: contiguous uint8")
        self._bind()
        _check(lib().repstep_image_write(self._ctx, int(step), _ptr(w), _ptr(m), _ptr(v),
                                         _ptr(dst), dst.numel(), 0 if dst.is_cuda else 1),
               "image_write")

    def image_read(self, src: torch.Tensor, w, m, v) -> int:
        self._state(w, m, v)
        if src.dtype != torch.uint8 or not src.is_contiguous():
            raise ValueError("image buffer: contiguous uint8")
        step = C.c_int32()
        self._bind()
        _check(lib().repstep_image_read(self._ctx, _ptr(src), src.numel(), 0 if src.is_cuda else 1,
                                        C.byref(step), _ptr(w), _ptr(m), _ptr(v)), "image_read")
        return int(step.value)

    def save_checkpoint(self, path: str, step: int, w, m, v):
        """Write the 8 + 12n-byte image of (step, w, m, v) to `path` (atomic rename)."""
        self._state(w, m, v)
        self._bind()
        _check(lib().repstep_checkpoint_save(self._ctx, os.fsencode(path), int(step), _ptr(w),
                                             _ptr(m), _ptr(v)), "checkpoint_save")

    def load_checkpoint(self, path: str, w, m, v) -> int:
        """Load an image file into (w, m, v); returns its step.  Size and header checked
        before anything is copied."""
        self._state(w, m, v)
        step = C.c_int32()
        self._bind()
        _check(lib().repstep_checkpoint_load(self._ctx, os.fsencode(path), C.byref(step), _ptr(w),
                                             _ptr(m), _ptr(v)), "checkpoint_load")
        return int(step.value)

    def sync(self) -> int:
        """Synchronise the stream; return the device flags (raises on a kernel timeout)."""
        flags = C.c_uint32()
        self._bind()
        rc = lib().repstep_sync(self._ctx, C.byref(flags))
        if rc == 6:
            raise RepstepError(rc, f"flags=0x{flags.value:x}")
        _check(rc, "sync")
        return int(flags.value)

    def launch_count(self) -> int:
        return int(lib().repstep_launch_count(self._ctx))

    def last_cuda_error(self) -> int:
        return int(lib().repstep_last_cuda_error(self._ctx))

    # ---------------------------------------------------------------- workspace views
    def _view(self, off: int, count: int, dtype):
        item = torch.empty(0, dtype=dtype).element_size()
        return self.workspace[off: off + count * item].view(dtype)

    def g_view(self):
        return self._view(self.layout.g, self.n, torch.float32)

    def chunk_sums_view(self):
        return self._view(self.layout.chunk_sums, self.c, torch.float32)

    def leaves_view(self):
        return self._view(self.layout.leaves, 1 + 3 * self.c, torch.int64)

    def scalars_view(self):
        return self._view(self.layout.scalars, 4, torch.int32)

    def destroy(self):
        if self._ctx:
            lib().repstep_destroy(self._ctx)
            self._ctx = C.c_void_p()

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass
