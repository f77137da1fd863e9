"""ctypes marshalling for the plain-C oracle (oracle.c).  Argument conversion only.

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the benchmark's
CPU-baseline leg; never by the product path.

Arrays are numpy arrays on the host: fp32 gradients/state as float32, bf16 gradients as
uint16 bit patterns, digests as uint64.
"""
import ctypes as C

import numpy as np

from . import build as _build

_lib = None

F32 = 0
BF16 = 1


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = C.CDLL(path)
        fp = C.c_void_p
        L.oracle_probe_mul_add.argtypes = [C.c_float, C.c_float, C.c_float]
        L.oracle_probe_mul_add.restype = C.c_float
        L.oracle_probe_subnormals.restype = C.c_int
        L.oracle_tree_sum.argtypes = [fp, C.c_uint64]
        L.oracle_tree_sum.restype = C.c_float
        L.oracle_reduce.argtypes = [fp, C.c_int, C.c_uint32, C.c_uint64, fp]
        L.oracle_reduce.restype = C.c_int
        L.oracle_reduce_topology.argtypes = [fp, C.c_int, C.c_uint32, C.c_uint32, C.c_uint64, fp]
        L.oracle_reduce_topology.restype = C.c_int
        L.oracle_norm.argtypes = [fp, C.c_uint64, fp]
        L.oracle_norm.restype = C.c_float
        L.oracle_clip_scale.argtypes = [C.c_float, C.c_float]
        L.oracle_clip_scale.restype = C.c_float
        L.oracle_bias_corrections.argtypes = [C.c_float, C.c_float, C.c_int32,
                                              C.POINTER(C.c_float), C.POINTER(C.c_float)]
        L.oracle_bias_corrections.restype = None
        L.oracle_adamw.argtypes = [fp, fp, fp, fp, C.c_uint64, C.c_float,
                                   C.c_float, C.c_float, C.c_float, C.c_float, C.c_float,
                                   C.c_float, C.c_float]
        L.oracle_adamw.restype = None
        L.oracle_pf61_constant.restype = C.c_uint64
        L.oracle_pf61.argtypes = [fp, C.c_uint64]
        L.oracle_pf61.restype = C.c_uint64
        L.oracle_blake2b.argtypes = [fp, C.c_uint64, fp, C.c_uint32]
        L.oracle_blake2b.restype = C.c_int
        L.oracle_node.argtypes = [C.c_uint64, C.c_uint64]
        L.oracle_node.restype = C.c_uint64
        L.oracle_merkle_root.argtypes = [fp, C.c_uint64]
        L.oracle_merkle_root.restype = C.c_uint64
        L.oracle_image_bytes.argtypes = [C.c_uint64]
        L.oracle_image_bytes.restype = C.c_uint64
        L.oracle_image.argtypes = [C.c_int32, C.c_uint64, fp, fp, fp, fp]
        L.oracle_image.restype = C.c_int
        L.oracle_num_leaves.argtypes = [C.c_uint64]
        L.oracle_num_leaves.restype = C.c_uint64
        L.oracle_leaves.argtypes = [C.c_int32, C.c_uint64, fp, fp, fp, fp]
        L.oracle_leaves.restype = C.c_int
        L.oracle_state_hash.argtypes = [C.c_int32, C.c_uint64, fp, fp, fp, C.POINTER(C.c_uint64)]
        L.oracle_state_hash.restype = C.c_int
        L.oracle_step.argtypes = [fp, C.c_int, C.c_uint32, C.c_uint32, C.c_uint64, fp, fp, fp,
                                  C.c_float, C.c_float, C.c_float, C.c_float, C.c_float,
                                  C.c_float, C.c_int32, C.POINTER(C.c_float),
                                  C.POINTER(C.c_float), C.POINTER(C.c_uint64)]
        L.oracle_step.restype = C.c_int
        L.oracle_leaves_mode.argtypes = [C.c_int32, C.c_uint64, fp, fp, fp, C.c_int, fp]
        L.oracle_leaves_mode.restype = C.c_int
        L.oracle_state_hash_mode.argtypes = [C.c_int32, C.c_uint64, fp, fp, fp, C.c_int,
                                             C.POINTER(C.c_uint64)]
        L.oracle_state_hash_mode.restype = C.c_int
        L.oracle_step_mode.argtypes = [fp, C.c_int, C.c_uint32, C.c_uint32, C.c_uint64, fp, fp,
                                       fp, C.c_float, C.c_float, C.c_float, C.c_float,
                                       C.c_float, C.c_float, C.c_int32, C.c_int,
                                       C.POINTER(C.c_float), C.POINTER(C.c_float),
                                       C.POINTER(C.c_uint64)]
        L.oracle_step_mode.restype = C.c_int
        L.oracle_reduce_alg1.argtypes = [fp, C.c_int, C.c_uint32, C.c_uint32, C.c_uint64, fp]
        L.oracle_reduce_alg1.restype = C.c_int
        L.oracle_reduce_alg1_accum.argtypes = [fp, C.c_int, C.c_uint32, C.c_uint32, C.c_uint32,
                                               C.c_uint64, fp]
        L.oracle_reduce_alg1_accum.restype = C.c_int
        L.oracle_f32_to_bf16.argtypes = [C.c_float]
        L.oracle_f32_to_bf16.restype = C.c_uint16
        L.oracle_adamw_bf16w.argtypes = [fp, fp, fp, fp, C.c_uint64, C.c_float, C.c_float,
                                         C.c_float, C.c_float, C.c_float, C.c_float, C.c_float,
                                         C.c_float]
        L.oracle_adamw_bf16w.restype = None
        L.oracle_flush.argtypes = [C.c_float]
        L.oracle_flush.restype = C.c_float
        for fn in (L.oracle_mul_ftz, L.oracle_div_ftz):
            fn.argtypes = [C.c_float, C.c_float]
            fn.restype = C.c_float
        L.oracle_tree_sum_ftz.argtypes = [fp, C.c_uint64]
        L.oracle_tree_sum_ftz.restype = C.c_float
        L.oracle_reduce_ftz.argtypes = [fp, C.c_int, C.c_uint32, C.c_uint64, fp]
        L.oracle_reduce_ftz.restype = C.c_int
        L.oracle_reduce_alg1_ftz.argtypes = [fp, C.c_int, C.c_uint32, C.c_uint32, C.c_uint32,
                                             C.c_uint64, fp]
        L.oracle_reduce_alg1_ftz.restype = C.c_int
        L.oracle_norm_ftz.argtypes = [fp, C.c_uint64, fp]
        L.oracle_norm_ftz.restype = C.c_float
        L.oracle_clip_scale_ftz.argtypes = [C.c_float, C.c_float]
        L.oracle_clip_scale_ftz.restype = C.c_float
        L.oracle_bias_corrections_ftz.argtypes = [C.c_float, C.c_float, C.c_int32,
                                                  C.POINTER(C.c_float), C.POINTER(C.c_float)]
        L.oracle_bias_corrections_ftz.restype = None
        L.oracle_adamw_ftz.argtypes = [fp, C.c_int, fp, fp, fp, C.c_uint64] + [C.c_float] * 8 + \
            [fp, fp, C.c_uint32]
        L.oracle_adamw_ftz.restype = C.c_int
        seg = [fp, fp, fp, fp, C.c_uint64] + [C.c_float] * 8 + [fp, fp, C.c_uint32]
        L.oracle_adamw_segments.argtypes = seg
        L.oracle_adamw_segments.restype = C.c_int
        L.oracle_adamw_bf16w_segments.argtypes = seg
        L.oracle_adamw_bf16w_segments.restype = C.c_int
        _lib = L
    return _lib


def _p(a: np.ndarray):
    assert a.flags.c_contiguous
    return C.c_void_p(a.ctypes.data)


def _f32(a):
    a = np.ascontiguousarray(a)
    assert a.dtype == np.float32, a.dtype
    return a


def _grad_arrays(grads):
    """Return (dtype code, list of contiguous arrays, ctypes pointer array)."""
    arrs = [np.ascontiguousarray(x) for x in grads]
    if arrs[0].dtype == np.float32:
        code = F32
    elif arrs[0].dtype == np.uint16:
        code = BF16
    else:
        raise TypeError(f"gradient dtype {arrs[0].dtype}: use float32 or uint16 (bf16 bits)")
    n = arrs[0].size
    for a in arrs:
        if a.dtype != arrs[0].dtype or a.size != n:
            raise ValueError("all replica gradients must share dtype and length")
    ptrs = (C.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])
    return code, arrs, ptrs


def probe_mul_add(a, b, c) -> float:
    return lib().oracle_probe_mul_add(a, b, c)


def probe_subnormals() -> bool:
    return bool(lib().oracle_probe_subnormals())


def tree_sum(x) -> np.float32:
    x = _f32(x)
    return np.float32(lib().oracle_tree_sum(_p(x), x.size))


def reduce(grads) -> np.ndarray:
    code, arrs, ptrs = _grad_arrays(grads)
    n = arrs[0].size
    g = np.empty(n, np.float32)
    rc = lib().oracle_reduce(C.cast(ptrs, C.c_void_p), code, len(arrs), n, _p(g))
    if rc != 0:
        raise ValueError(f"oracle_reduce rc={rc}")
    return g


def reduce_topology(grads, nodes: int, gpus_per_node: int) -> np.ndarray:
    code, arrs, ptrs = _grad_arrays(grads)
    if nodes * gpus_per_node != len(arrs):
        raise ValueError("nodes * gpus_per_node must equal the replica count")
    n = arrs[0].size
    g = np.empty(n, np.float32)
    rc = lib().oracle_reduce_topology(C.cast(ptrs, C.c_void_p), code, nodes, gpus_per_node,
                                      n, _p(g))
    if rc == -2:
        raise ValueError("topology breaks the canonical tree")
    if rc != 0:
        raise ValueError(f"oracle_reduce_topology rc={rc}")
    return g


def reduce_alg1(grads, dp_shard: int) -> np.ndarray:
    """Paper-exact reduction (OPEN-1B §6 Algorithm 1) over R = dp_replicate * dp_shard
    virtual-rank gradients in mesh order."""
    code, arrs, ptrs = _grad_arrays(grads)
    n = arrs[0].size
    g = np.empty(n, np.float32)
    rc = lib().oracle_reduce_alg1(C.cast(ptrs, C.c_void_p), code, len(arrs), dp_shard, n, _p(g))
    if rc != 0:
        raise ValueError(f"oracle_reduce_alg1 rc={rc}")
    return g


def reduce_alg1_accum(grads, dp_shard: int, accum: int) -> np.ndarray:
    """Paper-exact reduction with Algorithm 1's microbatch accumulation: grads holds
    R * accum microbatch gradients, rank-major (index r * accum + k)."""
    code, arrs, ptrs = _grad_arrays(grads)
    if accum < 1 or len(arrs) % accum:
        raise ValueError("the input count must be a multiple of accum >= 1")
    n = arrs[0].size
    g = np.empty(n, np.float32)
    rc = lib().oracle_reduce_alg1_accum(C.cast(ptrs, C.c_void_p), code, len(arrs) // accum,
                                        dp_shard, accum, n, _p(g))
    if rc != 0:
        raise ValueError(f"oracle_reduce_alg1_accum rc={rc}")
    return g


def norm(g, with_chunks: bool = False):
    g = _f32(g)
    c = (g.size + 4095) // 4096
    chunks = np.empty(max(c, 1), np.float32)
    nv = np.float32(lib().oracle_norm(_p(g), g.size, _p(chunks)))
    if with_chunks:
        return nv, chunks[:c].copy()
    return nv


def clip_scale(norm_value, clip) -> np.float32:
    return np.float32(lib().oracle_clip_scale(float(np.float32(norm_value)), float(np.float32(clip))))


def bias_corrections(beta1, beta2, t):
    b1, b2 = C.c_float(), C.c_float()
    lib().oracle_bias_corrections(float(np.float32(beta1)), float(np.float32(beta2)), int(t),
                                  C.byref(b1), C.byref(b2))
    return np.float32(b1.value), np.float32(b2.value)


def adamw(w, m, v, g, scale, lr, beta1, beta2, eps, wd, bc1, bc2):
    """In-place on copies; returns (w', m', v')."""
    w = _f32(w).copy(); m = _f32(m).copy(); v = _f32(v).copy(); g = _f32(g)
    n = w.size
    assert m.size == n and v.size == n and g.size == n
    f = lambda x: float(np.float32(x))  # noqa: E731
    lib().oracle_adamw(_p(w), _p(m), _p(v), _p(g), n, f(scale), f(lr), f(beta1), f(beta2),
                       f(eps), f(wd), f(bc1), f(bc2))
    return w, m, v


def f32_to_bf16(x) -> int:
    return int(lib().oracle_f32_to_bf16(float(np.float32(x))))


def adamw_bf16w(w16, m, v, g, scale, lr, beta1, beta2, eps, wd, bc1, bc2):
    """bf16 parameters (uint16 bit patterns): returns (w16', m', v') on copies."""
    w16 = np.ascontiguousarray(w16, dtype=np.uint16).copy()
    m = _f32(m).copy(); v = _f32(v).copy(); g = _f32(g)
    f = lambda x: float(np.float32(x))  # noqa: E731
    lib().oracle_adamw_bf16w(_p(w16), _p(m), _p(v), _p(g), w16.size, f(scale), f(lr), f(beta1),
                             f(beta2), f(eps), f(wd), f(bc1), f(bc2))
    return w16, m, v


def _segments(segments):
    """[(begin, decays), ...] -> (uint64 starts, uint8 flags)."""
    b = np.ascontiguousarray([int(s[0]) for s in segments] or [0], dtype=np.uint64)
    d = np.ascontiguousarray([1 if s[1] else 0 for s in segments] or [0], dtype=np.uint8)
    return b, d, len(segments)


def adamw_segments(w, m, v, g, scale, lr, beta1, beta2, eps, wd, bc1, bc2, segments):
    """AdamW with per-segment weight decay: segments = [(begin, decays), ...] cutting
    [0, n) in increasing order from 0; returns (w', m', v') on copies."""
    w = _f32(w).copy(); m = _f32(m).copy(); v = _f32(v).copy(); g = _f32(g)
    b, d, cnt = _segments(segments)
    f = lambda x: float(np.float32(x))  # noqa: E731
    rc = lib().oracle_adamw_segments(_p(w), _p(m), _p(v), _p(g), w.size, f(scale), f(lr),
                                     f(beta1), f(beta2), f(eps), f(wd), f(bc1), f(bc2), _p(b),
                                     _p(d), cnt)
    if rc != 0:
        raise ValueError("bad segment list")
    return w, m, v


def adamw_bf16w_segments(w16, m, v, g, scale, lr, beta1, beta2, eps, wd, bc1, bc2, segments):
    """bf16 parameters with per-segment weight decay; returns (w16', m', v') on copies."""
    w16 = np.ascontiguousarray(w16, dtype=np.uint16).copy()
    m = _f32(m).copy(); v = _f32(v).copy(); g = _f32(g)
    b, d, cnt = _segments(segments)
    f = lambda x: float(np.float32(x))  # noqa: E731
    rc = lib().oracle_adamw_bf16w_segments(_p(w16), _p(m), _p(v), _p(g), w16.size, f(scale),
                                           f(lr), f(beta1), f(beta2), f(eps), f(wd), f(bc1),
                                           f(bc2), _p(b), _p(d), cnt)
    if rc != 0:
        raise ValueError("bad segment list")
    return w16, m, v


# ---------------------------------------------------------------- software FTZ mode
def flush(x) -> np.float32:
    """A subnormal becomes a zero of the same sign; everything else is unchanged."""
    return np.float32(lib().oracle_flush(float(np.float32(x))))


def mul_ftz(a, b) -> np.float32:
    """One product in the flush-to-zero mode (operands flushed, tiny result zeroed)."""
    return np.float32(lib().oracle_mul_ftz(float(np.float32(a)), float(np.float32(b))))


def div_ftz(a, b) -> np.float32:
    """One quotient in the flush-to-zero mode."""
    return np.float32(lib().oracle_div_ftz(float(np.float32(a)), float(np.float32(b))))


def tree_sum_ftz(x) -> np.float32:
    x = _f32(x)
    return np.float32(lib().oracle_tree_sum_ftz(_p(x), x.size))


def reduce_ftz(grads) -> np.ndarray:
    code, arrs, ptrs = _grad_arrays(grads)
    g = np.empty(arrs[0].size, np.float32)
    if lib().oracle_reduce_ftz(C.cast(ptrs, C.c_void_p), code, len(arrs), g.size, _p(g)) != 0:
        raise ValueError("bad arguments")
    return g


def reduce_alg1_ftz(grads, dp_shard: int, accum: int = 0) -> np.ndarray:
    code, arrs, ptrs = _grad_arrays(grads)
    if accum and len(arrs) % accum:
        raise ValueError("the input count must be a multiple of accum")
    g = np.empty(arrs[0].size, np.float32)
    R = len(arrs) // accum if accum else len(arrs)
    if lib().oracle_reduce_alg1_ftz(C.cast(ptrs, C.c_void_p), code, R, dp_shard, accum, g.size,
                                    _p(g)) != 0:
        raise ValueError("bad arguments")
    return g


def norm_ftz(g, with_chunks: bool = False):
    g = _f32(g)
    c = (g.size + 4095) // 4096
    chunks = np.empty(max(c, 1), np.float32)
    nv = np.float32(lib().oracle_norm_ftz(_p(g), g.size, _p(chunks)))
    return (nv, chunks[:c].copy()) if with_chunks else nv


def clip_scale_ftz(norm_value, clip) -> np.float32:
    return np.float32(lib().oracle_clip_scale_ftz(float(np.float32(norm_value)),
                                                  float(np.float32(clip))))


def bias_corrections_ftz(beta1, beta2, t):
    b1, b2 = C.c_float(), C.c_float()
    lib().oracle_bias_corrections_ftz(float(np.float32(beta1)), float(np.float32(beta2)), int(t),
                                      C.byref(b1), C.byref(b2))
    return np.float32(b1.value), np.float32(b2.value)


def adamw_ftz(w, m, v, g, scale, lr, beta1, beta2, eps, wd, bc1, bc2, segments=None):
    """FTZ-mode AdamW on copies; w float32, or uint16 bf16 bit patterns (bf16 parameters);
    segments as in adamw_segments (None: every element decays).  Returns (w', m', v')."""
    w = np.ascontiguousarray(w).copy()
    bf = w.dtype == np.uint16
    if not bf:
        w = _f32(w).copy()
    m = _f32(m).copy(); v = _f32(v).copy(); g = _f32(g)
    b, d, cnt = _segments(segments) if segments else (np.zeros(1, np.uint64),
                                                      np.zeros(1, np.uint8), 0)
    f = lambda x: float(np.float32(x))  # noqa: E731
    rc = lib().oracle_adamw_ftz(_p(w), 1 if bf else 0, _p(m), _p(v), _p(g), w.size, f(scale),
                                f(lr), f(beta1), f(beta2), f(eps), f(wd), f(bc1), f(bc2), _p(b),
                                _p(d), cnt)
    if rc != 0:
        raise ValueError("bad segment list")
    return w, m, v


def widen_bf16(w16) -> np.ndarray:
    """bf16 bit patterns -> the fp32 values they denote (exact)."""
    return (np.ascontiguousarray(w16, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def pf61_constant() -> int:
    return int(lib().oracle_pf61_constant())


def pf61(words) -> int:
    words = np.ascontiguousarray(words, dtype=np.uint32)
    return int(lib().oracle_pf61(_p(words) if words.size else None, words.size))


def blake2b(data: bytes, outlen: int = 64) -> bytes:
    buf = np.frombuffer(bytes(data) + b"\0", dtype=np.uint8)
    out = np.zeros(outlen, np.uint8)
    rc = lib().oracle_blake2b(_p(buf), len(data), _p(out), outlen)
    if rc != 0:
        raise ValueError("bad outlen")
    return out.tobytes()


def node(a: int, b: int) -> int:
    return int(lib().oracle_node(a, b))


def merkle_root(leaves) -> int:
    leaves = np.ascontiguousarray(leaves, dtype=np.uint64)
    return int(lib().oracle_merkle_root(_p(leaves), leaves.size))


def image_bytes(n: int) -> int:
    return int(lib().oracle_image_bytes(n))


def image(step: int, w, m, v) -> bytes:
    w = _f32(w); m = _f32(m); v = _f32(v)
    n = w.size
    out = np.empty(image_bytes(n), np.uint8)
    rc = lib().oracle_image(step, n, _p(w), _p(m), _p(v), _p(out))
    if rc != 0:
        raise ValueError("n too large for the header")
    return out.tobytes()


def num_leaves(n: int) -> int:
    return int(lib().oracle_num_leaves(n))


def leaves(step: int, w, m, v, hash_mode: int = 0) -> np.ndarray:
    """Leaf digests: hash_mode 0 = PF61, 1 = BLAKE2b-64 (audit mode)."""
    w = _f32(w); m = _f32(m); v = _f32(v)
    n = w.size
    out = np.empty(num_leaves(n), np.uint64)
    rc = lib().oracle_leaves_mode(step, n, _p(w), _p(m), _p(v), hash_mode, _p(out))
    if rc != 0:
        raise ValueError("n too large for the header")
    return out


def state_hash(step: int, w, m, v, hash_mode: int = 0) -> int:
    w = _f32(w); m = _f32(m); v = _f32(v)
    r = C.c_uint64()
    rc = lib().oracle_state_hash_mode(step, w.size, _p(w), _p(m), _p(v), hash_mode, C.byref(r))
    if rc != 0:
        raise ValueError("n too large for the header")
    return int(r.value)


def step(grads, w, m, v, *, lr, beta1, beta2, eps, wd, clip, t, nodes=1, gpus_per_node=None,
         hash_mode=0):
    """One oracle step on copies of (w, m, v).  Returns dict(w, m, v, norm, scale, root)."""
    code, arrs, ptrs = _grad_arrays(grads)
    R = len(arrs)
    if gpus_per_node is None:
        gpus_per_node = R // nodes
    if nodes * gpus_per_node != R:
        raise ValueError("nodes * gpus_per_node must equal the replica count")
    w = _f32(w).copy(); m = _f32(m).copy(); v = _f32(v).copy()
    n = w.size
    nv, sv, root = C.c_float(), C.c_float(), C.c_uint64()
    f = lambda x: float(np.float32(x))  # noqa: E731
    rc = lib().oracle_step_mode(C.cast(ptrs, C.c_void_p), code, nodes, gpus_per_node, n,
                                _p(w), _p(m), _p(v), f(lr), f(beta1), f(beta2), f(eps), f(wd),
                                f(clip), int(t), int(hash_mode), C.byref(nv), C.byref(sv),
                                C.byref(root))
    if rc == -2:
        raise ValueError("topology breaks the canonical tree")
    if rc != 0:
        raise ValueError(f"oracle_step rc={rc}")
    return dict(w=w, m=m, v=v, norm=np.float32(nv.value), scale=np.float32(sv.value),
                root=int(root.value))
