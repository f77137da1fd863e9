"""Every slot of a full-size step compared with the oracle, run chunk-parallel on the host.

TEST INFRASTRUCTURE ONLY: it drives the oracle (oracle/oracle.c through oracle/oracle.py),
and only the GPU tests and the golden-fingerprint script use it.

The oracle's functions run unchanged; each call is single-threaded and covers one slice
[lo, hi) of the parameter range whose ends are multiples of the 4096-element chunk (or n).
A pool of host threads runs the calls for disjoint slices at the same time: ctypes
releases the GIL for the length of each foreign call, and no two calls touch the same
memory.  Because every slice starts on the chunk grid of the definition, the chunk sums
and the leaf digests a slice yields are exactly those of the same chunks of the whole
vector.  The global pieces are then formed once, from the oracle's own per-chunk results:
the canonical tree over all c chunk sums, its square root, the clip scale, and the Merkle
tree over all 1 + 3c leaves ("OPEN-1B: A Fully Auditable Training Run", §3.2 global-norm
clipping, App. B state hash).

The oracle keeps its own state (w, m, v) in host memory from step to step, starting from
the same initial bytes as the GPU, so after K steps it has followed its own trajectory; the
GPU's arrays are read only to be compared.  Host memory: the state (12n bytes, or 10n with
bf16 parameters), the reduced gradient g (4n) and pinned staging buffers of one slab.

The statistics reported per array are those of "Cross-process reproducibility, settled by
measurement" (section "The measurement"): differing slots, relative Frobenius difference
and the largest absolute difference.
"""
from __future__ import annotations

import ctypes as C
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

from oracle import oracle as O

CH = 4096
F32, BF16 = 0, 1


def _ptr(a: np.ndarray, lo: int = 0) -> C.c_void_p:
    return C.c_void_p(a.ctypes.data + lo * a.itemsize)


def _local_segments(segs, lo, hi):
    """The decay segment list [(begin, decays), ...] restricted to [lo, hi), re-based to lo."""
    starts = [b for b, _ in segs]
    k = int(np.searchsorted(starts, lo, side="right")) - 1
    out = [(0, segs[k][1])]
    for b, d in segs[k + 1:]:
        if b >= hi:
            break
        out.append((b - lo, d))
    b = np.ascontiguousarray([s[0] for s in out], dtype=np.uint64)
    f = np.ascontiguousarray([1 if s[1] else 0 for s in out], dtype=np.uint8)
    return b, f


def _as_f32(a: np.ndarray) -> np.ndarray:
    return (a.astype(np.uint32) << 16).view(np.float32) if a.dtype == np.uint16 else a


def diff_stats(got: np.ndarray, want: np.ndarray):
    """(differing slots, sum of squared finite differences, sum of squared finite reference
    values, max|d|) of two equal-length fp32 (or bf16 bit-pattern) arrays; NaNs are
    compared by class, as the contract on specials says."""
    bad = (got != want) if got.dtype == np.uint16 else (got.view(np.uint32) != want.view(np.uint32))
    if not bad.any():
        return 0, 0.0, 0.0, 0.0
    g, w = _as_f32(got), _as_f32(want)
    bad &= ~(np.isnan(g) & np.isnan(w))
    nbad = int(np.count_nonzero(bad))
    if nbad == 0:
        return 0, 0.0, 0.0, 0.0
    g64, w64 = g.astype(np.float64), w.astype(np.float64)
    fin = np.isfinite(g64) & np.isfinite(w64)
    with np.errstate(invalid="ignore"):
        d = np.where(fin, g64 - w64, 0.0)
    wf = np.where(fin, w64, 0.0)
    return nbad, float(np.dot(d, d)), float(np.dot(wf, wf)), float(np.max(np.abs(d)))


class Tally:
    """Per array: differing slots, relative Frobenius difference and max|d|, accumulated
    slab by slab.  The relFro denominator is the norm of the whole reference array, taken
    at report time (and only when some slot differs)."""

    def __init__(self):
        self.d = {}

    def add(self, name, got, want):
        nbad, num2, _, mx = diff_stats(got, want)
        tot = self.d.setdefault(name, [0, 0.0, 0.0, 0])
        tot[0] += nbad
        tot[1] += num2
        tot[2] = max(tot[2], mx)
        tot[3] += got.size

    def report(self, refs):
        """refs: name -> the whole reference (oracle) array."""
        out = {}
        for k, (nbad, num2, mx, size) in self.d.items():
            rel = 0.0
            if nbad:
                r = _as_f32(refs[k]).astype(np.float64)
                r = np.where(np.isfinite(r), r, 0.0)
                den = float(np.sqrt(np.dot(r, r)))
                rel = float(np.sqrt(num2)) / den if den > 0 else float(np.sqrt(num2))
            out[k] = dict(slots=size, differing=nbad, relFro=rel, max_abs=mx)
        return out


class FullOracle:
    """The oracle's trajectory of a workload at full size, compared slot by slot with the
    GPU's after every step.

    n, R: parameters and replicas; grad_dtype "f32" or "bf16"; param_dtype "f32" or "bf16";
    hash_mode 0 (PF61) or 1 (BLAKE2b-64 leaves); ftz: the flush-to-zero arithmetic;
    segments: decay segments [(begin, decays), ...] or None (every element decays).
    w0, m0, v0: host copies of the initial state (w0 as uint16 bit patterns for bf16
    parameters), which the oracle then owns and updates.
    """

    def __init__(self, n, R, w0, m0, v0, *, grad_dtype="f32", param_dtype="f32", hash_mode=0,
                 ftz=False, segments=None, threads=None, slab=1 << 26):
        self.n, self.R = n, R
        self.c = (n + CH - 1) // CH
        self.gcode = BF16 if grad_dtype == "bf16" else F32
        self.bf16w = param_dtype == "bf16"
        self.hash_mode, self.ftz, self.segments = hash_mode, ftz, segments
        self.threads = threads or max(1, os.cpu_count() or 1)
        assert slab % CH == 0
        self.slab = slab
        self.w = np.ascontiguousarray(w0, dtype=np.uint16 if self.bf16w else np.float32)
        self.m = np.ascontiguousarray(m0, dtype=np.float32)
        self.v = np.ascontiguousarray(v0, dtype=np.float32)
        assert self.w.size == self.m.size == self.v.size == n
        self.g = np.empty(n, np.float32)
        self.chunk_sums = np.empty(max(self.c, 1), np.float32)
        self.leaves = np.empty(1 + 3 * self.c, np.uint64)
        self.pool = ThreadPoolExecutor(self.threads)
        self.L = O.lib()
        gt = torch.bfloat16 if self.gcode == BF16 else torch.float32
        pin = torch.cuda.is_available()            # CPU tensors in the CPU self-test
        self.stage_grads = torch.empty((R, slab), dtype=gt, pin_memory=pin)
        self.stage_a = torch.empty(slab, dtype=torch.float32, pin_memory=pin)
        self.stage_b = torch.empty(slab, dtype=torch.float32, pin_memory=pin)
        self.stage_c = torch.empty(slab, dtype=torch.float32, pin_memory=pin)

    # ----------------------------------------------------------------- helpers
    def _slabs(self):
        for lo in range(0, self.n, self.slab):
            yield lo, min(lo + self.slab, self.n)

    def _parts(self, lo, hi):
        """Chunk-aligned sub-slices of [lo, hi) for the thread pool."""
        chunks = (hi - lo + CH - 1) // CH
        per = max(1, -(-chunks // self.threads))
        out = []
        for k in range(0, chunks, per):
            a = lo + k * CH
            out.append((a, min(lo + (k + per) * CH, hi)))
        return out

    def _run(self, fn, parts):
        for f in [self.pool.submit(fn, a, b) for a, b in parts]:
            f.result()

    @staticmethod
    def _sync():
        if torch.cuda.is_available():
            torch.cuda.current_stream().synchronize()

    def _host(self, stage: torch.Tensor, dev: torch.Tensor, cnt: int) -> np.ndarray:
        """Copy cnt elements of a device slice into a pinned buffer; numpy view of it."""
        dst = stage[:cnt]
        dst.copy_(dev, non_blocking=True)
        self._sync()
        return dst.numpy()

    # ----------------------------------------------------------------- one step
    def step(self, grads, t, hp, gpu, *, reducer="tree", nodes=1, gpus_per_node=None,
             dp_shard=1):
        """Run the oracle's step t on the device gradients `grads` (R torch tensors) and
        compare with the GPU's results.  hp: dict(lr, beta1, beta2, eps, wd, clip).
        gpu: None (the oracle's step only), or a dict of device tensors g (optional: a
        step that keeps g out of HBM has none to compare), chunk_sums, leaves (u64 as
        int64), w, m, v (the state after the GPU's step), norm (1 fp32) and root (1 int64).  reducer: "tree"
        (the canonical tree), "topology" (staged nodes x gpus_per_node) or "alg1" (the
        paper-exact order with dp_shard).  Returns the report dict."""
        L, n, c, R = self.L, self.n, self.c, self.R
        tally = Tally()
        assert len(grads) == R
        esz = 2 if self.gcode == BF16 else 4

        # ---- pass 1: reduce and the chunk sums of squares, slab by slab
        for lo, hi in self._slabs():
            cnt = hi - lo
            for r in range(R):
                self.stage_grads[r, :cnt].copy_(grads[r][lo:hi], non_blocking=True)
            self._sync()
            sg = self.stage_grads
            base = [sg[r].data_ptr() for r in range(R)]

            def reduce_part(a, b, lo=lo, base=base):
                ptrs = (C.c_void_p * R)(*[p + (a - lo) * esz for p in base])
                pp = C.cast(ptrs, C.c_void_p)
                if reducer == "tree":
                    fn = L.oracle_reduce_ftz if self.ftz else L.oracle_reduce
                    rc = fn(pp, self.gcode, R, b - a, _ptr(self.g, a))
                elif reducer == "topology":
                    assert not self.ftz
                    rc = L.oracle_reduce_topology(pp, self.gcode, nodes, gpus_per_node, b - a,
                                                  _ptr(self.g, a))
                elif reducer == "alg1":
                    if self.ftz:
                        rc = L.oracle_reduce_alg1_ftz(pp, self.gcode, R, dp_shard, 0, b - a,
                                                      _ptr(self.g, a))
                    else:
                        rc = L.oracle_reduce_alg1(pp, self.gcode, R, dp_shard, b - a,
                                                  _ptr(self.g, a))
                else:
                    raise ValueError(reducer)
                assert rc == 0, (reducer, rc)
                normf = L.oracle_norm_ftz if self.ftz else L.oracle_norm
                normf(_ptr(self.g, a), b - a, _ptr(self.chunk_sums, a // CH))

            self._run(reduce_part, self._parts(lo, hi))
            if gpu is not None and "g" in gpu:
                tally.add("g", self._host(self.stage_a, gpu["g"][lo:hi], cnt), self.g[lo:hi])

        # ---- the global norm and clip scale from the oracle's own chunk sums
        cs = self.chunk_sums[:c]
        if self.ftz:
            norm = O.flush(np.sqrt(O.tree_sum_ftz(cs), dtype=np.float32)) if c else np.float32(0)
            scale = O.clip_scale_ftz(norm, hp["clip"])
            bc1, bc2 = O.bias_corrections_ftz(hp["beta1"], hp["beta2"], t)
        else:
            norm = np.sqrt(O.tree_sum(cs), dtype=np.float32) if c else np.float32(0)
            scale = O.clip_scale(norm, hp["clip"])
            bc1, bc2 = O.bias_corrections(hp["beta1"], hp["beta2"], t)
        if gpu is not None:
            tally.add("chunk_sums", gpu["chunk_sums"][:c].cpu().numpy(), cs)

        # ---- pass 2: AdamW and the leaf digests, slab by slab
        f = lambda x: float(np.float32(x))  # noqa: E731
        hpf = (f(scale), f(hp["lr"]), f(hp["beta1"]), f(hp["beta2"]), f(hp["eps"]),
               f(hp["wd"]), f(bc1), f(bc2))

        def adamw_part(a, b):
            cnt = b - a
            wp = _ptr(self.w, a)
            if self.segments is not None:
                sb, sd = _local_segments(self.segments, a, b)
                segargs = (_ptr(sb), _ptr(sd), len(sb))
            else:
                sb = sd = None
                segargs = (None, None, 0)
            if self.ftz:
                rc = L.oracle_adamw_ftz(wp, 1 if self.bf16w else 0, _ptr(self.m, a),
                                        _ptr(self.v, a), _ptr(self.g, a), cnt, *hpf, *segargs)
                assert rc == 0
            elif self.segments is not None:
                fn = L.oracle_adamw_bf16w_segments if self.bf16w else L.oracle_adamw_segments
                assert fn(wp, _ptr(self.m, a), _ptr(self.v, a), _ptr(self.g, a), cnt, *hpf,
                          *segargs) == 0
            elif self.bf16w:
                L.oracle_adamw_bf16w(wp, _ptr(self.m, a), _ptr(self.v, a), _ptr(self.g, a),
                                     cnt, *hpf)
            else:
                L.oracle_adamw(wp, _ptr(self.m, a), _ptr(self.v, a), _ptr(self.g, a), cnt,
                               *hpf)
            # leaves of this slice's chunks (the header leaf of the call is discarded)
            cr = (cnt + CH - 1) // CH
            tmp = np.empty(1 + 3 * cr, np.uint64)
            wv = self.w[a:b]
            w32 = (wv.astype(np.uint32) << 16).view(np.float32) if self.bf16w else wv
            w32 = np.ascontiguousarray(w32)
            rc = L.oracle_leaves_mode(t, cnt, _ptr(w32), _ptr(self.m, a), _ptr(self.v, a),
                                      self.hash_mode, _ptr(tmp))
            assert rc == 0
            k0 = a // CH
            for arr in range(3):
                self.leaves[1 + arr * c + k0: 1 + arr * c + k0 + cr] = \
                    tmp[1 + arr * cr: 1 + (arr + 1) * cr]

        for lo, hi in self._slabs():
            cnt = hi - lo
            self._run(adamw_part, self._parts(lo, hi))
            if gpu is None:
                continue
            if self.bf16w:
                gw = gpu["w"][lo:hi].view(torch.int16).cpu().numpy().view(np.uint16)
            else:
                gw = self._host(self.stage_a, gpu["w"][lo:hi], cnt)
            tally.add("w", gw, self.w[lo:hi])
            tally.add("m", self._host(self.stage_b, gpu["m"][lo:hi], cnt), self.m[lo:hi])
            tally.add("v", self._host(self.stage_c, gpu["v"][lo:hi], cnt), self.v[lo:hi])

        # ---- header leaf and the root over the oracle's own leaves
        hdr = np.array([t & 0xFFFFFFFF, n], dtype=np.uint64).astype(np.uint32)
        if self.hash_mode == 0:
            self.leaves[0] = O.pf61(hdr)
        else:
            self.leaves[0] = int.from_bytes(O.blake2b(hdr.astype("<u4").tobytes(), 8), "little")
        root = O.merkle_root(self.leaves)
        norm_bits = f"{int(np.array([norm], np.float32).view(np.uint32)[0]):08x}"
        rep = dict(norm=dict(oracle=norm_bits), root=dict(oracle=f"{root:016x}"),
                   scale=float(scale))
        if gpu is None:
            return rep
        gpu_leaves = gpu["leaves"][:1 + 3 * c].cpu().numpy().view(np.uint64)
        gpu_root = int(gpu["root"].cpu().numpy().view(np.uint64)[0])
        gpu_norm = np.array([gpu["norm"].item()], np.float32).view(np.uint32)[0]
        rep.update(tally.report(dict(g=self.g, chunk_sums=cs, w=self.w, m=self.m, v=self.v)))
        rep["leaves"] = dict(slots=int(self.leaves.size),
                             differing=int(np.count_nonzero(gpu_leaves != self.leaves)))
        rep["norm"].update(gpu=f"{int(gpu_norm):08x}", equal=f"{int(gpu_norm):08x}" == norm_bits)
        rep["root"].update(gpu=f"{gpu_root:016x}", equal=root == gpu_root)
        return rep

    def close(self):
        self.pool.shutdown()


def assert_identical(rep, what=""):
    """Every compared slot equal: 0 differing slots (relFro 0) in every array, the same
    norm bits and the same root."""
    bad = {k: v for k, v in rep.items() if isinstance(v, dict) and v.get("differing", 0)}
    assert not bad, f"{what}: differing slots {bad}"
    assert rep["norm"]["equal"], f"{what}: norm {rep['norm']}"
    assert rep["root"]["equal"], f"{what}: root {rep['root']}"


def summary_line(rep) -> str:
    arrays = ["g", "chunk_sums", "w", "m", "v", "leaves"]
    parts = [f"{k} {rep[k]['differing']}/{rep[k]['slots']}" for k in arrays if k in rep]
    return (" ".join(parts) + f" | norm {rep['norm']['gpu']}/{rep['norm']['oracle']}"
            f" root {rep['root']['gpu']}/{rep['root']['oracle']}")
