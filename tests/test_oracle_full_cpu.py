"""CPU checks of the chunk-parallel oracle driver (tests/oracle_full.py) that the full-size
GPU tests compare with: cut into small slabs and run on several threads, it must give the
same bits as the oracle's single calls over the whole vector -- g, every chunk sum, the
norm, w, m, v, every leaf and the root -- over two steps, for fp32 and bf16 gradients, bf16
parameters with decay segments in the flush-to-zero mode, and audit-mode leaves.  And it
must notice a single changed slot (negative controls)."""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from tests import oracle_full as OF

CH = 4096
HP = dict(lr=3e-4, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.1, clip=1.0)


def _f32(x):
    return np.float32(x)


def _whole(grads_np, w, m, v, t, *, hash_mode=0, ftz=False, bf16w=False, segments=None):
    """The step from the oracle's single calls over the whole vector."""
    hp = {k: _f32(x) for k, x in HP.items()}
    if ftz:
        g = O.reduce_ftz(grads_np)
        norm, cs = O.norm_ftz(g, with_chunks=True)
        scale = O.clip_scale_ftz(norm, hp["clip"])
        bc1, bc2 = O.bias_corrections_ftz(hp["beta1"], hp["beta2"], t)
        w, m, v = O.adamw_ftz(w, m, v, g, scale, hp["lr"], hp["beta1"], hp["beta2"], hp["eps"],
                              hp["wd"], bc1, bc2, segments=segments)
    else:
        g = O.reduce(grads_np)
        norm, cs = O.norm(g, with_chunks=True)
        scale = O.clip_scale(norm, hp["clip"])
        bc1, bc2 = O.bias_corrections(hp["beta1"], hp["beta2"], t)
        args = (g, scale, hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], hp["wd"], bc1, bc2)
        if segments is not None:
            fn = O.adamw_bf16w_segments if bf16w else O.adamw_segments
            w, m, v = fn(w, m, v, *args, segments)
        else:
            w, m, v = (O.adamw_bf16w if bf16w else O.adamw)(w, m, v, *args)
    wide = O.widen_bf16(w) if bf16w else w
    leaves = O.leaves(t, wide, m, v, hash_mode)
    return dict(g=g, cs=cs, norm=norm, w=w, m=m, v=v, leaves=leaves,
                root=O.merkle_root(leaves))


def _as_gpu_dict(res):
    """The single-call results in the form the driver reads the GPU's (CPU tensors here)."""
    w = res["w"]
    wt = torch.from_numpy(w.view(np.int16).copy()).view(torch.bfloat16) \
        if w.dtype == np.uint16 else torch.from_numpy(w.copy())
    return dict(g=torch.from_numpy(res["g"].copy()), chunk_sums=torch.from_numpy(res["cs"].copy()),
                leaves=torch.from_numpy(res["leaves"].view(np.int64).copy()), w=wt,
                m=torch.from_numpy(res["m"].copy()), v=torch.from_numpy(res["v"].copy()),
                norm=torch.tensor([float(res["norm"])], dtype=torch.float32),
                root=torch.tensor([res["root"]], dtype=torch.uint64).view(torch.int64))


def _grads(rng, n, R, t, bf16=False):
    out_np, out_t = [], []
    for r in range(R):
        x = (rng.standard_normal(n) * 10.0 ** (-3 + (r + t) % 3)).astype(np.float32)
        if bf16:
            tt = torch.from_numpy(x).to(torch.bfloat16)
            out_t.append(tt)
            out_np.append(tt.view(torch.int16).numpy().view(np.uint16).copy())
        else:
            out_t.append(torch.from_numpy(x))
            out_np.append(x)
    return out_np, out_t


@pytest.mark.parametrize("case", ["f32", "bf16_grads", "audit", "bf16w_segments_ftz", "ragged_small"])
def test_chunk_parallel_driver_equals_single_calls(case):
    rng = np.random.default_rng(hash(case) % 2**32)
    n = 7 * CH + 1234 if case != "ragged_small" else 1234
    R = 3
    kw = {}
    bf16w = case == "bf16w_segments_ftz"
    segs = [(0, False), (CH + 17, True), (3 * CH - 5, False), (5 * CH + 2, True)] \
        if bf16w else None
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    if bf16w:
        w0 = torch.from_numpy(w0).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    m0 = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    v0 = (rng.standard_normal(n) * 1e-3).astype(np.float32) ** 2
    hash_mode = 1 if case == "audit" else 0
    fo = OF.FullOracle(n, R, w0.copy(), m0.copy(), v0.copy(),
                       grad_dtype="bf16" if case == "bf16_grads" else "f32",
                       param_dtype="bf16" if bf16w else "f32", hash_mode=hash_mode,
                       ftz=bf16w, segments=segs, threads=3, slab=2 * CH)
    w, m, v = w0, m0, v0
    for t in (1, 2):
        gnp, gt = _grads(rng, n, R, t, bf16=case == "bf16_grads")
        res = _whole(gnp, w, m, v, t, hash_mode=hash_mode, ftz=bf16w, bf16w=bf16w,
                     segments=segs)
        rep = fo.step(gt, t, HP, _as_gpu_dict(res), **kw)
        OF.assert_identical(rep, f"{case} step {t}")
        assert rep["w"]["slots"] == n and rep["leaves"]["slots"] == 1 + 3 * ((n + CH - 1) // CH)
        w, m, v = res["w"], res["m"], res["v"]
    fo.close()


def test_driver_reports_a_single_changed_slot():
    """Negative controls: one flipped bit in w, one changed leaf and one changed chunk sum
    are each counted, with the right relFro, and a wrong norm or root is flagged."""
    rng = np.random.default_rng(5)
    n, R = 5 * CH + 77, 2
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    z = np.zeros(n, np.float32)
    gnp, gt = _grads(rng, n, R, 1)
    res = _whole(gnp, w0, z, z, 1)
    for what in ["w", "leaves", "chunk_sums", "norm", "root"]:
        fo = OF.FullOracle(n, R, w0.copy(), z.copy(), z.copy(), threads=2, slab=2 * CH)
        gpu = _as_gpu_dict(res)
        if what == "w":
            wb = gpu["w"].view(torch.int32)
            wb[n - 3] ^= 1
        elif what == "leaves":
            gpu["leaves"][7] += 1
        elif what == "chunk_sums":
            gpu["chunk_sums"].view(torch.int32)[2] ^= 1
        elif what == "norm":
            gpu["norm"].view(torch.int32)[0] ^= 1
        else:
            gpu["root"][0] ^= 1
        rep = fo.step(gt, 1, HP, gpu)
        fo.close()
        if what in ("norm", "root"):
            assert not rep[what]["equal"]
            with pytest.raises(AssertionError):
                OF.assert_identical(rep)
            continue
        assert rep[what]["differing"] == 1, rep[what]
        if what == "w":
            d = abs(float(res["w"][n - 3]) - float(gpu["w"][n - 3]))
            assert rep["w"]["max_abs"] == pytest.approx(d)
            assert rep["w"]["relFro"] == pytest.approx(d / np.linalg.norm(res["w"].astype(np.float64)))
        with pytest.raises(AssertionError):
            OF.assert_identical(rep)
