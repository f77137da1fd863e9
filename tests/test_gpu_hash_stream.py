"""The state hash on a second stream (repstep_set_hash_stream): the root passes of step t
run beside step t+1's reduce, and every later writer of the leaves or the state waits for
them.  Each step's root must equal the single-stream run's, and so must the state."""
import numpy as np
import pytest
import torch

from bitwise_reproducible_step_gb300 import inputs as I
from bitwise_reproducible_step_gb300 import repstep as rs
from oracle import oracle as O
from tests import gpu_util as U

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module", autouse=True)
def _built():
    U.ensure_built()
    torch.cuda.set_device(0)


def run(n, R, steps, hash_mode, hash_stream, pdt=torch.float32, ranges=None):
    ctx = rs.Repstep(n, device=DEV, hash_mode=hash_mode, param_dtype=pdt)
    side = torch.cuda.Stream(DEV) if hash_stream else None
    ctx.set_hash_stream(side)
    w, m, v = I.gen_state(U.F32_WL, n=n, device=DEV)
    w = w.to(pdt)
    roots = torch.zeros(steps, dtype=torch.int64, device=DEV)
    grads_all = [U.gen_grads(n, R, t, scale=2000.0 if t == 2 else 1.0) for t in range(1, steps + 1)]
    for t in range(1, steps + 1):
        grads, hp = grads_all[t - 1], U.hp_for(t)
        if ranges:
            for lo, hi in ranges:
                ctx.reduce(grads, begin=lo, count=hi - lo)
            ctx.clip(hp.clip)
            for lo, hi in ranges:
                ctx.adamw(w, m, v, hp, begin=lo, count=hi - lo)
            ctx.root(t, root_out=roots[t - 1:t])
        else:
            ctx.step(grads, w, m, v, hp, step=t, root_out=roots[t - 1:t])
        # no synchronisation between steps: step t+1 is enqueued while step t's root passes
        # may still run on the hash stream
    if side is not None:
        ctx.wait_hash()
    ctx.sync()
    return roots.cpu().numpy().view(np.uint64), w, m, v


@pytest.mark.parametrize("hash_mode,pdt", [(0, torch.float32), (1, torch.float32),
                                           (0, torch.bfloat16), (1, torch.bfloat16)])
def test_pipelined_roots_equal_single_stream(hash_mode, pdt):
    n, R, T = 3 * 4096 * 5 + 123, 4, 4
    a = run(n, R, T, hash_mode, False, pdt)
    b = run(n, R, T, hash_mode, True, pdt)
    assert np.array_equal(a[0], b[0])
    for x, y in zip(a[1:], b[1:]):
        assert torch.equal(x.contiguous().view(torch.uint8), y.contiguous().view(torch.uint8))
    # and the last root is the oracle's hash of the final state
    wf = O.widen_bf16(U.bits16(b[1])) if pdt == torch.bfloat16 else b[1].cpu().numpy()
    assert int(b[0][-1]) == O.state_hash(T, wf, b[2].cpu().numpy(), b[3].cpu().numpy(),
                                         hash_mode=hash_mode)


def test_pipelined_roots_with_cut_chunks():
    """Shard ranges cut chunks, whose leaves are recomputed by the root passes -- on the
    hash stream, from w, m, v that the next step's AdamW must not overwrite first."""
    n, R, T = 50_001, 4, 3
    ranges = I.shard_ranges(n, 5)
    a = run(n, R, T, 0, False, ranges=ranges)
    b = run(n, R, T, 0, True, ranges=ranges)
    assert np.array_equal(a[0], b[0])
    assert torch.equal(a[1].view(torch.int32), b[1].view(torch.int32))


def test_image_read_waits_for_a_pending_root():
    n, R = 4 * 4096 + 9, 4
    ctx = rs.Repstep(n, device=DEV, hash_mode=rs.HASH_BLAKE2B)
    side = torch.cuda.Stream(DEV)
    ctx.set_hash_stream(side)
    w, m, v = I.gen_state(U.F32_WL, n=n, device=DEV)
    img = torch.empty(rs.image_bytes(n), dtype=torch.uint8, device=DEV)
    ctx.image_write(0, torch.zeros_like(w), torch.zeros_like(m), torch.zeros_like(v), img)
    grads = U.gen_grads(n, R, 1)
    root = torch.zeros(1, dtype=torch.int64, device=DEV)
    ow, om, ov = w.cpu().numpy(), m.cpu().numpy(), v.cpu().numpy()
    ctx.step(grads, w, m, v, U.hp_for(1), step=1, root_out=root)
    ctx.image_read(img, w, m, v)          # overwrites the state the audit leaves read
    ctx.sync()
    ref = U.oracle_step(U.oracle_grads(grads), ow, om, ov, 1, hash_mode=1)
    assert U.root_of(root) == ref["root"]
    assert not w.any()


def test_hash_stream_can_be_cleared():
    n, R = 9000, 2
    a = run(n, R, 2, 0, False)
    ctx = rs.Repstep(n, device=DEV)
    ctx.set_hash_stream(torch.cuda.Stream(DEV))
    ctx.set_hash_stream(None)
    w, m, v = I.gen_state(U.F32_WL, n=n, device=DEV)
    r = torch.zeros(2, dtype=torch.int64, device=DEV)
    for t in (1, 2):
        ctx.step(U.gen_grads(n, R, t, scale=2000.0 if t == 2 else 1.0), w, m, v, U.hp_for(t),
                 step=t, root_out=r[t - 1:t])
    ctx.sync()
    assert np.array_equal(r.cpu().numpy().view(np.uint64), a[0])
