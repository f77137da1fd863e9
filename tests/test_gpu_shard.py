"""The sharded step on one GB300, through the C ABI (repstep_reduce on routed slices,
repstep_clip_gathered, repstep_adamw, repstep_root_gathered).

* World size 1 over NCCL, through ShardedStep: the all-gathers run for real (trivially).
* N = 2, 3, 4 and 8 ranks emulated in one process: each virtual rank has its own context
  over its chunk-aligned range; the routing delivers exactly the slices grads[r][lo:hi],
  and an all-gather's result is by definition the ranks' contributions stacked in rank order,
  so the test stacks what shard.pack_* produces and unpacks it with shard.unpack_*.  No
  kernels wait on one another.

Every rank's norm and root, and the state, must equal the unsharded repstep_step's bit for
bit ("OPEN-1B: A Fully Auditable Training Run", App. A.2), over consecutive steps, for fp32
and bf16 gradients, PF61 and audit-mode leaves, ragged sizes and ranks that own nothing; and
at 1.2e9 parameters over 8 ranges."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist

from bitwise_reproducible_step_gb300 import inputs as I
from bitwise_reproducible_step_gb300 import repstep as rs
from bitwise_reproducible_step_gb300 import shard as S
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    U.ensure_built()
    torch.cuda.set_device(0)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def emulated_step(plan, ctxs, grads, w, m, v, hp, t, audit=False):
    """One sharded step of plan.world virtual ranks in one process; returns their norms and
    roots (host values)."""
    n, N = plan.n, plan.world
    dev = w.device
    for s in range(N):
        lo, hi = plan.range_of(s)
        ctxs[s].reduce([g[lo:hi] for g in grads])
    sums = S.unpack_chunk_sums(
        torch.stack([S.pack_chunk_sums(ctxs[s].chunk_sums_view(), plan, s) for s in range(N)]),
        plan)
    norms = torch.empty(N, dtype=torch.float32, device=dev)
    roots = torch.empty(N, dtype=torch.int64, device=dev)
    for s in range(N):
        lo, hi = plan.range_of(s)
        ctxs[s].clip_gathered(sums, hp.clip, norm_out=norms[s:s + 1])
        ctxs[s].adamw(w[lo:hi], m[lo:hi], v[lo:hi], hp)
        if audit:
            ctxs[s].leaves(t, w[lo:hi], m[lo:hi], v[lo:hi])
    leaves = S.unpack_leaves(
        torch.stack([S.pack_leaves(ctxs[s].leaves_view(), plan, s) for s in range(N)]), plan)
    for s in range(N):
        ctxs[s].root_gathered(t, n, leaves, root_out=roots[s:s + 1])
    for c in ctxs:
        assert c.sync() & ~rs.FLAG_NONFINITE_NORM == 0
    return norms.cpu().numpy(), roots.cpu().numpy().view(np.uint64)


def emulated_fused_step(plan, ctxs, grads, src, dst, hp, t, audit=False):
    """The sharded single-pass step of plan.world virtual ranks in one process, from the
    state buffers `src` into `dst` (full-length tensors; each rank updates its range)."""
    n, N = plan.n, plan.world
    dev = src[0].device
    sl = [tuple(x[plan.range_of(s)[0]:plan.range_of(s)[1]] for x in (*src, *dst))
          for s in range(N)]
    for s in range(N):
        lo, hi = plan.range_of(s)
        ctxs[s].fused_begin([g[lo:hi] for g in grads], *sl[s], hp)
    sums = S.unpack_chunk_sums(
        torch.stack([S.pack_chunk_sums(ctxs[s].chunk_sums_view(), plan, s) for s in range(N)]),
        plan)
    norms = torch.empty(N, dtype=torch.float32, device=dev)
    roots = torch.empty(N, dtype=torch.int64, device=dev)
    for s in range(N):
        lo, hi = plan.range_of(s)
        ctxs[s].clip_gathered(sums, hp.clip, norm_out=norms[s:s + 1])
        ctxs[s].fused_end([g[lo:hi] for g in grads], *sl[s], hp)
        if audit:
            ctxs[s].leaves(t, *sl[s][3:])
    leaves = S.unpack_leaves(
        torch.stack([S.pack_leaves(ctxs[s].leaves_view(), plan, s) for s in range(N)]), plan)
    for s in range(N):
        ctxs[s].root_gathered(t, n, leaves, root_out=roots[s:s + 1])
    for c in ctxs:
        assert c.sync() & ~rs.FLAG_NONFINITE_NORM == 0
    return norms.cpu().numpy(), roots.cpu().numpy().view(np.uint64)


FUSED_CASES = [
    # n, N, R, grad dtype, hash mode
    (5 * 4096 * 4 + 1234, 4, 8, torch.float32, rs.HASH_PF61),
    (5 * 4096 * 4 + 1234, 2, 4, torch.bfloat16, rs.HASH_BLAKE2B),
    (2 * 4096 + 5, 4, 4, torch.float32, rs.HASH_PF61),          # the last rank owns nothing
    (4096 * 4100, 2, 8, torch.float32, rs.HASH_PF61),           # c > 4096: two-pass norm
]


@pytest.mark.parametrize("n,N,R,gdt,hm", FUSED_CASES)
def test_emulated_ranks_fused_equal_unsharded_step(n, N, R, gdt, hm):
    """repstep_fused_begin / repstep_clip_gathered / repstep_fused_end on every virtual
    rank, steps that do not clip, clip, clip and do not (every path of the prediction), the
    state buffers alternating: the norm, root and state equal repstep_step's."""
    dev = torch.device("cuda", 0)
    plan = S.ShardPlan(n, N)
    ref = rs.Repstep(n, grad_dtype=gdt, device=dev, hash_mode=hm)
    ctxs = [rs.Repstep(plan.range_of(s)[1] - plan.range_of(s)[0], grad_dtype=gdt, device=dev,
                       hash_mode=hm) for s in range(N)]
    wa, ma, va = I.gen_state(U.F32_WL, n=n, device=dev)
    bufs = [(wa.clone(), ma.clone(), va.clone()),
            tuple(torch.empty_like(x) for x in (wa, ma, va))]
    nr = torch.empty(1, dtype=torch.float32, device=dev)
    rr = torch.empty(1, dtype=torch.int64, device=dev)
    for t in (1, 2, 3, 4):
        grads = U.gen_grads(n, R, 40 + t, gdt, scale=2000.0 if t in (2, 3) else 1e-3)
        hp = U.hp_for(t)
        ref.step(grads, wa, ma, va, hp, step=t, norm_out=nr, root_out=rr)
        ref.sync()
        norms, roots = emulated_fused_step(plan, ctxs, grads, bufs[(t - 1) % 2], bufs[t % 2],
                                           hp, t, audit=hm != 0)
        assert all(x.view(np.uint32) == np.float32(nr.item()).view(np.uint32) for x in norms)
        assert all(int(x) == U.root_of(rr) for x in roots), (roots, U.root_of(rr))
        for a, b in zip((wa, ma, va), bufs[t % 2]):
            assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_fused_halves_check_their_order():
    dev = torch.device("cuda", 0)
    n, R = 3 * 4096, 4
    ctx = rs.Repstep(n, device=dev)
    w, m, v = I.gen_state(U.F32_WL, n=n, device=dev)
    out = tuple(torch.empty_like(x) for x in (w, m, v))
    grads = U.gen_grads(n, R, 1)
    hp = U.hp_for(1)
    with pytest.raises(rs.RepstepError):            # no first half
        ctx.fused_end(grads, w, m, v, *out, hp)
    ctx.fused_begin(grads, w, m, v, *out, hp)
    with pytest.raises(rs.RepstepError):            # before the clip
        ctx.fused_end(grads, w, m, v, *out, hp)
    ctx.clip(hp.clip)
    other = tuple(torch.empty_like(x) for x in (w, m, v))
    with pytest.raises(rs.RepstepError):            # other output buffers than the first half's
        ctx.fused_end(grads, w, m, v, *other, hp)
    ctx.fused_end(grads, w, m, v, *out, hp)
    ctx.root(1)
    assert ctx.sync() == 0


CASES = [
    # n, N, R, grad dtype, hash mode
    (5 * 4096 * 4 + 1234, 4, 8, torch.float32, rs.HASH_PF61),
    (5 * 4096 * 4 + 1234, 3, 6, torch.bfloat16, rs.HASH_BLAKE2B),
    (2 * 4096 + 5, 4, 4, torch.float32, rs.HASH_PF61),          # the last rank owns nothing
    (300_001, 2, 2, torch.bfloat16, rs.HASH_PF61),
    (4096 * 4100, 2, 4, torch.float32, rs.HASH_PF61),           # c > 4096: two-pass norm
]


@pytest.mark.parametrize("n,N,R,gdt,hm", CASES)
def test_emulated_ranks_equal_unsharded_step(n, N, R, gdt, hm):
    dev = torch.device("cuda", 0)
    plan = S.ShardPlan(n, N)
    ref = rs.Repstep(n, grad_dtype=gdt, device=dev, hash_mode=hm)
    ctxs = [rs.Repstep(plan.range_of(s)[1] - plan.range_of(s)[0], grad_dtype=gdt, device=dev,
                       hash_mode=hm) for s in range(N)]
    wa, ma, va = I.gen_state(U.F32_WL, n=n, device=dev)
    wb, mb, vb = wa.clone(), ma.clone(), va.clone()
    nr = torch.empty(1, dtype=torch.float32, device=dev)
    rr = torch.empty(1, dtype=torch.int64, device=dev)
    for t in (1, 2, 3):
        grads = U.gen_grads(n, R, t, gdt, scale=2000.0 if t == 2 else 1.0)
        hp = U.hp_for(t)
        ref.step(grads, wa, ma, va, hp, step=t, norm_out=nr, root_out=rr)
        ref.sync()
        norms, roots = emulated_step(plan, ctxs, grads, wb, mb, vb, hp, t, audit=hm != 0)
        assert all(x.view(np.uint32) == np.float32(nr.item()).view(np.uint32) for x in norms)
        assert all(int(x) == U.root_of(rr) for x in roots), (roots, U.root_of(rr))
        for a, b in ((wa, wb), (ma, mb), (va, vb)):
            assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_gathered_calls_check_their_arguments():
    dev = torch.device("cuda", 0)
    plan = S.ShardPlan(3 * 4096, 3)
    ctx = rs.Repstep(4096, device=dev)
    sums = torch.zeros(plan.c, dtype=torch.float32, device=dev)
    with pytest.raises(rs.RepstepError):            # before the local reduce: call order
        ctx.clip_gathered(sums, 1.0)
    grads = U.gen_grads(4096, 2, 1)
    ctx.reduce(grads)
    with pytest.raises(rs.RepstepError):            # fewer chunk sums than the context's own
        ctx.clip_gathered(sums[:0], 1.0)
    ctx.clip_gathered(sums, 1.0)
    leaves = torch.zeros(1 + 3 * plan.c, dtype=torch.int64, device=dev)
    with pytest.raises(rs.RepstepError):            # before AdamW: call order
        ctx.root_gathered(1, plan.n, leaves)
    w, m, v = I.gen_state(U.F32_WL, n=4096, device=dev)
    ctx.adamw(w, m, v, U.hp_for(1))
    with pytest.raises(rs.RepstepError):            # n_total below the context's n
        ctx.root_gathered(1, 100, leaves)
    ctx.root_gathered(1, plan.n, leaves)
    assert ctx.sync() == 0


@pytest.mark.parametrize("gdt,hm", [(torch.float32, rs.HASH_PF61),
                                    (torch.bfloat16, rs.HASH_BLAKE2B)])
def test_world_one_over_nccl_equals_unsharded_step(gdt, hm):
    """ShardedStep with a real NCCL process group of one rank: the routing reads the rank's
    own slices in place, the two all-gathers run (as copies), and the bits equal
    repstep_step's."""
    dev = torch.device("cuda", 0)
    n, R = 3 * 4096 * 5 + 333, 4
    os.environ.setdefault("NCCL_NVLS_ENABLE", "0")
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{_free_port()}", rank=0,
                            world_size=1, device_id=dev)
    try:
        step = S.ShardedStep(n, R, 0, 1, dev, grad_dtype=gdt, hash_mode=hm)
        ref = rs.Repstep(n, grad_dtype=gdt, device=dev, hash_mode=hm)
        wa, ma, va = I.gen_state(U.F32_WL, n=n, device=dev)
        wb, mb, vb = wa.clone(), ma.clone(), va.clone()
        nr = torch.empty(2, dtype=torch.float32, device=dev)
        rr = torch.empty(2, dtype=torch.int64, device=dev)
        for t in (1, 2):
            grads = U.gen_grads(n, R, t, gdt)
            hp = U.hp_for(t)
            ref.step(grads, wa, ma, va, hp, step=t, norm_out=nr[0:1], root_out=rr[0:1])
            step.step(grads, wb, mb, vb, hp, t, norm_out=nr[1:2], root_out=rr[1:2])
            ref.sync()
            step.ctx.sync()
            assert nr[0].item() == nr[1].item()
            rh = rr.cpu().numpy().view(np.uint64)
            assert rh[0] == rh[1]
            for a, b in ((wa, wb), (ma, mb), (va, vb)):
                assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    finally:
        dist.destroy_process_group()


def test_world_one_over_nccl_fused_equals_unsharded_step():
    """ShardedStep.step_fused with a real NCCL process group of one rank, the state buffers
    alternating, over steps that clip and do not."""
    dev = torch.device("cuda", 0)
    n, R = 3 * 4096 * 5 + 333, 8
    os.environ.setdefault("NCCL_NVLS_ENABLE", "0")
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{_free_port()}", rank=0,
                            world_size=1, device_id=dev)
    try:
        step = S.ShardedStep(n, R, 0, 1, dev)
        ref = rs.Repstep(n, device=dev)
        wa, ma, va = I.gen_state(U.F32_WL, n=n, device=dev)
        bufs = [(wa.clone(), ma.clone(), va.clone()),
                tuple(torch.empty_like(x) for x in (wa, ma, va))]
        nr = torch.empty(2, dtype=torch.float32, device=dev)
        rr = torch.empty(2, dtype=torch.int64, device=dev)
        for t in (1, 2, 3):
            grads = U.gen_grads(n, R, t, scale=2000.0 if t == 2 else 1e-3)
            hp = U.hp_for(t)
            ref.step(grads, wa, ma, va, hp, step=t, norm_out=nr[0:1], root_out=rr[0:1])
            step.step_fused(grads, *bufs[(t - 1) % 2], *bufs[t % 2], hp, t, norm_out=nr[1:2],
                            root_out=rr[1:2])
            ref.sync()
            step.ctx.sync()
            assert nr[0].item() == nr[1].item()
            rh = rr.cpu().numpy().view(np.uint64)
            assert rh[0] == rh[1]
            for a, b in zip((wa, ma, va), bufs[t % 2]):
                assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    finally:
        dist.destroy_process_group()


@pytest.mark.big
def test_flat1200m_r8_eight_emulated_ranks():
    """The 1.2e9-parameter workload split over 8 ranges (c = 292,969 chunks: the gathered
    norm and the Merkle tree take several passes), one step, equal to the unsharded step."""
    wl = I.WORKLOADS["flat1200m_r8_segscale"]
    n, R, N = wl.n, wl.R, 8
    dev = torch.device("cuda", 0)
    plan = S.ShardPlan(n, N)
    grads = [I.gen_grad(wl, 1, r, device=dev) for r in range(R)]
    wa, ma, va = I.gen_state(wl, device=dev)
    wb, mb, vb = wa.clone(), ma.clone(), va.clone()
    hp = U.hp_for(1)
    ref = rs.Repstep(n, device=dev)
    nr = torch.empty(1, dtype=torch.float32, device=dev)
    rr = torch.empty(1, dtype=torch.int64, device=dev)
    ref.step(grads, wa, ma, va, hp, step=1, norm_out=nr, root_out=rr)
    ref.sync()
    del ref
    ctxs = [rs.Repstep(plan.range_of(s)[1] - plan.range_of(s)[0], device=dev) for s in range(N)]
    norms, roots = emulated_step(plan, ctxs, grads, wb, mb, vb, hp, 1)
    assert all(x.view(np.uint32) == np.float32(nr.item()).view(np.uint32) for x in norms)
    assert all(int(x) == U.root_of(rr) for x in roots)
    for a, b in ((wa, wb), (ma, mb), (va, vb)):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
