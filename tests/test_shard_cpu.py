"""The sharded step's exchange layer (bitwise_reproducible_step_gb300/shard.py) on CPU
processes over gloo, world sizes 2 and 4.

Each rank holds R/N replica gradients of the whole model and one chunk-aligned range of the
state.  The test checks the three exchanges byte for byte:
  * route_gradients delivers every replica's slice of the rank's range, in global replica
    order, bit-exact (fp32 and bf16), its own replicas' slices read in place;
  * gather_chunk_sums returns every chunk's sum of squares in chunk order;
  * gather_leaves returns every chunk leaf in image order.
The per-rank arithmetic here is the oracle's (the test's stand-in for the GPU kernels): the
reduce of the routed slices, the chunk sums and AdamW of the local range, its leaves.  Fed
the gathered arrays, the oracle's tree over the chunk sums and its Merkle tree must give the
unsharded step's norm and root, and every rank the same ones ("OPEN-1B: A Fully Auditable
Training Run", App. A.2: reduce-scatter into shards before the optimizer step)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from bitwise_reproducible_step_gb300 import shard as S

CH = 4096
HP = dict(lr=np.float32(3e-4), beta1=np.float32(0.9), beta2=np.float32(0.999),
          eps=np.float32(1e-8), wd=np.float32(0.1), clip=np.float32(1.0))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(n, R, bf16, seed):
    """Every replica's gradient (host numpy: fp32, or bf16 as uint16 bits) and the state."""
    rng = np.random.default_rng(seed)
    grads = []
    for r in range(R):
        x = (rng.standard_normal(n) * 10.0 ** (-3 + r % 3)).astype(np.float32)
        if bf16:
            x = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        grads.append(x)
    w = (rng.standard_normal(n) * 0.02).astype(np.float32)
    m = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    v = ((rng.standard_normal(n) * 1e-3) ** 2).astype(np.float32)
    return grads, w, m, v


def _as_tensor(x, bf16):
    """A gradient buffer as the exchange takes it."""
    if bf16:
        return torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16)
    return torch.from_numpy(x.copy())


def _host(t):
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def _rank_main(rank, world, port, n, R, bf16, t, seed):
    from oracle import oracle as O
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        plan = S.ShardPlan(n, world)
        grads, w, m, v = _inputs(n, R, bf16, seed)
        Rl = R // world
        mine = [_as_tensor(grads[rank * Rl + j], bf16) for j in range(Rl)]
        lo, hi = plan.range_of(rank)

        # 1. routing: every replica's slice of this range, global replica order, bit-exact
        slices = S.route_gradients(mine, plan, rank, R)
        assert len(slices) == R
        for r in range(R):
            got = _host(slices[r])
            assert got.shape == (hi - lo,)
            assert np.array_equal(got.view(np.uint16 if bf16 else np.uint32),
                                  grads[r][lo:hi].view(np.uint16 if bf16 else np.uint32)), r

        # the rank's arithmetic (oracle as the stand-in for the GPU kernels)
        g_loc = O.reduce([_host(s) for s in slices]) if hi > lo else np.zeros(0, np.float32)
        _, sums_loc = O.norm(g_loc, with_chunks=True) if hi > lo else (0, np.zeros(0, np.float32))

        # 2. chunk sums gathered in chunk order = the unsharded oracle's
        sums = S.gather_chunk_sums(torch.from_numpy(np.ascontiguousarray(sums_loc)), plan, rank)
        g_all = O.reduce(grads)
        norm_all, sums_all = O.norm(g_all, with_chunks=True)
        assert np.array_equal(sums.numpy().view(np.uint32), sums_all.view(np.uint32))
        norm = np.sqrt(O.tree_sum(sums.numpy()), dtype=np.float32)
        assert norm.view(np.uint32) == np.float32(norm_all).view(np.uint32)

        # 3. AdamW of the local range, its leaves, gathered in image order
        scale = O.clip_scale(norm, HP["clip"])
        bc1, bc2 = O.bias_corrections(HP["beta1"], HP["beta2"], t)
        hpv = (scale, HP["lr"], HP["beta1"], HP["beta2"], HP["eps"], HP["wd"], bc1, bc2)
        w1, m1, v1 = O.adamw(w[lo:hi], m[lo:hi], v[lo:hi], g_loc, *hpv)
        leaves_loc = O.leaves(t, w1, m1, v1) if hi > lo else np.zeros(1, np.uint64)
        leaves = S.gather_leaves(torch.from_numpy(leaves_loc.view(np.int64)), plan, rank)
        W, M, V = O.adamw(w, m, v, g_all, *hpv)
        want = O.leaves(t, W, M, V)
        got = leaves.numpy().view(np.uint64)
        assert got[0] == 0 and np.array_equal(got[1:], want[1:])
        got = got.copy()
        got[0] = O.pf61(np.array([t, n], np.uint32))
        assert O.merkle_root(got) == O.state_hash(t, W, M, V)
        # every rank ends with the same norm and root
        both = torch.tensor([int(norm.view(np.uint32)), O.merkle_root(got) & (2 ** 62 - 1)],
                            dtype=torch.int64)
        allv = [torch.empty_like(both) for _ in range(world)]
        dist.all_gather(allv, both)
        assert all(torch.equal(x, allv[0]) for x in allv)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,n,R,bf16", [
    (2, 5 * CH * 2 + 1234, 8, False),        # ragged last chunk
    (2, 3 * CH, 2, True),                    # one replica per rank, bf16
    (4, 7 * CH + 17, 8, False),              # uneven: cr = 2, the last rank owns 2 chunks
    (4, 2 * CH + 5, 4, True),                # c = 3 < world: the last rank owns nothing
])
def test_sharded_exchange_equals_unsharded_oracle(world, n, R, bf16):
    mp.spawn(_rank_main, args=(world, _free_port(), n, R, bf16, 2, 11 + world), nprocs=world,
             join=True)


def test_plan_ranges_cover_the_chunk_grid():
    for n, N in [(1, 1), (4096, 3), (5 * CH + 7, 2), (10 ** 6, 8), (1_200_000_000, 8),
                 (3_000_000_000, 8), (2 * CH + 5, 4)]:
        p = S.ShardPlan(n, N)
        ranges = [p.range_of(s) for s in range(N)]
        assert ranges[0][0] == 0 and ranges[-1][1] == n
        for (a, b), (c, d) in zip(ranges, ranges[1:]):
            assert b == c
        for lo, hi in ranges:
            assert (lo % CH == 0 or lo == n) and (hi % CH == 0 or hi == n) and hi - lo <= p.stride
        assert sum(p.chunks_of(s) for s in range(N)) == p.c
        assert p.stride % CH == 0 and N * p.stride >= n


def test_route_rejects_short_or_miscounted_buffers():
    p = S.ShardPlan(3 * CH + 1, 2)
    with pytest.raises(ValueError):
        S.route_gradients([torch.zeros(3 * CH)], p, 0, 2)            # shorter than n
    with pytest.raises(ValueError):
        S.route_gradients([torch.zeros(p.n)] * 2, p, 0, 2)           # R/N = 1 expected
    with pytest.raises(ValueError):
        S.route_gradients([torch.zeros(p.n)], p, 0, 3)               # N does not divide R


class OracleCtx:
    """The test's stand-in for one rank's repstep context on the CPU: the calls ShardedStep
    makes, computed by the oracle on CPU tensors.  It lets ShardedStep's own sequence of
    exchanges and calls run across gloo ranks without a GPU."""

    def __init__(self, n, hash_mode=0):
        self.n, self.c, self.hash_mode = n, (n + CH - 1) // CH, hash_mode
        self.g = np.zeros(n, np.float32)
        self.cs = np.zeros(self.c, np.float32)
        self.lv = np.zeros(1 + 3 * self.c, np.uint64)
        self.scale = np.float32(1.0)

    def reduce(self, slices):
        from oracle import oracle as O
        if self.n:
            self.g = O.reduce([_host(s) for s in slices])
            _, self.cs = O.norm(self.g, with_chunks=True)

    def chunk_sums_view(self):
        return torch.from_numpy(self.cs)

    def clip_gathered(self, sums, clip, norm_out=None):
        from oracle import oracle as O
        norm = np.sqrt(O.tree_sum(sums.numpy()), dtype=np.float32)
        self.scale = O.clip_scale(norm, clip)
        if norm_out is not None:
            norm_out[0] = float(norm)

    def adamw(self, w, m, v, hp):
        from oracle import oracle as O
        if not self.n:
            return
        w1, m1, v1 = O.adamw(w.numpy(), m.numpy(), v.numpy(), self.g, self.scale, hp.lr,
                             hp.beta1, hp.beta2, hp.eps, hp.weight_decay, hp.bc1, hp.bc2)
        w.copy_(torch.from_numpy(w1)); m.copy_(torch.from_numpy(m1)); v.copy_(torch.from_numpy(v1))
        self.lv = O.leaves(0, w1, m1, v1)          # the chunk leaves; the header is not used

    def fused_begin(self, slices, w, m, v, w_out, m_out, v_out, hp):
        self.reduce(slices)

    def fused_end(self, slices, w, m, v, w_out, m_out, v_out, hp):
        for dst, src in ((w_out, w), (m_out, m), (v_out, v)):
            dst.copy_(src)
        self.adamw(w_out, m_out, v_out, hp)

    def leaves(self, step, w, m, v):
        from oracle import oracle as O
        if self.n:
            self.lv = O.leaves(step, w.numpy(), m.numpy(), v.numpy(), self.hash_mode)

    def leaves_view(self):
        return torch.from_numpy(self.lv.view(np.int64))

    def root_gathered(self, step, n_total, leaves, root_out=None):
        from oracle import oracle as O
        L = leaves.numpy().view(np.uint64).copy()
        hdr = np.array([step, n_total], np.uint32)
        L[0] = O.pf61(hdr) if self.hash_mode == 0 else \
            int.from_bytes(O.blake2b(hdr.astype("<u4").tobytes(), 8), "little")
        if root_out is not None:
            root_out[0] = int(np.array([O.merkle_root(L)], np.uint64).view(np.int64)[0])


def _sharded_step_main(rank, world, port, n, R, bf16, hash_mode, seed, fused=False):
    from bitwise_reproducible_step_gb300 import repstep as rs
    from oracle import oracle as O
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        gdt = torch.bfloat16 if bf16 else torch.float32
        lo, hi = S.ShardPlan(n, world).range_of(rank)
        step = S.ShardedStep(n, R, rank, world, "cpu", grad_dtype=gdt,
                             ctx=OracleCtx(hi - lo, hash_mode))
        assert (step.lo, step.hi) == (lo, hi)
        _, W, M, V = _inputs(n, R, bf16, seed)
        w, m, v = (torch.from_numpy(x[lo:hi].copy()) for x in (W, M, V))
        other = tuple(torch.empty_like(x) for x in (w, m, v))
        Rl = R // world
        for t in (1, 2):
            grads, _, _, _ = _inputs(n, R, bf16, seed + 100 * t)
            mine = [_as_tensor(grads[rank * Rl + j], bf16) for j in range(Rl)]
            hp = rs.hparams(lr=HP["lr"], beta1=HP["beta1"], beta2=HP["beta2"], eps=HP["eps"],
                            weight_decay=HP["wd"], clip=HP["clip"], t=t)
            norm = torch.zeros(1, dtype=torch.float32)
            root = torch.zeros(1, dtype=torch.int64)
            if fused:                    # from (w, m, v) into the other buffers, then swap
                step.step_fused(mine, w, m, v, *other, hp, t, norm_out=norm, root_out=root)
                (w, m, v), other = other, (w, m, v)
            else:
                step.step(mine, w, m, v, hp, t, norm_out=norm, root_out=root)
            ref = O.step(grads, W, M, V, lr=HP["lr"], beta1=HP["beta1"], beta2=HP["beta2"],
                         eps=HP["eps"], wd=HP["wd"], clip=HP["clip"], t=t, hash_mode=hash_mode)
            W, M, V = ref["w"], ref["m"], ref["v"]
            assert np.float32(norm.item()).view(np.uint32) == np.float32(ref["norm"]).view(np.uint32)
            assert int(root.numpy().view(np.uint64)[0]) == ref["root"], (rank, t)
            for a, b in ((w, W), (m, M), (v, V)):
                assert np.array_equal(a.numpy().view(np.uint32), b[lo:hi].view(np.uint32))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,n,R,bf16,hash_mode", [
    (2, 4 * CH * 2 + 999, 4, False, 0),
    (4, 9 * CH + 1, 8, True, 1),             # bf16 gradients, audit-mode leaves
    (4, 2 * CH + 5, 4, False, 0),            # the last rank owns nothing
])
def test_sharded_step_across_ranks_equals_unsharded_oracle(world, n, R, bf16, hash_mode):
    """ShardedStep's own sequence -- routing, local reduce, chunk-sum gather, gathered clip,
    AdamW, leaf gather, gathered root -- over gloo ranks, two steps, against the unsharded
    oracle step: every rank's norm, root and state range bit for bit."""
    from bitwise_reproducible_step_gb300 import build
    build.build()                             # the host-side bias corrections
    mp.spawn(_sharded_step_main, args=(world, _free_port(), n, R, bf16, hash_mode, 31 + world),
             nprocs=world, join=True)


@pytest.mark.parametrize("world,n,R,bf16,hash_mode", [
    (2, 4 * CH * 2 + 999, 4, False, 0),
    (4, 9 * CH + 1, 8, True, 1),
])
def test_sharded_fused_step_across_ranks_equals_unsharded_oracle(world, n, R, bf16, hash_mode):
    """ShardedStep.step_fused's sequence -- routing, the first half of the single-pass
    step, chunk-sum gather, gathered clip, the second half into the other state buffer,
    leaf gather, gathered root -- over gloo ranks, two steps with the buffers alternating,
    against the unsharded oracle step."""
    from bitwise_reproducible_step_gb300 import build
    build.build()
    mp.spawn(_sharded_step_main,
             args=(world, _free_port(), n, R, bf16, hash_mode, 77 + world, True),
             nprocs=world, join=True)
