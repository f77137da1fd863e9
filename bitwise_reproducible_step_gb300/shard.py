"""Sharded optimizer step: each GPU owns one chunk-aligned range of the flat parameters.

"OPEN-1B: A Fully Auditable Training Run", App. A.2 (reduce-scatter over shards): every
replica's slice of a shard's range is routed to the shard's owner, which sums the slices in
a fixed order.  Here the exchanges carry data only, through torch.distributed (NCCL
between GPUs, gloo between CPU processes):

  1. route_gradients -- point-to-point sends of gradient slices (an all-to-all that skips
     each rank's own slices); afterwards rank s holds every
     replica's slice of range s, in global replica order;
  2. gather_chunk_sums -- one all-gather of the ranges' 4096-element chunk sums of
     squares, which come out in chunk order;
  3. gather_leaves -- one all-gather of the ranges' chunk leaf digests, assembled in the
     image's leaf order (all w chunks, then all m chunks, then all v chunks).

Every floating-point sum -- the replica tree of each element, the chunk sums, the tree
over all chunk sums -- and the Merkle tree run in this library's kernels
(repstep_reduce or the single pass of repstep_fused_begin, repstep_clip_gathered,
repstep_root_gathered) in the canonical order of the unsharded step, so every bit equals
it.  No collective reduces anything.

Layout.  With c = ceil(n/4096) chunks and N ranks, rank s owns chunks [s*cr, (s+1)*cr) with
cr = ceil(c/N) (the last ranges may be shorter or empty): elements [s*S, min((s+1)*S, n))
with the stride S = cr*4096.  Rank p holds replicas [p*R/N, (p+1)*R/N) of the whole model
(N divides R).  The routing is point-to-point: each rank sends every peer the slices of its
replicas that fall in the peer's range and receives the peers' slices of its own range
into slots of S elements (so each starts on a 16-byte boundary); the slices of its own
replicas it reads in place, so one rank moves nothing.
"""
from __future__ import annotations

import dataclasses

import torch
import torch.distributed as dist

CHUNK = 4096


@dataclasses.dataclass(frozen=True)
class ShardPlan:
    n: int          # parameters of the whole model
    world: int      # ranks (one range each)

    @property
    def c(self) -> int:
        return (self.n + CHUNK - 1) // CHUNK

    @property
    def cr(self) -> int:
        """Chunks per rank (the last ranks may own fewer)."""
        return max(1, -(-self.c // self.world))

    @property
    def stride(self) -> int:
        """Elements per rank's slot: cr whole chunks."""
        return self.cr * CHUNK

    def range_of(self, rank: int) -> tuple[int, int]:
        lo = min(rank * self.stride, self.n)
        return lo, min(lo + self.stride, self.n)

    def chunks_of(self, rank: int) -> int:
        lo, hi = self.range_of(rank)
        return (hi - lo + CHUNK - 1) // CHUNK


def _bytes(t: torch.Tensor) -> torch.Tensor:
    return t.view(torch.uint8)


def route_gradients(local_grads, plan: ShardPlan, rank: int, R: int, out=None, group=None):
    """Route gradient slices to their range's owner (data movement only: point-to-point
    sends and receives of bytes).

    local_grads: this rank's R/N replica gradients (global replicas rank*R/N + j), each a
    contiguous buffer of at least n elements.  Returns R tensors of len(range) elements in
    global replica order: replica r's slice of this rank's range -- a view into
    local_grads for this rank's own replicas, into `out` for the peers'.  out: optional
    receive buffer of shape (R/N, world - 1, stride) and the gradient dtype."""
    N = plan.world
    if R % N:
        raise ValueError("the replica count must be a multiple of the world size")
    Rl = R // N
    local_grads = list(local_grads)
    if len(local_grads) != Rl:
        raise ValueError(f"rank holds {len(local_grads)} replicas, expected R/N = {Rl}")
    dt, dev = local_grads[0].dtype, local_grads[0].device
    for g in local_grads:
        if g.dtype != dt or not g.is_contiguous() or g.numel() < plan.n:
            raise ValueError(f"gradients: contiguous {dt} buffers of at least n = {plan.n} "
                             "elements")
    if out is None:
        out = torch.empty((Rl, max(N - 1, 0), plan.stride), dtype=dt, device=dev)
    lo, hi = plan.range_of(rank)

    def slot(q):                   # the receive slot of peer q
        return q if q < rank else q - 1

    ops = []
    for j, g in enumerate(local_grads):
        for p in range(N):
            if p == rank:
                continue
            plo, phi = plan.range_of(p)
            if phi > plo:
                ops.append(dist.P2POp(dist.isend, _bytes(g[plo:phi]), p, group))
            if hi > lo:
                ops.append(dist.P2POp(dist.irecv, _bytes(out[j, slot(p), :hi - lo]), p, group))
    if ops:
        for req in dist.batch_isend_irecv(ops):
            req.wait()
    routed = []
    for r in range(R):
        q, j = divmod(r, Rl)       # global replica r = q * Rl + j, peer q's j-th replica
        routed.append(local_grads[j][lo:hi] if q == rank else out[j, slot(q), :hi - lo])
    return routed


def pack_chunk_sums(local_sums: torch.Tensor, plan: ShardPlan, rank: int) -> torch.Tensor:
    """This rank's contribution to the chunk-sum all-gather: its plan.chunks_of(rank) sums
    in a slot of cr, zero-padded."""
    send = torch.zeros(plan.cr, dtype=torch.float32, device=local_sums.device)
    k = plan.chunks_of(rank)
    send[:k].copy_(local_sums[:k])
    return send


def unpack_chunk_sums(gathered: torch.Tensor, plan: ShardPlan) -> torch.Tensor:
    """The world slots of cr gathered in rank order hold the c chunk sums in chunk order,
    then padding."""
    return gathered.view(-1)[:plan.c]


def gather_chunk_sums(local_sums: torch.Tensor, plan: ShardPlan, rank: int, group=None):
    """All-gather of the ranges' chunk sums of squares (fp32, this rank's
    plan.chunks_of(rank) of them); returns all c sums in chunk order."""
    send = pack_chunk_sums(local_sums, plan, rank)
    out = torch.empty(plan.world * plan.cr, dtype=torch.float32, device=send.device)
    dist.all_gather_into_tensor(out, send, group=group)
    return unpack_chunk_sums(out, plan)


def pack_leaves(local_leaves: torch.Tensor, plan: ShardPlan, rank: int) -> torch.Tensor:
    """This rank's contribution to the leaf all-gather: from its leaf array (u64 as int64)
    [header, w chunks, m chunks, v chunks] of its own range, the three chunk rows, each
    zero-padded to cr: shape (3, cr)."""
    k = plan.chunks_of(rank)
    send = torch.zeros((3, plan.cr), dtype=torch.int64, device=local_leaves.device)
    if k:
        send[:, :k].copy_(local_leaves[1:1 + 3 * k].view(3, k))
    return send


def unpack_leaves(gathered: torch.Tensor, plan: ShardPlan) -> torch.Tensor:
    """From the gathered (world, 3, cr) rows, the 1 + 3c leaves of the whole state in image
    order (all w chunks, all m chunks, all v chunks), slot 0 (the header leaf) zero."""
    N, cr, c = plan.world, plan.cr, plan.c
    leaves = torch.zeros(1 + 3 * c, dtype=torch.int64, device=gathered.device)
    leaves[1:].view(3, c).copy_(gathered.view(N, 3, cr).permute(1, 0, 2).reshape(3, N * cr)[:, :c])
    return leaves


def gather_leaves(local_leaves: torch.Tensor, plan: ShardPlan, rank: int, group=None):
    """All-gather of the ranges' chunk leaf digests: the 1 + 3c leaves of the whole state in
    image order, slot 0 zero (repstep_root_gathered writes the header leaf there)."""
    send = pack_leaves(local_leaves, plan, rank)
    gathered = torch.empty((plan.world, 3, plan.cr), dtype=torch.int64, device=send.device)
    dist.all_gather_into_tensor(gathered.view(-1), send.view(-1), group=group)
    return unpack_leaves(gathered, plan)


class ShardedStep:
    """One rank's part of a sharded step on its GPU, through the C ABI.

    The rank owns the state (w, m, v) of its range, allocated by the caller with
    len(range) elements each; its context's n is that length.  step() runs: route the
    gradients -> repstep_reduce on the received slices -> gather the chunk sums ->
    repstep_clip_gathered -> repstep_adamw (its chunk leaves fused) -> (audit mode:
    repstep_leaves) -> gather the leaves -> repstep_root_gathered.  The norm and the root
    are the whole model's, the same on every rank and equal to the unsharded step's."""

    def __init__(self, n: int, R: int, rank: int, world: int, device, group=None,
                 grad_dtype=torch.float32, ctx=None, **ctx_kw):
        """ctx: the rank's context over its range (default: a new Repstep of n = the
        range's length on `device`, built with ctx_kw); anything with the same calls
        works, which lets the exchanges be exercised without a GPU."""
        self.plan = ShardPlan(n, world)
        self.R, self.rank, self.group = R, rank, group
        self.lo, self.hi = self.plan.range_of(rank)
        if ctx is None:
            from . import repstep as rs
            ctx = rs.Repstep(self.hi - self.lo, grad_dtype=grad_dtype, device=device, **ctx_kw)
        self.ctx = ctx
        self.recv = torch.empty((R // world, world - 1, self.plan.stride), dtype=grad_dtype,
                                device=device)
        self.audit = self.ctx.hash_mode != 0

    def step(self, local_grads, w, m, v, hp, step: int, norm_out=None, root_out=None):
        slices = route_gradients(local_grads, self.plan, self.rank, self.R, out=self.recv,
                                 group=self.group)
        ctx = self.ctx
        ctx.reduce(slices)
        sums = gather_chunk_sums(ctx.chunk_sums_view(), self.plan, self.rank, self.group)
        ctx.clip_gathered(sums, hp.clip, norm_out=norm_out)
        ctx.adamw(w, m, v, hp)
        if self.audit:
            ctx.leaves(step, w, m, v)
        leaves = gather_leaves(ctx.leaves_view(), self.plan, self.rank, self.group)
        ctx.root_gathered(step, self.plan.n, leaves, root_out=root_out)
        return leaves

    def step_fused(self, local_grads, w, m, v, w_out, m_out, v_out, hp, step: int,
                   norm_out=None, root_out=None):
        """The same step from (w, m, v) into (w_out, m_out, v_out) with the single pass:
        route -> repstep_fused_begin on the received slices -> gather the chunk sums ->
        repstep_clip_gathered -> repstep_fused_end -> (audit mode: repstep_leaves of the
        new state) -> gather the leaves -> repstep_root_gathered.  Every rank gets the same
        norm, so every rank takes the same path; the bits equal step()'s."""
        slices = route_gradients(local_grads, self.plan, self.rank, self.R, out=self.recv,
                                 group=self.group)
        ctx = self.ctx
        ctx.fused_begin(slices, w, m, v, w_out, m_out, v_out, hp)
        sums = gather_chunk_sums(ctx.chunk_sums_view(), self.plan, self.rank, self.group)
        ctx.clip_gathered(sums, hp.clip, norm_out=norm_out)
        ctx.fused_end(slices, w, m, v, w_out, m_out, v_out, hp)
        if self.audit:
            ctx.leaves(step, w_out, m_out, v_out)
        leaves = gather_leaves(ctx.leaves_view(), self.plan, self.rank, self.group)
        ctx.root_gathered(step, self.plan.n, leaves, root_out=root_out)
        return leaves
