"""Full-size workloads on one GB300, in the launch configuration the benchmark times.

The oracle cannot redo a 1.2e9- or 3e9-parameter step in seconds, so each step is checked
as a chain of pieces the oracle computes exactly:
  * sampled whole chunks (first, last/ragged, and ~250 seeded random ones): g, the chunk
    sum of squares, the AdamW outputs and the three leaf digests, from the same gathered
    inputs, bit for bit;
  * the pre-clip norm and clip scale: the oracle's canonical tree over ALL chunk sums;
  * the Merkle root: the oracle's tree over ALL leaf digests;
and every invariance (launch shape, topology, shard ranges) is checked on the full arrays
by exact equality on the device.
"""
import hashlib

import numpy as np
import pytest
import torch

from bitwise_reproducible_step_gb300 import inputs as I
from bitwise_reproducible_step_gb300 import repstep as rs
from oracle import oracle as O
from tests import gpu_util as U

pytestmark = [pytest.mark.gpu, pytest.mark.big]

CH = 4096


@pytest.fixture(scope="module", autouse=True)
def _built():
    U.ensure_built()
    torch.cuda.set_device(0)
    yield
    torch.cuda.empty_cache()


def sample_chunks(c, k=254, seed=0):
    rng = np.random.default_rng(seed)
    pick = set(rng.choice(c, size=min(k, c), replace=False).tolist())
    pick.update([0, c - 1])
    return np.array(sorted(pick), dtype=np.int64)


def gather(t: torch.Tensor, chunks, n):
    """Host copy of whole chunks of a device array (ragged last chunk kept short)."""
    out = []
    for k in chunks:
        lo, hi = int(k) * CH, min(int(k) * CH + CH, n)
        out.append(t[lo:hi])
    return [x.cpu() for x in out]


def leaf_of(words: np.ndarray, hash_mode: int) -> int:
    if hash_mode == 0:
        return O.pf61(words.view(np.uint32))
    return int.from_bytes(hashlib.blake2b(words.astype("<f4").tobytes(), digest_size=8).digest(),
                          "little")


def check_step_chain(ctx, grads_before, state_before, w, m, v, t, chunks, n, norm_t, root_t,
                     hash_mode=0, reducer=O.reduce):
    """grads_before / state_before: host chunk lists gathered before the step."""
    c = (n + CH - 1) // CH
    chunk_sums = ctx.chunk_sums_view().cpu().numpy()
    # norm and scale: oracle tree over all GPU chunk sums
    S = O.tree_sum(chunk_sums)
    norm = np.sqrt(S, dtype=np.float32)
    norm_o = np.float32(np.sqrt(np.float32(S)))
    assert np.float32(norm_t.item()) == norm_o == norm
    scale = O.clip_scale(norm_o, U.HP["clip"])
    bc1, bc2 = O.bias_corrections(U.HP["beta1"], U.HP["beta2"], t)
    leaves = ctx.leaves_view().cpu().numpy().view(np.uint64)
    g_dev = ctx.g_view()
    new_w, new_m, new_v = gather(w, chunks, n), gather(m, chunks, n), gather(v, chunks, n)
    g_got = gather(g_dev, chunks, n)
    for i, k in enumerate(chunks):
        G = [I.to_numpy(gr[i]) for gr in grads_before]
        g = reducer(G)
        U.assert_same_f32(g_got[i], g, f"g chunk {k}")
        _, s = O.norm(g, with_chunks=True)
        assert s.view(np.uint32)[0] == chunk_sums[k:k + 1].view(np.uint32)[0], f"chunk sum {k}"
        w0, m0, v0 = (x[i].numpy() for x in state_before)
        w1, m1, v1 = O.adamw(w0, m0, v0, g, scale, U.HP["lr"], U.HP["beta1"], U.HP["beta2"],
                             U.HP["eps"], U.HP["wd"], bc1, bc2)
        U.assert_same_f32(new_w[i], w1, f"w chunk {k}")
        U.assert_same_f32(new_m[i], m1, f"m chunk {k}")
        U.assert_same_f32(new_v[i], v1, f"v chunk {k}")
        for a, arr in enumerate((w1, m1, v1)):
            assert leaves[1 + a * c + k] == leaf_of(arr, hash_mode), f"leaf {a} chunk {k}"
    hdr_words = np.array([t, n], dtype=np.uint64).astype(np.uint32)
    hdr = O.pf61(hdr_words) if hash_mode == 0 else int.from_bytes(
        hashlib.blake2b(hdr_words.astype("<u4").tobytes(), digest_size=8).digest(), "little")
    assert leaves[0] == hdr
    assert U.root_of(root_t) == O.merkle_root(leaves)
    return float(norm_o)


def run_big(wl, steps, ranges=None, compare_unsharded=False, hash_mode=0):
    n, R = wl.n, wl.R
    dev = torch.device("cuda", 0)
    gdt = torch.bfloat16 if wl.grad_dtype == "bf16" else torch.float32
    c = (n + CH - 1) // CH
    chunks = sample_chunks(c)
    if ranges:   # also sample the chunks the shard boundaries cut
        extra = {lo // CH for lo, _ in ranges[1:]}
        chunks = np.array(sorted(set(chunks.tolist()) | extra), dtype=np.int64)
    ctx = rs.Repstep(n, grad_dtype=gdt, device=dev, hash_mode=hash_mode)
    w, m, v = I.gen_state(wl, device=dev)
    twin = None
    if compare_unsharded:
        twin = (rs.Repstep(n, grad_dtype=gdt, device=dev), w.clone(), m.clone(), v.clone())
    grads = [torch.empty(n, dtype=gdt, device=dev) for _ in range(R)]
    norm = torch.empty(1, dtype=torch.float32, device=dev)
    root = torch.empty(1, dtype=torch.int64, device=dev)
    norms = []
    for t in range(1, steps + 1):
        for r in range(R):
            I.gen_grad(wl, t, r, device=dev, out=grads[r])
        g_before = [gather(gr, chunks, n) for gr in grads]
        s_before = (gather(w, chunks, n), gather(m, chunks, n), gather(v, chunks, n))
        hp = U.hp_for(t)
        if ranges:
            for lo, hi in ranges:
                ctx.reduce(grads, begin=lo, count=hi - lo)
            ctx.clip(hp.clip, norm_out=norm)
            for lo, hi in ranges:
                ctx.adamw(w, m, v, hp, begin=lo, count=hi - lo)
            ctx.root(t, root_out=root)
        else:
            ctx.step(grads, w, m, v, hp, step=t, norm_out=norm, root_out=root)
        assert ctx.sync() & ~rs.FLAG_NONFINITE_NORM == 0
        norms.append(check_step_chain(ctx, g_before, s_before, w, m, v, t, chunks, n, norm, root,
                                      hash_mode))
        if twin is not None:
            tc, tw, tm, tv = twin
            tn = torch.empty(1, dtype=torch.float32, device=dev)
            tr = torch.empty(1, dtype=torch.int64, device=dev)
            tc.step(grads, tw, tm, tv, hp, step=t, norm_out=tn, root_out=tr)
            tc.sync()
            assert torch.equal(tw.view(torch.int32), w.view(torch.int32))
            assert torch.equal(tm.view(torch.int32), m.view(torch.int32))
            assert torch.equal(tv.view(torch.int32), v.view(torch.int32))
            assert tn.item() == norm.item() and U.root_of(tr) == U.root_of(root)
    return norms


def test_flat1200m_r8_segscale():
    wl = I.WORKLOADS["flat1200m_r8_segscale"]
    norms = run_big(wl, steps=2)
    assert all(x < 1.0 for x in norms)              # tiny segment-scaled grads: no clip


def test_flat1200m_r8_segscale_audit_mode():
    """The bench workload with BLAKE2b-64 audit-mode leaves, one step."""
    wl = I.WORKLOADS["flat1200m_r8_segscale"]
    run_big(wl, steps=1, hash_mode=rs.HASH_BLAKE2B)


def test_flat3000m_r8_bf16_spiked_shards():
    wl = I.WORKLOADS["flat3000m_r8_bf16_spiked_shards"]
    norms = run_big(wl, steps=2, ranges=I.shard_ranges(wl.n, wl.shards), compare_unsharded=True)
    assert all(x > 1.0 for x in norms)              # 1% spikes x 1e3 force the clip


def test_flat268m_r32_topologies_grids_blocks():
    """4 topologies x 5 grid sizes x 3 block sizes: every output bit equal, and the
    default configuration equal to the oracle on the sampled chain."""
    wl = I.WORKLOADS["flat268m_r32_topologies"]
    n, R = wl.n, wl.R
    dev = torch.device("cuda", 0)
    c = (n + CH - 1) // CH
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    grads = [I.gen_grad(wl, 1, r, device=dev) for r in range(R)]
    w0, m0, v0 = I.gen_state(wl, device=dev)
    m0.copy_(I.gen_grad(wl, 9, 0, device=dev))       # non-zero moments: a mid-run step
    v0.copy_(I.gen_grad(wl, 9, 1, device=dev).square())
    chunks = sample_chunks(c, k=126, seed=4)
    g_before = [gather(gr, chunks, n) for gr in grads]
    s_before = (gather(w0, chunks, n), gather(m0, chunks, n), gather(v0, chunks, n))
    hp = U.hp_for(3)
    w, m, v = w0.clone(), m0.clone(), v0.clone()
    ref = None
    for nodes, gpn in wl.topologies:
        for grid in [0, 1, 7, sm, 2 * sm + 1, c]:
            for nt in ([128, 256, 512] if grid in (0, sm) else [256]):
                ctx = rs.Repstep(n, device=dev, grid_blocks=grid, block_threads=nt)
                w.copy_(w0); m.copy_(m0); v.copy_(v0)
                norm = torch.empty(1, dtype=torch.float32, device=dev)
                root = torch.empty(1, dtype=torch.int64, device=dev)
                ctx.step(grads, w, m, v, hp, step=3, norm_out=norm, root_out=root,
                         nodes=nodes, gpus_per_node=gpn)
                ctx.sync()
                if ref is None:
                    check_step_chain(ctx, g_before, s_before, w, m, v, 3, chunks, n, norm, root)
                    ref = (w.clone(), m.clone(), v.clone(), norm.item(), U.root_of(root))
                else:
                    assert torch.equal(w.view(torch.int32), ref[0].view(torch.int32)), (nodes, grid, nt)
                    assert torch.equal(m.view(torch.int32), ref[1].view(torch.int32))
                    assert torch.equal(v.view(torch.int32), ref[2].view(torch.int32))
                    assert norm.item() == ref[3] and U.root_of(root) == ref[4]
                ctx.destroy()


def test_fixed_division_is_ieee_for_every_significand_pair():
    """The AdamW kernel divides by the step's bias corrections with Markstein's correction
    from a precomputed reciprocal; compare it with IEEE division for all 2^46 pairs."""
    assert rs.selftest_fixed_division(0, 1 << 23) == 0


def test_flat268m_r32_paper_exact_order():
    """OPEN-1B Algorithm 1 order on 268M parameters: 4 replicas x 8 shards (linear shard
    sums, TreeFold over replicas), sampled chunks against the oracle's restatement."""
    wl = I.WORKLOADS["flat268m_r32_topologies"]
    n, R, dps = wl.n, wl.R, 8
    dev = torch.device("cuda", 0)
    c = (n + CH - 1) // CH
    grads = [I.gen_grad(wl, 1, r, device=dev) for r in range(R)]
    w, m, v = I.gen_state(wl, device=dev)
    chunks = sample_chunks(c, k=126, seed=5)
    g_before = [gather(gr, chunks, n) for gr in grads]
    s_before = (gather(w, chunks, n), gather(m, chunks, n), gather(v, chunks, n))
    ctx = rs.Repstep(n, device=dev)
    hp = U.hp_for(1)
    norm = torch.empty(1, dtype=torch.float32, device=dev)
    root = torch.empty(1, dtype=torch.int64, device=dev)
    ctx.reduce_paper(grads, dps)
    ctx.clip(hp.clip, norm_out=norm)
    ctx.adamw(w, m, v, hp)
    ctx.root(1, root_out=root)
    ctx.sync()
    check_step_chain(ctx, g_before, s_before, w, m, v, 1, chunks, n, norm, root,
                     reducer=lambda G: O.reduce_alg1(G, dps))


def bench_segments(n):
    """The decay segments of the benchmark's --decay-mask: no decay on a 5% embedding and
    on a 4096-element gain after every 16.7M-element block of matrices."""
    segs, e = [(0, False)], n // 20 | 1
    while e < n:
        segs.append((e, True))
        e += 16_777_216 + 3
        if e < n:
            segs.append((e, False))
            e += 4096
    return segs


def local_segments(segs, lo, hi):
    """The segment list restricted to [lo, hi), re-based to lo."""
    starts = [b for b, _ in segs]
    k = int(np.searchsorted(starts, lo, side="right")) - 1
    out = [(0, segs[k][1])]
    for b, d in segs[k + 1:]:
        if b >= hi:
            break
        out.append((b - lo, d))
    return out


def test_flat1200m_r8_bf16w_decay_mask_ftz():
    """The bench workload with all three optimizer variants at once -- bf16 parameters,
    the benchmark's decay segments and software flush-to-zero -- one step, checked on
    sampled whole chunks against the oracle's FTZ functions, the norm over all chunk sums
    and the root over all leaves."""
    wl = I.WORKLOADS["flat1200m_r8_segscale"]
    n, R = wl.n, wl.R
    dev = torch.device("cuda", 0)
    c = (n + CH - 1) // CH
    chunks = sample_chunks(c, k=190, seed=7)
    segs = bench_segments(n)
    # also sample the chunks that hold segment boundaries
    chunks = np.array(sorted(set(chunks.tolist()) | {b // CH for b, _ in segs[1:8]}), np.int64)
    ctx = rs.Repstep(n, device=dev, param_dtype=torch.bfloat16, subnormals=rs.SUBNORMALS_FTZ)
    ctx.set_decay_mask(rs.decay_mask_from_segments(n, segs).to(dev))
    w32, m, v = I.gen_state(wl, device=dev)
    w = w32.to(torch.bfloat16)
    del w32
    m.copy_(I.gen_grad(wl, 9, 0, device=dev))           # non-zero moments: a mid-run step
    v.copy_(I.gen_grad(wl, 9, 1, device=dev).square())
    grads = [I.gen_grad(wl, 3, r, device=dev) for r in range(R)]
    g_before = [gather(gr, chunks, n) for gr in grads]
    s_before = (gather(w, chunks, n), gather(m, chunks, n), gather(v, chunks, n))
    hp = U.hp_for(3)
    norm = torch.empty(1, dtype=torch.float32, device=dev)
    root = torch.empty(1, dtype=torch.int64, device=dev)
    ctx.step(grads, w, m, v, hp, step=3, norm_out=norm, root_out=root)
    assert ctx.sync() & ~rs.FLAG_NONFINITE_NORM == 0
    chunk_sums = ctx.chunk_sums_view().cpu().numpy()
    norm_o = O.flush(np.sqrt(O.tree_sum_ftz(chunk_sums), dtype=np.float32))
    assert np.float32(norm.item()) == norm_o
    scale = O.clip_scale_ftz(norm_o, U.HP["clip"])
    bc1, bc2 = O.bias_corrections_ftz(U.HP["beta1"], U.HP["beta2"], 3)
    leaves = ctx.leaves_view().cpu().numpy().view(np.uint64)
    new_w, new_m, new_v = gather(w, chunks, n), gather(m, chunks, n), gather(v, chunks, n)
    g_got = gather(ctx.g_view(), chunks, n)
    for i, k in enumerate(chunks):
        lo, hi = int(k) * CH, min(int(k) * CH + CH, n)
        g = O.reduce_ftz([I.to_numpy(gr[i]) for gr in g_before])
        U.assert_same_f32(g_got[i], g, f"g chunk {k}")
        _, s = O.norm_ftz(g, with_chunks=True)
        assert s.view(np.uint32)[0] == chunk_sums[k:k + 1].view(np.uint32)[0], f"chunk sum {k}"
        w0 = I.to_numpy(s_before[0][i])
        w1, m1, v1 = O.adamw_ftz(w0, s_before[1][i].numpy(), s_before[2][i].numpy(), g, scale,
                                 U.HP["lr"], U.HP["beta1"], U.HP["beta2"], U.HP["eps"],
                                 U.HP["wd"], bc1, bc2, segments=local_segments(segs, lo, hi))
        U.assert_same_bf16(new_w[i], w1, f"w chunk {k}")
        U.assert_same_f32(new_m[i], m1, f"m chunk {k}")
        U.assert_same_f32(new_v[i], v1, f"v chunk {k}")
        for a, arr in enumerate((O.widen_bf16(w1), m1, v1)):
            assert leaves[1 + a * c + k] == O.pf61(arr.view(np.uint32)), f"leaf {a} chunk {k}"
    assert U.root_of(root) == O.merkle_root(leaves)


@pytest.mark.parametrize("nt", [256, 512])
def test_repeated_steps_are_bit_identical(nt):
    """The same step, from the same state, 200 times: every output bit must repeat.  This
    caught a ring-refill race (a bulk copy overtaking a consumer's read of the previous
    tile) that hit about one run in 80 with 256-thread AdamW CTAs."""
    wl = I.WORKLOADS["flat268m_r32_topologies"]
    n, R = wl.n, wl.R
    dev = torch.device("cuda", 0)
    grads = [I.gen_grad(wl, 1, r, device=dev) for r in range(R)]
    w0, m0, v0 = I.gen_state(wl, device=dev)
    m0.copy_(I.gen_grad(wl, 9, 0, device=dev))
    v0.copy_(I.gen_grad(wl, 9, 1, device=dev).square())
    hp = U.hp_for(3)
    ctx = rs.Repstep(n, device=dev, block_threads=nt)
    w, m, v = w0.clone(), m0.clone(), v0.clone()
    root = torch.empty(1, dtype=torch.int64, device=dev)
    ref = None
    for _ in range(200):
        w.copy_(w0); m.copy_(m0); v.copy_(v0)
        ctx.step(grads, w, m, v, hp, step=3, root_out=root)
        assert ctx.sync() == 0
        if ref is None:
            ref = (w.clone(), m.clone(), v.clone(), U.root_of(root))
            continue
        assert U.root_of(root) == ref[3]
        assert torch.equal(w.view(torch.int32), ref[0].view(torch.int32))
    assert torch.equal(m.view(torch.int32), ref[1].view(torch.int32))
    assert torch.equal(v.view(torch.int32), ref[2].view(torch.int32))
