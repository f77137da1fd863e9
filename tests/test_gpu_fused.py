"""repstep_step_fused through the C ABI: the single-pass step (reduce, chunk sums, AdamW with
the clip scale taken as 1 into a second state buffer, PF61 leaves) with its second pass when
the step clips, and the two passes taken directly after a step that clipped.  Every output
bit -- the new w, m, v, the pre-clip norm, the root and the leaves -- must equal
repstep_step's on the same inputs, step after step with the two state buffers alternating,
on all four paths (predicted no clip and none; predicted no clip and a clip; predicted a
clip and one; predicted a clip and none); the input state must be left untouched.
The single pass covers R = 4, 8 and 16 with any gradient and parameter dtype,
arithmetic mode, decay mask and hash mode; other replica counts and launch shapes take the
two ordinary passes into the output buffers, with the same bits."""
import ctypes as C

import numpy as np
import pytest
import torch

from bitwise_reproducible_step_gb300 import inputs as I
from bitwise_reproducible_step_gb300 import repstep as rs
from tests import gpu_util as U

pytestmark = pytest.mark.gpu

CH = 4096


@pytest.fixture(scope="module", autouse=True)
def _built():
    U.ensure_built()
    torch.cuda.set_device(0)


# no clip, then three that clip, then two that do not: every path of the prediction
CLIPS = (2, 3, 4)


def run_pair(n, R, gdt=torch.float32, steps=6, clip_steps=CLIPS, ctx_kw=None,
             hash_stream=False, mask_segs=None):
    """Steps of repstep_step (in place) and of repstep_step_fused (alternating buffers) on the
    same gradients; steps in clip_steps get gradients large enough to clip."""
    dev = torch.device("cuda", 0)
    ctx_kw = dict(ctx_kw or {})
    a = rs.Repstep(n, grad_dtype=gdt, device=dev, **ctx_kw)
    b = rs.Repstep(n, grad_dtype=gdt, device=dev, **ctx_kw)
    if hash_stream:
        a.set_hash_stream(torch.cuda.Stream(dev))
        b.set_hash_stream(torch.cuda.Stream(dev))
    if mask_segs:
        mask = rs.decay_mask_from_segments(n, mask_segs).to(dev)
        a.set_decay_mask(mask)
        b.set_decay_mask(mask)
    pdt = ctx_kw.get("param_dtype", torch.float32)
    w, m, v = I.gen_state(U.F32_WL, n=n, device=dev)
    m.copy_(I.gen_grad(U.F32_WL, 9, 0, n=n, device=dev))           # mid-run moments
    v.copy_(I.gen_grad(U.F32_WL, 9, 1, n=n, device=dev).square())
    w = w.to(pdt)
    bufs = [(w.clone(), m.clone(), v.clone()),
            (torch.full_like(w, float("nan")), torch.full_like(m, float("nan")),
             torch.full_like(v, float("nan")))]
    nr = torch.empty(2, dtype=torch.float32, device=dev)
    rr = torch.empty(2, dtype=torch.int64, device=dev)
    clipped = 0
    for t in range(1, steps + 1):
        scale = 3000.0 if t in clip_steps else 1e-3
        grads = U.gen_grads(n, R, 60 + t, gdt, scale=scale)
        hp = U.hp_for(t)
        a.step(grads, w, m, v, hp, step=t, norm_out=nr[0:1], root_out=rr[0:1])
        src, dst = bufs[(t - 1) % 2], bufs[t % 2]
        before = [x.clone() for x in src]
        b.step_fused(grads, *src, *dst, hp, step=t, norm_out=nr[1:2], root_out=rr[1:2])
        assert a.sync() & ~rs.FLAG_NONFINITE_NORM == 0
        assert b.sync() & ~rs.FLAG_NONFINITE_NORM == 0
        for x, y in zip(before, src):                         # the inputs are untouched
            assert torch.equal(x.view(torch.int16 if x.dtype == torch.bfloat16 else torch.int32),
                               y.view(torch.int16 if y.dtype == torch.bfloat16 else torch.int32))
        nb = nr.cpu().numpy().view(np.uint32)
        assert nb[0] == nb[1], (t, nr)
        rh = rr.cpu().numpy().view(np.uint64)
        assert rh[0] == rh[1], t
        for x, y, what in zip((w, m, v), dst, "wmv"):
            xi = x.view(torch.int16 if x.dtype == torch.bfloat16 else torch.int32)
            yi = y.view(torch.int16 if y.dtype == torch.bfloat16 else torch.int32)
            assert torch.equal(xi, yi), (what, t)
        assert torch.equal(a.leaves_view(), b.leaves_view()), t
        clipped += float(nr[0].item()) > 1.0
    return clipped


@pytest.mark.parametrize("n,R,hm", [(64 * CH + 1234, 8, rs.HASH_PF61),
                                    (300 * CH + 5, 4, rs.HASH_PF61),
                                    (64 * CH + 1234, 4, rs.HASH_BLAKE2B)])
def test_fused_steps_beside_pending_roots(n, R, hm):
    """With the hash stream, step t+1's single pass runs while step t's Merkle passes may
    still read their leaf snapshot: the fused steps are enqueued with no synchronisation
    between them, and every step's norm and root, and the final state and leaves, must
    equal repstep_step's run step by step on one stream."""
    dev = torch.device("cuda", 0)
    steps, clips = 7, (3, 4)
    a = rs.Repstep(n, device=dev, hash_mode=hm)
    b = rs.Repstep(n, device=dev, hash_mode=hm)
    b.set_hash_stream(torch.cuda.Stream(dev))
    w, m, v = I.gen_state(U.F32_WL, n=n, device=dev)
    bufs = [(w.clone(), m.clone(), v.clone()), tuple(torch.empty_like(x) for x in (w, m, v))]
    grads = [U.gen_grads(n, R, 90 + t, scale=3000.0 if t in clips else 1e-3)
             for t in range(1, steps + 1)]
    na = torch.empty(steps, dtype=torch.float32, device=dev)
    ra = torch.empty(steps, dtype=torch.int64, device=dev)
    nb, rb = torch.empty_like(na), torch.empty_like(ra)
    for t in range(1, steps + 1):
        a.step(grads[t - 1], w, m, v, U.hp_for(t), step=t, norm_out=na[t - 1:t],
               root_out=ra[t - 1:t])
        a.sync()
    for t in range(1, steps + 1):
        b.step_fused(grads[t - 1], *bufs[(t - 1) % 2], *bufs[t % 2], U.hp_for(t), step=t,
                     norm_out=nb[t - 1:t], root_out=rb[t - 1:t])
    assert b.sync() & ~rs.FLAG_NONFINITE_NORM == 0
    assert torch.equal(na.view(torch.int32), nb.view(torch.int32))
    assert torch.equal(ra, rb)
    for x, y in zip((w, m, v), bufs[steps % 2]):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))
    assert torch.equal(a.leaves_view(), b.leaves_view())


@pytest.mark.parametrize("n,R,gdt", [
    (5 * CH * 3 + 77, 8, torch.float32),
    (5 * CH * 3 + 77, 4, torch.float32),
    (300_001, 8, torch.bfloat16),
    (2 * CH + 2049, 4, torch.bfloat16),       # the last chunk's second tile is partial
    (1000, 8, torch.float32),                 # one short chunk: its second tile is empty
    (1, 4, torch.float32),
    (64 * CH, 8, torch.float32),
    (3 * CH + 5, 16, torch.float32),          # two replica stages per tile
    (2 * CH + 2049, 16, torch.bfloat16),
    (20 * CH + 999, 32, torch.float32),       # R = 32: the two passes
])
def test_fused_equals_two_pass_step(n, R, gdt):
    clipped = run_pair(n, R, gdt)
    assert clipped == 3 or n == 1              # the clipping steps clipped


def test_fused_audit_mode_and_hash_stream():
    run_pair(5 * CH * 3 + 77, 8, ctx_kw=dict(hash_mode=rs.HASH_BLAKE2B), hash_stream=True)
    run_pair(5 * CH * 3 + 77, 4, torch.bfloat16, hash_stream=True)


@pytest.mark.parametrize("kw,R,gdt", [
    (dict(param_dtype=torch.bfloat16), 8, torch.float32),       # in the single pass
    (dict(param_dtype=torch.bfloat16), 4, torch.bfloat16),
    (dict(subnormals=rs.SUBNORMALS_FTZ), 8, torch.float32),
    (dict(subnormals=rs.SUBNORMALS_FTZ, param_dtype=torch.bfloat16), 4, torch.bfloat16),
    (dict(subnormals=rs.SUBNORMALS_FTZ, param_dtype=torch.bfloat16), 16, torch.float32),
    (dict(), 3, torch.float32),                                 # R not 4, 8, 16: two passes
    (dict(), 12, torch.bfloat16),
    (dict(block_threads=256), 8, torch.float32),                # launch shape: two passes
])
def test_configuration_variants(kw, R, gdt):
    run_pair(3 * CH + 5, R, gdt, ctx_kw=kw)
    run_pair(2 * CH + 2049, R, gdt, ctx_kw=kw)                  # ragged: bulk-copy edges


@pytest.mark.parametrize("kw", [dict(), dict(param_dtype=torch.bfloat16),
                                dict(subnormals=rs.SUBNORMALS_FTZ)])
def test_decay_mask(kw):
    run_pair(3 * CH + 5, 8, mask_segs=[(0, False), (CH + 3, True), (2 * CH + 7, False)],
             ctx_kw=kw)


def test_prediction_follows_other_calls():
    """The clip outcome the prediction reads is the context's: a two-pass step or a lone
    clip between fused steps moves it, and the bits stay repstep_step's."""
    n, R = 3 * CH + 5, 8
    dev = torch.device("cuda", 0)
    a, b = rs.Repstep(n, device=dev), rs.Repstep(n, device=dev)
    w, m, v = I.gen_state(U.F32_WL, n=n, device=dev)
    bufs = [(w.clone(), m.clone(), v.clone()), tuple(torch.empty_like(x) for x in (w, m, v))]
    cur = 0
    for t, (clip, via_step) in enumerate([(True, False), (False, True), (True, True),
                                          (False, False), (True, False)], start=1):
        grads = U.gen_grads(n, R, 80 + t, scale=3000.0 if clip else 1e-3)
        hp = U.hp_for(t)
        a.step(grads, w, m, v, hp, step=t)
        if via_step:                           # b steps in place on its current buffer
            b.step(grads, *bufs[cur], hp, step=t)
        else:
            b.step_fused(grads, *bufs[cur], *bufs[1 - cur], hp, step=t)
            cur = 1 - cur
        a.sync()
        b.sync()
        for x, y in zip((w, m, v), bufs[cur]):
            assert torch.equal(x.view(torch.int32), y.view(torch.int32)), t
        assert torch.equal(a.leaves_view(), b.leaves_view()), t


def test_fused_matches_the_oracle():
    n, R = 2 * CH + 333, 8
    dev = torch.device("cuda", 0)
    ctx = rs.Repstep(n, device=dev)
    w, m, v = I.gen_state(U.F32_WL, n=n, device=dev)
    ow, om, ov = (x.cpu().numpy() for x in (w, m, v))
    bufs = [(w, m, v), (torch.empty_like(w), torch.empty_like(m), torch.empty_like(v))]
    nr = torch.empty(1, dtype=torch.float32, device=dev)
    rr = torch.empty(1, dtype=torch.int64, device=dev)
    for t in (1, 2, 3):
        grads = U.gen_grads(n, R, 70 + t, scale=3000.0 if t == 2 else 1.0)
        ctx.step_fused(grads, *bufs[(t - 1) % 2], *bufs[t % 2], U.hp_for(t), step=t,
                       norm_out=nr, root_out=rr)
        ctx.sync()
        ref = U.oracle_step(U.oracle_grads(grads), ow, om, ov, t)
        ow, om, ov = ref["w"], ref["m"], ref["v"]
        for got, want, what in zip(bufs[t % 2], (ow, om, ov), "wmv"):
            U.assert_same_f32(got, want, f"{what} step {t}")
        assert np.float32(nr.item()) == ref["norm"] and U.root_of(rr) == ref["root"]


def test_fused_rejects_overlapping_buffers():
    n, R = CH, 4
    dev = torch.device("cuda", 0)
    ctx = rs.Repstep(n, device=dev)
    w, m, v = I.gen_state(U.F32_WL, n=n, device=dev)
    grads = U.gen_grads(n, R, 1)
    hp = U.hp_for(1)
    big = torch.zeros(2 * n, device=dev)
    with pytest.raises(rs.RepstepError):
        ctx.step_fused(grads, w, m, v, w, torch.empty_like(m), torch.empty_like(v), hp, 1)
    with pytest.raises(rs.RepstepError):             # partial overlap
        ctx.step_fused(grads, big[:n], m, v, big[n // 2:n // 2 + n], torch.empty_like(m),
                       torch.empty_like(v), hp, 1)
    L = rs.lib()
    arr = (C.c_void_p * R)(*[g.data_ptr() for g in grads])
    rc = L.repstep_step_fused(ctx._ctx, arr, R, C.c_void_p(w.data_ptr() + 4), None, None, None,
                              None, None, C.byref(hp), 1, None, None)
    assert rc in (1, 2)
    assert ctx.sync() == 0


@pytest.mark.big
def test_flat1200m_r8_fused_equals_two_pass():
    """The benchmark workload, 3 steps: the single pass every step (no clipping), equal to
    repstep_step bit for bit, and the input state untouched."""
    wl = I.WORKLOADS["flat1200m_r8_segscale"]
    n, R = wl.n, wl.R
    dev = torch.device("cuda", 0)
    a, b = rs.Repstep(n, device=dev), rs.Repstep(n, device=dev)
    b.set_hash_stream(torch.cuda.Stream(dev))          # the roots beside the next pass
    w, m, v = I.gen_state(wl, device=dev)
    bufs = [(w.clone(), m.clone(), v.clone()),
            (torch.empty_like(w), torch.empty_like(m), torch.empty_like(v))]
    grads = [torch.empty(n, device=dev) for _ in range(R)]
    nr = torch.empty(2, dtype=torch.float32, device=dev)
    rr = torch.empty(2, dtype=torch.int64, device=dev)
    for t in (1, 2, 3):
        for r in range(R):
            I.gen_grad(wl, t, r, device=dev, out=grads[r])
        hp = U.hp_for(t)
        a.step(grads, w, m, v, hp, step=t, norm_out=nr[0:1], root_out=rr[0:1])
        b.step_fused(grads, *bufs[(t - 1) % 2], *bufs[t % 2], hp, step=t, norm_out=nr[1:2],
                     root_out=rr[1:2])
        a.sync()
        b.sync()
        assert nr[0].item() == nr[1].item() < 1.0
        rh = rr.cpu().numpy().view(np.uint64)
        assert rh[0] == rh[1]
        for x, y in zip((w, m, v), bufs[t % 2]):
            assert torch.equal(x.view(torch.int32), y.view(torch.int32))


def test_pass_events_time_the_single_pass():
    """repstep_set_pass_events: the events bracket the single pass of each call while set;
    cleared, they are left alone; one null and one event is an argument error."""
    n, R = 64 * CH, 8
    dev = torch.device("cuda", 0)
    ctx = rs.Repstep(n, device=dev)
    st = torch.cuda.current_stream(dev)
    w, m, v = I.gen_state(U.F32_WL, n=n, device=dev)
    bufs = [(w, m, v), tuple(torch.empty_like(x) for x in (w, m, v))]
    ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with pytest.raises(rs.RepstepError):          # not yet created
        ctx.set_pass_events(ea, eb)
    ea.record(st)
    eb.record(st)
    with pytest.raises(rs.RepstepError):
        rs._check(rs.lib().repstep_set_pass_events(ctx._ctx, C.c_void_p(ea.cuda_event), None),
                  "one event")
    grads = U.gen_grads(n, R, 5, scale=1e-3)
    outer_a, outer_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ctx.set_pass_events(ea, eb)
    outer_a.record(st)
    ctx.step_fused(grads, *bufs[0], *bufs[1], U.hp_for(1), step=1)
    outer_b.record(st)
    ctx.set_pass_events(None, None)
    ctx.sync()
    inner = ea.elapsed_time(eb)
    assert 0.0 < inner <= outer_a.elapsed_time(outer_b)
    ctx.step_fused(grads, *bufs[1], *bufs[0], U.hp_for(2), step=2)   # cleared: not recorded
    ctx.sync()
    assert ea.elapsed_time(eb) == inner


def test_empty_state():
    """n = 0: no arrays are read; the root is the header's, as repstep_step's."""
    dev = torch.device("cuda", 0)
    a, b = rs.Repstep(0, device=dev), rs.Repstep(0, device=dev)
    e = torch.empty(0, device=dev)
    grads = [torch.empty(0, device=dev) for _ in range(4)]
    nr = torch.empty(2, dtype=torch.float32, device=dev)
    rr = torch.empty(2, dtype=torch.int64, device=dev)
    hp = U.hp_for(1)
    a.step(grads, e, e.clone(), e.clone(), hp, step=1, norm_out=nr[0:1], root_out=rr[0:1])
    b.step_fused(grads, e, e.clone(), e.clone(), torch.empty(0, device=dev),
                 torch.empty(0, device=dev), torch.empty(0, device=dev), hp, step=1,
                 norm_out=nr[1:2], root_out=rr[1:2])
    assert a.sync() == 0 and b.sync() == 0
    assert nr[0].item() == nr[1].item() == 0.0
    rh = rr.cpu().numpy().view(np.uint64)
    assert rh[0] == rh[1]


def test_prediction_chooses_the_path():
    """The host's prediction, seen through the library's launch count: after a step that
    did not clip (or at the start) the call launches the single pass and the two gated
    second-pass kernels; after one that clipped, the reduce and AdamW of the two passes --
    one launch fewer.  Synchronising after each step makes the outcome visible to the host
    before the next call."""
    n, R = 5 * CH + 77, 8
    dev = torch.device("cuda", 0)
    ctx = rs.Repstep(n, device=dev)
    w, m, v = I.gen_state(U.F32_WL, n=n, device=dev)
    bufs = [(w, m, v), tuple(torch.empty_like(x) for x in (w, m, v))]
    launches = []
    clips = [False, True, True, False, False]
    for t, clip in enumerate(clips, start=1):
        grads = U.gen_grads(n, R, 120 + t, scale=3000.0 if clip else 1e-3)
        before = ctx.launch_count()
        ctx.step_fused(grads, *bufs[(t - 1) % 2], *bufs[t % 2], U.hp_for(t), step=t)
        launches.append(ctx.launch_count() - before)
        ctx.sync()
    single, two = launches[0], launches[0] - 1
    # step 2 is predicted not to clip (step 1 did not), step 3 and 4 to clip, step 5 not
    assert launches == [single, single, two, two, single], launches
